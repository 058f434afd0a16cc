"""GPU parity for speculative tree verify and commit.

* tree outputs vs the oracle's root-path replay (tolerance);
* the committed state vs the oracle (tolerance);
* bit-exact GPU vs GPU: a node's verify output == decode of its root path,
  the committed state == decode of the accepted path, and the conv tail is
  exactly the last four inputs."""
import numpy as np
import pytest
import torch

from gdn_testutil import (assert_out_close, assert_state_close, bf16, f32, gdn, gen, host, oracle,
                          oracle_conv_then_round)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from hybrid_linear_attention_conv_gb300 import build
    build.build()
    gdn.load()


def _tree_case(shape, N, seed, max_depth=8, parents=None):
    s1 = shape.with_batch(1)
    if parents is None:
        parents = gen.random_tree(seed, N, max_depth)
    d = gen.decode_inputs(seed, s1, N, tag="tree")
    return parents, {"qkv": d["qkv"][0], "alpha": d["alpha"][0], "beta": d["beta"][0],
                     "state": d["state"][0]}


def _verify(shape, parents, d, **kw):
    st = f32(d["state"])
    before = st.clone()
    out = gdn.tree_verify(parents, bf16(d["qkv"]), f32(d["alpha"]), f32(d["beta"]), st, shape.Hk,
                          shape.Hv, shape.dk, shape.dv, **kw)
    torch.cuda.synchronize()
    assert torch.equal(st, before), "tree verify must not write the committed state"
    return out


def _path_decode(shape, d, path):
    """GPU linear decode of the gathered path inputs: (outputs, final state)."""
    st = f32(d["state"][None])
    out = gdn.decode_step(bf16(d["qkv"][None, path]), f32(d["alpha"][None, path]),
                          f32(d["beta"][None, path]), st, shape.Hk, shape.Hv, shape.dk, shape.dv)
    torch.cuda.synchronize()
    return out[0], st[0]


@pytest.mark.parametrize("shape", [gen.TINY, gen.QWEN_27B])
def test_tree_verify_vs_oracle(shape):
    parents, d = _tree_case(shape, 32, 1)
    out = _verify(shape, parents, d)
    ref = oracle.tree_verify(parents, d["qkv"], d["alpha"], d["beta"], d["state"], shape.Hk, shape.Hv,
                             shape.dk, shape.dv)
    assert_out_close(host(out), ref)


def test_tree_verify_outputs_equal_decode_bitwise():
    shape = gen.QWEN_27B
    parents, d = _tree_case(shape, 32, 2)
    out = _verify(shape, parents, d)
    for n in range(32):
        path = gdn.tree_root_path(parents, n)
        o, _ = _path_decode(shape, d, path)
        assert torch.equal(out[n], o[-1]), f"node {n}"


def _binary_tree(n):
    return np.array([-1] + [(i - 1) // 2 for i in range(1, n)], np.int32)


def _caterpillar(n):
    """A spine whose every node also has one leaf."""
    parents = [-1]
    spine = 0
    while len(parents) < n:
        parents.append(spine)
        nxt = len(parents) - 1
        if len(parents) < n:
            parents.append(spine)
        spine = nxt
    return np.array(parents, np.int32)


@pytest.mark.parametrize("parents", [_binary_tree(63), _caterpillar(17), gen.random_tree(11, 64, 8),
                                     gen.random_tree(12, 48, 12), gen.random_tree(13, 64, 4)])
def test_tree_walk_shapes_equal_decode_bitwise(parents):
    """Whatever walk the host schedules (the tree split between walkers where
    that shortens the walk and their branch states fit, else one depth-first
    walk), every node's output is the bits of the linear decode of its root
    path."""
    shape = gen.QWEN_27B
    _, d = _tree_case(shape, len(parents), 5, parents=parents)
    out = _verify(shape, parents, d)
    for n in range(len(parents)):
        o, _ = _path_decode(shape, d, gdn.tree_root_path(parents, n))
        assert torch.equal(out[n], o[-1]), f"node {n}"


@pytest.mark.parametrize("parents", [gen.random_tree(1234, 32, 8), gen.random_tree(0, 32, 8), _caterpillar(17),
                                     gen.random_tree(12, 48, 12), gen.random_tree(3, 8, 8), _binary_tree(63),
                                     np.arange(-1, 31, dtype=np.int32)])
def test_walkers_equal_one_walker_bitwise(parents):
    """A single tree's verify splits the tree between up to three walkers
    (CTAs holding the same rows, each walking part of the tree) when that
    shortens the walk; the joint verify (one tree here) always walks it whole.
    Both give the same bits, with post-conv and pre-conv inputs."""
    shape = gen.QWEN_27B
    N = len(parents)
    _, d = _tree_case(shape, N, 21, parents=parents)
    out = _verify(shape, parents, d)
    joint = gdn.tree_verify_batched(np.array([N], np.int32), parents[None], bf16(d["qkv"][None]),
                                    f32(d["alpha"][None]), f32(d["beta"][None]), f32(d["state"][None]),
                                    shape.Hk, shape.Hv, shape.dk, shape.dv)
    torch.cuda.synchronize()
    assert torch.equal(out, joint[0])
    c = gen.conv_inputs(22, 1, N, shape.C, tag="walkers")
    w = bf16(c["w"])
    fused = gdn.conv_tree_verify(parents, bf16(c["x"][0]), w, bf16(c["tail"][0]), f32(d["alpha"]),
                                 f32(d["beta"]), f32(d["state"]), shape.Hk, shape.Hv, shape.dk, shape.dv)
    fused_joint = gdn.conv_tree_verify_batched(np.array([N], np.int32), parents[None], bf16(c["x"]), w,
                                               bf16(c["tail"]), f32(d["alpha"][None]), f32(d["beta"][None]),
                                               f32(d["state"][None]), shape.Hk, shape.Hv, shape.dk, shape.dv)
    torch.cuda.synchronize()
    assert torch.equal(fused, fused_joint[0])


@pytest.mark.parametrize("parents", [
    np.array([-1], np.int32),                                  # a single node
    np.arange(-1, 63, dtype=np.int32),                         # a 64-long chain (no branch states)
    np.array([-1] + [0] * 31, np.int32),                       # a star: 31 children of the root
    np.array([-1, 0, 0, 1, 1, 2, 3, 3, 4, 6, 6, 9, 10], np.int32),  # 13 nodes (not a multiple of 4)
])
def test_tree_verify_degenerate_shapes(parents):
    shape = gen.Shape(1, 2, 4, 64, 64)
    _, d = _tree_case(shape, len(parents), 3, parents=parents)
    out = _verify(shape, parents, d)
    ref = oracle.tree_verify(parents, d["qkv"], d["alpha"], d["beta"], d["state"], shape.Hk, shape.Hv,
                             shape.dk, shape.dv)
    assert_out_close(host(out), ref)


def _nested_branch_tree(levels):
    parents = [-1]
    spine = 0
    for _ in range(levels):
        parents.append(spine)
        nxt = len(parents) - 1
        parents.append(spine)
        spine = nxt
    return np.array(parents, np.int32)


def test_tree_verify_max_branch_states():
    """Exactly GDN_MAX_TREE_SLOTS nested branching nodes is accepted and correct."""
    shape = gen.Shape(1, 2, 4, 128, 128)
    parents = _nested_branch_tree(gdn.GDN_MAX_TREE_SLOTS)
    _, d = _tree_case(shape, len(parents), 4, parents=parents)
    out = _verify(shape, parents, d)
    ref = oracle.tree_verify(parents, d["qkv"], d["alpha"], d["beta"], d["state"], shape.Hk, shape.Hv,
                             shape.dk, shape.dv)
    assert_out_close(host(out), ref)


def test_tree_verify_bf16_out_and_scale():
    shape = gen.Shape(1, 2, 6, 64, 64)
    parents, d = _tree_case(shape, 20, 5)
    out = _verify(shape, parents, d, q_scale=0.5, out_bf16=True)
    ref = oracle.tree_verify(parents, d["qkv"], d["alpha"], d["beta"], d["state"], shape.Hk, shape.Hv,
                             shape.dk, shape.dv, q_scale=0.5)
    got = gen.bf16_bits_to_f32(host(out)).astype(np.float64)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-3)


@pytest.mark.parametrize("shape", [gen.TINY, gen.QWEN_27B])
def test_commit_vs_oracle_and_decode_bitwise(shape):
    N = 32
    parents, d = _tree_case(shape, N, 6)
    c = gen.conv_inputs(6, 1, N, shape.C)
    leaf = gen.random_leaf(6, parents)
    path = gdn.tree_root_path(parents, leaf)
    assert np.array_equal(path, oracle.root_path(parents, leaf))
    st = f32(d["state"])
    tail = bf16(c["tail"][0])
    gdn.commit_path(parents, path, bf16(d["qkv"]), f32(d["alpha"]), f32(d["beta"]), st, shape.Hk,
                    shape.Hv, shape.dk, shape.dv, x_tree=bf16(c["x"][0]), tail=tail)
    torch.cuda.synchronize()
    st_ref, tail_ref = oracle.commit(parents, path, d["qkv"], d["alpha"], d["beta"], d["state"],
                                     shape.Hk, shape.Hv, shape.dk, shape.dv, x_tree=c["x"][0],
                                     tail=c["tail"][0])
    assert_state_close(host(st), st_ref)
    assert np.array_equal(host(tail), tail_ref)
    _, st_dec = _path_decode(shape, d, path)
    assert torch.equal(st, st_dec), "commit must equal the linear decode of the path bit for bit"


def test_commit_every_prefix_length():
    shape = gen.Shape(1, 2, 4, 64, 64)
    parents = np.arange(-1, 11, dtype=np.int32)  # chain of 12
    _, d = _tree_case(shape, 12, 7, parents=parents)
    c = gen.conv_inputs(7, 1, 12, shape.C)
    for L in range(0, 13):
        path = np.arange(L, dtype=np.int32)
        st = f32(d["state"])
        tail = bf16(c["tail"][0])
        gdn.commit_path(parents, path, bf16(d["qkv"]), f32(d["alpha"]), f32(d["beta"]), st, shape.Hk,
                        shape.Hv, shape.dk, shape.dv, x_tree=bf16(c["x"][0]), tail=tail)
        torch.cuda.synchronize()
        st_ref, tail_ref = oracle.commit(parents, path, d["qkv"], d["alpha"], d["beta"], d["state"],
                                         shape.Hk, shape.Hv, shape.dk, shape.dv, x_tree=c["x"][0],
                                         tail=c["tail"][0])
        assert np.array_equal(host(tail), tail_ref), L
        if L == 0:
            assert np.array_equal(host(st), d["state"])
        else:
            assert_state_close(host(st), st_ref)


def test_speculative_round_end_to_end():
    """One round at the 27B shape: tree conv -> verify -> commit (state and
    tail), compared with the oracle's conv + verify + commit, and the commit
    compared bitwise with conv + decode of the accepted path from scratch."""
    shape = gen.QWEN_27B
    N = 32
    parents = gen.random_tree(8, N, 8)
    c = gen.conv_inputs(8, 1, N, shape.C)
    d = gen.decode_inputs(8, shape, N, tag="round")
    w = bf16(c["w"])
    tail = bf16(c["tail"])
    x_tree = bf16(c["x"])
    y_tree = gdn.conv_step(x_tree, w, tail, parents=parents)
    st = f32(d["state"][0])
    al, be = f32(d["alpha"][0]), f32(d["beta"][0])
    out = gdn.tree_verify(parents, y_tree[0], al, be, st, shape.Hk, shape.Hv, shape.dk, shape.dv)
    leaf = gen.random_leaf(8, parents)
    path = gdn.tree_root_path(parents, leaf)
    gdn.commit_path(parents, path, y_tree[0], al, be, st, shape.Hk, shape.Hv, shape.dk, shape.dv,
                    x_tree=x_tree[0], tail=tail[0])
    torch.cuda.synchronize()

    y_ref = oracle.conv_tree_r32(parents, c["x"][0], c["w"], c["tail"][0])  # bf16 rounding decided in binary32
    out_ref = oracle.tree_verify(parents, y_ref, d["alpha"][0], d["beta"][0], d["state"][0], shape.Hk,
                                 shape.Hv, shape.dk, shape.dv)
    st_ref, tail_ref = oracle.commit(parents, path, y_ref, d["alpha"][0], d["beta"][0], d["state"][0],
                                     shape.Hk, shape.Hv, shape.dk, shape.dv, x_tree=c["x"][0],
                                     tail=c["tail"][0])
    assert_out_close(host(out), out_ref)
    assert_state_close(host(st), st_ref)
    assert np.array_equal(host(tail[0]), tail_ref)

    # the same tokens decoded linearly from the pre-round state and tail
    tail2 = bf16(c["tail"])
    y_lin = gdn.conv_step(bf16(c["x"][:, path]), w, tail2)
    st2 = f32(d["state"][0:1])
    gdn.decode_step(y_lin, f32(d["alpha"][:, path]), f32(d["beta"][:, path]), st2, shape.Hk, shape.Hv,
                    shape.dk, shape.dv)
    torch.cuda.synchronize()
    assert torch.equal(st2[0], st)
    assert torch.equal(tail2[0], tail[0])


# ---------------------------------------------------------------------------
# joint verify of several sequences' trees (different sizes and shapes)
# ---------------------------------------------------------------------------
def _pad_parents(trees, N):
    out = np.full((len(trees), N), -7, np.int32)  # junk past each tree's size
    for b, t in enumerate(trees):
        out[b, :len(t)] = t
    return out


@pytest.mark.parametrize("shape", [gen.QWEN_27B, gen.Shape(1, 2, 4, 64, 64)])
def test_tree_verify_batched_equals_single_and_oracle(shape):
    N = 32
    trees = [gen.random_tree(40, 32, 8), np.array([-1], np.int32), gen.random_tree(41, 13, 5),
             gen.random_tree(42, 20, 8), np.arange(-1, 6, dtype=np.int32)]
    B = len(trees)
    counts = np.array([len(t) for t in trees], np.int32)
    parents = _pad_parents(trees, N)
    d = gen.decode_inputs(43, shape.with_batch(B), N, tag="treeb")
    st = f32(d["state"])
    before = st.clone()
    out = torch.full((B, N, shape.Hv, shape.dv), float("nan"), device="cuda")
    gdn.tree_verify_batched(counts, parents, bf16(d["qkv"]), f32(d["alpha"]), f32(d["beta"]), st, shape.Hk,
                            shape.Hv, shape.dk, shape.dv, out=out)
    torch.cuda.synchronize()
    assert torch.equal(st, before), "verify must not write the committed states"
    for b, t in enumerate(trees):
        n = len(t)
        assert torch.isnan(out[b, n:]).all(), "rows past the tree's size must stay untouched"
        single = gdn.tree_verify(t, bf16(d["qkv"][b, :n]), f32(d["alpha"][b, :n]), f32(d["beta"][b, :n]),
                                 f32(d["state"][b]), shape.Hk, shape.Hv, shape.dk, shape.dv)
        torch.cuda.synchronize()
        assert torch.equal(out[b, :n], single), f"tree {b}"
        ref = oracle.tree_verify(t, d["qkv"][b, :n], d["alpha"][b, :n], d["beta"][b, :n], d["state"][b], shape.Hk,
                                 shape.Hv, shape.dk, shape.dv)
        assert_out_close(host(out[b, :n]), ref)


@pytest.mark.parametrize("shape", [gen.QWEN_27B, gen.Shape(1, 2, 4, 64, 64)])
def test_commit_path_batched_equals_single_commits_and_oracle(shape):
    """A joint verify's sequences commit their accepted paths in one launch:
    each sequence's state and tail equal gdn_commit_path on its tree alone, bit
    for bit, and the oracle's commit within the bars; a sequence that accepts
    nothing keeps its state and tail."""
    N = 32
    trees = [gen.random_tree(50, 32, 8), np.array([-1], np.int32), gen.random_tree(51, 13, 5),
             gen.random_tree(52, 20, 8), np.arange(-1, 6, dtype=np.int32)]
    B = len(trees)
    counts = np.array([len(t) for t in trees], np.int32)
    parents = _pad_parents(trees, N)
    paths = np.full((B, N), -9, np.int32)
    lengths = np.zeros(B, np.int32)
    for b, t in enumerate(trees):
        if b == 3:
            continue  # nothing accepted
        p = gdn.tree_root_path(t, gen.random_leaf(60 + b, t))
        paths[b, :len(p)] = p
        lengths[b] = len(p)
    d = gen.decode_inputs(53, shape.with_batch(B), N, tag="commitb")
    c = gen.conv_inputs(54, B, N, shape.C, tag="commitb")
    qkv, al, be, xt = bf16(d["qkv"]), f32(d["alpha"]), f32(d["beta"]), bf16(c["x"])
    st = f32(d["state"])
    tail = bf16(c["tail"])
    gdn.commit_path_batched(counts, parents, paths, lengths, qkv, al, be, st, shape.Hk, shape.Hv, shape.dk,
                            shape.dv, x_tree=xt, tail=tail)
    torch.cuda.synchronize()
    for b, t in enumerate(trees):
        n, L = len(t), int(lengths[b])
        st_1 = f32(d["state"][b])
        tail_1 = bf16(c["tail"][b])
        gdn.commit_path(t, paths[b, :L], qkv[b, :n].contiguous(), al[b, :n].contiguous(), be[b, :n].contiguous(),
                        st_1, shape.Hk, shape.Hv, shape.dk, shape.dv, x_tree=xt[b, :n].contiguous(), tail=tail_1)
        torch.cuda.synchronize()
        assert torch.equal(st[b], st_1), f"sequence {b}: state"
        assert torch.equal(tail[b], tail_1), f"sequence {b}: tail"
        if L == 0:
            assert np.array_equal(host(st[b]), d["state"][b]) and np.array_equal(host(tail[b]), c["tail"][b])
            continue
        st_ref, tail_ref = oracle.commit(t, paths[b, :L], d["qkv"][b, :n], d["alpha"][b, :n], d["beta"][b, :n],
                                         d["state"][b], shape.Hk, shape.Hv, shape.dk, shape.dv,
                                         x_tree=c["x"][b, :n], tail=c["tail"][b])
        assert_state_close(host(st[b]), st_ref)
        assert np.array_equal(host(tail[b]), tail_ref)


# ---------------------------------------------------------------------------
# the round with the conv fused into verify and commit (pre-conv inputs)
# ---------------------------------------------------------------------------
_FUSED_TREES = {
    "random32": gen.random_tree(70, 32, 8),
    "chain64": np.arange(-1, 63, dtype=np.int32),   # no branch states: the conv outputs alone size the slot region
    "binary63": _binary_tree(63),                    # several branch states
    "single": np.array([-1], np.int32),
    "random13": np.array([-1, 0, 0, 1, 1, 2, 3, 3, 4, 6, 6, 9, 10], np.int32),
}


def _conv_case(shape, N, seed, B=1, tag="fused"):
    c = gen.conv_inputs(seed, B, N, shape.C, tag=tag)
    d = gen.decode_inputs(seed + 1, shape.with_batch(B), N, tag=tag)
    return c, d


@pytest.mark.parametrize("shape", [gen.TINY, gen.QWEN_27B, gen.Shape(1, 2, 4, 64, 64)])
@pytest.mark.parametrize("tree", sorted(_FUSED_TREES))
def test_conv_tree_verify_equals_conv_then_verify(shape, tree):
    """gdn_conv_tree_verify == gdn_conv_step (tree mode) + gdn_tree_verify, bit
    for bit; the committed state and the tail are left untouched."""
    parents = _FUSED_TREES[tree]
    N = len(parents)
    c, d = _conv_case(shape, N, 72)
    x, w, tail = bf16(c["x"][0]), bf16(c["w"]), bf16(c["tail"][0])
    al, be, st = f32(d["alpha"][0]), f32(d["beta"][0]), f32(d["state"][0])
    y = gdn.conv_step(x[None], w, tail[None].clone(), parents=parents)[0]
    ref = gdn.tree_verify(parents, y, al, be, st, shape.Hk, shape.Hv, shape.dk, shape.dv)
    out = gdn.conv_tree_verify(parents, x, w, tail, al, be, st, shape.Hk, shape.Hv, shape.dk, shape.dv)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert np.array_equal(host(st), d["state"][0]) and np.array_equal(host(tail), c["tail"][0])


@pytest.mark.parametrize("out_bf16,q_scale", [(True, 1.0), (False, 0.0884), (True, 0.0884)])
def test_conv_tree_verify_flags_equal_unfused(out_bf16, q_scale):
    """bf16 outputs and a q scale (1/sqrt(128)) through the fused verify: the
    bits of conv + unfused verify with the same flags, on the 27B shape."""
    shape = gen.QWEN_27B
    parents = _FUSED_TREES["random32"]
    N = len(parents)
    c, d = _conv_case(shape, N, 73)
    x, w, tail = bf16(c["x"][0]), bf16(c["w"]), bf16(c["tail"][0])
    al, be, st = f32(d["alpha"][0]), f32(d["beta"][0]), f32(d["state"][0])
    y = gdn.conv_step(x[None], w, tail[None].clone(), parents=parents)[0]
    ref = gdn.tree_verify(parents, y, al, be, st, shape.Hk, shape.Hv, shape.dk, shape.dv, q_scale=q_scale,
                          out_bf16=out_bf16)
    out = gdn.conv_tree_verify(parents, x, w, tail, al, be, st, shape.Hk, shape.Hv, shape.dk, shape.dv,
                               q_scale=q_scale, out_bf16=out_bf16)
    torch.cuda.synchronize()
    assert out.dtype == (torch.bfloat16 if out_bf16 else torch.float32)
    assert torch.equal(out, ref)


@pytest.mark.parametrize("shape", [gen.TINY, gen.Shape(1, 2, 4, 64, 64)])
def test_conv_round_batched_small_shapes(shape):
    """The joint fused verify and batched fused commit at the small head
    shapes (clusters of two CTAs): equal to the per-sequence fused calls."""
    N = 20
    trees = [gen.random_tree(120, 20, 6), gen.random_tree(121, 7, 4), np.array([-1], np.int32)]
    B = len(trees)
    counts = np.array([len(t) for t in trees], np.int32)
    parents = _pad_parents(trees, N)
    paths = np.full((B, N), -9, np.int32)
    lengths = np.zeros(B, np.int32)
    for b, t in enumerate(trees):
        p = gdn.tree_root_path(t, gen.random_leaf(130 + b, t))
        paths[b, :len(p)] = p
        lengths[b] = len(p)
    c, d = _conv_case(shape, N, 131, B=B, tag="roundsmall")
    x, w, tail = bf16(c["x"]), bf16(c["w"]), bf16(c["tail"])
    al, be, st = f32(d["alpha"]), f32(d["beta"]), f32(d["state"])
    out = gdn.conv_tree_verify_batched(counts, parents, x, w, tail, al, be, st, shape.Hk, shape.Hv, shape.dk,
                                       shape.dv)
    tail_out = torch.empty_like(tail)
    gdn.conv_commit_path_batched(counts, parents, paths, lengths, x, w, tail, tail_out, al, be, st, shape.Hk,
                                 shape.Hv, shape.dk, shape.dv)
    torch.cuda.synchronize()
    for b, t in enumerate(trees):
        n, L = len(t), int(lengths[b])
        xb, alb, beb = x[b, :n].contiguous(), al[b, :n].contiguous(), be[b, :n].contiguous()
        st1 = f32(d["state"][b])
        o1 = gdn.conv_tree_verify(t, xb, w, tail[b], alb, beb, st1, shape.Hk, shape.Hv, shape.dk, shape.dv)
        t1 = torch.empty_like(tail[b])
        gdn.conv_commit_path(t, paths[b, :L], xb, w, tail[b], t1, alb, beb, st1, shape.Hk, shape.Hv, shape.dk,
                             shape.dv)
        torch.cuda.synchronize()
        assert torch.equal(out[b, :n], o1) and torch.equal(st[b], st1) and torch.equal(tail_out[b], t1), b
        # and the oracle (conv outputs rounded from binary32, as the kernels round them)
        y_ref = oracle.conv_tree_r32(t, c["x"][b, :n], c["w"], c["tail"][b])
        out_ref = oracle.tree_verify(t, y_ref, d["alpha"][b, :n], d["beta"][b, :n], d["state"][b], shape.Hk,
                                     shape.Hv, shape.dk, shape.dv)
        assert_out_close(host(o1), out_ref)


@pytest.mark.parametrize("shape", [gen.TINY, gen.QWEN_27B])
def test_conv_commit_equals_conv_then_commit_every_prefix(shape):
    """gdn_conv_commit_path == gdn_conv_step (tree mode) + gdn_commit_path with
    x_tree, bit for bit, for every prefix of a root-to-leaf path (L = 0
    included: the state stays and tail_in is copied to tail_out)."""
    parents = gen.random_tree(74, 32, 8)
    path = gdn.tree_root_path(parents, gen.random_leaf(74, parents))
    N = len(parents)
    c, d = _conv_case(shape, N, 75)
    x, w = bf16(c["x"][0]), bf16(c["w"])
    al, be = f32(d["alpha"][0]), f32(d["beta"][0])
    y = gdn.conv_step(x[None], w, bf16(c["tail"]), parents=parents)[0]
    for L in range(len(path) + 1):
        st1, tail1 = f32(d["state"][0]), bf16(c["tail"][0])
        gdn.commit_path(parents, path[:L], y, al, be, st1, shape.Hk, shape.Hv, shape.dk, shape.dv, x_tree=x,
                        tail=tail1)
        st2, tail_in = f32(d["state"][0]), bf16(c["tail"][0])
        tail_out = torch.full_like(tail_in, 0x7FC0)  # junk: every entry must be written
        gdn.conv_commit_path(parents, path[:L], x, w, tail_in, tail_out, al, be, st2, shape.Hk, shape.Hv, shape.dk,
                             shape.dv)
        torch.cuda.synchronize()
        assert torch.equal(st1, st2), f"L={L}: state"
        assert torch.equal(tail1, tail_out), f"L={L}: tail"
        assert np.array_equal(host(tail_in), c["tail"][0]), "tail_in is read only"


def test_conv_commit_long_path():
    """A 64-node chain accepted whole: the longest path (64 tokens of conv
    outputs in shared memory)."""
    shape = gen.QWEN_27B
    parents = np.arange(-1, 63, dtype=np.int32)
    path = np.arange(64, dtype=np.int32)
    c, d = _conv_case(shape, 64, 76)
    x, w = bf16(c["x"][0]), bf16(c["w"])
    al, be = f32(d["alpha"][0]), f32(d["beta"][0])
    y = gdn.conv_step(x[None], w, bf16(c["tail"]), parents=parents)[0]
    st1, tail1 = f32(d["state"][0]), bf16(c["tail"][0])
    gdn.commit_path(parents, path, y, al, be, st1, shape.Hk, shape.Hv, shape.dk, shape.dv, x_tree=x, tail=tail1)
    st2, tail_out = f32(d["state"][0]), torch.empty_like(tail1)
    gdn.conv_commit_path(parents, path, x, w, bf16(c["tail"][0]), tail_out, al, be, st2, shape.Hk, shape.Hv,
                         shape.dk, shape.dv)
    torch.cuda.synchronize()
    assert torch.equal(st1, st2) and torch.equal(tail1, tail_out)


def test_fused_rounds_vs_oracle_and_unfused():
    """Two speculative rounds at the 27B shape with the conv fused in (tails
    alternating between two buffers): each round's outputs, the state and the
    tail equal the three-launch round bit for bit, and the oracle's conv +
    verify + commit within the bars.  The oracle's conv rounds its outputs to
    bf16 from binary32, as the kernels do: from fp64, the rare outputs within
    an ulp or two of a bf16 midpoint land one bf16 ulp apart, and a single
    such v input moves a node's output by about 1e-3."""
    shape = gen.QWEN_27B
    N = 32
    c, d = _conv_case(shape, N, 78, B=2, tag="rounds")
    w = bf16(c["w"])
    st_f, st_u = f32(d["state"][0]), f32(d["state"][0])
    tails = [bf16(c["tail"][0]), torch.empty_like(bf16(c["tail"][0]))]
    tail_u = bf16(c["tail"][0])
    st_ref, tail_ref = d["state"][0], c["tail"][0]
    for r in range(2):
        parents = gen.random_tree(80 + r, N, 8)
        path = gdn.tree_root_path(parents, gen.random_leaf(80 + r, parents))
        x = bf16(c["x"][r])
        al, be = f32(d["alpha"][r]), f32(d["beta"][r])
        tin, tout = tails[r % 2], tails[(r + 1) % 2]
        out_f = gdn.conv_tree_verify(parents, x, w, tin, al, be, st_f, shape.Hk, shape.Hv, shape.dk, shape.dv)
        gdn.conv_commit_path(parents, path, x, w, tin, tout, al, be, st_f, shape.Hk, shape.Hv, shape.dk, shape.dv)
        y = gdn.conv_step(x[None], w, tail_u[None].clone(), parents=parents)[0]
        out_u = gdn.tree_verify(parents, y, al, be, st_u, shape.Hk, shape.Hv, shape.dk, shape.dv)
        gdn.commit_path(parents, path, y, al, be, st_u, shape.Hk, shape.Hv, shape.dk, shape.dv, x_tree=x,
                        tail=tail_u)
        torch.cuda.synchronize()
        assert torch.equal(out_f, out_u), f"round {r}: outputs"
        assert torch.equal(st_f, st_u), f"round {r}: state"
        assert torch.equal(tout, tail_u), f"round {r}: tail"
        # the conv outputs' bf16 rounding decided in binary32 on both sides
        y_ref = oracle.conv_tree_r32(parents, c["x"][r], c["w"], tail_ref)
        out_ref = oracle.tree_verify(parents, y_ref, d["alpha"][r], d["beta"][r], st_ref, shape.Hk, shape.Hv,
                                     shape.dk, shape.dv)
        st_ref, tail_ref = oracle.commit(parents, path, y_ref, d["alpha"][r], d["beta"][r], st_ref, shape.Hk,
                                         shape.Hv, shape.dk, shape.dv, x_tree=c["x"][r], tail=tail_ref)
        assert_out_close(host(out_f), out_ref)
        assert_state_close(host(st_f), st_ref)
        assert np.array_equal(host(tout), tail_ref)


@pytest.mark.parametrize("B", [5, 8, 14])  # one, two and four rows per thread in the commit at the 27B shape
def test_conv_round_batched_equals_single(B):
    """The joint verify and the batched commit with the conv fused in equal
    the single-sequence fused calls bit for bit (sequence 1 accepts nothing:
    its state stays and its tail is copied)."""
    shape = gen.QWEN_27B
    N = 32
    base = [gen.random_tree(90, 32, 8), np.array([-1], np.int32), gen.random_tree(91, 13, 5),
            gen.random_tree(92, 20, 8), np.arange(-1, 6, dtype=np.int32)]
    trees = [base[b % len(base)] if b < len(base) else gen.random_tree(93 + b, 32, 8) for b in range(B)]
    counts = np.array([len(t) for t in trees], np.int32)
    parents = _pad_parents(trees, N)
    paths = np.full((B, N), -9, np.int32)
    lengths = np.zeros(B, np.int32)
    for b, t in enumerate(trees):
        if b == 1:
            continue
        p = gdn.tree_root_path(t, gen.random_leaf(100 + b, t))
        paths[b, :len(p)] = p
        lengths[b] = len(p)
    c, d = _conv_case(shape, N, 95, B=B, tag="roundb")
    x, w, tail = bf16(c["x"]), bf16(c["w"]), bf16(c["tail"])
    al, be, st = f32(d["alpha"]), f32(d["beta"]), f32(d["state"])
    out = torch.full((B, N, shape.Hv, shape.dv), float("nan"), device="cuda")
    gdn.conv_tree_verify_batched(counts, parents, x, w, tail, al, be, st, shape.Hk, shape.Hv, shape.dk, shape.dv,
                                 out=out)
    tail_out = torch.full_like(tail, 0x7FC0)
    gdn.conv_commit_path_batched(counts, parents, paths, lengths, x, w, tail, tail_out, al, be, st, shape.Hk,
                                 shape.Hv, shape.dk, shape.dv)
    torch.cuda.synchronize()
    assert np.array_equal(host(tail), c["tail"]), "tail_in is read only"
    for b, t in enumerate(trees):
        n, L = len(t), int(lengths[b])
        xb = x[b, :n].contiguous()
        alb, beb = al[b, :n].contiguous(), be[b, :n].contiguous()
        st1 = f32(d["state"][b])
        o1 = gdn.conv_tree_verify(t, xb, w, tail[b], alb, beb, st1, shape.Hk, shape.Hv, shape.dk, shape.dv)
        t1 = torch.empty_like(tail[b])
        gdn.conv_commit_path(t, paths[b, :L], xb, w, tail[b], t1, alb, beb, st1, shape.Hk, shape.Hv, shape.dk,
                             shape.dv)
        torch.cuda.synchronize()
        assert torch.equal(out[b, :n], o1), f"sequence {b}: outputs"
        assert torch.isnan(out[b, n:]).all(), f"sequence {b}: rows past the tree"
        assert torch.equal(st[b], st1), f"sequence {b}: state"
        assert torch.equal(tail_out[b], t1), f"sequence {b}: tail"
    assert np.array_equal(host(st[1]), d["state"][1]) and np.array_equal(host(tail_out[1]), c["tail"][1])


def test_tree_verify_batched_at_the_maximum():
    """The joint verify at its limits: 32 sequences, node capacity 64, trees of
    1 to 64 nodes with branching states up to the slot limit; each tree equals
    its single-tree verify bit for bit, and three of them the oracle."""
    shape = gen.QWEN_27B
    B, N = 32, 64
    trees = [gen.random_tree(200 + b, 1 + (b * 37) % 64, 2 + b % 7) for b in range(B)]
    trees[0] = np.arange(-1, 63, dtype=np.int32)  # the longest chain
    counts = np.array([len(t) for t in trees], np.int32)
    parents = _pad_parents(trees, N)
    d = gen.decode_inputs(240, shape.with_batch(B), N, tag="treemax")
    st = f32(d["state"])
    out = torch.full((B, N, shape.Hv, shape.dv), float("nan"), device="cuda")
    gdn.tree_verify_batched(counts, parents, bf16(d["qkv"]), f32(d["alpha"]), f32(d["beta"]), st, shape.Hk,
                            shape.Hv, shape.dk, shape.dv, out=out)
    torch.cuda.synchronize()
    for b, t in enumerate(trees):
        n = len(t)
        single = gdn.tree_verify(t, bf16(d["qkv"][b, :n]), f32(d["alpha"][b, :n]), f32(d["beta"][b, :n]),
                                 f32(d["state"][b]), shape.Hk, shape.Hv, shape.dk, shape.dv)
        torch.cuda.synchronize()
        assert torch.equal(out[b, :n], single), f"tree {b}"
        assert torch.isnan(out[b, n:]).all()
        if b in (0, 13, 31):
            ref = oracle.tree_verify(t, d["qkv"][b, :n], d["alpha"][b, :n], d["beta"][b, :n], d["state"][b],
                                     shape.Hk, shape.Hv, shape.dk, shape.dv)
            assert_out_close(host(out[b, :n]), ref)
