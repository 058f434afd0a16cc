"""GPU parity for the KDA variant (a decay per key channel): the decode step
and the fused conv + decode step against the fp64 oracle, through the C ABI."""
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
    assert torch.cuda.is_available()


def _run(shape, T, seed, tag="kdag", **kw):
    d = gen.kda_inputs(seed, shape, T, tag=tag)
    st = f32(d["state"])
    out = gdn.kda_decode_step(bf16(d["qkv"]), f32(d["alpha"]), f32(d["beta"]), st, shape.Hk, shape.Hv,
                              shape.dk, shape.dv, **kw)
    torch.cuda.synchronize()
    out_ref, st_ref = oracle.kda_decode(d["qkv"], d["alpha"], d["beta"], d["state"], shape.Hk, shape.Hv,
                                        shape.dk, shape.dv, q_scale=kw.get("q_scale", 1.0))
    return d, out, st, out_ref, st_ref


@pytest.mark.parametrize("shape,T", [
    (gen.TINY, 16),
    (gen.Shape(3, 2, 4, 64, 64), 5),
    (gen.Shape(2, 1, 3, 128, 128), 9),
    (gen.Shape(2, 2, 4, 32, 64), 4),      # dk != dv
    (gen.Shape(1, 2, 2, 128, 32), 3),
    (gen.QWEN_27B.with_batch(2), 7),
])
def test_kda_decode_vs_oracle(shape, T):
    _, out, st, out_ref, st_ref = _run(shape, T, 40 + T)
    assert_out_close(host(out), out_ref)
    assert_state_close(host(st), st_ref)


def test_kda_decode_batched_27b_full_parity():
    """Batch 64 at the 27B head shape, one token: every output and state."""
    _, out, st, out_ref, st_ref = _run(gen.QWEN_27B.with_batch(64), 1, 41, tag="kdabatch")
    assert_out_close(host(out), out_ref)
    assert_state_close(host(st), st_ref)


def test_kda_decode_strong_and_zero_gates():
    """Gates over the whole of [0, 1), some exactly 0 (that key channel is
    wiped before the write) and some exactly 1."""
    s = gen.Shape(2, 2, 4, 64, 64)
    T = 6
    d = gen.kda_inputs(42, s, T, tag="kdawide")
    a = gen.uniform(42, "kdawide.gate", d["alpha"].size).astype(np.float32).reshape(d["alpha"].shape)
    a[..., ::7] = 0.0
    a[..., 3::11] = 1.0
    st = f32(d["state"])
    out = gdn.kda_decode_step(bf16(d["qkv"]), f32(a), f32(d["beta"]), st, s.Hk, s.Hv, s.dk, s.dv)
    torch.cuda.synchronize()
    out_ref, st_ref = oracle.kda_decode(d["qkv"], a, d["beta"], d["state"], s.Hk, s.Hv, s.dk, s.dv)
    assert_out_close(host(out), out_ref)
    assert_state_close(host(st), st_ref)


def test_kda_decode_options():
    s = gen.Shape(2, 2, 4, 64, 64)
    _, out, st, out_ref, st_ref = _run(s, 3, 43, q_scale=64 ** -0.5)
    assert_out_close(host(out), out_ref)
    assert_state_close(host(st), st_ref)
    _, out, st, out_ref, st_ref = _run(s, 3, 44, out_bf16=True)
    got = gen.bf16_bits_to_f32(host(out)).astype(np.float64)
    assert np.all(np.abs(got - out_ref) <= np.abs(out_ref) * 2.0 ** -8 + 1e-3)


def test_kda_equal_gates_match_scalar_gate_decode():
    """A gate equal on every channel gives the scalar-gated step's results
    (same map, another rounding order: compared within the parity bar)."""
    s = gen.QWEN_27B.with_batch(2)
    d = gen.decode_inputs(45, s, 4, tag="kdaeq")
    a_vec = np.repeat(d["alpha"][..., None], s.dk, axis=-1)
    st_g, st_k = f32(d["state"]), f32(d["state"])
    out_g = gdn.decode_step(bf16(d["qkv"]), f32(d["alpha"]), f32(d["beta"]), st_g, s.Hk, s.Hv, s.dk, s.dv)
    out_k = gdn.kda_decode_step(bf16(d["qkv"]), f32(a_vec), f32(d["beta"]), st_k, s.Hk, s.Hv, s.dk, s.dv)
    torch.cuda.synchronize()
    assert_out_close(host(out_k), host(out_g).astype(np.float64))
    assert_state_close(host(st_k), host(st_g).astype(np.float64))


def test_kda_multi_token_equals_single_steps_bitwise():
    s = gen.QWEN_27B.with_batch(2)
    T = 5
    d = gen.kda_inputs(46, s, T)
    st_a = f32(d["state"])
    out_a = gdn.kda_decode_step(bf16(d["qkv"]), f32(d["alpha"]), f32(d["beta"]), st_a, s.Hk, s.Hv, s.dk, s.dv)
    st_b = f32(d["state"])
    outs = [gdn.kda_decode_step(bf16(d["qkv"][:, t:t + 1]), f32(d["alpha"][:, t:t + 1]),
                                f32(d["beta"][:, t:t + 1]), st_b, s.Hk, s.Hv, s.dk, s.dv) for t in range(T)]
    torch.cuda.synchronize()
    assert torch.equal(st_a, st_b)
    assert torch.equal(out_a, torch.cat(outs, dim=1))


def test_kda_zero_tokens_is_noop():
    s = gen.TINY
    d = gen.kda_inputs(47, s, 1)
    st = f32(d["state"])
    before = st.clone()
    qkv = torch.empty((1, 0, s.C), dtype=torch.bfloat16, device="cuda")
    a = torch.empty((1, 0, s.Hv, s.dk), dtype=torch.float32, device="cuda")
    b = torch.empty((1, 0, s.Hv), dtype=torch.float32, device="cuda")
    gdn.kda_decode_step(qkv, a, b, st, s.Hk, s.Hv, s.dk, s.dv)
    torch.cuda.synchronize()
    assert torch.equal(st, before)


# ---------------------------------------------------------------------------
# fused conv + KDA decode
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("shape,T,pingpong", [
    (gen.QWEN_27B.with_batch(64), 1, False),    # the batched decode shape
    (gen.QWEN_27B.with_batch(1), 1, True),      # rows split over CTAs
    (gen.QWEN_27B.with_batch(2), 3, True),
    (gen.TINY, 16, False),
    (gen.Shape(3, 2, 4, 32, 64), 2, True),
])
def test_kda_conv_decode_fused_equals_unfused(shape, T, pingpong):
    c = gen.conv_inputs(51 + T, shape.B, T, shape.C)
    d = gen.kda_inputs(51 + T, shape, T, tag="kdafused")
    w = bf16(c["w"])
    tail_a = bf16(c["tail"])
    y = gdn.conv_step(bf16(c["x"]), w, tail_a)
    st_a = f32(d["state"])
    out_a = gdn.kda_decode_step(y, f32(d["alpha"]), f32(d["beta"]), st_a, shape.Hk, shape.Hv, shape.dk, shape.dv)
    tail_in = bf16(c["tail"])
    tail_out = torch.zeros_like(tail_in) if pingpong else None
    st_b = f32(d["state"])
    out_b = gdn.kda_conv_decode_step(bf16(c["x"]), w, tail_in, f32(d["alpha"]), f32(d["beta"]), st_b,
                                     shape.Hk, shape.Hv, shape.dk, shape.dv, tail_out=tail_out)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    assert torch.equal(st_a, st_b)
    assert torch.equal(tail_a, tail_out if pingpong else tail_in)


def test_kda_conv_decode_fused_vs_oracle_27b():
    shape = gen.QWEN_27B.with_batch(3)
    T = 2
    c = gen.conv_inputs(55, shape.B, T, shape.C)
    d = gen.kda_inputs(55, shape, T, tag="kdafo")
    tail = bf16(c["tail"])
    st = f32(d["state"])
    out = gdn.kda_conv_decode_step(bf16(c["x"]), bf16(c["w"]), tail, f32(d["alpha"]), f32(d["beta"]), st,
                                   shape.Hk, shape.Hv, shape.dk, shape.dv)
    torch.cuda.synchronize()
    y_ref, tail_ref = oracle_conv_then_round(c["x"], c["w"], c["tail"])
    out_ref, st_ref = oracle.kda_decode(y_ref, d["alpha"], d["beta"], d["state"], shape.Hk, shape.Hv, shape.dk,
                                        shape.dv)
    assert np.array_equal(host(tail), tail_ref)
    assert_out_close(host(out), out_ref)
    assert_state_close(host(st), st_ref)


# ---------------------------------------------------------------------------
# the speculative round with the KDA step: tree verify and commit
# ---------------------------------------------------------------------------
def _kda_tree_case(shape, N, seed, tag="kdatree"):
    d = gen.kda_inputs(seed, shape.with_batch(1), N, tag=tag)
    return {"qkv": d["qkv"][0], "alpha": d["alpha"][0], "beta": d["beta"][0], "state": d["state"][0]}


def _kda_path_decode(shape, d, path):
    st = f32(d["state"][None])
    out = gdn.kda_decode_step(bf16(d["qkv"][None, path]), f32(d["alpha"][None, path]), f32(d["beta"][None, path]),
                              st, shape.Hk, shape.Hv, shape.dk, shape.dv)
    torch.cuda.synchronize()
    return out[0], st[0]


@pytest.mark.parametrize("shape,parents", [
    (gen.QWEN_27B, gen.random_tree(150, 32, 8)),
    (gen.TINY, gen.random_tree(151, 20, 6)),
    (gen.Shape(1, 2, 4, 64, 64), np.array([-1] + [0] * 15, np.int32)),      # a star
    (gen.Shape(1, 2, 4, 64, 64), np.arange(-1, 40, dtype=np.int32)),        # a 41-long chain
])
def test_kda_tree_verify_equals_kda_decode_of_root_paths(shape, parents):
    """Every node's output is the bits of the KDA decode of its root path; the
    committed state is untouched; and the outputs agree with the oracle's KDA
    decode of the root paths (a sample of nodes at the 27B shape)."""
    N = len(parents)
    d = _kda_tree_case(shape, N, 152)
    st = f32(d["state"])
    out = gdn.kda_tree_verify(parents, bf16(d["qkv"]), f32(d["alpha"]), f32(d["beta"]), st, shape.Hk, shape.Hv,
                              shape.dk, shape.dv)
    torch.cuda.synchronize()
    assert np.array_equal(host(st), d["state"]), "verify must not write the committed state"
    nodes = range(N) if shape is not gen.QWEN_27B else [0, 1, 7, 15, N - 1]
    for n in range(N):
        path = gdn.tree_root_path(parents, n)
        o, _ = _kda_path_decode(shape, d, path)
        assert torch.equal(out[n], o[-1]), f"node {n}"
        if n in nodes:
            o_ref, _ = oracle.kda_decode(d["qkv"][None, path], d["alpha"][None, path], d["beta"][None, path],
                                         d["state"][None], shape.Hk, shape.Hv, shape.dk, shape.dv)
            assert_out_close(host(out[n]), o_ref[0, -1])


@pytest.mark.parametrize("shape", [gen.QWEN_27B, gen.TINY])
def test_kda_commit_equals_kda_decode_every_prefix(shape):
    """The KDA commit of every prefix of a root-to-leaf path: the bits of the
    KDA decode of the gathered path, the tail the last four inputs, and the
    state within the oracle's bar."""
    N = 32
    parents = gen.random_tree(153, N, 8)
    path = gdn.tree_root_path(parents, gen.random_leaf(153, parents))
    d = _kda_tree_case(shape, N, 154)
    c = gen.conv_inputs(155, 1, N, shape.C, tag="kdacommit")
    for L in range(len(path) + 1):
        st = f32(d["state"])
        tail = bf16(c["tail"][0])
        gdn.kda_commit_path(parents, path[:L], bf16(d["qkv"]), f32(d["alpha"]), f32(d["beta"]), st, shape.Hk,
                            shape.Hv, shape.dk, shape.dv, x_tree=bf16(c["x"][0]), tail=tail)
        torch.cuda.synchronize()
        hist = np.concatenate([c["tail"][0], c["x"][0][path[:L]]], axis=0)
        assert np.array_equal(host(tail), hist[-4:]), f"L={L}: tail"
        if L == 0:
            assert np.array_equal(host(st), d["state"])
            continue
        _, st_dec = _kda_path_decode(shape, d, path[:L])
        assert torch.equal(st, st_dec), f"L={L}: state"
    _, st_ref = oracle.kda_decode(d["qkv"][None, path], d["alpha"][None, path], d["beta"][None, path],
                                  d["state"][None], shape.Hk, shape.Hv, shape.dk, shape.dv)
    assert_state_close(host(st), st_ref[0])


def test_kda_tree_verify_batched_equals_single():
    """The joint KDA verify (trees of 32, 1, 13 and 20 nodes; capacity 32):
    each tree equals gdn_kda_tree_verify of that tree alone, bit for bit; rows
    past a tree's size are not written; the states are untouched."""
    shape = gen.QWEN_27B
    N = 32
    trees = [gen.random_tree(160, 32, 8), np.array([-1], np.int32), gen.random_tree(161, 13, 5),
             gen.random_tree(162, 20, 8)]
    B = len(trees)
    counts = np.array([len(t) for t in trees], np.int32)
    parents = np.full((B, N), -7, np.int32)
    for b, t in enumerate(trees):
        parents[b, :len(t)] = t
    d = gen.kda_inputs(163, shape.with_batch(B), N, tag="kdajoint")
    st = f32(d["state"])
    out = torch.full((B, N, shape.Hv, shape.dv), float("nan"), device="cuda")
    gdn.kda_tree_verify_batched(counts, parents, bf16(d["qkv"]), f32(d["alpha"]), f32(d["beta"]), st, shape.Hk,
                                shape.Hv, shape.dk, shape.dv, out=out)
    torch.cuda.synchronize()
    assert np.array_equal(host(st), d["state"])
    for b, t in enumerate(trees):
        n = len(t)
        single = gdn.kda_tree_verify(t, bf16(d["qkv"][b, :n]), f32(d["alpha"][b, :n]), f32(d["beta"][b, :n]),
                                     f32(d["state"][b]), shape.Hk, shape.Hv, shape.dk, shape.dv)
        torch.cuda.synchronize()
        assert torch.equal(out[b, :n], single), f"tree {b}"
        assert torch.isnan(out[b, n:]).all()
