"""GPU parity for chunked prefill against the sequential fp64 oracle.

The chunk form rounds differently from the sequential recurrence (the same
mathematics accumulated in another order), so parity is the stated tolerance,
not bits.  At the full 8,192-token size the oracle runs per key head on all
host cores (the key heads are independent problems), and every output and the
whole final state are compared."""
import numpy as np
import pytest
import torch

from gdn_testutil import (assert_out_close, assert_state_close, bf16, f32, gdn, gen, host, oracle,
                          oracle_decode_parallel)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from hybrid_linear_attention_conv_gb300 import build
    build.build()
    gdn.load()


def _slice_key_head(qkv, shape, g):
    """Packed rows of one key head g and its value heads, as a (Hk=1) problem."""
    Hk, dk, dv = shape.Hk, shape.dk, shape.dv
    grp = shape.Hv // Hk
    q = qkv[..., g * dk:(g + 1) * dk]
    k = qkv[..., Hk * dk + g * dk: Hk * dk + (g + 1) * dk]
    v = qkv[..., 2 * Hk * dk + g * grp * dv: 2 * Hk * dk + (g + 1) * grp * dv]
    return np.ascontiguousarray(np.concatenate([q, k, v], axis=-1)), slice(g * grp, (g + 1) * grp)


def _run(shape, T, seed, heads=None, **kw):
    d = gen.decode_inputs(seed, shape.with_batch(1), T, tag="prefill")
    st = f32(d["state"][0])
    ws = torch.full((gdn.prefill_workspace_bytes(T, shape.Hk, shape.Hv, shape.dk, shape.dv),), 7,
                    dtype=torch.uint8, device="cuda")
    out = gdn.chunk_prefill(bf16(d["qkv"][0]), f32(d["alpha"][0]), f32(d["beta"][0]), st, shape.Hk,
                            shape.Hv, shape.dk, shape.dv, workspace=ws, **kw)
    torch.cuda.synchronize()
    if T > 0:
        assert int(ws[:4].view(torch.int32).item()) == 0, "a bounded tensor-core wait gave up"
    out_h, st_h = host(out), host(st)
    if heads is None:
        out_ref, st_ref = oracle.prefill(d["qkv"], d["alpha"], d["beta"], d["state"], shape.Hk, shape.Hv,
                                         shape.dk, shape.dv, q_scale=kw.get("q_scale", 1.0))
        return out_h, st_h, out_ref[0], st_ref[0]
    grp = shape.Hv // shape.Hk
    outs, sts, refs_o, refs_s = [], [], [], []
    for g in heads:
        qkv_g, hs = _slice_key_head(d["qkv"], shape, g)
        o_ref, s_ref = oracle.prefill(qkv_g, d["alpha"][..., hs], d["beta"][..., hs], d["state"][:, hs],
                                      1, grp, shape.dk, shape.dv, q_scale=kw.get("q_scale", 1.0))
        outs.append(out_h[:, hs])
        sts.append(st_h[hs])
        refs_o.append(o_ref[0])
        refs_s.append(s_ref[0])
    return (np.concatenate(outs, 1), np.concatenate(sts, 0), np.concatenate(refs_o, 1),
            np.concatenate(refs_s, 0))


@pytest.mark.parametrize("shape,T", [(gen.TINY, 64), (gen.TINY, 300), (gen.QWEN_27B, 129),
                                     (gen.Shape(1, 2, 4, 64, 64), 1), (gen.Shape(1, 1, 2, 128, 128), 511),
                                     (gen.Shape(1, 1, 3, 128, 128), 1), (gen.Shape(1, 1, 3, 128, 128), 64),
                                     (gen.Shape(1, 2, 2, 128, 128), 65), (gen.QWEN_27B, 1000)])
def test_prefill_small_vs_oracle(shape, T):
    out, st, out_ref, st_ref = _run(shape, T, 40 + T)
    assert_out_close(out, out_ref)
    assert_state_close(st, st_ref)


def test_prefill_27b_8192_all_heads():
    """1 sequence, 8,192 tokens, 27B head shape, chunk 64: every output of
    all 48 value heads and the whole final state against the sequential oracle."""
    shape = gen.QWEN_27B
    T = 8192
    d = gen.decode_inputs(0, shape.with_batch(1), T, tag="prefill")
    st = f32(d["state"][0])
    out = gdn.chunk_prefill(bf16(d["qkv"][0]), f32(d["alpha"][0]), f32(d["beta"][0]), st, shape.Hk, shape.Hv,
                            shape.dk, shape.dv)
    torch.cuda.synchronize()
    out_ref, st_ref = oracle_decode_parallel(d["qkv"], d["alpha"], d["beta"], d["state"], shape)
    assert_out_close(host(out), out_ref[0])
    assert_state_close(host(st), st_ref[0])


# ---------------------------------------------------------------------------
# gates at their extremes on the tensor-core path
# ---------------------------------------------------------------------------
def _edge_gates(kind, T, Hv, seed):
    """(alpha, beta) fp32 [1, T, Hv] for the strong- and edge-gate cases:
    'layer'  the layer's own gates from its projections (the published Gated
             DeltaNet initialisation), computed by the oracle: some heads decay
             hard (alpha far below 0.9);
    'edges'  alpha and beta at exactly 0 and 1, mixed with ordinary values
             inside the same chunks;
    'front'  every chunk's first 8 tokens decay hard (alpha ~ U(0.01, 0.2)),
             the rest keep alpha within 1e-4 of 1."""
    alpha, beta = gen.gates(seed, "edge." + kind, (1, T, Hv))
    u = gen.uniform(seed, "edge.pick." + kind, T * Hv).reshape(1, T, Hv)
    if kind == "layer":
        L = gen.layer_inputs(seed, gen.Shape(1, 1, Hv, 32, 32), T, tag="edge.layer")
        alpha, beta = oracle.gates_from_projections(L["a"], L["b"], L["A_log"], L["dt_bias"])
        alpha, beta = alpha.astype(np.float32), beta.astype(np.float32)
    elif kind == "edges":
        alpha = np.where(u < 0.1, 0.0, np.where(u < 0.3, 1.0, alpha)).astype(np.float32)
        v = gen.uniform(seed, "edge.pick2", T * Hv).reshape(1, T, Hv)
        beta = np.where(v < 0.15, 0.0, np.where(v < 0.35, 1.0, beta)).astype(np.float32)
    else:
        t = np.arange(T).reshape(1, T, 1) % 64
        hard = (0.01 + 0.19 * u).astype(np.float32)
        soft = (1.0 - 1e-4 * u).astype(np.float32)
        alpha = np.where(t < 8, hard, soft).astype(np.float32)
    return alpha, beta


@pytest.mark.parametrize("kind", ["layer", "edges", "front"])
@pytest.mark.parametrize("form", ["cooperative", "two_launch", "noalloc"])
def test_prefill_edge_gates_vs_oracle(kind, form):
    shape = gen.QWEN_27B
    T = 700  # ten full chunks and a ragged one
    d = gen.decode_inputs(300, shape.with_batch(1), T, tag="edgegates")
    d["alpha"], d["beta"] = _edge_gates(kind, T, shape.Hv, 301)
    if kind == "layer":
        assert d["alpha"].min() < 0.14 and d["alpha"].max() > 0.99
    st = f32(d["state"][0])
    args = (bf16(d["qkv"][0]), f32(d["alpha"][0]), f32(d["beta"][0]), st, shape.Hk, shape.Hv, shape.dk, shape.dv)
    if form == "noalloc":
        out = gdn.chunk_prefill_noalloc(*args)
        assert gdn.chunk_prefill_noalloc_status() == 0
    else:
        ws = torch.empty(gdn.prefill_workspace_bytes(T, shape.Hk, shape.Hv, shape.dk, shape.dv), dtype=torch.uint8,
                         device="cuda")
        out = gdn.chunk_prefill(*args, workspace=ws, two_launch=form == "two_launch")
        assert gdn.prefill_status(ws) == 0
    torch.cuda.synchronize()
    out_ref, st_ref = oracle_decode_parallel(d["qkv"], d["alpha"], d["beta"], d["state"], shape)
    assert_out_close(host(out), out_ref[0])
    assert_state_close(host(st), st_ref[0])


def test_prefill_options_27b():
    """q scale and bf16 outputs on the tensor-core path."""
    shape = gen.Shape(1, 2, 6, 128, 128)
    out, st, out_ref, st_ref = _run(shape, 200, 3, q_scale=0.25)
    assert_out_close(out, out_ref)
    assert_state_close(st, st_ref)
    out, st, out_ref, st_ref = _run(shape, 150, 4, out_bf16=True)
    got = gen.bf16_bits_to_f32(out).astype(np.float64)
    assert np.all(np.abs(got - out_ref) <= np.abs(out_ref) * 2.0 ** -8 + 1e-3)
    assert_state_close(st, st_ref)


def test_prefill_zero_tokens_keeps_state():
    shape = gen.TINY
    d = gen.decode_inputs(1, shape, 1)
    st = f32(d["state"][0])
    before = st.clone()
    qkv = torch.empty((0, shape.C), dtype=torch.bfloat16, device="cuda")
    e = torch.empty((0, shape.Hv), dtype=torch.float32, device="cuda")
    gdn.chunk_prefill(qkv, e, e, st, shape.Hk, shape.Hv, shape.dk, shape.dv)
    torch.cuda.synchronize()
    assert torch.equal(st, before)


def test_prefill_then_decode_continues():
    """Prefill leaves a state that decode continues from (prompt then one token)."""
    shape = gen.QWEN_27B
    T = 200
    d = gen.decode_inputs(9, shape, T + 1, tag="pd")
    st = f32(d["state"][0])
    gdn.chunk_prefill(bf16(d["qkv"][0, :T]), f32(d["alpha"][0, :T]), f32(d["beta"][0, :T]), st, shape.Hk,
                      shape.Hv, shape.dk, shape.dv)
    st_b = st[None].contiguous()
    out = gdn.decode_step(bf16(d["qkv"][:, T:]), f32(d["alpha"][:, T:]), f32(d["beta"][:, T:]), st_b,
                          shape.Hk, shape.Hv, shape.dk, shape.dv)
    torch.cuda.synchronize()
    out_ref, st_ref = oracle.decode(d["qkv"], d["alpha"], d["beta"], d["state"], shape.Hk, shape.Hv,
                                    shape.dk, shape.dv)
    assert_out_close(host(out)[0, 0], out_ref[0, T])
    assert_state_close(host(st_b)[0], st_ref[0])


@pytest.mark.parametrize("T", [64, 300, 1000])
def test_prefill_prepass_and_self_contained_agree(T):
    """The pre-pass path (T, the state-update factor T^T diag(c) K and the
    output factor P T computed for all chunks in parallel, then read by the
    chain) and the self-contained chain (which forms U = T X between its
    MMAs) group the same algebra differently, so they round differently:
    each must meet the oracle bars, and they must agree with each other."""
    import ctypes
    shape = gen.QWEN_27B
    d = gen.decode_inputs(90 + T, shape.with_batch(1), T, tag="prepass")
    qkv, al, be = bf16(d["qkv"][0]), f32(d["alpha"][0]), f32(d["beta"][0])
    st_a = f32(d["state"][0])
    out_a = gdn.chunk_prefill(qkv, al, be, st_a, shape.Hk, shape.Hv, shape.dk, shape.dv)
    st_b = f32(d["state"][0])
    out_b = torch.empty_like(out_a)
    P = ctypes.c_void_p
    sh = gdn.gdn_shape(1, shape.Hk, shape.Hv, shape.dk, shape.dv)
    rc = gdn.load().gdn_chunk_prefill_noalloc(ctypes.byref(sh), T, 64, P(qkv.data_ptr()), P(al.data_ptr()),
                                              P(be.data_ptr()), P(st_b.data_ptr()), P(out_b.data_ptr()), 1.0,
                                              gdn.GDN_NORMALIZE_QK, P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, gdn.last_error()
    torch.cuda.synchronize()
    out_ref, st_ref = oracle.prefill(d["qkv"], d["alpha"], d["beta"], d["state"], shape.Hk, shape.Hv,
                                     shape.dk, shape.dv)
    for out, st in ((out_a, st_a), (out_b, st_b)):
        assert_out_close(host(out), out_ref[0])
        assert_state_close(host(st), st_ref[0])
    assert_out_close(host(out_a), host(out_b).astype(np.float64))
    assert_state_close(host(st_a), host(st_b).astype(np.float64))


@pytest.mark.parametrize("T", [300, 1000])
def test_prefill_cooperative_equals_two_launch_bitwise(T):
    """One cooperative launch (pre-pass workers beside the chains) and the
    pre-pass over all chunks followed by the chain run the same code on the
    same records: the same bits."""
    shape = gen.QWEN_27B
    d = gen.decode_inputs(110 + T, shape.with_batch(1), T, tag="forms")
    qkv, al, be = bf16(d["qkv"][0]), f32(d["alpha"][0]), f32(d["beta"][0])
    st_a, st_b = f32(d["state"][0]), f32(d["state"][0])
    out_a = gdn.chunk_prefill(qkv, al, be, st_a, shape.Hk, shape.Hv, shape.dk, shape.dv)
    out_b = gdn.chunk_prefill(qkv, al, be, st_b, shape.Hk, shape.Hv, shape.dk, shape.dv, two_launch=True)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    assert torch.equal(st_a, st_b)



# ---------------------------------------------------------------------------
# the bounded waits: a wait that gives up is reported, and the next call is clean
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("two_launch", [False, True])
def test_prefill_wait_timeout_is_reported_and_recovers(two_launch):
    """With the wait limit at 0, a wait gives up at the first empty probe (the
    chains wait for pre-pass records, copies and MMAs that cannot be done yet):
    the kernels return, the status word is non-zero and gdn_prefill_status
    returns GDN_ERR_TIMEOUT.  With the default limit back, the same workspace
    serves a clean call whose results meet the oracle bars."""
    import ctypes
    shape = gen.QWEN_27B
    T = 1000
    d = gen.decode_inputs(320, shape.with_batch(1), T, tag="timeout")
    qkv, al, be = bf16(d["qkv"][0]), f32(d["alpha"][0]), f32(d["beta"][0])
    ws = torch.empty(gdn.prefill_workspace_bytes(T, shape.Hk, shape.Hv, shape.dk, shape.dv), dtype=torch.uint8,
                     device="cuda")
    prev = gdn.set_wait_limit_ns(0)
    try:
        gdn.chunk_prefill(qkv, al, be, f32(d["state"][0]), shape.Hk, shape.Hv, shape.dk, shape.dv, workspace=ws,
                          two_launch=two_launch)
        status = gdn.prefill_status(ws)
    finally:
        assert gdn.set_wait_limit_ns(prev) == 0
    assert status != 0
    word = ctypes.c_int32(0)
    rc = gdn.load().gdn_prefill_status(ctypes.c_void_p(ws.data_ptr()),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(word))
    assert rc == -8 and word.value == status  # GDN_ERR_TIMEOUT
    st = f32(d["state"][0])
    out = gdn.chunk_prefill(qkv, al, be, st, shape.Hk, shape.Hv, shape.dk, shape.dv, workspace=ws,
                            two_launch=two_launch)
    assert gdn.prefill_status(ws) == 0
    out_ref, st_ref = oracle_decode_parallel(d["qkv"], d["alpha"], d["beta"], d["state"], shape)
    assert_out_close(host(out), out_ref[0])
    assert_state_close(host(st), st_ref[0])


def test_prefill_long_prompt_split_calls_and_sampled_heads():
    """32,768 tokens (four times the config's prompt) at the 27B shape, in one
    call and as four calls of 8,192 with the state carried (chunk boundaries
    unchanged, so the same bits); key heads 0 and 15 -- all their value heads,
    every output and the final state -- against the oracle (key heads are
    independent problems, run on two host cores)."""
    shape = gen.QWEN_27B
    T, P = 32768, 8192
    d = gen.decode_inputs(32, shape.with_batch(1), T, tag="prefill-long")
    qkv, al, be = bf16(d["qkv"][0]), f32(d["alpha"][0]), f32(d["beta"][0])
    st = f32(d["state"][0])
    out = gdn.chunk_prefill(qkv, al, be, st, shape.Hk, shape.Hv, shape.dk, shape.dv)
    st2 = f32(d["state"][0])
    outs = [gdn.chunk_prefill(qkv[i:i + P], al[i:i + P], be[i:i + P], st2, shape.Hk, shape.Hv, shape.dk,
                              shape.dv) for i in range(0, T, P)]
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(outs, 0), out) and torch.equal(st2, st)
    keys = [0, shape.Hk - 1]
    out_ref, st_ref = oracle_decode_parallel(d["qkv"], d["alpha"], d["beta"], d["state"], shape, keys=keys)
    grp = shape.Hv // shape.Hk
    heads = np.concatenate([np.arange(g * grp, (g + 1) * grp) for g in keys])
    assert_out_close(host(out)[:, heads], out_ref[0][:, heads])
    assert_state_close(host(st)[heads], st_ref[0][heads])
