"""The allocation-free prefill entry point, checked against the regular one.

gdn_chunk_prefill_noalloc serves callers that cannot allocate device memory
when they run a prefill -- for example a serving loop whose device footprint
is fixed at start-up, or a host whose device memory belongs to another
allocator.  It keeps the kernel's scratch in an array inside the library
instead of a caller-provided workspace.  Here two calls in a row (the second
continuing from the first one's state) must agree with gdn_chunk_prefill on
the same inputs, within the tolerances every parity test uses, at the 27B
head shape (the tensor-core chain) and at the tiny shape (narrow heads, run
token by token).  The status word the calls leave in the library's array is
read back with gdn_chunk_prefill_noalloc_status: 0 after good calls, and
GDN_ERR_TIMEOUT when a bounded wait was made to give up.

The file is named so that pytest collects it last: if it fails, a run that
stops at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from gdn_testutil import assert_out_close, assert_state_close, bf16, f32, gdn, gen, host, oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from hybrid_linear_attention_conv_gb300 import build
    build.build()
    return gdn.load()


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _prefill_noalloc(lib, shape, qkv, alpha, beta, state, out):
    """One call of the C entry point (no workspace argument)."""
    sh = gdn.gdn_shape(1, shape.Hk, shape.Hv, shape.dk, shape.dv)
    P = ctypes.c_void_p
    T = qkv.shape[0]
    rc = lib.gdn_chunk_prefill_noalloc(ctypes.byref(sh), T, 64, P(qkv.data_ptr()), P(alpha.data_ptr()),
                                       P(beta.data_ptr()), P(state.data_ptr()), P(out.data_ptr()), 1.0,
                                       gdn.GDN_NORMALIZE_QK, _stream())
    assert rc == 0, gdn.last_error()


def _noalloc_status(lib):
    """(return code, status word) of gdn_chunk_prefill_noalloc_status."""
    word = ctypes.c_int32(-1)
    rc = lib.gdn_chunk_prefill_noalloc_status(_stream(), ctypes.byref(word))
    return rc, word.value


@pytest.mark.parametrize("shape,T", [(gen.QWEN_27B, 300), (gen.TINY, 16)],
                         ids=["27b_tensor_core", "tiny_token_by_token"])
def test_noalloc_prefill_matches_workspace_prefill_on_two_calls(lib, shape, T):
    # 27B: four full chunks and a ragged one per call; tiny: the config's 16 tokens
    d = gen.decode_inputs(17, shape, 2 * T, tag="noalloc")
    qkv, al, be = bf16(d["qkv"][0]), f32(d["alpha"][0]), f32(d["beta"][0])

    st_ref = f32(d["state"][0])
    st_new = f32(d["state"][0])
    for call in range(2):
        sl = slice(call * T, (call + 1) * T)
        q_c, a_c, b_c = qkv[sl].contiguous(), al[sl].contiguous(), be[sl].contiguous()
        out_ref = gdn.chunk_prefill(q_c, a_c, b_c, st_ref, shape.Hk, shape.Hv, shape.dk, shape.dv)
        out_new = torch.empty_like(out_ref)
        _prefill_noalloc(lib, shape, q_c, a_c, b_c, st_new, out_new)
        assert _noalloc_status(lib) == (0, 0)
        torch.cuda.synchronize()
        assert_out_close(host(out_new), host(out_ref).astype("float64"))
        assert_state_close(host(st_new), host(st_ref).astype("float64"))
        if call == 0:
            # and against the oracle itself, over the first call's tokens
            o_or, s_or = oracle.decode(d["qkv"][:, sl], d["alpha"][:, sl], d["beta"][:, sl], d["state"], shape.Hk,
                                       shape.Hv, shape.dk, shape.dv)
            assert_out_close(host(out_new), o_or[0])
            assert_state_close(host(st_new), s_or[0])


def test_noalloc_prefill_timeout_is_readable_and_recovers(lib):
    """A wait limit of 0 makes the chain's bounded tensor-core waits give up at
    their first empty probe: the status word in the library's array is then
    non-zero and gdn_chunk_prefill_noalloc_status returns GDN_ERR_TIMEOUT.  The
    next call, with the default limit back, clears the word and is correct."""
    shape = gen.QWEN_27B
    T = 300
    d = gen.decode_inputs(19, shape, T, tag="noalloc_timeout")
    qkv, al, be = bf16(d["qkv"][0]), f32(d["alpha"][0]), f32(d["beta"][0])
    out = torch.empty((T, shape.Hv, shape.dv), dtype=torch.float32, device="cuda")
    prev = gdn.set_wait_limit_ns(0)
    try:
        _prefill_noalloc(lib, shape, qkv, al, be, f32(d["state"][0]), out)
        rc, word = _noalloc_status(lib)
    finally:
        assert gdn.set_wait_limit_ns(prev) == 0
    assert rc == -8 and word != 0  # GDN_ERR_TIMEOUT
    st = f32(d["state"][0])
    _prefill_noalloc(lib, shape, qkv, al, be, st, out)
    assert _noalloc_status(lib) == (0, 0)
    o_or, s_or = oracle.decode(d["qkv"], d["alpha"], d["beta"], d["state"], shape.Hk, shape.Hv, shape.dk, shape.dv)
    assert_out_close(host(out), o_or[0])
    assert_state_close(host(st), s_or[0])


def test_noalloc_prefill_refuses_bad_arguments(lib):
    shape = gen.QWEN_27B
    d = gen.decode_inputs(18, shape, 64, tag="noalloc_bad")
    st = f32(d["state"][0])
    before = st.clone()
    out = torch.empty((64, shape.Hv, shape.dv), dtype=torch.float32, device="cuda")
    sh = gdn.gdn_shape(1, shape.Hk, shape.Hv, shape.dk, shape.dv)
    P = ctypes.c_void_p
    rc = lib.gdn_chunk_prefill_noalloc(ctypes.byref(sh), 64, 32, P(bf16(d["qkv"][0]).data_ptr()),
                                       P(f32(d["alpha"][0]).data_ptr()), P(f32(d["beta"][0]).data_ptr()),
                                       P(st.data_ptr()), P(out.data_ptr()), 1.0, gdn.GDN_NORMALIZE_QK, None)
    torch.cuda.synchronize()
    assert rc == -1 and "chunk" in gdn.last_error()
    assert torch.equal(st, before)
