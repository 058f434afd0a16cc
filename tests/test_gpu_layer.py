"""GPU parity for the layer's decode step around the mixer: gates from the
projections, conv + L2-norm + delta step, gated RMS-norm output -- against
the fp64 oracle, and bit for bit against the separate gates and fused-step
calls it stands for."""
import numpy as np
import pytest
import torch

from gdn_testutil import assert_out_close, assert_state_close, bf16, f32, gdn, gen, host, oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from hybrid_linear_attention_conv_gb300 import build
    build.build()
    gdn.load()
    assert torch.cuda.is_available()


def _run(shape, T, seed, pingpong=False, eps=1e-6):
    d = gen.layer_inputs(seed, shape, T)
    tail_in = bf16(d["tail"])
    tail_out = torch.zeros_like(tail_in) if pingpong else None
    st = f32(d["state"])
    o = torch.empty((shape.B, T, shape.Hv, shape.dv), dtype=torch.float32, device="cuda")
    y = gdn.layer_decode_step(bf16(d["x"]), bf16(d["w"]), tail_in, bf16(d["a"]), bf16(d["b"]), f32(d["A_log"]),
                              f32(d["dt_bias"]), bf16(d["z"]), f32(d["norm_w"]), st, shape.Hk, shape.Hv, shape.dk,
                              shape.dv, tail_out=tail_out, o=o, norm_eps=eps)
    torch.cuda.synchronize()
    ref = oracle.layer_decode(d["x"], d["w"], d["tail"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["z"],
                              d["norm_w"], d["state"], shape.Hk, shape.Hv, shape.dk, shape.dv, eps=eps)
    return d, y, o, st, tail_out if pingpong else tail_in, ref


def _assert_y_close(y, y_ref, o, o_ref, d, eps=1e-6):
    """y = o / rms(o) * g with g = w * SiLU(z).  Two checks:
    (1) the epilogue alone: y against the fp64 gated norm of the kernel's own o,
        within one bf16 rounding (half an ulp <= 2^-8 |y|) plus fp32 slack;
    (2) end to end against the oracle: o's error e_o (per head, measured, and
        itself within the 1e-3 bar) propagates through 1/rms, so
        |dy_i| <= 2^-8 |y_i| + |g_i| e_o / rms (1 + |o_i| / rms).
    Heads whose output is nearly zero (strongly decaying gates) have a small
    rms and a correspondingly larger, but still exact-arithmetic-bounded, y error."""
    got = gen.bf16_bits_to_f32(host(y)).astype(np.float64)
    assert np.all(np.isfinite(got))
    o_gpu = host(o).astype(np.float64)
    zf = gen.bf16_bits_to_f32(d["z"]).astype(np.float64)
    g = d["norm_w"].astype(np.float64) * zf / (1.0 + np.exp(-zf))
    y_own = o_gpu / np.sqrt((o_gpu ** 2).mean(-1, keepdims=True) + eps) * g
    assert np.all(np.abs(got - y_own) <= np.abs(y_own) * 2.0 ** -8 + 1e-5 * np.abs(g) + 1e-6)
    rms = np.sqrt((o_ref ** 2).mean(-1, keepdims=True) + eps)
    e_o = np.abs(o_gpu - o_ref).max(-1, keepdims=True)
    bound = np.abs(y_ref) * 2.0 ** -8 + 1.01 * np.abs(g) * e_o / rms * (1.0 + np.abs(o_ref) / rms) + 1e-6
    assert np.all(np.abs(got - y_ref) <= bound), float((np.abs(got - y_ref) - bound).max())


@pytest.mark.parametrize("shape,T,pingpong", [
    (gen.TINY, 16, False),
    (gen.QWEN_27B.with_batch(4), 1, False),
    (gen.QWEN_27B.with_batch(2), 3, True),
    (gen.Shape(3, 2, 4, 32, 64), 2, False),     # dk != dv
    (gen.Shape(2, 1, 3, 64, 128), 5, True),
])
def test_layer_step_vs_oracle(shape, T, pingpong):
    d, y, o, st, tail, (o_ref, y_ref, st_ref, tail_ref) = _run(shape, T, 70 + T, pingpong)
    assert np.array_equal(host(tail), tail_ref)
    assert_out_close(host(o), o_ref)
    assert_state_close(host(st), st_ref)
    _assert_y_close(y, y_ref, o, o_ref, d)


def test_layer_step_batched_27b_full_parity():
    """Batch 64 at the 27B shape, one token: every y, o and state vs the oracle."""
    d, y, o, st, tail, (o_ref, y_ref, st_ref, tail_ref) = _run(gen.QWEN_27B.with_batch(64), 1, 77)
    assert np.array_equal(host(tail), tail_ref)
    assert_out_close(host(o), o_ref)
    assert_state_close(host(st), st_ref)
    _assert_y_close(y, y_ref, o, o_ref, d)


def test_gates_kernel_vs_oracle():
    s = gen.QWEN_27B.with_batch(8)
    d = gen.layer_inputs(78, s, 5)
    al, be = gdn.gates(bf16(d["a"]), bf16(d["b"]), f32(d["A_log"]), f32(d["dt_bias"]))
    torch.cuda.synchronize()
    al_ref, be_ref = oracle.gates_from_projections(d["a"], d["b"], d["A_log"], d["dt_bias"])
    np.testing.assert_allclose(host(al), al_ref, rtol=2e-6, atol=0)
    np.testing.assert_allclose(host(be), be_ref, rtol=2e-6, atol=0)


@pytest.mark.parametrize("shape,T", [(gen.QWEN_27B.with_batch(64), 1), (gen.QWEN_27B.with_batch(2), 4),
                                     (gen.TINY, 7)])
def test_layer_step_o_equals_gates_then_fused_step(shape, T):
    """o of the layer step == gdn_gates, then gdn_conv_decode_step on those
    gates, bit for bit (the same gate function, the same fused step)."""
    d = gen.layer_inputs(79 + T, shape, T)
    a, b_ = bf16(d["a"]), bf16(d["b"])
    al, be = gdn.gates(a, b_, f32(d["A_log"]), f32(d["dt_bias"]))
    tail_a = bf16(d["tail"])
    st_a = f32(d["state"])
    o_a = gdn.conv_decode_step(bf16(d["x"]), bf16(d["w"]), tail_a, al, be, st_a, shape.Hk, shape.Hv, shape.dk,
                               shape.dv)
    tail_b = bf16(d["tail"])
    st_b = f32(d["state"])
    o_b = torch.empty_like(o_a)
    gdn.layer_decode_step(bf16(d["x"]), bf16(d["w"]), tail_b, a, b_, f32(d["A_log"]), f32(d["dt_bias"]),
                          bf16(d["z"]), f32(d["norm_w"]), st_b, shape.Hk, shape.Hv, shape.dk, shape.dv, o=o_b)
    torch.cuda.synchronize()
    assert torch.equal(o_a, o_b)
    assert torch.equal(st_a, st_b)
    assert torch.equal(tail_a, tail_b)


def test_layer_step_zero_gate_projection_and_no_o():
    """z = 0 gives y = 0 exactly (SiLU(0) = 0); o may be omitted."""
    s = gen.Shape(2, 2, 4, 64, 64)
    d = gen.layer_inputs(80, s, 2)
    st = f32(d["state"])
    y = gdn.layer_decode_step(bf16(d["x"]), bf16(d["w"]), bf16(d["tail"]), bf16(d["a"]), bf16(d["b"]),
                              f32(d["A_log"]), f32(d["dt_bias"]), torch.zeros((s.B, 2, s.Hv, s.dv),
                                                                              dtype=torch.bfloat16, device="cuda"),
                              f32(d["norm_w"]), st, s.Hk, s.Hv, s.dk, s.dv)
    torch.cuda.synchronize()
    assert not y.float().abs().sum().item()
