"""Shared helpers for the GPU parity tests: tolerances, device transfer, and
running the oracle on the same generator bytes the kernels see."""
import numpy as np
import torch

import oracle
from hybrid_linear_attention_conv_gb300 import gdn
from hybrid_linear_attention_conv_gb300 import inputs as gen

# Tolerances of the parity bar: outputs within 1e-3 absolute of the fp64
# oracle; the state after the run within 1e-4 relative Frobenius error.
OUT_ATOL = 1e-3
STATE_RTOL_F = 1e-4


def rel_frob(got, want) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def f32(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)


def bf16(a, device="cuda"):
    return gdn.bf16_tensor(a, device)


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return gdn.bf16_bits(t)
    return t.detach().cpu().numpy()


def assert_out_close(got, want, atol=OUT_ATOL):
    err = np.abs(np.asarray(got, np.float64) - want)
    assert np.all(np.isfinite(got)), "non-finite output"
    assert err.max() <= atol, f"max abs error {err.max():.3e} > {atol:g}"
    return float(err.max())


def assert_state_close(got, want, rtol=STATE_RTOL_F):
    r = rel_frob(got, want)
    assert r <= rtol, f"relative Frobenius error {r:.3e} > {rtol:g}"
    return r


def bf16_ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in units of last place between two bf16 arrays (finite values)."""
    def key(h):
        h = h.astype(np.int32)
        return np.where(h & 0x8000, -(h & 0x7FFF), h & 0x7FFF)
    return np.abs(key(a_bits) - key(b_bits))


def oracle_conv_then_round(x, w, tail):
    """Oracle conv in fp64, rounded to bf16 where the kernel stores bf16."""
    y, tail2 = oracle.conv_linear(x, w, tail)
    return oracle.f64_to_bf16(y), tail2


def _key_head_slice(qkv, shape, g):
    """Packed rows of key head g and its value heads, as an Hk = 1 problem."""
    Hk, dk, dv = shape.Hk, shape.dk, shape.dv
    grp = shape.Hv // Hk
    q = qkv[..., g * dk:(g + 1) * dk]
    k = qkv[..., Hk * dk + g * dk: Hk * dk + (g + 1) * dk]
    v = qkv[..., 2 * Hk * dk + g * grp * dv: 2 * Hk * dk + (g + 1) * grp * dv]
    return np.ascontiguousarray(np.concatenate([q, k, v], axis=-1)), slice(g * grp, (g + 1) * grp)


def oracle_decode_parallel(qkv, alpha, beta, state, shape, q_scale=1.0, normalize=True, keys=None):
    """The oracle's sequential decode, run per key head on all host cores.

    qkv [B,T,C] bf16 bits, alpha/beta [B,T,Hv], state [B,Hv,dv,dk].  Key heads
    are independent problems (each value head reads only its own key head), so
    each is the oracle on that head's slice; ctypes releases the GIL during the
    C call, so the slices run on separate cores.  `keys` picks key heads
    (default all); returns (out [B,T,Hv,dv], state [B,Hv,dv,dk]) with only the
    picked heads filled (NaN elsewhere)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    B, T = qkv.shape[0], qkv.shape[1]
    grp = shape.Hv // shape.Hk
    keys = list(range(shape.Hk)) if keys is None else list(keys)
    out = np.full((B, T, shape.Hv, shape.dv), np.nan)
    st = np.full((B, shape.Hv, shape.dv, shape.dk), np.nan)

    def one(g):
        q_g, hs = _key_head_slice(qkv, shape, g)
        o, s_ = oracle.decode(q_g, alpha[..., hs], beta[..., hs], state[:, hs], 1, grp, shape.dk, shape.dv,
                              q_scale=q_scale, normalize=normalize)
        return hs, o, s_

    with ThreadPoolExecutor(max_workers=min(len(keys), os.cpu_count() or 1)) as ex:
        for hs, o, s_ in ex.map(one, keys):
            out[:, :, hs] = o
            st[:, hs] = s_
    return out, st


__all__ = ["OUT_ATOL", "STATE_RTOL_F", "rel_frob", "f32", "bf16", "host", "assert_out_close",
           "assert_state_close", "bf16_ulp_diff", "oracle_conv_then_round", "oracle_decode_parallel", "gen", "gdn",
           "oracle"]
