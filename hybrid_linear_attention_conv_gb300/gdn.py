"""Thin Python binding over ``libgdn.so`` (the C ABI in ``include/gdn.h``).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, and their ``data_ptr()`` plus the current CUDA stream are passed to
the C entry point of the same name.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU fallback, and a missing library is an
error.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_CONV_W = 4
GDN_MAX_TREE_NODES = 64
GDN_MAX_TREE_SLOTS = 8
GDN_NORMALIZE_QK = 0x1
GDN_OUT_BF16 = 0x2
GDN_PREFILL_TWO_LAUNCH = 0x4
GDN_IN_F32 = 0x8

STATUS = {
    0: "GDN_OK",
    -1: "GDN_ERR_INVALID_ARG",
    -2: "GDN_ERR_UNSUPPORTED_SHAPE",
    -3: "GDN_ERR_BAD_PARENTS",
    -4: "GDN_ERR_BAD_PATH",
    -5: "GDN_ERR_DEPTH_EXCEEDED",
    -6: "GDN_ERR_MISALIGNED",
    -7: "GDN_ERR_CUDA",
    -8: "GDN_ERR_TIMEOUT",
    -9: "GDN_ERR_WORKSPACE",
}

# Every symbol include/gdn.h declares.
EXPORTS = [
    "gdn_abi_version",
    "gdn_last_error",
    "gdn_state_bytes",
    "gdn_tree_root_path",
    "gdn_conv_step",
    "gdn_decode_step",
    "gdn_conv_decode_step",
    "gdn_kda_decode_step",
    "gdn_kda_conv_decode_step",
    "gdn_layer_decode_step",
    "gdn_gates",
    "gdn_tree_verify",
    "gdn_tree_verify_batched",
    "gdn_commit_path",
    "gdn_commit_path_batched",
    "gdn_kda_tree_verify",
    "gdn_kda_tree_verify_batched",
    "gdn_kda_commit_path",
    "gdn_conv_tree_verify",
    "gdn_conv_tree_verify_batched",
    "gdn_conv_commit_path",
    "gdn_conv_commit_path_batched",
    "gdn_prefill_workspace_bytes",
    "gdn_chunk_prefill",
    "gdn_prefill_status",
    "gdn_set_wait_limit_ns",
    "gdn_chunk_prefill_noalloc",
    "gdn_chunk_prefill_noalloc_status",
    "gdn_snapshot_bytes",
    "gdn_snapshot_signature",
    "gdn_snapshot_save",
    "gdn_snapshot_restore",
]


class GdnError(RuntimeError):
    def __init__(self, code: int, fn: str, msg: str):
        super().__init__(f"{fn} -> {STATUS.get(code, code)}: {msg}")
        self.code = code


class gdn_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hk", ctypes.c_int32), ("Hv", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load the shared library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                               "(the CUDA library is required; there is no fallback)")
        lib = ctypes.CDLL(path)
        P, I32, U32, F, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_float,
                              ctypes.c_size_t)
        I64 = ctypes.c_int64
        SH = ctypes.POINTER(gdn_shape)
        sig = {
            "gdn_abi_version": (ctypes.c_int, []),
            "gdn_last_error": (ctypes.c_char_p, []),
            "gdn_state_bytes": (SZ, [SH]),
            "gdn_tree_root_path": (ctypes.c_int, [I32, P, I32, P, I32]),
            "gdn_conv_step": (ctypes.c_int, [I32, I32, I32, P, P, P, P, P, U32, P]),
            "gdn_decode_step": (ctypes.c_int, [SH, I32, P, P, P, P, P, F, U32, P]),
            "gdn_conv_decode_step": (ctypes.c_int, [SH, I32, P, P, P, P, P, P, P, P, F, U32, P]),
            "gdn_kda_decode_step": (ctypes.c_int, [SH, I32, P, P, P, P, P, F, U32, P]),
            "gdn_kda_conv_decode_step": (ctypes.c_int, [SH, I32, P, P, P, P, P, P, P, P, F, U32, P]),
            "gdn_layer_decode_step": (ctypes.c_int, [SH, I32, P, P, P, P, P, P, P, P, P, P, F, P, P, P, F, U32,
                                                     P]),
            "gdn_gates": (ctypes.c_int, [I64, I32, P, P, P, P, P, P, P]),
            "gdn_tree_verify": (ctypes.c_int, [SH, I32, P, P, P, P, P, P, F, U32, P]),
            "gdn_tree_verify_batched": (ctypes.c_int, [SH, I32, P, P, P, P, P, P, P, F, U32, P]),
            "gdn_commit_path": (ctypes.c_int, [SH, I32, P, P, I32, P, P, P, P, P, P, U32, P]),
            "gdn_commit_path_batched": (ctypes.c_int, [SH, I32, P, P, P, P, P, P, P, P, P, P, U32, P]),
            "gdn_kda_tree_verify": (ctypes.c_int, [SH, I32, P, P, P, P, P, P, F, U32, P]),
            "gdn_kda_tree_verify_batched": (ctypes.c_int, [SH, I32, P, P, P, P, P, P, P, F, U32, P]),
            "gdn_kda_commit_path": (ctypes.c_int, [SH, I32, P, P, I32, P, P, P, P, P, P, U32, P]),
            "gdn_conv_tree_verify": (ctypes.c_int, [SH, I32, P, P, P, P, P, P, P, P, F, U32, P]),
            "gdn_conv_tree_verify_batched": (ctypes.c_int, [SH, I32, P, P, P, P, P, P, P, P, P, F, U32, P]),
            "gdn_conv_commit_path": (ctypes.c_int, [SH, I32, P, P, I32, P, P, P, P, P, P, P, U32, P]),
            "gdn_conv_commit_path_batched": (ctypes.c_int, [SH, I32, P, P, P, P, P, P, P, P, P, P, P, U32, P]),
            "gdn_prefill_workspace_bytes": (SZ, [SH, I32, I32]),
            "gdn_chunk_prefill": (ctypes.c_int, [SH, I32, I32, P, P, P, P, P, P, SZ, F, U32, P]),
            "gdn_prefill_status": (ctypes.c_int, [P, P, ctypes.POINTER(I32)]),
            "gdn_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
            "gdn_chunk_prefill_noalloc": (ctypes.c_int, [SH, I32, I32, P, P, P, P, P, F, U32, P]),
            "gdn_chunk_prefill_noalloc_status": (ctypes.c_int, [P, ctypes.POINTER(I32)]),
            "gdn_snapshot_bytes": (SZ, [SH, I32]),
            "gdn_snapshot_signature": (ctypes.c_uint64, [SH, I32]),
            "gdn_snapshot_save": (ctypes.c_int, [SH, I32, I32, P, I64, P, I64, P, SZ, P, SZ, P]),
            "gdn_snapshot_restore": (ctypes.c_int, [SH, I32, I32, P, SZ, P, I64, P, I64, P, SZ, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def last_error() -> str:
    return load().gdn_last_error().decode()


def _check(rc: int, fn: str):
    if rc != 0:
        raise GdnError(rc, fn, last_error())


def _shape(B, Hk, Hv, dk, dv) -> gdn_shape:
    return gdn_shape(int(B), int(Hk), int(Hv), int(dk), int(dv))


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dev(t: torch.Tensor | None, dtype, name: str, shape=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _host_i32(a, name):
    if a is None:
        return None, None
    arr = np.ascontiguousarray(a, dtype=np.int32)
    return arr, arr.ctypes.data_as(ctypes.c_void_p)


def packed_channels(Hk, Hv, dk, dv) -> int:
    """Length of a packed [q | k | v] row."""
    return 2 * Hk * dk + Hv * dv


def _flags(normalize: bool, out_bf16: bool) -> int:
    return (GDN_NORMALIZE_QK if normalize else 0) | (GDN_OUT_BF16 if out_bf16 else 0)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------
def abi_version() -> int:
    return load().gdn_abi_version()


def state_bytes(B, Hk, Hv, dk, dv) -> int:
    sh = _shape(B, Hk, Hv, dk, dv)
    return load().gdn_state_bytes(ctypes.byref(sh))


def tree_root_path(parents, node: int) -> np.ndarray:
    par, pp = _host_i32(parents, "parents")
    path = np.zeros(max(len(par), 1), np.int32)
    n = load().gdn_tree_root_path(len(par), pp, int(node), path.ctypes.data_as(ctypes.c_void_p),
                                  len(path))
    if n < 0:
        _check(n, "gdn_tree_root_path")
    return path[:n].copy()


def conv_step(x: torch.Tensor, w: torch.Tensor, tail: torch.Tensor, y: torch.Tensor | None = None,
              parents=None) -> torch.Tensor:
    """x bf16 [B,T,C], w bf16 [C,4], tail bf16 [B,4,C] (updated in place in linear mode).
    With fp32 x, every tensor is fp32 (GDN_IN_F32: y is not rounded to bf16)."""
    B, T, C = x.shape
    dt = torch.float32 if x.dtype == torch.float32 else torch.bfloat16
    if y is None:
        y = torch.empty_like(x)
    par, pp = _host_i32(parents, "parents")
    rc = load().gdn_conv_step(B, T, C, pp, _dev(x, dt, "x"),
                              _dev(w, dt, "w", (C, GDN_CONV_W)),
                              _dev(tail, dt, "tail", (B, GDN_CONV_W, C)),
                              _dev(y, dt, "y", (B, T, C)), GDN_IN_F32 if dt == torch.float32 else 0,
                              _stream())
    _check(rc, "gdn_conv_step")
    return y


def _decode(fn, qkv, alpha, beta, state, Hk, Hv, dk, dv, out, q_scale, normalize, out_bf16, gate_shape):
    B, T, C = qkv.shape
    if out is None:
        out = torch.empty((B, T, Hv, dv), dtype=torch.bfloat16 if out_bf16 else torch.float32,
                          device=qkv.device)
    sh = _shape(B, Hk, Hv, dk, dv)
    in_f32 = qkv.dtype == torch.float32  # GDN_IN_F32 (the library refuses it where unsupported)
    rc = getattr(load(), fn)(ctypes.byref(sh), T,
                             _dev(qkv, torch.float32 if in_f32 else torch.bfloat16, "qkv",
                                  (B, T, packed_channels(Hk, Hv, dk, dv))),
                             _dev(alpha, torch.float32, "alpha", gate_shape(B, T)),
                             _dev(beta, torch.float32, "beta", (B, T, Hv)),
                             _dev(state, torch.float32, "state", (B, Hv, dv, dk)),
                             _dev(out, torch.bfloat16 if out_bf16 else torch.float32, "out", (B, T, Hv, dv)),
                             float(q_scale), _flags(normalize, out_bf16) | (GDN_IN_F32 if in_f32 else 0),
                             _stream())
    _check(rc, fn)
    return out


def decode_step(qkv, alpha, beta, state, Hk, Hv, dk, dv, out=None, q_scale=1.0, normalize=True,
                out_bf16=False) -> torch.Tensor:
    """qkv bf16 [B,T,C] (or fp32: GDN_IN_F32), alpha/beta fp32 [B,T,Hv], state fp32
    [B,Hv,dv,dk] (in place)."""
    return _decode("gdn_decode_step", qkv, alpha, beta, state, Hk, Hv, dk, dv, out, q_scale, normalize,
                   out_bf16, lambda B, T: (B, T, Hv))


def kda_decode_step(qkv, alpha, beta, state, Hk, Hv, dk, dv, out=None, q_scale=1.0, normalize=True,
                    out_bf16=False) -> torch.Tensor:
    """KDA: alpha fp32 [B,T,Hv,dk] (a decay per key channel); the rest as decode_step."""
    return _decode("gdn_kda_decode_step", qkv, alpha, beta, state, Hk, Hv, dk, dv, out, q_scale, normalize,
                   out_bf16, lambda B, T: (B, T, Hv, dk))


def _conv_decode(fn, x, w, tail_in, alpha, beta, state, Hk, Hv, dk, dv, tail_out, out, q_scale, normalize,
                 out_bf16, gate_shape):
    B, T, C = x.shape
    if tail_out is None:
        tail_out = tail_in
    if out is None:
        out = torch.empty((B, T, Hv, dv), dtype=torch.bfloat16 if out_bf16 else torch.float32,
                          device=x.device)
    sh = _shape(B, Hk, Hv, dk, dv)
    C_ = packed_channels(Hk, Hv, dk, dv)
    rc = getattr(load(), fn)(ctypes.byref(sh), T, _dev(x, torch.bfloat16, "x", (B, T, C_)),
                             _dev(w, torch.bfloat16, "w", (C_, GDN_CONV_W)),
                             _dev(tail_in, torch.bfloat16, "tail_in", (B, GDN_CONV_W, C_)),
                             _dev(tail_out, torch.bfloat16, "tail_out", (B, GDN_CONV_W, C_)),
                             _dev(alpha, torch.float32, "alpha", gate_shape(B, T)),
                             _dev(beta, torch.float32, "beta", (B, T, Hv)),
                             _dev(state, torch.float32, "state", (B, Hv, dv, dk)),
                             _dev(out, torch.bfloat16 if out_bf16 else torch.float32, "out", (B, T, Hv, dv)),
                             float(q_scale), _flags(normalize, out_bf16), _stream())
    _check(rc, fn)
    return out


def conv_decode_step(x, w, tail_in, alpha, beta, state, Hk, Hv, dk, dv, tail_out=None, out=None,
                     q_scale=1.0, normalize=True, out_bf16=False) -> torch.Tensor:
    """Fused conv + decode.  x bf16 [B,T,C] pre-conv, w bf16 [C,4], tail_in bf16
    [B,4,C]; tail_out defaults to tail_in (in place).  Returns out [B,T,Hv,dv]."""
    return _conv_decode("gdn_conv_decode_step", x, w, tail_in, alpha, beta, state, Hk, Hv, dk, dv, tail_out,
                        out, q_scale, normalize, out_bf16, lambda B, T: (B, T, Hv))


def kda_conv_decode_step(x, w, tail_in, alpha, beta, state, Hk, Hv, dk, dv, tail_out=None, out=None,
                         q_scale=1.0, normalize=True, out_bf16=False) -> torch.Tensor:
    """Fused conv + KDA decode: alpha fp32 [B,T,Hv,dk]; the rest as conv_decode_step."""
    return _conv_decode("gdn_kda_conv_decode_step", x, w, tail_in, alpha, beta, state, Hk, Hv, dk, dv,
                        tail_out, out, q_scale, normalize, out_bf16, lambda B, T: (B, T, Hv, dk))


def layer_decode_step(x, conv_w, tail_in, a, b, A_log, dt_bias, z, norm_w, state, Hk, Hv, dk, dv, tail_out=None,
                      y=None, o=None, norm_eps=1e-6, q_scale=1.0, normalize=True) -> torch.Tensor:
    """The layer's decode step: x bf16 [B,T,C] pre-conv, conv_w bf16 [C,4], tail_in bf16 [B,4,C],
    a/b bf16 [B,T,Hv], A_log/dt_bias fp32 [Hv], z bf16 [B,T,Hv,dv], norm_w fp32 [dv],
    state fp32 [B,Hv,dv,dk] (in place).  Returns y bf16 [B,T,Hv,dv]; o (fp32, pre-norm) if given."""
    B, T, C = x.shape
    if tail_out is None:
        tail_out = tail_in
    if y is None:
        y = torch.empty((B, T, Hv, dv), dtype=torch.bfloat16, device=x.device)
    C_ = packed_channels(Hk, Hv, dk, dv)
    rc = load().gdn_layer_decode_step(
        ctypes.byref(_shape(B, Hk, Hv, dk, dv)), T, _dev(x, torch.bfloat16, "x", (B, T, C_)),
        _dev(conv_w, torch.bfloat16, "conv_w", (C_, GDN_CONV_W)),
        _dev(tail_in, torch.bfloat16, "tail_in", (B, GDN_CONV_W, C_)),
        _dev(tail_out, torch.bfloat16, "tail_out", (B, GDN_CONV_W, C_)),
        _dev(a, torch.bfloat16, "a", (B, T, Hv)), _dev(b, torch.bfloat16, "b", (B, T, Hv)),
        _dev(A_log, torch.float32, "A_log", (Hv,)), _dev(dt_bias, torch.float32, "dt_bias", (Hv,)),
        _dev(z, torch.bfloat16, "z", (B, T, Hv, dv)), _dev(norm_w, torch.float32, "norm_w", (dv,)), float(norm_eps),
        _dev(state, torch.float32, "state", (B, Hv, dv, dk)), _dev(o, torch.float32, "o", (B, T, Hv, dv)),
        _dev(y, torch.bfloat16, "y", (B, T, Hv, dv)), float(q_scale), _flags(normalize, False), _stream())
    _check(rc, "gdn_layer_decode_step")
    return y


def gates(a, b, A_log, dt_bias):
    """a, b bf16 [..., Hv]; A_log, dt_bias fp32 [Hv] -> (alpha, beta) fp32 [..., Hv]."""
    Hv = a.shape[-1]
    n = a.numel() // Hv
    alpha = torch.empty(a.shape, dtype=torch.float32, device=a.device)
    beta = torch.empty(a.shape, dtype=torch.float32, device=a.device)
    rc = load().gdn_gates(n, Hv, _dev(a, torch.bfloat16, "a"), _dev(b, torch.bfloat16, "b", tuple(a.shape)),
                          _dev(A_log, torch.float32, "A_log", (Hv,)), _dev(dt_bias, torch.float32, "dt_bias", (Hv,)),
                          _dev(alpha, torch.float32, "alpha"), _dev(beta, torch.float32, "beta"), _stream())
    _check(rc, "gdn_gates")
    return alpha, beta


def tree_verify(parents, qkv, alpha, beta, state, Hk, Hv, dk, dv, out=None, q_scale=1.0,
                normalize=True, out_bf16=False) -> torch.Tensor:
    """qkv bf16 [N,C], alpha/beta fp32 [N,Hv], state fp32 [Hv,dv,dk] (read only)."""
    par, pp = _host_i32(parents, "parents")
    N = len(par)
    if out is None:
        out = torch.empty((N, Hv, dv), dtype=torch.bfloat16 if out_bf16 else torch.float32,
                          device=qkv.device)
    sh = _shape(1, Hk, Hv, dk, dv)
    rc = load().gdn_tree_verify(ctypes.byref(sh), N, pp,
                                _dev(qkv, torch.bfloat16, "qkv", (N, packed_channels(Hk, Hv, dk, dv))),
                                _dev(alpha, torch.float32, "alpha", (N, Hv)),
                                _dev(beta, torch.float32, "beta", (N, Hv)),
                                _dev(state, torch.float32, "state", (Hv, dv, dk)),
                                _dev(out, torch.bfloat16 if out_bf16 else torch.float32, "out",
                                     (N, Hv, dv)),
                                float(q_scale), _flags(normalize, out_bf16), _stream())
    _check(rc, "gdn_tree_verify")
    return out


def tree_verify_batched(counts, parents, qkv, alpha, beta, state, Hk, Hv, dk, dv, out=None, q_scale=1.0,
                        normalize=True, out_bf16=False) -> torch.Tensor:
    """B trees in one launch.  counts [B], parents [B,N] (host), qkv bf16 [B,N,C],
    alpha/beta fp32 [B,N,Hv], state fp32 [B,Hv,dv,dk] (read only) -> out [B,N,Hv,dv]."""
    cnt, pc = _host_i32(counts, "counts")
    par, pp = _host_i32(parents, "parents")
    B, N = par.shape
    if out is None:
        out = torch.empty((B, N, Hv, dv), dtype=torch.bfloat16 if out_bf16 else torch.float32,
                          device=qkv.device)
    sh = _shape(B, Hk, Hv, dk, dv)
    rc = load().gdn_tree_verify_batched(
        ctypes.byref(sh), N, pc, pp,
        _dev(qkv, torch.bfloat16, "qkv", (B, N, packed_channels(Hk, Hv, dk, dv))),
        _dev(alpha, torch.float32, "alpha", (B, N, Hv)), _dev(beta, torch.float32, "beta", (B, N, Hv)),
        _dev(state, torch.float32, "state", (B, Hv, dv, dk)),
        _dev(out, torch.bfloat16 if out_bf16 else torch.float32, "out", (B, N, Hv, dv)),
        float(q_scale), _flags(normalize, out_bf16), _stream())
    _check(rc, "gdn_tree_verify_batched")
    return out


def commit_path(parents, path, qkv, alpha, beta, state, Hk, Hv, dk, dv, x_tree=None, tail=None,
                normalize=True) -> None:
    """Replays `path` through the step in place on state [Hv,dv,dk]; updates tail [4,C]."""
    par, pp = _host_i32(parents, "parents")
    pa, ppa = _host_i32(path, "path")
    N = len(par)
    sh = _shape(1, Hk, Hv, dk, dv)
    rc = load().gdn_commit_path(ctypes.byref(sh), N, pp, ppa, len(pa),
                                _dev(qkv, torch.bfloat16, "qkv", (N, packed_channels(Hk, Hv, dk, dv))),
                                _dev(alpha, torch.float32, "alpha", (N, Hv)),
                                _dev(beta, torch.float32, "beta", (N, Hv)),
                                _dev(x_tree, torch.bfloat16, "x_tree", (N, packed_channels(Hk, Hv, dk, dv))),
                                _dev(state, torch.float32, "state", (Hv, dv, dk)),
                                _dev(tail, torch.bfloat16, "tail", (GDN_CONV_W, packed_channels(Hk, Hv, dk, dv))), _flags(normalize, False),
                                _stream())
    _check(rc, "gdn_commit_path")


def commit_path_batched(counts, parents, paths, lengths, qkv, alpha, beta, state, Hk, Hv, dk, dv, x_tree=None,
                        tail=None, normalize=True) -> None:
    """B sequences' accepted paths in one launch.  counts [B], parents [B,N],
    paths [B,N] (first lengths[b] entries used), lengths [B] (host); qkv bf16
    [B,N,C], alpha/beta fp32 [B,N,Hv], x_tree bf16 [B,N,C] or None; state fp32
    [B,Hv,dv,dk] and tail bf16 [B,4,C] updated in place."""
    cnt, pc = _host_i32(counts, "counts")
    par, pp = _host_i32(parents, "parents")
    pth, ppth = _host_i32(paths, "paths")
    ln, pl = _host_i32(lengths, "lengths")
    B, N = par.shape
    C = packed_channels(Hk, Hv, dk, dv)
    rc = load().gdn_commit_path_batched(
        ctypes.byref(_shape(B, Hk, Hv, dk, dv)), N, pc, pp, ppth, pl,
        _dev(qkv, torch.bfloat16, "qkv", (B, N, C)), _dev(alpha, torch.float32, "alpha", (B, N, Hv)),
        _dev(beta, torch.float32, "beta", (B, N, Hv)), _dev(x_tree, torch.bfloat16, "x_tree", (B, N, C)),
        _dev(state, torch.float32, "state", (B, Hv, dv, dk)), _dev(tail, torch.bfloat16, "tail", (B, GDN_CONV_W, C)),
        _flags(normalize, False), _stream())
    _check(rc, "gdn_commit_path_batched")


def kda_tree_verify(parents, qkv, alpha, beta, state, Hk, Hv, dk, dv, out=None, q_scale=1.0,
                    normalize=True, out_bf16=False) -> torch.Tensor:
    """The KDA tree verify.  qkv bf16 [N,C], alpha fp32 [N,Hv,dk], beta fp32 [N,Hv],
    state fp32 [Hv,dv,dk] (read only) -> out [N,Hv,dv]."""
    par, pp = _host_i32(parents, "parents")
    N = len(par)
    if out is None:
        out = torch.empty((N, Hv, dv), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=qkv.device)
    rc = load().gdn_kda_tree_verify(
        ctypes.byref(_shape(1, Hk, Hv, dk, dv)), N, pp,
        _dev(qkv, torch.bfloat16, "qkv", (N, packed_channels(Hk, Hv, dk, dv))),
        _dev(alpha, torch.float32, "alpha", (N, Hv, dk)), _dev(beta, torch.float32, "beta", (N, Hv)),
        _dev(state, torch.float32, "state", (Hv, dv, dk)),
        _dev(out, torch.bfloat16 if out_bf16 else torch.float32, "out", (N, Hv, dv)),
        float(q_scale), _flags(normalize, out_bf16), _stream())
    _check(rc, "gdn_kda_tree_verify")
    return out


def kda_tree_verify_batched(counts, parents, qkv, alpha, beta, state, Hk, Hv, dk, dv, out=None, q_scale=1.0,
                            normalize=True, out_bf16=False) -> torch.Tensor:
    """B trees' KDA verify in one launch.  counts [B], parents [B,N] (host), qkv bf16 [B,N,C],
    alpha fp32 [B,N,Hv,dk], beta fp32 [B,N,Hv], state fp32 [B,Hv,dv,dk] (read only) -> out [B,N,Hv,dv]."""
    cnt, pc = _host_i32(counts, "counts")
    par, pp = _host_i32(parents, "parents")
    B, N = par.shape
    if out is None:
        out = torch.empty((B, N, Hv, dv), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=qkv.device)
    rc = load().gdn_kda_tree_verify_batched(
        ctypes.byref(_shape(B, Hk, Hv, dk, dv)), N, pc, pp,
        _dev(qkv, torch.bfloat16, "qkv", (B, N, packed_channels(Hk, Hv, dk, dv))),
        _dev(alpha, torch.float32, "alpha", (B, N, Hv, dk)), _dev(beta, torch.float32, "beta", (B, N, Hv)),
        _dev(state, torch.float32, "state", (B, Hv, dv, dk)),
        _dev(out, torch.bfloat16 if out_bf16 else torch.float32, "out", (B, N, Hv, dv)),
        float(q_scale), _flags(normalize, out_bf16), _stream())
    _check(rc, "gdn_kda_tree_verify_batched")
    return out


def kda_commit_path(parents, path, qkv, alpha, beta, state, Hk, Hv, dk, dv, x_tree=None, tail=None,
                    normalize=True) -> None:
    """The KDA commit: replays `path` in place on state [Hv,dv,dk]; alpha fp32 [N,Hv,dk]; updates tail [4,C]."""
    par, pp = _host_i32(parents, "parents")
    pa, ppa = _host_i32(path, "path")
    N = len(par)
    C = packed_channels(Hk, Hv, dk, dv)
    rc = load().gdn_kda_commit_path(
        ctypes.byref(_shape(1, Hk, Hv, dk, dv)), N, pp, ppa, len(pa), _dev(qkv, torch.bfloat16, "qkv", (N, C)),
        _dev(alpha, torch.float32, "alpha", (N, Hv, dk)), _dev(beta, torch.float32, "beta", (N, Hv)),
        _dev(x_tree, torch.bfloat16, "x_tree", (N, C)), _dev(state, torch.float32, "state", (Hv, dv, dk)),
        _dev(tail, torch.bfloat16, "tail", (GDN_CONV_W, C)), _flags(normalize, False), _stream())
    _check(rc, "gdn_kda_commit_path")


def conv_tree_verify(parents, x, w, tail, alpha, beta, state, Hk, Hv, dk, dv, out=None, q_scale=1.0,
                     normalize=True, out_bf16=False) -> torch.Tensor:
    """The tree conv and verify in one launch.  x bf16 [N,C] pre-conv, w bf16 [C,4],
    tail bf16 [4,C] (read only), alpha/beta fp32 [N,Hv], state fp32 [Hv,dv,dk] (read only)."""
    par, pp = _host_i32(parents, "parents")
    N = len(par)
    C = packed_channels(Hk, Hv, dk, dv)
    if out is None:
        out = torch.empty((N, Hv, dv), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=x.device)
    rc = load().gdn_conv_tree_verify(
        ctypes.byref(_shape(1, Hk, Hv, dk, dv)), N, pp, _dev(x, torch.bfloat16, "x", (N, C)),
        _dev(w, torch.bfloat16, "w", (C, GDN_CONV_W)), _dev(tail, torch.bfloat16, "tail", (GDN_CONV_W, C)),
        _dev(alpha, torch.float32, "alpha", (N, Hv)), _dev(beta, torch.float32, "beta", (N, Hv)),
        _dev(state, torch.float32, "state", (Hv, dv, dk)),
        _dev(out, torch.bfloat16 if out_bf16 else torch.float32, "out", (N, Hv, dv)),
        float(q_scale), _flags(normalize, out_bf16), _stream())
    _check(rc, "gdn_conv_tree_verify")
    return out


def conv_tree_verify_batched(counts, parents, x, w, tail, alpha, beta, state, Hk, Hv, dk, dv, out=None,
                             q_scale=1.0, normalize=True, out_bf16=False) -> torch.Tensor:
    """B trees' conv and joint verify in one launch.  counts [B], parents [B,N] (host),
    x bf16 [B,N,C], w bf16 [C,4], tail bf16 [B,4,C] (read only), alpha/beta fp32 [B,N,Hv],
    state fp32 [B,Hv,dv,dk] (read only) -> out [B,N,Hv,dv]."""
    cnt, pc = _host_i32(counts, "counts")
    par, pp = _host_i32(parents, "parents")
    B, N = par.shape
    C = packed_channels(Hk, Hv, dk, dv)
    if out is None:
        out = torch.empty((B, N, Hv, dv), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=x.device)
    rc = load().gdn_conv_tree_verify_batched(
        ctypes.byref(_shape(B, Hk, Hv, dk, dv)), N, pc, pp, _dev(x, torch.bfloat16, "x", (B, N, C)),
        _dev(w, torch.bfloat16, "w", (C, GDN_CONV_W)), _dev(tail, torch.bfloat16, "tail", (B, GDN_CONV_W, C)),
        _dev(alpha, torch.float32, "alpha", (B, N, Hv)), _dev(beta, torch.float32, "beta", (B, N, Hv)),
        _dev(state, torch.float32, "state", (B, Hv, dv, dk)),
        _dev(out, torch.bfloat16 if out_bf16 else torch.float32, "out", (B, N, Hv, dv)),
        float(q_scale), _flags(normalize, out_bf16), _stream())
    _check(rc, "gdn_conv_tree_verify_batched")
    return out


def conv_commit_path(parents, path, x, w, tail_in, tail_out, alpha, beta, state, Hk, Hv, dk, dv,
                     normalize=True) -> None:
    """The commit from pre-conv inputs: x bf16 [N,C], w bf16 [C,4]; tail_in bf16 [4,C] read,
    tail_out bf16 [4,C] written (a distinct buffer); state fp32 [Hv,dv,dk] in place."""
    par, pp = _host_i32(parents, "parents")
    pa, ppa = _host_i32(path, "path")
    N = len(par)
    C = packed_channels(Hk, Hv, dk, dv)
    rc = load().gdn_conv_commit_path(
        ctypes.byref(_shape(1, Hk, Hv, dk, dv)), N, pp, ppa, len(pa), _dev(x, torch.bfloat16, "x", (N, C)),
        _dev(w, torch.bfloat16, "w", (C, GDN_CONV_W)), _dev(tail_in, torch.bfloat16, "tail_in", (GDN_CONV_W, C)),
        _dev(tail_out, torch.bfloat16, "tail_out", (GDN_CONV_W, C)),
        _dev(alpha, torch.float32, "alpha", (N, Hv)), _dev(beta, torch.float32, "beta", (N, Hv)),
        _dev(state, torch.float32, "state", (Hv, dv, dk)), _flags(normalize, False), _stream())
    _check(rc, "gdn_conv_commit_path")


def conv_commit_path_batched(counts, parents, paths, lengths, x, w, tail_in, tail_out, alpha, beta, state,
                             Hk, Hv, dk, dv, normalize=True) -> None:
    """B sequences' commits from pre-conv inputs in one launch.  counts [B], parents [B,N],
    paths [B,N], lengths [B] (host); x bf16 [B,N,C], w bf16 [C,4]; tail_in bf16 [B,4,C] read,
    tail_out bf16 [B,4,C] written for every sequence; state fp32 [B,Hv,dv,dk] in place."""
    cnt, pc = _host_i32(counts, "counts")
    par, pp = _host_i32(parents, "parents")
    pth, ppth = _host_i32(paths, "paths")
    ln, pl = _host_i32(lengths, "lengths")
    B, N = par.shape
    C = packed_channels(Hk, Hv, dk, dv)
    rc = load().gdn_conv_commit_path_batched(
        ctypes.byref(_shape(B, Hk, Hv, dk, dv)), N, pc, pp, ppth, pl, _dev(x, torch.bfloat16, "x", (B, N, C)),
        _dev(w, torch.bfloat16, "w", (C, GDN_CONV_W)),
        _dev(tail_in, torch.bfloat16, "tail_in", (B, GDN_CONV_W, C)),
        _dev(tail_out, torch.bfloat16, "tail_out", (B, GDN_CONV_W, C)),
        _dev(alpha, torch.float32, "alpha", (B, N, Hv)), _dev(beta, torch.float32, "beta", (B, N, Hv)),
        _dev(state, torch.float32, "state", (B, Hv, dv, dk)), _flags(normalize, False), _stream())
    _check(rc, "gdn_conv_commit_path_batched")


def prefill_workspace_bytes(T, Hk, Hv, dk, dv, chunk=64) -> int:
    sh = _shape(1, Hk, Hv, dk, dv)
    return load().gdn_prefill_workspace_bytes(ctypes.byref(sh), int(T), int(chunk))


def chunk_prefill(qkv, alpha, beta, state, Hk, Hv, dk, dv, out=None, workspace=None, chunk=64,
                  q_scale=1.0, normalize=True, out_bf16=False, two_launch=False) -> torch.Tensor:
    """qkv bf16 [T,C], alpha/beta fp32 [T,Hv], state fp32 [Hv,dv,dk] (S_0 in, S_T out).
    two_launch: the pre-pass, then the chain, as two launches (GDN_PREFILL_TWO_LAUNCH)."""
    T = qkv.shape[0]
    if out is None:
        out = torch.empty((T, Hv, dv), dtype=torch.bfloat16 if out_bf16 else torch.float32,
                          device=qkv.device)
    ws_bytes = prefill_workspace_bytes(T, Hk, Hv, dk, dv, chunk)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=qkv.device)
    sh = _shape(1, Hk, Hv, dk, dv)
    rc = load().gdn_chunk_prefill(ctypes.byref(sh), T, int(chunk),
                                  _dev(qkv, torch.bfloat16, "qkv", (T, packed_channels(Hk, Hv, dk, dv))),
                                  _dev(alpha, torch.float32, "alpha", (T, Hv)),
                                  _dev(beta, torch.float32, "beta", (T, Hv)),
                                  _dev(state, torch.float32, "state", (Hv, dv, dk)),
                                  _dev(out, torch.bfloat16 if out_bf16 else torch.float32, "out",
                                       (T, Hv, dv)),
                                  _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                                  float(q_scale),
                                  _flags(normalize, out_bf16) | (GDN_PREFILL_TWO_LAUNCH if two_launch else 0),
                                  _stream())
    _check(rc, "gdn_chunk_prefill")
    return out


def prefill_status(workspace: torch.Tensor) -> int:
    """Synchronise the current stream and return the status word of the last
    gdn_chunk_prefill call that used `workspace` (0: the results are valid;
    non-zero: a bounded device wait gave up)."""
    st = ctypes.c_int32(0)
    rc = load().gdn_prefill_status(_dev(workspace, torch.uint8, "workspace"), _stream(), ctypes.byref(st))
    if rc not in (0, -8):
        _check(rc, "gdn_prefill_status")
    return int(st.value)


def set_wait_limit_ns(ns: int) -> int:
    """Limit of every bounded device wait of the prefill kernels (process-wide,
    read at each later launch); returns the previous limit."""
    return int(load().gdn_set_wait_limit_ns(int(ns)))


def chunk_prefill_noalloc(qkv, alpha, beta, state, Hk, Hv, dk, dv, out=None, chunk=64, q_scale=1.0,
                          normalize=True, out_bf16=False) -> torch.Tensor:
    """gdn_chunk_prefill_noalloc: chunk_prefill without a workspace (its
    scratch lives in the library).  Same arguments and layouts."""
    T = qkv.shape[0]
    if out is None:
        out = torch.empty((T, Hv, dv), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=qkv.device)
    sh = _shape(1, Hk, Hv, dk, dv)
    rc = load().gdn_chunk_prefill_noalloc(ctypes.byref(sh), T, int(chunk),
                                          _dev(qkv, torch.bfloat16, "qkv", (T, packed_channels(Hk, Hv, dk, dv))),
                                          _dev(alpha, torch.float32, "alpha", (T, Hv)),
                                          _dev(beta, torch.float32, "beta", (T, Hv)),
                                          _dev(state, torch.float32, "state", (Hv, dv, dk)),
                                          _dev(out, torch.bfloat16 if out_bf16 else torch.float32, "out",
                                               (T, Hv, dv)),
                                          float(q_scale), _flags(normalize, out_bf16), _stream())
    _check(rc, "gdn_chunk_prefill_noalloc")
    return out


def chunk_prefill_noalloc_status() -> int:
    """Synchronise the current stream and return the status word the last
    gdn_chunk_prefill_noalloc call on this device left (0: valid results)."""
    st = ctypes.c_int32(0)
    rc = load().gdn_chunk_prefill_noalloc_status(_stream(), ctypes.byref(st))
    if rc not in (0, -8):
        _check(rc, "gdn_chunk_prefill_noalloc_status")
    return int(st.value)


# ---------------------------------------------------------------------------
# snapshot / restore of one sequence's recurrent sections
# ---------------------------------------------------------------------------
SNAPSHOT_WORKSPACE_BYTES = 256
SNAPSHOT_STATUS = {0: "ok", 1: "header does not match this shape (magic/version/layers/shape/signature/size)",
                   2: "payload checksum does not match"}


def snapshot_bytes(layers, Hk, Hv, dk, dv) -> int:
    return int(load().gdn_snapshot_bytes(ctypes.byref(_shape(1, Hk, Hv, dk, dv)), int(layers)))


def snapshot_signature(layers, Hk, Hv, dk, dv) -> int:
    return int(load().gdn_snapshot_signature(ctypes.byref(_shape(1, Hk, Hv, dk, dv)), int(layers)))


def _layered(t: torch.Tensor, dtype, name: str, inner) -> tuple[ctypes.c_void_p, int]:
    """A [layers, *inner] CUDA tensor whose layers may be strided apart but are
    each contiguous: (pointer, layer stride in elements)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape[1:]) != tuple(inner):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected (layers, {', '.join(map(str, inner))})")
    if not t[0].is_contiguous():
        raise ValueError(f"each layer of {name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr()), int(t.stride(0))


def _blob(t: torch.Tensor, name: str) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor) or t.dtype != torch.uint8 or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous uint8 tensor")
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be device memory or pinned host memory")
    return ctypes.c_void_p(t.data_ptr())


def snapshot_save(state, tail, seq, Hk, Hv, dk, dv, dst=None, workspace=None, host=False) -> torch.Tensor:
    """Blob of sequence `seq` from state fp32 [L,B,Hv,dv,dk] and tail bf16
    [L,B,4,C].  dst: a uint8 tensor (device, or pinned host) of at least
    snapshot_bytes(); by default a new device tensor (pinned host with host=True)."""
    L, B = state.shape[0], state.shape[1]
    C = packed_channels(Hk, Hv, dk, dv)
    sp, ss = _layered(state, torch.float32, "state", (B, Hv, dv, dk))
    tp, ts = _layered(tail, torch.bfloat16, "tail", (B, 4, C))
    n = snapshot_bytes(L, Hk, Hv, dk, dv)
    if dst is None:
        dst = (torch.empty(n, dtype=torch.uint8, pin_memory=True) if host
               else torch.empty(n, dtype=torch.uint8, device=state.device))
    if workspace is None:
        workspace = torch.empty(SNAPSHOT_WORKSPACE_BYTES, dtype=torch.uint8, device=state.device)
    rc = load().gdn_snapshot_save(ctypes.byref(_shape(B, Hk, Hv, dk, dv)), L, int(seq), sp, ss, tp, ts,
                                  _blob(dst, "dst"), dst.numel(), _dev(workspace, torch.uint8, "workspace"),
                                  workspace.numel(), _stream())
    _check(rc, "gdn_snapshot_save")
    return dst


def snapshot_restore(src, state, tail, seq, Hk, Hv, dk, dv, workspace=None, check=True) -> int:
    """Verify the blob `src` and write it into sequence `seq` of state/tail.
    With check=True, synchronise and raise GdnError when the device refused
    the blob (nothing is written then); return the status word (0 = done)."""
    L, B = state.shape[0], state.shape[1]
    C = packed_channels(Hk, Hv, dk, dv)
    sp, ss = _layered(state, torch.float32, "state", (B, Hv, dv, dk))
    tp, ts = _layered(tail, torch.bfloat16, "tail", (B, 4, C))
    if workspace is None:
        workspace = torch.empty(SNAPSHOT_WORKSPACE_BYTES, dtype=torch.uint8, device=state.device)
    rc = load().gdn_snapshot_restore(ctypes.byref(_shape(B, Hk, Hv, dk, dv)), L, int(seq), _blob(src, "src"),
                                     src.numel(), sp, ss, tp, ts, _dev(workspace, torch.uint8, "workspace"),
                                     workspace.numel(), _stream())
    _check(rc, "gdn_snapshot_restore")
    if not check:
        return 0
    torch.cuda.current_stream().synchronize()
    status = int(workspace[:4].view(torch.int32).item())
    if status != 0:
        raise GdnError(-100 - status, "gdn_snapshot_restore", SNAPSHOT_STATUS.get(status, str(status)))
    return status


def write_snapshot_file(blob: torch.Tensor, path: str) -> None:
    """Write a blob to a file as it is (the format carries its own header)."""
    blob.detach().cpu().numpy().tofile(path)


def read_snapshot_file(path: str, pinned: bool = True) -> torch.Tensor:
    """Read a blob file into (pinned) host memory, ready for snapshot_restore."""
    t = torch.from_numpy(np.fromfile(path, dtype=np.uint8))
    return t.pin_memory() if pinned else t


# ---------------------------------------------------------------------------
# conversions between the generator's numpy arrays and device tensors
# ---------------------------------------------------------------------------
def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """Raw bf16 bits (uint16 numpy) -> bf16 tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> raw bits as uint16 numpy."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
