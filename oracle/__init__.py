"""fp64 CPU oracle for the Gated DeltaNet mixer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The CUDA library never does, and shares no code with
it.  This module only marshals numpy arrays into the plain C oracle in
``gdn_oracle.c`` (built with gcc on first use); every step of the arithmetic is
in that C file, with its sources cited in ``gdn_oracle.h``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_HDR = os.path.join(_HERE, "gdn_oracle.h")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

CONV_W = 4


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, no FMA contraction); return the path."""
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest_src:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        sig = {
            "orc_bf16_to_f64": (D, [ctypes.c_uint16]),
            "orc_f64_to_bf16": (ctypes.c_uint16, [D]),
            "orc_bf16_to_f64_n": (None, [P, P, ctypes.c_int64]),
            "orc_f64_to_bf16_n": (None, [P, P, ctypes.c_int64]),
            "orc_silu": (D, [D]),
            "orc_conv_linear": (None, [I, I, I, I, P, P, P, P]),
            "orc_conv_tree": (None, [I, I, I, P, P, P, P, P]),
            "orc_conv_linear_f32": (None, [I, I, I, I, P, P, P, P]),
            "orc_conv_linear_r32": (None, [I, I, I, I, P, P, P, P]),
            "orc_conv_tree_r32": (None, [I, I, I, P, P, P, P, P]),
            "orc_decode_f32": (None, [I, I, I, I, I, I, P, P, P, P, P, D, I]),
            "orc_tree_check": (I, [I, P, P]),
            "orc_root_path": (I, [I, P, I, P]),
            "orc_path_check": (I, [I, P, P, I]),
            "orc_l2norm": (None, [P, I, D, P]),
            "orc_delta_token": (None, [I, I, P, P, P, P, D, D, P]),
            "orc_delta_token_matrix": (None, [I, I, P, P, P, P, D, D, P]),
            "orc_decode": (None, [I, I, I, I, I, I, P, P, P, P, P, D, I]),
            "orc_tree_verify": (None, [I, I, I, I, I, P, P, P, P, P, P, D, I]),
            "orc_commit": (None, [I, I, I, I, I, P, P, I, P, P, P, P, I, P, P, I]),
            "orc_kda_token": (None, [I, I, P, P, P, P, P, D, P]),
            "orc_kda_token_matrix": (None, [I, I, P, P, P, P, P, D, P]),
            "orc_kda_decode": (None, [I, I, I, I, I, I, P, P, P, P, P, D, I]),
            "orc_softplus": (D, [D]),
            "orc_sigmoid": (D, [D]),
            "orc_gates": (None, [I, I, P, P, P, P, P, P]),
            "orc_gated_rmsnorm": (None, [I, P, P, P, D, P]),
            "orc_layer_decode": (None, [I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, D, P, P, P, D, I]),
            "orc_fnv1a64": (ctypes.c_uint64, [P, ctypes.c_size_t]),
            "orc_mix64": (ctypes.c_uint64, [ctypes.c_uint64]),
            "orc_snapshot_checksum": (ctypes.c_uint64, [P, ctypes.c_size_t]),
            "orc_snapshot_signature": (ctypes.c_uint64, [I, I, I, I, I]),
            "orc_snapshot_bytes": (ctypes.c_size_t, [I, I, I, I, I]),
            "orc_snapshot_save": (None, [I, I, I, I, I, I, I, P, P, P]),
            "orc_snapshot_restore": (I, [I, I, I, I, I, I, I, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# bf16 storage
# --------------------------------------------------------------------------
def bf16_to_f64(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float64)
    _load().orc_bf16_to_f64_n(_ptr(h), _ptr(out), h.size)
    return out


def f64_to_bf16(x) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().orc_f64_to_bf16_n(_ptr(x), _ptr(out), x.size)
    return out


def silu(z: float) -> float:
    return _load().orc_silu(float(z))


# --------------------------------------------------------------------------
# convolution
# --------------------------------------------------------------------------
def conv_linear(x, w, tail):
    """x bf16 [B,T,C], w bf16 [C,4], tail bf16 [B,4,C] -> (y f64 [B,T,C], new tail)."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    tail = _c(tail, np.uint16).copy()
    B, T, C = x.shape
    W = w.shape[1]
    y = np.empty((B, T, C), np.float64)
    _load().orc_conv_linear(B, T, C, W, _ptr(x), _ptr(w), _ptr(tail), _ptr(y))
    return y, tail


def conv_linear_f32(x, w, tail):
    """conv_linear over fp32 x [B,T,C], w [C,4], tail [B,4,C] -> (y f64, new fp32 tail)."""
    x = _c(x, np.float32)
    w = _c(w, np.float32)
    tail = _c(tail, np.float32).copy()
    B, T, C = x.shape
    W = w.shape[1]
    y = np.empty((B, T, C), np.float64)
    _load().orc_conv_linear_f32(B, T, C, W, _ptr(x), _ptr(w), _ptr(tail), _ptr(y))
    return y, tail


def conv_tree(parents, x, w, tail):
    """x bf16 [N,C], tail bf16 [4,C] (read only) -> y f64 [N,C]."""
    parents = _c(parents, np.int32)
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    tail = _c(tail, np.uint16)
    N, C = x.shape
    y = np.empty((N, C), np.float64)
    _load().orc_conv_tree(N, C, w.shape[1], _ptr(parents), _ptr(x), _ptr(w), _ptr(tail), _ptr(y))
    return y


def conv_linear_r32(x, w, tail):
    """conv_linear with the outputs as bf16 bits, rounded from binary32 (the
    precision the CUDA conv rounds in) -> (y bf16 [B,T,C], new tail)."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    tail = _c(tail, np.uint16).copy()
    B, T, C = x.shape
    y = np.empty((B, T, C), np.uint16)
    _load().orc_conv_linear_r32(B, T, C, w.shape[1], _ptr(x), _ptr(w), _ptr(tail), _ptr(y))
    return y, tail


def conv_tree_r32(parents, x, w, tail):
    """conv_tree with the outputs as bf16 bits, rounded from binary32 -> y bf16 [N,C]."""
    parents = _c(parents, np.int32)
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    tail = _c(tail, np.uint16)
    N, C = x.shape
    y = np.empty((N, C), np.uint16)
    _load().orc_conv_tree_r32(N, C, w.shape[1], _ptr(parents), _ptr(x), _ptr(w), _ptr(tail), _ptr(y))
    return y


# --------------------------------------------------------------------------
# tree bookkeeping
# --------------------------------------------------------------------------
def tree_check(parents):
    parents = _c(parents, np.int32)
    depth = np.zeros(max(len(parents), 1), np.int32)
    rc = _load().orc_tree_check(len(parents), _ptr(parents), _ptr(depth))
    return rc, depth[: len(parents)]


def root_path(parents, node: int) -> np.ndarray:
    parents = _c(parents, np.int32)
    path = np.zeros(len(parents), np.int32)
    L = _load().orc_root_path(len(parents), _ptr(parents), int(node), _ptr(path))
    return path[:L].copy()


def path_check(parents, path) -> int:
    parents = _c(parents, np.int32)
    path = _c(path, np.int32)
    return _load().orc_path_check(len(parents), _ptr(parents), _ptr(path) if path.size else None,
                                  int(path.size))


# --------------------------------------------------------------------------
# gated delta rule
# --------------------------------------------------------------------------
def l2norm(x, eps=1e-6):
    x = _c(x, np.float64)
    out = np.empty_like(x)
    _load().orc_l2norm(_ptr(x), x.size, float(eps), _ptr(out))
    return out


def delta_token(S, k, v, q, alpha, beta, matrix_form=False):
    """One token, one head, fp64 vectors.  Returns (S_new, o)."""
    S = _c(S, np.float64).copy()
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    q = _c(q, np.float64)
    dv, dk = S.shape
    o = np.empty(dv, np.float64)
    fn = _load().orc_delta_token_matrix if matrix_form else _load().orc_delta_token
    fn(dk, dv, _ptr(S), _ptr(k), _ptr(v), _ptr(q), float(alpha), float(beta), _ptr(o))
    return S, o


def decode(qkv, alpha, beta, state, Hk, Hv, dk, dv, q_scale=1.0, normalize=True):
    """qkv bf16 [B,T,C], alpha/beta f32 [B,T,Hv], state [B,Hv,dv,dk] (any float).

    Returns (out f64 [B,T,Hv,dv], state f64)."""
    qkv = _c(qkv, np.uint16)
    alpha = _c(alpha, np.float32)
    beta = _c(beta, np.float32)
    st = _c(state, np.float64).copy()
    B, T = qkv.shape[0], qkv.shape[1]
    assert qkv.shape[2] == 2 * Hk * dk + Hv * dv
    assert st.shape == (B, Hv, dv, dk)
    out = np.empty((B, T, Hv, dv), np.float64)
    _load().orc_decode(B, T, Hk, Hv, dk, dv, _ptr(qkv), _ptr(alpha), _ptr(beta), _ptr(st),
                       _ptr(out), float(q_scale), int(bool(normalize)))
    return out, st


def decode_f32(qkv, alpha, beta, state, Hk, Hv, dk, dv, q_scale=1.0, normalize=True):
    """decode() over fp32 activations qkv [B,T,C] (no bf16 rounding anywhere)."""
    qkv = _c(qkv, np.float32)
    alpha = _c(alpha, np.float32)
    beta = _c(beta, np.float32)
    st = _c(state, np.float64).copy()
    B, T = qkv.shape[0], qkv.shape[1]
    assert qkv.shape[2] == 2 * Hk * dk + Hv * dv
    assert st.shape == (B, Hv, dv, dk)
    out = np.empty((B, T, Hv, dv), np.float64)
    _load().orc_decode_f32(B, T, Hk, Hv, dk, dv, _ptr(qkv), _ptr(alpha), _ptr(beta), _ptr(st),
                           _ptr(out), float(q_scale), int(bool(normalize)))
    return out, st


def tree_verify(parents, qkv, alpha, beta, state, Hk, Hv, dk, dv, q_scale=1.0, normalize=True):
    """qkv bf16 [N,C], alpha/beta f32 [N,Hv], state [Hv,dv,dk] -> out f64 [N,Hv,dv]."""
    parents = _c(parents, np.int32)
    qkv = _c(qkv, np.uint16)
    alpha = _c(alpha, np.float32)
    beta = _c(beta, np.float32)
    st = _c(state, np.float64)
    N = len(parents)
    out = np.empty((N, Hv, dv), np.float64)
    _load().orc_tree_verify(N, Hk, Hv, dk, dv, _ptr(parents), _ptr(qkv), _ptr(alpha), _ptr(beta),
                            _ptr(st), _ptr(out), float(q_scale), int(bool(normalize)))
    return out


def commit(parents, path, qkv, alpha, beta, state, Hk, Hv, dk, dv, x_tree=None, tail=None,
           normalize=True):
    """Returns (state f64 [Hv,dv,dk], tail bf16 [4,C] or None)."""
    parents = _c(parents, np.int32)
    path = _c(path, np.int32)
    qkv = _c(qkv, np.uint16)
    alpha = _c(alpha, np.float32)
    beta = _c(beta, np.float32)
    st = _c(state, np.float64).copy()
    xt = None if x_tree is None else _c(x_tree, np.uint16)
    tl = None if tail is None else _c(tail, np.uint16).copy()
    W = CONV_W if tl is None else tl.shape[0]
    _load().orc_commit(len(parents), Hk, Hv, dk, dv, _ptr(parents), _ptr(path) if path.size else None,
                       int(path.size), _ptr(qkv), _ptr(alpha), _ptr(beta), _ptr(xt), W, _ptr(st),
                       _ptr(tl), int(bool(normalize)))
    return st, tl


def prefill(qkv, alpha, beta, state, Hk, Hv, dk, dv, q_scale=1.0, normalize=True):
    """Chunked prefill's definition: the plain sequential recurrence over all T
    tokens of one sequence (the chunk form is an exact reorganisation of it)."""
    return decode(qkv, alpha, beta, state, Hk, Hv, dk, dv, q_scale, normalize)


# --------------------------------------------------------------------------
# KDA variant (a decay per key channel)
# --------------------------------------------------------------------------
def kda_token(S, k, v, q, alpha, beta, matrix_form=False):
    """One KDA token, one head: alpha is a vector of dk decays.  Returns (S_new, o)."""
    S = _c(S, np.float64).copy()
    k, v, q, a = (_c(x, np.float64) for x in (k, v, q, alpha))
    dv, dk = S.shape
    o = np.empty(dv, np.float64)
    fn = _load().orc_kda_token_matrix if matrix_form else _load().orc_kda_token
    fn(dk, dv, _ptr(S), _ptr(k), _ptr(v), _ptr(q), _ptr(a), float(beta), _ptr(o))
    return S, o


def kda_decode(qkv, alpha, beta, state, Hk, Hv, dk, dv, q_scale=1.0, normalize=True):
    """qkv bf16 [B,T,C], alpha f32 [B,T,Hv,dk], beta f32 [B,T,Hv], state [B,Hv,dv,dk]."""
    qkv = _c(qkv, np.uint16)
    alpha = _c(alpha, np.float32)
    beta = _c(beta, np.float32)
    st = _c(state, np.float64).copy()
    B, T = qkv.shape[0], qkv.shape[1]
    assert alpha.shape == (B, T, Hv, dk)
    out = np.empty((B, T, Hv, dv), np.float64)
    _load().orc_kda_decode(B, T, Hk, Hv, dk, dv, _ptr(qkv), _ptr(alpha), _ptr(beta), _ptr(st), _ptr(out),
                           float(q_scale), int(bool(normalize)))
    return out, st


# --------------------------------------------------------------------------
# state snapshot / restore
# --------------------------------------------------------------------------
def fnv1a64(data: bytes) -> int:
    buf = np.frombuffer(bytes(data), np.uint8).copy() if len(data) else np.zeros(1, np.uint8)
    return int(_load().orc_fnv1a64(_ptr(buf), len(data)))


def mix64(z: int) -> int:
    return int(_load().orc_mix64(ctypes.c_uint64(z & 0xFFFFFFFFFFFFFFFF)))


def snapshot_checksum(payload) -> int:
    payload = np.ascontiguousarray(np.frombuffer(bytes(payload), np.uint8) if isinstance(payload, (bytes, bytearray))
                                   else payload).view(np.uint8)
    return int(_load().orc_snapshot_checksum(_ptr(payload), payload.size))


def snapshot_signature(layers, Hk, Hv, dk, dv) -> int:
    return int(_load().orc_snapshot_signature(layers, Hk, Hv, dk, dv))


def snapshot_bytes(layers, Hk, Hv, dk, dv) -> int:
    return int(_load().orc_snapshot_bytes(layers, Hk, Hv, dk, dv))


def snapshot_save(state, tail, seq, Hk, Hv, dk, dv) -> np.ndarray:
    """state fp32 [L,B,Hv,dv,dk], tail bf16 bits [L,B,4,C]: the blob of sequence seq (uint8)."""
    state = _c(state, np.float32)
    tail = _c(tail, np.uint16)
    L, B = state.shape[0], state.shape[1]
    blob = np.zeros(snapshot_bytes(L, Hk, Hv, dk, dv), np.uint8)
    _load().orc_snapshot_save(L, B, Hk, Hv, dk, dv, int(seq), _ptr(state), _ptr(tail), _ptr(blob))
    return blob


def snapshot_restore(blob, state, tail, seq, Hk, Hv, dk, dv):
    """Restore sequence seq in copies of state/tail; returns (rc, state, tail)."""
    blob = np.ascontiguousarray(blob, np.uint8)
    st = _c(state, np.float32).copy()
    tl = _c(tail, np.uint16).copy()
    rc = _load().orc_snapshot_restore(st.shape[0], st.shape[1], Hk, Hv, dk, dv, int(seq), _ptr(blob), _ptr(st),
                                      _ptr(tl))
    return int(rc), st, tl


# --------------------------------------------------------------------------
# gate front end and gated-norm output
# --------------------------------------------------------------------------
def softplus(x: float) -> float:
    return float(_load().orc_softplus(float(x)))


def sigmoid(x: float) -> float:
    return float(_load().orc_sigmoid(float(x)))


def gates_from_projections(a, b, A_log, dt_bias):
    """a, b bf16 bits [..., Hv]; A_log, dt_bias fp32 [Hv] -> (alpha, beta) fp64 [..., Hv]."""
    a = _c(a, np.uint16)
    b = _c(b, np.uint16)
    Hv = a.shape[-1]
    n = a.size // Hv
    al = np.empty(a.shape, np.float64)
    be = np.empty(a.shape, np.float64)
    _load().orc_gates(n, Hv, _ptr(a), _ptr(b), _ptr(_c(A_log, np.float32)), _ptr(_c(dt_bias, np.float32)),
                      _ptr(al), _ptr(be))
    return al, be


def gated_rmsnorm(o, z, w, eps=1e-6):
    """o fp64 [dv], z bf16 bits [dv], w fp32 [dv] -> y fp64 [dv]."""
    o = _c(o, np.float64)
    y = np.empty(o.size, np.float64)
    _load().orc_gated_rmsnorm(o.size, _ptr(o), _ptr(_c(z, np.uint16)), _ptr(_c(w, np.float32)), float(eps),
                              _ptr(y))
    return y


def layer_decode(x, conv_w, tail, a, b, A_log, dt_bias, z, norm_w, state, Hk, Hv, dk, dv, eps=1e-6,
                 q_scale=1.0, normalize=True):
    """The layer's decode step.  Returns (o, y, state, tail); inputs are not modified."""
    x = _c(x, np.uint16)
    B, T, C = x.shape
    tl = _c(tail, np.uint16).copy()
    st = _c(state, np.float64).copy()
    o = np.empty((B, T, Hv, dv), np.float64)
    y = np.empty((B, T, Hv, dv), np.float64)
    _load().orc_layer_decode(B, T, Hk, Hv, dk, dv, _ptr(x), _ptr(_c(conv_w, np.uint16)), _ptr(tl),
                             _ptr(_c(a, np.uint16)), _ptr(_c(b, np.uint16)), _ptr(_c(A_log, np.float32)),
                             _ptr(_c(dt_bias, np.float32)), _ptr(_c(z, np.uint16)), _ptr(_c(norm_w, np.float32)),
                             float(eps), _ptr(st), _ptr(o), _ptr(y), float(q_scale), int(bool(normalize)))
    return o, y, st, tl
