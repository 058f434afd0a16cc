"""Seeded synthetic inputs for the Gated DeltaNet mixer.

This module is shared by the tests, the benchmark and the CPU oracle's callers.
It holds only random-number generation and storage rounding -- none of the
mixer's arithmetic -- so that the CUDA path and the oracle see the same bytes
without sharing any code.

Generator (fixed so that "seed s" names one sequence of numbers):
  * splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014) over a counter: value i of a stream is
    mix64(base + (i + 1) * 0x9E3779B97F4A7C15), base = mix64(seed-and-stream key);
  * a 53-bit uniform in (0, 1): ((z >> 11) + 0.5) * 2^-53;
  * normals by Box-Muller on consecutive pairs (u1, u2):
    sqrt(-2 ln u1) * (cos 2 pi u2, sin 2 pi u2).
Values are produced in fp64 and rounded once to their storage type (fp32 by
numpy's round-to-nearest-even cast; bf16 by round-to-nearest-even on the fp32
bit pattern).

Distributions follow the mixer workloads: q, k, v and pre-conv inputs ~ N(0, 1);
alpha ~ U(0.9, 1.0); beta = sigmoid(N(0, 1)); initial state ~ N(0, 0.1^2);
conv taps ~ N(0, 0.5^2); draft trees of up to 32 nodes, branching 1-4, depth <= 8.
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

CONV_W = 4


@dataclass(frozen=True)
class Shape:
    """Head shape of one Gated DeltaNet layer, plus the batch of sequences."""

    B: int
    Hk: int
    Hv: int
    dk: int
    dv: int

    @property
    def C(self) -> int:
        """Channels of the packed [q | k | v] activation row."""
        return 2 * self.Hk * self.dk + self.Hv * self.dv

    def with_batch(self, B: int) -> "Shape":
        return Shape(B, self.Hk, self.Hv, self.dk, self.dv)


# 2 key heads / 4 value heads of 32: the small correctness case.
TINY = Shape(1, 2, 4, 32, 32)
# The 27B hybrid's Gated DeltaNet head shape: 16 key heads and 48 value heads of 128.
QWEN_27B = Shape(1, 16, 48, 128, 128)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _base(seed: int, stream: str) -> np.uint64:
    key = (int(seed) & 0xFFFFFFFF) << 32 | zlib.crc32(stream.encode())
    return _mix64(np.array([key], np.uint64))[0]


def uniform(seed: int, stream: str, n: int) -> np.ndarray:
    """n fp64 uniforms in (0, 1) from stream `stream` of seed `seed`."""
    base = _base(seed, stream)
    out = np.empty(n, np.float64)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        ctr = np.arange(s + 1, e + 1, dtype=np.uint64)
        z = _mix64(base + ctr * _GOLDEN)
        out[s:e] = ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)
    return out


def normal(seed: int, stream: str, n: int) -> np.ndarray:
    """n fp64 standard normals (Box-Muller over consecutive uniform pairs)."""
    m = (n + 1) // 2
    u = uniform(seed, stream, 2 * m)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * m, np.float64)
    out[0::2] = r * np.cos(2.0 * np.pi * u2)
    out[1::2] = r * np.sin(2.0 * np.pi * u2)
    return out[:n]


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return the raw bits."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & np.uint64(0x7FFFFFFF)) > np.uint64(0x7F800000)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(h) -> np.ndarray:
    """Widen raw bf16 bits to fp32 (exact)."""
    return (np.ascontiguousarray(h, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, stream: str, shape, scale: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return f32_to_bf16_bits((scale * normal(seed, stream, n)).astype(np.float32)).reshape(shape)


def normal_f32(seed: int, stream: str, shape, scale: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return (scale * normal(seed, stream, n)).astype(np.float32).reshape(shape)


def gates(seed: int, stream: str, shape):
    """(alpha, beta) fp32: alpha ~ U(0.9, 1.0), beta = sigmoid(N(0, 1))."""
    n = int(np.prod(shape))
    alpha = (0.9 + 0.1 * uniform(seed, stream + ".alpha", n)).astype(np.float32).reshape(shape)
    z = normal(seed, stream + ".beta", n)
    beta = (1.0 / (1.0 + np.exp(-z))).astype(np.float32).reshape(shape)
    return alpha, beta


def decode_inputs(seed: int, shape: Shape, T: int, tag: str = "decode") -> dict:
    """Packed bf16 qkv [B,T,C], fp32 alpha/beta [B,T,Hv], fp32 state [B,Hv,dv,dk]."""
    B = shape.B
    qkv = normal_bf16(seed, tag + ".qkv", (B, T, shape.C))
    alpha, beta = gates(seed, tag, (B, T, shape.Hv))
    state = normal_f32(seed, tag + ".state", (B, shape.Hv, shape.dv, shape.dk), 0.1)
    return {"qkv": qkv, "alpha": alpha, "beta": beta, "state": state}


def conv_inputs(seed: int, B: int, T: int, C: int, tag: str = "conv", zero_tail: bool = False) -> dict:
    """Pre-conv x bf16 [B,T,C], taps w bf16 [C,4], tail bf16 [B,4,C]."""
    x = normal_bf16(seed, tag + ".x", (B, T, C))
    w = normal_bf16(seed, tag + ".w", (C, CONV_W), 0.5)
    if zero_tail:
        tail = np.zeros((B, CONV_W, C), np.uint16)
    else:
        tail = normal_bf16(seed, tag + ".tail", (B, CONV_W, C))
    return {"x": x, "w": w, "tail": tail}


def decode_inputs_f32(seed: int, shape: Shape, T: int, tag: str = "decode_f32") -> dict:
    """As decode_inputs, with the packed activations qkv [B,T,C] drawn and kept
    in fp32 (~N(0, 1), never rounded to bf16)."""
    d = decode_inputs(seed, shape, T, tag=tag)
    d["qkv"] = normal_f32(seed, tag + ".qkv32", (shape.B, T, shape.C))
    return d


def conv_inputs_f32(seed: int, B: int, T: int, C: int, tag: str = "conv_f32", zero_tail: bool = True) -> dict:
    """Pre-conv x fp32 [B,T,C] ~ N(0, 1), taps w fp32 [C,4] ~ N(0, 0.5^2), tail
    fp32 [B,4,C] (zeros: the start of a sequence, unless zero_tail is False)."""
    x = normal_f32(seed, tag + ".x", (B, T, C))
    w = normal_f32(seed, tag + ".w", (C, CONV_W), 0.5)
    tail = np.zeros((B, CONV_W, C), np.float32) if zero_tail else normal_f32(seed, tag + ".tail", (B, CONV_W, C))
    return {"x": x, "w": w, "tail": tail}


def random_tree(seed: int, N: int = 32, max_depth: int = 8, branch=(1, 4)) -> np.ndarray:
    """Draft-tree parent array: node 0 is the root (parent -1); nodes are added
    in breadth-first order, each visited node drawing U{branch} children, never
    past `max_depth` (root depth 1).  If the frontier empties first, the
    shallow nodes are visited again in index order."""
    lo, hi = branch
    draws = uniform(seed, "tree", 4 * N + 64)
    di = 0
    parents = [-1]
    depth = [1]
    order = [0]
    pos = 0
    while len(parents) < N:
        if pos >= len(order):
            order.extend(i for i in range(len(parents)) if depth[i] < max_depth)
            if pos >= len(order):
                break
        node = order[pos]
        pos += 1
        if depth[node] >= max_depth:
            continue
        if di >= len(draws):
            draws = np.concatenate([draws, uniform(seed, f"tree.{di}", 4 * N)])
        kids = lo + int(draws[di] * (hi - lo + 1))
        di += 1
        for _ in range(kids):
            if len(parents) >= N:
                break
            parents.append(node)
            depth.append(depth[node] + 1)
            order.append(len(parents) - 1)
    return np.array(parents, np.int32)


def random_leaf(seed: int, parents) -> int:
    """A uniformly chosen leaf (node with no children) of the tree."""
    parents = np.asarray(parents)
    has_child = np.zeros(len(parents), bool)
    has_child[parents[parents >= 0]] = True
    leaves = np.nonzero(~has_child)[0]
    u = uniform(seed, "leaf", 1)[0]
    return int(leaves[min(int(u * len(leaves)), len(leaves) - 1)])


def kda_inputs(seed: int, shape: Shape, T: int, tag: str = "kda") -> dict:
    """As decode_inputs, with alpha fp32 [B,T,Hv,dk]: one decay per key channel,
    each ~ U(0.9, 1.0)."""
    d = decode_inputs(seed, shape, T, tag=tag)
    n = shape.B * T * shape.Hv * shape.dk
    d["alpha"] = (0.9 + 0.1 * uniform(seed, tag + ".alpha_vec", n)).astype(np.float32).reshape(
        shape.B, T, shape.Hv, shape.dk)
    return d


def layer_inputs(seed: int, shape: Shape, T: int, tag: str = "layer") -> dict:
    """Inputs of the layer's decode step around the mixer: pre-conv x, taps and
    tail (as conv_inputs), the gate projections a, b bf16 [B,T,Hv] ~ N(0, 1),
    the per-head parameters A_log = log(U(1, 16)) and dt_bias = the inverse
    softplus of dt, log-uniform in [1e-3, 1e-1] (the published initialisation),
    the output-gate projection z bf16 [B,T,Hv,dv] ~ N(0, 1), the norm weight
    w fp32 [dv] ~ N(1, 0.1^2) and the fp32 state [B,Hv,dv,dk] ~ N(0, 0.1^2)."""
    B, Hv, dv = shape.B, shape.Hv, shape.dv
    d = conv_inputs(seed, B, T, shape.C, tag=tag + ".conv")
    d["a"] = normal_bf16(seed, tag + ".a", (B, T, Hv))
    d["b"] = normal_bf16(seed, tag + ".b", (B, T, Hv))
    d["A_log"] = np.log(1.0 + 15.0 * uniform(seed, tag + ".A", Hv)).astype(np.float32)
    dt = np.exp(np.log(1e-3) + (np.log(1e-1) - np.log(1e-3)) * uniform(seed, tag + ".dt", Hv))
    d["dt_bias"] = (dt + np.log(-np.expm1(-dt))).astype(np.float32)
    d["z"] = normal_bf16(seed, tag + ".z", (B, T, Hv, dv))
    d["norm_w"] = (1.0 + 0.1 * normal(seed, tag + ".w", dv)).astype(np.float32)
    d["state"] = normal_f32(seed, tag + ".state", (B, Hv, dv, shape.dk), 0.1)
    return d
