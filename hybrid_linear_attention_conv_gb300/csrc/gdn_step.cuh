// gdn_step.cuh -- the one per-row gated delta-rule step used by every kernel
// that advances a state token by token (decode, commit, tree verify).
//
// Because decode, commit and tree verify all call these functions with the
// same lane layout, a committed path's state equals a linear decode of that
// path bit for bit, and a tree node's output equals the decode output of the
// last token of its root path.  The speculative round needs exactly that
// (TandemLLM "Architecture" v0.11.1: a model whose verify rows equal its decode
// rows bit for bit can speculate with no change to its greedy text).  All
// floating-point operations use explicit round-to-nearest intrinsics so that no
// compiler contraction can differ between call sites.
//
// The row arithmetic runs on the packed fp32x2 pipe (fma.rn.f32x2 etc.), which
// rounds every element exactly as the scalar instruction would.
//
// Layout: a row of the state (dk fp32 values) is owned by a group of 8 lanes;
// lane l of the group holds float4 number m at columns 32*m + 4*l, for
// m = 0 .. dk/32 - 1.  A warp therefore covers 4 rows, and each load/store
// instruction of a warp touches 4 x 128 contiguous bytes.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace gdn {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr float kNormEps = 1e-6f;

// Sum over the 8 lanes of a row group (xor butterfly: every lane of the group
// ends with the same bits, since a + b == b + a exactly).
__device__ __forceinline__ float group_sum8(float x) {
    x = __fadd_rn(x, __shfl_xor_sync(kFullMask, x, 4));
    x = __fadd_rn(x, __shfl_xor_sync(kFullMask, x, 2));
    x = __fadd_rn(x, __shfl_xor_sync(kFullMask, x, 1));
    return x;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One activation as fp32: a bf16 bit pattern widened exactly, or an fp32 value.
__device__ __forceinline__ float act_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ float act_f(float f) { return f; }

// This lane's V*4 elements of a dk-long bf16 head vector.
template <int V>
__device__ __forceinline__ void load_head_vec(const uint16_t* head, int lane8, float (&x)[V][4]) {
#pragma unroll
    for (int m = 0; m < V; ++m) {
        const uint2 raw = *reinterpret_cast<const uint2*>(head + 32 * m + 4 * lane8);
        x[m][0] = bf16_lo(raw.x);
        x[m][1] = bf16_hi(raw.x);
        x[m][2] = bf16_lo(raw.y);
        x[m][3] = bf16_hi(raw.y);
    }
}

// The same for an fp32 head vector (the fp32-activation decode).
template <int V>
__device__ __forceinline__ void load_head_vec(const float* head, int lane8, float (&x)[V][4]) {
#pragma unroll
    for (int m = 0; m < V; ++m) {
        const float4 f = *reinterpret_cast<const float4*>(head + 32 * m + 4 * lane8);
        x[m][0] = f.x;
        x[m][1] = f.y;
        x[m][2] = f.z;
        x[m][3] = f.w;
    }
}

// Dot product of this lane's slice with another, reduced over the row group.
// Per float4 a short fma chain, then a fixed pairwise tree over the float4s.
template <int V>
__device__ __forceinline__ float lane_dot(const float (&a)[V][4], const float (&b)[V][4]) {
    float part[V];
#pragma unroll
    for (int m = 0; m < V; ++m) {
        float acc = __fmul_rn(a[m][0], b[m][0]);
        acc = __fmaf_rn(a[m][1], b[m][1], acc);
        acc = __fmaf_rn(a[m][2], b[m][2], acc);
        acc = __fmaf_rn(a[m][3], b[m][3], acc);
        part[m] = acc;
    }
#pragma unroll
    for (int w = 1; w < V; w *= 2)
#pragma unroll
        for (int m = 0; m + w < V; m += 2 * w) part[m] = __fadd_rn(part[m], part[m + w]);
    return group_sum8(part[0]);
}

// Dot product of this lane's slice of a state row with a vector slice, on the
// packed fp32x2 pipe: two float2 accumulators (even and odd float4s), each a
// short fma2 chain, then summed in a fixed order.
template <int V>
__device__ __forceinline__ float lane_dot4(const float4 (&s)[V], const float (&b)[V][4]) {
    float2 acc[2];
#pragma unroll
    for (int m = 0; m < V && m < 2; ++m) {
        acc[m] = __fmul2_rn(make_float2(s[m].x, s[m].y), make_float2(b[m][0], b[m][1]));
        acc[m] = __ffma2_rn(make_float2(s[m].z, s[m].w), make_float2(b[m][2], b[m][3]), acc[m]);
    }
#pragma unroll
    for (int m = 2; m < V; ++m) {
        acc[m & 1] = __ffma2_rn(make_float2(s[m].x, s[m].y), make_float2(b[m][0], b[m][1]), acc[m & 1]);
        acc[m & 1] = __ffma2_rn(make_float2(s[m].z, s[m].w), make_float2(b[m][2], b[m][3]), acc[m & 1]);
    }
    float2 t = acc[0];
    if (V > 1) t = __fadd2_rn(acc[0], acc[1]);
    return __fadd_rn(t.x, t.y);
}

// q^ = scale * q / sqrt(|q|^2 + eps) (or scale * q without normalisation).
template <int V>
__device__ __forceinline__ void normalize_vec(float (&x)[V][4], float scale, bool normalize) {
    float inv = scale;
    if (normalize) {
        const float ss = lane_dot<V>(x, x);
        inv = __fmul_rn(rsqrtf(__fadd_rn(ss, kNormEps)), scale);
    }
#pragma unroll
    for (int m = 0; m < V; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[m][e] = __fmul_rn(x[m][e], inv);
}

// Per-token key-head vectors of one row group: normalised q, k and k.q.
template <int V>
struct TokenKQ {
    float k[V][4];
    float q[V][4];
    float kq;
};

template <int V, typename In>
__device__ __forceinline__ void token_kq(const In* q_head, const In* k_head,
                                         int lane8, float q_scale, bool normalize,
                                         TokenKQ<V>& t) {
    load_head_vec<V>(k_head, lane8, t.k);
    load_head_vec<V>(q_head, lane8, t.q);
    normalize_vec<V>(t.k, 1.0f, normalize);
    normalize_vec<V>(t.q, q_scale, normalize);
    t.kq = lane_dot<V>(t.k, t.q);
}

// One token on one state row s (this lane's slice), in place:
//   a = s.k, c = s.q  (row-group sums),  u = beta * (v_i - alpha * a),
//   o_i = alpha * c + u * (k.q),         s <- alpha * s + u * k.
// This is row i of S <- alpha S (I - beta k k^T) + beta v k^T followed by
// o = S q (expand S_new q = alpha S q + u (k.q)).  Returns o_i in every lane.
template <int V>
__device__ __forceinline__ float row_step(float4 (&s)[V], const TokenKQ<V>& t, float v_i,
                                          float alpha, float beta) {
    const float a_part = lane_dot4<V>(s, t.k);
    const float c_part = lane_dot4<V>(s, t.q);
    const float a = group_sum8(a_part);
    const float c = group_sum8(c_part);
    const float u = __fmul_rn(beta, __fmaf_rn(-alpha, a, v_i));
    const float o = __fmaf_rn(alpha, c, __fmul_rn(u, t.kq));
    const float2 uu = make_float2(u, u), aa = make_float2(alpha, alpha);
#pragma unroll
    for (int m = 0; m < V; ++m) {
        const float2 lo = __ffma2_rn(uu, make_float2(t.k[m][0], t.k[m][1]), __fmul2_rn(aa, make_float2(s[m].x, s[m].y)));
        const float2 hi = __ffma2_rn(uu, make_float2(t.k[m][2], t.k[m][3]), __fmul2_rn(aa, make_float2(s[m].z, s[m].w)));
        s[m] = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    return o;
}

// KDA (Kimi Delta Attention) replaces the scalar decay by one per key channel:
// row i of S <- (S diag(g)) (I - beta k k^T) + beta v k^T, then o = S q.  The
// decay comes first, s' = g o s (kda_decay, applied to all of a thread's rows
// before their delta steps, so that the decay slice is live only briefly);
// then on s' (delta_row_step)
//   a = s'.k, c = s'.q,  u = beta * (v_i - a),  o_i = c + u * (k.q),
//   s <- s' + u * k.
// With g equal on every channel this is the same map as row_step; the
// rounding order differs (the decay is applied before the dot products).

// This lane's slice of a decay vector (dk fp32) staged in shared memory.
template <int V>
__device__ __forceinline__ void load_gate_smem(const float4* gate, int lane8, float4 (&g)[V]) {
#pragma unroll
    for (int m = 0; m < V; ++m) g[m] = gate[8 * m + lane8];
}

template <int V>
__device__ __forceinline__ void kda_decay(float4 (&s)[V], const float4 (&g)[V]) {
#pragma unroll
    for (int m = 0; m < V; ++m) {
        const float2 lo = __fmul2_rn(make_float2(g[m].x, g[m].y), make_float2(s[m].x, s[m].y));
        const float2 hi = __fmul2_rn(make_float2(g[m].z, g[m].w), make_float2(s[m].z, s[m].w));
        s[m] = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
}

template <int V>
__device__ __forceinline__ float delta_row_step(float4 (&s)[V], const TokenKQ<V>& t, float v_i, float beta) {
    const float a_part = lane_dot4<V>(s, t.k);
    const float c_part = lane_dot4<V>(s, t.q);
    const float a = group_sum8(a_part);
    const float c = group_sum8(c_part);
    const float u = __fmul_rn(beta, __fsub_rn(v_i, a));
    const float o = __fmaf_rn(u, t.kq, c);
    const float2 uu = make_float2(u, u);
#pragma unroll
    for (int m = 0; m < V; ++m) {
        const float2 lo = __ffma2_rn(uu, make_float2(t.k[m][0], t.k[m][1]), make_float2(s[m].x, s[m].y));
        const float2 hi = __ffma2_rn(uu, make_float2(t.k[m][2], t.k[m][3]), make_float2(s[m].z, s[m].w));
        s[m] = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    return o;
}

__device__ __forceinline__ void store_out(void* out, size_t idx, float o, bool as_bf16) {
    if (as_bf16) {
        reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(o);
    } else {
        reinterpret_cast<float*>(out)[idx] = o;
    }
}

}  // namespace gdn
