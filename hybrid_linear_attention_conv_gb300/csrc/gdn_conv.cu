// gdn_conv.cu -- 4-tap causal depthwise convolution + SiLU, and the conv-tail
// update of a commit (sm_103a).
//
// The layer keeps, per sequence, the last four pre-conv inputs of every q/k/v
// channel (TandemLLM "Architecture" v0.14.2 section 8.1: a 4-wide convolution
// tail of 80 KB per layer = 4 x 10,240 channels x bf16).  Each thread owns 8
// consecutive channels (one 16-byte vector of bf16) of one sequence, so a warp
// reads and writes 512 contiguous bytes per token.  The per-channel arithmetic
// is identical in linear and tree mode (same order of the four products), so a
// tree node's conv output equals the linear conv of its root path bit for bit.
#include <cuda_runtime.h>

#include "gdn_internal.h"
#include "gdn_step.cuh"

namespace gdn {

constexpr int kConvThreads = 128;
constexpr int kConvTok = 16;  // tokens per thread in a linear run

struct Vec8 {
    float v[8];
};

__device__ __forceinline__ Vec8 load8(const uint16_t* p) {
    const uint4 raw = *reinterpret_cast<const uint4*>(p);
    Vec8 r;
    r.v[0] = bf16_lo(raw.x);
    r.v[1] = bf16_hi(raw.x);
    r.v[2] = bf16_lo(raw.y);
    r.v[3] = bf16_hi(raw.y);
    r.v[4] = bf16_lo(raw.z);
    r.v[5] = bf16_hi(raw.z);
    r.v[6] = bf16_lo(raw.w);
    r.v[7] = bf16_hi(raw.w);
    return r;
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
}

// y = SiLU(w0*u0 + w1*u1 + w2*u2 + w3*u3), u0 oldest, u3 newest.
__device__ __forceinline__ float conv_silu(const float (&w)[4], float u0, float u1, float u2,
                                           float u3) {
    float acc = __fmul_rn(w[0], u0);
    acc = __fmaf_rn(w[1], u1, acc);
    acc = __fmaf_rn(w[2], u2, acc);
    acc = __fmaf_rn(w[3], u3, acc);
    return __fdiv_rn(acc, __fadd_rn(1.0f, expf(-acc)));
}

__device__ __forceinline__ void store_y(uint16_t* dst, const float (&w)[8][4], const Vec8& u0,
                                        const Vec8& u1, const Vec8& u2, const Vec8& u3) {
    float y[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) y[c] = conv_silu(w[c], u0.v[c], u1.v[c], u2.v[c], u3.v[c]);
    uint4 out;
    out.x = pack2(y[0], y[1]);
    out.y = pack2(y[2], y[3]);
    out.z = pack2(y[4], y[5]);
    out.w = pack2(y[6], y[7]);
    *reinterpret_cast<uint4*>(dst) = out;
}

__global__ void __launch_bounds__(kConvThreads) gdn_conv_kernel(const __grid_constant__ ConvParams p) {
    const int cv = blockIdx.x * kConvThreads + threadIdx.x;
    const int c0 = cv * 8;
    if (c0 >= p.C) return;
    const int b = blockIdx.z;
    const size_t C = (size_t)p.C;
    const uint16_t* xb = p.x + (size_t)b * p.T * C + c0;
    uint16_t* yb = p.y + (size_t)b * p.T * C + c0;
    uint16_t* tb = p.tail + (size_t)b * GDN_CONV_W * C + c0;

    float w[8][4];
    {
        const uint4* wp = reinterpret_cast<const uint4*>(p.w + (size_t)c0 * GDN_CONV_W);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 raw = wp[q];  // channels c0+2q, c0+2q+1
            w[2 * q][0] = bf16_lo(raw.x);
            w[2 * q][1] = bf16_hi(raw.x);
            w[2 * q][2] = bf16_lo(raw.y);
            w[2 * q][3] = bf16_hi(raw.y);
            w[2 * q + 1][0] = bf16_lo(raw.z);
            w[2 * q + 1][1] = bf16_hi(raw.z);
            w[2 * q + 1][2] = bf16_lo(raw.w);
            w[2 * q + 1][3] = bf16_hi(raw.w);
        }
    }

    if (!p.tree && gridDim.y == 1) {
        // The whole run in one pass (T <= kConvTok, e.g. a decode step): a
        // window of the four most recent inputs starts as the tail, every
        // load is issued up front, and the new tail is the final window.
        Vec8 h0 = load8(tb), h1 = load8(tb + C), h2 = load8(tb + 2 * C), h3 = load8(tb + 3 * C);
        Vec8 xn = p.T > 0 ? load8(xb) : h3;
        for (int t = 0; t < p.T; ++t) {
            h0 = h1;
            h1 = h2;
            h2 = h3;
            h3 = xn;
            if (t + 1 < p.T) xn = load8(xb + (size_t)(t + 1) * C);
            store_y(yb + (size_t)t * C, w, h0, h1, h2, h3);
        }
        auto put = [&](uint16_t* dst, const Vec8& v) {
            uint4 o;
            o.x = pack2(v.v[0], v.v[1]);
            o.y = pack2(v.v[2], v.v[3]);
            o.z = pack2(v.v[4], v.v[5]);
            o.w = pack2(v.v[6], v.v[7]);
            *reinterpret_cast<uint4*>(dst) = o;
        };
        put(tb, h0);
        put(tb + C, h1);
        put(tb + 2 * C, h2);
        put(tb + 3 * C, h3);
    } else if (!p.tree) {
        // inputs before token t0: t < 0 reads tail slot 4 + t
        const int t0 = blockIdx.y * kConvTok;
        const int t1 = min(p.T, t0 + kConvTok);
        auto in = [&](int t) -> Vec8 {
            return t >= 0 ? load8(xb + (size_t)t * C) : load8(tb + (size_t)(GDN_CONV_W + t) * C);
        };
        Vec8 u0 = in(t0 - 3), u1 = in(t0 - 2), u2 = in(t0 - 1);
        for (int t = t0; t < t1; ++t) {
            const Vec8 u3 = load8(xb + (size_t)t * C);
            store_y(yb + (size_t)t * C, w, u0, u1, u2, u3);
            u0 = u1;
            u1 = u2;
            u2 = u3;
        }
        if (blockIdx.y == 0) {
            // New tail = the last four of (tail ++ x).  Only this thread touches
            // these channels of the tail, and it has finished reading it.
            uint4 nt[GDN_CONV_W];
#pragma unroll
            for (int j = 0; j < GDN_CONV_W; ++j) {
                const int pos = p.T + j;  // index into tail ++ x
                const uint16_t* src = pos < GDN_CONV_W ? tb + (size_t)pos * C
                                                       : xb + (size_t)(pos - GDN_CONV_W) * C;
                nt[j] = *reinterpret_cast<const uint4*>(src);
            }
#pragma unroll
            for (int j = 0; j < GDN_CONV_W; ++j) *reinterpret_cast<uint4*>(tb + (size_t)j * C) = nt[j];
        }
    } else {
        const int n = blockIdx.y;
        auto src = [&](int a) -> Vec8 {
            return a >= 0 ? load8(xb + (size_t)a * C) : load8(tb + (size_t)(-1 - a) * C);
        };
        const Vec8 u3 = load8(xb + (size_t)n * C);
        const Vec8 u2 = src(p.anc[n][0]);
        const Vec8 u1 = src(p.anc[n][1]);
        const Vec8 u0 = src(p.anc[n][2]);
        store_y(yb + (size_t)n * C, w, u0, u1, u2, u3);
    }
}

__global__ void __launch_bounds__(kConvThreads)
gdn_commit_tail_kernel(const __grid_constant__ TailParams p) {
    const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * 8;
    if (c0 >= p.C) return;
    const size_t C = (size_t)p.C;
    uint4 nt[GDN_CONV_W];
#pragma unroll
    for (int j = 0; j < GDN_CONV_W; ++j) {
        const int pos = p.L + j;  // index into tail ++ x_tree[path]
        const uint16_t* src = pos < GDN_CONV_W ? p.tail + (size_t)pos * C + c0
                                               : p.x_tree + (size_t)p.path[pos - GDN_CONV_W] * C + c0;
        nt[j] = *reinterpret_cast<const uint4*>(src);
    }
#pragma unroll
    for (int j = 0; j < GDN_CONV_W; ++j) *reinterpret_cast<uint4*>(p.tail + (size_t)j * C + c0) = nt[j];
}

cudaError_t launch_conv(const ConvParams& p, cudaStream_t s) {
    const int cvecs = p.C / 8;
    const int gy = p.tree ? p.T : (p.T + kConvTok - 1) / kConvTok;
    dim3 grid((cvecs + kConvThreads - 1) / kConvThreads, gy, p.B);
    gdn_conv_kernel<<<grid, kConvThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_commit_tail(const TailParams& p, cudaStream_t s) {
    const int cvecs = p.C / 8;
    dim3 grid((cvecs + kConvThreads - 1) / kConvThreads, 1, 1);
    gdn_commit_tail_kernel<<<grid, kConvThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
