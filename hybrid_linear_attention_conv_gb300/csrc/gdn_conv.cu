// gdn_conv.cu -- 4-tap causal depthwise convolution + SiLU (sm_103a).
//
// The layer keeps, per sequence, the last four pre-conv inputs of every q/k/v
// channel (TandemLLM "Architecture" v0.14.2 section 8.1: a 4-wide convolution
// tail of 80 KB per layer = 4 x 10,240 channels x bf16).  Each thread owns 8
// consecutive channels (one 16-byte vector of bf16) of one sequence, so a warp
// reads and writes 512 contiguous bytes per token.  The per-channel arithmetic
// is identical in linear and tree mode (same order of the four products), so a
// tree node's conv output equals the linear conv of its root path bit for bit.
#include <cuda_runtime.h>

#include "gdn_conv.cuh"
#include "gdn_internal.h"

namespace gdn {

constexpr int kConvThreads = 128;
constexpr int kConvTok = 16;  // tokens per thread in a single-pass linear run

// Tokens per thread when a long linear run is split over blocks: every input
// of a thread's tokens is loaded before any is used, held as raw 16-byte
// words (11 loads of one word for bf16, of two for fp32).  A long run is
// bound by the SiLU's arithmetic (an IEEE divide and an accurate exp per
// output), not by its loads: on GB300 an 8,192-token prompt took 141 us with
// 8 tokens per thread, 155 us with 16 and 159 us with 4.
constexpr int kConvSplitTok = 8;

// 8 channels from their raw 16-byte words: one word of bf16, two of fp32.
__device__ __forceinline__ Vec8 vec8_of(const uint4 (&r)[1]) {
    Vec8 v;
    v.v[0] = bf16_lo(r[0].x);
    v.v[1] = bf16_hi(r[0].x);
    v.v[2] = bf16_lo(r[0].y);
    v.v[3] = bf16_hi(r[0].y);
    v.v[4] = bf16_lo(r[0].z);
    v.v[5] = bf16_hi(r[0].z);
    v.v[6] = bf16_lo(r[0].w);
    v.v[7] = bf16_hi(r[0].w);
    return v;
}

__device__ __forceinline__ Vec8 vec8_of(const uint4 (&r)[2]) {
    Vec8 v;
    v.v[0] = __uint_as_float(r[0].x);
    v.v[1] = __uint_as_float(r[0].y);
    v.v[2] = __uint_as_float(r[0].z);
    v.v[3] = __uint_as_float(r[0].w);
    v.v[4] = __uint_as_float(r[1].x);
    v.v[5] = __uint_as_float(r[1].y);
    v.v[6] = __uint_as_float(r[1].z);
    v.v[7] = __uint_as_float(r[1].w);
    return v;
}

// E is the element type of x, w, tail and y: uint16_t (bf16 bits; y rounded
// to bf16) or float (the fp32-activation conv; y kept in fp32).
template <typename E>
__global__ void __launch_bounds__(kConvThreads) gdn_conv_kernel(const __grid_constant__ ConvParams p) {
    const int cv = blockIdx.x * kConvThreads + threadIdx.x;
    const int c0 = cv * 8;
    if (c0 >= p.C) return;
    const int b = blockIdx.z;
    const size_t C = (size_t)p.C;
    const E* xb = static_cast<const E*>(p.x) + (size_t)b * p.T * C + c0;
    E* yb = static_cast<E*>(p.y) + (size_t)b * p.T * C + c0;
    E* tb = static_cast<E*>(p.tail) + (size_t)b * GDN_CONV_W * C + c0;

    float w[8][4];
    load_taps8(static_cast<const E*>(p.w) + (size_t)c0 * GDN_CONV_W, w);

    if (!p.tree && gridDim.y == 1) {
        // The whole run in one pass (T <= kConvTok, e.g. a decode step): a
        // window of the four most recent inputs starts as the tail, every
        // load is issued up front, and the new tail is the final window.
        // T >= 1 here (the API returns early on T == 0): tail[0] is shifted
        // out by the first token, so it is not read
        Vec8 h1 = load8(tb + C), h2 = load8(tb + 2 * C), h3 = load8(tb + 3 * C);
        Vec8 h0 = h1;
        Vec8 xn = load8(xb);
        for (int t = 0; t < p.T; ++t) {
            h0 = h1;
            h1 = h2;
            h2 = h3;
            h3 = xn;
            if (t + 1 < p.T) xn = load8(xb + (size_t)(t + 1) * C);
            store_y(yb + (size_t)t * C, w, h0, h1, h2, h3);
        }
        put8(tb, h0);
        put8(tb + C, h1);
        put8(tb + 2 * C, h2);
        put8(tb + 3 * C, h3);
    } else if (!p.tree) {
        // A block of TOK tokens: the three inputs before it (t < 0 reads tail
        // slot 4 + t) and its own, all requested before the first is used, so
        // that a thread waits for one DRAM round trip, not one per token.
        constexpr int TOK = kConvSplitTok;
        constexpr int W16 = (int)sizeof(E) / 2;  // 16-byte words per 8 channels
        const int t0 = blockIdx.y * TOK;
        const int n = min(p.T - t0, TOK);
        uint4 raw[3 + TOK][W16];
#pragma unroll
        for (int j = 0; j < 3 + TOK; ++j) {
            const int t = t0 - 3 + j;
            if (j < 3 + n) {
                const E* src = t >= 0 ? xb + (size_t)t * C : tb + (size_t)(GDN_CONV_W + t) * C;
#pragma unroll
                for (int q = 0; q < W16; ++q) raw[j][q] = reinterpret_cast<const uint4*>(src)[q];
            }
        }
        Vec8 u0 = vec8_of(raw[0]), u1 = vec8_of(raw[1]), u2 = vec8_of(raw[2]);
#pragma unroll
        for (int i = 0; i < TOK; ++i) {
            if (i < n) {
                const Vec8 u3 = vec8_of(raw[3 + i]);
                store_y(yb + (size_t)(t0 + i) * C, w, u0, u1, u2, u3);
                u0 = u1;
                u1 = u2;
                u2 = u3;
            }
        }
        if (blockIdx.y == 0) {
            // New tail = the last four of (tail ++ x).  Only this thread touches
            // these channels of the tail, and it has finished reading it.
            // (raw 16-byte words: the bytes are copied as they are)
            constexpr int W16 = (int)sizeof(E) / 2;  // 16-byte words per 8 channels
            uint4 nt[GDN_CONV_W][W16];
#pragma unroll
            for (int j = 0; j < GDN_CONV_W; ++j) {
                const int pos = p.T + j;  // index into tail ++ x
                const E* src = pos < GDN_CONV_W ? tb + (size_t)pos * C : xb + (size_t)(pos - GDN_CONV_W) * C;
#pragma unroll
                for (int q = 0; q < W16; ++q) nt[j][q] = reinterpret_cast<const uint4*>(src)[q];
            }
#pragma unroll
            for (int j = 0; j < GDN_CONV_W; ++j)
#pragma unroll
                for (int q = 0; q < W16; ++q) reinterpret_cast<uint4*>(tb + (size_t)j * C)[q] = nt[j][q];
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

cudaError_t launch_conv(const ConvParams& p, cudaStream_t s) {
    const int cvecs = p.C / 8;
    // a linear run of up to kConvTok tokens is one pass per thread; a longer
    // one is split into blocks of kConvSplitTok tokens along grid y
    const int gy = p.tree ? p.T : p.T <= kConvTok ? 1 : (p.T + kConvSplitTok - 1) / kConvSplitTok;
    dim3 grid((cvecs + kConvThreads - 1) / kConvThreads, gy, p.B);
    if (p.f32) gdn_conv_kernel<float><<<grid, kConvThreads, 0, s>>>(p);
    else gdn_conv_kernel<uint16_t><<<grid, kConvThreads, 0, s>>>(p);
    return cudaGetLastError();
}



}  // namespace gdn
