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
constexpr int kConvTok = 16;  // tokens per thread in a linear run

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
    const int gy = p.tree ? p.T : (p.T + kConvTok - 1) / kConvTok;
    dim3 grid((cvecs + kConvThreads - 1) / kConvThreads, gy, p.B);
    if (p.f32) gdn_conv_kernel<float><<<grid, kConvThreads, 0, s>>>(p);
    else gdn_conv_kernel<uint16_t><<<grid, kConvThreads, 0, s>>>(p);
    return cudaGetLastError();
}



}  // namespace gdn
