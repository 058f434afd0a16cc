// gdn_conv.cuh -- the per-channel arithmetic of the 4-tap causal conv + SiLU,
// shared by the standalone conv kernel and the fused conv + decode kernel so
// that both produce the same bf16 bits for the same inputs.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_step.cuh"

namespace gdn {

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

// 8 consecutive fp32 channels (the fp32-activation conv).
__device__ __forceinline__ Vec8 load8(const float* p) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    Vec8 r;
    r.v[0] = a.x;
    r.v[1] = a.y;
    r.v[2] = a.z;
    r.v[3] = a.w;
    r.v[4] = b.x;
    r.v[5] = b.y;
    r.v[6] = b.z;
    r.v[7] = b.w;
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

// 8 conv outputs rounded to bf16, packed as they are stored.
__device__ __forceinline__ uint4 conv8_bf16(const float (&w)[8][4], const Vec8& u0, const Vec8& u1, const Vec8& u2,
                                            const Vec8& u3) {
    float y[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) y[c] = conv_silu(w[c], u0.v[c], u1.v[c], u2.v[c], u3.v[c]);
    uint4 out;
    out.x = pack2(y[0], y[1]);
    out.y = pack2(y[2], y[3]);
    out.z = pack2(y[4], y[5]);
    out.w = pack2(y[6], y[7]);
    return out;
}

__device__ __forceinline__ void store_y(uint16_t* dst, const float (&w)[8][4], const Vec8& u0,
                                        const Vec8& u1, const Vec8& u2, const Vec8& u3) {
    *reinterpret_cast<uint4*>(dst) = conv8_bf16(w, u0, u1, u2, u3);
}

// The same 8 outputs kept in fp32 (the fp32-activation conv stores no bf16).
__device__ __forceinline__ void store_y(float* dst, const float (&w)[8][4], const Vec8& u0, const Vec8& u1,
                                        const Vec8& u2, const Vec8& u3) {
    float y[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) y[c] = conv_silu(w[c], u0.v[c], u1.v[c], u2.v[c], u3.v[c]);
    *reinterpret_cast<float4*>(dst) = make_float4(y[0], y[1], y[2], y[3]);
    *reinterpret_cast<float4*>(dst + 4) = make_float4(y[4], y[5], y[6], y[7]);
}

// Taps of 8 consecutive channels, fp32 [C][4].
__device__ __forceinline__ void load_taps8(const float* wp, float (&w)[8][4]) {
    const float4* w4 = reinterpret_cast<const float4*>(wp);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 t = w4[c];
        w[c][0] = t.x;
        w[c][1] = t.y;
        w[c][2] = t.z;
        w[c][3] = t.w;
    }
}

// Taps of 8 consecutive channels (w is [C][4] bf16, channel-major).
__device__ __forceinline__ void load_taps8(const uint16_t* wp, float (&w)[8][4]) {
    const uint4* w4 = reinterpret_cast<const uint4*>(wp);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 raw = w4[q];  // channels 2q, 2q+1
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

// Store 8 fp32 inputs as they are (the fp32-activation tail).
__device__ __forceinline__ void put8(float* dst, const Vec8& v) {
    *reinterpret_cast<float4*>(dst) = make_float4(v.v[0], v.v[1], v.v[2], v.v[3]);
    *reinterpret_cast<float4*>(dst + 4) = make_float4(v.v[4], v.v[5], v.v[6], v.v[7]);
}

// Store 8 values that are exact in bf16 (a window of inputs) as bf16.
__device__ __forceinline__ void put8(uint16_t* dst, const Vec8& v) {
    uint4 o;
    o.x = pack2(v.v[0], v.v[1]);
    o.y = pack2(v.v[2], v.v[3]);
    o.z = pack2(v.v[4], v.v[5]);
    o.w = pack2(v.v[6], v.v[7]);
    *reinterpret_cast<uint4*>(dst) = o;
}

}  // namespace gdn
