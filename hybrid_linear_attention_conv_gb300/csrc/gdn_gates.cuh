// gdn_gates.cuh -- the steps either side of the mixer in the Gated DeltaNet
// layer: the gate front end (decay and write strength from the token's
// projections) and the gated RMS-norm output.  The pages name the layer but
// print neither step; both follow the published Gated DeltaNet layer (Yang,
// Kautz & Hatamizadeh 2024, as shipped with the Qwen3-Next models):
//     alpha = exp(-exp(A_log[h]) * softplus(a + dt_bias[h])),  beta = sigmoid(b),
//     y_i   = o_i / sqrt(mean(o^2) + eps) * w_i * SiLU(z_i).
// One device function per step, shared by the standalone gates kernel and
// the fused layer step, so that both produce the same bits.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace gdn {

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// softplus(x) = log(1 + e^x), as max(x, 0) + log1p(e^-|x|) (no overflow).
__device__ __forceinline__ float softplus_f(float x) { return __fadd_rn(fmaxf(x, 0.0f), log1pf(expf(-fabsf(x)))); }

__device__ __forceinline__ void gate_pair(float a, float b, float A_log, float dt_bias, float& alpha, float& beta) {
    const float dt = softplus_f(__fadd_rn(a, dt_bias));
    alpha = expf(-__fmul_rn(expf(A_log), dt));
    beta = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-b)));
}

// w_i * SiLU(z_i) * o_i * inv_rms, rounded once per step as written.
__device__ __forceinline__ float gated_norm_out(float o, float inv_rms, float w, float z) {
    const float silu = __fdiv_rn(z, __fadd_rn(1.0f, expf(-z)));
    return __fmul_rn(__fmul_rn(__fmul_rn(o, inv_rms), w), silu);
}

}  // namespace gdn
