// gdn_prefill.cu -- chunked prefill entry points.
//
// This revision evaluates the recurrence for the whole prompt with the decode
// kernel: one launch, state in registers across all T tokens, read once and
// written once.  It is exact to the same rounding as decode.  The tensor-core
// WY/UT chunk form replaces it behind the same entry points.
#include <cuda_runtime.h>

#include "gdn_internal.h"

extern "C" {

size_t gdn_prefill_workspace_bytes(const gdn_shape* shape, int32_t T, int32_t chunk) {
    if (shape == nullptr || T < 0 || chunk != 64) return 0;
    return 256;
}

int gdn_chunk_prefill(const gdn_shape* shape, int32_t T, int32_t chunk, const gdn_bf16* qkv,
                      const float* alpha, const float* beta, float* state, void* out,
                      void* workspace, size_t workspace_bytes, float q_scale, uint32_t flags,
                      void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    if (shape == nullptr || shape->B != 1) {
        return gdn_decode_step(nullptr, 0, nullptr, nullptr, nullptr, nullptr, nullptr, 0.f, 0u,
                               nullptr);
    }
    if (chunk != 64) return GDN_ERR_INVALID_ARG;
    return gdn_decode_step(shape, T, qkv, alpha, beta, state, out, q_scale, flags, stream);
}

}  // extern "C"
