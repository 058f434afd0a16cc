// gdn_snapshot.cu -- bit-exact snapshot and restore of one sequence's
// recurrent sections (fp32 delta-rule state + bf16 conv tail of every layer).
//
// A serving cache restores a sequence's state exactly: the recurrent state has
// absorbed every token and has no inverse, so it is restored, not recomputed
// (TandemLLM "Architecture" v0.14.2, section 8.1), and a signature over the
// sections' names, shapes and dtypes refuses a restore across models (same
// page, "ModelState: sections and views").
//
// GB300 design: the blob is written (or read) by the kernels themselves, so its
// home can be device memory or pinned host memory mapped into the device's
// address space (on Grace-Blackwell the NVLink-C2C link carries it); no staging
// copy is made.  Save is one gather pass that also accumulates the checksum;
// its last CTA writes the header.  Restore is a verify pass (header fields and
// checksum) and a scatter pass that writes nothing unless the verify passed,
// so a corrupted or foreign blob leaves the state untouched.  All passes are
// HBM- (or link-) bound streaming copies: 16-byte vectors, four in flight per
// thread, a grid of 8 CTAs per SM, streaming cache hints.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kSnapThreads = 256;
constexpr int kSnapUnroll = 4;
constexpr size_t kHeaderBytes = 64;

struct SnapParams {
    const uint8_t* state;     // layer 0's state of the sequence (bytes)
    const uint8_t* tail;      // layer 0's tail of the sequence
    uint8_t* state_w;         // the same, writable (restore)
    uint8_t* tail_w;
    int64_t state_stride;     // bytes between layers
    int64_t tail_stride;
    const uint8_t* blob_in;   // restore: the blob (header + payload)
    uint8_t* blob_out;        // save: the blob
    uint64_t sb16, tb16;      // 16-byte vectors per layer: state, tail
    uint64_t n16;             // payload vectors in all
    unsigned long long* acc;  // checksum accumulator (workspace + 8)
    int* status;              // workspace + 0
    unsigned int* done;       // CTAs finished (workspace + 16)
    uint64_t header[6];       // expected header words 0..5 (magic .. payload bytes)
};

// SplitMix64's output function (Steele, Lea & Flood 2014).
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

// SplitMix64's increment (the golden-ratio gamma).
constexpr uint64_t kGamma = 0x9e3779b97f4a7c15ULL;

// Checksum terms of one 16-byte vector: its 64-bit words j = 2v and 2v + 1,
// each keyed by adding (j + 1) gamma before mixing.
__device__ __forceinline__ uint64_t vec_terms(uint4 x, uint64_t v) {
    const uint64_t key = (2 * v + 1) * kGamma;
    const uint64_t d0 = (uint64_t)x.x | ((uint64_t)x.y << 32);
    const uint64_t d1 = (uint64_t)x.z | ((uint64_t)x.w << 32);
    return mix64(d0 + key) + mix64(d1 + key + kGamma);
}

// Byte offset, in the state/tail arrays, of payload vector v.
__device__ __forceinline__ const uint8_t* src_of(const SnapParams& p, uint64_t v) {
    const uint64_t per = p.sb16 + p.tb16;
    const uint64_t l = v / per, r = v % per;
    return r < p.sb16 ? p.state + (int64_t)l * p.state_stride + r * 16
                      : p.tail + (int64_t)l * p.tail_stride + (r - p.sb16) * 16;
}
__device__ __forceinline__ uint8_t* dst_of(const SnapParams& p, uint64_t v) {
    const uint64_t per = p.sb16 + p.tb16;
    const uint64_t l = v / per, r = v % per;
    return r < p.sb16 ? p.state_w + (int64_t)l * p.state_stride + r * 16
                      : p.tail_w + (int64_t)l * p.tail_stride + (r - p.sb16) * 16;
}

__device__ __forceinline__ void add_block_sum(uint64_t sum, unsigned long long* acc) {
    __shared__ uint64_t warp_sum[kSnapThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint64_t s = 0;
        for (int w = 0; w < kSnapThreads / 32; ++w) s += warp_sum[w];
        atomicAdd(acc, (unsigned long long)s);  // wraps modulo 2^64
    }
}

// Save: gather the payload into the blob and sum its checksum terms; the last
// CTA to finish writes the header with the complete sum.
__global__ void __launch_bounds__(kSnapThreads) gdn_snapshot_gather_kernel(const __grid_constant__ SnapParams p) {
    uint64_t sum = 0;
    const uint64_t stride = (uint64_t)gridDim.x * kSnapThreads;
    uint8_t* out = p.blob_out + kHeaderBytes;
    for (uint64_t v0 = (uint64_t)blockIdx.x * kSnapThreads + threadIdx.x; v0 < p.n16; v0 += stride * kSnapUnroll) {
        uint4 x[kSnapUnroll];
#pragma unroll
        for (int u = 0; u < kSnapUnroll; ++u) {
            const uint64_t v = v0 + u * stride;
            if (v < p.n16) x[u] = __ldcs(reinterpret_cast<const uint4*>(src_of(p, v)));
        }
#pragma unroll
        for (int u = 0; u < kSnapUnroll; ++u) {
            const uint64_t v = v0 + u * stride;
            if (v < p.n16) {
                __stcs(reinterpret_cast<uint4*>(out + v * 16), x[u]);
                sum += vec_terms(x[u], v);
            }
        }
    }
    add_block_sum(sum, p.acc);
    if (threadIdx.x == 0) {
        __threadfence();  // this CTA's sum is visible before it counts itself done
        if (atomicAdd(p.done, 1u) == gridDim.x - 1) {
            __threadfence();
            const unsigned long long total = atomicAdd(p.acc, 0ull);  // every CTA's sum is in
            uint64_t* h = reinterpret_cast<uint64_t*>(p.blob_out);
            for (int i = 0; i < 6; ++i) h[i] = p.header[i];
            h[6] = total;
            h[7] = 0;
        }
    }
}

// Restore, pass 1: check the header against the expected one and sum the
// payload's checksum terms.
__global__ void __launch_bounds__(kSnapThreads) gdn_snapshot_verify_kernel(const __grid_constant__ SnapParams p) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const uint64_t* h = reinterpret_cast<const uint64_t*>(p.blob_in);
        bool ok = true;
        for (int i = 0; i < 6; ++i) ok = ok && (h[i] == p.header[i]);
        if (!ok) atomicOr(p.status, 1);
    }
    uint64_t sum = 0;
    const uint64_t stride = (uint64_t)gridDim.x * kSnapThreads;
    const uint8_t* in = p.blob_in + kHeaderBytes;
    for (uint64_t v0 = (uint64_t)blockIdx.x * kSnapThreads + threadIdx.x; v0 < p.n16; v0 += stride * kSnapUnroll) {
        uint4 x[kSnapUnroll];
#pragma unroll
        for (int u = 0; u < kSnapUnroll; ++u) {
            const uint64_t v = v0 + u * stride;
            if (v < p.n16) x[u] = __ldcs(reinterpret_cast<const uint4*>(in + v * 16));
        }
#pragma unroll
        for (int u = 0; u < kSnapUnroll; ++u) {
            const uint64_t v = v0 + u * stride;
            if (v < p.n16) sum += vec_terms(x[u], v);
        }
    }
    add_block_sum(sum, p.acc);
}

// Restore, pass 2: scatter the payload, only if pass 1 found the header equal
// to the expected one and the checksum equal to the stored one.
__global__ void __launch_bounds__(kSnapThreads) gdn_snapshot_scatter_kernel(const __grid_constant__ SnapParams p) {
    const uint64_t stored = reinterpret_cast<const uint64_t*>(p.blob_in)[6];
    const bool header_bad = *p.status != 0;
    const bool sum_bad = *p.acc != stored;
    if (header_bad || sum_bad) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && !header_bad) atomicOr(p.status, 2);
        return;
    }
    const uint64_t stride = (uint64_t)gridDim.x * kSnapThreads;
    const uint8_t* in = p.blob_in + kHeaderBytes;
    for (uint64_t v0 = (uint64_t)blockIdx.x * kSnapThreads + threadIdx.x; v0 < p.n16; v0 += stride * kSnapUnroll) {
        uint4 x[kSnapUnroll];
#pragma unroll
        for (int u = 0; u < kSnapUnroll; ++u) {
            const uint64_t v = v0 + u * stride;
            if (v < p.n16) x[u] = __ldcs(reinterpret_cast<const uint4*>(in + v * 16));
        }
#pragma unroll
        for (int u = 0; u < kSnapUnroll; ++u) {
            const uint64_t v = v0 + u * stride;
            if (v < p.n16) __stcs(reinterpret_cast<uint4*>(dst_of(p, v)), x[u]);
        }
    }
}

// FNV-1a 64 (Fowler, Noll, Vo) of a byte string.
uint64_t fnv1a64(const char* s, size_t n) {
    uint64_t h = 0xcbf29ce484222325ULL;
    for (size_t i = 0; i < n; ++i) {
        h ^= (uint8_t)s[i];
        h *= 0x100000001b3ULL;
    }
    return h;
}

int channels_of(const gdn_shape* s) { return 2 * s->Hk * s->dk + s->Hv * s->dv; }

uint64_t signature_of(const gdn_shape* s, int layers) {
    char text[256];
    const int n = snprintf(text, sizeof text, "gdn-snapshot/1;layers=%d;state:f32[%d,%d,%d];tail:bf16[4,%d]",
                           layers, s->Hv, s->dv, s->dk, channels_of(s));
    return fnv1a64(text, (size_t)n);
}

// Header words 0..5: magic, version | layers, Hk | Hv, dk | dv, signature, payload bytes.
void header_words(const gdn_shape* s, int layers, uint64_t payload, uint64_t (&h)[6]) {
    uint64_t magic = 0;
    memcpy(&magic, "GDNSNAP1", 8);  // little-endian on every supported host
    h[0] = magic;
    h[1] = 1ULL | ((uint64_t)(uint32_t)layers << 32);
    h[2] = (uint64_t)(uint32_t)s->Hk | ((uint64_t)(uint32_t)s->Hv << 32);
    h[3] = (uint64_t)(uint32_t)s->dk | ((uint64_t)(uint32_t)s->dv << 32);
    h[4] = signature_of(s, layers);
    h[5] = payload;
}

uint64_t state_seq_bytes(const gdn_shape* s) { return (uint64_t)s->Hv * s->dv * s->dk * 4; }
uint64_t tail_seq_bytes(const gdn_shape* s) { return (uint64_t)4 * channels_of(s) * 2; }

// Refuse blob memory the device cannot reach (pageable host memory).
int check_device_reachable(const void* ptr, const char* name) {
    cudaPointerAttributes a{};
    cudaError_t e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return report_error(GDN_ERR_INVALID_ARG, "%s: cannot query the pointer (%s)", name, cudaGetErrorString(e));
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return GDN_OK;
    if (a.type == cudaMemoryTypeHost && a.devicePointer == ptr) return GDN_OK;
    return report_error(GDN_ERR_INVALID_ARG,
                        "%s (%p) is not device-accessible memory: use device memory or pinned, mapped host memory",
                        name, ptr);
}

int snap_grid() { return 8 * device_sm_count(); }

// Validation shared by save and restore.  Fills the parameters common to both.
int prepare(const gdn_shape* shape, int32_t layers, int32_t seq, const void* state, int64_t state_layer_stride,
            const void* tail, int64_t tail_layer_stride, const void* blob, size_t blob_bytes, void* workspace,
            size_t workspace_bytes, SnapParams& p) {
    int rc;
    if ((rc = check_shape_arg(shape, false)) != GDN_OK) return rc;
    if (layers < 1) return report_error(GDN_ERR_INVALID_ARG, "layers=%d < 1", layers);
    if (shape->B < 1) return report_error(GDN_ERR_INVALID_ARG, "B=%d: the arrays hold no sequence", shape->B);
    if (seq < 0 || seq >= shape->B)
        return report_error(GDN_ERR_INVALID_ARG, "seq=%d outside [0, B=%d)", seq, shape->B);
    const uint64_t sb = state_seq_bytes(shape), tb = tail_seq_bytes(shape);
    const int64_t s_elems = (int64_t)shape->B * shape->Hv * shape->dv * shape->dk;
    const int64_t t_elems = (int64_t)shape->B * 4 * channels_of(shape);
    if (layers > 1 && (state_layer_stride < s_elems || tail_layer_stride < t_elems))
        return report_error(GDN_ERR_INVALID_ARG,
                            "layer strides (%lld, %lld elements) smaller than one layer's arrays (%lld, %lld)",
                            (long long)state_layer_stride, (long long)tail_layer_stride, (long long)s_elems,
                            (long long)t_elems);
    if ((state_layer_stride * 4) % 16 != 0 || (tail_layer_stride * 2) % 16 != 0)
        return report_error(GDN_ERR_MISALIGNED, "layer strides must be multiples of 16 bytes");
    if ((rc = check_pointer(state, "state")) || (rc = check_pointer(tail, "tail")) ||
        (rc = check_pointer(blob, "blob")))
        return rc;
    const uint64_t payload = (uint64_t)layers * (sb + tb);
    if (blob_bytes < kHeaderBytes + payload)
        return report_error(GDN_ERR_INVALID_ARG, "blob of %zu bytes, the snapshot needs %llu", blob_bytes,
                            (unsigned long long)(kHeaderBytes + payload));
    if (workspace == nullptr) return report_error(GDN_ERR_WORKSPACE, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return report_error(GDN_ERR_MISALIGNED, "workspace (%p) is not 256-byte aligned", workspace);
    if (workspace_bytes < 256)
        return report_error(GDN_ERR_WORKSPACE, "workspace of %zu bytes, need 256", workspace_bytes);
    if ((rc = check_device_reachable(blob, "blob")) != GDN_OK) return rc;
    p = SnapParams{};
    const size_t sidx = (size_t)seq;
    p.state = static_cast<const uint8_t*>(state) + sidx * sb;
    p.tail = static_cast<const uint8_t*>(tail) + sidx * tb;
    p.state_stride = state_layer_stride * 4;
    p.tail_stride = tail_layer_stride * 2;
    p.sb16 = sb / 16;
    p.tb16 = tb / 16;
    p.n16 = payload / 16;
    p.status = static_cast<int*>(workspace);
    p.acc = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(workspace) + 8);
    p.done = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) + 16);
    header_words(shape, layers, payload, p.header);
    return GDN_OK;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

size_t gdn_snapshot_bytes(const gdn_shape* shape, int32_t layers) {
    if (check_shape_arg(shape, false) != GDN_OK || layers < 1) return 0;
    return kHeaderBytes + (size_t)layers * (state_seq_bytes(shape) + tail_seq_bytes(shape));
}

uint64_t gdn_snapshot_signature(const gdn_shape* shape, int32_t layers) {
    if (check_shape_arg(shape, false) != GDN_OK || layers < 1) return 0;
    return signature_of(shape, layers);
}

int gdn_snapshot_save(const gdn_shape* shape, int32_t layers, int32_t seq, const float* state,
                      int64_t state_layer_stride, const gdn_bf16* tail, int64_t tail_layer_stride, void* dst,
                      size_t dst_bytes, void* workspace, size_t workspace_bytes, void* stream) {
    SnapParams p;
    int rc = prepare(shape, layers, seq, state, state_layer_stride, tail, tail_layer_stride, dst, dst_bytes,
                     workspace, workspace_bytes, p);
    if (rc != GDN_OK) return rc;
    p.blob_out = static_cast<uint8_t*>(dst);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(workspace, 0, 24, st);
    if (e != cudaSuccess) return cuda_error(e, "snapshot workspace reset");
    gdn_snapshot_gather_kernel<<<snap_grid(), kSnapThreads, 0, st>>>(p);
    e = cudaGetLastError();
    return e == cudaSuccess ? GDN_OK : cuda_error(e, "snapshot launch");
}

int gdn_snapshot_restore(const gdn_shape* shape, int32_t layers, int32_t seq, const void* src, size_t src_bytes,
                         float* state, int64_t state_layer_stride, gdn_bf16* tail, int64_t tail_layer_stride,
                         void* workspace, size_t workspace_bytes, void* stream) {
    SnapParams p;
    int rc = prepare(shape, layers, seq, state, state_layer_stride, tail, tail_layer_stride, src, src_bytes,
                     workspace, workspace_bytes, p);
    if (rc != GDN_OK) return rc;
    p.blob_in = static_cast<const uint8_t*>(src);
    p.state_w = const_cast<uint8_t*>(p.state);
    p.tail_w = const_cast<uint8_t*>(p.tail);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(workspace, 0, 16, st);
    if (e != cudaSuccess) return cuda_error(e, "restore workspace reset");
    gdn_snapshot_verify_kernel<<<snap_grid(), kSnapThreads, 0, st>>>(p);
    gdn_snapshot_scatter_kernel<<<snap_grid(), kSnapThreads, 0, st>>>(p);
    e = cudaGetLastError();
    return e == cudaSuccess ? GDN_OK : cuda_error(e, "restore launch");
}

}  // extern "C"
