// gdn_tc.cuh -- thin inline-PTX wrappers for the 5th-generation tensor cores
// (tcgen05) and mbarriers on sm_103a, used by the chunked-prefill kernel.
//
// Operand tiles live in shared memory in the K-major, non-swizzled canonical
// layout: "core matrices" of 8 rows x 16 bytes (8 bf16) stored contiguously
// (128 B); core matrices adjacent along K are 128 B apart (leading byte
// offset), groups of 8 rows are 16*Kd bytes apart (stride byte offset) for a
// tile with Kd columns.  One MMA instruction consumes K = 16 (two core
// matrices along K), so step ks of a tile starts 256 B further on.
// Accumulators live in tensor memory (TMEM): row m of an M = 128 tile is TMEM
// lane m, column n is TMEM column base + n (fp32).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace gdn {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of element (r, k) in a K-major tile with Kd columns.
__device__ __forceinline__ uint32_t core_off(int r, int k, int Kd) {
    return (uint32_t)((r >> 3) * (Kd * 16) + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// Shared-memory matrix descriptor: start address, leading byte offset 128,
// stride byte offset `sbo`, fixed version bits 46-48 = 0b001, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128u >> 4) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Shared-memory matrix descriptor of a K-major tile stored with the 128-byte
// swizzle (as a TMA load with that swizzle leaves it): rows of 128 B (64
// bf16), groups of 8 rows 1,024 B apart, layout type 2 in bits 61..63.  Step
// k of K = 16 inside a 64-wide slab starts 32 B further on.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;              // leading byte offset (unused with this swizzle)
    d |= (uint64_t)(1024u >> 4) << 32;   // stride byte offset
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// The same with A read from tensor memory: an M = 128 x K = 16 bf16 slice is
// 128 lanes x 8 columns starting at `a_tmem`, column c of a lane holding
// elements k = 2c (low 16 bits) and 2c + 1 (high 16 bits); the next K slice
// starts 8 columns on.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make generic-proxy shared-memory writes visible to the tensor cores.
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_saddr, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}
// 8 consecutive 32-bit columns of this thread's TMEM lane (raw words).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&w)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One bounded try: true once phase `parity` of `bar` has completed.  The
// thread may be suspended (up to the hint) until the phase completes, so
// waiting warps do not take issue slots from working ones.
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// One probe that never suspends the thread: true if phase `parity` of `bar`
// has already completed.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; give up after `limit_ns`.  The
// clock is read only once the first try has come back empty (reading it costs
// more than a try on a completed phase).  A limit of 0 gives up at once unless
// the phase has already completed (one probe, no suspension).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (limit_ns == 0) return mbar_test(bar, parity);
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// Split x into bf16 hi + lo with x ~= hi + lo (x - hi is exact in fp32).
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(__fsub_rn(x, __bfloat162float(hi)));
}

__device__ __forceinline__ uint32_t pack_bf16(__nv_bfloat16 a, __nv_bfloat16 b) {
    return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// Split a pair (a, b) into packed bf16 hi and lo words (a in the low 16
// bits): hi = RNE(x), lo = RNE(x - hi), where x - hi is exact in fp32 -- the
// same roundings as split_bf16, with paired conversions and one fp32x2 FMA.
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const uint32_t hw = *reinterpret_cast<const uint32_t*>(&h);
    const float2 r = __ffma2_rn(make_float2(__uint_as_float(hw << 16), __uint_as_float(hw & 0xffff0000u)),
                                make_float2(-1.0f, -1.0f), make_float2(a, b));
    const __nv_bfloat162 l = __floats2bfloat162_rn(r.x, r.y);
    hi = hw;
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Split 8 floats and store them as one 16-byte row segment of a hi and a lo tile.
__device__ __forceinline__ void store_split8(uint8_t* hi_dst, uint8_t* lo_dst, const float* x) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split_pair(x[2 * e], x[2 * e + 1], h[e], l[e]);
    *reinterpret_cast<uint4*>(hi_dst) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo_dst) = make_uint4(l[0], l[1], l[2], l[3]);
}

// Split 16 floats into bf16 hi and lo halves packed two per word (element
// 2e in the low 16 bits), the layout of an A operand slice in tensor memory.
__device__ __forceinline__ void split_pack16(const float (&x)[16], uint32_t (&hi)[8], uint32_t (&lo)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) split_pair(x[2 * e], x[2 * e + 1], hi[e], lo[e]);
}

// x[j] *= f[j] for 16 values on the fp32x2 pipe (each element rounded as the
// scalar multiply would be); f is 16 floats in shared memory, 16-byte aligned.
__device__ __forceinline__ void mul16(float (&x)[16], const float* f) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 m = reinterpret_cast<const float4*>(f)[q];
        const float2 a = __fmul2_rn(make_float2(x[4 * q], x[4 * q + 1]), make_float2(m.x, m.y));
        const float2 b = __fmul2_rn(make_float2(x[4 * q + 2], x[4 * q + 3]), make_float2(m.z, m.w));
        x[4 * q] = a.x;
        x[4 * q + 1] = a.y;
        x[4 * q + 2] = b.x;
        x[4 * q + 3] = b.y;
    }
}

// Arrive once on `bar` and announce `bytes` of copy-engine data that will
// complete on it (the phase completes when both have happened).
// One arrival on an mbarrier (release at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global to shared memory by the copy engine, counted on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Tiled TMA load of one box of a 2-D tensor map at element coordinates
// (x, y) into shared memory, counted on `bar`; rows past the tensor's end
// read as zeros.  x times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Order this thread's earlier generic-proxy view of global memory before its
// later copy-engine accesses (data another CTA published through a flag).
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Asynchronous 16-byte global -> shared copy; zero-fills when !valid.
__device__ __forceinline__ void cp_async16(uint32_t dst_saddr, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_saddr), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Transpose four 8x8 b16 matrices: lane l gives row (l & 7) of matrix (l >> 3)
// of the source (src) and of the destination (dst).
__device__ __forceinline__ void transpose_8x8x4(uint32_t src, uint32_t dst) {
    uint32_t r0, r1, r2, r3;
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(src));
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(r0), "r"(r1),
                 "r"(r2), "r"(r3)
                 : "memory");
}

}  // namespace tc
}  // namespace gdn
