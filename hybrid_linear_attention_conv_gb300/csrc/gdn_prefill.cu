// gdn_prefill.cu -- chunked prefill on the tcgen05 tensor cores (sm_103a).
//
// The prompt's T tokens are processed in chunks of 64 with the WY/UT chunk
// form of the gated delta rule (Yang et al. 2024, "Parallelizing Linear
// Transformers with the Delta Rule over Sequence Length"; gated extension in
// "Gated Delta Networks").  Per value head and chunk, with gamma_t the running
// product of alpha inside the chunk and r the L2-norm reciprocals:
//   L[t][s] = beta_t (gamma_t/gamma_s) r_k,t r_k,s (k_t . k_s)   (s < t)
//   T       = (I + L)^-1                                          (unit lower)
//   X       = diag(beta) (V - diag(gamma r_k) K S^T)              (64 x dv)
//   U       = T X
//   O       = diag(gamma r_q) Q S^T + P U,  P[t][s] = (gamma_t/gamma_s) r_q,t r_k,s (q_t . k_s), s <= t
//   S      <- gamma_C S + (diag(gamma_C/gamma r_k) U)^T K
// which is the sequential recurrence reorganised exactly (the reorganisation
// is pinned in fp64 against the sequential oracle by the test suite).  This is
// the "block" form of the rule the recurrent-layer kernels provide (TandemLLM
// "Architecture" v0.11.1, "The parts"); chunk-parallel and sequential forms
// agree mathematically but round differently ("Serving A Research Architecture
// On CPU", third exactness layer).
//
// One CTA owns one value head; thread i owns state row i, which is TMEM lane i
// of every accumulator, so all products are written in the transposed form
// (value rows as M = 128): S [K;Q]^T, X^T T^T, Uhat^T K and U^T P^T.  The state
// stays in TMEM as an fp32 accumulator across all chunks and crosses HBM once
// in and once out.  Operands that are not exact in bf16 (S, X, T, U, P) are
// split into bf16 hi + lo and multiplied in 2 or 3 passes (hi.hi + hi.lo +
// lo.hi) so the result keeps close to fp32 accuracy; q, k, v enter as the raw
// bf16 inputs (exact) with the norms applied as fp32 scalings.  T is solved
// on the CUDA cores by column-parallel forward substitution.
//
// Heads smaller than 128 run the same recurrence token by token with the
// decode kernel (still on the GPU; the chunk form here is written for the
// 128-wide heads of the 27B layer).
#include <cuda_runtime.h>

#include <cmath>

#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

using namespace gdn::tc;

constexpr int kChunk = 64;
constexpr int kD = 128;
constexpr int kPrefillThreads = 128;

// Shared memory map (bytes).
constexpr uint32_t OFF_S_HI = 0;        // S hi  [128 i][128 j]   A of S [K;Q]^T
constexpr uint32_t OFF_S_LO = 32768;    // S lo
constexpr uint32_t OFF_KQ = 65536;      // [K;Q] [128 t'][128 j]  B of S [K;Q]^T, A and B of [K;Q] K^T
constexpr uint32_t OFF_KT = 98304;      // K^T   [128 j][64 t]    B of Uhat^T K
constexpr uint32_t OFF_V = 114688;      // V     [64 t][128 i]    plain row-major
constexpr uint32_t OFF_T_HI = 131072;   // T     [64 t][64 s]     B of X^T T^T
constexpr uint32_t OFF_T_LO = 139264;
constexpr uint32_t OFF_P_HI = 147456;   // P     [64 t][64 s]     B of U^T P^T
constexpr uint32_t OFF_P_LO = 155648;
constexpr uint32_t OFF_X_HI = 163840;   // X^T, then Uhat^T [128 i][64 s]  A
constexpr uint32_t OFF_X_LO = 180224;
constexpr uint32_t OFF_U_HI = 196608;   // U^T   [128 i][64 s]    A of U^T P^T
constexpr uint32_t OFF_U_LO = 212992;
constexpr uint32_t OFF_L = 196608;      // L fp32 [64][64] (aliases U^T, used before it)
constexpr uint32_t OFF_SCAL = 229376;   // alpha, beta, log gamma, r_k, r_q: 5 x 64 fp32
constexpr uint32_t OFF_MISC = OFF_SCAL + 5 * 64 * 4;  // mbarrier, TMEM base, abort flag
constexpr uint32_t kPrefillSmem = OFF_MISC + 32;

// TMEM columns (fp32 accumulators, 128 lanes each).
constexpr uint32_t COL_S = 0;     // S [i][j]                 128 columns
constexpr uint32_t COL_KQ = 128;  // (S K^T) [i][t]           64 columns
constexpr uint32_t COL_O = 192;   // (S Q^T), then O^T [i][t] 64 columns
constexpr uint32_t COL_U = 256;   // U^T [i][t]               64 columns
constexpr uint32_t COL_G = 320;   // [K;Q] K^T [t'][s]        64 columns
constexpr uint32_t kTmemCols = 512;

constexpr uint64_t kWaitLimitNs = 200000000ull;  // 0.2 s per tensor-core batch

struct PrefillParams {
    const uint16_t* qkv;
    const float* alpha;
    const float* beta;
    float* state;
    void* out;
    int* status;
    int T, Hk, Hv, C, group;
    float q_scale;
    int normalize;
    int out_bf16;
};

__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__global__ void __launch_bounds__(kPrefillThreads, 1)
gdn_prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t sm[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int h = blockIdx.x;
    const int g = h / p.group;
    float* s_alpha = reinterpret_cast<float*>(sm + OFF_SCAL);
    float* s_beta = s_alpha + 64;
    float* s_lg = s_alpha + 128;
    float* s_rk = s_alpha + 192;
    float* s_rq = s_alpha + 256;
    uint64_t* bar_ptr = reinterpret_cast<uint64_t*>(sm + OFF_MISC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC + 8);
    int* abort_flag = reinterpret_cast<int*>(sm + OFF_MISC + 12);
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar = smem_u32(bar_ptr);

    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    if (tid == 0) {
        mbar_init(bar, 1);
        *abort_flag = 0;
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);  // this thread's lane
    uint32_t parity = 0;

    // wait for the tensor cores; on a timeout every thread leaves the chunk loop
    auto wait_mma = [&]() -> bool {
        const bool ok = mbar_wait(bar, parity, kWaitLimitNs);
        if (ok) parity ^= 1u;  // on a timeout keep the phase, to drain it below
        else atomicOr(abort_flag, 1);
        __syncthreads();
        fence_after_sync();
        return *abort_flag == 0;
    };

    // ---- prologue: state row i -> TMEM lane i and the bf16 hi/lo operand tiles
    float* srow = p.state + ((size_t)h * kD + tid) * kD;
#pragma unroll 1
    for (int c0 = 0; c0 < kD; c0 += 16) {
        float v[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 f = *reinterpret_cast<const float4*>(srow + c0 + 4 * q);
            v[4 * q] = f.x;
            v[4 * q + 1] = f.y;
            v[4 * q + 2] = f.z;
            v[4 * q + 3] = f.w;
        }
        tmem_st16(trow + COL_S + c0, v);
        store_split8(sm + OFF_S_HI + core_off(tid, c0, kD), sm + OFF_S_LO + core_off(tid, c0, kD), v);
        store_split8(sm + OFF_S_HI + core_off(tid, c0 + 8, kD), sm + OFF_S_LO + core_off(tid, c0 + 8, kD), v + 8);
    }
    tmem_wait_st();

    const int nchunks = (p.T + kChunk - 1) / kChunk;
    const size_t C = (size_t)p.C;
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = c * kChunk;
        const int n = min(kChunk, p.T - t0);

        // ---- A: stage the chunk's inputs ---------------------------------
        {
            // thread t' loads row t' of [K;Q] (t' < 64: k_t, else q_t) and its norm
            const int t = tid & 63;
            const bool is_q = tid >= 64;
            const bool valid = t < n;
            const uint16_t* src = p.qkv + (size_t)(t0 + t) * C + (is_q ? 0 : (size_t)p.Hk * kD) + (size_t)g * kD;
            float ss = 0.f;
#pragma unroll 4
            for (int kb = 0; kb < 16; ++kb) {
                uint4 w = make_uint4(0, 0, 0, 0);
                if (valid) w = __ldg(reinterpret_cast<const uint4*>(src + kb * 8));
                const uint16_t* e = reinterpret_cast<const uint16_t*>(&w);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float x = bf16_to_f(e[j]);
                    ss = __fmaf_rn(x, x, ss);
                }
                *reinterpret_cast<uint4*>(sm + OFF_KQ + core_off(tid, kb * 8, kD)) = w;
                if (!is_q) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint16_t*>(sm + OFF_KT + core_off(kb * 8 + j, t, kChunk)) = e[j];
                }
            }
            const float r = p.normalize ? rsqrtf(__fadd_rn(ss, 1e-6f)) : 1.0f;
            if (is_q) s_rq[t] = __fmul_rn(r, p.q_scale);
            else s_rk[t] = r;
            // v rows of this value head (plain row-major)
#pragma unroll 2
            for (int e = tid; e < kChunk * 16; e += kPrefillThreads) {
                const int tt = e >> 4, kb = e & 15;
                uint4 w = make_uint4(0, 0, 0, 0);
                if (tt < n)
                    w = __ldg(reinterpret_cast<const uint4*>(p.qkv + (size_t)(t0 + tt) * C + (size_t)2 * p.Hk * kD +
                                                             (size_t)h * kD + kb * 8));
                *reinterpret_cast<uint4*>(sm + OFF_V + tt * 256 + kb * 16) = w;
            }
            if (tid < kChunk) {
                const bool ok = tid < n;
                s_alpha[tid] = ok ? p.alpha[(size_t)(t0 + tid) * p.Hv + h] : 1.0f;
                s_beta[tid] = ok ? p.beta[(size_t)(t0 + tid) * p.Hv + h] : 0.0f;
            }
        }
        __syncthreads();
        if (warp == 0) {
            // log gamma: inclusive prefix sum of log(alpha) (two tokens per lane)
            const int l = tid;
            const float a0 = logf(fmaxf(s_alpha[2 * l], 1e-30f));
            const float a1 = logf(fmaxf(s_alpha[2 * l + 1], 1e-30f));
            const float pair = __fadd_rn(a0, a1);
            float incl = pair;
#pragma unroll
            for (int o = 1; o < 32; o *= 2) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (l >= o) incl = __fadd_rn(incl, y);
            }
            const float excl = __fsub_rn(incl, pair);
            s_lg[2 * l] = __fadd_rn(excl, a0);
            s_lg[2 * l + 1] = incl;
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        // ---- B: [K;Q] K^T (1 pass) and S [K;Q]^T (S hi, S lo) -------------
        if (tid == 0) {
            fence_after_sync();
            constexpr uint32_t id_g = idesc_bf16(128, 64);
            constexpr uint32_t id_kq = idesc_bf16(128, 128);
#pragma unroll 1
            for (int ks = 0; ks < kD / 16; ++ks)
                mma_bf16(tmem + COL_G, smem_desc(sbase + OFF_KQ + ks * 256, kD * 16),
                         smem_desc(sbase + OFF_KQ + ks * 256, kD * 16), id_g, ks > 0);
#pragma unroll 1
            for (int pass = 0; pass < 2; ++pass)
#pragma unroll 1
                for (int ks = 0; ks < kD / 16; ++ks)
                    mma_bf16(tmem + COL_KQ, smem_desc(sbase + (pass ? OFF_S_LO : OFF_S_HI) + ks * 256, kD * 16),
                             smem_desc(sbase + OFF_KQ + ks * 256, kD * 16), id_kq, (pass > 0 || ks > 0));
            mma_commit(bar);
        }
        if (!wait_mma()) break;

        // ---- C: L, P, X^T and the scaled Q S^T ----------------------------
        {
            const int t = tid & 63;
            const float lg_t = s_lg[t];
#pragma unroll 1
            for (int s0 = 0; s0 < kChunk; s0 += 16) {
                float a[16];
                tmem_ld16(trow + COL_G + s0, a);
                if (tid < 64) {
                    // L row t (strictly lower), fp32 for the solve
                    const float f = __fmul_rn(s_beta[t], s_rk[t]);
                    float lrow[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int s = s0 + j;
                        const float ratio = expf(__fsub_rn(lg_t, s_lg[s]));
                        lrow[j] = (s < t) ? __fmul_rn(__fmul_rn(f, __fmul_rn(s_rk[s], ratio)), a[j]) : 0.f;
                    }
                    float4* dst = reinterpret_cast<float4*>(sm + OFF_L + (t * kChunk + s0) * 4);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = make_float4(lrow[4 * q], lrow[4 * q + 1], lrow[4 * q + 2], lrow[4 * q + 3]);
                } else {
                    // P row t (lower incl. diagonal), split for the B operand
                    const float f = s_rq[t];
                    float prow[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int s = s0 + j;
                        const float ratio = expf(__fsub_rn(lg_t, s_lg[s]));
                        prow[j] = (s <= t) ? __fmul_rn(__fmul_rn(f, __fmul_rn(s_rk[s], ratio)), a[j]) : 0.f;
                    }
                    store_split8(sm + OFF_P_HI + core_off(t, s0, kChunk), sm + OFF_P_LO + core_off(t, s0, kChunk), prow);
                    store_split8(sm + OFF_P_HI + core_off(t, s0 + 8, kChunk),
                                 sm + OFF_P_LO + core_off(t, s0 + 8, kChunk), prow + 8);
                }
            }
            // thread i: X^T[i][s] = beta_s (v_s[i] - gamma_s r_k,s (S k_s)[i])
            const int i = tid;
            const uint16_t* vcol = reinterpret_cast<const uint16_t*>(sm + OFF_V) + i;
#pragma unroll 1
            for (int s0 = 0; s0 < kChunk; s0 += 16) {
                float ks[16], x[16];
                tmem_ld16(trow + COL_KQ + s0, ks);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int s = s0 + j;
                    const float gk = __fmul_rn(expf(s_lg[s]), s_rk[s]);
                    x[j] = __fmul_rn(s_beta[s], __fmaf_rn(-gk, ks[j], bf16_to_f(vcol[s * kD])));
                }
                store_split8(sm + OFF_X_HI + core_off(i, s0, kChunk), sm + OFF_X_LO + core_off(i, s0, kChunk), x);
                store_split8(sm + OFF_X_HI + core_off(i, s0 + 8, kChunk), sm + OFF_X_LO + core_off(i, s0 + 8, kChunk),
                             x + 8);
            }
            // scaled (S q_t)[i] * gamma_t r_q,t, written back as the start of O^T
#pragma unroll 1
            for (int s0 = 0; s0 < kChunk; s0 += 16) {
                float qs[16];
                tmem_ld16(trow + COL_O + s0, qs);
#pragma unroll
                for (int j = 0; j < 16; ++j) qs[j] = __fmul_rn(qs[j], __fmul_rn(expf(s_lg[s0 + j]), s_rq[s0 + j]));
                tmem_st16(trow + COL_O + s0, qs);
            }
            tmem_wait_st();
        }
        __syncthreads();

        // ---- D: T = (I + L)^-1, column c per thread (threads 0..63) --------
        if (tid < kChunk) {
            const int cc = tid;
            const float4* L4 = reinterpret_cast<const float4*>(sm + OFF_L);
            float col[kChunk];
#pragma unroll
            for (int t = 0; t < kChunk; ++t) col[t] = (t == cc) ? 1.f : 0.f;
#pragma unroll
            for (int t = 1; t < kChunk; ++t) {
                float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
                for (int s4 = 0; s4 < (t + 3) / 4; ++s4) {
                    const float4 l = L4[t * 16 + s4];
                    acc0 = __fmaf_rn(l.x, col[4 * s4], acc0);
                    if (4 * s4 + 1 < t) acc1 = __fmaf_rn(l.y, col[4 * s4 + 1], acc1);
                    if (4 * s4 + 2 < t) acc2 = __fmaf_rn(l.z, col[4 * s4 + 2], acc2);
                    if (4 * s4 + 3 < t) acc3 = __fmaf_rn(l.w, col[4 * s4 + 3], acc3);
                }
                const float v = -__fadd_rn(__fadd_rn(acc0, acc1), __fadd_rn(acc2, acc3));
                if (t > cc) col[t] = v;
            }
#pragma unroll
            for (int t = 0; t < kChunk; ++t) {
                __nv_bfloat16 hi, lo;
                split_bf16(col[t], hi, lo);
                *reinterpret_cast<__nv_bfloat16*>(sm + OFF_T_HI + core_off(t, cc, kChunk)) = hi;
                *reinterpret_cast<__nv_bfloat16*>(sm + OFF_T_LO + core_off(t, cc, kChunk)) = lo;
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        // ---- E: U^T = X^T T^T (3 passes) ----------------------------------
        if (tid == 0) {
            fence_after_sync();
            constexpr uint32_t id = idesc_bf16(128, 64);
            const uint32_t a_off[3] = {OFF_X_HI, OFF_X_HI, OFF_X_LO};
            const uint32_t b_off[3] = {OFF_T_HI, OFF_T_LO, OFF_T_HI};
#pragma unroll 1
            for (int pass = 0; pass < 3; ++pass)
#pragma unroll 1
                for (int ks = 0; ks < kChunk / 16; ++ks)
                    mma_bf16(tmem + COL_U, smem_desc(sbase + a_off[pass] + ks * 256, kChunk * 16),
                             smem_desc(sbase + b_off[pass] + ks * 256, kChunk * 16), id, (pass > 0 || ks > 0));
            mma_commit(bar);
        }
        if (!wait_mma()) break;

        // ---- F: Uhat^T and U^T operands; S <- gamma_C S -------------------
        {
            const int i = tid;
            const float lg_c = s_lg[kChunk - 1];
#pragma unroll 1
            for (int s0 = 0; s0 < kChunk; s0 += 16) {
                float u[16], uh[16];
                tmem_ld16(trow + COL_U + s0, u);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    uh[j] = __fmul_rn(u[j], __fmul_rn(expf(__fsub_rn(lg_c, s_lg[s0 + j])), s_rk[s0 + j]));
                store_split8(sm + OFF_X_HI + core_off(i, s0, kChunk), sm + OFF_X_LO + core_off(i, s0, kChunk), uh);
                store_split8(sm + OFF_X_HI + core_off(i, s0 + 8, kChunk), sm + OFF_X_LO + core_off(i, s0 + 8, kChunk),
                             uh + 8);
                store_split8(sm + OFF_U_HI + core_off(i, s0, kChunk), sm + OFF_U_LO + core_off(i, s0, kChunk), u);
                store_split8(sm + OFF_U_HI + core_off(i, s0 + 8, kChunk), sm + OFF_U_LO + core_off(i, s0 + 8, kChunk),
                             u + 8);
            }
            const float gamma_c = expf(lg_c);
#pragma unroll 1
            for (int c0 = 0; c0 < kD; c0 += 16) {
                float sv[16];
                tmem_ld16(trow + COL_S + c0, sv);
#pragma unroll
                for (int j = 0; j < 16; ++j) sv[j] = __fmul_rn(sv[j], gamma_c);
                tmem_st16(trow + COL_S + c0, sv);
            }
            tmem_wait_st();
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        // ---- G: S += Uhat^T K (2 passes); O^T += U^T P^T (3 passes) --------
        if (tid == 0) {
            fence_after_sync();
            constexpr uint32_t id_s = idesc_bf16(128, 128);
            constexpr uint32_t id_o = idesc_bf16(128, 64);
#pragma unroll 1
            for (int pass = 0; pass < 2; ++pass)
#pragma unroll 1
                for (int ks = 0; ks < kChunk / 16; ++ks)
                    mma_bf16(tmem + COL_S, smem_desc(sbase + (pass ? OFF_X_LO : OFF_X_HI) + ks * 256, kChunk * 16),
                             smem_desc(sbase + OFF_KT + ks * 256, kChunk * 16), id_s, 1u);
            const uint32_t a_off[3] = {OFF_U_HI, OFF_U_HI, OFF_U_LO};
            const uint32_t b_off[3] = {OFF_P_HI, OFF_P_LO, OFF_P_HI};
#pragma unroll 1
            for (int pass = 0; pass < 3; ++pass)
#pragma unroll 1
                for (int ks = 0; ks < kChunk / 16; ++ks)
                    mma_bf16(tmem + COL_O, smem_desc(sbase + a_off[pass] + ks * 256, kChunk * 16),
                             smem_desc(sbase + b_off[pass] + ks * 256, kChunk * 16), id_o, 1u);
            mma_commit(bar);
        }
        if (!wait_mma()) break;

        // ---- H: outputs, next chunk's S operands, final state -------------
        {
            const int i = tid;
            const size_t ostride = (size_t)p.Hv * kD;
            const size_t obase = (size_t)t0 * ostride + (size_t)h * kD + i;
#pragma unroll 1
            for (int s0 = 0; s0 < kChunk; s0 += 16) {
                float o[16];
                tmem_ld16(trow + COL_O + s0, o);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if (s0 + j < n) {
                        const size_t idx = obase + (size_t)(s0 + j) * ostride;
                        if (p.out_bf16) reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(o[j]);
                        else reinterpret_cast<float*>(p.out)[idx] = o[j];
                    }
                }
            }
            const bool last = (c == nchunks - 1);
#pragma unroll 1
            for (int c0 = 0; c0 < kD; c0 += 16) {
                float sv[16];
                tmem_ld16(trow + COL_S + c0, sv);
                if (last) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<float4*>(srow + c0 + 4 * q) =
                            make_float4(sv[4 * q], sv[4 * q + 1], sv[4 * q + 2], sv[4 * q + 3]);
                } else {
                    store_split8(sm + OFF_S_HI + core_off(i, c0, kD), sm + OFF_S_LO + core_off(i, c0, kD), sv);
                    store_split8(sm + OFF_S_HI + core_off(i, c0 + 8, kD), sm + OFF_S_LO + core_off(i, c0 + 8, kD),
                                 sv + 8);
                }
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
    }

    if (*abort_flag != 0) {
        if (tid == 0) atomicExch(p.status, 1);
        // give in-flight tensor-core work one more bounded chance to drain
        mbar_wait(bar, parity, kWaitLimitNs);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

size_t gdn_prefill_workspace_bytes(const gdn_shape* shape, int32_t T, int32_t chunk) {
    if (shape == nullptr || T < 0 || chunk != kChunk) return 0;
    return 256;  // status word (int32 at offset 0), padded
}

int gdn_chunk_prefill(const gdn_shape* shape, int32_t T, int32_t chunk, const gdn_bf16* qkv,
                      const float* alpha, const float* beta, float* state, void* out, void* workspace,
                      size_t workspace_bytes, float q_scale, uint32_t flags, void* stream) {
    int rc = check_prefill_args(shape, T, chunk, qkv, alpha, beta, state, out, workspace,
                                        workspace_bytes, flags);
    if (rc != GDN_OK || T == 0) return rc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(workspace, 0, 16, st);
    if (e != cudaSuccess) return cuda_error(e, "prefill status reset");
    if (shape->dk != kD || shape->dv != kD) {
        // narrower heads: the same recurrence token by token on the GPU
        return gdn_decode_step(shape, T, qkv, alpha, beta, state, out, q_scale, flags, stream);
    }
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(gdn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kPrefillSmem);
        if (e != cudaSuccess) return cuda_error(e, "prefill smem attribute");
        configured[dev] = true;
    }
    PrefillParams p{};
    p.qkv = qkv;
    p.alpha = alpha;
    p.beta = beta;
    p.state = state;
    p.out = out;
    p.status = static_cast<int*>(workspace);
    p.T = T;
    p.Hk = shape->Hk;
    p.Hv = shape->Hv;
    p.C = 2 * shape->Hk * shape->dk + shape->Hv * shape->dv;
    p.group = shape->Hv / shape->Hk;
    p.q_scale = q_scale;
    p.normalize = (flags & GDN_NORMALIZE_QK) != 0;
    p.out_bf16 = (flags & GDN_OUT_BF16) != 0;
    gdn_prefill_tc_kernel<<<shape->Hv, kPrefillThreads, kPrefillSmem, st>>>(p);
    e = cudaGetLastError();
    return e == cudaSuccess ? GDN_OK : cuda_error(e, "prefill launch");
}

}  // extern "C"
