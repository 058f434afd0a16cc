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
// Substituting U = T X gives the form the pipelined chain runs, which never
// forms U:
//   S  <- gamma_C S + X^T W,                W  = T^T diag(c) K,  c_t = (gamma_C/gamma_t) r_k,t
//   O^T = (S Q^T) diag(gamma r_q) + X^T PT^T, PT = P T
// W and PT depend only on the chunk's own q, k, alpha and beta, so a pre-pass
// computes them for every chunk in parallel and the chain per value head only
// carries S [K;Q]^T -> X^T -> S += X^T W from chunk to chunk.
//
// A chain CTA owns one value head; thread i owns state row i, which is TMEM
// lane i of every accumulator, so all products are written in the transposed
// form (value rows as M = 128).  The state stays in TMEM as an fp32
// accumulator across all chunks and crosses HBM once in and once out.
// Operands that are not exact in bf16 (S, X, T, P, W, PT) are split into bf16
// hi + lo and multiplied in 2 or 3 passes (hi.hi + hi.lo + lo.hi) so the
// result keeps close to fp32 accuracy; q, k, v enter as the raw bf16 inputs
// (exact) with the norms applied as fp32 scalings.  T is solved on the CUDA
// cores by blocked forward substitution.
//
// The kernels in this file:
//   gdn_prefill_prep_kernel   the pre-pass: W, PT and the per-token scalars of
//                             every (chunk, value head), written as records;
//   gdn_prefill_chain_kernel  the pipelined chain reading those records;
//   gdn_prefill_fused_kernel  both in one cooperative launch, the pre-pass
//                             workers running ahead of the chains (the form
//                             gdn_chunk_prefill takes where the GPU holds it);
//   gdn_prefill_tc_kernel     the self-contained chain in the U form, computing
//                             each chunk's T and P itself
//                             (gdn_chunk_prefill_noalloc).
// The first three run the same code on the same records, so the cooperative
// and two-launch forms give the same bits; the self-contained chain groups the
// same algebra differently and agrees within rounding.
//
// Heads smaller than 128 run the same recurrence token by token with the
// decode kernel (still on the GPU; the chunk form here is written for the
// 128-wide heads of the 27B layer).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

using namespace gdn::tc;

constexpr int kChunk = 64;
constexpr int kD = 128;
constexpr int kPrefillThreads = 256;  // two warpgroups over the same 128 TMEM lanes

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
constexpr uint32_t OFF_TF = 212992;     // T fp32 [64][64] while it is solved (aliases U^T lo)
constexpr uint32_t OFF_R = 131072;      // block-solve scratch fp32 [16][48] (aliases T hi)
constexpr uint32_t OFF_SCAL = 229376;   // per-token scalars: 9 x 64 fp32 (see kernel)
constexpr uint32_t OFF_MISC = OFF_SCAL + 9 * 64 * 4;  // mbarrier, TMEM base, abort flag
constexpr uint32_t kPrefillSmem = OFF_MISC + 32;

// TMEM columns (fp32 accumulators, 128 lanes each).
constexpr uint32_t COL_S = 0;     // S [i][j]                 128 columns
constexpr uint32_t COL_KQ = 128;  // (S K^T) [i][t]           64 columns
constexpr uint32_t COL_O = 192;   // (S Q^T), then O^T [i][t] 64 columns
constexpr uint32_t COL_U = 256;   // U^T [i][t]               64 columns
constexpr uint32_t COL_G = 320;   // [K;Q] K^T [t'][s]        64 columns
constexpr uint32_t kTmemCols = 512;

// Bounded waits.  A wait for the tensor cores, a copy or another CTA's record
// gives up after PrefillParams::wait_ns (0.2 s unless the caller set another
// limit; 0 gives up at the first empty probe).  After a wait gave up, the
// kernel still lets the work it started finish before it frees tensor memory
// or exits (the drain), with this fixed limit.
constexpr uint64_t kDrainLimitNs = 200000000ull;

// Kernel parameters.  The two tensor maps describe the packed q/k/v rows
// [T][C] (bf16) for the chain's TMA loads: 64 x 64 boxes with the 128-byte
// swizzle (64 columns of 64 tokens) for K and Q, 128 x 64 plain boxes for V.
// (CUtensorMap carries its own 128-byte alignment, and so the struct.)
struct PrefillParams {
    CUtensorMap tm_kq;
    CUtensorMap tm_v;
    const uint16_t* qkv;
    const float* alpha;
    const float* beta;
    float* state;
    void* out;
    int* status;
    uint64_t wait_ns;   // limit of each bounded wait (see kDrainLimitNs)
    int* ready;         // per (chunk, value head): 1 once the pre-pass record is written (cooperative form)
    int n_workers;      // pre-pass worker CTAs of the cooperative form
    int T, Hk, Hv, C, group;
    float q_scale;
    int normalize;
    int out_bf16;
};

__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Barriers over the threads that run a chunk-local step: the whole CTA, or
// the first N threads of it (named barrier ID) when other warps of the CTA
// do something else meanwhile.
struct CtaSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};
template <int ID, int N>
struct NamedSync {
    __device__ __forceinline__ void operator()() const { asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(N) : "memory"); }
};

// The blocks of T below its diagonal in column block J (16 J .. 16 J + 15),
// one 8-column half per warp: for I = J + 1 .. 3 in turn,
//   R = L[I][J:I] T[J:I][J],   T[I][J] = -T_II R.
// Lane (column c, row group rg) keeps R[4 rg .. 4 rg + 3][c] in registers and
// gathers the rest of column c from the lanes of the same column.  L comes
// transposed (sLT[k][t] = L[t][k]) and T_II transposed (tiit[I][m][r]), so
// that every shared-memory read of a warp is one contiguous run.
template <int J>
__device__ __forceinline__ void solve_column_block(const float* sLT, float* Tf, const float* tiit, int c, int rg,
                                                   int lane) {
#pragma unroll
    for (int I = J + 1; I < 4; ++I) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 16 * J; k < 16 * I; ++k) {
            const float4 l4 = *reinterpret_cast<const float4*>(sLT + k * kChunk + 16 * I + 4 * rg);
            const float tv = Tf[k * kChunk + c];
            acc[0] = __fmaf_rn(l4.x, tv, acc[0]);
            acc[1] = __fmaf_rn(l4.y, tv, acc[1]);
            acc[2] = __fmaf_rn(l4.z, tv, acc[2]);
            acc[3] = __fmaf_rn(l4.w, tv, acc[3]);
        }
        float out[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const float rm = __shfl_sync(0xffffffffu, acc[m & 3], (m >> 2) * 8 + (lane & 7));
            const float4 t4 = *reinterpret_cast<const float4*>(tiit + I * 256 + m * 16 + 4 * rg);
            out[0] = __fmaf_rn(t4.x, rm, out[0]);
            out[1] = __fmaf_rn(t4.y, rm, out[1]);
            out[2] = __fmaf_rn(t4.z, rm, out[2]);
            out[3] = __fmaf_rn(t4.w, rm, out[3]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) Tf[(16 * I + 4 * rg + q) * kChunk + c] = -out[q];
        __syncwarp();  // the next block row reads this one's column c from the other lanes
    }
}

// ---------------------------------------------------------------------------
// Chunk-local steps, shared by the pre-pass kernel and the self-contained
// prefill kernel (the same code, so both produce the same bits).
// ---------------------------------------------------------------------------

// r_k,t = 1/|k_t| and q_scale r_q,t from the staged [K;Q] rows (threads 0..127).
__device__ __forceinline__ void kq_norms(const uint8_t* kq_tile, float* s_rk, float* s_rq, int tid, bool normalize,
                                         float q_scale) {
    if (tid < 128) {
        float ss = 0.f;
#pragma unroll 4
        for (int kb = 0; kb < 16; ++kb) {
            const uint4 w = *reinterpret_cast<const uint4*>(kq_tile + core_off(tid, kb * 8, kD));
            const uint16_t* e = reinterpret_cast<const uint16_t*>(&w);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float x = bf16_to_f(e[j]);
                ss = __fmaf_rn(x, x, ss);
            }
        }
        const float r = normalize ? rsqrtf(__fadd_rn(ss, 1e-6f)) : 1.0f;
        if (tid >= 64) s_rq[tid - 64] = __fmul_rn(r, q_scale);
        else s_rk[tid] = r;
    }
}

// log2 gamma_t: inclusive prefix sum of log2(alpha) over the chunk (warp 0,
// two tokens per lane).
__device__ __forceinline__ void log2_gamma_scan(const float* s_alpha, float* s_lg, int tid) {
    if (tid < 32) {
        const int l = tid;
        const float a0 = log2f(fmaxf(s_alpha[2 * l], 1e-30f));
        const float a1 = log2f(fmaxf(s_alpha[2 * l + 1], 1e-30f));
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
}

// Per-token products of the chunk form (threads 0..63).
__device__ __forceinline__ void chunk_scalars(const float* s_lg, const float* s_rk, const float* s_rq,
                                              const float* s_beta, float* s_gk, float* s_gq, float* s_ck,
                                              float* s_brk, int tid) {
    if (tid < kChunk) {
        const float lg = s_lg[tid];
        const float gam = exp2f(lg);
        s_gk[tid] = __fmul_rn(gam, s_rk[tid]);
        s_gq[tid] = __fmul_rn(gam, s_rq[tid]);
        s_ck[tid] = __fmul_rn(exp2f(__fsub_rn(s_lg[kChunk - 1], lg)), s_rk[tid]);
        s_brk[tid] = __fmul_rn(s_beta[tid], s_rk[tid]);
    }
}

// L (strictly lower, fp32, stored transposed: sLT[s][t] = L[t][s]) and P
// (lower with the diagonal, bf16 hi/lo tiles [t][s], K-major) from the
// [K;Q] K^T accumulator: thread i_row holds row i_row of it (K rows 0..63 give
// L, Q rows 64..127 give P); warpgroup wg takes columns 32 wg .. 32 wg + 31.
// The transposed L makes a warp's stores (consecutive t) one contiguous run.
__device__ __forceinline__ void form_l_p(uint32_t g_cols, int i_row, int wg, const float* s_lg, const float* s_brk,
                                         const float* s_rq, const float* s_rk, float* sLT, uint8_t* p_hi,
                                         uint8_t* p_lo) {
    const int t = i_row & 63;
    const bool krow = i_row < 64;
    const float lg_t = s_lg[t];
    const float f = krow ? s_brk[t] : s_rq[t];
#pragma unroll 1
    for (int s0 = wg * 32; s0 < wg * 32 + 32; s0 += 16) {
        float a[16];
        tmem_ld16(g_cols + s0, a);
        float row[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int sj = s0 + j;
            const float ratio = exp2f(__fsub_rn(lg_t, s_lg[sj]));  // gamma_t / gamma_s
            const float v = __fmul_rn(__fmul_rn(f, __fmul_rn(s_rk[sj], ratio)), a[j]);
            // L: strictly lower (rows of K); P: lower incl. diagonal (rows of Q)
            row[j] = (krow ? sj < t : sj <= t) ? v : 0.f;
        }
        if (krow) {
#pragma unroll
            for (int j = 0; j < 16; ++j) sLT[(s0 + j) * kChunk + t] = row[j];
        } else {
            store_split8(p_hi + core_off(t, s0, kChunk), p_lo + core_off(t, s0, kChunk), row);
            store_split8(p_hi + core_off(t, s0 + 8, kChunk), p_lo + core_off(t, s0 + 8, kChunk), row + 8);
        }
    }
}

// T = (I + L)^-1 (L strictly lower, given transposed), blocked by 16, into Tf
// (fp32 [64][64], zeros above the diagonal) and, when t_hi is given, bf16
// hi/lo B-operand tiles [t][s].  tiit is 4 KB of fp32 scratch (the diagonal
// blocks, transposed).  All kPrefillThreads threads; two barriers.
//  1. Warp b < 4 inverts diagonal block b, lane = column: forward substitution
//     in right-looking order (once x_q is final it enters every later row's
//     sum, each sum still running over q in increasing order).  The other
//     warps write the zero blocks above the diagonal.
//  2. Warps 2 J and 2 J + 1 fill the blocks below the diagonal in column
//     block J (solve_column_block): columns of T never mix, so no barrier
//     between them.
static_assert(kPrefillThreads == 256, "solve_t splits its work over exactly eight warps");
template <class Sync>
__device__ __forceinline__ void solve_t(const float* sLT, float* Tf, float* tiit, uint8_t* t_hi, uint8_t* t_lo,
                                        int tid, Sync sync) {
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < 4) {
        if (lane < 16) {
            const int b = warp * 16, cc = lane;
            float x[16], acc[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) acc[r] = 0.f;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                x[q] = q == cc ? 1.f : (q > cc ? -acc[q] : 0.f);
#pragma unroll
                for (int r = q + 1; r < 16; ++r) acc[r] = __fmaf_rn(sLT[(b + q) * kChunk + b + r], x[q], acc[r]);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Tf[(b + r) * kChunk + b + cc] = x[r];
            float4* dst = reinterpret_cast<float4*>(tiit + warp * 256 + cc * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        }
    } else {
        // the six 16 x 16 blocks (bi, bk) above the diagonal, in the order
        // (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const int idx = (tid - 128) + 128 * k;  // 0 .. 383: block, row, float4
            const int blk = idx >> 6, r = (idx >> 2) & 15, f4 = idx & 3;
            const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
            const int bk = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
            *reinterpret_cast<float4*>(Tf + (16 * bi + r) * kChunk + 16 * bk + 4 * f4) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    sync();
    if (warp < 6) {
        const int c = 16 * (warp >> 1) + 8 * (warp & 1) + (lane & 7), rg = lane >> 3;
        if (warp < 2) solve_column_block<0>(sLT, Tf, tiit, c, rg, lane);
        else if (warp < 4) solve_column_block<1>(sLT, Tf, tiit, c, rg, lane);
        else solve_column_block<2>(sLT, Tf, tiit, c, rg, lane);
    }
    sync();
    // T -> bf16 hi/lo B-operand tiles (rows t, K = s)
    for (int e = tid; t_hi != nullptr && e < kChunk * 8; e += kPrefillThreads) {
        const int t = e >> 3, s0 = (e & 7) * 8;
        const float4 a = *reinterpret_cast<const float4*>(Tf + t * kChunk + s0);
        const float4 b = *reinterpret_cast<const float4*>(Tf + t * kChunk + s0 + 4);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        store_split8(t_hi + core_off(t, s0, kChunk), t_lo + core_off(t, s0, kChunk), v);
    }
}

// ---------------------------------------------------------------------------
// Pre-pass: the chunk-local part of every chunk, all chunks in parallel.
// T, P and the per-token scalars depend only on the chunk's own q, k, alpha
// and beta, not on the state, so they need not sit on the chunk-to-chunk
// chain of the main kernel.  One CTA per (chunk, key head): [K;Q] K^T once,
// then for each of the key head's value heads its L, P, T and scalars, written
// to a per-(chunk, value head) record in the workspace in the layout the main
// kernel copies into shared memory as it is.
// ---------------------------------------------------------------------------
constexpr uint32_t REC_W_HI = 0;         // W^T hi [128 j][64 s]  B of X^T W (the state update)
constexpr uint32_t REC_W_LO = 16384;     // W^T lo
constexpr uint32_t REC_PT_HI = 32768;    // (P T) hi [64 t][64 s]  B of X^T (P T)^T (the outputs)
constexpr uint32_t REC_PT_LO = 40960;    // (P T) lo
constexpr uint32_t REC_SCAL = 49152;     // beta, log2 gamma, gamma r_k, gamma q_scale r_q, (gamma_C/gamma) r_k
constexpr uint32_t kRecBytes = REC_SCAL + 5 * 64 * 4;
constexpr uint32_t kRecBase = 256;       // records start after the status word

// Shared memory of one pre-pass pipeline.  Regions whose contents are dead
// are reused: once [K;Q] K^T and K^T are made, the [K;Q] tile holds P and
// T^T; once T is solved, L's region holds (diag(c) T)^T.
constexpr uint32_t Q_OFF_KQ = 0;         // [K;Q] 32 KB (K-major core matrices, 128 rows)
constexpr uint32_t Q_OFF_P = 0;          // P hi, lo [64 t][64 u] 2 x 8 KB, A of P T (after [K;Q] is consumed)
constexpr uint32_t Q_OFF_TT = 16384;     // T^T hi, lo [64 s][64 u] 2 x 8 KB, B of P T
constexpr uint32_t Q_OFF_KT = 32768;     // K^T [128 j][64 t] 16 KB, A of K^T (diag(c) T)
constexpr uint32_t Q_OFF_L = 49152;      // L^T fp32 16 KB
constexpr uint32_t Q_OFF_CT = 49152;     // (diag(c) T)^T hi, lo [64 s][64 t] 2 x 8 KB (after the solve)
constexpr uint32_t Q_OFF_TF = 65536;     // T fp32 16 KB
constexpr uint32_t Q_OFF_R = 81920;      // solve scratch 4 KB (the diagonal blocks of T, transposed)
constexpr uint32_t Q_OFF_SCAL = 86016;   // 9 x 64 fp32
constexpr uint32_t Q_OFF_AB = Q_OFF_SCAL + 9 * 64 * 4;  // alpha, beta of the group's heads: 2 x 64 x kMaxGroup fp32
constexpr int kMaxGroup = 8;                             // value heads per key head staged at once
constexpr uint32_t Q_OFF_MISC = Q_OFF_AB + 2 * 64 * kMaxGroup * 4;  // 2 mbarriers, TMEM base, abort flag
constexpr uint32_t kPrepSmem = Q_OFF_MISC + 32;
constexpr uint32_t kPrepStride = (kPrepSmem + 1023) / 1024 * 1024;  // one pipeline's share of a worker CTA
constexpr uint32_t kPrepTmemCols = 256;  // [K;Q] K^T, W^T and P T (64 columns each)

// One pre-pass item: chunk c of key head g, giving the records of the key
// head's value heads.  Per value head, from the chunk's own inputs:
//   L, P and T = (I + L)^-1 as in the chunk form;
//   W  = T^T diag(c) K with c_t = (gamma_C / gamma_t) r_k,t (64 x dk), the
//        state-update factor: S_new = gamma_C S + X^T W;
//   PT = P T (64 x 64), the output factor: O = diag(gamma r_q) Q S^T + PT X.
// (With U = T X these are the chunk form's U^T diag(c) K and P U, regrouped
// so that the chain never forms U.)  Both run on tcgen05: W^T = K^T (diag(c) T)
// with K exact in bf16 and diag(c) T split hi + lo (two passes), P T with
// both factors split (three passes: hi hi, hi lo, lo hi).  Runs on threads
// 0 .. kPrefillThreads - 1 of the CTA (tid), `sync` being a barrier over
// exactly those threads; `tmem` holds kPrepTmemCols
// columns; `bars` are two mbarriers whose phases this CTA's MMAs complete in
// turn (`*phase` counts them).  Returns false (after raising the status word)
// when a tensor-core wait timed out.
template <class Sync>
__device__ bool prep_item(const PrefillParams& p, uint8_t* sm, uint32_t tmem, uint32_t bars, uint32_t* phase, int c,
                          int g, int j0, int j1, bool publish, int tid, Sync sync) {
    const int warp = tid >> 5, lane = tid & 31;
    float* s_alpha = reinterpret_cast<float*>(sm + Q_OFF_SCAL);
    float* s_beta = s_alpha + 64;
    float* s_lg = s_alpha + 128;
    float* s_rk = s_alpha + 192;
    float* s_rq = s_alpha + 256;
    float* s_gk = s_alpha + 320;
    float* s_gq = s_alpha + 384;
    float* s_ck = s_alpha + 448;
    float* s_brk = s_alpha + 512;
    int* abort_flag = reinterpret_cast<int*>(sm + Q_OFF_MISC + 20);
    const uint32_t sbase = smem_u32(sm);
    const int t0 = c * kChunk;
    const int n = min(kChunk, p.T - t0);
    const size_t C = (size_t)p.C;
    const uint32_t bar_g = bars, bar_w = bars + 8;
    // a bounded wait for the next phase of one of the two barriers; if it gives
    // up, the MMAs are still let finish (drain) before TMEM is reused or freed
    auto wait_mma = [&](uint32_t b, uint32_t ph) {
        if (!mbar_wait(b, ph & 1u, p.wait_ns)) {
            atomicOr(abort_flag, 1);
            mbar_wait(b, ph & 1u, kDrainLimitNs);
        }
    };

    // [K;Q] rows of the chunk (zero-filled past the last token)
    for (int idx = tid; idx < 2 * kChunk * 16; idx += kPrefillThreads) {
        const int r = ((idx >> 7) << 3) | (idx & 7), kb = (idx >> 3) & 15;  // 8 rows x 4 chunks per warp
        const int t = r & 63;
        const bool ok = t < n;
        const uint16_t* src = p.qkv + (size_t)(t0 + (ok ? t : 0)) * C + (r >= 64 ? 0 : (size_t)p.Hk * kD) +
                              (size_t)g * kD + kb * 8;
        cp_async16(sbase + Q_OFF_KQ + core_off(r, kb * 8, kD), src, ok);
    }
    cp_async_commit();
    cp_async_wait_all();
    fence_async_smem();
    fence_before_sync();
    sync();
    fence_after_sync();
    const int i_row = tid & 127;
    const int wg = tid >> 7;
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);

    if (tid == 0) {
        constexpr uint32_t id_g = idesc_bf16(128, 64);
#pragma unroll 1
        for (int ks = 0; ks < kD / 16; ++ks)
            mma_bf16(tmem, smem_desc(sbase + Q_OFF_KQ + ks * 256, kD * 16),
                     smem_desc(sbase + Q_OFF_KQ + ks * 256, kD * 16), id_g, ks > 0);
        mma_commit(bar_g);
    }
    // K^T (A operand of K^T (diag(c) T)): each warp transposes 16 of the 128
    // 8 x 8 core matrices of K
#pragma unroll
    for (int it = 0; it < 128 / (kPrefillThreads / 32) / 4; ++it) {
        const int q = warp * (128 / (kPrefillThreads / 32)) + it * 4 + (lane >> 3);
        const int tb = q >> 4, jb = q & 15;
        transpose_8x8x4(sbase + Q_OFF_KQ + tb * (kD * 16) + jb * 128 + (lane & 7) * 16,
                        sbase + Q_OFF_KT + jb * (kChunk * 16) + tb * 128 + (lane & 7) * 16);
    }
    kq_norms(sm + Q_OFF_KQ, s_rk, s_rq, tid, p.normalize != 0, p.q_scale);
    // alpha and beta of the first kMaxGroup value heads of the group, all
    // requested at once ([head][token]; padding tokens: alpha 1, beta 0)
    float* s_ab = reinterpret_cast<float*>(sm + Q_OFF_AB);
    const int staged = min(p.group, kMaxGroup);
    for (int idx = tid; idx < staged * kChunk; idx += kPrefillThreads) {
        const int j = idx / kChunk, t = idx % kChunk;
        const bool in = t < n;
        const size_t at = (size_t)(t0 + (in ? t : 0)) * p.Hv + g * p.group + j;
        s_ab[idx] = in ? p.alpha[at] : 1.0f;
        s_ab[kMaxGroup * kChunk + idx] = in ? p.beta[at] : 0.0f;
    }
    wait_mma(bar_g, phase[0]++);
    sync();
    fence_after_sync();
    bool fine = *abort_flag == 0;

    float* sLT = reinterpret_cast<float*>(sm + Q_OFF_L);
    float* Tf = reinterpret_cast<float*>(sm + Q_OFF_TF);
#pragma unroll 1
    for (int j = j0; fine && j < j1; ++j) {
        const int h = g * p.group + j;
        if (tid < kChunk) {
            const bool in = tid < n;
            if (j < kMaxGroup) {
                s_alpha[tid] = s_ab[j * kChunk + tid];
                s_beta[tid] = s_ab[kMaxGroup * kChunk + j * kChunk + tid];
            } else {
                s_alpha[tid] = in ? p.alpha[(size_t)(t0 + tid) * p.Hv + h] : 1.0f;
                s_beta[tid] = in ? p.beta[(size_t)(t0 + tid) * p.Hv + h] : 0.0f;
            }
        }
        sync();
        log2_gamma_scan(s_alpha, s_lg, tid);
        sync();
        chunk_scalars(s_lg, s_rk, s_rq, s_beta, s_gk, s_gq, s_ck, s_brk, tid);
        sync();
        form_l_p(trow, i_row, wg, s_lg, s_brk, s_rq, s_rk, sLT, sm + Q_OFF_P, sm + Q_OFF_P + 8192);
        sync();
        solve_t(sLT, Tf, reinterpret_cast<float*>(sm + Q_OFF_R), nullptr, nullptr, tid, sync);
        // (diag(c) T)^T and T^T as the B operands [s][t] of K^T (diag(c) T) and
        // P T, hi/lo (a warp's lanes take consecutive s: conflict-free column
        // reads of T)
        for (int e = tid; e < kChunk * 8; e += kPrefillThreads) {
            const int sc = e & 63, tb = (e >> 6) * 8;
            float v[8], w[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                w[q] = Tf[(tb + q) * kChunk + sc];
                v[q] = __fmul_rn(s_ck[tb + q], w[q]);
            }
            store_split8(sm + Q_OFF_CT + core_off(sc, tb, kChunk), sm + Q_OFF_CT + 8192 + core_off(sc, tb, kChunk), v);
            store_split8(sm + Q_OFF_TT + core_off(sc, tb, kChunk), sm + Q_OFF_TT + 8192 + core_off(sc, tb, kChunk), w);
        }
        fence_async_smem();
        fence_before_sync();
        sync();
        if (tid == 0) {
            fence_after_sync();
            constexpr uint32_t id_w = idesc_bf16(128, 64);
#pragma unroll
            for (int pass = 0; pass < 2; ++pass)
#pragma unroll
                for (int ks = 0; ks < kChunk / 16; ++ks)
                    mma_bf16(tmem + 64, smem_desc(sbase + Q_OFF_KT + ks * 256, kChunk * 16),
                             smem_desc(sbase + Q_OFF_CT + (pass ? 8192 : 0) + ks * 256, kChunk * 16),
                             id_w, (pass > 0 || ks > 0));
            // P T: (P hi, T hi), (P hi, T lo), (P lo, T hi); M = 64, so row t
            // of the result sits in TMEM lane 32 (t / 16) + t % 16
            constexpr uint32_t id_pt = idesc_bf16(64, 64);
#pragma unroll
            for (int pass = 0; pass < 3; ++pass)
#pragma unroll
                for (int ks = 0; ks < kChunk / 16; ++ks)
                    mma_bf16(tmem + 128, smem_desc(sbase + Q_OFF_P + (pass == 2 ? 8192 : 0) + ks * 256, kChunk * 16),
                             smem_desc(sbase + Q_OFF_TT + (pass == 1 ? 8192 : 0) + ks * 256, kChunk * 16),
                             id_pt, (pass > 0 || ks > 0));
            mma_commit(bar_w);
        }
        uint8_t* rec = reinterpret_cast<uint8_t*>(p.status) + kRecBase + ((size_t)c * p.Hv + h) * kRecBytes;
        // meanwhile the per-token scalars
        if (tid < 5 * 16) {
            const float* src[5] = {s_beta, s_lg, s_gk, s_gq, s_ck};
            reinterpret_cast<uint4*>(rec + REC_SCAL)[tid] = reinterpret_cast<const uint4*>(src[tid >> 4])[tid & 15];
        }
        wait_mma(bar_w, phase[1]++);
        sync();
        fence_after_sync();
        if (*abort_flag != 0) {
            fine = false;
            break;
        }
        // the record of (chunk c, value head h): W^T (lane j, this warpgroup's
        // 32 columns s) and P T (lanes 0..15 of each warp: row t, this
        // warpgroup's 32 columns s) from TMEM as hi/lo tiles
        {
            float w[2][16];
            tmem_ld16(trow + 64 + wg * 32, w[0]);
            tmem_ld16(trow + 64 + wg * 32 + 16, w[1]);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int sc = wg * 32 + hh * 16 + q * 8;
                    store_split8(rec + REC_W_HI + core_off(i_row, sc, kChunk), rec + REC_W_LO + core_off(i_row, sc, kChunk),
                                 w[hh] + q * 8);
                }
            float pt[2][16];
            tmem_ld16(trow + 128 + wg * 32, pt[0]);
            tmem_ld16(trow + 128 + wg * 32 + 16, pt[1]);
            if (lane < 16) {
                const int t = 16 * (warp & 3) + lane;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int sc = wg * 32 + hh * 16 + q * 8;
                        store_split8(rec + REC_PT_HI + core_off(t, sc, kChunk), rec + REC_PT_LO + core_off(t, sc, kChunk),
                                     pt[hh] + q * 8);
                    }
            }
        }
        __threadfence();  // this thread's record stores, before the flag
        fence_before_sync();
        sync();  // every thread is past this head's TMEM reads, tiles and record stores
        fence_after_sync();
        if (publish && tid == 0)
            asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p.ready + (size_t)c * p.Hv + h), "r"(1) : "memory");
    }
    if (!fine && tid == 0) atomicExch(p.status, 1);
    fence_before_sync();
    sync();  // every thread is past the abort flag and the TMEM reads of this item
    fence_after_sync();
    return fine;
}

// TMEM, mbarriers and abort flag of a pre-pass CTA (threads 0 .. kPrefillThreads - 1).
template <class Sync>
__device__ uint32_t prep_setup(uint8_t* sm, int tid, Sync sync) {
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Q_OFF_MISC + 16);
    if ((tid >> 5) == 0) tmem_alloc(smem_u32(tmem_slot), kPrepTmemCols);
    if (tid == 0) {
        mbar_init(smem_u32(sm + Q_OFF_MISC), 1);
        mbar_init(smem_u32(sm + Q_OFF_MISC + 8), 1);
        *reinterpret_cast<int*>(sm + Q_OFF_MISC + 20) = 0;
    }
    fence_before_sync();
    sync();
    fence_after_sync();
    return *tmem_slot;
}

__global__ void __launch_bounds__(kPrefillThreads, 2)
gdn_prefill_prep_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t sm[];
    const int tid = threadIdx.x;
    const uint32_t tmem = prep_setup(sm, tid, CtaSync{});
    uint32_t phase[2] = {0, 0};
    prep_item(p, sm, tmem, smem_u32(sm + Q_OFF_MISC), phase, blockIdx.x, blockIdx.y, 0, p.group, false, tid, CtaSync{});
    if ((tid >> 5) == 0) tmem_dealloc(tmem, kPrepTmemCols);
}

// The self-contained chain over chunks: T, P and the per-token scalars are
// computed here, between the chunk's MMAs, with the same helper functions as
// the pre-pass (so the two paths give the same bits).  It needs no workspace
// beyond the status word, which is what the allocation-free entry point
// offers.  Two warpgroups share the 128 TMEM lanes (each takes half of every
// row's columns).
__global__ void __launch_bounds__(kPrefillThreads, 1)
gdn_prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
    constexpr int NT = kPrefillThreads;
    constexpr int NWG = NT / 128;      // warpgroups
    constexpr int CW = kChunk / NWG;   // columns of a 64-wide tile per warpgroup
    constexpr int CS = kD / NWG;       // columns of the state per warpgroup
    extern __shared__ __align__(1024) uint8_t sm[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int h = blockIdx.x;
    const int g = h / p.group;
    float* s_alpha = reinterpret_cast<float*>(sm + OFF_SCAL);
    float* s_beta = s_alpha + 64;
    float* s_lg = s_alpha + 128;   // log2 gamma_t (prefix sums of log2 alpha)
    float* s_rk = s_alpha + 192;   // r_k,t
    float* s_rq = s_alpha + 256;   // q_scale r_q,t
    float* s_gk = s_alpha + 320;   // gamma_t r_k,t
    float* s_gq = s_alpha + 384;   // gamma_t q_scale r_q,t
    float* s_ck = s_alpha + 448;   // (gamma_C / gamma_t) r_k,t
    float* s_brk = s_alpha + 512;  // beta_t r_k,t
    uint64_t* bar_ptr = reinterpret_cast<uint64_t*>(sm + OFF_MISC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC + 8);
    int* abort_flag = reinterpret_cast<int*>(sm + OFF_MISC + 12);
    uint64_t* barg_ptr = reinterpret_cast<uint64_t*>(sm + OFF_MISC + 16);
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar = smem_u32(bar_ptr);    // every MMA batch except [K;Q] K^T
    const uint32_t barg = smem_u32(barg_ptr);  // [K;Q] K^T, so L and T need not wait for S [K;Q]^T

    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(barg, 1);
        *abort_flag = 0;
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // Thread tid owns TMEM lane / state row i = tid % 128; the warpgroups
    // (wg = tid / 128) split every row's columns.
    const int i_row = tid & 127;
    const int wg = tid >> 7;
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // this thread's lane
    uint32_t parity = 0, parity_g = 0;

    // wait for the tensor cores; on a timeout every thread leaves the chunk loop
    // with the same phase kept (every thread's), to drain it below
    auto wait_on = [&](uint32_t b, uint32_t& par) -> bool {
        if (!mbar_wait(b, par, p.wait_ns)) atomicOr(abort_flag, 1);
        __syncthreads();
        fence_after_sync();
        if (*abort_flag != 0) return false;
        par ^= 1u;
        return true;
    };

    // ---- prologue: state row i -> TMEM lane i and the bf16 hi/lo operand tiles
    float* srow = p.state + ((size_t)h * kD + i_row) * kD;
#pragma unroll 1
    for (int c0 = wg * CS; c0 < wg * CS + CS; c0 += 16) {
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
        store_split8(sm + OFF_S_HI + core_off(i_row, c0, kD), sm + OFF_S_LO + core_off(i_row, c0, kD), v);
        store_split8(sm + OFF_S_HI + core_off(i_row, c0 + 8, kD), sm + OFF_S_LO + core_off(i_row, c0 + 8, kD), v + 8);
    }
    tmem_wait_st();

    const int nchunks = (p.T + kChunk - 1) / kChunk;
    const size_t C = (size_t)p.C;
    // [K;Q] rows into the K-major core layout and v rows row-major, as
    // asynchronous 16-byte copies (zero-filled past the last token)
    auto issue_kq = [&](int t0, int n) {
#pragma unroll 4
        for (int idx = tid; idx < 2 * kChunk * 16; idx += NT) {
            const int r = ((idx >> 7) << 3) | (idx & 7), kb = (idx >> 3) & 15;  // 8 rows x 4 chunks per warp
            const int t = r & 63;
            const bool ok = t < n;
            const uint16_t* src = p.qkv + (size_t)(t0 + (ok ? t : 0)) * C + (r >= 64 ? 0 : (size_t)p.Hk * kD) +
                                  (size_t)g * kD + kb * 8;
            cp_async16(sbase + OFF_KQ + core_off(r, kb * 8, kD), src, ok);
        }
    };
    auto issue_v = [&](int t0, int n) {
#pragma unroll 4
        for (int idx = tid; idx < kChunk * 16; idx += NT) {
            const int t = idx >> 4, kb = idx & 15;
            const bool ok = t < n;
            const uint16_t* src =
                p.qkv + (size_t)(t0 + (ok ? t : 0)) * C + (size_t)2 * p.Hk * kD + (size_t)h * kD + kb * 8;
            cp_async16(sbase + OFF_V + t * 256 + kb * 16, src, ok);
        }
    };
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = c * kChunk;
        const int n = min(kChunk, p.T - t0);

        // ---- A: stage the chunk's inputs ---------------------------------
        // ([K;Q] and v of chunk c > 0 were prefetched during chunk c - 1)
        {
            if (c == 0) {
                issue_kq(t0, n);
                issue_v(t0, n);
                cp_async_commit();
            }
            cp_async_wait_all();
            if (tid < kChunk) {
                const bool ok = tid < n;
                s_alpha[tid] = ok ? p.alpha[(size_t)(t0 + tid) * p.Hv + h] : 1.0f;
                s_beta[tid] = ok ? p.beta[(size_t)(t0 + tid) * p.Hv + h] : 0.0f;
            }
        }
        __syncthreads();
        kq_norms(sm + OFF_KQ, s_rk, s_rq, tid, p.normalize != 0, p.q_scale);
        {
            // K^T: each warp transposes 16 of the 128 8x8 core matrices of K
            const int lane = tid & 31;
#pragma unroll
            for (int it = 0; it < 128 / (NT / 32) / 4; ++it) {
                // core matrix (tb, jb) = (q / 16, q % 16); each warp takes 128 / (NT / 32) of them
                const int q = warp * (128 / (NT / 32)) + it * 4 + (lane >> 3);
                const int tb = q >> 4, jb = q & 15;
                const uint32_t src = sbase + OFF_KQ + tb * (kD * 16) + jb * 128 + (lane & 7) * 16;
                const uint32_t dst = sbase + OFF_KT + jb * (kChunk * 16) + tb * 128 + (lane & 7) * 16;
                transpose_8x8x4(src, dst);
            }
        }
        log2_gamma_scan(s_alpha, s_lg, tid);
        __syncthreads();
        chunk_scalars(s_lg, s_rk, s_rq, s_beta, s_gk, s_gq, s_ck, s_brk, tid);
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
            mma_commit(barg);
#pragma unroll 1
            for (int pass = 0; pass < 2; ++pass)
#pragma unroll 1
                for (int ks = 0; ks < kD / 16; ++ks)
                    mma_bf16(tmem + COL_KQ, smem_desc(sbase + (pass ? OFF_S_LO : OFF_S_HI) + ks * 256, kD * 16),
                             smem_desc(sbase + OFF_KQ + ks * 256, kD * 16), id_kq, (pass > 0 || ks > 0));
            mma_commit(bar);
        }
        {
            if (!wait_on(barg, parity_g)) break;
            // ---- C: L and P (from [K;Q] K^T), then the T solve, while S [K;Q]^T runs
            form_l_p(trow + COL_G, i_row, wg, s_lg, s_brk, s_rq, s_rk, reinterpret_cast<float*>(sm + OFF_L),
                     sm + OFF_P_HI, sm + OFF_P_LO);
            __syncthreads();
            // ---- D: T = (I + L)^-1, blocked by 16 --------------------------
            solve_t(reinterpret_cast<const float*>(sm + OFF_L), reinterpret_cast<float*>(sm + OFF_TF),
                    reinterpret_cast<float*>(sm + OFF_R), sm + OFF_T_HI, sm + OFF_T_LO, tid, CtaSync{});
            fence_async_smem();
            fence_before_sync();
            __syncthreads();
        }

        if (!wait_on(bar, parity)) break;
        // S [K;Q]^T has read [K;Q]: prefetch the next chunk's rows behind it
        if (c + 1 < nchunks) {
            issue_kq(t0 + kChunk, min(kChunk, p.T - t0 - kChunk));
            cp_async_commit();
        }

        // ---- C2: X^T and the scaled Q S^T --------------------------------
        {
            // thread i: X^T[i][s] = beta_s (v_s[i] - gamma_s r_k,s (S k_s)[i])
            const int i = i_row;
            const uint16_t* vcol = reinterpret_cast<const uint16_t*>(sm + OFF_V) + i;
#pragma unroll 1
            for (int s0 = wg * CW; s0 < wg * CW + CW; s0 += 16) {
                float ks[16], x[16];
                tmem_ld16(trow + COL_KQ + s0, ks);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int sj = s0 + j;
                    x[j] = __fmul_rn(s_beta[sj], __fmaf_rn(-s_gk[sj], ks[j], bf16_to_f(vcol[sj * kD])));
                }
                store_split8(sm + OFF_X_HI + core_off(i, s0, kChunk), sm + OFF_X_LO + core_off(i, s0, kChunk), x);
                store_split8(sm + OFF_X_HI + core_off(i, s0 + 8, kChunk), sm + OFF_X_LO + core_off(i, s0 + 8, kChunk),
                             x + 8);
            }
            // scaled (S q_t)[i] * gamma_t r_q,t, written back as the start of O^T
#pragma unroll 1
            for (int s0 = wg * CW; s0 < wg * CW + CW; s0 += 16) {
                float qs[16];
                tmem_ld16(trow + COL_O + s0, qs);
#pragma unroll
                for (int j = 0; j < 16; ++j) qs[j] = __fmul_rn(qs[j], s_gq[s0 + j]);
                tmem_st16(trow + COL_O + s0, qs);
            }
            tmem_wait_st();
        }
        __syncthreads();
        // X^T has read this chunk's v rows: prefetch the next chunk's
        if (c + 1 < nchunks) {
            issue_v(t0 + kChunk, min(kChunk, p.T - t0 - kChunk));
            cp_async_commit();
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
        if (!wait_on(bar, parity)) break;

        // ---- F: Uhat^T and U^T operands; S <- gamma_C S -------------------
        {
            const int i = i_row;
            const float lg_c = s_lg[kChunk - 1];
#pragma unroll 1
            for (int s0 = wg * CW; s0 < wg * CW + CW; s0 += 16) {
                float u[16], uh[16];
                tmem_ld16(trow + COL_U + s0, u);
#pragma unroll
                for (int j = 0; j < 16; ++j) uh[j] = __fmul_rn(u[j], s_ck[s0 + j]);
                store_split8(sm + OFF_X_HI + core_off(i, s0, kChunk), sm + OFF_X_LO + core_off(i, s0, kChunk), uh);
                store_split8(sm + OFF_X_HI + core_off(i, s0 + 8, kChunk), sm + OFF_X_LO + core_off(i, s0 + 8, kChunk),
                             uh + 8);
                store_split8(sm + OFF_U_HI + core_off(i, s0, kChunk), sm + OFF_U_LO + core_off(i, s0, kChunk), u);
                store_split8(sm + OFF_U_HI + core_off(i, s0 + 8, kChunk), sm + OFF_U_LO + core_off(i, s0 + 8, kChunk),
                             u + 8);
            }
            const float gamma_c = exp2f(lg_c);
#pragma unroll 1
            for (int c0 = wg * CS; c0 < wg * CS + CS; c0 += 16) {
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
        if (!wait_on(bar, parity)) break;

        // ---- H: outputs, next chunk's S operands, final state -------------
        {
            const int i = i_row;
            const size_t ostride = (size_t)p.Hv * kD;
            const size_t obase = (size_t)t0 * ostride + (size_t)h * kD + i;
#pragma unroll 1
            for (int s0 = wg * CW; s0 < wg * CW + CW; s0 += 16) {
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
            for (int c0 = wg * CS; c0 < wg * CS + CS; c0 += 16) {
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

    cp_async_wait_all();  // no prefetch may still be writing shared memory at exit
    if (*abort_flag != 0) {
        if (tid == 0) atomicExch(p.status, 1);
        // let in-flight tensor-core work drain (the last commit covers every
        // MMA issued before it) before TMEM is freed
        mbar_wait(bar, parity, kDrainLimitNs);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}


// ---------------------------------------------------------------------------
// The pipelined chain (pre-pass path).  The chunk form regrouped so that the
// chain never forms U = T X: with the pre-pass factors W = T^T diag(c) K and
// PT = P T,
//   S_new = gamma_C S + X^T W,      O^T = (S Q^T) diag(gamma r_q) + X^T PT^T,
// so that only S [K;Q]^T -> X^T -> S += X^T W -> the next S operand carry the
// state from chunk to chunk, while the output side (the S Q^T scaling,
// X^T PT^T and the output stores) runs in the shadow of those MMAs.  X^T is
// the A operand of both products, written by the epilogue threads straight
// to tensor memory as bf16 pairs, as is the S operand of S [K;Q]^T.  A chunk's
// inputs ([K;Q], v, the record) arrive by the copy engine into double
// buffers, requested by a copy warp of their own up to a chunk ahead; the
// output accumulator is double-buffered in tensor memory, so that chunk c's
// outputs are read out while chunk c + 1 runs.  Per chunk the MMA warp learns
// from mbarriers that X^T and the S Q^T scaling are in place; one barrier
// over the epilogue and MMA warps closes the chunk (the next S operand).
// ---------------------------------------------------------------------------
constexpr int kEpiThreads = 512;    // four epilogue warpgroups over the 128 TMEM lanes
constexpr int kLoopThreads = kEpiThreads + 32;   // and one warp that only issues the MMAs
constexpr int kChainThreads = kLoopThreads + 32;  // and one warp that only requests the inputs
constexpr uint32_t kRecStride = (kRecBytes + 1023) / 1024 * 1024;  // a record slot, padded to 1 KB

// Inputs of a chunk are double-buffered by chunk parity and loaded by the
// copy engine a whole chunk ahead.  [K;Q] is two 16 KB slabs (columns 0..63,
// 64..127), each 128 rows of 128 B with the 128-byte swizzle (K rows 0..63,
// then Q rows 64..127): four TMA boxes, read by the MMAs through swizzled
// K-major descriptors.
constexpr uint32_t C_OFF_KQ = 0;         // [K;Q] x 2   B of S [K;Q]^T
constexpr uint32_t C_OFF_V = 65536;      // V     [64 t][128 i] x 2, plain row-major
constexpr uint32_t C_OFF_REC = 98304;    // two record slots (W^T hi/lo, PT hi/lo, scalars)
constexpr uint32_t kKqBytes = 32768, kVBytes = 16384;
constexpr uint32_t kInputTx = kKqBytes + kVBytes + kRecBytes;  // bytes a chunk's inputs bring
constexpr uint32_t C_OFF_MISC = C_OFF_REC + 2 * kRecStride;  // mbarriers, TMEM base, abort flag
constexpr uint32_t kChainSmem = C_OFF_MISC + 128;
// A chain CTA takes all 512 TMEM columns of its SM, so no two may share an SM:
// its shared memory must exceed half of the 227 KB an SM offers.  The
// cooperative kernel's workers run the pre-pass in the same allocation.
static_assert(kChainSmem > 232448 / 2, "chain CTAs must not fit two to an SM");
static_assert(kChainSmem <= 232448 && kPrepStride + kPrepSmem <= kChainSmem, "shared-memory layouts");

// TMEM columns.  The state and S [K;Q]^T are fp32 accumulators.  S [K;Q]^T
// is double-buffered by chunk parity: its S K^T half feeds X^T, its S Q^T
// half becomes O^T, which is read out while the next chunk runs.  X^T as an A
// operand holds bf16 hi in its first 32 columns and lo in the next 32.  The S
// operand of the next chunk (64 columns each = 128 bf16 per lane) has hi in
// T_SH and lo in the S K^T half of the current chunk's buffer, which the X^T
// epilogue has consumed (and which the chunk after next rewrites, after the
// next chunk's MMAs have read it).
constexpr uint32_t T_S = 0;      // S [i][j]                               128 columns
constexpr uint32_t T_D = 128;    // [S K^T | S Q^T -> O^T] [i][t], 2 x 128 (by chunk parity)
constexpr uint32_t T_SH = 384;   // S hi (the next chunk's operand)        64
constexpr uint32_t T_XA = 448;   // X^T                    hi 32 + lo 32  64

// Wait (bounded by limit_ns) until ready flag `item` (chunk * Hv + value
// head) is set.
__device__ __forceinline__ bool wait_ready(const int* ready, int item, uint64_t limit_ns) {
    const uint64_t t0 = global_ns();
    while (true) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ready + item) : "memory");
        if (v != 0) return true;
        if (global_ns() - t0 >= limit_ns) return false;
        __nanosleep(100);
    }
}

// The chain of value head h.  READY: the records are produced concurrently
// by the pre-pass workers of the cooperative kernel; the copy warp waits for
// a record's flag before it requests the record, up to a chunk ahead of use.
template <bool READY>
__device__ __forceinline__ void chain_body(const PrefillParams& p, uint8_t* sm, int h) {
    constexpr int CW = kChunk / 4;  // columns of a 64-wide tile per warpgroup
    constexpr int CS = kD / 4;      // columns of the state per warpgroup
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const bool issuer = tid == kEpiThreads;    // lane 0 of the MMA warp
    const bool epi = tid < kEpiThreads;        // an epilogue thread
    const bool copier = tid >= kLoopThreads;   // the copy warp
    const int g = h / p.group;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C_OFF_MISC);  // 10 mbarriers
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C_OFF_MISC + 96);
    // raised by the threads of the chunk loop before the barrier that closes
    // a chunk, so that they all leave the loop together
    int* abort_flag = reinterpret_cast<int*>(sm + C_OFF_MISC + 100);
    int* copy_fail = reinterpret_cast<int*>(sm + C_OFF_MISC + 104);  // the copy warp gave up
    const NamedSync<1, kLoopThreads> loop_sync;  // the epilogue and MMA warps
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar_ks = smem_u32(bars + 0);    // S [K;Q]^T
    const uint32_t bar_x = smem_u32(bars + 1);     // every epilogue warp has written its part of X^T
    const uint32_t bar_qs = smem_u32(bars + 2);    // every epilogue warp has scaled its part of S Q^T
    const uint32_t bar_s = smem_u32(bars + 3);     // state update X^T W
    const uint32_t bar_o = smem_u32(bars + 4);     // outputs X^T PT^T
    const uint32_t bar_fin = smem_u32(bars + 5);   // every MMA issued, before TMEM is freed
    const uint32_t bar_in0 = smem_u32(bars + 6);   // a chunk's inputs landed in buffer 0 (bar_in0 + 8: buffer 1)
    const uint32_t bar_free0 = smem_u32(bars + 8);  // buffer 0's chunk is done with it (bar_free0 + 8: buffer 1)

    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    if (tid == 0) {
        for (int b = 0; b < 10; ++b) mbar_init(smem_u32(bars + b), (b == 1 || b == 2) ? kEpiThreads / 32 : 1);
        *abort_flag = 0;
        *copy_fail = 0;
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int i = tid & 127;   // TMEM lane = state row
    const int wg = tid >> 7;   // warpgroup: a quarter of every row's columns
    const int s0 = wg * CW;
    const int c0 = wg * CS;
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);

    // a bounded wait on one of the per-chunk barriers (each completes once per
    // chunk); a timeout only raises the flag, which every thread checks at the
    // end of the chunk, so no thread leaves a barrier the others still reach
    auto wait_mma = [&](uint32_t b, int chunk) {
        if (!mbar_wait(b, (uint32_t)chunk & 1u, p.wait_ns)) atomicOr(abort_flag, 1);
        __syncwarp();  // the tcgen05.ld that follow are warp-collective
        fence_after_sync();
    };

    // ---- prologue: state row i -> TMEM lane i and the bf16 hi/lo operand tiles
    float* srow = p.state + ((size_t)h * kD + i) * kD;
#pragma unroll 1
    for (int cc = c0; cc < (epi ? c0 + CS : c0); cc += 16) {
        float v[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 f = *reinterpret_cast<const float4*>(srow + cc + 4 * q);
            v[4 * q] = f.x;
            v[4 * q + 1] = f.y;
            v[4 * q + 2] = f.z;
            v[4 * q + 3] = f.w;
        }
        tmem_st16(trow + T_S + cc, v);
        uint32_t hi[8], lo[8];
        split_pack16(v, hi, lo);
        tmem_st8(trow + T_SH + cc / 2, hi);
        tmem_st8(trow + T_D + 128 + cc / 2, lo);  // chunk 0 reads lo from buffer 1
    }
    tmem_wait_st();

    const int nchunks = (p.T + kChunk - 1) / kChunk;
    const int lane = tid & 31;
    // The copy warp loads chunk cc's inputs into buffer cc & 1 with the copy
    // engine: four TMA boxes for [K;Q], one for V and one bulk copy of the
    // record, all counted on that buffer's barrier.  Rows past the end of the
    // prompt read as zeros.  (The barrier expects all of a chunk's bytes when
    // [K;Q] and V are requested; the record follows once its flag is set.)
    // Chunk cc's inputs, requested by the copy warp once chunk cc - 2, the
    // previous user of buffer cc & 1, is done with it (its output MMAs, the
    // last readers, committed that buffer's free barrier).  False when a wait
    // gave up.
    int in_last = -1;  // copy warp: the last chunk whose inputs it requested
    auto issue_inputs = [&](int cc) -> bool {
        const uint32_t b = bar_in0 + 8u * (uint32_t)(cc & 1);
        const int t0 = cc * kChunk;
        // the record's ready flag first (no buffer needed for that)
        int ok = 1;
        if (READY && lane == 0) ok = wait_ready(p.ready, cc * p.Hv + h, p.wait_ns);
        if (__shfl_sync(0xffffffffu, ok, 0) == 0) return false;
        if (cc >= 2) {
            if (lane == 0)
                ok = mbar_wait(bar_free0 + 8u * (uint32_t)(cc & 1), (uint32_t)((cc - 2) >> 1) & 1u, p.wait_ns);
            if (__shfl_sync(0xffffffffu, ok, 0) == 0) return false;
        }
        in_last = cc;
        if (lane == 0) mbar_arrive_expect_tx(b, kInputTx);
        __syncwarp();
        // lanes 0..3: K slab 0, Q slab 0, K slab 1, Q slab 1; lane 4: V
        if (lane < 4) {
            const uint32_t kq = sbase + C_OFF_KQ + (uint32_t)(cc & 1) * kKqBytes;
            const int is_q = lane & 1, slab = lane >> 1;
            const int x = (is_q ? 0 : p.Hk * kD) + g * kD + slab * 64;
            tma_load_2d(kq + (uint32_t)slab * 16384u + (uint32_t)is_q * 8192u, &p.tm_kq, x, t0, b);
        } else if (lane == 4) {
            tma_load_2d(sbase + C_OFF_V + (uint32_t)(cc & 1) * kVBytes, &p.tm_v, 2 * p.Hk * kD + h * kD, t0, b);
        }
        // the record (published above)
        if (lane == 0) {
            fence_proxy_async_global();
            const uint8_t* rec =
                reinterpret_cast<const uint8_t*>(p.status) + kRecBase + ((size_t)cc * p.Hv + h) * kRecBytes;
            bulk_g2s(sbase + C_OFF_REC + (uint32_t)(cc & 1) * kRecStride, rec, kRecBytes, b);
        }
        return true;
    };
    // every thread that reads a buffer waits for its phase (chunk cc is the
    // (cc >> 1)-th use of buffer cc & 1)
    auto wait_inputs = [&](int cc) {
        if (!mbar_wait(bar_in0 + 8u * (uint32_t)(cc & 1), (uint32_t)(cc >> 1) & 1u, p.wait_ns))
            atomicOr(abort_flag, 1);
    };

    // Operand descriptors, computed once: an MMA issue is then a 64-bit add
    // and the instruction (step ks of a K-major tile starts 256 B, i.e. 16
    // descriptor units, further on).  The issuing thread shares its SM
    // sub-partition with busy epilogue warps, so its instruction stream must
    // stay short for the tensor pipe to be fed at its own rate.
    const uint64_t d_kq0 = smem_desc_sw128(sbase + C_OFF_KQ);  // [K;Q] of buffer 0
    constexpr uint64_t kKqDesc = kKqBytes >> 4;                    // buffer 1 vs buffer 0
    const uint64_t d_rec0 = smem_desc(sbase + C_OFF_REC, kChunk * 16);  // record slot 0, 64-wide K-major tiles
    constexpr uint64_t kRecDesc = kRecStride >> 4;  // slot 1 vs slot 0
    constexpr uint64_t kWHi = REC_W_HI >> 4, kWLo = REC_W_LO >> 4, kPtHi = REC_PT_HI >> 4, kPtLo = REC_PT_LO >> 4;

    const size_t ostride = (size_t)p.Hv * kD;
    // outputs of chunk cc (its O^T buffer, after U^T P^T completed)
    auto store_outputs = [&](int cc) {
        const int t0 = cc * kChunk;
        const int n = min(kChunk, p.T - t0);
        float o[16];
        tmem_ld16(trow + T_D + (uint32_t)(cc & 1) * 128 + 64 + s0, o);
        const size_t obase = (size_t)(t0 + s0) * ostride + (size_t)h * kD + i;
        if (p.out_bf16) {
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + obase;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (s0 + j < n) dst[(size_t)j * ostride] = __float2bfloat16_rn(o[j]);
        } else if (n == kChunk) {
            float* dst = reinterpret_cast<float*>(p.out) + obase;
#pragma unroll
            for (int j = 0; j < 16; ++j) dst[(size_t)j * ostride] = o[j];
        } else {
            float* dst = reinterpret_cast<float*>(p.out) + obase;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (s0 + j < n) dst[(size_t)j * ostride] = o[j];
        }
    };

    if (copier) {
        // runs up to a chunk ahead of the chain, bounded by the two buffers
#pragma unroll 1
        for (int cc = 0; cc < nchunks; ++cc) {
            if (*reinterpret_cast<volatile int*>(abort_flag) != 0) break;
            if (!issue_inputs(cc)) {
                if (lane == 0) *copy_fail = 1;
                break;
            }
        }
        // no copy may still be writing shared memory at exit: wait for the
        // last requested phase of each input buffer
        if (lane == 0)
            for (int cc = in_last; cc >= 0 && cc > in_last - 2; --cc)
                if (!mbar_wait(bar_in0 + 8u * (uint32_t)(cc & 1), (uint32_t)(cc >> 1) & 1u, kDrainLimitNs))
                    *copy_fail = 1;
    } else {
        // the first chunk's MMAs read the operands of the prologue (later chunks'
        // are ordered by the barrier that closes each chunk)
        fence_before_sync();
        loop_sync();
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
            const uint32_t d_col = T_D + (uint32_t)(c & 1) * 128;  // S K^T here, O^T at + 64
            const uint32_t s_lo = T_D + (uint32_t)((c + 1) & 1) * 128;  // this chunk's S lo operand
            const uint8_t* rec = sm + C_OFF_REC + (uint32_t)(c & 1) * kRecStride;
            const float* s_beta = reinterpret_cast<const float*>(rec + REC_SCAL);  // beta_t
            const float* s_lg = s_beta + 64;   // log2 gamma_t
            const float* s_gk = s_beta + 128;  // gamma_t r_k,t
            const float* s_gq = s_beta + 192;  // gamma_t q_scale r_q,t
            const uint64_t d_rec = d_rec0 + (uint64_t)(c & 1) * kRecDesc;

            // ---- A: chunk c's inputs have landed (each thread that reads them
            // waits on the barrier itself; the S operand is in place since the
            // barrier that closed the previous chunk)
            if (epi || issuer) wait_inputs(c);

            // ---- B: S [K;Q]^T (S hi, S lo from tensor memory) into this chunk's buffer
            if (issuer) {
                fence_after_sync();
                constexpr uint32_t id = idesc_bf16(128, 128);
#pragma unroll
                for (int pass = 0; pass < 2; ++pass)
#pragma unroll
                    for (int ks = 0; ks < kD / 16; ++ks)
                        mma_bf16_ts(tmem + d_col, tmem + (pass ? s_lo : T_SH) + ks * 8,
                                    d_kq0 + (uint64_t)(c & 1) * kKqDesc + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2), id,
                                    (pass > 0 || ks > 0));
                mma_commit(bar_ks);
            }
            if (epi) {
                // in the shadow of S [K;Q]^T: S <- gamma_C S
                {
                    const float gamma_c = exp2f(s_lg[kChunk - 1]);
                    const float2 g2 = make_float2(gamma_c, gamma_c);
#pragma unroll 1
                    for (int cc = c0; cc < c0 + CS; cc += 16) {
                        float sv[16];
                        tmem_ld16(trow + T_S + cc, sv);
#pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            const float2 r = __fmul2_rn(make_float2(sv[j], sv[j + 1]), g2);
                            sv[j] = r.x;
                            sv[j + 1] = r.y;
                        }
                        tmem_st16(trow + T_S + cc, sv);
                    }
                }
                wait_mma(bar_ks, c);

                // ---- C: X^T[i][s] = beta_s (v_s[i] - gamma_s r_k,s (S k_s)[i]) as the A operand
                // of both X^T W and X^T PT^T
                {
                    const uint16_t* vcol =
                        reinterpret_cast<const uint16_t*>(sm + C_OFF_V + (uint32_t)(c & 1) * kVBytes) + i;
                    float ks[16], x[16];
                    tmem_ld16(trow + d_col + s0, ks);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 b4 = reinterpret_cast<const float4*>(s_beta + s0)[q];
                        const float4 g4 = reinterpret_cast<const float4*>(s_gk + s0)[q];
                        const int sj = s0 + 4 * q;
                        const float2 v01 = make_float2(bf16_to_f(vcol[sj * kD]), bf16_to_f(vcol[(sj + 1) * kD]));
                        const float2 v23 = make_float2(bf16_to_f(vcol[(sj + 2) * kD]), bf16_to_f(vcol[(sj + 3) * kD]));
                        const float2 lo = __fmul2_rn(make_float2(b4.x, b4.y),
                                                     __ffma2_rn(make_float2(-g4.x, -g4.y),
                                                                make_float2(ks[4 * q], ks[4 * q + 1]), v01));
                        const float2 hi = __fmul2_rn(make_float2(b4.z, b4.w),
                                                     __ffma2_rn(make_float2(-g4.z, -g4.w),
                                                                make_float2(ks[4 * q + 2], ks[4 * q + 3]), v23));
                        x[4 * q] = lo.x;
                        x[4 * q + 1] = lo.y;
                        x[4 * q + 2] = hi.x;
                        x[4 * q + 3] = hi.y;
                    }
                    uint32_t hi[8], lo[8];
                    split_pack16(x, hi, lo);
                    tmem_st8(trow + T_XA + s0 / 2, hi);
                    tmem_st8(trow + T_XA + 32 + s0 / 2, lo);
                    tmem_wait_st();  // also covers the S rescale above
                }
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_x);
            }

            // ---- G: S += X^T W (3 passes); then O^T += X^T PT^T (3 passes)
            if (issuer) {
                if (!mbar_wait(bar_x, (uint32_t)c & 1u, p.wait_ns)) atomicOr(abort_flag, 1);
                fence_after_sync();
                constexpr uint32_t id_s = idesc_bf16(128, 128);
                constexpr uint32_t id_o = idesc_bf16(128, 64);
#pragma unroll
                for (int pass = 0; pass < 3; ++pass)  // (X hi, W hi), (X hi, W lo), (X lo, W hi)
#pragma unroll
                    for (int ks = 0; ks < kChunk / 16; ++ks)
                        mma_bf16_ts(tmem + T_S, tmem + T_XA + (pass == 2 ? 32 : 0) + ks * 8,
                                    d_rec + (pass == 1 ? kWLo : kWHi) + 16 * ks, id_s, 1u);
                mma_commit(bar_s);
                // the output MMAs accumulate onto S Q^T once every epilogue warp has scaled its part
                if (!mbar_wait(bar_qs, (uint32_t)c & 1u, p.wait_ns)) atomicOr(abort_flag, 1);
                fence_after_sync();
#pragma unroll
                for (int pass = 0; pass < 3; ++pass)  // (X hi, PT hi), (X hi, PT lo), (X lo, PT hi)
#pragma unroll
                    for (int ks = 0; ks < kChunk / 16; ++ks)
                        mma_bf16_ts(tmem + d_col + 64, tmem + T_XA + (pass == 2 ? 32 : 0) + ks * 8,
                                    d_rec + (pass == 1 ? kPtLo : kPtHi) + 16 * ks, id_o, 1u);
                mma_commit(bar_o);
                mma_commit(bar_free0 + 8u * (uint32_t)(c & 1));  // the last readers of this chunk's buffers
            }
            if (epi) {
                // in the shadow of the state update: S Q^T scaled by gamma_t q_scale r_q,t
                // (the start of O^T), then the previous chunk's outputs
                {
                    float qs[16];
                    tmem_ld16(trow + d_col + 64 + s0, qs);
                    mul16(qs, s_gq + s0);
                    tmem_st16(trow + d_col + 64 + s0, qs);
                    tmem_wait_st();
                }
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_qs);
                if (c > 0) {
                    wait_mma(bar_o, c - 1);
                    store_outputs(c - 1);
                }
                wait_mma(bar_s, c);

                // ---- H: the next chunk's S operand (hi into T_SH; lo into this
                // chunk's consumed S K^T half), or the final state
                const bool last = (c == nchunks - 1);
                float sv[2][16];
                tmem_ld16(trow + T_S + c0, sv[0]);
                tmem_ld16(trow + T_S + c0 + 16, sv[1]);
                if (last) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<float4*>(srow + c0 + 16 * hh + 4 * q) =
                                make_float4(sv[hh][4 * q], sv[hh][4 * q + 1], sv[hh][4 * q + 2], sv[hh][4 * q + 3]);
                } else {
                    uint32_t hi[2][8], lo[2][8];
                    split_pack16(sv[0], hi[0], lo[0]);
                    split_pack16(sv[1], hi[1], lo[1]);
                    tmem_st8(trow + T_SH + c0 / 2, hi[0]);
                    tmem_st8(trow + T_SH + c0 / 2 + 8, hi[1]);
                    tmem_st8(trow + d_col + c0 / 2, lo[0]);
                    tmem_st8(trow + d_col + c0 / 2 + 8, lo[1]);
                    tmem_wait_st();
                }
            }
            fence_before_sync();
            loop_sync();
            if (*abort_flag != 0) break;
        }

        if (epi && *abort_flag == 0 && nchunks > 0) {
            wait_mma(bar_o, nchunks - 1);
            store_outputs(nchunks - 1);
        }
    }
    // every MMA this CTA issued has completed before TMEM is released
    fence_before_sync();
    __syncthreads();
    if (issuer) {
        fence_after_sync();
        mma_commit(bar_fin);
    }
    if (!mbar_wait(bar_fin, 0, kDrainLimitNs)) atomicOr(abort_flag, 1);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if ((*abort_flag != 0 || *copy_fail != 0) && tid == 0) atomicExch(p.status, 1);
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

__global__ void __launch_bounds__(kChainThreads, 1)
gdn_prefill_chain_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t sm[];
    chain_body<false>(p, sm, blockIdx.x);
}

// Pre-pass worker w of the cooperative kernel: two independent pipelines of
// kPrefillThreads threads (each with its own shared memory, named barrier and
// kPrepTmemCols TMEM columns of one shared allocation), pipeline q taking the
// items 2w + q, 2w + q + 2 n_workers, ... in chunk order.  The first chunk,
// which every chain waits for before it can start, is split into one item per
// value head; later chunks have one item per key head (its value heads share
// [K;Q] K^T).  Each record is published with a release store of its ready
// flag once it is written.
template <int Q>
__device__ __forceinline__ void prep_pipeline(const PrefillParams& p, uint8_t* sm, uint32_t tmem, int w) {
    const int tid = threadIdx.x - Q * kPrefillThreads;
    const NamedSync<2 + Q, kPrefillThreads> sync;
    uint8_t* smq = sm + Q * kPrepStride;
    const uint32_t bars = smem_u32(smq + Q_OFF_MISC);
    const int nchunks = (p.T + kChunk - 1) / kChunk;
    const int items = nchunks > 0 ? p.Hv + (nchunks - 1) * p.Hk : 0;
    uint32_t phase[2] = {0, 0};
#pragma unroll 1
    for (int item = 2 * w + Q; item < items; item += 2 * p.n_workers) {
        int c, g, j0, j1;
        if (item < p.Hv) {  // chunk 0, value head `item`
            c = 0;
            g = item / p.group;
            j0 = item % p.group;
            j1 = j0 + 1;
        } else {
            c = 1 + (item - p.Hv) / p.Hk;
            g = (item - p.Hv) % p.Hk;
            j0 = 0;
            j1 = p.group;
        }
        if (!prep_item(p, smq, tmem + Q * kPrepTmemCols, bars, phase, c, g, j0, j1, true, tid, sync)) break;
    }
}

__device__ __forceinline__ void prep_worker(const PrefillParams& p, uint8_t* sm, int w) {
    const int tid = threadIdx.x;  // 0 .. 2 kPrefillThreads - 1
    const NamedSync<1, 2 * kPrefillThreads> all;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Q_OFF_MISC + 16);
    if ((tid >> 5) == 0) tmem_alloc(smem_u32(tmem_slot), 2 * kPrepTmemCols);
    if (tid == 0) {
        for (int q = 0; q < 2; ++q) {
            uint8_t* smq = sm + q * kPrepStride;
            mbar_init(smem_u32(smq + Q_OFF_MISC), 1);
            mbar_init(smem_u32(smq + Q_OFF_MISC + 8), 1);
            *reinterpret_cast<int*>(smq + Q_OFF_MISC + 20) = 0;
        }
    }
    fence_before_sync();
    all();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    if (tid < kPrefillThreads) prep_pipeline<0>(p, sm, tmem, w);
    else prep_pipeline<1>(p, sm, tmem, w);
    fence_before_sync();
    all();
    fence_after_sync();
    if ((tid >> 5) == 0) tmem_dealloc(tmem, 2 * kPrepTmemCols);
}

// Pre-pass and chain in one cooperative launch (every CTA resident at once, so
// a chain may wait for a worker): CTAs 0 .. Hv - 1 run the value heads'
// chains, the others the pre-pass, so that the records of later chunks are
// computed while earlier chunks run through the chain.
__global__ void __launch_bounds__(kChainThreads, 1)
gdn_prefill_fused_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t sm[];
    if ((int)blockIdx.x < p.Hv) {
        chain_body<true>(p, sm, blockIdx.x);
    } else if ((int)threadIdx.x < 2 * kPrefillThreads) {
        prep_worker(p, sm, blockIdx.x - p.Hv);
    }
}

}  // namespace
}  // namespace gdn

using namespace gdn;

namespace {
int launch_prefill(const gdn_shape* shape, int32_t T, const gdn_bf16* qkv, const float* alpha, const float* beta,
                   float* state, void* out, void* workspace, float q_scale, uint32_t flags, cudaStream_t st,
                   bool prep);
// bytes of the ready flags (one int32 per chunk and key head), padded to 16
size_t ready_bytes(size_t nchunks, int Hv) { return (nchunks * (size_t)Hv * 4 + 15) / 16 * 16; }
constexpr int kMinWorkers = 8;  // fewest pre-pass workers worth a cooperative launch

// Limit of each bounded device wait of the prefill kernels, read at every launch.
constexpr uint64_t kDefaultWaitNs = 200000000ull;   // 0.2 s
constexpr uint64_t kMaxWaitNs = 10000000000ull;     // 10 s
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

// Copy a prefill status word (int32 in device memory) to the host once the
// stream has reached it: GDN_OK (0), GDN_ERR_TIMEOUT (non-zero) or GDN_ERR_CUDA.
int read_status_word(const void* word, void* stream, int32_t* status) {
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, word, sizeof v, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_error(e, "reading the prefill status word");
    if (status != nullptr) *status = v;
    if (v != 0)
        return report_error(GDN_ERR_TIMEOUT, "a bounded device wait of the prefill gave up (status %d): its outputs "
                            "and state are not valid", v);
    return GDN_OK;
}
}  // namespace

extern "C" {

uint64_t gdn_set_wait_limit_ns(uint64_t ns) {
    if (ns > kMaxWaitNs) ns = kMaxWaitNs;
    return g_wait_ns.exchange(ns);
}

int gdn_prefill_status(const void* workspace, void* stream, int32_t* status) {
    if (workspace == nullptr) return report_error(GDN_ERR_INVALID_ARG, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return report_error(GDN_ERR_MISALIGNED, "workspace (%p) is not 256-byte aligned", workspace);
    return read_status_word(workspace, stream, status);
}

size_t gdn_prefill_workspace_bytes(const gdn_shape* shape, int32_t T, int32_t chunk) {
    if (shape == nullptr || T < 0 || chunk != kChunk) return 0;
    // the status word (int32 at offset 0, padded), then for 128-wide heads one
    // pre-pass record per (chunk, value head) and one ready flag (int32) per
    // (chunk, key head)
    if (shape->dk != kD || shape->dv != kD || shape->Hv < 1) return kRecBase;
    const size_t nchunks = ((size_t)T + kChunk - 1) / kChunk;
    return kRecBase + nchunks * (size_t)shape->Hv * kRecBytes + ready_bytes(nchunks, shape->Hv);
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
    // the ready flags start at zero on every call
    const size_t nchunks = ((size_t)T + kChunk - 1) / kChunk;
    e = cudaMemsetAsync(static_cast<uint8_t*>(workspace) + kRecBase + nchunks * (size_t)shape->Hv * kRecBytes, 0,
                        ready_bytes(nchunks, shape->Hv), st);
    if (e != cudaSuccess) return cuda_error(e, "prefill flag reset");
    return launch_prefill(shape, T, qkv, alpha, beta, state, out, workspace, q_scale, flags, st, true);
}

}  // extern "C"

namespace {

// cuTensorMapEncodeTiled from the driver, looked up once (no link-time
// dependency on the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        (void)cudaGetLastError();
    });
    return fn;
}

// The chain's tensor maps over the packed rows qkv [T][C] (bf16): 64 x 64
// boxes with the 128-byte swizzle for the K and Q columns, 128 x 64 for V.  Returns false if the driver
// refuses them.
bool encode_qkv_maps(PrefillParams& p, const void* qkv, int T, int C) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)C * 2};
    const cuuint32_t box_kq[2] = {64, (cuuint32_t)kChunk}, box_v[2] = {(cuuint32_t)kD, (cuuint32_t)kChunk};
    const cuuint32_t unit[2] = {1, 1};
    void* base = const_cast<void*>(qkv);
    return enc(&p.tm_kq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box_kq, unit,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
           enc(&p.tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box_v, unit,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-device set-up of the prefill kernels, done once per device (with that
// device current) however many host threads make their first call at once:
// the shared-memory opt-ins, then the number of cooperative-kernel CTAs the
// device holds at once (0: no cooperative launch).
struct PrefillDevice {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int capacity = 0;
};
PrefillDevice g_prefill_dev[64];

const PrefillDevice* prefill_device(int dev) {
    if (dev < 0 || dev >= 64) return nullptr;
    PrefillDevice& d = g_prefill_dev[dev];
    std::call_once(d.once, [&d, dev] {
        cudaError_t e = cudaFuncSetAttribute(gdn_prefill_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kChainSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_prefill_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kChainSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kPrefillSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_prefill_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kPrepSmem);
        d.err = e;
        if (e != cudaSuccess) return;
        int coop = 0, sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) coop = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gdn_prefill_fused_kernel, kChainThreads,
                                                          kChainSmem) != cudaSuccess)
            per_sm = 0;
        (void)cudaGetLastError();
        d.capacity = coop ? sms * per_sm : 0;
    });
    return &d;
}

// The chunk-form launch(es): with `prep`, the pre-pass and the chain reading
// its records (the workspace holds them), as one cooperative kernel where the
// device allows it; without, the self-contained chain (the workspace holds
// only the status word).
int launch_prefill(const gdn_shape* shape, int32_t T, const gdn_bf16* qkv, const float* alpha, const float* beta,
                   float* state, void* out, void* workspace, float q_scale, uint32_t flags, cudaStream_t st,
                   bool prep) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "prefill device");
    const PrefillDevice* pd = prefill_device(dev);
    if (pd == nullptr) return report_error(GDN_ERR_CUDA, "device %d outside the 64 this library tracks", dev);
    if (pd->err != cudaSuccess) return cuda_error(pd->err, "prefill smem attribute");
    PrefillParams p{};
    p.qkv = qkv;
    p.alpha = alpha;
    p.beta = beta;
    p.state = state;
    p.out = out;
    p.status = static_cast<int*>(workspace);
    p.wait_ns = g_wait_ns.load();
    p.T = T;
    p.Hk = shape->Hk;
    p.Hv = shape->Hv;
    p.C = 2 * shape->Hk * shape->dk + shape->Hv * shape->dv;
    p.group = shape->Hv / shape->Hk;
    p.q_scale = q_scale;
    p.normalize = (flags & GDN_NORMALIZE_QK) != 0;
    p.out_bf16 = (flags & GDN_OUT_BF16) != 0;
    if (prep) {
        if (!encode_qkv_maps(p, qkv, T, p.C))
            return report_error(GDN_ERR_CUDA, "the driver refused the prefill's tensor maps");
        const int nchunks = (T + kChunk - 1) / kChunk;
        p.ready = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + kRecBase +
                                         (size_t)nchunks * shape->Hv * kRecBytes);
        // The cooperative form when the GPU holds a chain CTA per value head
        // and at least a few pre-pass workers at once; otherwise the pre-pass
        // over all chunks, then the chain.
        const int resident = pd->capacity;
        const int items = shape->Hv + (nchunks - 1) * shape->Hk;  // chunk 0 per value head, then per key head
        const int workers = std::min(resident - shape->Hv, items);
        if (workers >= kMinWorkers && (flags & GDN_PREFILL_TWO_LAUNCH) == 0) {
            p.n_workers = workers;
            void* args[] = {&p};
            e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(gdn_prefill_fused_kernel),
                                            dim3((unsigned)(shape->Hv + workers)), dim3(kChainThreads), args,
                                            kChainSmem, st);
            if (e == cudaSuccess) return GDN_OK;
            (void)cudaGetLastError();  // not launched: take the two-kernel form
        }
        const dim3 grid((unsigned)nchunks, (unsigned)shape->Hk);
        gdn_prefill_prep_kernel<<<grid, kPrefillThreads, kPrepSmem, st>>>(p);
        gdn_prefill_chain_kernel<<<shape->Hv, kChainThreads, kChainSmem, st>>>(p);
    } else {
        gdn_prefill_tc_kernel<<<shape->Hv, kPrefillThreads, kPrefillSmem, st>>>(p);
    }
    e = cudaGetLastError();
    return e == cudaSuccess ? GDN_OK : cuda_error(e, "prefill launch");
}

}  // namespace

// ---------------------------------------------------------------------------
// Prefill without caller-provided workspace.
//
// Some callers cannot allocate device memory when they run the prefill: a
// serving loop whose device memory is fixed once at start-up (it must not
// allocate while it serves, so that its footprint stays constant), or a host
// program whose device memory belongs to another allocator and which can only
// hand this library the tensors it already has.  For them the scratch the
// prefill kernel needs lives in the array below, which every GPU that loads
// this library holds until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = 256;  // largest workspace the variant can serve
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {};

// Device address of g_noalloc_scratch on the current device, looked up once per
// device (in host code the array's name is only a host-side stand-in).
cudaError_t noalloc_scratch(void** ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int gdn_chunk_prefill_noalloc_status(void* stream, int32_t* status) {
    void* scratch = nullptr;
    cudaError_t e = noalloc_scratch(&scratch);
    if (e != cudaSuccess) return cuda_error(e, "locating the built-in prefill scratch");
    return read_status_word(scratch, stream, status);
}

extern "C" int gdn_chunk_prefill_noalloc(const gdn_shape* shape, int32_t T, int32_t chunk, const gdn_bf16* qkv,
                                         const float* alpha, const float* beta, float* state, void* out,
                                         float q_scale, uint32_t flags, void* stream) {
    // the self-contained chain needs only the status word
    const size_t need = kRecBase;
    if (need > kNoAllocScratchBytes)
        return report_error(GDN_ERR_WORKSPACE, "prefill needs %zu bytes of scratch; the built-in array holds %zu",
                            need, kNoAllocScratchBytes);
    void* scratch = nullptr;
    cudaError_t e = noalloc_scratch(&scratch);
    if (e != cudaSuccess) return cuda_error(e, "locating the built-in prefill scratch");
    int rc = check_prefill_args(shape, T, chunk, qkv, alpha, beta, state, out, scratch, kNoAllocScratchBytes, flags,
                                false);
    if (rc != GDN_OK || T == 0) return rc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(scratch, 0, 16, st);
    if (e != cudaSuccess) return cuda_error(e, "prefill status reset");
    if (shape->dk != kD || shape->dv != kD)
        return gdn_decode_step(shape, T, qkv, alpha, beta, state, out, q_scale, flags, stream);
    return launch_prefill(shape, T, qkv, alpha, beta, state, out, scratch, q_scale, flags, st, false);
}
