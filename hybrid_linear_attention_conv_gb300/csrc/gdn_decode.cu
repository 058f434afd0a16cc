// gdn_decode.cu -- decode, commit and tree-verify kernels (sm_103a).
//
// Decode / commit: one CTA owns 32*R rows of one value head of one sequence.
// Its rows of the state are loaded into registers once, advanced through all
// T tokens, and stored once: the state crosses HBM exactly twice per call,
// whatever T is (the recurrent state is updated in place and never grows --
// "Serving A Research Architecture On CPU", constant-state section).  Loads and
// stores use the streaming cache hint, since a batched decode touches each
// state exactly once per step and it should not evict the activations from L2.
//
// Tree verify: one CTA owns 32 R rows of one value head and walks the draft
// tree depth-first.  The current node's rows stay in registers; the rows of a
// node with two or more children are parked in tensor memory (or, for deep
// nests, shared memory) until its last child starts (host-computed slots).
// A single tree's preorder is cut into up to three walks, each run by its own
// CTA over the same rows, so that the dependent chain of node steps is
// shorter.  The committed state is read once and node states never reach HBM
// (TandemLLM "Architecture" v0.14.2 section 8.3: each draft node's state
// branches from its parent's and the whole tree is verified in one pass).
// Given pre-conv inputs, the CTA also runs the tree conv of the channels it
// reads (a key head's CTAs share its q/k conv as one thread-block cluster; a
// walker convolves its own walk's nodes); a KDA variant applies a decay per
// key channel.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "gdn_conv.cuh"
#include "gdn_gates.cuh"
#include "gdn_internal.h"
#include "gdn_step.cuh"

namespace gdn {

constexpr int kThreads = 256;        // 8 warps = 32 row groups of 8 lanes
constexpr int kRowsPerPass = 32;
constexpr int kMaxSmemPerCta = 232448;  // the opt-in shared memory of one CTA (227 KB)
constexpr size_t kSmemTwoCtas = 233472 / 2 - 1024;  // two CTAs on one SM (228 KB, 1 KB reserved per CTA)

// Fused step (plain and KDA), several value heads per CTA: each thread copies
// its rows of the next head's state into shared memory (cp.async, its own
// slots only) while it advances the current head, so the head loop does not
// wait on DRAM between heads.  [R * V][kThreads] float4 (element-major: a warp's accesses
// are contiguous).
template <int DK, int R>
__host__ __device__ constexpr size_t conv_decode_prefetch_bytes() {
    return (size_t)R * (DK / 32) * kThreads * 16;
}
__host__ __device__ constexpr size_t align16(size_t n) { return (n + 15) / 16 * 16; }

// One 16-byte global -> shared copy (cp.async, L2 only); both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(gsrc) : "memory");
}

// One 4-byte global -> shared copy (cp.async); both addresses 4-byte aligned.
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc) {
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(gsrc) : "memory");
}

// Thread-block cluster helpers (the fused verify's shared q/k conv).
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster: shared-memory writes before it,
// local or remote, are visible to all of them after it.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store 16 bytes at the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ void st_cluster16(const void* local, uint32_t rank, uint4 v) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Tensor memory as the tree walk's branch slots.  A thread's rows of one slot
// (R V float4) sit in its own TMEM lane, 4 R V consecutive columns: warp w
// uses the lanes of quarter w mod 4 and the columns of half w / 4, so a slot
// takes 8 R V columns.  Loads and stores are exact 32-bit moves, and they
// leave the shared-memory pipe to the walk's record fetches.
template <int R, int V>
__device__ __forceinline__ void tmem_put_rows(uint32_t taddr, const float4 (&s)[R][V]) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < V; ++m)
            asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             taddr + (uint32_t)(4 * (r * V + m))),
                         "f"(s[r][m].x), "f"(s[r][m].y), "f"(s[r][m].z), "f"(s[r][m].w)
                         : "memory");
}
template <int R, int V>
__device__ __forceinline__ void tmem_get_rows(uint32_t taddr, float4 (&s)[R][V]) {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");  // this thread's earlier saves
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < V; ++m)
            asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(s[r][m].x), "=f"(s[r][m].y), "=f"(s[r][m].z), "=f"(s[r][m].w)
                         : "r"(taddr + (uint32_t)(4 * (r * V + m))));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// The conv-tail update of a commit, done by the commit's own launch: the
// tail becomes the last four inputs of (tail ++ x_tree[path[0]] ++ ...), 8
// channels (one 16-byte vector) per thread of the grid, copied as they are.
// Each vector is read and written by one thread only.  The loads are issued
// with the state loads and the stores made at the end, so that the tail adds
// no DRAM round trip to the commit.
struct CommitTail {
    uint4 v[GDN_CONV_W];
    size_t c0;
    bool mine;
};

template <typename PathIndex>
__device__ __forceinline__ void commit_tail_load(CommitTail& t, const uint16_t* x_tree, const uint16_t* tail, int C,
                                                 int L, const PathIndex* path, long long gi) {
    t.mine = gi < C / 8;
    if (!t.mine) return;
    t.c0 = (size_t)gi * 8;
#pragma unroll
    for (int j = 0; j < GDN_CONV_W; ++j) {
        const int pos = L + j;  // index into tail ++ x_tree[path]
        const uint16_t* src = pos < GDN_CONV_W ? tail + (size_t)pos * C + t.c0
                                               : x_tree + (size_t)path[pos - GDN_CONV_W] * C + t.c0;
        t.v[j] = *reinterpret_cast<const uint4*>(src);
    }
}

__device__ __forceinline__ void commit_tail_store(const CommitTail& t, uint16_t* tail, int C) {
    if (!t.mine) return;
#pragma unroll
    for (int j = 0; j < GDN_CONV_W; ++j) *reinterpret_cast<uint4*>(tail + (size_t)j * C + t.c0) = t.v[j];
}

// KDA selects a decay per key channel: alpha is then [B, Tsrc, Hv, dk].
// In is the activations' element type: uint16_t (bf16 bits) or float.
template <int DK, int R, bool GATHER, bool KDA, typename In>
__global__ void __launch_bounds__(kThreads, 2)
gdn_decode_kernel(const __grid_constant__ DecodeParams p) {
    constexpr int V = DK / 32;
    const In* qkv = reinterpret_cast<const In*>(p.qkv);
    const int lane8 = threadIdx.x & 7;
    const int rg = threadIdx.x >> 3;
    const int h = blockIdx.y;
    const int b = blockIdx.z;
    const int g = h / p.group;
    const int row0 = blockIdx.x * (kRowsPerPass * R) + rg;
    float* S = p.state + ((size_t)b * p.Hv + h) * (size_t)p.dv * DK;

    CommitTail ct;  // commit: the conv tail too (one sequence); the grid has far more threads than C / 8
    ct.mine = false;
    if (GATHER && p.x_tree != nullptr)
        commit_tail_load(ct, p.x_tree, p.tail, p.C, p.T, p.tok,
                         (((long long)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) * kThreads +
                             threadIdx.x);

    float4 s[R][V];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < V; ++m)
            s[r][m] = __ldcs(reinterpret_cast<const float4*>(
                S + (size_t)(row0 + kRowsPerPass * r) * DK + 32 * m + 4 * lane8));

    // KDA: each token's decay vector, staged in shared memory (two buffers, so
    // one barrier per token separates a buffer's readers from its next writer)
    __shared__ float4 s_gate[KDA ? 2 : 1][KDA ? DK / 4 : 1];
    const bool normalize = p.normalize != 0;
    const bool out_bf16 = p.out_bf16 != 0;
    for (int t = 0; t < p.T; ++t) {
        const int tok = GATHER ? p.tok[t] : t;
        const size_t trow = (size_t)b * p.Tsrc + tok;
        if constexpr (KDA) {
            if (threadIdx.x < DK / 4)
                s_gate[t & 1][threadIdx.x] =
                    __ldg(reinterpret_cast<const float4*>(p.alpha + (trow * p.Hv + h) * DK) + threadIdx.x);
            __syncthreads();
        }
        const In* row = qkv + trow * (size_t)p.C;
        TokenKQ<V> kq;
        token_kq<V>(row + g * DK, row + (size_t)p.Hk * DK + g * DK, lane8, p.q_scale,
                    normalize, kq);
        float alpha = 0.0f;
        if constexpr (!KDA) alpha = p.alpha[trow * p.Hv + h];
        const float beta = p.beta[trow * p.Hv + h];
        const In* vrow = row + (size_t)2 * p.Hk * DK + (size_t)h * p.dv;
        if constexpr (KDA) {
            float4 g[V];
            load_gate_smem<V>(s_gate[t & 1], lane8, g);
#pragma unroll
            for (int r = 0; r < R; ++r) kda_decay<V>(s[r], g);
        }
        float my_o = 0.0f;  // lane l < R of a row group stores row r = l (all lanes hold the same o)
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int i = row0 + kRowsPerPass * r;
            const float v_i = act_f(vrow[i]);
            float o;
            if constexpr (KDA) o = delta_row_step<V>(s[r], kq, v_i, beta);
            else o = row_step<V>(s[r], kq, v_i, alpha, beta);
            if (lane8 == r) my_o = o;
        }
        if (p.out != nullptr && lane8 < R)
            store_out(p.out, (((size_t)b * p.T + t) * p.Hv + h) * p.dv + row0 + kRowsPerPass * lane8, my_o, out_bf16);
    }

#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < V; ++m)
            __stcs(reinterpret_cast<float4*>(S + (size_t)(row0 + kRowsPerPass * r) * DK + 32 * m +
                                             4 * lane8),
                   s[r][m]);
    if (GATHER) commit_tail_store(ct, p.tail, p.C);
}

// Commit of several sequences' accepted paths in one launch.  A CTA owns 32 R
// rows of one value head of one sequence and replays that sequence's path
// through the shared step, exactly as gdn_decode_kernel does with a gather
// map (the same functions in the same order), so each sequence's result is the
// bits of gdn_commit_path on its tree alone.
//
// Fused conv (p.w set): before the replay, the CTA computes the conv outputs
// of the path's tokens for the channels it reads (q and k of its key head, v
// of its own rows) into shared memory, [L][2 DK + 32 R] bf16, with the
// arithmetic and rounding of gdn_conv_step.  The path is a root path, so the
// inputs before token t are path[t-1], path[t-2], ... then the tail's newest
// entries: the tree conv of node path[t].
template <int DK, int R>
__host__ __device__ constexpr size_t commit_conv_bytes(int L) {
    return (size_t)L * (2 * DK + kRowsPerPass * R) * 2;
}

template <int DK, int R>
__global__ void __launch_bounds__(kThreads, 2)
gdn_commit_batched_kernel(const __grid_constant__ CommitBatchParams p) {
    constexpr int V = DK / 32;
    constexpr int ROWS = kRowsPerPass * R;
    constexpr int YW = 2 * DK + ROWS;  // one token's conv outputs in shared memory
    const int lane8 = threadIdx.x & 7;
    const int rg = threadIdx.x >> 3;
    const int h = blockIdx.y;
    const int b = blockIdx.z;
    const int L = p.L[b];
    const bool conv = p.w != nullptr;
    if (L == 0 && !conv) return;  // nothing accepted for this sequence
    CommitTail ct;  // sequence b's conv tail, by sequence b's CTAs (far more threads than C / 8)
    ct.mine = false;
    if (p.x_tree != nullptr)
        commit_tail_load(ct, p.x_tree + (size_t)b * p.N * p.C,
                         (conv ? p.tail_in : p.tail) + (size_t)b * GDN_CONV_W * p.C, p.C, L, p.path[b],
                         ((long long)blockIdx.y * gridDim.x + blockIdx.x) * kThreads + threadIdx.x);
    if (L == 0) {  // the fused conv: the tail is carried over to the output buffer as it is
        commit_tail_store(ct, p.tail + (size_t)b * GDN_CONV_W * p.C, p.C);
        return;
    }
    const int g = h / p.group;
    const int row0 = blockIdx.x * ROWS + rg;
    float* S = p.state + ((size_t)b * p.Hv + h) * (size_t)p.dv * DK;
    float4 s[R][V];
    auto load_state = [&]() {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < V; ++m)
                s[r][m] = __ldcs(reinterpret_cast<const float4*>(S + (size_t)(row0 + kRowsPerPass * r) * DK +
                                                                 32 * m + 4 * lane8));
    };
    // The state rows are requested before the fused conv's loads, so that the
    // two DRAM round trips overlap -- except with four rows per thread, where
    // the 64 state registers and the conv's taps and windows would not fit
    // together in the register budget of two CTAs per SM.
    constexpr bool kStateFirst = R < 4;
    if (kStateFirst || !conv) load_state();
    extern __shared__ uint4 smem_commit[];
    uint16_t* ys = reinterpret_cast<uint16_t*>(smem_commit);  // the fused conv's outputs, [L][YW]
    if (conv) {
        const uint16_t* xb = p.x_tree + (size_t)b * p.N * p.C;
        const uint16_t* tb = p.tail_in + (size_t)b * GDN_CONV_W * p.C;
        const int8_t* path = p.path[b];
        constexpr int QK8 = 2 * DK / 8, PER = YW / 8;
        for (int idx = threadIdx.x; idx < L * PER; idx += kThreads) {
            const int t = idx / PER, c = idx % PER;
            const int gc = c < DK / 8 ? g * DK + 8 * c
                         : c < QK8    ? p.Hk * DK + g * DK + 8 * (c - DK / 8)
                                      : 2 * p.Hk * DK + h * p.dv + blockIdx.x * ROWS + 8 * (c - QK8);
            float w[8][4];
            load_taps8(p.w + (size_t)gc * GDN_CONV_W, w);
            // input j of (tail ++ x_tree[path]) counted from the path's start: j < 0 is tail slot 4 + j
            auto in = [&](int j) -> Vec8 {
                return j >= 0 ? load8(xb + (size_t)path[j] * p.C + gc) : load8(tb + (size_t)(GDN_CONV_W + j) * p.C + gc);
            };
            store_y(ys + (size_t)t * YW + 8 * c, w, in(t - 3), in(t - 2), in(t - 1), in(t));
        }
        if (!kStateFirst) load_state();
        __syncthreads();
    }
    const bool normalize = p.normalize != 0;
    for (int t = 0; t < L; ++t) {
        const size_t trow = (size_t)b * p.N + p.path[b][t];
        TokenKQ<V> kq;
        const uint16_t* vrow;  // v of this CTA's row r at vrow[kRowsPerPass * r]
        if (conv) {
            const uint16_t* yt = ys + (size_t)t * YW;
            token_kq<V>(yt, yt + DK, lane8, 1.0f, normalize, kq);
            vrow = yt + 2 * DK + rg;
        } else {
            const uint16_t* row = p.qkv + trow * (size_t)p.C;
            token_kq<V>(row + g * DK, row + (size_t)p.Hk * DK + g * DK, lane8, 1.0f, normalize, kq);
            vrow = row + (size_t)2 * p.Hk * DK + (size_t)h * p.dv + row0;
        }
        const float alpha = p.alpha[trow * p.Hv + h];
        const float beta = p.beta[trow * p.Hv + h];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float v_i = act_f(vrow[kRowsPerPass * r]);
            row_step<V>(s[r], kq, v_i, alpha, beta);
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < V; ++m)
            __stcs(reinterpret_cast<float4*>(S + (size_t)(row0 + kRowsPerPass * r) * DK + 32 * m + 4 * lane8),
                   s[r][m]);
    commit_tail_store(ct, p.tail + (size_t)b * GDN_CONV_W * p.C, p.C);
}

template <int DK, int R>
static cudaError_t launch_commit_batched_t(const CommitBatchParams& p, cudaStream_t s) {
    dim3 grid(p.dv / (kRowsPerPass * R), p.Hv, p.B);
    int lmax = 0;
    for (int b = 0; b < p.B; ++b) lmax = std::max(lmax, (int)p.L[b]);
    const size_t smem = p.w != nullptr ? commit_conv_bytes<DK, R>(lmax) : 0;
    // at most 64 tokens x (2 x 128 + 128) channels x 2 bytes = 48 KB: no opt-in needed
    if (smem > 48 * 1024) return cudaErrorInvalidValue;
    gdn_commit_batched_kernel<DK, R><<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <int DK>
static cudaError_t launch_commit_batched_r(const CommitBatchParams& p, int rows_per_cta, cudaStream_t s) {
    switch (rows_per_cta) {
        case 32: return launch_commit_batched_t<DK, 1>(p, s);
        case 64: return launch_commit_batched_t<DK, 2>(p, s);
        case 128: return launch_commit_batched_t<DK, 4>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_commit_batched(const CommitBatchParams& p, int dk, int rows_per_cta, cudaStream_t s) {
    switch (dk) {
        case 32: return launch_commit_batched_r<32>(p, rows_per_cta, s);
        case 64: return launch_commit_batched_r<64>(p, rows_per_cta, s);
        case 128: return launch_commit_batched_r<128>(p, rows_per_cta, s);
    }
    return cudaErrorInvalidValue;
}

// Shared-memory staging of the tree's inputs for one CTA (after the slots):
// q and k of this CTA's key head for every node, this CTA's 32 R rows of v,
// and alpha/beta -- loaded once, all loads in flight together, before the walk.
// Per node, the normalised k and q in the lane layout of TokenKQ plus k.q,
// computed once per CTA (by one row group per node, with token_kq itself).
template <int DK>
__host__ __device__ constexpr size_t tree_kq_bytes(int N) {
    return (size_t)N * (8 * 2 * (DK / 32) * 4 * 4 + 16);
}

template <int DK, int R>
__host__ __device__ constexpr size_t tree_stage_bytes(int N) {
    // per node: the record, v, alpha/beta, the schedule step and (fused conv) its 3 ancestors + pad
    return tree_kq_bytes<DK>(N) + (size_t)N * (kRowsPerPass * R * 2 + 2 * 4 + sizeof(TreeStep) + 4);
}

// The region in front of the staging: the walk's branch slots, which the
// fused conv uses first (it is done before the walk writes its first slot):
//   y_qk  [N][2 DK] bf16      the conv outputs of the key head's q and k
//   xs    [N + 3][2 DK + 32 R] bf16  the conv inputs of the CTA's channels:
//         tail slots 1..3, then the N nodes
//   ws    [2 DK + 32 R][4] bf16      their taps
template <int DK, int R>
__host__ __device__ constexpr size_t tree_conv_bytes(int N) {
    return (size_t)N * 2 * DK * 2 + ((size_t)N + 3 + 4) * (2 * DK + kRowsPerPass * R) * 2;
}

template <int DK, int R>
__host__ __device__ constexpr size_t tree_slot_bytes(int n_slots, int N, bool conv) {
    // without the conv the region still holds y_qk, the staged q and k rows
    const size_t slots = (size_t)n_slots * kRowsPerPass * R * DK * sizeof(float);
    const size_t c = conv ? tree_conv_bytes<DK, R>(N) : (size_t)N * 2 * DK * 2;
    return slots > c ? slots : c;
}

// The tree walk.  A thread keeps R rows of the state (rows rg + 32 r of this
// CTA's 32 R), so that each node's k and q, fetched from shared memory once
// per thread, serve R rows: the walk is bound by those fetches (every row of
// every value head reads the whole record), and R rows per fetch divide that
// traffic by R while giving each thread R independent row chains.
// KDA: a decay vector per node and head (alpha [B, Nmax, Hv, dk]) staged after
// the other inputs, [N][dk] fp32; each step applies kda_decay and the delta
// step of the KDA decode, so a node's output is the bits of gdn_kda_decode_step
// over its root path.
// Walkers: with p.walkers = W > 1 (one tree), W CTAs hold the same rows and
// each walks its own part of the tree (walk[w]), the host having cut the
// tree's preorder into W ranges.  Each walk is a dependent chain of node
// steps, so W shorter chains in parallel (two CTAs to an SM) end sooner than
// one long one; every CTA stages the inputs and records it reads.
template <int DK, int MB, int R, bool KDA>
__global__ void __launch_bounds__(kThreads, 2)
gdn_tree_kernel(const __grid_constant__ TreeParamsT<MB> p) {
    constexpr int V = DK / 32;
    constexpr int ROWS = kRowsPerPass * R;  // rows of one value head per CTA
    constexpr int NT = kThreads;
    // z: the sequence b (its own tree and state), or with one tree the walker
    const int tree = MB == 1 ? 0 : (int)blockIdx.z;
    const int N = p.N[tree];
    const uint16_t* qkv = p.qkv + (size_t)tree * p.Nmax * p.C;
    const float* alpha_b = p.alpha + (size_t)tree * p.Nmax * p.Hv;
    const float* beta_b = p.beta + (size_t)tree * p.Nmax * p.Hv;
    const bool conv = p.x != nullptr;  // pre-conv inputs: the tree conv runs here
    extern __shared__ float4 smem4[];
    float4* slots = smem4;  // [n_slots][R][32 row groups][V][8 lanes]
    const int W = MB == 1 ? p.walkers : 1;   // walkers (CTAs) per row block
    const int walker = MB == 1 ? (int)blockIdx.z : 0;
    uint8_t* stage = reinterpret_cast<uint8_t*>(smem4) +
                     tree_slot_bytes<DK, R>(p.tmem_cols > 0 ? 0 : W == 1 ? p.n_slots : p.walk_slots, p.Nmax, conv);
    float4* s_kq = reinterpret_cast<float4*>(stage);                                   // per-node records
    uint16_t* s_v = reinterpret_cast<uint16_t*>(stage + tree_kq_bytes<DK>(p.Nmax));        // [N][32 R]
    float* s_ab = reinterpret_cast<float*>(s_v + (size_t)p.Nmax * ROWS);                    // [N][alpha, beta]
    // the walk's schedule (this walker's), staged from the parameters below
    TreeStep* steps = reinterpret_cast<TreeStep*>(s_ab + 2 * (size_t)p.Nmax);
    // the fused conv's ancestor table, [N] x (3 ancestors + pad), copied out of the parameters
    char4* s_anc = reinterpret_cast<char4*>(steps + p.Nmax);
    // KDA: the nodes' decay vectors for head h, [N][DK / 4] float4, after the staging
    float4* s_gate = reinterpret_cast<float4*>(stage + tree_stage_bytes<DK, R>(p.Nmax));
    const int lane8 = threadIdx.x & 7;
    const int rg = threadIdx.x >> 3;
    const int h = blockIdx.y;
    const int g = h / p.group;
    const int row0 = blockIdx.x * ROWS;
    const int row = row0 + rg;  // this thread's rows: row + 32 r
    // node n's record in s_kq: [V float4 of k, V float4 of q][8 lanes], then k.q
    constexpr int KQ_REC = 8 * 2 * V + 1;  // float4 units

    // branch slots in tensor memory (p.tmem_cols columns, at most half of an
    // SM's, so that two CTAs fit), allocated by warp 0 before the staging; the
    // allocation's address goes to the last word of the dynamic shared memory
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(stage + tree_stage_bytes<DK, R>(p.Nmax) +
                                                   (KDA ? (size_t)p.Nmax * DK * 4 : 0));
    const bool tm = p.tmem_cols > 0;
    if (tm && threadIdx.x < 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         (uint32_t)__cvta_generic_to_shared(s_tmem)),
                     "r"((uint32_t)p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    }

    // this thread's rows of the committed state, requested before the staging
    // loads so that the two DRAM round trips overlap
    const float* S = p.state + ((size_t)tree * p.Hv + h) * p.dv * DK + (size_t)row * DK;
    float4 s[R][V];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < V; ++m)
            s[r][m] = __ldg(reinterpret_cast<const float4*>(S + (size_t)kRowsPerPass * r * DK + 32 * m + 4 * lane8));

    // the walks' schedules, copied out of the parameter block (read once per
    // step on the walk's dependent chain)
    const int NS = W == 1 ? N : p.walk_n[walker];  // steps of this walk
    auto stage_steps = [&] {
        if (W == 1) {
            for (int n = threadIdx.x; n < N; n += NT) steps[n] = p.steps[tree][n];
        } else {
            for (int k = threadIdx.x; k < NS; k += NT) steps[k] = p.walk[MB == 1 ? walker : 0][MB == 1 ? k : 0];
        }
    };

    // conv: node n's q and k of key head g, [N][2 DK] bf16, in the slot region
    uint16_t* y_qk = reinterpret_cast<uint16_t*>(smem4);
    if (conv) {
        // The tree conv of every node, for the channels this CTA reads: q and
        // k of key head g and its own rows of v (the arithmetic and bf16
        // rounding of gdn_conv_step in tree mode).  A node's earlier inputs are
        // its nearest ancestors, then the tail.  First every input row and the
        // taps of these channels are copied to shared memory, all copies in
        // flight together (one DRAM round trip, beside the state loads above);
        // then each task (a node and 8 channels) computes from there.
        constexpr int QK8 = 2 * DK / 8, PER = QK8 + ROWS / 8, CW = 8 * PER;
        uint16_t* xs = y_qk + (size_t)p.Nmax * 2 * DK;   // [N + 3][CW]
        uint16_t* ws = xs + ((size_t)p.Nmax + 3) * CW;   // [CW][4]
        const uint16_t* xb = p.x + (size_t)tree * p.Nmax * p.C;
        const uint16_t* tb = p.tail + (size_t)tree * GDN_CONV_W * p.C;
        auto chan = [&](int c) {  // the packed channel of this CTA's vector c
            return c < DK / 8 ? g * DK + 8 * c
                 : c < QK8    ? p.Hk * DK + g * DK + 8 * (c - DK / 8)
                              : 2 * p.Hk * DK + h * p.dv + row0 + 8 * (c - QK8);
        };
        for (int idx = threadIdx.x; idx < (N + 3) * PER; idx += NT) {
            const int r = idx / PER, c = idx % PER;
            const uint16_t* src = r < 3 ? tb + (size_t)(r + 1) * p.C + chan(c) : xb + (size_t)(r - 3) * p.C + chan(c);
            cp_async16(xs + (size_t)r * CW + 8 * c, src);
        }
        for (int idx = threadIdx.x; idx < PER * 4; idx += NT) {  // 8 channels x 4 taps = 4 x 16 bytes
            const int c = idx >> 2, q = idx & 3;
            cp_async16(ws + (size_t)c * 32 + 8 * q, p.w + (size_t)chan(c) * GDN_CONV_W + 8 * q);
        }
        // the gates too, in the same round trip (after the conv they would cost another);
        // and the per-node tables read with a per-node index out of the
        // parameters (constant-cache misses), while the copies are in flight
        for (int n = threadIdx.x; n < N; n += NT) {
            if (!KDA) cp_async4(s_ab + 2 * n, alpha_b + (size_t)n * p.Hv + h);
            cp_async4(s_ab + 2 * n + 1, beta_b + (size_t)n * p.Hv + h);
        }
        if constexpr (KDA) {
            for (int idx = threadIdx.x; idx < N * (DK / 4); idx += NT) {
                const int n = idx / (DK / 4), c4 = idx % (DK / 4);
                cp_async16(s_gate + idx, p.alpha + (((size_t)tree * p.Nmax + n) * p.Hv + h) * DK + 4 * c4);
            }
        }
        for (int n = threadIdx.x; n < N; n += NT)
            s_anc[n] = make_char4(p.anc[tree][n][0], p.anc[tree][n][1], p.anc[tree][n][2], 0);
        stage_steps();
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
        // With a cluster (the CTAs of one key head: its value heads' row
        // blocks), the q/k outputs are computed once per cluster: task j goes
        // to CTA j mod csize, which stores the result into every CTA's y_qk.
        // The first cluster barrier also makes sure every CTA of the cluster
        // is running before any remote store.  A walker (no cluster) computes
        // the outputs of its own walk's nodes only.
        const int csize = p.cluster;
        const uint32_t rank = csize > 1 ? cluster_rank() : 0u;
        if (csize > 1) cluster_sync_all();
        else __syncthreads();
        // staged row of input a: a node (a >= 0) or tail slot -1 - a (1 .. 3)
        auto row_of = [&](int a) { return a >= 0 ? a + 3 : -2 - a; };
        // vector c of node n: c < QK8 a q/k vector, else one of this CTA's v vectors
        auto conv_task = [&](int n, int c) -> uint4 {
            float w[8][4];
            load_taps8(ws + (size_t)c * 32, w);
            const char4 a4 = s_anc[n];
            const int anc[3] = {a4.x, a4.y, a4.z};
            const uint16_t* xc = xs + 8 * c;
            const Vec8 u3 = load8(xc + (size_t)(n + 3) * CW);
            const Vec8 u2 = load8(xc + (size_t)row_of(anc[0]) * CW);
            const Vec8 u1 = load8(xc + (size_t)row_of(anc[1]) * CW);
            const Vec8 u0 = load8(xc + (size_t)row_of(anc[2]) * CW);
            return conv8_bf16(w, u0, u1, u2, u3);
        };
        if (W > 1) {
            // a walker needs the conv outputs of its own walk's nodes only:
            // its range and the ancestors it replays
            for (int idx = threadIdx.x; idx < NS * PER; idx += NT) {
                const int i = idx / PER, c = idx % PER;
                const int n = steps[i].node;
                const uint4 y = conv_task(n, c);
                if (c < QK8) *reinterpret_cast<uint4*>(y_qk + (size_t)n * 2 * DK + 8 * c) = y;
                else *reinterpret_cast<uint4*>(s_v + (size_t)n * ROWS + 8 * (c - QK8)) = y;
            }
        }
        const int n_qk = W > 1 ? 0 : N * QK8;  // q/k tasks of the tree
        for (int t = threadIdx.x; t * csize + (int)rank < n_qk; t += NT) {
            const int j = t * csize + (int)rank;
            const int n = j / QK8, c = j % QK8;
            const uint4 y = conv_task(n, c);
            uint16_t* dst = y_qk + (size_t)n * 2 * DK + 8 * c;
            if (csize > 1) {
                for (int r = 0; r < csize; ++r) st_cluster16(dst, (uint32_t)r, y);
            } else {
                *reinterpret_cast<uint4*>(dst) = y;
            }
        }
        if (W == 1) {
            for (int idx = threadIdx.x; idx < N * (ROWS / 8); idx += NT) {
                const int n = idx / (ROWS / 8), c = idx % (ROWS / 8);
                *reinterpret_cast<uint4*>(s_v + (size_t)n * ROWS + 8 * c) = conv_task(n, QK8 + c);
            }
        }
        // every CTA's y_qk is complete (and no remote store is still to come:
        // a CTA may leave the cluster only after this point)
        if (csize > 1) cluster_sync_all();
    } else {
        // Post-conv inputs: the key head's q and k rows of every node (into
        // y_qk, as the fused conv leaves them), this CTA's v rows, the gates
        // and (KDA) the decay vectors, all copies in flight together beside
        // the state loads: one DRAM round trip before the records.
        constexpr int QK8 = 2 * DK / 8;
        for (int idx = threadIdx.x; idx < N * QK8; idx += NT) {
            const int n = idx / QK8, c = idx % QK8;
            const size_t ch = c < DK / 8 ? (size_t)g * DK + 8 * c : (size_t)p.Hk * DK + g * DK + 8 * (c - DK / 8);
            cp_async16(y_qk + (size_t)n * 2 * DK + 8 * c, qkv + (size_t)n * p.C + ch);
        }
        for (int idx = threadIdx.x; idx < N * (ROWS / 8); idx += NT) {
            const int n = idx / (ROWS / 8), c = idx % (ROWS / 8);
            cp_async16(s_v + (size_t)n * ROWS + c * 8,
                       qkv + (size_t)n * p.C + (size_t)2 * p.Hk * DK + (size_t)h * p.dv + row0 + c * 8);
        }
        for (int n = threadIdx.x; n < N; n += NT) {
            if (!KDA) cp_async4(s_ab + 2 * n, alpha_b + (size_t)n * p.Hv + h);
            cp_async4(s_ab + 2 * n + 1, beta_b + (size_t)n * p.Hv + h);
        }
        if constexpr (KDA) {
            for (int idx = threadIdx.x; idx < N * (DK / 4); idx += NT) {
                const int n = idx / (DK / 4), c4 = idx % (DK / 4);
                cp_async16(s_gate + idx, p.alpha + (((size_t)tree * p.Nmax + n) * p.Hv + h) * DK + 4 * c4);
            }
        }
        stage_steps();
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
    }
    __syncthreads();

    const bool normalize = p.normalize != 0;
    const bool out_bf16 = p.out_bf16 != 0;
    // The key-head vectors do not depend on the state: row group n computes
    // node n's with the same token_kq every decode row group runs (so the bits
    // match decode), and the walk reads them back.
    // token_kq reduces with full-warp shuffles, so the loop is warp-uniform:
    // all four row groups of a warp iterate together (on a clamped node when
    // they run past N) and only the groups with a real node write.
    // (a walker: the records of its own walk's nodes only)
    const int NR = W > 1 ? NS : N;
    for (int i0 = rg & ~3; i0 < NR; i0 += kRowsPerPass) {
        const int i = i0 + (rg & 3);
        const bool real = i < NR;
        TokenKQ<V> t;
        const int ic = real ? i : NR - 1;
        const int n = W > 1 ? (int)steps[ic].node : ic;
        const uint16_t* yn = y_qk + (size_t)n * 2 * DK;
        token_kq<V>(yn, yn + DK, lane8, p.q_scale, normalize, t);
        if (real) {
            float4* rec = s_kq + (size_t)n * KQ_REC + lane8;
#pragma unroll
            for (int m = 0; m < V; ++m) {
                rec[8 * m] = make_float4(t.k[m][0], t.k[m][1], t.k[m][2], t.k[m][3]);
                rec[8 * (V + m)] = make_float4(t.q[m][0], t.q[m][1], t.q[m][2], t.q[m][3]);
            }
            if (lane8 == 0) s_kq[(size_t)n * KQ_REC + 8 * 2 * V] = make_float4(t.kq, 0.f, 0.f, 0.f);
        }
    }
    __syncthreads();
    auto fetch = [&](int n, TokenKQ<V>& t) {
        const float4* rec = s_kq + (size_t)n * KQ_REC + lane8;
#pragma unroll
        for (int m = 0; m < V; ++m) {
            const float4 a = rec[8 * m], b = rec[8 * (V + m)];
            t.k[m][0] = a.x; t.k[m][1] = a.y; t.k[m][2] = a.z; t.k[m][3] = a.w;
            t.q[m][0] = b.x; t.q[m][1] = b.y; t.q[m][2] = b.z; t.q[m][3] = b.w;
        }
        t.kq = s_kq[(size_t)n * KQ_REC + 8 * 2 * V].x;
    };
    // one step of the walk on the node record `cur`, fetching the next
    // step's record into `nxt` (the loop below alternates the two, so no
    // record is copied between steps)
    auto slot_at = [&](int slot, int r, int m) -> float4& {
        return slots[(((slot * R + r) * kRowsPerPass + rg) * V + m) * 8 + lane8];
    };
    uint32_t tm_warp = 0;  // this warp's first slot column block (lane quarter, column half)
    if (tm) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const int warp = threadIdx.x >> 5;
        tm_warp = *s_tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((warp >> 2) * 4 * R * V);
    }
    constexpr uint32_t kSlotCols = 8 * R * V;
    const TreeStep* my_steps = steps;
    auto walk_step = [&](int step, const TokenKQ<V>& cur, TokenKQ<V>& nxt) {
        const TreeStep st = my_steps[step];
        if (st.restore >= 0) {
            if (tm) {
                tmem_get_rows<R, V>(tm_warp + (uint32_t)st.restore * kSlotCols, s);
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int m = 0; m < V; ++m) s[r][m] = slot_at(st.restore, r, m);
            }
        }
        const int node = st.node;
        if (step + 1 < NS) fetch(my_steps[step + 1].node, nxt);
        const float beta = s_ab[2 * node + 1];
        float o[R];
        if constexpr (KDA) {
            float4 gv[V];
            load_gate_smem<V>(s_gate + (size_t)node * (DK / 4), lane8, gv);
#pragma unroll
            for (int r = 0; r < R; ++r) kda_decay<V>(s[r], gv);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float v_i = __uint_as_float((uint32_t)s_v[(size_t)node * ROWS + kRowsPerPass * r + rg] << 16);
                o[r] = delta_row_step<V>(s[r], cur, v_i, beta);
            }
        } else {
            const float alpha = s_ab[2 * node];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float v_i = __uint_as_float((uint32_t)s_v[(size_t)node * ROWS + kRowsPerPass * r + rg] << 16);
                o[r] = row_step<V>(s[r], cur, v_i, alpha, beta);
            }
        }
        // lane r of a row group stores row r's output (every lane holds the same bits)
        float my_o = o[0];
#pragma unroll
        for (int r = 1; r < R; ++r)
            if (lane8 == r) my_o = o[r];
        if (lane8 < R && st.store)
            store_out(p.out, (((size_t)tree * p.Nmax + node) * p.Hv + h) * p.dv + row + kRowsPerPass * lane8, my_o,
                      out_bf16);
        if (st.save >= 0) {
            if (tm) {
                tmem_put_rows<R, V>(tm_warp + (uint32_t)st.save * kSlotCols, s);
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int m = 0; m < V; ++m) slot_at(st.save, r, m) = s[r][m];
            }
        }
    };
    TokenKQ<V> ka, kb;
    fetch(my_steps[0].node, ka);
    for (int step = 0; step < NS; step += 2) {
        walk_step(step, ka, kb);
        if (step + 1 < NS) walk_step(step + 1, kb, ka);
    }
    if (tm) {  // every thread's TMEM stores done, then warp 0 frees the columns
        asm volatile("tcgen05.wait::st.sync.aligned;\n\ttcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        if (threadIdx.x < 32) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(*s_tmem), "r"((uint32_t)p.tmem_cols)
                         : "memory");
        }
    }
}

// Fused conv + decode.  A CTA owns one key-head group (its q and k channels
// and the v channels of the group's value heads) of one sequence, and 32*R
// rows of each of the group's value heads it runs: all of them, or one each
// when the heads are split over CTAs (head_parts = group) to widen the grid of
// a small batch.  It runs the conv for all of the group's channels into shared
// memory (rounded to bf16 exactly as gdn_conv_step stores it), then advances
// its value heads' rows through the T tokens with the shared step.  Every tail
// entry is written by one CTA only (row block 0 of head part 0); with several
// row blocks or head parts the tail is read from tail_in and written to a
// distinct tail_out, so no CTA reads an entry another CTA has overwritten.
// KIND 0: the step as it is; 1: KDA (a decay per key channel); 2: the layer
// step -- gates computed from the token's projections in front, and the
// gated RMS norm of each head's output after (the CTA holds all the head's
// rows: one value-row block).
template <int DK, int R, int KIND>
__global__ void __launch_bounds__(kThreads, 2)
gdn_conv_decode_kernel(const __grid_constant__ ConvDecodeParams p) {
    constexpr bool KDA = KIND == 1;
    constexpr bool LAYER = KIND == 2;
    constexpr int V = DK / 32;
    extern __shared__ uint4 smem_y[];
    uint16_t* ys = reinterpret_cast<uint16_t*>(smem_y);  // [T][CC] bf16 conv outputs
    // KDA: the group's decay vectors [T][group][DK] fp32, after the conv outputs
    float4* gs = reinterpret_cast<float4*>(ys + (size_t)p.T * p.CC);
    const int lane8 = threadIdx.x & 7;
    const int rg = threadIdx.x >> 3;
    // blockIdx.x = (group g, head part hp, row block rb); a head part runs
    // group / head_parts of the group's value heads
    const int g = blockIdx.x / (p.head_parts * p.row_blocks);
    const int hp = (blockIdx.x / p.row_blocks) % p.head_parts;
    const int rb = blockIdx.x % p.row_blocks;
    const int nh = p.group / p.head_parts;
    const int j0 = hp * nh;
    const int b = blockIdx.y;
    const size_t C = (size_t)p.C;
    const int CC = p.CC;
    const int row0 = rb * (kRowsPerPass * R) + rg;
    auto state_of = [&](int j) { return p.state + ((size_t)b * p.Hv + g * p.group + j) * (size_t)p.dv * DK; };

    // Launched as a programmatic dependent of the previous kernel on the
    // stream: this grid's CTAs may be placed while that kernel drains.  Each
    // lets the next kernel launch in turn, then waits for the previous one to
    // complete (and its writes to be visible) before it touches any memory.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // the next head's state rows, prefetched by each thread into its own slots
    // (not in the layer step, whose per-head norm barrier already overlaps the
    // next head's loads, and which measured slower with it)
    const bool prefetch = !LAYER && nh > 1;
    float4* s_pref = reinterpret_cast<float4*>(
        reinterpret_cast<uint8_t*>(smem_y) +
        align16((size_t)p.T * p.CC * 2 + (KDA ? (size_t)p.T * p.group * DK * 4 : 0) + (LAYER ? (size_t)p.T * p.group * 8 : 0)));
    auto prefetch_head = [&](int j) {
        const float* S = state_of(j);
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < V; ++m) {
                const uint32_t dst = (uint32_t)__cvta_generic_to_shared(s_pref + (size_t)(r * V + m) * kThreads + threadIdx.x);
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
                             "l"(S + (size_t)(row0 + kRowsPerPass * r) * DK + 32 * m + 4 * lane8)
                             : "memory");
            }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    // The first value head's state rows are requested before the conv, so that
    // their DRAM round trip overlaps the conv inputs' instead of following it:
    // into registers with one row per thread (small batches), else, for the
    // plain step, into the prefetch slots (several heads per CTA: no registers
    // held across the conv; batch 64: 69.28 -> 68.97 us a layer; the KDA step,
    // whose decay vectors are also loaded before the conv, measured no gain).
    constexpr bool kEarlyState = R == 1;
    const bool early_slots = !kEarlyState && KIND == 0 && prefetch;
    if (early_slots) prefetch_head(j0);
    float4 s_first[kEarlyState ? 1 : R][V];
    if constexpr (kEarlyState) {
        const float* S = state_of(j0);
#pragma unroll
        for (int m = 0; m < V; ++m)
            s_first[0][m] = __ldcs(reinterpret_cast<const float4*>(S + (size_t)row0 * DK + 32 * m + 4 * lane8));
    }

    // KDA: the group's decay vectors [T][group][DK] go to shared memory after
    // the conv outputs; the first kThreads float4s are loaded before the conv
    // so that their latency overlaps it.
    constexpr int G4 = DK / 4;  // float4s of one decay vector
    const int n_gate4 = KDA ? p.T * p.group * G4 : 0;
    auto gate_src = [&](int idx) {
        const int tj = idx / G4, c4 = idx % G4;
        const int t = tj / p.group, j = tj % p.group;
        return reinterpret_cast<const float4*>(p.alpha + (((size_t)b * p.T + t) * p.Hv + g * p.group + j) * DK) + c4;
    };
    float4 gate_first = make_float4(0.f, 0.f, 0.f, 0.f);
    if (KDA && threadIdx.x < n_gate4) gate_first = __ldg(gate_src(threadIdx.x));

    // ---- conv of this group's channels (8 per thread)
    for (int cv = threadIdx.x; cv < CC / 8; cv += kThreads) {
        const int c = cv * 8;
        const int gc = c < DK ? g * DK + c
                     : c < 2 * DK ? p.Hk * DK + g * DK + (c - DK)
                     : 2 * p.Hk * DK + g * p.group * p.dv + (c - 2 * DK);
        float w[8][4];
        load_taps8(p.w + (size_t)gc * GDN_CONV_W, w);
        const uint16_t* tb = p.tail_in + (size_t)b * GDN_CONV_W * C + gc;
        const uint16_t* xb = p.x + (size_t)b * p.T * C + gc;
        // tail[0] is shifted out by the first token (T >= 1), so it is not read
        Vec8 h1 = load8(tb + C), h2 = load8(tb + 2 * C), h3 = load8(tb + 3 * C);
        Vec8 h0 = h1;
        for (int t = 0; t < p.T; ++t) {
            h0 = h1;
            h1 = h2;
            h2 = h3;
            h3 = load8(xb + (size_t)t * C);
            store_y(ys + (size_t)t * CC + c, w, h0, h1, h2, h3);
        }
        if (rb == 0 && hp == 0) {
            uint16_t* to = p.tail_out + (size_t)b * GDN_CONV_W * C + gc;
            put8(to, h0);
            put8(to + C, h1);
            put8(to + 2 * C, h2);
            put8(to + 3 * C, h3);
        }
    }
    if constexpr (KDA) {
        if (threadIdx.x < n_gate4) gs[threadIdx.x] = gate_first;
        for (int idx = threadIdx.x + kThreads; idx < n_gate4; idx += kThreads) gs[idx] = __ldg(gate_src(idx));
    }
    // layer: the group's (alpha, beta) per token and head, [T][group], computed once
    float2* s_ab = reinterpret_cast<float2*>(ys + (size_t)p.T * p.CC);
    if constexpr (LAYER) {
        for (int idx = threadIdx.x; idx < p.T * p.group; idx += kThreads) {
            const int t = idx / p.group, h = g * p.group + idx % p.group;
            const size_t ti = ((size_t)b * p.T + t) * p.Hv + h;
            float al, be;
            gate_pair(bf16_bits_to_float(p.layer.a[ti]), bf16_bits_to_float(p.layer.b[ti]), p.layer.A_log[h],
                      p.layer.dt_bias[h], al, be);
            s_ab[idx] = make_float2(al, be);
        }
    }
    // the row this lane writes outputs for: lane l < R of a row group takes
    // row r = l (every lane of the group holds the same o bits)
    const int my_row = row0 + kRowsPerPass * (lane8 < R ? lane8 : 0);
    float my_w = 0.0f;
    if constexpr (LAYER) my_w = p.layer.norm_w[my_row];
    __syncthreads();

    // ---- the group's value heads, one after another
    const bool normalize = p.normalize != 0;
    const bool out_bf16 = p.out_bf16 != 0;
    // layer: per-warp sums of o^2 (two buffers).  A head's norm needs every
    // warp's sum, i.e. a barrier; the last token's epilogue is deferred until
    // the next head's state loads are in flight, so that the barrier wait
    // overlaps them.
    __shared__ float red[LAYER ? 2 : 1][kThreads / 32];
    int red_buf = 0;
    bool pend = false;      // an epilogue waiting for its barrier
    float pend_o = 0.0f;    // this lane's o for it
    size_t pend_at = 0;     // where its y goes
    int pend_buf = 0;
    auto finish_pending = [&]() {
        __syncthreads();
        float tot = red[pend_buf][0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) tot = __fadd_rn(tot, red[pend_buf][w]);
        const float inv_rms = rsqrtf(__fadd_rn(__fmul_rn(tot, 1.0f / (float)(kRowsPerPass * R)), p.layer.norm_eps));
        if (lane8 < R) {
            const float yv = gated_norm_out(pend_o, inv_rms, my_w, bf16_bits_to_float(p.layer.z[pend_at]));
            reinterpret_cast<__nv_bfloat16*>(p.layer.y)[pend_at] = __float2bfloat16_rn(yv);
        }
        pend = false;
    };
    for (int j = j0; j < j0 + nh; ++j) {
        const int h = g * p.group + j;
        float* S = state_of(j);
        float4 s[R][V];
        if (kEarlyState && j == j0) {
#pragma unroll
            for (int m = 0; m < V; ++m) s[0][m] = s_first[0][m];
        } else if (prefetch && (j > j0 || early_slots)) {
            // this thread's own copies of head j (issued during head j - 1, or
            // before the conv for the first head)
            asm volatile("cp.async.wait_all;" ::: "memory");
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < V; ++m) s[r][m] = s_pref[(size_t)(r * V + m) * kThreads + threadIdx.x];
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < V; ++m)
                    s[r][m] = __ldcs(reinterpret_cast<const float4*>(
                        S + (size_t)(row0 + kRowsPerPass * r) * DK + 32 * m + 4 * lane8));
        }
        if (prefetch && j + 1 < j0 + nh) prefetch_head(j + 1);
        if constexpr (LAYER) {
            if (pend) finish_pending();  // the previous head's last token, behind these loads
        }
        for (int t = 0; t < p.T; ++t) {
            const uint16_t* yt = ys + (size_t)t * CC;
            TokenKQ<V> kq;
            token_kq<V>(yt, yt + DK, lane8, p.q_scale, normalize, kq);
            const size_t trow = (size_t)b * p.T + t;
            float alpha = 0.0f, beta;
            if constexpr (LAYER) {
                const float2 ab = s_ab[t * p.group + j];
                alpha = ab.x;
                beta = ab.y;
            } else {
                if constexpr (!KDA) alpha = p.alpha[trow * p.Hv + h];
                beta = p.beta[trow * p.Hv + h];
            }
            const uint16_t* vrow = yt + 2 * DK + j * p.dv;
            if constexpr (KDA) {
                float4 g[V];
                load_gate_smem<V>(gs + ((size_t)t * p.group + j) * (DK / 4), lane8, g);
#pragma unroll
                for (int r = 0; r < R; ++r) kda_decay<V>(s[r], g);
            }
            float o_r[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int i = row0 + kRowsPerPass * r;
                const float v_i = __uint_as_float((uint32_t)vrow[i] << 16);
                float o;
                if constexpr (KDA) o = delta_row_step<V>(s[r], kq, v_i, beta);
                else o = row_step<V>(s[r], kq, v_i, alpha, beta);
                o_r[r] = o;
            }
            float my_o = o_r[0];
#pragma unroll
            for (int r = 1; r < R; ++r)
                if (lane8 == r) my_o = o_r[r];  // compile-time indices: o_r stays in registers
            if (p.out != nullptr && lane8 < R) store_out(p.out, ((trow * p.Hv) + h) * p.dv + my_row, my_o, out_bf16);
            if constexpr (LAYER) {
                // mean of o^2 over the head's dv rows: this thread's rows in
                // order, the warp's four row groups (xor butterfly: the same
                // bits in every lane), then the eight warps in order
                float ss = __fmul_rn(o_r[0], o_r[0]);
#pragma unroll
                for (int r = 1; r < R; ++r) ss = __fmaf_rn(o_r[r], o_r[r], ss);
                ss = __fadd_rn(ss, __shfl_xor_sync(kFullMask, ss, 8));
                ss = __fadd_rn(ss, __shfl_xor_sync(kFullMask, ss, 16));
                if ((threadIdx.x & 31) == 0) red[red_buf][threadIdx.x >> 5] = ss;
                pend = true;
                pend_o = my_o;
                pend_at = ((trow * p.Hv) + h) * p.dv + my_row;
                pend_buf = red_buf;
                red_buf ^= 1;
                if (t + 1 < p.T) finish_pending();  // nothing to overlap within a head's tokens
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < V; ++m)
                __stcs(reinterpret_cast<float4*>(S + (size_t)(row0 + kRowsPerPass * r) * DK + 32 * m + 4 * lane8),
                       s[r][m]);
    }
    if constexpr (LAYER) {
        if (pend) finish_pending();
    }
}

template <int DK, int R, int KIND>
static cudaError_t launch_conv_decode_t(const ConvDecodeParams& p, cudaStream_t s) {
    dim3 grid(p.Hk * p.head_parts * p.row_blocks, p.B, 1);
    const bool prefetch = KIND != 2 && p.group / p.head_parts > 1;
    const size_t smem = align16((size_t)p.T * p.CC * 2 + (KIND == 1 ? (size_t)p.T * p.group * DK * 4 : 0) +
                                (KIND == 2 ? (size_t)p.T * p.group * 8 : 0)) +
                        (prefetch ? conv_decode_prefetch_bytes<DK, R>() : 0);
    // above 48 KB the kernel's dynamic shared memory must be opted into (to
    // what this launch needs: the opt-in limit counts its static memory too);
    // the per-device record of what was opted into is shared by host threads
    if (smem > 48 * 1024) {
        static std::mutex mu;
        static size_t opted[64] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lock(mu);
        if (smem > opted[dev]) {
            e = cudaFuncSetAttribute(gdn_conv_decode_kernel<DK, R, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem);
            if (e != cudaSuccess) return e;
            opted[dev] = smem;
        }
    }
    // a programmatic dependent launch (see the kernel): consecutive layer
    // steps overlap one's start with the other's drain
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gdn_conv_decode_kernel<DK, R, KIND>, p);
}

template <int DK, int KIND>
static cudaError_t launch_conv_decode_r(const ConvDecodeParams& p, int rows_per_cta, cudaStream_t s) {
    switch (rows_per_cta) {
        case 32: return launch_conv_decode_t<DK, 1, KIND>(p, s);
        case 64: return launch_conv_decode_t<DK, 2, KIND>(p, s);
        case 128: return launch_conv_decode_t<DK, 4, KIND>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int KIND>
static cudaError_t launch_conv_decode_k(const ConvDecodeParams& p, int dk, int rows_per_cta, cudaStream_t s) {
    switch (dk) {
        case 32: return launch_conv_decode_r<32, KIND>(p, rows_per_cta, s);
        case 64: return launch_conv_decode_r<64, KIND>(p, rows_per_cta, s);
        case 128: return launch_conv_decode_r<128, KIND>(p, rows_per_cta, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_conv_decode(const ConvDecodeParams& p, int dk, int rows_per_cta, int kind, cudaStream_t s) {
    switch (kind) {
        case 0: return launch_conv_decode_k<0>(p, dk, rows_per_cta, s);
        case 1: return launch_conv_decode_k<1>(p, dk, rows_per_cta, s);
        case 2: return launch_conv_decode_k<2>(p, dk, rows_per_cta, s);
    }
    return cudaErrorInvalidValue;
}

// Gates from projections for n tokens x Hv heads (one thread per pair).
__global__ void __launch_bounds__(kThreads) gdn_gates_kernel(const __grid_constant__ GatesParams p) {
    const int64_t idx = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (idx >= p.n * p.Hv) return;
    const int h = (int)(idx % p.Hv);
    float alpha, beta;
    gate_pair(bf16_bits_to_float(p.a[idx]), bf16_bits_to_float(p.b[idx]), p.A_log[h], p.dt_bias[h], alpha, beta);
    p.alpha[idx] = alpha;
    p.beta[idx] = beta;
}

cudaError_t launch_gates(const GatesParams& p, cudaStream_t s) {
    const int64_t n = p.n * p.Hv;
    const unsigned blocks = (unsigned)((n + kThreads - 1) / kThreads);
    gdn_gates_kernel<<<blocks, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

template <int DK, int R, bool GATHER, bool KDA, typename In>
static cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t s) {
    dim3 grid(p.dv / (kRowsPerPass * R), p.Hv, p.B);
    gdn_decode_kernel<DK, R, GATHER, KDA, In><<<grid, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

template <int DK, bool GATHER, bool KDA, typename In>
static cudaError_t launch_decode_r(const DecodeParams& p, int rows_per_cta, cudaStream_t s) {
    switch (rows_per_cta) {
        case 32: return launch_decode_t<DK, 1, GATHER, KDA, In>(p, s);
        case 64: return launch_decode_t<DK, 2, GATHER, KDA, In>(p, s);
        case 128: return launch_decode_t<DK, 4, GATHER, KDA, In>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

template <bool GATHER, bool KDA, typename In = uint16_t>
static cudaError_t launch_decode_k(const DecodeParams& p, int dk, int rows_per_cta, cudaStream_t s) {
    switch (dk) {
        case 32: return launch_decode_r<32, GATHER, KDA, In>(p, rows_per_cta, s);
        case 64: return launch_decode_r<64, GATHER, KDA, In>(p, rows_per_cta, s);
        case 128: return launch_decode_r<128, GATHER, KDA, In>(p, rows_per_cta, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeParams& p, int dk, int rows_per_cta, int gather, bool kda, bool in_f32,
                          cudaStream_t s) {
    // fp32 activations: the plain step only (the host refuses other combinations)
    if (in_f32) return (gather || kda) ? cudaErrorInvalidValue : launch_decode_k<false, false, float>(p, dk, rows_per_cta, s);
    // commit (gather) replays short paths: one row pass per CTA keeps the grid wide
    if (gather) return kda ? launch_decode_k<true, true>(p, dk, rows_per_cta, s)
                           : launch_decode_k<true, false>(p, dk, rows_per_cta, s);
    return kda ? launch_decode_k<false, true>(p, dk, rows_per_cta, s)
               : launch_decode_k<false, false>(p, dk, rows_per_cta, s);
}

template <int DK, int R>
static size_t tree_smem_bytes(int n_slots, int N, bool conv, bool kda) {
    // + the word for the tensor-memory address
    return tree_slot_bytes<DK, R>(n_slots, N, conv) + tree_stage_bytes<DK, R>(N) + (kda ? (size_t)N * DK * 4 : 0) + 16;
}

// Tensor-memory columns for n_slots branch slots (8 R V each, allocated in a
// power of two of at least 32), or 0 to keep them in shared memory: more
// than 256 columns would leave no room for a second CTA on the SM.
template <int DK, int R>
static int tree_tmem_cols(int n_slots) {
    if (n_slots <= 0) return 0;
    const int need = n_slots * 8 * R * (DK / 32);
    int cols = 32;
    while (cols < need) cols *= 2;
    return cols <= 256 ? cols : 0;
}

// Shared memory of a launch whose slots go to tensor memory when they fit.
template <int DK, int R>
static size_t tree_smem_bytes_tm(int n_slots, int N, bool conv, bool kda) {
    return tree_smem_bytes<DK, R>(tree_tmem_cols<DK, R>(n_slots) > 0 ? 0 : n_slots, N, conv, kda);
}

template <int DK, int MB, int R, bool KDA>
static cudaError_t launch_tree_t(TreeParamsT<MB>& p, cudaStream_t s) {
    constexpr int ROWS = kRowsPerPass * R;
    const int W = MB == 1 ? p.walkers : 1;
    const int n_slots = W == 1 ? p.n_slots : p.walk_slots;
    p.tmem_cols = tree_tmem_cols<DK, R>(n_slots);
    const size_t smem = tree_smem_bytes_tm<DK, R>(n_slots, p.Nmax, p.x != nullptr, KDA);
    // the shared-memory opt-in, once per device whatever the host threads
    static std::once_flag once[64];
    static cudaError_t setup_err[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev] {
        const int max_smem = std::min((int)tree_smem_bytes<DK, R>(GDN_MAX_TREE_SLOTS, GDN_MAX_TREE_NODES, true, KDA),
                                      kMaxSmemPerCta);
        setup_err[dev] = cudaFuncSetAttribute(gdn_tree_kernel<DK, MB, R, KDA>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    });
    if (setup_err[dev] != cudaSuccess) return setup_err[dev];
    dim3 grid(p.dv / ROWS, p.Hv, MB == 1 ? W : p.B);
    // The fused conv shares each key head's q/k conv among the CTAs that read
    // it -- the row blocks of its value heads, adjacent in the grid -- as one
    // thread-block cluster (at most the portable 8 CTAs).  Walkers run
    // without one: each computes only its own walk's nodes, which measured
    // faster than sharing all of a row block's conv in clusters of three.  If
    // the cluster cannot be placed, the launch falls back to one CTA per
    // cluster.
    const int cx = p.dv / ROWS, cy = p.group;
    const int csize = cx * cy;
    if (p.x != nullptr && csize > 1 && csize <= 8 && W == 1) {
        p.cluster = csize;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)cx;
        attr[0].val.clusterDim.y = (unsigned)cy;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, gdn_tree_kernel<DK, MB, R, KDA>, p) == cudaSuccess) return cudaSuccess;
        (void)cudaGetLastError();  // a configuration error, not sticky: take the plain launch
    }
    p.cluster = 1;
    gdn_tree_kernel<DK, MB, R, KDA><<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

// Rows per thread: 2 when the value head has a multiple of 64 rows and the
// slots for them fit in shared memory (each node's record then serves two
// rows per fetch), else 1.
// Walkers (one tree): when the host split the tree, the value head has a
// multiple of 64 rows, and two CTAs fit on an SM (registers: the launch
// bounds; shared memory: the walkers' slots and staging), so that the grid
// of W x row blocks x heads CTAs runs in one wave.
template <int DK, int MB, bool KDA>
static cudaError_t launch_tree_r(TreeParamsT<MB>& p, cudaStream_t s) {
    if constexpr (MB == 1) {
        if (p.walkers > 1) {
            const bool fits = p.dv % (2 * kRowsPerPass) == 0 &&
                              (p.dv / (2 * kRowsPerPass)) * p.Hv * p.walkers <= 2 * device_sm_count() &&
                              tree_smem_bytes_tm<DK, 2>(p.walk_slots, p.Nmax, p.x != nullptr, KDA) <= kSmemTwoCtas;
            if (fits) return launch_tree_t<DK, MB, 2, KDA>(p, s);
            p.walkers = 1;
        }
    }
    const size_t smem2 = tree_smem_bytes_tm<DK, 2>(p.n_slots, p.Nmax, p.x != nullptr, KDA);
    if (p.dv % (2 * kRowsPerPass) == 0 && smem2 <= (size_t)kMaxSmemPerCta) return launch_tree_t<DK, MB, 2, KDA>(p, s);
    return launch_tree_t<DK, MB, 1, KDA>(p, s);
}

template <int MB>
cudaError_t launch_tree(TreeParamsT<MB>& p, int dk, cudaStream_t s) {
    if (p.kda) {
        switch (dk) {
            case 32: return launch_tree_r<32, MB, true>(p, s);
            case 64: return launch_tree_r<64, MB, true>(p, s);
            case 128: return launch_tree_r<128, MB, true>(p, s);
        }
        return cudaErrorInvalidValue;
    }
    switch (dk) {
        case 32: return launch_tree_r<32, MB, false>(p, s);
        case 64: return launch_tree_r<64, MB, false>(p, s);
        case 128: return launch_tree_r<128, MB, false>(p, s);
    }
    return cudaErrorInvalidValue;
}
template cudaError_t launch_tree<1>(TreeParamsT<1>&, int, cudaStream_t);
template cudaError_t launch_tree<kMaxTreeBatch>(TreeParamsT<kMaxTreeBatch>&, int, cudaStream_t);

}  // namespace gdn
