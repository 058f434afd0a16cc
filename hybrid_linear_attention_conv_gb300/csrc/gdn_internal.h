// gdn_internal.h -- launch parameters shared by the host API and the kernels.
// Host validation (gdn_api.cu) fills these; the kernels (gdn_decode.cu,
// gdn_conv.cu, gdn_prefill.cu) consume them.  Nothing here is part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

// Decode / commit: T sequential tokens per sequence, optionally gathered
// through an index map (commit replays a tree path).
struct DecodeParams {
    const uint16_t* qkv;   // bf16 [B, Tsrc, C] (fp32 for the fp32-activation step, cast by the kernel)
    const float* alpha;    // [B, Tsrc, Hv], or [B, Tsrc, Hv, dk] for KDA
    const float* beta;     // [B, Tsrc, Hv]
    float* state;          // [B, Hv, dv, dk]
    void* out;             // [B, T, Hv, dv] or nullptr
    int B, T, Tsrc, Hk, Hv, dv, group;  // group = Hv / Hk
    int C;                 // packed row length
    float q_scale;
    int normalize;
    int out_bf16;
    int32_t tok[GDN_MAX_TREE_NODES];  // gather map when used (commit)
    // commit only: the tree's pre-conv inputs [Tsrc, C] and the conv tail
    // [4, C] to update from them (nullptr: the tail is left alone)
    const uint16_t* x_tree;
    uint16_t* tail;
};

// One step of the tree walk, computed on the host (depth-first preorder).
struct TreeStep {
    int8_t node;      // node processed at this step
    int8_t restore;   // slot holding the parent's state, or -1 (registers)
    int8_t save;      // slot to keep this node's state in, or -1
    int8_t store;     // 1: write the node's output; 0: an ancestor replayed
                      // by the second walker, whose output the first writes
};

constexpr int kMaxWalkers = 3;

// Tree verify over up to MB trees (one per sequence) in one launch.
template <int MB>
struct TreeParamsT {
    const uint16_t* qkv;   // bf16 [B, Nmax, C]
    const float* alpha;    // [B, Nmax, Hv]
    const float* beta;     // [B, Nmax, Hv]
    const float* state;    // [B, Hv, dv, dk] read only
    void* out;             // [B, Nmax, Hv, dv]
    int B, Nmax, Hk, Hv, dv, group, C;
    float q_scale;
    int normalize;
    int out_bf16;
    int n_slots;           // largest number of branch states any tree needs
    int N[MB];             // nodes of tree b
    TreeStep steps[MB][GDN_MAX_TREE_NODES];
    // Fused conv (x != nullptr; qkv unused): the tree conv of the pre-conv
    // inputs runs in the kernel.  anc as in ConvParams, per tree.
    const uint16_t* x;     // bf16 [B, Nmax, C] pre-conv inputs
    const uint16_t* w;     // bf16 [C, 4]
    const uint16_t* tail;  // bf16 [B, 4, C] read only
    int8_t anc[MB][GDN_MAX_TREE_NODES][3];
    int cluster;           // CTAs per thread-block cluster sharing the q/k conv (1: no cluster; set by the launcher)
    int kda;               // a decay per key channel: alpha is [B, Nmax, Hv, dk]
    // Walkers (one tree, walkers > 1): the tree's preorder cut into
    // `walkers` ranges, walker w's CTAs running walk[w][0 .. walk_n[w] - 1]
    // over their rows with branch slots 0 .. walk_slots - 1 of their own.  The
    // launcher takes this schedule instead of steps[0] when the walkers fit
    // (and sets walkers back to 1 when they do not).
    TreeStep walk[MB == 1 ? kMaxWalkers : 1][MB == 1 ? GDN_MAX_TREE_NODES : 1];
    int walk_n[kMaxWalkers];
    int walk_slots;
    int walkers;           // CTAs walking one row block's part of the tree (1 .. kMaxWalkers)
    int tmem_cols;         // > 0: the branch slots live in this many tensor-memory columns (set by the launcher)
};
constexpr int kMaxTreeBatch = 32;
using TreeParams = TreeParamsT<1>;
using TreeParamsBatch = TreeParamsT<kMaxTreeBatch>;

struct ConvParams {
    // bf16 bits, or fp32 for the fp32-activation conv (f32 = 1; cast by the kernel)
    const void* x;         // [B, T, C]
    const void* w;         // [C, 4]
    void* tail;            // [B, 4, C]
    void* y;               // [B, T, C]
    int f32;
    int B, T, C;
    int tree;              // 0: linear run, 1: tree (ancestor table below)
    // tree mode: for node n, source of its m-th earlier input (m = 1..3):
    // >= 0 a node index, < 0 tail slot (-1 - s).
    int8_t anc[GDN_MAX_TREE_NODES][3];
};

// Fused conv + decode: one CTA per (key-head group, row block, sequence).
// The layer step's extra inputs around the mixer (gdn_layer_decode_step).
struct LayerParams {
    const uint16_t* a;       // bf16 [B, T, Hv] decay projection
    const uint16_t* b;       // bf16 [B, T, Hv] write-strength projection
    const float* A_log;      // [Hv]
    const float* dt_bias;    // [Hv]
    const uint16_t* z;       // bf16 [B, T, Hv, dv] output-gate projection
    const float* norm_w;     // [dv]
    uint16_t* y;             // bf16 [B, T, Hv, dv]
    float norm_eps;
};

struct GatesParams {
    const uint16_t* a;
    const uint16_t* b;
    const float* A_log;
    const float* dt_bias;
    float* alpha;            // [n, Hv]
    float* beta;
    int64_t n;               // tokens
    int Hv;
};

struct ConvDecodeParams {
    const uint16_t* x;        // [B, T, C] pre-conv inputs
    const uint16_t* w;        // [C, 4]
    const uint16_t* tail_in;  // [B, 4, C]
    uint16_t* tail_out;       // [B, 4, C] (equal to tail_in when row_blocks == 1)
    const float* alpha;       // [B, T, Hv], or [B, T, Hv, dk] for KDA
    const float* beta;        // [B, T, Hv]
    float* state;             // [B, Hv, dv, dk]
    void* out;                // [B, T, Hv, dv] or nullptr
    int B, T, Hk, Hv, dv, group, C;
    int CC;                   // channels of one key-head group: 2 dk + group dv
    int row_blocks;           // CTAs along the value rows of one group
    int head_parts;           // CTAs along the value heads of one group (1 or group)
    float q_scale;
    int normalize;
    int out_bf16;
    LayerParams layer;        // the layer step only (gates from projections, gated-norm output)
};

// Commit of the accepted paths of up to kMaxTreeBatch sequences (a joint
// verify's trees) in one launch: sequence b replays path[b][0 .. L[b] - 1] of
// its own tree, and its tail takes the last four inputs of (tail ++ x_tree[path]).
// With w set (the fused conv), the path's conv outputs are computed in the
// kernel from x_tree and tail_in, qkv is unused, and the new tail goes to
// `tail`, a buffer distinct from tail_in (every sequence's, L[b] == 0 too).
struct CommitBatchParams {
    const uint16_t* qkv;     // bf16 [B, N, C] the trees' inputs (post-conv)
    const float* alpha;      // [B, N, Hv]
    const float* beta;       // [B, N, Hv]
    float* state;            // [B, Hv, dv, dk] in place
    const uint16_t* x_tree;  // bf16 [B, N, C] pre-conv inputs, or nullptr (tails untouched)
    uint16_t* tail;          // bf16 [B, 4, C] (in place; the fused conv: written only)
    const uint16_t* w;       // bf16 [C, 4] the fused conv's taps, or nullptr
    const uint16_t* tail_in; // bf16 [B, 4, C] the fused conv's tail before the commit
    int B, N, Hk, Hv, dv, group, C;
    int normalize;
    int32_t L[32];                         // path length of sequence b (0: nothing to commit)
    int8_t path[32][GDN_MAX_TREE_NODES];   // its path, root first (node indices)
};


// Host validation shared by the entry points (gdn_api.cu).  Both record a
// message for gdn_last_error() and return a gdn_status.
int check_prefill_args(const gdn_shape* shape, int T, int chunk, const void* qkv, const void* alpha,
                       const void* beta, const void* state, const void* out, const void* workspace,
                       size_t workspace_bytes, uint32_t flags, bool records = true);
int cuda_error(cudaError_t e, const char* what);
int report_error(int code, const char* fmt, ...);
int check_shape_arg(const gdn_shape* s, bool need_single);  // head sizes, Hv % Hk, grid limits
int check_pointer(const void* p, const char* name);          // non-NULL and 16-byte aligned
int device_sm_count();                                        // SMs of the current device (cached)

// Launchers (return the cudaError_t of the launch).
// kda: a decay per key channel (alpha [.., Hv, dk]) instead of one per head.
// in_f32: the activations (qkv) are fp32 instead of bf16 (plain step only).
cudaError_t launch_decode(const DecodeParams& p, int dk, int rows_per_cta, int gather, bool kda, bool in_f32,
                          cudaStream_t s);
template <int MB>
cudaError_t launch_tree(TreeParamsT<MB>& p, int dk, cudaStream_t s);  // sets p.cluster
// kind: 0 the plain step, 1 KDA, 2 the layer step (gates in front, gated norm after)
cudaError_t launch_conv_decode(const ConvDecodeParams& p, int dk, int rows_per_cta, int kind, cudaStream_t s);
cudaError_t launch_gates(const GatesParams& p, cudaStream_t s);
constexpr int kFusedMaxTokens = 16;
constexpr int kFusedMaxSmem = 48 * 1024;
cudaError_t launch_conv(const ConvParams& p, cudaStream_t s);
cudaError_t launch_commit_batched(const CommitBatchParams& p, int dk, int rows_per_cta, cudaStream_t s);

}  // namespace gdn
