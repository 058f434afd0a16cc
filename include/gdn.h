/*
 * gdn.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet mixer library.
 *
 * The library runs the recurrent mixer of a hybrid DeltaNet/attention decoder on
 * one GPU: the short causal convolution in front of it, decode of one or more
 * tokens, speculative tree verify, commit of the accepted path, and chunked
 * prefill.  Sources for what each call computes:
 *
 *  - Layer and state: TandemLLM "Architecture" (v0.14.2) section 8.1, table of
 *    layer kinds: 48 Gated DeltaNet layers, each keeping per sequence an fp32
 *    state of 48 heads x 128 x 128 (3.15 MB) and a 4-wide convolution tail
 *    (80 KB); the state is fixed-size and has no inverse.
 *  - Recurrence: the pages name "the gated delta rule for one token, a block, a
 *    tree" (TandemLLM "Architecture" v0.11.1, "The parts" diagram) but print no
 *    equation.  The update is the published Gated DeltaNet rule (Yang, Kautz &
 *    Hatamizadeh 2024): per value head h and token t,
 *        S_h <- alpha * S_h (I - beta k k^T) + beta v k^T,   o = S_h q
 *    with q, k the L2-normalised key-head vectors (eps 1e-6) after a 4-tap
 *    causal depthwise convolution + SiLU over the q/k/v channels.
 *  - In-place, constant-size state with no allocation inside the decode loop:
 *    "Serving A Research Architecture On CPU", section on the constant-state
 *    guarantee.  This library never allocates or frees device memory; every
 *    buffer is owned by the caller.
 *  - Tree verify and commit: "Architecture" (v0.14.2) section 8.3 and the
 *    round sequence diagram of v0.11.1: a draft tree of up to 32 nodes is
 *    verified in one pass with each node's state branched from its parent's;
 *    the accepted root-to-node path's state is then committed exactly.
 *  - Refusing unsupported shapes loudly instead of corrupting memory: "Serving
 *    A Research Architecture On CPU", the hardcoded-head-size bug.
 *
 * Conventions for every call
 *  - Tensor pointers are DEVICE pointers to caller-owned, dense, row-major
 *    memory, unless marked "host".  Layouts are given per argument.
 *  - bf16 tensors are raw bfloat16 bit patterns (gdn_bf16).
 *  - Packed activations: one token's row holds C_qkv = 2*Hk*dk + Hv*dv channels
 *    ordered [q | k | v]; q and k are key-head-major (key head g in channels
 *    g*dk .. g*dk+dk-1 of its block), v is value-head-major.
 *  - Value head h reads key head h / (Hv / Hk).
 *  - State S_h is dv x dk fp32, row i contiguous over the key index:
 *    state[b][h][i][j].
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t, NULL = the
 *    legacy default stream).  Host arrays (parents, path) are read before the
 *    call returns and may be reused at once.
 *  - Return value: GDN_OK (0) or a negative gdn_status.  A call that fails
 *    validation enqueues nothing and leaves every buffer untouched.
 *    gdn_last_error() returns a message for the calling thread's last failure.
 *  - Supported shapes: dk, dv in {32, 64, 128}; Hk >= 1; Hv a multiple of Hk;
 *    B >= 0; token counts >= 0 (0 is a no-op).  Device pointers must be 16-byte
 *    aligned (GDN_ERR_MISALIGNED otherwise).
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_ABI_VERSION 1

/* Taps of the causal depthwise convolution; the tail keeps this many inputs. */
#define GDN_CONV_W 4
/* Largest draft tree accepted by tree verify / commit / tree-mode conv. */
#define GDN_MAX_TREE_NODES 64
/* Largest number of branch states a tree verify keeps at once (nested nodes
 * with two or more children on one root path). */
#define GDN_MAX_TREE_SLOTS 8

typedef uint16_t gdn_bf16;

typedef struct gdn_shape {
    int32_t B;   /* sequences in the batch */
    int32_t Hk;  /* key heads (q and k) */
    int32_t Hv;  /* value heads (v, state, output) */
    int32_t dk;  /* key head size: state columns */
    int32_t dv;  /* value head size: state rows */
} gdn_shape;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = -1,       /* null pointer, negative count, bad flag */
    GDN_ERR_UNSUPPORTED_SHAPE = -2, /* head sizes / head counts not supported */
    GDN_ERR_BAD_PARENTS = -3,       /* parent array is not one tree rooted at 0 */
    GDN_ERR_BAD_PATH = -4,          /* path is not a root-to-node path */
    GDN_ERR_DEPTH_EXCEEDED = -5,    /* tree needs more than GDN_MAX_TREE_SLOTS */
    GDN_ERR_MISALIGNED = -6,        /* device pointer not 16-byte aligned */
    GDN_ERR_CUDA = -7,              /* a CUDA runtime call failed */
    GDN_ERR_TIMEOUT = -8,           /* a bounded device wait gave up */
    GDN_ERR_WORKSPACE = -9          /* workspace missing or too small */
} gdn_status;

/* flags */
#define GDN_NORMALIZE_QK 0x1u  /* L2-normalise q and k per key head (eps 1e-6) */
#define GDN_OUT_BF16 0x2u      /* outputs stored as bf16 (RNE) instead of fp32 */
/* gdn_chunk_prefill only: run the pre-pass over all chunks, then the chain,
 * as two launches, even where one cooperative launch would fit (the results
 * are the same bits; for comparisons).  Other entry points refuse it. */
#define GDN_PREFILL_TWO_LAUNCH 0x4u
/* gdn_conv_step and gdn_decode_step only: the activations are fp32 instead
 * of bf16 (conv: x, w, tail and y; decode: qkv), for inputs drawn or kept in
 * fp32.  The arithmetic is the same; nothing is rounded to bf16 on the way.
 * Other entry points refuse it. */
#define GDN_IN_F32 0x8u

/* ABI version of the loaded library (GDN_ABI_VERSION it was built with). */
int gdn_abi_version(void);

/* Message for the calling thread's most recent failed call ("" if none). */
const char* gdn_last_error(void);

/* Bytes of fp32 state for the shape: B * Hv * dv * dk * 4 (0 on a bad shape). */
size_t gdn_state_bytes(const gdn_shape* shape);

/* Host-only tree bookkeeping, the same code the tree calls validate with.
 * Writes the root-to-node path of `node` (root first) into path[0..cap-1] and
 * returns its length, or a negative gdn_status for a bad tree, node or cap. */
int gdn_tree_root_path(int32_t N, const int32_t* parents, int32_t node, int32_t* path,
                       int32_t cap);

/*
 * gdn_conv_step -- 4-tap causal depthwise convolution + SiLU.
 *   y[b,t,c] = SiLU( sum_{j=0..3} w[c][j] * u_j ),   u_3 = x[b,t,c] (newest),
 *   u_{3-m} = the m-th earlier input of that token's history.
 * Linear mode (parents == NULL): the history of token t is x[b,0..t-1] after
 *   tail[b]; on return tail[b] holds the last 4 inputs of (tail[b] ++ x[b]).
 * Tree mode (parents != NULL, host int32[T]; T = N draft nodes): the history
 *   of node n is its ancestors' inputs, nearest first, then tail[b]; the tail
 *   is read only.  All B sequences share the tree.
 *   B, T, C   sequences, tokens (or nodes), channels; C % 8 == 0.
 *   x         bf16 [B, T, C]  pre-conv inputs.
 *   w         bf16 [C, 4]     taps, oldest input first.
 *   tail      bf16 [B, 4, C]  the last four inputs, oldest first (in/out in
 *                             linear mode, read-only in tree mode).
 *   y         bf16 [B, T, C]  output (fp32 math, rounded to nearest even).
 *   flags     0, or GDN_IN_F32: x, w, tail and y are all fp32 (y not rounded).
 * The conv takes its sizes as (B, T, C) rather than a gdn_shape: it is a
 * per-channel operation, and C need not be a packed q/k/v row (C % 8 == 0).
 * Source: the per-layer 4-wide convolution tail, "Architecture" (v0.14.2)
 * section 8.1; short convolution rings carried between steps, "Serving A
 * Research Architecture On CPU" (engine design).
 */
int gdn_conv_step(int32_t B, int32_t T, int32_t C, const int32_t* parents,
                  const void* x, const void* w, void* tail, void* y,
                  uint32_t flags, void* stream);

/*
 * gdn_decode_step -- T sequential tokens of the gated delta rule, in place.
 * For each sequence b, token t, value head h (key head g = h / (Hv/Hk)):
 *   q^ = q_scale * q / |q|,  k^ = k / |k|   (if GDN_NORMALIZE_QK),
 *   S_h <- alpha S_h (I - beta k^ k^T) + beta v k^T,   out = S_h q^.
 * The state is read from HBM once and written once per call, whatever T.
 *   qkv     bf16 [B, T, C_qkv]   packed post-conv activations (fp32 with
 *                                GDN_IN_F32).
 *   alpha   fp32 [B, T, Hv]      decay, beta fp32 [B, T, Hv] write strength.
 *   state   fp32 [B, Hv, dv, dk] in/out.
 *   out     [B, T, Hv, dv] fp32, or bf16 with GDN_OUT_BF16; may be NULL.
 * Source: "Architecture" (v0.11.1) "The parts" (one token, a block);
 * "Architecture" (v0.14.2) section 8.3 (decode without speculation).
 */
int gdn_decode_step(const gdn_shape* shape, int32_t T, const void* qkv,
                    const float* alpha, const float* beta, float* state, void* out,
                    float q_scale, uint32_t flags, void* stream);

/*
 * gdn_conv_decode_step -- gdn_conv_step (linear mode) followed by
 * gdn_decode_step on its output, in one launch: the conv output never
 * reaches HBM.  Results (out, state, the new tail) are identical, bit for
 * bit, to the two separate calls.
 *   T          1 .. 16 tokens per sequence (0 is a no-op); T * (2 dk +
 *              (Hv/Hk) dv) * 2 bytes must not exceed 48 KB.
 *   x          bf16 [B, T, C_qkv] pre-conv inputs (packed [q | k | v]).
 *   w          bf16 [C_qkv, 4] conv taps.
 *   tail_in    bf16 [B, 4, C_qkv] the last four inputs before this call.
 *   tail_out   bf16 [B, 4, C_qkv] receives the last four inputs after it.
 *              It may be tail_in itself (updated in place); a distinct
 *              buffer (ping-pong between calls) lets small batches spread
 *              each head's rows over more CTAs.  Partial overlap is refused.
 *   alpha, beta, state, out, q_scale, flags: as for gdn_decode_step.
 * The launch is a programmatic dependent launch: its CTAs may be placed
 * while the previous kernel on the stream drains, but they touch no memory
 * before that kernel has completed, so stream order is kept (consecutive
 * layer steps overlap one's start with the other's end).
 * Source: the per-layer decode step of "Architecture" (v0.14.2) section 8.1
 * (conv tail + recurrent state per layer) and section 8.3 (decode loop).
 */
int gdn_conv_decode_step(const gdn_shape* shape, int32_t T, const gdn_bf16* x, const gdn_bf16* w,
                         const gdn_bf16* tail_in, gdn_bf16* tail_out, const float* alpha,
                         const float* beta, float* state, void* out, float q_scale, uint32_t flags,
                         void* stream);

/*
 * gdn_kda_decode_step -- gdn_decode_step with a decay per key channel (KDA,
 * Kimi Delta Attention) instead of one per head:
 *   S_h <- (S_h diag(a)) (I - beta k^ k^T) + beta v k^T,   out = S_h q^,
 * with a = alpha[b, t, h, 0 .. dk-1] (column j of S, the j-th key channel,
 * decays by a[j]).  With a[j] equal for all j this is gdn_decode_step's map;
 * rounding differs (the decay is applied before the dot products).
 *   alpha   fp32 [B, T, Hv, dk]; every other argument as for gdn_decode_step.
 * Source: the metrale_model_arch API page lists a KDA mixer with a CPU
 * reference (module index: glm5next_kda, glm5next_kda_ref, kimi_k3) and prints
 * no update rule; the rule above is the gated delta rule of "Architecture"
 * (v0.11.1) "The parts" with its scalar decay made diagonal on the key side.
 */
int gdn_kda_decode_step(const gdn_shape* shape, int32_t T, const gdn_bf16* qkv,
                        const float* alpha, const float* beta, float* state, void* out,
                        float q_scale, uint32_t flags, void* stream);

/*
 * gdn_kda_conv_decode_step -- gdn_conv_decode_step with the KDA step of
 * gdn_kda_decode_step: conv + SiLU, L2-norm and the per-channel-decay delta
 * step in one launch.  Results equal, bit for bit, gdn_conv_step followed by
 * gdn_kda_decode_step.  alpha fp32 [B, T, Hv, dk]; every other argument and
 * limit as for gdn_conv_decode_step.
 */
int gdn_kda_conv_decode_step(const gdn_shape* shape, int32_t T, const gdn_bf16* x,
                             const gdn_bf16* w, const gdn_bf16* tail_in, gdn_bf16* tail_out,
                             const float* alpha, const float* beta, float* state, void* out,
                             float q_scale, uint32_t flags, void* stream);

/*
 * gdn_layer_decode_step -- the layer's whole decode step around the mixer, in
 * one launch: conv + SiLU and L2-norm as in gdn_conv_decode_step, the gates
 * computed from the token's projections, the delta step, and the gated RMS
 * norm of each head's output:
 *   alpha = exp(-exp(A_log[h]) * softplus(a + dt_bias[h])),  beta = sigmoid(b),
 *   o = S_h q^ (after the update),
 *   y_i = o_i / sqrt(mean_i(o_i^2) + norm_eps) * norm_w[i] * SiLU(z_i).
 *   x, conv_w, tail_in, tail_out, state, q_scale, T: as gdn_conv_decode_step
 *               (T * (2 dk + (Hv/Hk) dv) * 2 bytes <= 48 KB).
 *   a, b        bf16 [B, T, Hv] the decay and write-strength projections.
 *   A_log, dt_bias  fp32 [Hv] per-head parameters.
 *   z           bf16 [B, T, Hv, dv] the output-gate projection.
 *   norm_w      fp32 [dv] the norm weight (shared by the heads); norm_eps in [0, 1].
 *   o           fp32 [B, T, Hv, dv] the mixer outputs before the norm, or NULL.
 *   y           bf16 [B, T, Hv, dv] the layer's mixer output.
 *   flags       GDN_NORMALIZE_QK only.
 * o equals, bit for bit, gdn_gates followed by gdn_conv_decode_step.
 * Source: the pages name the layer but print neither the gates nor the
 * output norm ("Architecture" v0.14.2 section 8.1; v0.11.1 "The parts"); both
 * follow the published Gated DeltaNet layer (Yang, Kautz & Hatamizadeh 2024,
 * as shipped with the Qwen3-Next models).
 */
int gdn_layer_decode_step(const gdn_shape* shape, int32_t T, const gdn_bf16* x,
                          const gdn_bf16* conv_w, const gdn_bf16* tail_in, gdn_bf16* tail_out,
                          const gdn_bf16* a, const gdn_bf16* b, const float* A_log,
                          const float* dt_bias, const gdn_bf16* z, const float* norm_w,
                          float norm_eps, float* state, float* o, gdn_bf16* y, float q_scale,
                          uint32_t flags, void* stream);

/*
 * gdn_gates -- the gates of gdn_layer_decode_step alone, for n tokens:
 *   a, b bf16 [n, Hv] -> alpha, beta fp32 [n, Hv] (A_log, dt_bias fp32 [Hv]).
 * Same arithmetic, same bits as inside the layer step.
 */
int gdn_gates(int64_t n, int32_t Hv, const gdn_bf16* a, const gdn_bf16* b, const float* A_log,
              const float* dt_bias, float* alpha, float* beta, void* stream);

/*
 * gdn_tree_verify -- outputs of every node of a draft tree in one pass.
 * Node n's state is the committed state advanced through the root..n path
 * (each node branches from its parent's state); out[n] = S_n q^_n.  The
 * committed state is read once and NOT modified; node states never reach HBM.
 *   shape->B must be 1.  N in [1, GDN_MAX_TREE_NODES].
 *   parents host int32 [N]: parents[0] == -1 (the root follows the committed
 *           state), 0 <= parents[n] < n otherwise.
 *   qkv     bf16 [N, C_qkv]; alpha, beta fp32 [N, Hv].
 *   state   fp32 [Hv, dv, dk] read only.
 *   out     [N, Hv, dv] fp32 (or bf16 with GDN_OUT_BF16).
 * A node's output equals, bit for bit, the output gdn_decode_step gives for
 * the last token of that node's root path (same step arithmetic).
 * Source: "Architecture" (v0.14.2) section 8.3 and the v0.11.1 round diagram
 * (verify the whole tree in one pass, trees of up to 32 nodes).
 */
int gdn_tree_verify(const gdn_shape* shape, int32_t N, const int32_t* parents,
                    const gdn_bf16* qkv, const float* alpha, const float* beta,
                    const float* state, void* out, float q_scale, uint32_t flags,
                    void* stream);

/*
 * gdn_tree_verify_batched -- gdn_tree_verify for B sequences in one launch,
 * each with its own draft tree (own size and shape) and its own state.
 *   shape->B  trees, 1 .. 32.   N  node capacity per tree, 1 .. 64.
 *   counts    host int32 [B]: nodes of tree b, 1 .. N.
 *   parents   host int32 [B, N]: tree b's parent array in parents[b*N ..],
 *             as for gdn_tree_verify; entries past counts[b] are ignored.
 *   qkv       bf16 [B, N, C_qkv]; alpha, beta fp32 [B, N, Hv].
 *   state     fp32 [B, Hv, dv, dk] read only.
 *   out       [B, N, Hv, dv] fp32 (or bf16); rows past counts[b] are not written.
 * Each tree's outputs equal, bit for bit, gdn_tree_verify of that tree alone.
 * Source: "Architecture" (v0.14.2) section 8.5 and v0.11.1 "One request, one
 * engine": with several sequences held over one copy of the weights, the
 * trees of concurrent requests are verified in one joint pass.
 */
int gdn_tree_verify_batched(const gdn_shape* shape, int32_t N, const int32_t* counts,
                            const int32_t* parents, const gdn_bf16* qkv, const float* alpha,
                            const float* beta, const float* state, void* out, float q_scale,
                            uint32_t flags, void* stream);

/*
 * gdn_commit_path -- keep the accepted path's state: replay path[0..L-1]
 * (a root-to-node path of the tree) through the step, in place.  The result
 * equals, bit for bit, gdn_decode_step over the path's gathered inputs.
 *   shape->B must be 1.  parents host int32 [N]; path host int32 [L], L >= 0
 *   (L == 0 leaves everything unchanged).
 *   qkv, alpha, beta  the tree's inputs as given to gdn_tree_verify.
 *   x_tree  bf16 [N, C_qkv] the tree's pre-conv inputs, or NULL.
 *   state   fp32 [Hv, dv, dk] in/out.
 *   tail    bf16 [4, C_qkv]: when x_tree != NULL, replaced by the last four
 *           inputs of (tail ++ x_tree[path[0]] ++ ... ++ x_tree[path[L-1]]).
 * Source: "Architecture" (v0.14.2) section 8.3 (commit the state of the
 * accepted path), v0.11.1 round diagram (commit KV rows and recurrent state).
 */
int gdn_commit_path(const gdn_shape* shape, int32_t N, const int32_t* parents,
                    const int32_t* path, int32_t L, const gdn_bf16* qkv,
                    const float* alpha, const float* beta, const gdn_bf16* x_tree,
                    float* state, gdn_bf16* tail, uint32_t flags, void* stream);

/*
 * gdn_commit_path_batched -- gdn_commit_path for B sequences in one launch
 * (after a joint gdn_tree_verify_batched): sequence b replays its accepted
 * path through the step in place, and its tail takes the path's inputs.  Each
 * sequence's state and tail equal, bit for bit, gdn_commit_path on its tree
 * alone.
 *   shape->B  trees, 1 .. 32.   N  node capacity per tree, 1 .. 64.
 *   counts    host int32 [B]: nodes of tree b, 1 .. N.
 *   parents   host int32 [B, N]: tree b's parent array (as for
 *             gdn_tree_verify_batched).
 *   paths     host int32 [B, N]: tree b's accepted root-to-node path in
 *             paths[b*N .. b*N + lengths[b] - 1]; may be NULL when every
 *             length is 0.
 *   lengths   host int32 [B]: path lengths, 0 .. counts[b] (0: sequence b
 *             keeps its state and tail).
 *   qkv, alpha, beta  the trees' inputs as given to the joint verify:
 *             bf16 [B, N, C_qkv], fp32 [B, N, Hv].
 *   x_tree    bf16 [B, N, C_qkv] the trees' pre-conv inputs, or NULL.
 *   state     fp32 [B, Hv, dv, dk] in/out.
 *   tail      bf16 [B, 4, C_qkv]: when x_tree != NULL, sequence b's tail is
 *             replaced by the last four inputs of (tail ++ x_tree[b][path]).
 *   flags     GDN_NORMALIZE_QK only.
 * A tree or path that fails validation refuses the whole call (nothing is
 * enqueued).  Source: "Architecture" (v0.14.2) section 8.5 (several requests'
 * trees verified in one joint pass) and section 8.3 (commit the state of the
 * accepted path).
 */
int gdn_commit_path_batched(const gdn_shape* shape, int32_t N, const int32_t* counts,
                            const int32_t* parents, const int32_t* paths, const int32_t* lengths,
                            const gdn_bf16* qkv, const float* alpha, const float* beta,
                            const gdn_bf16* x_tree, float* state, gdn_bf16* tail, uint32_t flags,
                            void* stream);

/*
 * gdn_kda_tree_verify -- gdn_tree_verify with the KDA step of
 * gdn_kda_decode_step (a decay per key channel): node n's state is the
 * committed state advanced through the root..n path by
 *   S <- (S diag(a_t)) (I - beta_t k^_t k^_t^T) + beta_t v_t k^_t^T,
 * and out[n] = S_n q^_n.  Each node's output equals, bit for bit, the output
 * gdn_kda_decode_step gives for the last token of that node's root path.
 *   alpha  fp32 [N, Hv, dk] (node n's decay vector for head h at
 *          alpha[(n * Hv + h) * dk]); every other argument as for
 *          gdn_tree_verify.
 * Source: the KDA mixer of the metrale_model_arch API page (see
 * gdn_kda_decode_step) run over "a tree" ("Architecture" v0.11.1, "The parts";
 * v0.14.2 section 8.3).
 */
int gdn_kda_tree_verify(const gdn_shape* shape, int32_t N, const int32_t* parents,
                        const gdn_bf16* qkv, const float* alpha, const float* beta,
                        const float* state, void* out, float q_scale, uint32_t flags,
                        void* stream);

/*
 * gdn_kda_tree_verify_batched -- gdn_kda_tree_verify for B sequences in one
 * launch (the joint verify of gdn_tree_verify_batched with the KDA step).
 *   alpha  fp32 [B, N, Hv, dk]; every other argument as for
 *          gdn_tree_verify_batched.
 * Each tree's outputs equal, bit for bit, gdn_kda_tree_verify of that tree
 * alone.  Source: "Architecture" (v0.14.2) section 8.5 (joint verify) with the
 * KDA mixer of gdn_kda_decode_step.
 */
int gdn_kda_tree_verify_batched(const gdn_shape* shape, int32_t N, const int32_t* counts,
                                const int32_t* parents, const gdn_bf16* qkv, const float* alpha,
                                const float* beta, const float* state, void* out, float q_scale,
                                uint32_t flags, void* stream);

/*
 * gdn_kda_commit_path -- gdn_commit_path with the KDA step: replays the
 * accepted path through gdn_kda_decode_step's arithmetic in place (bit for
 * bit the KDA decode of the path's gathered inputs), and updates the conv
 * tail as gdn_commit_path does.
 *   alpha  fp32 [N, Hv, dk]; every other argument as for gdn_commit_path.
 */
int gdn_kda_commit_path(const gdn_shape* shape, int32_t N, const int32_t* parents,
                        const int32_t* path, int32_t L, const gdn_bf16* qkv,
                        const float* alpha, const float* beta, const gdn_bf16* x_tree,
                        float* state, gdn_bf16* tail, uint32_t flags, void* stream);

/*
 * The speculative round with the conv fused in.  A round is a tree conv, the
 * verify and the commit; these entry points take the tree's PRE-conv inputs
 * and run the 4-tap conv + SiLU inside the verify and commit kernels, so the
 * conv outputs never reach HBM and the round is two launches instead of three.
 * The kernels compute the conv outputs they read (a key head's q and k, shared
 * by the CTAs that read them or computed for just the nodes a CTA walks, and
 * each CTA's own rows of v) with the arithmetic and bf16 rounding of
 * gdn_conv_step, so the results are the same bits as the unfused calls.
 *
 * gdn_conv_tree_verify -- gdn_conv_step in tree mode (x -> y) followed by
 * gdn_tree_verify on y, in one launch.  out equals that pair's, bit for bit.
 *   x       bf16 [N, C_qkv] the nodes' pre-conv inputs (packed [q | k | v]).
 *   w       bf16 [C_qkv, 4] conv taps (as for gdn_conv_step).
 *   tail    bf16 [4, C_qkv] the committed conv tail, read only.
 *   the other arguments as for gdn_tree_verify.
 * Source: the rule run over "a tree" ("Architecture" v0.11.1, "The parts")
 * with the per-layer conv tail of v0.14.2 section 8.1; verify the whole tree
 * in one pass (v0.14.2 section 8.3).
 */
int gdn_conv_tree_verify(const gdn_shape* shape, int32_t N, const int32_t* parents,
                         const gdn_bf16* x, const gdn_bf16* w, const gdn_bf16* tail,
                         const float* alpha, const float* beta, const float* state, void* out,
                         float q_scale, uint32_t flags, void* stream);

/*
 * gdn_conv_tree_verify_batched -- gdn_conv_tree_verify for B sequences in one
 * launch (the joint verify of gdn_tree_verify_batched with the conv fused in).
 *   x     bf16 [B, N, C_qkv];  tail  bf16 [B, 4, C_qkv] read only;
 *   w     bf16 [C_qkv, 4] (one layer's taps, shared by the sequences);
 *   the other arguments as for gdn_tree_verify_batched.
 * Each tree's outputs equal, bit for bit, gdn_conv_tree_verify of that tree
 * alone.  Source: "Architecture" (v0.14.2) section 8.5 (joint verify).
 */
int gdn_conv_tree_verify_batched(const gdn_shape* shape, int32_t N, const int32_t* counts,
                                 const int32_t* parents, const gdn_bf16* x, const gdn_bf16* w,
                                 const gdn_bf16* tail, const float* alpha, const float* beta,
                                 const float* state, void* out, float q_scale, uint32_t flags,
                                 void* stream);

/*
 * gdn_conv_commit_path -- the commit of the accepted path from the tree's
 * pre-conv inputs: the path's conv outputs are computed in the kernel, the
 * state is replayed in place, and the new tail -- the last four inputs of
 * (tail_in ++ x[path[0]] ++ ... ++ x[path[L-1]]) -- is written to tail_out.
 * state and tail_out equal, bit for bit, gdn_conv_step (tree mode) followed by
 * gdn_commit_path with x_tree = x.
 *   shape->B must be 1.  parents, path, L as for gdn_commit_path; L == 0
 *             leaves the state unchanged and copies tail_in to tail_out.
 *   x         bf16 [N, C_qkv] pre-conv inputs;  w  bf16 [C_qkv, 4].
 *   tail_in   bf16 [4, C_qkv] read;  tail_out  bf16 [4, C_qkv] written.  The
 *             two must not overlap (GDN_ERR_INVALID_ARG): every CTA reads
 *             tail_in for the conv while others write the new tail, so the
 *             caller alternates two tail buffers between rounds.
 *   alpha, beta, state, flags  as for gdn_commit_path.
 * Source: "Architecture" (v0.14.2) section 8.3 (commit the state of the
 * accepted path) and section 8.1 (the per-layer conv tail).
 */
int gdn_conv_commit_path(const gdn_shape* shape, int32_t N, const int32_t* parents,
                         const int32_t* path, int32_t L, const gdn_bf16* x, const gdn_bf16* w,
                         const gdn_bf16* tail_in, gdn_bf16* tail_out, const float* alpha,
                         const float* beta, float* state, uint32_t flags, void* stream);

/*
 * gdn_conv_commit_path_batched -- gdn_conv_commit_path for B sequences in one
 * launch (after gdn_conv_tree_verify_batched).
 *   counts, parents, paths, lengths  as for gdn_commit_path_batched.
 *   x         bf16 [B, N, C_qkv];  w  bf16 [C_qkv, 4].
 *   tail_in   bf16 [B, 4, C_qkv] read;  tail_out  bf16 [B, 4, C_qkv] written
 *             for every sequence (a sequence with lengths[b] == 0 gets its
 *             tail_in copied); the two must not overlap.
 *   alpha, beta fp32 [B, N, Hv];  state fp32 [B, Hv, dv, dk] in/out.
 * Each sequence's state and tail equal, bit for bit, gdn_conv_commit_path on
 * its tree alone.  Source: "Architecture" (v0.14.2) sections 8.3 and 8.5.
 */
int gdn_conv_commit_path_batched(const gdn_shape* shape, int32_t N, const int32_t* counts,
                                 const int32_t* parents, const int32_t* paths,
                                 const int32_t* lengths, const gdn_bf16* x, const gdn_bf16* w,
                                 const gdn_bf16* tail_in, gdn_bf16* tail_out, const float* alpha,
                                 const float* beta, float* state, uint32_t flags, void* stream);

/*
 * gdn_prefill_workspace_bytes -- device workspace gdn_chunk_prefill needs for
 * T tokens in chunks of `chunk` (0 on a bad shape or chunk).  The workspace
 * holds the call's status word (int32 at offset 0, padded to 256 bytes) and,
 * for 128-wide heads, one 50,432-byte pre-pass record per (chunk, value
 * head) and one int32 ready flag per (chunk, value head), padded to 16
 * bytes: 256 + ceil(T / 64) * Hv * (50,432 + 4) bytes, the flags rounded up
 * to 16 (310 MB at T = 8,192 with 48 value heads).
 */
size_t gdn_prefill_workspace_bytes(const gdn_shape* shape, int32_t T, int32_t chunk);

/*
 * gdn_chunk_prefill -- T tokens of one sequence by the chunk-parallel (WY/UT)
 * form of the same recurrence, on the tcgen05 tensor cores.  Mathematically
 * identical to gdn_decode_step over the T tokens; rounding differs (bf16
 * operand splits with fp32 accumulation, in another order).
 *   shape->B must be 1.  chunk == 64.  T >= 0 (a ragged last chunk is masked).
 *   qkv bf16 [T, C_qkv]; alpha, beta fp32 [T, Hv];
 *   state fp32 [Hv, dv, dk] in: S_0, out: S_T;  out [T, Hv, dv] fp32 / bf16.
 *   workspace  device, >= gdn_prefill_workspace_bytes(), 256-byte aligned,
 *              caller-owned.  Its int32 at offset 0 is reset to 0 by the call
 *              and set non-zero on the device if a bounded wait (for the
 *              tensor cores, a copy, or a pre-pass record) gave up; the
 *              results are then invalid.  gdn_prefill_status() reads it.
 * The chunk form runs for dk = dv = 128 (the 27B layer's heads); narrower
 * heads run the same recurrence token by token on the GPU.  A pre-pass
 * computes every chunk's state-independent part into the workspace: with
 * T = (I + L)^-1, the state-update factor T^T diag(c) K, the output factor
 * P T (P the masked, decayed Q K^T) and the per-token decays.  A chain per
 * value head then walks the chunks in order.  Where the
 * GPU can hold one chain CTA per value head plus pre-pass workers at once, both
 * run in one cooperative launch (the chain of chunk c waits, bounded, for its
 * record's ready flag, so later chunks' pre-pass overlaps earlier chunks'
 * chain); otherwise the pre-pass over all chunks runs first.  The results are
 * the same bits either way.
 * Source: "Architecture" (v0.11.1) "The parts" (the rule over a block);
 * chunk-parallel versus sequential evaluation of the recurrence, "Serving A
 * Research Architecture On CPU" (third exactness layer).  Chunk form: Yang et
 * al. 2024, "Parallelizing Linear Transformers with the Delta Rule over
 * Sequence Length", with the gated extension of "Gated Delta Networks".
 */
int gdn_chunk_prefill(const gdn_shape* shape, int32_t T, int32_t chunk,
                      const gdn_bf16* qkv, const float* alpha, const float* beta,
                      float* state, void* out, void* workspace, size_t workspace_bytes,
                      float q_scale, uint32_t flags, void* stream);

/*
 * gdn_prefill_status -- the status word of a gdn_chunk_prefill call: waits
 * for `stream` to reach this point (cudaStreamSynchronize), copies the int32
 * at offset 0 of `workspace` to *status (if status != NULL) and returns
 * GDN_OK when it is 0, GDN_ERR_TIMEOUT when a bounded device wait of the call
 * gave up (its outputs and state are then not valid), GDN_ERR_CUDA if the
 * copy failed.  Source: failing loudly rather than handing back corrupt
 * results, "Serving A Research Architecture On CPU" (the head-size bug).
 */
int gdn_prefill_status(const void* workspace, void* stream, int32_t* status);

/*
 * gdn_set_wait_limit_ns -- the limit, in nanoseconds, of every bounded device
 * wait of the prefill kernels (for the tensor cores, a copy, or another CTA's
 * pre-pass record), read at each later launch; returns the previous limit.
 * Default 200,000,000 (0.2 s); values above 10 s are clamped to 10 s; 0 makes
 * a wait give up at once unless what it waits for has already happened (for
 * tests of the timeout path).  A wait that gives up sets the call's status
 * word; the kernel still lets the work it started finish before it returns.
 * Process-wide; launches already enqueued keep the limit they were given.
 */
uint64_t gdn_set_wait_limit_ns(uint64_t ns);

/*
 * gdn_chunk_prefill_noalloc -- gdn_chunk_prefill for callers that cannot
 * allocate device memory, e.g. a serving loop whose device footprint is fixed
 * at start-up and must not grow while it serves, or a host whose device memory
 * is owned by another allocator.  (The pages describe no such call; it exists
 * for those callers.)
 *   Arguments as gdn_chunk_prefill, without the workspace.  It runs the
 *   single-launch form of the chain that computes each chunk's
 *   state-independent part itself, so its results agree with
 *   gdn_chunk_prefill's within the parity tolerances (max abs error 1e-3 on
 *   the outputs, relative Frobenius error 1e-4 on the state), not bit for bit:
 *   the same algebra is grouped differently.  The only scratch it needs is the
 *   status word, in a 256-byte array inside this library, which every GPU
 *   that loads the library keeps until the process exits.  Returns
 *   GDN_ERR_WORKSPACE if the call would need more scratch than that.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture.  Every call on a device shares the one array and clears the part
 *   that must start at zero; calls that overlap on the GPU (different streams,
 *   no ordering between them) race on it.  The status word of the last call
 *   is read with gdn_chunk_prefill_noalloc_status().
 */
int gdn_chunk_prefill_noalloc(const gdn_shape* shape, int32_t T, int32_t chunk, const gdn_bf16* qkv,
                              const float* alpha, const float* beta, float* state, void* out,
                              float q_scale, uint32_t flags, void* stream);

/*
 * gdn_chunk_prefill_noalloc_status -- the status word that the last
 * gdn_chunk_prefill_noalloc call on the current device left in the library's
 * array, read as gdn_prefill_status() reads a workspace's (it synchronises
 * `stream`, which should be the stream of that call): GDN_OK, or
 * GDN_ERR_TIMEOUT when a bounded device wait of the call gave up and its
 * outputs and state are not valid.  Allocates nothing.
 */
int gdn_chunk_prefill_noalloc_status(void* stream, int32_t* status);

/*
 * ---- Snapshot and restore of one sequence's recurrent sections -------------
 * A cache restores a sequence's state exactly: the recurrent state has
 * absorbed every token and cannot be undone, so it is restored rather than
 * recomputed ("Architecture" v0.14.2 section 8.1), and a signature over the
 * sections' names, shapes and dtypes refuses a restore across models (same
 * page, "ModelState: sections and views").  The sections of a sequence are,
 * for each of `layers` layers in order, its fp32 state [Hv, dv, dk] and its
 * bf16 conv tail [4, C_qkv].
 *
 * Blob (little-endian), gdn_snapshot_bytes() long:
 *   bytes  0..63  header: "GDNSNAP1" | u32 version 1 | u32 layers |
 *                 i32 Hk, Hv, dk, dv | u64 signature | u64 payload bytes |
 *                 u64 checksum | u64 0
 *   bytes 64..    payload: layer 0 state, layer 0 tail, layer 1 state, ...
 *                 (raw bits: the restore is bit-exact).
 *   signature  FNV-1a 64 of the text
 *              "gdn-snapshot/1;layers=<L>;state:f32[<Hv>,<dv>,<dk>];tail:bf16[4,<C>]".
 *   checksum   sum over the payload's 64-bit words d_j (j = 0, 1, ...) of
 *              mix64(d_j + (j + 1) * 0x9e3779b97f4a7c15) modulo 2^64, mix64
 *              being SplitMix64's output function and the constant its
 *              increment.
 *
 * Arrays: layer l's state is at state + l * state_layer_stride (fp32
 * elements), laid out [B, Hv, dv, dk]; its tail at tail + l *
 * tail_layer_stride (bf16 elements), [B, 4, C_qkv]; strides are multiples of
 * 16 bytes and at least one layer's array (any value when layers == 1).
 * `seq` in [0, shape->B) picks the sequence.  The blob may be device memory
 * or pinned host memory mapped into the device's address space (the kernels
 * read and write it directly); pageable host memory is refused.
 * workspace  device, >= 256 bytes, 256-byte aligned, caller-owned.  Its int32
 * at offset 0 is the call's status (read it after the stream synchronises):
 *   0  done;  1  restore refused: the blob's header (magic, version, layers,
 *   shape, signature, size) is not this shape's;  2  restore refused: the
 *   payload's checksum does not match the header's.  A refused restore writes
 *   nothing.
 */
size_t gdn_snapshot_bytes(const gdn_shape* shape, int32_t layers);       /* 0 on a bad shape */
uint64_t gdn_snapshot_signature(const gdn_shape* shape, int32_t layers); /* 0 on a bad shape */

/* gdn_snapshot_save -- write sequence seq's sections into the blob dst. */
int gdn_snapshot_save(const gdn_shape* shape, int32_t layers, int32_t seq, const float* state,
                      int64_t state_layer_stride, const gdn_bf16* tail, int64_t tail_layer_stride,
                      void* dst, size_t dst_bytes, void* workspace, size_t workspace_bytes,
                      void* stream);

/* gdn_snapshot_restore -- verify the blob src (header and checksum, on the
 * device) and, only if it verifies, write it into sequence seq's sections. */
int gdn_snapshot_restore(const gdn_shape* shape, int32_t layers, int32_t seq, const void* src,
                         size_t src_bytes, float* state, int64_t state_layer_stride, gdn_bf16* tail,
                         int64_t tail_layer_stride, void* workspace, size_t workspace_bytes,
                         void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GDN_H */
