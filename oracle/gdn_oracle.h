/*
 * gdn_oracle.h -- fp64 CPU oracle for the Gated DeltaNet mixer.
 *
 * TEST INFRASTRUCTURE ONLY.  This oracle is the slow, plain definition that the
 * CUDA library is checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table or
 * helper with the CUDA path, and the CUDA path never calls it.
 *
 * What it computes (sources):
 *  - The recurrent state: one matrix per value head, updated in place once per
 *    token, fixed size, never re-allocated.  TandemLLM "Architecture" (v0.14.2)
 *    section 8.1, table of layer kinds (48 Gated DeltaNet layers, fp32 state of
 *    48 heads x 128 x 128 plus a 4-wide convolution tail per layer);
 *    "Serving A Research Architecture On CPU", the constant-state section
 *    (rank-1 update of a fixed [d, d] matrix per head, no allocation in the loop).
 *  - The gated delta rule for one token, a block and a tree: TandemLLM
 *    "Architecture" (v0.11.1), "The parts" diagram, recurrent-layer kernels box.
 *    The pages name the rule but print no equation; the recurrence used is the
 *    published Gated DeltaNet update (Yang, Kautz & Hatamizadeh, "Gated Delta
 *    Networks: Improving Mamba2 with Delta Rule", 2024, eq. for S_t):
 *        S <- alpha * S * (I - beta * k k^T) + beta * v k^T,   o = S q
 *    with q, k L2-normalised per key head and a 4-tap causal depthwise
 *    convolution + SiLU in front of q, k, v.
 *  - Tree verify and commit: "Architecture" (v0.14.2) section 8.3 and the
 *    v0.11.1 round sequence diagram: a tree of up to 32 draft nodes is verified
 *    in one pass, each node's state branched from its parent's, and the state of
 *    the accepted root-to-node path is then kept exactly.
 *
 * Layouts (row-major, all dense):
 *   qkv    bf16 [.., C_qkv] with C_qkv = 2*Hk*dk + Hv*dv, channels [q | k | v],
 *          q and k head-major (key head g occupies channels g*dk .. g*dk+dk-1).
 *   alpha, beta  fp32 [.., Hv]
 *   state  fp64 [Hv, dv, dk]   (row i of S_h is contiguous over the key index j)
 *   out    fp64 [.., Hv, dv]
 *   conv   x bf16 [.., C], w bf16 [C, W], tail bf16 [W, C] oldest first, W = 4.
 * Value head h reads key head h / (Hv / Hk).
 *
 * Error behaviour: functions that validate (tree / path checks) return 0 or a
 * negative code; the numeric functions assume valid arguments (test code).
 */
#ifndef GDN_ORACLE_H
#define GDN_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- bf16 storage conversion -------------------------------------------- */
double   orc_bf16_to_f64(uint16_t h);
uint16_t orc_f64_to_bf16(double x);           /* round to nearest, ties to even */
void     orc_bf16_to_f64_n(const uint16_t* h, double* out, int64_t n);
void     orc_f64_to_bf16_n(const double* x, uint16_t* out, int64_t n);

/* ---- short causal convolution + SiLU ------------------------------------ */
double orc_silu(double z);

/* Linear run: per sequence b, inputs x[b, 0..T-1, :] follow the history held in
 * tail[b] (W inputs, oldest first).  y[b,t,c] = SiLU(sum_j w[c][j] * u_j) where
 * u_{W-1} is x[b,t,c] and u_{W-1-m} is the m-th earlier input.  tail[b] is
 * replaced by the last W inputs of (tail ++ x).  y is fp64 (not rounded). */
void orc_conv_linear(int B, int T, int C, int W, const uint16_t* x,
                     const uint16_t* w, uint16_t* tail, double* y);

/* The linear run over fp32 x, w and tail (widened exactly; tail stays fp32). */
void orc_conv_linear_f32(int B, int T, int C, int W, const float* x, const float* w,
                         float* tail, double* y);

/* Tree run (one sequence): node n's earlier inputs are its ancestors' inputs,
 * nearest first, and then the committed tail.  tail is not modified. */
void orc_conv_tree(int N, int C, int W, const int32_t* parents, const uint16_t* x,
                   const uint16_t* w, const uint16_t* tail, double* y);

/* The linear and tree runs with the output stored as bf16 and its rounding
 * decided in binary32 (the tap sum in tap order, SiLU, then one rounding to
 * bf16, ties to even), the precision the CUDA conv decides it in: where a
 * floating-point value is quantised, both sides quantise the same-precision
 * value.  Within one bf16 ulp of rounding the fp64 output. */
void orc_conv_linear_r32(int B, int T, int C, int W, const uint16_t* x,
                         const uint16_t* w, uint16_t* tail, uint16_t* y);
void orc_conv_tree_r32(int N, int C, int W, const int32_t* parents, const uint16_t* x,
                       const uint16_t* w, const uint16_t* tail, uint16_t* y);

/* ---- tree bookkeeping ---------------------------------------------------- */
/* 0 if parents[] describes one tree rooted at node 0 (parents[0] == -1 and
 * 0 <= parents[i] < i for i > 0); negative otherwise.  depth[n] (optional)
 * gets the number of nodes on the root..n path (root depth 1). */
int orc_tree_check(int N, const int32_t* parents, int32_t* depth);
/* Root-to-node path of `node`; returns its length. */
int orc_root_path(int N, const int32_t* parents, int node, int32_t* path);
/* 0 if path[0..L-1] is a root-to-node path of the tree, negative otherwise. */
int orc_path_check(int N, const int32_t* parents, const int32_t* path, int L);

/* ---- gated delta rule ---------------------------------------------------- */
/* out = x / sqrt(sum x^2 + eps) */
void orc_l2norm(const double* x, int n, double eps, double* out);

/* One token on one value head, row form (S is dv x dk, row-major):
 *   a_i = s_i . k ;  s_i <- alpha*s_i + beta*(v_i - alpha*a_i) * k
 * then o = S_new q computed as a plain matrix-vector product. */
void orc_delta_token(int dk, int dv, double* S, const double* k, const double* v,
                     const double* q, double alpha, double beta, double* o);

/* The same token written as the textbook matrix product, with explicit dk x dk
 * and dv x dk temporaries:  S <- alpha * S (I - beta k k^T) + beta v k^T. */
void orc_delta_token_matrix(int dk, int dv, double* S, const double* k,
                            const double* v, const double* q, double alpha,
                            double beta, double* o);

/* T sequential tokens for B independent sequences.
 * qkv bf16 [B,T,C_qkv]; alpha, beta fp32 [B,T,Hv]; state fp64 [B,Hv,dv,dk]
 * (in/out); out fp64 [B,T,Hv,dv].  normalize != 0 applies the L2 norm to q, k
 * (eps = 1e-6); q is then multiplied by q_scale. */
void orc_decode(int B, int T, int Hk, int Hv, int dk, int dv, const uint16_t* qkv,
                const float* alpha, const float* beta, double* state, double* out,
                double q_scale, int normalize);

/* orc_decode over fp32 activations qkv [B,T,C_qkv] (widened exactly). */
void orc_decode_f32(int B, int T, int Hk, int Hv, int dk, int dv, const float* qkv,
                    const float* alpha, const float* beta, double* state, double* out,
                    double q_scale, int normalize);

/* Tree verify (one sequence): node n's state is the committed state advanced
 * through the root..n path; out[n] is that node's output.  Computed by replaying
 * each node's root path from the committed state (state is not modified). */
void orc_tree_verify(int N, int Hk, int Hv, int dk, int dv, const int32_t* parents,
                     const uint16_t* qkv, const float* alpha, const float* beta,
                     const double* state, double* out, double q_scale, int normalize);

/* Commit: advance state through the accepted path's nodes, in order.  If
 * x_tree is not NULL, tail [W, C] becomes the last W inputs of
 * (tail ++ x_tree[path[0]] ++ ... ++ x_tree[path[L-1]]). */
void orc_commit(int N, int Hk, int Hv, int dk, int dv, const int32_t* parents,
                const int32_t* path, int L, const uint16_t* qkv, const float* alpha,
                const float* beta, const uint16_t* x_tree, int W, double* state,
                uint16_t* tail, int normalize);

/* ---- KDA variant: a decay per key channel ---------------------------------
 * Kimi Delta Attention is listed, with a CPU reference, in the module index of
 * the metrale_model_arch API page (Modules: glm5next_kda, kimi_k3); the page
 * prints no update rule.  Read here as the gated delta rule with the scalar
 * decay replaced by a diagonal one on the key dimension:
 *     S <- (S diag(a)) (I - beta k k^T) + beta v k^T,   o = S q
 * with a = alpha[0..dk-1].  Row form: s' = a o s (elementwise);
 * s <- s' + beta (v_i - s'.k) k.  Then o = S_new q as a plain product. */
void orc_kda_token(int dk, int dv, double* S, const double* k, const double* v,
                   const double* q, const double* alpha, double beta, double* o);
void orc_kda_token_matrix(int dk, int dv, double* S, const double* k, const double* v,
                          const double* q, const double* alpha, double beta, double* o);
/* As orc_decode, with alpha fp32 [B,T,Hv,dk] (one decay per key channel). */
void orc_kda_decode(int B, int T, int Hk, int Hv, int dk, int dv, const uint16_t* qkv,
                    const float* alpha, const float* beta, double* state, double* out,
                    double q_scale, int normalize);

/* ---- gate front end and gated-norm output (the layer around the mixer) -----
 * The pages name the layer but print neither step; both are read from the
 * published Gated DeltaNet layer (Yang, Kautz & Hatamizadeh 2024, as shipped
 * with the Qwen3-Next models): per value head h, from bf16 projections a, b
 * and fp32 parameters A_log[h], dt_bias[h]:
 *     alpha = exp(-exp(A_log[h]) * softplus(a + dt_bias[h])),
 *     beta  = sigmoid(b),
 * and after the mixer, with bf16 projection z [dv] and fp32 weight w [dv]:
 *     y_i = o_i / sqrt(mean_i(o_i^2) + eps) * w_i * SiLU(z_i).
 * softplus(x) = log(1 + e^x), evaluated as max(x, 0) + log1p(e^-|x|). */
double orc_softplus(double x);
double orc_sigmoid(double x);
/* a, b bf16 [n, Hv]; alpha, beta fp64 [n, Hv]. */
void orc_gates(int n, int Hv, const uint16_t* a, const uint16_t* b, const float* A_log, const float* dt_bias,
               double* alpha, double* beta);
void orc_gated_rmsnorm(int dv, const double* o, const uint16_t* z, const float* w, double eps, double* y);
/* The whole decode step of one layer for T tokens of B sequences:
 * conv + SiLU (tail in/out, conv output rounded to bf16 as stored), gates
 * from a/b, L2-norm, the delta step (state in/out), o = S q, then y.
 *   x bf16 [B,T,C]; conv_w bf16 [C,4]; tail bf16 [B,4,C] in/out;
 *   a, b bf16 [B,T,Hv]; A_log, dt_bias fp32 [Hv]; z bf16 [B,T,Hv,dv];
 *   norm_w fp32 [dv]; state fp64 [B,Hv,dv,dk]; o, y fp64 [B,T,Hv,dv]. */
void orc_layer_decode(int B, int T, int Hk, int Hv, int dk, int dv, const uint16_t* x, const uint16_t* conv_w,
                      uint16_t* tail, const uint16_t* a, const uint16_t* b, const float* A_log,
                      const float* dt_bias, const uint16_t* z, const float* norm_w, double eps, double* state,
                      double* o, double* y, double q_scale, int normalize);

/* ---- state snapshot / restore ----------------------------------------------
 * A cache restores a sequence's recurrent state exactly ("Architecture"
 * v0.14.2, section 8.1: the state has absorbed every token and has no inverse,
 * so it is restored from a cache); a signature over section names, shapes and
 * dtypes refuses a restore across models (section "ModelState: sections and
 * views").  Blob format (little-endian):
 *   header, 64 bytes: magic "GDNSNAP1" | u32 version 1 | u32 layers |
 *     i32 Hk, Hv, dk, dv | u64 signature | u64 payload bytes | u64 checksum |
 *     u64 0
 *   payload: for each layer l in order, the sequence's state [Hv][dv][dk] fp32
 *     then its conv tail [4][C] bf16, C = 2 Hk dk + Hv dv.
 * signature = FNV-1a 64 (Fowler, Noll, Vo; offset basis 0xcbf29ce484222325,
 *   prime 0x100000001b3) of the text
 *   "gdn-snapshot/1;layers=<L>;state:f32[<Hv>,<dv>,<dk>];tail:bf16[4,<C>]".
 * checksum = sum over the payload's little-endian 64-bit words d_j
 *   (j = 0, 1, ...) of mix64(d_j + (j + 1) * 0x9e3779b97f4a7c15), modulo
 *   2^64, where mix64 is the output function of Steele, Lea & Flood's
 *   SplitMix64 (shift 30, multiply 0xbf58476d1ce4e5b9, shift 27, multiply
 *   0x94d049bb133111eb, shift 31) and 0x9e3779b97f4a7c15 its increment: for
 *   an all-zero payload the terms are the generator's outputs from seed 0. */
uint64_t orc_fnv1a64(const uint8_t* p, size_t n);
uint64_t orc_mix64(uint64_t z);
uint64_t orc_snapshot_checksum(const uint8_t* payload, size_t bytes);
uint64_t orc_snapshot_signature(int layers, int Hk, int Hv, int dk, int dv);
size_t orc_snapshot_bytes(int layers, int Hk, int Hv, int dk, int dv);
/* state [layers][B][Hv][dv][dk], tail [layers][B][4][C]; seq in [0, B). */
void orc_snapshot_save(int layers, int B, int Hk, int Hv, int dk, int dv, int seq, const float* state,
                       const uint16_t* tail, uint8_t* blob);
/* Returns 0 and writes sequence seq's sections; 1 if the header does not
 * match (magic, version, layers, shape, signature, payload size); 2 if the
 * payload's checksum does not match.  Nothing is written unless 0. */
int orc_snapshot_restore(int layers, int B, int Hk, int Hv, int dk, int dv, int seq, const uint8_t* blob,
                         float* state, uint16_t* tail);

#ifdef __cplusplus
}
#endif
#endif
