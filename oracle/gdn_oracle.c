/*
 * gdn_oracle.c -- fp64 CPU oracle for the Gated DeltaNet mixer.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the test suite, the smoke check and the
 * benchmark's CPU-baseline leg; never by the CUDA library.  Plain loops, no
 * blocking, fusion or reordering beyond the definitions cited in gdn_oracle.h.
 * Everything is fp64 except where the data is stored as bf16/fp32, which is
 * converted exactly on the way in.
 */
#include "gdn_oracle.h"

#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 storage                                                               */
/* ------------------------------------------------------------------------ */

/* bf16 is the top 16 bits of an IEEE binary32: 1 sign, 8 exponent, 7 fraction
 * bits.  Widening is exact. */
double orc_bf16_to_f64(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16, ties to even.  Done by decomposing the
 * value (frexp) rather than by bit tricks on binary32, so that it is a direct
 * rounding of the fp64 value (no double rounding through fp32). */
uint16_t orc_f64_to_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0x0000;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    /* Spacing of bf16 values around a: normal numbers have 8 significant bits
     * (2^(e-8) for a in [2^(e-1), 2^e)); subnormals are multiples of 2^-133. */
    int e;
    frexp(a, &e);                       /* a = m * 2^e, m in [0.5, 1) */
    int q = e - 8;                      /* ulp exponent for normals */
    if (q < -133) q = -133;             /* subnormal range: fixed ulp 2^-133 */
    double scaled = ldexp(a, -q);       /* exact: power-of-two scaling */
    double fl = floor(scaled);
    double rem = scaled - fl;           /* exact */
    double n = fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) n = fl + 1.0;
    double r = ldexp(n, q);             /* the rounded magnitude */
    if (r > 0x1.FEp127) return sign | 0x7F80;   /* past the largest finite bf16 */
    float rf = (float)r;                /* exact: r is representable in bf16 */
    uint32_t bits;
    memcpy(&bits, &rf, sizeof bits);
    return sign | (uint16_t)(bits >> 16);
}

void orc_bf16_to_f64_n(const uint16_t* h, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f64(h[i]);
}

void orc_f64_to_bf16_n(const double* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* short causal convolution                                                   */
/* ------------------------------------------------------------------------ */

/* SiLU(z) = z * sigmoid(z) = z / (1 + e^-z) */
double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* One output channel: taps w[0..W-1] against inputs u[0..W-1] (oldest first). */
static double conv_channel(int W, const uint16_t* wc, const double* u) {
    double acc = 0.0;
    for (int j = 0; j < W; ++j) acc += orc_bf16_to_f64(wc[j]) * u[j];
    return orc_silu(acc);
}

/* The same channel where the output is stored as bf16 and the rounding is
 * decided in binary32, the precision of the CUDA conv: the sum over the taps in
 * binary32 in tap order (the first product is exact, each further term one
 * fused multiply-add), SiLU(z) = z / (1 + e^-z) in binary32 with the host
 * libm's expf, then round to the nearest bf16, ties to even.  Rounding a conv
 * output to bf16 is a quantisation, so both sides take it in one precision. */
static uint16_t conv_channel_r32(int W, const uint16_t* wc, const double* u) {
    float acc = (float)orc_bf16_to_f64(wc[0]) * (float)u[0];
    for (int j = 1; j < W; ++j) acc = fmaf((float)orc_bf16_to_f64(wc[j]), (float)u[j], acc);
    const float z = acc / (1.0f + expf(-acc));
    return orc_f64_to_bf16((double)z); /* exact widening, then one rounding */
}

/* y64 != NULL: fp64 outputs; else y16 gets the bf16 outputs decided in binary32 */
static void conv_linear_impl(int B, int T, int C, int W, const uint16_t* x, const uint16_t* w, uint16_t* tail,
                             double* y64, uint16_t* y16) {
    /* history per sequence: W tail inputs followed by the T new inputs */
    double* u = (double*)malloc(sizeof(double) * (size_t)W);
    uint16_t* hist = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(W + T));
    for (int b = 0; b < B; ++b) {
        for (int c = 0; c < C; ++c) {
            for (int j = 0; j < W; ++j) hist[j] = tail[((size_t)b * W + j) * C + c];
            for (int t = 0; t < T; ++t) hist[W + t] = x[((size_t)b * T + t) * C + c];
            for (int t = 0; t < T; ++t) {
                /* inputs x_{t-W+1} .. x_t sit at hist[t+1 .. t+W] */
                for (int j = 0; j < W; ++j) u[j] = orc_bf16_to_f64(hist[t + 1 + j]);
                const size_t at = ((size_t)b * T + t) * C + c;
                if (y64) y64[at] = conv_channel(W, w + (size_t)c * W, u);
                else y16[at] = conv_channel_r32(W, w + (size_t)c * W, u);
            }
            for (int j = 0; j < W; ++j) tail[((size_t)b * W + j) * C + c] = hist[T + j];
        }
    }
    free(hist);
    free(u);
}

void orc_conv_linear(int B, int T, int C, int W, const uint16_t* x,
                     const uint16_t* w, uint16_t* tail, double* y) {
    conv_linear_impl(B, T, C, W, x, w, tail, y, NULL);
}

void orc_conv_linear_r32(int B, int T, int C, int W, const uint16_t* x,
                         const uint16_t* w, uint16_t* tail, uint16_t* y) {
    conv_linear_impl(B, T, C, W, x, w, tail, NULL, y);
}

/* The same linear run over fp32 activations and taps (widened exactly to fp64;
 * nothing is rounded to bf16). */
void orc_conv_linear_f32(int B, int T, int C, int W, const float* x, const float* w,
                         float* tail, double* y) {
    double* u = (double*)malloc(sizeof(double) * (size_t)W);
    float* hist = (float*)malloc(sizeof(float) * (size_t)(W + T));
    for (int b = 0; b < B; ++b) {
        for (int c = 0; c < C; ++c) {
            for (int j = 0; j < W; ++j) hist[j] = tail[((size_t)b * W + j) * C + c];
            for (int t = 0; t < T; ++t) hist[W + t] = x[((size_t)b * T + t) * C + c];
            for (int t = 0; t < T; ++t) {
                double acc = 0.0;
                for (int j = 0; j < W; ++j) {
                    u[j] = (double)hist[t + 1 + j];
                    acc += (double)w[(size_t)c * W + j] * u[j];
                }
                y[((size_t)b * T + t) * C + c] = orc_silu(acc);
            }
            for (int j = 0; j < W; ++j) tail[((size_t)b * W + j) * C + c] = hist[T + j];
        }
    }
    free(hist);
    free(u);
}

static void conv_tree_impl(int N, int C, int W, const int32_t* parents, const uint16_t* x, const uint16_t* w,
                           const uint16_t* tail, double* y64, uint16_t* y16) {
    double* u = (double*)malloc(sizeof(double) * (size_t)W);
    for (int n = 0; n < N; ++n) {
        for (int c = 0; c < C; ++c) {
            /* walk back from n: the newest input is x[n], then its parent's ... */
            int node = n;
            int tail_pos = W - 1;            /* next tail entry once nodes run out */
            for (int j = W - 1; j >= 0; --j) {
                if (node >= 0) {
                    u[j] = orc_bf16_to_f64(x[(size_t)node * C + c]);
                    node = parents[node];
                } else {
                    u[j] = orc_bf16_to_f64(tail[(size_t)tail_pos * C + c]);
                    tail_pos -= 1;
                }
            }
            if (y64) y64[(size_t)n * C + c] = conv_channel(W, w + (size_t)c * W, u);
            else y16[(size_t)n * C + c] = conv_channel_r32(W, w + (size_t)c * W, u);
        }
    }
    free(u);
}

void orc_conv_tree(int N, int C, int W, const int32_t* parents, const uint16_t* x,
                   const uint16_t* w, const uint16_t* tail, double* y) {
    conv_tree_impl(N, C, W, parents, x, w, tail, y, NULL);
}

void orc_conv_tree_r32(int N, int C, int W, const int32_t* parents, const uint16_t* x,
                       const uint16_t* w, const uint16_t* tail, uint16_t* y) {
    conv_tree_impl(N, C, W, parents, x, w, tail, NULL, y);
}

/* ------------------------------------------------------------------------ */
/* tree bookkeeping                                                           */
/* ------------------------------------------------------------------------ */

int orc_tree_check(int N, const int32_t* parents, int32_t* depth) {
    if (N < 1 || parents == NULL) return -1;
    if (parents[0] != -1) return -2;
    for (int i = 1; i < N; ++i)
        if (parents[i] < 0 || parents[i] >= i) return -3;
    if (depth) {
        depth[0] = 1;
        for (int i = 1; i < N; ++i) depth[i] = depth[parents[i]] + 1;
    }
    return 0;
}

int orc_root_path(int N, const int32_t* parents, int node, int32_t* path) {
    (void)N;
    int len = 0;
    for (int m = node; m >= 0; m = parents[m]) len += 1;
    int pos = len - 1;
    for (int m = node; m >= 0; m = parents[m]) path[pos--] = m;
    return len;
}

int orc_path_check(int N, const int32_t* parents, const int32_t* path, int L) {
    if (L < 0) return -1;
    for (int i = 0; i < L; ++i)
        if (path[i] < 0 || path[i] >= N) return -2;
    if (L == 0) return 0;
    if (parents[path[0]] != -1) return -3;
    for (int i = 1; i < L; ++i)
        if (parents[path[i]] != path[i - 1]) return -4;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* gated delta rule                                                           */
/* ------------------------------------------------------------------------ */

void orc_l2norm(const double* x, int n, double eps, double* out) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < n; ++i) out[i] = x[i] * inv;
}

void orc_delta_token(int dk, int dv, double* S, const double* k, const double* v,
                     const double* q, double alpha, double beta, double* o) {
    for (int i = 0; i < dv; ++i) {
        double* s = S + (size_t)i * dk;
        double a = 0.0;
        for (int j = 0; j < dk; ++j) a += s[j] * k[j];
        double u = beta * (v[i] - alpha * a);
        for (int j = 0; j < dk; ++j) s[j] = alpha * s[j] + u * k[j];
    }
    for (int i = 0; i < dv; ++i) {
        const double* s = S + (size_t)i * dk;
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += s[j] * q[j];
        o[i] = acc;
    }
}

void orc_delta_token_matrix(int dk, int dv, double* S, const double* k,
                            const double* v, const double* q, double alpha,
                            double beta, double* o) {
    /* A = I - beta k k^T  (dk x dk) */
    double* A = (double*)malloc(sizeof(double) * (size_t)dk * dk);
    double* R = (double*)malloc(sizeof(double) * (size_t)dv * dk);
    for (int a = 0; a < dk; ++a)
        for (int b = 0; b < dk; ++b)
            A[(size_t)a * dk + b] = (a == b ? 1.0 : 0.0) - beta * k[a] * k[b];
    /* R = alpha * S A + beta v k^T */
    for (int i = 0; i < dv; ++i)
        for (int b = 0; b < dk; ++b) {
            double acc = 0.0;
            for (int a = 0; a < dk; ++a) acc += S[(size_t)i * dk + a] * A[(size_t)a * dk + b];
            R[(size_t)i * dk + b] = alpha * acc + beta * v[i] * k[b];
        }
    memcpy(S, R, sizeof(double) * (size_t)dv * dk);
    for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * q[j];
        o[i] = acc;
    }
    free(R);
    free(A);
}

/* Gather one token's q (key head g), k (key head g) and v (value head h) from
 * the packed bf16 row, widen, and normalise q and k. */
static void token_vectors(int Hk, int dk, int dv, const uint16_t* row, int g, int h,
                          double q_scale, int normalize, double* q, double* k,
                          double* v) {
    const uint16_t* qs = row + (size_t)g * dk;
    const uint16_t* ks = row + (size_t)Hk * dk + (size_t)g * dk;
    const uint16_t* vs = row + (size_t)2 * Hk * dk + (size_t)h * dv;
    double* tmp = (double*)malloc(sizeof(double) * (size_t)dk);
    for (int j = 0; j < dk; ++j) tmp[j] = orc_bf16_to_f64(qs[j]);
    if (normalize) orc_l2norm(tmp, dk, 1e-6, q); else memcpy(q, tmp, sizeof(double) * dk);
    for (int j = 0; j < dk; ++j) q[j] *= q_scale;
    for (int j = 0; j < dk; ++j) tmp[j] = orc_bf16_to_f64(ks[j]);
    if (normalize) orc_l2norm(tmp, dk, 1e-6, k); else memcpy(k, tmp, sizeof(double) * dk);
    for (int i = 0; i < dv; ++i) v[i] = orc_bf16_to_f64(vs[i]);
    free(tmp);
}

void orc_decode(int B, int T, int Hk, int Hv, int dk, int dv, const uint16_t* qkv,
                const float* alpha, const float* beta, double* state, double* out,
                double q_scale, int normalize) {
    const size_t C = (size_t)2 * Hk * dk + (size_t)Hv * dv;
    const int group = Hv / Hk;
    double* q = (double*)malloc(sizeof(double) * (size_t)dk);
    double* k = (double*)malloc(sizeof(double) * (size_t)dk);
    double* v = (double*)malloc(sizeof(double) * (size_t)dv);
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t) {
            const size_t tok = (size_t)b * T + t;
            for (int h = 0; h < Hv; ++h) {
                token_vectors(Hk, dk, dv, qkv + tok * C, h / group, h, q_scale,
                              normalize, q, k, v);
                double* S = state + ((size_t)b * Hv + h) * (size_t)dv * dk;
                orc_delta_token(dk, dv, S, k, v, q, (double)alpha[tok * Hv + h],
                                (double)beta[tok * Hv + h], out + (tok * Hv + h) * dv);
            }
        }
    free(v);
    free(k);
    free(q);
}

/* orc_decode over fp32 activations: each token's q, k, v widened exactly to
 * fp64, then the same normalisation and row-form step. */
void orc_decode_f32(int B, int T, int Hk, int Hv, int dk, int dv, const float* qkv,
                    const float* alpha, const float* beta, double* state, double* out,
                    double q_scale, int normalize) {
    const size_t C = (size_t)2 * Hk * dk + (size_t)Hv * dv;
    const int group = Hv / Hk;
    double* raw = (double*)malloc(sizeof(double) * (size_t)dk);
    double* q = (double*)malloc(sizeof(double) * (size_t)dk);
    double* k = (double*)malloc(sizeof(double) * (size_t)dk);
    double* v = (double*)malloc(sizeof(double) * (size_t)dv);
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t) {
            const size_t tok = (size_t)b * T + t;
            const float* row = qkv + tok * C;
            for (int h = 0; h < Hv; ++h) {
                const int g = h / group;
                for (int j = 0; j < dk; ++j) raw[j] = (double)row[(size_t)g * dk + j];
                if (normalize) orc_l2norm(raw, dk, 1e-6, q); else memcpy(q, raw, sizeof(double) * dk);
                for (int j = 0; j < dk; ++j) q[j] *= q_scale;
                for (int j = 0; j < dk; ++j) raw[j] = (double)row[(size_t)Hk * dk + (size_t)g * dk + j];
                if (normalize) orc_l2norm(raw, dk, 1e-6, k); else memcpy(k, raw, sizeof(double) * dk);
                for (int i = 0; i < dv; ++i) v[i] = (double)row[(size_t)2 * Hk * dk + (size_t)h * dv + i];
                double* S = state + ((size_t)b * Hv + h) * (size_t)dv * dk;
                orc_delta_token(dk, dv, S, k, v, q, (double)alpha[tok * Hv + h],
                                (double)beta[tok * Hv + h], out + (tok * Hv + h) * dv);
            }
        }
    free(v);
    free(k);
    free(q);
    free(raw);
}

void orc_tree_verify(int N, int Hk, int Hv, int dk, int dv, const int32_t* parents,
                     const uint16_t* qkv, const float* alpha, const float* beta,
                     const double* state, double* out, double q_scale, int normalize) {
    const size_t C = (size_t)2 * Hk * dk + (size_t)Hv * dv;
    const int group = Hv / Hk;
    const size_t hs = (size_t)dv * dk;
    double* S = (double*)malloc(sizeof(double) * hs);
    double* q = (double*)malloc(sizeof(double) * (size_t)dk);
    double* k = (double*)malloc(sizeof(double) * (size_t)dk);
    double* v = (double*)malloc(sizeof(double) * (size_t)dv);
    double* o = (double*)malloc(sizeof(double) * (size_t)dv);
    int32_t* path = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    for (int n = 0; n < N; ++n) {
        int L = orc_root_path(N, parents, n, path);
        for (int h = 0; h < Hv; ++h) {
            memcpy(S, state + (size_t)h * hs, sizeof(double) * hs);
            for (int m = 0; m < L; ++m) {
                const int node = path[m];
                token_vectors(Hk, dk, dv, qkv + (size_t)node * C, h / group, h, q_scale,
                              normalize, q, k, v);
                orc_delta_token(dk, dv, S, k, v, q, (double)alpha[(size_t)node * Hv + h],
                                (double)beta[(size_t)node * Hv + h], o);
            }
            memcpy(out + ((size_t)n * Hv + h) * dv, o, sizeof(double) * (size_t)dv);
        }
    }
    free(path);
    free(o);
    free(v);
    free(k);
    free(q);
    free(S);
}

void orc_commit(int N, int Hk, int Hv, int dk, int dv, const int32_t* parents,
                const int32_t* path, int L, const uint16_t* qkv, const float* alpha,
                const float* beta, const uint16_t* x_tree, int W, double* state,
                uint16_t* tail, int normalize) {
    (void)N;
    (void)parents;
    const size_t C = (size_t)2 * Hk * dk + (size_t)Hv * dv;
    const int group = Hv / Hk;
    const size_t hs = (size_t)dv * dk;
    double* q = (double*)malloc(sizeof(double) * (size_t)dk);
    double* k = (double*)malloc(sizeof(double) * (size_t)dk);
    double* v = (double*)malloc(sizeof(double) * (size_t)dv);
    double* o = (double*)malloc(sizeof(double) * (size_t)dv);
    for (int m = 0; m < L; ++m) {
        const int node = path[m];
        for (int h = 0; h < Hv; ++h) {
            token_vectors(Hk, dk, dv, qkv + (size_t)node * C, h / group, h, 1.0,
                          normalize, q, k, v);
            orc_delta_token(dk, dv, state + (size_t)h * hs, k, v, q,
                            (double)alpha[(size_t)node * Hv + h],
                            (double)beta[(size_t)node * Hv + h], o);
        }
    }
    if (x_tree != NULL && tail != NULL) {
        /* history = W tail entries followed by the path's inputs; keep the last W */
        const int total = W + L;
        uint16_t* hist = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)total * C);
        memcpy(hist, tail, sizeof(uint16_t) * (size_t)W * C);
        for (int m = 0; m < L; ++m)
            memcpy(hist + (size_t)(W + m) * C, x_tree + (size_t)path[m] * C,
                   sizeof(uint16_t) * C);
        memcpy(tail, hist + (size_t)(total - W) * C, sizeof(uint16_t) * (size_t)W * C);
        free(hist);
    }
    free(o);
    free(v);
    free(k);
    free(q);
}

/* ------------------------------------------------------------------------ */
/* KDA variant                                                                */
/* ------------------------------------------------------------------------ */

void orc_kda_token(int dk, int dv, double* S, const double* k, const double* v,
                   const double* q, const double* alpha, double beta, double* o) {
    for (int i = 0; i < dv; ++i) {
        double* s = S + (size_t)i * dk;
        for (int j = 0; j < dk; ++j) s[j] *= alpha[j];      /* s' = a o s */
        double a = 0.0;
        for (int j = 0; j < dk; ++j) a += s[j] * k[j];
        double u = beta * (v[i] - a);
        for (int j = 0; j < dk; ++j) s[j] += u * k[j];
    }
    for (int i = 0; i < dv; ++i) {
        const double* s = S + (size_t)i * dk;
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += s[j] * q[j];
        o[i] = acc;
    }
}

void orc_kda_token_matrix(int dk, int dv, double* S, const double* k, const double* v,
                          const double* q, const double* alpha, double beta, double* o) {
    /* D A with D = diag(alpha), A = I - beta k k^T: (D A)[a][b] = alpha[a] A[a][b] */
    double* DA = (double*)malloc(sizeof(double) * (size_t)dk * dk);
    double* R = (double*)malloc(sizeof(double) * (size_t)dv * dk);
    for (int a = 0; a < dk; ++a)
        for (int b = 0; b < dk; ++b)
            DA[(size_t)a * dk + b] = alpha[a] * ((a == b ? 1.0 : 0.0) - beta * k[a] * k[b]);
    /* R = S (D A) + beta v k^T */
    for (int i = 0; i < dv; ++i)
        for (int b = 0; b < dk; ++b) {
            double acc = 0.0;
            for (int a = 0; a < dk; ++a) acc += S[(size_t)i * dk + a] * DA[(size_t)a * dk + b];
            R[(size_t)i * dk + b] = acc + beta * v[i] * k[b];
        }
    memcpy(S, R, sizeof(double) * (size_t)dv * dk);
    for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * q[j];
        o[i] = acc;
    }
    free(R);
    free(DA);
}

void orc_kda_decode(int B, int T, int Hk, int Hv, int dk, int dv, const uint16_t* qkv,
                    const float* alpha, const float* beta, double* state, double* out,
                    double q_scale, int normalize) {
    const size_t C = (size_t)2 * Hk * dk + (size_t)Hv * dv;
    const int group = Hv / Hk;
    double* q = (double*)malloc(sizeof(double) * (size_t)dk);
    double* k = (double*)malloc(sizeof(double) * (size_t)dk);
    double* v = (double*)malloc(sizeof(double) * (size_t)dv);
    double* a = (double*)malloc(sizeof(double) * (size_t)dk);
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t) {
            const size_t tok = (size_t)b * T + t;
            for (int h = 0; h < Hv; ++h) {
                token_vectors(Hk, dk, dv, qkv + tok * C, h / group, h, q_scale, normalize, q, k, v);
                for (int j = 0; j < dk; ++j) a[j] = (double)alpha[(tok * Hv + h) * dk + j];
                double* S = state + ((size_t)b * Hv + h) * (size_t)dv * dk;
                orc_kda_token(dk, dv, S, k, v, q, a, (double)beta[tok * Hv + h],
                              out + (tok * Hv + h) * dv);
            }
        }
    free(a);
    free(v);
    free(k);
    free(q);
}

/* ------------------------------------------------------------------------ */
/* state snapshot / restore                                                   */
/* ------------------------------------------------------------------------ */

uint64_t orc_fnv1a64(const uint8_t* p, size_t n) {
    uint64_t h = 0xcbf29ce484222325ULL;
    for (size_t i = 0; i < n; ++i) {
        h ^= (uint64_t)p[i];
        h *= 0x100000001b3ULL;
    }
    return h;
}

uint64_t orc_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

uint64_t orc_snapshot_checksum(const uint8_t* payload, size_t bytes) {
    uint64_t sum = 0;
    for (size_t j = 0; j < bytes / 8; ++j) {
        uint64_t d = 0;
        for (int b = 0; b < 8; ++b) d |= (uint64_t)payload[8 * j + b] << (8 * b);
        sum += orc_mix64(d + (uint64_t)(j + 1) * 0x9e3779b97f4a7c15ULL);
    }
    return sum;
}

static int snap_channels(int Hk, int Hv, int dk, int dv) { return 2 * Hk * dk + Hv * dv; }

uint64_t orc_snapshot_signature(int layers, int Hk, int Hv, int dk, int dv) {
    char text[256];
    int n = snprintf(text, sizeof text, "gdn-snapshot/1;layers=%d;state:f32[%d,%d,%d];tail:bf16[4,%d]", layers,
                     Hv, dv, dk, snap_channels(Hk, Hv, dk, dv));
    return orc_fnv1a64((const uint8_t*)text, (size_t)n);
}

static size_t snap_state_bytes(int Hv, int dk, int dv) { return (size_t)Hv * dv * dk * 4; }
static size_t snap_tail_bytes(int Hk, int Hv, int dk, int dv) {
    return (size_t)4 * snap_channels(Hk, Hv, dk, dv) * 2;
}

size_t orc_snapshot_bytes(int layers, int Hk, int Hv, int dk, int dv) {
    return 64 + (size_t)layers * (snap_state_bytes(Hv, dk, dv) + snap_tail_bytes(Hk, Hv, dk, dv));
}

static void put_u32(uint8_t* p, uint32_t v) {
    for (int i = 0; i < 4; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
static void put_u64(uint8_t* p, uint64_t v) {
    for (int i = 0; i < 8; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
static uint32_t get_u32(const uint8_t* p) {
    uint32_t v = 0;
    for (int i = 0; i < 4; ++i) v |= (uint32_t)p[i] << (8 * i);
    return v;
}
static uint64_t get_u64(const uint8_t* p) {
    uint64_t v = 0;
    for (int i = 0; i < 8; ++i) v |= (uint64_t)p[i] << (8 * i);
    return v;
}

/* fp32 and bf16 values are stored as their little-endian bit patterns */
static void put_f32(uint8_t* p, float f) {
    uint32_t bits;
    memcpy(&bits, &f, 4);
    put_u32(p, bits);
}

static void write_header(uint8_t* h, int layers, int Hk, int Hv, int dk, int dv, uint64_t checksum) {
    memcpy(h, "GDNSNAP1", 8);
    put_u32(h + 8, 1);
    put_u32(h + 12, (uint32_t)layers);
    put_u32(h + 16, (uint32_t)Hk);
    put_u32(h + 20, (uint32_t)Hv);
    put_u32(h + 24, (uint32_t)dk);
    put_u32(h + 28, (uint32_t)dv);
    put_u64(h + 32, orc_snapshot_signature(layers, Hk, Hv, dk, dv));
    put_u64(h + 40, orc_snapshot_bytes(layers, Hk, Hv, dk, dv) - 64);
    put_u64(h + 48, checksum);
    put_u64(h + 56, 0);
}

void orc_snapshot_save(int layers, int B, int Hk, int Hv, int dk, int dv, int seq, const float* state,
                       const uint16_t* tail, uint8_t* blob) {
    const size_t S = (size_t)Hv * dv * dk;           /* state values of one sequence */
    const size_t TL = (size_t)4 * snap_channels(Hk, Hv, dk, dv);  /* tail values of one sequence */
    uint8_t* p = blob + 64;
    for (int l = 0; l < layers; ++l) {
        const float* st = state + ((size_t)l * B + seq) * S;
        for (size_t i = 0; i < S; ++i, p += 4) put_f32(p, st[i]);
        const uint16_t* tl = tail + ((size_t)l * B + seq) * TL;
        for (size_t i = 0; i < TL; ++i, p += 2) {
            p[0] = (uint8_t)(tl[i] & 0xff);
            p[1] = (uint8_t)(tl[i] >> 8);
        }
    }
    const size_t payload = orc_snapshot_bytes(layers, Hk, Hv, dk, dv) - 64;
    write_header(blob, layers, Hk, Hv, dk, dv, orc_snapshot_checksum(blob + 64, payload));
}

int orc_snapshot_restore(int layers, int B, int Hk, int Hv, int dk, int dv, int seq, const uint8_t* blob,
                         float* state, uint16_t* tail) {
    const size_t payload = orc_snapshot_bytes(layers, Hk, Hv, dk, dv) - 64;
    if (memcmp(blob, "GDNSNAP1", 8) != 0 || get_u32(blob + 8) != 1 || get_u32(blob + 12) != (uint32_t)layers ||
        get_u32(blob + 16) != (uint32_t)Hk || get_u32(blob + 20) != (uint32_t)Hv ||
        get_u32(blob + 24) != (uint32_t)dk || get_u32(blob + 28) != (uint32_t)dv ||
        get_u64(blob + 32) != orc_snapshot_signature(layers, Hk, Hv, dk, dv) || get_u64(blob + 40) != payload)
        return 1;
    if (orc_snapshot_checksum(blob + 64, payload) != get_u64(blob + 48)) return 2;
    const size_t S = (size_t)Hv * dv * dk;
    const size_t TL = (size_t)4 * snap_channels(Hk, Hv, dk, dv);
    const uint8_t* p = blob + 64;
    for (int l = 0; l < layers; ++l) {
        float* st = state + ((size_t)l * B + seq) * S;
        for (size_t i = 0; i < S; ++i, p += 4) {
            const uint32_t bits = get_u32(p);
            memcpy(&st[i], &bits, 4);
        }
        uint16_t* tl = tail + ((size_t)l * B + seq) * TL;
        for (size_t i = 0; i < TL; ++i, p += 2) tl[i] = (uint16_t)(p[0] | (p[1] << 8));
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* gate front end and gated-norm output                                       */
/* ------------------------------------------------------------------------ */

double orc_softplus(double x) { return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x))); }

double orc_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

void orc_gates(int n, int Hv, const uint16_t* a, const uint16_t* b, const float* A_log, const float* dt_bias,
               double* alpha, double* beta) {
    for (int t = 0; t < n; ++t)
        for (int h = 0; h < Hv; ++h) {
            const size_t i = (size_t)t * Hv + h;
            const double dt = orc_softplus(orc_bf16_to_f64(a[i]) + (double)dt_bias[h]);
            alpha[i] = exp(-exp((double)A_log[h]) * dt);
            beta[i] = orc_sigmoid(orc_bf16_to_f64(b[i]));
        }
}

void orc_gated_rmsnorm(int dv, const double* o, const uint16_t* z, const float* w, double eps, double* y) {
    double ss = 0.0;
    for (int i = 0; i < dv; ++i) ss += o[i] * o[i];
    const double inv = 1.0 / sqrt(ss / dv + eps);
    for (int i = 0; i < dv; ++i) y[i] = o[i] * inv * (double)w[i] * orc_silu(orc_bf16_to_f64(z[i]));
}

void orc_layer_decode(int B, int T, int Hk, int Hv, int dk, int dv, const uint16_t* x, const uint16_t* conv_w,
                      uint16_t* tail, const uint16_t* a, const uint16_t* b, const float* A_log,
                      const float* dt_bias, const uint16_t* z, const float* norm_w, double eps, double* state,
                      double* o, double* y, double q_scale, int normalize) {
    const size_t C = (size_t)2 * Hk * dk + (size_t)Hv * dv;
    const int group = Hv / Hk;
    const size_t n = (size_t)B * T;
    double* yc = (double*)malloc(sizeof(double) * n * C);
    uint16_t* qkv = (uint16_t*)malloc(sizeof(uint16_t) * n * C);
    double* alpha = (double*)malloc(sizeof(double) * n * Hv);
    double* beta = (double*)malloc(sizeof(double) * n * Hv);
    double* q = (double*)malloc(sizeof(double) * (size_t)dk);
    double* k = (double*)malloc(sizeof(double) * (size_t)dk);
    double* v = (double*)malloc(sizeof(double) * (size_t)dv);
    orc_conv_linear(B, T, (int)C, 4, x, conv_w, tail, yc);
    orc_f64_to_bf16_n(yc, qkv, (int64_t)(n * C));       /* the conv output is stored as bf16 */
    orc_gates((int)n, Hv, a, b, A_log, dt_bias, alpha, beta);
    for (size_t tok = 0; tok < n; ++tok)
        for (int h = 0; h < Hv; ++h) {
            token_vectors(Hk, dk, dv, qkv + tok * C, h / group, h, q_scale, normalize, q, k, v);
            double* S = state + ((tok / T) * Hv + h) * (size_t)dv * dk;
            double* oh = o + (tok * Hv + h) * dv;
            orc_delta_token(dk, dv, S, k, v, q, alpha[tok * Hv + h], beta[tok * Hv + h], oh);
            orc_gated_rmsnorm(dv, oh, z + (tok * Hv + h) * dv, norm_w, eps, y + (tok * Hv + h) * dv);
        }
    free(v);
    free(k);
    free(q);
    free(beta);
    free(alpha);
    free(qkv);
    free(yc);
}
