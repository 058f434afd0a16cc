// gdn_api.cu -- host side of the C ABI declared in include/gdn.h: argument
// validation, tree bookkeeping and kernel launches.  Every check runs before
// anything is enqueued, so a failing call leaves all buffers untouched and
// the stream unchanged.  Unsupported shapes are refused with an error code
// rather than run (the lesson of the hardcoded head-size bug in "Serving A
// Research Architecture On CPU").  Nothing here allocates device memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "gdn_internal.h"

using namespace gdn;

namespace {

thread_local std::string t_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(GDN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool head_size_ok(int d) { return d == 32 || d == 64 || d == 128; }

int check_shape(const gdn_shape* s, bool need_single) {
    if (s == nullptr) return fail(GDN_ERR_INVALID_ARG, "shape is NULL");
    if (s->B < 0 || s->Hk < 1 || s->Hv < 1)
        return fail(GDN_ERR_UNSUPPORTED_SHAPE, "bad head counts / batch: B=%d Hk=%d Hv=%d", s->B,
                    s->Hk, s->Hv);
    if (s->Hv % s->Hk != 0)
        return fail(GDN_ERR_UNSUPPORTED_SHAPE, "Hv=%d is not a multiple of Hk=%d", s->Hv, s->Hk);
    if (!head_size_ok(s->dk) || !head_size_ok(s->dv))
        return fail(GDN_ERR_UNSUPPORTED_SHAPE, "head sizes dk=%d dv=%d not in {32, 64, 128}", s->dk,
                    s->dv);
    if (s->Hv > 65535 || s->B > 65535)
        return fail(GDN_ERR_UNSUPPORTED_SHAPE, "B=%d / Hv=%d exceed the grid limit 65535", s->B, s->Hv);
    if (need_single && s->B != 1)
        return fail(GDN_ERR_UNSUPPORTED_SHAPE, "this call takes one sequence (B=%d)", s->B);
    return GDN_OK;
}

int packed_channels(const gdn_shape* s) { return 2 * s->Hk * s->dk + s->Hv * s->dv; }

// `extra`: flag bits this call accepts beyond the common two.
int check_flags(uint32_t flags, uint32_t extra = 0) {
    if (flags & ~(GDN_NORMALIZE_QK | GDN_OUT_BF16 | extra))
        return fail(GDN_ERR_INVALID_ARG, "unknown flag bits 0x%x for this call", flags);
    return GDN_OK;
}

int check_ptr(const void* p, const char* name, bool required = true) {
    if (p == nullptr) {
        if (required) return fail(GDN_ERR_INVALID_ARG, "%s is NULL", name);
        return GDN_OK;
    }
    if (!aligned16(p)) return fail(GDN_ERR_MISALIGNED, "%s (%p) is not 16-byte aligned", name, p);
    return GDN_OK;
}

// Parent array -> OK or GDN_ERR_BAD_PARENTS (one tree rooted at node 0).
int check_parents(int N, const int32_t* parents) {
    if (parents == nullptr) return fail(GDN_ERR_INVALID_ARG, "parents is NULL");
    if (N < 1 || N > GDN_MAX_TREE_NODES)
        return fail(GDN_ERR_BAD_PARENTS, "tree size N=%d outside [1, %d]", N, GDN_MAX_TREE_NODES);
    if (parents[0] != -1) return fail(GDN_ERR_BAD_PARENTS, "parents[0]=%d, the root must be -1", parents[0]);
    for (int i = 1; i < N; ++i)
        if (parents[i] < 0 || parents[i] >= i)
            return fail(GDN_ERR_BAD_PARENTS, "parents[%d]=%d, need 0 <= parent < %d", i, parents[i], i);
    return GDN_OK;
}

// Depth-first preorder walk with branch-state slots (see TreeStep).
int schedule_tree(int N, const int32_t* parents, TreeStep* steps, int* n_slots) {
    std::vector<std::vector<int>> children(N);
    for (int i = 1; i < N; ++i) children[parents[i]].push_back(i);
    std::vector<int> order;
    order.reserve(N);
    std::vector<int> stack{0};
    while (!stack.empty()) {
        const int n = stack.back();
        stack.pop_back();
        order.push_back(n);
        for (int c = (int)children[n].size() - 1; c >= 0; --c) stack.push_back(children[n][c]);
    }
    std::vector<int> slot_of(N, -1);
    int depth = 0, max_depth = 0, prev = -1;
    for (int k = 0; k < N; ++k) {
        const int n = order[k];
        int restore = -1;
        if (n != 0) {
            const int par = parents[n];
            if (prev != par) {
                restore = slot_of[par];
                if (restore < 0) return fail(GDN_ERR_BAD_PARENTS, "internal: no saved state for node %d", par);
            }
            if (slot_of[par] >= 0 && n == children[par].back()) {
                if (slot_of[par] != depth - 1)
                    return fail(GDN_ERR_BAD_PARENTS, "internal: slot stack out of order at node %d", n);
                depth -= 1;
            }
        }
        int save = -1;
        if (children[n].size() >= 2) {
            save = depth++;
            slot_of[n] = save;
            if (depth > max_depth) max_depth = depth;
        }
        if (max_depth > GDN_MAX_TREE_SLOTS)
            return fail(GDN_ERR_DEPTH_EXCEEDED,
                        "tree keeps %d branch states at once (more than %d nested branching nodes)",
                        max_depth, GDN_MAX_TREE_SLOTS);
        steps[k].node = (int8_t)n;
        steps[k].restore = (int8_t)restore;
        steps[k].save = (int8_t)save;
        steps[k].store = 1;
        prev = n;
    }
    *n_slots = max_depth;
    return GDN_OK;
}

// The walk of one walker: a depth-first preorder over `member` (a
// set of nodes closed under taking parents, so a subtree holding the root),
// writing the outputs of the nodes in `own`.  The children of a node are
// visited in increasing order of the branch slots their own subtrees need,
// so that the parent's slot is released before the most demanding child
// (the fewest slots any preorder can use); slots are numbered from `base`.
// Returns the steps taken; *n_slots gets the slots used.
int schedule_walker(int N, const int32_t* parents, const char* member, const char* own, int base, TreeStep* steps,
                    int* n_slots) {
    // children lists in fixed arrays (N <= GDN_MAX_TREE_NODES): kids[n][0 .. nk[n])
    int8_t kids[GDN_MAX_TREE_NODES][GDN_MAX_TREE_NODES];
    int nk[GDN_MAX_TREE_NODES] = {};
    for (int i = 1; i < N; ++i)
        if (member[i]) kids[parents[i]][nk[parents[i]]++] = (int8_t)i;
    // slots a subtree needs (children in increasing order of need): the
    // parent's slot is held through every child but the last
    int need[GDN_MAX_TREE_NODES] = {};
    for (int n = N - 1; n >= 0; --n) {  // children have larger indices than their parent
        if (!member[n]) continue;
        int8_t* c = kids[n];
        for (int a = 1; a < nk[n]; ++a)  // stable insertion sort by need
            for (int b = a; b > 0 && need[c[b - 1]] > need[c[b]]; --b) std::swap(c[b - 1], c[b]);
        if (nk[n] == 1) need[n] = need[c[0]];
        else if (nk[n] >= 2) need[n] = std::max(need[c[nk[n] - 1]], need[c[nk[n] - 2]] + 1);
    }
    int slot_of[GDN_MAX_TREE_NODES];
    int stack[GDN_MAX_TREE_NODES];
    int sp = 0, k = 0, depth = 0, max_depth = 0, prev = -1;
    stack[sp++] = 0;
    while (sp > 0) {
        const int n = stack[--sp];
        for (int c = nk[n] - 1; c >= 0; --c) stack[sp++] = kids[n][c];
        slot_of[n] = -1;
        int restore = -1;
        if (n != 0) {
            const int par = parents[n];
            if (prev != par) restore = slot_of[par];
            if (slot_of[par] >= 0 && n == kids[par][nk[par] - 1]) depth -= 1;  // the last child frees the slot
        }
        int save = -1;
        if (nk[n] >= 2) {
            save = base + depth++;
            slot_of[n] = save;
            max_depth = std::max(max_depth, depth);
        }
        steps[k].node = (int8_t)n;
        steps[k].restore = (int8_t)restore;
        steps[k].save = (int8_t)save;
        steps[k].store = own[n] ? 1 : 0;
        prev = n;
        ++k;
    }
    *n_slots = max_depth;
    return k;
}

// Walkers for one tree: the preorder (children by slot need) cut into P
// contiguous ranges, walker w taking range w and replaying, without storing
// them, the ancestors of its nodes that lie before the range.  Each node's
// output is written by exactly one walker, with the arithmetic and operand
// order of the single walk, so the bits are the same.  The cuts minimise the
// longest walk: for a bound L, ranges taken greedily as long as their walks
// stay within L (a walk only grows as its range does) cover the tree iff any
// cuts do, and L rises from N / P until they do.  Left at walkers = 1 when
// the longest walk would not be at least a quarter shorter than the single
// walk (chains, small trees).
void split_walkers(int N, const int32_t* parents, int P, TreeParams& p) {
    p.walkers = 1;
    if (P < 2 || N < 8) return;
    char all[GDN_MAX_TREE_NODES];
    memset(all, 1, sizeof all);
    TreeStep order_steps[GDN_MAX_TREE_NODES];
    int slots = 0;
    schedule_walker(N, parents, all, all, 0, order_steps, &slots);
    int order[GDN_MAX_TREE_NODES];
    for (int k = 0; k < N; ++k) order[k] = order_steps[k].node;
    // a walk is at least as long as its deepest node's root path
    int depth[GDN_MAX_TREE_NODES], max_depth = 1;
    depth[0] = 1;
    for (int n = 1; n < N; ++n) max_depth = std::max(max_depth, depth[n] = depth[parents[n]] + 1);
    int cut[kMaxWalkers + 1] = {};
    int best = N;
    for (int L = std::max((N + P - 1) / P, max_depth); 4 * L <= 3 * N; ++L) {
        int k = 0, w = 0;
        for (; w < P && k < N; ++w) {
            char m[GDN_MAX_TREE_NODES] = {};
            int len = 0;
            cut[w] = k;
            for (; k < N; ++k) {
                int add = 0;
                for (int a = order[k]; a >= 0 && !m[a]; a = parents[a]) ++add;
                if (len + add > L) break;
                for (int a = order[k]; a >= 0 && !m[a]; a = parents[a]) m[a] = 1;
                len += add;
            }
        }
        if (k == N) {
            best = L;
            P = w;  // the walkers the cuts use
            cut[P] = N;
            break;
        }
    }
    if (P < 2 || 4 * best > 3 * N) return;
    int s_max = 0;
    for (int w = 0; w < P; ++w) {
        char mw[GDN_MAX_TREE_NODES] = {}, own[GDN_MAX_TREE_NODES] = {};
        for (int j = cut[w]; j < cut[w + 1]; ++j) {
            own[order[j]] = 1;
            for (int a = order[j]; a >= 0 && !mw[a]; a = parents[a]) mw[a] = 1;
        }
        int sw = 0;
        p.walk_n[w] = schedule_walker(N, parents, mw, own, 0, p.walk[w], &sw);
        s_max = std::max(s_max, sw);
    }
    p.walk_slots = s_max;
    p.walkers = P;
}

int check_path(int N, const int32_t* parents, const int32_t* path, int L) {
    if (L < 0) return fail(GDN_ERR_INVALID_ARG, "path length L=%d < 0", L);
    if (L == 0) return GDN_OK;
    if (path == nullptr) return fail(GDN_ERR_INVALID_ARG, "path is NULL");
    for (int i = 0; i < L; ++i)
        if (path[i] < 0 || path[i] >= N) return fail(GDN_ERR_BAD_PATH, "path[%d]=%d outside [0, %d)", i, path[i], N);
    if (parents[path[0]] != -1) return fail(GDN_ERR_BAD_PATH, "path[0]=%d is not the root", path[0]);
    for (int i = 1; i < L; ++i)
        if (parents[path[i]] != path[i - 1])
            return fail(GDN_ERR_BAD_PATH, "path[%d]=%d is not a child of path[%d]=%d", i, path[i], i - 1,
                        path[i - 1]);
    return GDN_OK;
}

// The tree conv's ancestor table: node n's m-th earlier input (m = 0 .. 2,
// nearest first) is its m+1-th ancestor, or, past the root, the tail's slots
// from the newest down (-1 - slot).
void conv_ancestors(int N, const int32_t* parents, int8_t (*anc)[3]) {
    for (int n = 0; n < N; ++n) {
        int a = n, tail_slot = GDN_CONV_W - 1;
        for (int m = 0; m < GDN_CONV_W - 1; ++m) {
            if (a >= 0) a = parents[a];
            if (a >= 0) {
                anc[n][m] = (int8_t)a;
            } else {
                anc[n][m] = (int8_t)(-1 - tail_slot);
                tail_slot -= 1;
            }
        }
    }
}

// true when [a, a + n) and [b, b + n) share a byte
bool overlaps(const void* a, const void* b, size_t n) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + n && y < x + n;
}

int sm_count() {
    // relaxed atomics: host threads may race to fill an entry, all with the same value
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Rows of one head per CTA for decode: the widest (fewest CTAs, most loads in
// flight per thread) that still gives every SM a few CTAs.
int decode_rows_per_cta(int B, int Hv, int dv) {
    const long heads = (long)B * Hv;
    const long want = 4L * sm_count();
    for (int rows = 128; rows > 32; rows /= 2) {
        if (dv % rows != 0) continue;
        if (heads * (dv / rows) >= want) return rows;
    }
    return 32;
}

}  // namespace

namespace gdn {

int cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }

int check_shape_arg(const gdn_shape* s, bool need_single) { return check_shape(s, need_single); }

int check_pointer(const void* p, const char* name) { return check_ptr(p, name); }

int device_sm_count() { return sm_count(); }

int report_error(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    return fail(code, "%s", buf);
}

int check_prefill_args(const gdn_shape* shape, int T, int chunk, const void* qkv, const void* alpha,
                       const void* beta, const void* state, const void* out, const void* workspace,
                       size_t workspace_bytes, uint32_t flags, bool records) {
    int rc;
    if ((rc = check_shape(shape, true)) != GDN_OK) return rc;
    if ((rc = check_flags(flags & ~(records ? GDN_PREFILL_TWO_LAUNCH : 0u))) != GDN_OK) return rc;
    if (chunk != 64) return fail(GDN_ERR_INVALID_ARG, "chunk=%d, only 64 is supported", chunk);
    if (T < 0) return fail(GDN_ERR_INVALID_ARG, "T=%d < 0", T);
    if (T == 0) return GDN_OK;  // nothing to do; pointers may be NULL
    if ((rc = check_ptr(qkv, "qkv")) || (rc = check_ptr(alpha, "alpha")) || (rc = check_ptr(beta, "beta")) ||
        (rc = check_ptr(state, "state")) || (rc = check_ptr(out, "out")))
        return rc;
    if (workspace == nullptr) return fail(GDN_ERR_WORKSPACE, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(GDN_ERR_MISALIGNED, "workspace (%p) is not 256-byte aligned", workspace);
    // with records: the pre-pass records as well as the status word
    const size_t need = records ? gdn_prefill_workspace_bytes(shape, T, chunk) : 256;
    if (workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
    return GDN_OK;
}

}  // namespace gdn

extern "C" {

int gdn_abi_version(void) { return GDN_ABI_VERSION; }

const char* gdn_last_error(void) { return t_error.c_str(); }

size_t gdn_state_bytes(const gdn_shape* s) {
    if (check_shape(s, false) != GDN_OK) return 0;
    return (size_t)s->B * s->Hv * s->dv * s->dk * sizeof(float);
}

int gdn_tree_root_path(int32_t N, const int32_t* parents, int32_t node, int32_t* path, int32_t cap) {
    int rc = check_parents(N, parents);
    if (rc != GDN_OK) return rc;
    if (node < 0 || node >= N) return fail(GDN_ERR_INVALID_ARG, "node %d outside [0, %d)", node, N);
    if (path == nullptr) return fail(GDN_ERR_INVALID_ARG, "path is NULL");
    int len = 0;
    for (int m = node; m >= 0; m = parents[m]) ++len;
    if (len > cap) return fail(GDN_ERR_INVALID_ARG, "path of length %d does not fit cap=%d", len, cap);
    int pos = len - 1;
    for (int m = node; m >= 0; m = parents[m]) path[pos--] = m;
    return len;
}

int gdn_conv_step(int32_t B, int32_t T, int32_t C, const int32_t* parents, const void* x, const void* w,
                  void* tail, void* y, uint32_t flags, void* stream) {
    int rc;
    if ((rc = check_flags(flags, GDN_IN_F32)) != GDN_OK) return rc;
    if (flags & (GDN_NORMALIZE_QK | GDN_OUT_BF16))
        return fail(GDN_ERR_INVALID_ARG, "the conv takes only GDN_IN_F32 (flags 0x%x)", flags);
    if (B < 0 || T < 0 || C < 0) return fail(GDN_ERR_INVALID_ARG, "negative size B=%d T=%d C=%d", B, T, C);
    if (C % 8 != 0) return fail(GDN_ERR_UNSUPPORTED_SHAPE, "channels C=%d not a multiple of 8", C);
    if (B > 65535) return fail(GDN_ERR_UNSUPPORTED_SHAPE, "B=%d exceeds 65535", B);
    if (parents != nullptr && (rc = check_parents(T, parents)) != GDN_OK) return rc;
    if (B == 0 || T == 0 || C == 0) return GDN_OK;  // nothing to do; pointers may be NULL
    if ((rc = check_ptr(x, "x")) || (rc = check_ptr(w, "w")) || (rc = check_ptr(tail, "tail")) ||
        (rc = check_ptr(y, "y")))
        return rc;
    ConvParams p{};
    p.x = x;
    p.w = w;
    p.tail = tail;
    p.y = y;
    p.B = B;
    p.T = T;
    p.C = C;
    p.f32 = (flags & GDN_IN_F32) != 0;
    p.tree = parents != nullptr;
    if (p.tree) conv_ancestors(T, parents, p.anc);
    cudaError_t e = launch_conv(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "conv launch");
}

// The decode step with a decay per head (kda = false) or per key channel.
static int decode_impl(const gdn_shape* shape, int32_t T, const void* qkv, const float* alpha,
                       const float* beta, float* state, void* out, float q_scale, uint32_t flags,
                       void* stream, bool kda) {
    int rc;
    if ((rc = check_shape(shape, false)) != GDN_OK) return rc;
    if ((rc = check_flags(flags, kda ? 0u : GDN_IN_F32)) != GDN_OK) return rc;
    if (T < 0) return fail(GDN_ERR_INVALID_ARG, "T=%d < 0", T);
    if (shape->B == 0 || T == 0) return GDN_OK;  // nothing to do; pointers may be NULL
    if ((rc = check_ptr(qkv, "qkv")) || (rc = check_ptr(alpha, "alpha")) || (rc = check_ptr(beta, "beta")) ||
        (rc = check_ptr(state, "state")) || (rc = check_ptr(out, "out", false)))
        return rc;
    const bool in_f32 = (flags & GDN_IN_F32) != 0;
    DecodeParams p{};
    p.qkv = static_cast<const uint16_t*>(qkv);
    p.alpha = alpha;
    p.beta = beta;
    p.state = state;
    p.out = out;
    p.B = shape->B;
    p.T = T;
    p.Tsrc = T;
    p.Hk = shape->Hk;
    p.Hv = shape->Hv;
    p.dv = shape->dv;
    p.group = shape->Hv / shape->Hk;
    p.C = packed_channels(shape);
    p.q_scale = q_scale;
    p.normalize = (flags & GDN_NORMALIZE_QK) != 0;
    p.out_bf16 = (flags & GDN_OUT_BF16) != 0;
    const int rows = decode_rows_per_cta(shape->B, shape->Hv, shape->dv);
    cudaError_t e = launch_decode(p, shape->dk, rows, 0, kda, in_f32, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, kda ? "KDA decode launch" : "decode launch");
}

int gdn_decode_step(const gdn_shape* shape, int32_t T, const void* qkv, const float* alpha,
                    const float* beta, float* state, void* out, float q_scale, uint32_t flags,
                    void* stream) {
    return decode_impl(shape, T, qkv, alpha, beta, state, out, q_scale, flags, stream, false);
}

int gdn_kda_decode_step(const gdn_shape* shape, int32_t T, const gdn_bf16* qkv, const float* alpha,
                        const float* beta, float* state, void* out, float q_scale, uint32_t flags,
                        void* stream) {
    return decode_impl(shape, T, qkv, alpha, beta, state, out, q_scale, flags, stream, true);
}

// The fused step: kind 0 plain, 1 KDA, 2 the layer step (gates from the
// projections in `layer`, alpha/beta unused; gated-norm output to layer->y).
static int conv_decode_impl(const gdn_shape* shape, int32_t T, const gdn_bf16* x, const gdn_bf16* w,
                            const gdn_bf16* tail_in, gdn_bf16* tail_out, const float* alpha, const float* beta,
                            float* state, void* out, float q_scale, uint32_t flags, void* stream, int kind,
                            const LayerParams* layer = nullptr) {
    const bool kda = kind == 1;
    int rc;
    if ((rc = check_shape(shape, false)) != GDN_OK) return rc;
    if ((rc = check_flags(flags)) != GDN_OK) return rc;
    if (T < 0) return fail(GDN_ERR_INVALID_ARG, "T=%d < 0", T);
    if (T > kFusedMaxTokens)
        return fail(GDN_ERR_UNSUPPORTED_SHAPE, "T=%d tokens, the fused step takes at most %d", T, kFusedMaxTokens);
    const int group = shape->Hv / shape->Hk;
    const int CC = 2 * shape->dk + group * shape->dv;
    // staged per token: the group's conv outputs (bf16) and, for KDA, its decay vectors (fp32)
    const long per_token = (long)CC * 2 + (kda ? (long)group * shape->dk * 4 : 0) + (kind == 2 ? (long)group * 8 : 0);
    if ((long)T * per_token > kFusedMaxSmem)
        return fail(GDN_ERR_UNSUPPORTED_SHAPE, "T=%d x %ld staged bytes per key-head group exceed the fused "
                    "step's %d-byte staging", T, per_token, kFusedMaxSmem);
    if (shape->B == 0 || T == 0) return GDN_OK;  // nothing to do; pointers may be NULL
    if ((rc = check_ptr(x, "x")) || (rc = check_ptr(w, "w")) || (rc = check_ptr(tail_in, "tail_in")) ||
        (rc = check_ptr(tail_out, "tail_out")) || (rc = check_ptr(state, "state")) ||
        (rc = check_ptr(out, "out", false)))
        return rc;
    if (kind != 2 && ((rc = check_ptr(alpha, "alpha")) || (rc = check_ptr(beta, "beta")))) return rc;
    const int C = packed_channels(shape);
    const size_t tail_bytes = (size_t)shape->B * GDN_CONV_W * C * 2;
    const uintptr_t ti = reinterpret_cast<uintptr_t>(tail_in), to = reinterpret_cast<uintptr_t>(tail_out);
    if (ti != to && (ti < to + tail_bytes && to < ti + tail_bytes))
        return fail(GDN_ERR_INVALID_ARG, "tail_in and tail_out overlap without being equal");
    ConvDecodeParams p{};
    p.x = x;
    p.w = w;
    p.tail_in = tail_in;
    p.tail_out = tail_out;
    p.alpha = alpha;
    p.beta = beta;
    p.state = state;
    p.out = out;
    p.B = shape->B;
    p.T = T;
    p.Hk = shape->Hk;
    p.Hv = shape->Hv;
    p.dv = shape->dv;
    p.group = group;
    p.C = C;
    p.CC = CC;
    p.q_scale = q_scale;
    p.normalize = (flags & GDN_NORMALIZE_QK) != 0;
    p.out_bf16 = (flags & GDN_OUT_BF16) != 0;
    // Rows of each value head per CTA: all of them when the tail is updated in
    // place (one writer per tail entry); with distinct tails, split the rows
    // until every SM has a few CTAs.
    if (layer != nullptr) p.layer = *layer;
    int row_blocks = 1, head_parts = 1;
    if (ti != to) {
        const long want = 4L * sm_count();
        if (kind != 2) {  // the layer step's norm needs every row of a head in one CTA
            while (row_blocks < 4 && shape->dv / (row_blocks * 2) >= 32 &&
                   (long)shape->Hk * shape->B * row_blocks < want)
                row_blocks *= 2;
        }
        // still short of a few CTAs per SM: one value head per CTA
        if ((long)shape->Hk * shape->B * row_blocks < want) head_parts = group;
    }
    p.row_blocks = row_blocks;
    p.head_parts = head_parts;
    cudaError_t e =
        launch_conv_decode(p, shape->dk, shape->dv / row_blocks, kind, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK
                            : cuda_fail(e, kind == 1 ? "conv+KDA decode launch"
                                                     : kind == 2 ? "layer decode launch" : "conv+decode launch");
}

int gdn_conv_decode_step(const gdn_shape* shape, int32_t T, const gdn_bf16* x, const gdn_bf16* w,
                         const gdn_bf16* tail_in, gdn_bf16* tail_out, const float* alpha, const float* beta,
                         float* state, void* out, float q_scale, uint32_t flags, void* stream) {
    return conv_decode_impl(shape, T, x, w, tail_in, tail_out, alpha, beta, state, out, q_scale, flags, stream,
                            0);
}

int gdn_kda_conv_decode_step(const gdn_shape* shape, int32_t T, const gdn_bf16* x, const gdn_bf16* w,
                             const gdn_bf16* tail_in, gdn_bf16* tail_out, const float* alpha, const float* beta,
                             float* state, void* out, float q_scale, uint32_t flags, void* stream) {
    return conv_decode_impl(shape, T, x, w, tail_in, tail_out, alpha, beta, state, out, q_scale, flags, stream,
                            1);
}

int gdn_layer_decode_step(const gdn_shape* shape, int32_t T, const gdn_bf16* x, const gdn_bf16* conv_w,
                          const gdn_bf16* tail_in, gdn_bf16* tail_out, const gdn_bf16* a, const gdn_bf16* b,
                          const float* A_log, const float* dt_bias, const gdn_bf16* z, const float* norm_w,
                          float norm_eps, float* state, float* o, gdn_bf16* y, float q_scale, uint32_t flags,
                          void* stream) {
    int rc;
    if ((rc = check_shape(shape, false)) != GDN_OK) return rc;
    if (flags & GDN_OUT_BF16)
        return fail(GDN_ERR_INVALID_ARG, "the layer step writes y in bf16 and o in fp32; GDN_OUT_BF16 not allowed");
    if (!(norm_eps >= 0.0f) || norm_eps > 1.0f)
        return fail(GDN_ERR_INVALID_ARG, "norm_eps=%g outside [0, 1]", (double)norm_eps);
    if (T < 0) return fail(GDN_ERR_INVALID_ARG, "T=%d < 0", T);
    if (shape->B == 0 || T == 0) return GDN_OK;  // nothing to do; pointers may be NULL
    if ((rc = check_ptr(a, "a")) || (rc = check_ptr(b, "b")) || (rc = check_ptr(A_log, "A_log")) ||
        (rc = check_ptr(dt_bias, "dt_bias")) || (rc = check_ptr(z, "z")) || (rc = check_ptr(norm_w, "norm_w")) ||
        (rc = check_ptr(y, "y")))
        return rc;
    LayerParams lp{};
    lp.a = a;
    lp.b = b;
    lp.A_log = A_log;
    lp.dt_bias = dt_bias;
    lp.z = z;
    lp.norm_w = norm_w;
    lp.y = y;
    lp.norm_eps = norm_eps;
    return conv_decode_impl(shape, T, x, conv_w, tail_in, tail_out, nullptr, nullptr, state, o, q_scale, flags,
                            stream, 2, &lp);
}

int gdn_gates(int64_t n, int32_t Hv, const gdn_bf16* a, const gdn_bf16* b, const float* A_log,
              const float* dt_bias, float* alpha, float* beta, void* stream) {
    int rc;
    if (n < 0 || Hv < 1) return fail(GDN_ERR_INVALID_ARG, "n=%lld tokens, Hv=%d heads", (long long)n, Hv);
    if (n == 0) return GDN_OK;
    if ((rc = check_ptr(a, "a")) || (rc = check_ptr(b, "b")) || (rc = check_ptr(A_log, "A_log")) ||
        (rc = check_ptr(dt_bias, "dt_bias")) || (rc = check_ptr(alpha, "alpha")) || (rc = check_ptr(beta, "beta")))
        return rc;
    if (n * (int64_t)Hv > (int64_t)1 << 38) return fail(GDN_ERR_INVALID_ARG, "n * Hv above 2^38");
    GatesParams p{};
    p.a = a;
    p.b = b;
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    p.alpha = alpha;
    p.beta = beta;
    p.n = n;
    p.Hv = Hv;
    cudaError_t e = launch_gates(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gates launch");
}

}  // extern "C"

namespace {

// Tree verify of one tree (conv == false: post-conv qkv) or with the tree
// conv fused in (x, w, tail: pre-conv inputs).
int tree_verify_impl(const gdn_shape* shape, int32_t N, const int32_t* parents, const gdn_bf16* qkv,
                     const gdn_bf16* x, const gdn_bf16* w, const gdn_bf16* tail, bool conv, const float* alpha,
                     const float* beta, const float* state, void* out, float q_scale, uint32_t flags,
                     void* stream, bool kda = false) {
    int rc;
    if ((rc = check_shape(shape, true)) != GDN_OK) return rc;
    if ((rc = check_flags(flags)) != GDN_OK) return rc;
    if ((rc = check_parents(N, parents)) != GDN_OK) return rc;
    if (conv) {
        if ((rc = check_ptr(x, "x")) || (rc = check_ptr(w, "w")) || (rc = check_ptr(tail, "tail"))) return rc;
    } else if ((rc = check_ptr(qkv, "qkv")) != GDN_OK) {
        return rc;
    }
    if ((rc = check_ptr(alpha, "alpha")) || (rc = check_ptr(beta, "beta")) || (rc = check_ptr(state, "state")) ||
        (rc = check_ptr(out, "out")))
        return rc;
    TreeParams p{};
    if ((rc = schedule_tree(N, parents, p.steps[0], &p.n_slots)) != GDN_OK) return rc;
    // As many walkers (up to kMaxWalkers) as keep the grid -- walkers x row
    // blocks of 64 x value heads -- within two CTAs per SM.
    int walkers = kMaxWalkers;
    while (walkers > 1 && (long)walkers * (shape->dv / 64) * shape->Hv > 2L * sm_count()) --walkers;
    split_walkers(N, parents, walkers, p);
    p.qkv = qkv;
    if (conv) {
        p.x = x;
        p.w = w;
        p.tail = tail;
        conv_ancestors(N, parents, p.anc[0]);
    }
    p.alpha = alpha;
    p.beta = beta;
    p.state = state;
    p.out = out;
    p.B = 1;
    p.Nmax = N;
    p.N[0] = N;
    p.Hk = shape->Hk;
    p.Hv = shape->Hv;
    p.dv = shape->dv;
    p.group = shape->Hv / shape->Hk;
    p.C = packed_channels(shape);
    p.q_scale = q_scale;
    p.normalize = (flags & GDN_NORMALIZE_QK) != 0;
    p.out_bf16 = (flags & GDN_OUT_BF16) != 0;
    p.kda = kda;
    cudaError_t e = launch_tree(p, shape->dk, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK
                            : cuda_fail(e, kda ? "KDA tree verify launch"
                                               : conv ? "conv + tree verify launch" : "tree verify launch");
}

int tree_verify_batched_impl(const gdn_shape* shape, int32_t N, const int32_t* counts, const int32_t* parents,
                             const gdn_bf16* qkv, const gdn_bf16* x, const gdn_bf16* w, const gdn_bf16* tail,
                             bool conv, const float* alpha, const float* beta, const float* state, void* out,
                             float q_scale, uint32_t flags, void* stream, bool kda = false) {
    int rc;
    if ((rc = check_shape(shape, false)) != GDN_OK) return rc;
    if ((rc = check_flags(flags)) != GDN_OK) return rc;
    if (shape->B < 1 || shape->B > kMaxTreeBatch)
        return fail(GDN_ERR_UNSUPPORTED_SHAPE, "B=%d trees, one call verifies 1 .. %d", shape->B, kMaxTreeBatch);
    if (N < 1 || N > GDN_MAX_TREE_NODES)
        return fail(GDN_ERR_BAD_PARENTS, "node capacity N=%d outside [1, %d]", N, GDN_MAX_TREE_NODES);
    if (counts == nullptr || parents == nullptr) return fail(GDN_ERR_INVALID_ARG, "counts / parents is NULL");
    if (conv) {
        if ((rc = check_ptr(x, "x")) || (rc = check_ptr(w, "w")) || (rc = check_ptr(tail, "tail"))) return rc;
    } else if ((rc = check_ptr(qkv, "qkv")) != GDN_OK) {
        return rc;
    }
    if ((rc = check_ptr(alpha, "alpha")) || (rc = check_ptr(beta, "beta")) || (rc = check_ptr(state, "state")) ||
        (rc = check_ptr(out, "out")))
        return rc;
    static thread_local TreeParamsBatch p;  // 14 KB of schedules and ancestor tables: kept off the stack
    p = TreeParamsBatch{};
    for (int b = 0; b < shape->B; ++b) {
        if (counts[b] < 1 || counts[b] > N)
            return fail(GDN_ERR_BAD_PARENTS, "tree %d has %d nodes, need 1 .. %d", b, counts[b], N);
        if ((rc = check_parents(counts[b], parents + (size_t)b * N)) != GDN_OK) {
            const std::string why = t_error;
            return fail(rc, "tree %d: %s", b, why.c_str());
        }
        int slots = 0;
        if ((rc = schedule_tree(counts[b], parents + (size_t)b * N, p.steps[b], &slots)) != GDN_OK) {
            const std::string why = t_error;
            return fail(rc, "tree %d: %s", b, why.c_str());
        }
        if (conv) conv_ancestors(counts[b], parents + (size_t)b * N, p.anc[b]);
        p.N[b] = counts[b];
        if (slots > p.n_slots) p.n_slots = slots;
    }
    p.qkv = qkv;
    if (conv) {
        p.x = x;
        p.w = w;
        p.tail = tail;
    }
    p.alpha = alpha;
    p.beta = beta;
    p.state = state;
    p.out = out;
    p.B = shape->B;
    p.Nmax = N;
    p.Hk = shape->Hk;
    p.Hv = shape->Hv;
    p.dv = shape->dv;
    p.group = shape->Hv / shape->Hk;
    p.C = packed_channels(shape);
    p.q_scale = q_scale;
    p.normalize = (flags & GDN_NORMALIZE_QK) != 0;
    p.out_bf16 = (flags & GDN_OUT_BF16) != 0;
    p.kda = kda;
    cudaError_t e = launch_tree(p, shape->dk, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK
                            : cuda_fail(e, kda ? "batched KDA tree verify launch"
                                               : conv ? "batched conv + tree verify launch" : "batched tree verify launch");
}

// Commit of B sequences' paths through the batched kernel.  Fused conv when
// w != nullptr: x_tree and tail_in required, tail_out written for every
// sequence (distinct from tail_in); else qkv required and tail updated in
// place when x_tree is given.
int commit_batched_impl(const gdn_shape* shape, int32_t N, const int32_t* counts, const int32_t* parents,
                        const int32_t* paths, const int32_t* lengths, const gdn_bf16* qkv, const float* alpha,
                        const float* beta, const gdn_bf16* x_tree, float* state, gdn_bf16* tail,
                        const gdn_bf16* w, const gdn_bf16* tail_in, uint32_t flags, void* stream) {
    const bool conv = w != nullptr;
    int rc;
    if ((rc = check_shape(shape, false)) != GDN_OK) return rc;
    if (flags & GDN_OUT_BF16) return fail(GDN_ERR_INVALID_ARG, "commit writes no output; GDN_OUT_BF16 not allowed");
    if ((rc = check_flags(flags)) != GDN_OK) return rc;
    if (shape->B < 1 || shape->B > kMaxTreeBatch)
        return fail(GDN_ERR_UNSUPPORTED_SHAPE, "B=%d trees, one call commits 1 .. %d", shape->B, kMaxTreeBatch);
    if (N < 1 || N > GDN_MAX_TREE_NODES)
        return fail(GDN_ERR_BAD_PARENTS, "node capacity N=%d outside [1, %d]", N, GDN_MAX_TREE_NODES);
    if (counts == nullptr || parents == nullptr || lengths == nullptr)
        return fail(GDN_ERR_INVALID_ARG, "counts / parents / lengths is NULL");
    static thread_local CommitBatchParams p;  // 2 KB of paths: kept off the stack
    p = CommitBatchParams{};
    int total = 0;
    for (int b = 0; b < shape->B; ++b) {
        if (counts[b] < 1 || counts[b] > N)
            return fail(GDN_ERR_BAD_PARENTS, "tree %d has %d nodes, need 1 .. %d", b, counts[b], N);
        const int32_t* par = parents + (size_t)b * N;
        if ((rc = check_parents(counts[b], par)) != GDN_OK) {
            const std::string why = t_error;
            return fail(rc, "tree %d: %s", b, why.c_str());
        }
        const int L = lengths[b];
        if (L > 0 && paths == nullptr) return fail(GDN_ERR_INVALID_ARG, "paths is NULL");
        if ((rc = check_path(counts[b], par, L > 0 ? paths + (size_t)b * N : nullptr, L)) != GDN_OK) {
            const std::string why = t_error;
            return fail(rc, "tree %d: %s", b, why.c_str());
        }
        p.L[b] = L;
        for (int i = 0; i < L; ++i) p.path[b][i] = (int8_t)paths[(size_t)b * N + i];
        total += L;
    }
    if (conv) {
        if ((rc = check_ptr(x_tree, "x")) || (rc = check_ptr(tail_in, "tail_in")) ||
            (rc = check_ptr(tail, "tail_out")))
            return rc;
        const size_t tail_bytes = (size_t)shape->B * GDN_CONV_W * packed_channels(shape) * sizeof(gdn_bf16);
        if (overlaps(tail_in, tail, tail_bytes))
            return fail(GDN_ERR_INVALID_ARG, "tail_in and tail_out overlap (they must be distinct buffers)");
    } else {
        if ((rc = check_ptr(qkv, "qkv")) || (rc = check_ptr(x_tree, "x_tree", false))) return rc;
        if (x_tree != nullptr && (rc = check_ptr(tail, "tail")) != GDN_OK) return rc;
    }
    if ((rc = check_ptr(alpha, "alpha")) || (rc = check_ptr(beta, "beta")) || (rc = check_ptr(state, "state")))
        return rc;
    if (total == 0 && !conv) return GDN_OK;  // no sequence accepted anything (the fused conv still moves the tails)
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    p.qkv = conv ? nullptr : qkv;
    p.alpha = alpha;
    p.beta = beta;
    p.state = state;
    p.x_tree = x_tree;
    p.tail = tail;
    p.w = w;
    p.tail_in = conv ? tail_in : nullptr;
    p.B = shape->B;
    p.N = N;
    p.Hk = shape->Hk;
    p.Hv = shape->Hv;
    p.dv = shape->dv;
    p.group = shape->Hv / shape->Hk;
    p.C = packed_channels(shape);
    p.normalize = (flags & GDN_NORMALIZE_QK) != 0;
    const int rows = decode_rows_per_cta(shape->B, shape->Hv, shape->dv);
    cudaError_t e = launch_commit_batched(p, shape->dk, rows, st);  // the tails too, when x_tree is given
    if (e != cudaSuccess) return cuda_fail(e, conv ? "conv + commit launch" : "batched commit launch");
    return GDN_OK;
}

}  // namespace

extern "C" {

int gdn_tree_verify(const gdn_shape* shape, int32_t N, const int32_t* parents, const gdn_bf16* qkv,
                    const float* alpha, const float* beta, const float* state, void* out,
                    float q_scale, uint32_t flags, void* stream) {
    return tree_verify_impl(shape, N, parents, qkv, nullptr, nullptr, nullptr, false, alpha, beta, state, out,
                            q_scale, flags, stream);
}

int gdn_kda_tree_verify(const gdn_shape* shape, int32_t N, const int32_t* parents, const gdn_bf16* qkv,
                        const float* alpha, const float* beta, const float* state, void* out, float q_scale,
                        uint32_t flags, void* stream) {
    return tree_verify_impl(shape, N, parents, qkv, nullptr, nullptr, nullptr, false, alpha, beta, state, out,
                            q_scale, flags, stream, true);
}

int gdn_conv_tree_verify(const gdn_shape* shape, int32_t N, const int32_t* parents, const gdn_bf16* x,
                         const gdn_bf16* w, const gdn_bf16* tail, const float* alpha, const float* beta,
                         const float* state, void* out, float q_scale, uint32_t flags, void* stream) {
    return tree_verify_impl(shape, N, parents, nullptr, x, w, tail, true, alpha, beta, state, out, q_scale, flags,
                            stream);
}

int gdn_tree_verify_batched(const gdn_shape* shape, int32_t N, const int32_t* counts, const int32_t* parents,
                            const gdn_bf16* qkv, const float* alpha, const float* beta, const float* state,
                            void* out, float q_scale, uint32_t flags, void* stream) {
    return tree_verify_batched_impl(shape, N, counts, parents, qkv, nullptr, nullptr, nullptr, false, alpha, beta,
                                    state, out, q_scale, flags, stream);
}

int gdn_kda_tree_verify_batched(const gdn_shape* shape, int32_t N, const int32_t* counts, const int32_t* parents,
                                const gdn_bf16* qkv, const float* alpha, const float* beta, const float* state,
                                void* out, float q_scale, uint32_t flags, void* stream) {
    return tree_verify_batched_impl(shape, N, counts, parents, qkv, nullptr, nullptr, nullptr, false, alpha, beta,
                                    state, out, q_scale, flags, stream, true);
}

int gdn_conv_tree_verify_batched(const gdn_shape* shape, int32_t N, const int32_t* counts, const int32_t* parents,
                                 const gdn_bf16* x, const gdn_bf16* w, const gdn_bf16* tail, const float* alpha,
                                 const float* beta, const float* state, void* out, float q_scale, uint32_t flags,
                                 void* stream) {
    return tree_verify_batched_impl(shape, N, counts, parents, nullptr, x, w, tail, true, alpha, beta, state, out,
                                    q_scale, flags, stream);
}

}  // extern "C"

// The single-sequence commit through the decode kernel's gather path (kda:
// a decay per key channel, alpha [N, Hv, dk]).
static int commit_path_impl(const gdn_shape* shape, int32_t N, const int32_t* parents, const int32_t* path,
                            int32_t L, const gdn_bf16* qkv, const float* alpha, const float* beta,
                            const gdn_bf16* x_tree, float* state, gdn_bf16* tail, uint32_t flags, void* stream,
                            bool kda) {
    int rc;
    if ((rc = check_shape(shape, true)) != GDN_OK) return rc;
    if (flags & GDN_OUT_BF16) return fail(GDN_ERR_INVALID_ARG, "commit writes no output; GDN_OUT_BF16 not allowed");
    if ((rc = check_flags(flags)) != GDN_OK) return rc;
    if ((rc = check_parents(N, parents)) != GDN_OK) return rc;
    if ((rc = check_path(N, parents, path, L)) != GDN_OK) return rc;
    if ((rc = check_ptr(qkv, "qkv")) || (rc = check_ptr(alpha, "alpha")) || (rc = check_ptr(beta, "beta")) ||
        (rc = check_ptr(state, "state")) || (rc = check_ptr(x_tree, "x_tree", false)))
        return rc;
    if (x_tree != nullptr && (rc = check_ptr(tail, "tail")) != GDN_OK) return rc;
    if (L == 0) return GDN_OK;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    DecodeParams p{};
    p.qkv = qkv;
    p.alpha = alpha;
    p.beta = beta;
    p.state = state;
    p.out = nullptr;
    p.B = 1;
    p.T = L;
    p.Tsrc = N;
    p.Hk = shape->Hk;
    p.Hv = shape->Hv;
    p.dv = shape->dv;
    p.group = shape->Hv / shape->Hk;
    p.C = packed_channels(shape);
    p.q_scale = 1.0f;
    p.normalize = (flags & GDN_NORMALIZE_QK) != 0;
    p.out_bf16 = 0;
    for (int i = 0; i < L; ++i) p.tok[i] = path[i];
    p.x_tree = x_tree;  // the conv tail is updated by the same launch
    p.tail = x_tree != nullptr ? tail : nullptr;
    const int rows = decode_rows_per_cta(1, shape->Hv, shape->dv);
    cudaError_t e = launch_decode(p, shape->dk, rows, 1, kda, false, st);
    if (e != cudaSuccess) return cuda_fail(e, kda ? "KDA commit launch" : "commit launch");
    return GDN_OK;
}

extern "C" {

int gdn_commit_path(const gdn_shape* shape, int32_t N, const int32_t* parents, const int32_t* path, int32_t L,
                    const gdn_bf16* qkv, const float* alpha, const float* beta, const gdn_bf16* x_tree, float* state,
                    gdn_bf16* tail, uint32_t flags, void* stream) {
    return commit_path_impl(shape, N, parents, path, L, qkv, alpha, beta, x_tree, state, tail, flags, stream, false);
}

int gdn_kda_commit_path(const gdn_shape* shape, int32_t N, const int32_t* parents, const int32_t* path, int32_t L,
                        const gdn_bf16* qkv, const float* alpha, const float* beta, const gdn_bf16* x_tree,
                        float* state, gdn_bf16* tail, uint32_t flags, void* stream) {
    return commit_path_impl(shape, N, parents, path, L, qkv, alpha, beta, x_tree, state, tail, flags, stream, true);
}


int gdn_commit_path_batched(const gdn_shape* shape, int32_t N, const int32_t* counts, const int32_t* parents,
                            const int32_t* paths, const int32_t* lengths, const gdn_bf16* qkv, const float* alpha,
                            const float* beta, const gdn_bf16* x_tree, float* state, gdn_bf16* tail, uint32_t flags,
                            void* stream) {
    return commit_batched_impl(shape, N, counts, parents, paths, lengths, qkv, alpha, beta, x_tree, state, tail,
                               nullptr, nullptr, flags, stream);
}

int gdn_conv_commit_path(const gdn_shape* shape, int32_t N, const int32_t* parents, const int32_t* path, int32_t L,
                         const gdn_bf16* x, const gdn_bf16* w, const gdn_bf16* tail_in, gdn_bf16* tail_out,
                         const float* alpha, const float* beta, float* state, uint32_t flags, void* stream) {
    int rc;
    if ((rc = check_shape(shape, true)) != GDN_OK) return rc;
    if ((rc = check_ptr(w, "w")) != GDN_OK) return rc;
    if (N < 1 || N > GDN_MAX_TREE_NODES)
        return fail(GDN_ERR_BAD_PARENTS, "tree size N=%d outside [1, %d]", N, GDN_MAX_TREE_NODES);
    const int32_t counts[1] = {N}, lengths[1] = {L};
    return commit_batched_impl(shape, N, counts, parents, path, lengths, nullptr, alpha, beta, x, state, tail_out,
                               w, tail_in, flags, stream);
}

int gdn_conv_commit_path_batched(const gdn_shape* shape, int32_t N, const int32_t* counts, const int32_t* parents,
                                 const int32_t* paths, const int32_t* lengths, const gdn_bf16* x, const gdn_bf16* w,
                                 const gdn_bf16* tail_in, gdn_bf16* tail_out, const float* alpha, const float* beta,
                                 float* state, uint32_t flags, void* stream) {
    int rc;
    if ((rc = check_ptr(w, "w")) != GDN_OK) return rc;
    return commit_batched_impl(shape, N, counts, parents, paths, lengths, nullptr, alpha, beta, x, state, tail_out,
                               w, tail_in, flags, stream);
}

}  // extern "C"
