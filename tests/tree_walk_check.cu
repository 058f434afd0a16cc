// Host-only check of the tree verify's walk schedules (built and run by
// test_tree_walk_host.py; no GPU).  It includes the host API's translation
// unit to reach its internal schedule builders, replays every schedule the
// way the kernel walks it, and checks, for random trees of every size:
//   - each step's parent state is where the step takes it from (the previous
//     step's registers, or a slot holding exactly the parent's state);
//   - slots stay within the count the launch sizes for;
//   - every node's output is stored exactly once over all walkers;
//   - a split shortens the longest walk to at most 3/4 of the tree.
#include "../hybrid_linear_attention_conv_gb300/csrc/gdn_api.cu"

#include <cstdio>
#include <map>
#include <random>

namespace {

// Replays one walk; returns 0 or an error code.
int replay(const int32_t* parents, const TreeStep* steps, int n_steps, int slot_lo, int slot_hi,
           std::vector<int>& stored) {
    int regs = -2;  // -2: the committed state
    std::map<int, int> slot;
    for (int k = 0; k < n_steps; ++k) {
        const int v = steps[k].node;
        const int want = parents[v] < 0 ? -2 : parents[v];
        if (steps[k].restore >= 0) {
            if (steps[k].restore < slot_lo || steps[k].restore >= slot_hi) return 1;
            if (!slot.count(steps[k].restore) || slot[steps[k].restore] != want) return 2;
        } else if (regs != want) {
            return 3;
        }
        regs = v;
        if (steps[k].save >= 0) {
            if (steps[k].save < slot_lo || steps[k].save >= slot_hi) return 4;
            slot[steps[k].save] = v;
        }
        if (steps[k].store) stored[v] += 1;
    }
    return 0;
}

}  // namespace

int main() {
    std::mt19937 rng(2024);
    long trees = 0, splits = 0;
    for (int it = 0; it < 6000; ++it) {
        const int N = 1 + (int)(rng() % GDN_MAX_TREE_NODES);
        std::vector<int32_t> parents(N);
        parents[0] = -1;
        for (int i = 1; i < N; ++i) {
            switch (it % 3) {
                case 0: parents[i] = (int32_t)(rng() % i); break;                           // any earlier node
                case 1: parents[i] = std::max(0, i - 1 - (int)(rng() % 3)); break;          // long and thin
                default: parents[i] = (int32_t)((i - 1) / (1 + (int)(rng() % 4))); break;  // bushy
            }
        }
        TreeParams p{};
        if (schedule_tree(N, parents.data(), p.steps[0], &p.n_slots) != GDN_OK) continue;  // too many nested branches
        ++trees;
        std::vector<int> stored(N, 0);
        int rc = replay(parents.data(), p.steps[0], N, 0, p.n_slots, stored);
        for (int v = 0; v < N && rc == 0; ++v)
            if (stored[v] != 1) rc = 5;
        if (rc) {
            printf("FAIL single walk: tree %d (N=%d) code %d\n", it, N, rc);
            return 1;
        }
        for (int P = 2; P <= kMaxWalkers; ++P) {
            TreeParams q{};
            split_walkers(N, parents.data(), P, q);
            if (q.walkers == 1) continue;
            ++splits;
            std::vector<int> st(N, 0);
            int longest = 0;
            for (int w = 0; w < q.walkers && rc == 0; ++w) {
                rc = replay(parents.data(), q.walk[w], q.walk_n[w], 0, q.walk_slots, st);
                longest = std::max(longest, q.walk_n[w]);
                if (q.walk_n[w] > N) rc = 6;
            }
            for (int v = 0; v < N && rc == 0; ++v)
                if (st[v] != 1) rc = 7;
            if (rc == 0 && (q.walkers > P || 4 * longest > 3 * N)) rc = 8;
            if (rc) {
                printf("FAIL %d walkers: tree %d (N=%d) code %d\n", P, it, N, rc);
                return 1;
            }
        }
    }
    printf("tree walk schedules OK: %ld trees, %ld splits\n", trees, splits);
    return 0;
}
