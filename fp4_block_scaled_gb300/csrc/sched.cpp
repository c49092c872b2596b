// sched.cpp -- expert-sharing batch planner (host code, no GPU).
//
// Sequences whose prompts are alike route their tokens to alike experts, so a
// batch of alike sequences touches fewer distinct experts per layer, and the
// weights a decode step streams fall with them ("把不支持 FP4 的 A100 拉到 673
// tok/s", §批处理不是「同时处理几个人」: 216 -> 156 distinct experts in one
// layer).  The planner cuts N sequences into batches of B so that each batch
// adds as few experts as it can: every sequence carries a signature (its
// recent top-k expert ids per layer); a batch starts from the lowest-numbered
// sequence not yet placed and grows by the sequence that adds the fewest
// experts not yet in the batch, summed over the layers (ties to the lower
// number), until it holds B.  Per-layer expert sets are bitsets of E bits, so
// choosing one sequence costs O(N L topk) and the plan O(N^2 L topk).
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "../../include/moe_ffn.h"

namespace {

struct Bits {
    int words;
    std::vector<uint64_t> w;
    Bits(int nsets, int nbits) : words((nbits + 63) / 64), w((size_t)nsets * words, 0) {}
    uint64_t* set(int i) { return w.data() + (size_t)i * words; }
};

inline bool test_bit(const uint64_t* s, int e) { return (s[e >> 6] >> (e & 63)) & 1u; }
inline void set_bit(uint64_t* s, int e) { s[e >> 6] |= 1ull << (e & 63); }

bool valid_args(const int32_t* sig, int N, int L, int topk, int E, int B)
{
    if (N < 0 || L <= 0 || topk <= 0 || E <= 0 || E > (1 << 20) || B <= 0) return false;
    if (N > 0 && !sig) return false;
    const size_t n = (size_t)N * L * topk;
    for (size_t i = 0; i < n; i++)
        if (sig[i] < -1 || sig[i] >= E) return false;
    return true;
}

}  // namespace

extern "C" int moe_batch_plan(const int32_t* sig, int N, int L, int topk, int E, int B, int32_t* order)
{
    if (!valid_args(sig, N, L, topk, E, B) || (N > 0 && !order)) return MOE_ERR_INVALID_ARG;
    if (N == 0) return MOE_OK;
    std::vector<char> placed((size_t)N, 0);
    Bits cur(L, E);                                  // the batch's experts, per layer
    int out = 0, next_seed = 0;
    while (out < N) {
        while (placed[next_seed]) next_seed++;
        std::fill(cur.w.begin(), cur.w.end(), 0);
        int in_batch = 0;
        int pick = next_seed;
        for (;;) {
            placed[pick] = 1;
            order[out++] = pick;
            in_batch++;
            for (int l = 0; l < L; l++) {
                const int32_t* ids = sig + ((size_t)pick * L + l) * topk;
                for (int k = 0; k < topk; k++)
                    if (ids[k] >= 0) set_bit(cur.set(l), ids[k]);
            }
            if (in_batch == B || out == N) break;
            // the unplaced sequence adding the fewest new experts (lowest number on ties)
            long best_cost = -1;
            pick = -1;
            for (int i = 0; i < N; i++) {
                if (placed[i]) continue;
                long cost = 0;
                for (int l = 0; l < L && (best_cost < 0 || cost < best_cost); l++) {
                    const int32_t* ids = sig + ((size_t)i * L + l) * topk;
                    const uint64_t* s = cur.set(l);
                    for (int k = 0; k < topk; k++) {
                        const int e = ids[k];
                        if (e < 0 || test_bit(s, e)) continue;
                        bool dup = false;                     // an id repeated within the row counts once
                        for (int k2 = 0; k2 < k; k2++) dup |= ids[k2] == e;
                        cost += dup ? 0 : 1;
                    }
                }
                if (best_cost < 0 || cost < best_cost) {
                    best_cost = cost;
                    pick = i;
                }
            }
        }
    }
    return MOE_OK;
}

extern "C" int moe_batch_distinct(const int32_t* routing, const int32_t* order, int N, int L, int topk, int E,
                                  int B, int32_t* distinct)
{
    if (!valid_args(routing, N, L, topk, E, B) || (N > 0 && (!order || !distinct))) return MOE_ERR_INVALID_ARG;
    std::vector<char> seen((size_t)N, 0);
    for (int i = 0; i < N; i++) {
        if (order[i] < 0 || order[i] >= N || seen[order[i]]) return MOE_ERR_INVALID_ARG;   // not a permutation
        seen[order[i]] = 1;
    }
    Bits cur(1, E);
    const int nb = (N + B - 1) / B;
    for (int b = 0; b < nb; b++) {
        const int i1 = (b + 1) * B < N ? (b + 1) * B : N;
        for (int l = 0; l < L; l++) {
            std::fill(cur.w.begin(), cur.w.end(), 0);
            int count = 0;
            for (int i = b * B; i < i1; i++) {
                const int32_t* ids = routing + ((size_t)order[i] * L + l) * topk;
                for (int k = 0; k < topk; k++) {
                    const int e = ids[k];
                    if (e < 0 || test_bit(cur.set(0), e)) continue;
                    set_bit(cur.set(0), e);
                    count++;
                }
            }
            distinct[(size_t)b * L + l] = count;
        }
    }
    return MOE_OK;
}
