// shared_prefix.cpp -- host planning of the shared-prefix decode: which
// sequences share their leading partitions' KV blocks ("TGI PagedAttention
// deep-dive" (lpnh.cn) sec. 5: requests with a common prompt prefix reuse its
// cached blocks; "Lecture 3: PagedAttention and vLLM", "shared prefix": several
// sequences' block tables point at the same physical blocks).
//
// Two sequences share partition j (tokens [jP, (j+1)P)) when their block
// tables name the same blocks over it. A sequence can share only partitions
// that lie wholly before its newest token: at most floor((L - 1) / P) of them.
// Sequences are sorted by their tables (lexicographically), so that those with
// long common prefixes are neighbours; units of up to PA_SHARED_UNIT_MEMBERS
// neighbours are formed greedily, choosing the size that saves the most
// partition reads: (members - 1) x (partitions common to all of them).
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "pagedkv.h"

namespace {

struct Plan {
    const int32_t* tables;
    int max_blocks;
    int bpp;                     // blocks per partition
    std::vector<int> shareable;  // whole partitions before each sequence's newest token

    const int32_t* row(int s) const { return tables + (size_t)s * max_blocks; }

    // leading partitions whose blocks agree, up to both sequences' limits
    int common(int a, int b) const {
        const int n = std::min(shareable[a], shareable[b]);
        const int32_t* ra = row(a);
        const int32_t* rb = row(b);
        for (int j = 0; j < n; ++j)
            for (int i = j * bpp; i < (j + 1) * bpp; ++i)
                if (ra[i] != rb[i]) return j;
        return n;
    }

    // table order over the shareable blocks; shorter first on a tie, then index
    bool before(int a, int b) const {
        const int n = std::min(shareable[a], shareable[b]) * bpp;
        const int32_t* ra = row(a);
        const int32_t* rb = row(b);
        for (int i = 0; i < n; ++i)
            if (ra[i] != rb[i]) return ra[i] < rb[i];
        if (shareable[a] != shareable[b]) return shareable[a] < shareable[b];
        return a < b;
    }
};

}  // namespace

extern "C" pa_status pa_shared_prefix_plan(const int32_t* block_tables, const int32_t* context_lens,
                                           int num_seqs, int max_blocks_per_seq, int block_size,
                                           int partition_size, int32_t* seq_shared_parts,
                                           int32_t* unit_seqs, int32_t* unit_parts, int max_units,
                                           int* num_units, int* max_unit_parts) {
    if (num_seqs < 0 || max_blocks_per_seq < 0 || block_size <= 0 || partition_size <= 0 ||
        max_units < 0 || !num_units || !max_unit_parts)
        return PA_ERR_INVALID_ARG;
    if (partition_size % 32 != 0 || partition_size % block_size != 0) return PA_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!block_tables || !context_lens || !seq_shared_parts))
        return PA_ERR_INVALID_ARG;
    if (max_units > 0 && (!unit_seqs || !unit_parts)) return PA_ERR_INVALID_ARG;
    *num_units = 0;
    *max_unit_parts = 0;
    Plan pl{block_tables, max_blocks_per_seq, partition_size / block_size, {}};
    pl.shareable.assign(num_seqs, 0);
    std::vector<int> cand;
    for (int s = 0; s < num_seqs; ++s) {
        seq_shared_parts[s] = 0;
        const int L = context_lens[s];
        if (L <= 0) continue;
        const int by_len = (L - 1) / partition_size;
        const int by_table = max_blocks_per_seq / pl.bpp;
        pl.shareable[s] = std::min(by_len, by_table);
        if (pl.shareable[s] > 0) cand.push_back(s);
    }
    std::sort(cand.begin(), cand.end(), [&](int a, int b) { return pl.before(a, b); });
    const int M = PA_SHARED_UNIT_MEMBERS;
    size_t i = 0;
    while (i < cand.size() && *num_units < max_units) {
        // common partitions with the first member fall along the sorted order
        int best_k = 1, best_parts = 0;
        long long best_saved = 0;
        int parts = 1 << 30;
        for (int k = 2; k <= M && i + k - 1 < cand.size(); ++k) {
            parts = std::min(parts, pl.common(cand[i], cand[i + k - 1]));
            if (parts <= 0) break;
            const long long saved = (long long)(k - 1) * parts;
            if (saved > best_saved) {
                best_saved = saved;
                best_k = k;
                best_parts = parts;
            }
        }
        if (best_k < 2) {
            ++i;
            continue;
        }
        const int u = (*num_units)++;
        for (int m = 0; m < M; ++m) {
            const int s = m < best_k ? cand[i + m] : -1;
            unit_seqs[(size_t)u * M + m] = s;
            if (s >= 0) seq_shared_parts[s] = best_parts;
        }
        unit_parts[u] = best_parts;
        *max_unit_parts = std::max(*max_unit_parts, best_parts);
        i += best_k;
    }
    return PA_OK;
}
