// pkv_plan.cpp -- host-side work plan for the paged prefill attention.
//
// The prefill kernel's work comes in units (sequence s, pair of 128-row
// query tiles qt, KV head h); a unit's work is its causal key range, which
// grows with the sequence's context (tokens already in the pool) and with
// qt.  A batch of chunks over contexts of different lengths ([P1] on chunked
// prefill: a long prompt is cut into chunks that each attend to the KV of
// the earlier ones) gives units of very different lengths, and the kernel's
// persistent CTAs take units in list order as they become free.  The plan
// lists the units (s, qt) longest key range first, so that the last units
// to start are the shortest ones (longest-processing-time first list
// scheduling).  The host knows the batch (it scheduled it), so the plan is
// built here, in plain C++, and passed to the kernel as a short device
// array.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "../../include/pagedkv.h"

namespace {
constexpr int kTileRows = 128;  // query rows per tensor-core tile
}

extern "C" pkv_status pkv_prefill_plan(const int32_t* query_start, const int32_t* seq_lens, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t num_kv_heads, int32_t max_query_len,
                                       int32_t* units, int32_t units_cap, int32_t* num_units) {
    if (!num_units) return PKV_ERR_INVALID;
    *num_units = 0;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_query_len < 0 || units_cap < 0)
        return PKV_ERR_INVALID;
    if (num_q_heads % num_kv_heads) return PKV_ERR_INVALID;
    const int G = num_q_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 || max_query_len == 0) return PKV_OK;
    if (!query_start || !seq_lens) return PKV_ERR_INVALID;
    const int64_t rows = 2 * (kTileRows / G);  // query tokens per CTA
    const int64_t nq = (max_query_len + rows - 1) / rows;
    if (nq * num_seqs > INT32_MAX) return PKV_ERR_UNSUPPORTED;

    struct Unit {
        int64_t keys;  // causal key range of the CTA's last row
        int32_t id;    // s * nq + qt
    };
    std::vector<Unit> list;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int64_t q0 = query_start[s], q1 = query_start[s + 1];
        const int64_t n = q1 - q0, L = seq_lens[s];
        if (q0 < 0 || n < 0 || n > max_query_len || L < n) return PKV_ERR_INVALID;
        const int64_t ctx = L - n;
        for (int64_t qt = 0; qt * rows < n; ++qt)
            list.push_back({ctx + std::min(n, (qt + 1) * rows), static_cast<int32_t>(s * nq + qt)});
    }
    // longest first; equal lengths keep (sequence, query tile) order
    std::stable_sort(list.begin(), list.end(), [](const Unit& a, const Unit& b) { return a.keys > b.keys; });
    *num_units = static_cast<int32_t>(list.size());
    if (static_cast<int64_t>(list.size()) > units_cap) return PKV_ERR_WORKSPACE;
    if (!list.empty() && !units) return PKV_ERR_INVALID;
    for (size_t i = 0; i < list.size(); ++i) units[i] = list[i].id;
    return PKV_OK;
}
