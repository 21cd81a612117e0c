// gqa_items.cuh -- the persistent work list of the GQA decode kernels.
//
// Work item = (sequence b, KV head, key slice p).  Sequence b has
// n_b = max(1, ceil(min(kv_len[b], P * chunk) / chunk)) slices per KV head
// (an empty sequence still has one item, which writes its empty result).
// cum[b] = num_kv_heads * sum_{b' < b} n_b' is built once per CTA in shared
// memory by one warp; item j is then found by binary search.  Items are
// handed to CTAs round-robin (item j -> CTA j mod gridDim.x).
#pragma once

#include "launch.h"
#include "ptx.cuh"

namespace attn {

struct GqaItem {
    int b, kvh, part, L, start, end, ntiles;
    bool direct;  // the sequence needs at most one slice: write the final rows
};

// Build cum[0..batch] with warp `warp_id` (all 32 lanes must call).
__device__ __forceinline__ void gqa_build_items(const GqaParams &p, int hkv, int *cum, int lane) {
    const uint32_t cap = uint32_t(p.num_partitions) * uint32_t(p.chunk);
    const int per_lane = (p.batch + 31) / 32;
    const int b0 = lane * per_lane;
    int local = 0;
    for (int i = 0; i < per_lane; ++i) {
        const int b = b0 + i;
        if (b < p.batch) {
            const uint32_t len_in = p.kv_len[b];
            if (len_in > cap && blockIdx.x == 0) atomicOr(p.err, kErrBadLength);
            const uint32_t L = min(len_in, cap);
            const int ns = static_cast<int>((L + p.chunk - 1) / p.chunk);
            local += max(ns, 1) * hkv;
        }
    }
    int incl = local;  // inclusive warp scan of the per-lane sums
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int i = 0; i < per_lane; ++i) {
        const int b = b0 + i;
        if (b < p.batch) {
            cum[b] = run;
            const uint32_t L = min(p.kv_len[b], cap);
            const int ns = static_cast<int>((L + p.chunk - 1) / p.chunk);
            run += max(ns, 1) * hkv;
        }
    }
    if (lane == 31) cum[p.batch] = incl;
}

template <int kTileKeys>
__device__ __forceinline__ GqaItem gqa_item(const GqaParams &p, const int *cum, int j, int hkv) {
    int lo = 0, hi = p.batch;  // find b: cum[b] <= j < cum[b+1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cum[mid] <= j) lo = mid; else hi = mid;
    }
    GqaItem it;
    it.b = lo;
    const int per_head = (cum[lo + 1] - cum[lo]) / hkv;  // n_b
    const int r = j - cum[lo];
    it.kvh = r / per_head;
    it.part = r - it.kvh * per_head;
    const uint32_t cap = uint32_t(p.num_partitions) * uint32_t(p.chunk);
    it.L = static_cast<int>(min(p.kv_len[lo], cap));
    it.start = it.part * p.chunk;
    it.end = min(it.start + p.chunk, it.L);
    it.ntiles = it.start < it.end ? (it.end - it.start + kTileKeys - 1) / kTileKeys : 0;
    it.direct = per_head <= 1;
    return it;
}

}  // namespace attn
