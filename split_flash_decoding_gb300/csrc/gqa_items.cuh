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
    // balanced split: the unit (sequence, KV head), whether this piece holds
    // its first tile, and the global tile index of that first tile and its
    // tile count
    int unit, unit_x, unit_tiles;
    bool first;
};

// This CTA's items: j = first, first + stride, ... < count.  The balanced
// split also keeps the CTA's tile range [x0, x1) of the concatenation of
// every unit's tiles (tiles in all; wtiles weighted positions dealt over
// ctas CTAs) and the unit of its first tile.
struct GqaWalk {
    int first, stride, count;
    long long x0, x1, tiles, wtiles, ctas;
    int u0;
};

// Balanced split: a CTA's time is its tiles plus a fixed cost for every unit
// it opens (the unit's Q, the pipeline refill, the epilogue and partial),
// about this many tiles' worth.  The split deals out a weighted
// concatenation in which every unit is preceded by that many virtual tiles,
// so a CTA whose range meets more units gets fewer tiles.
constexpr int kGqaUnitCost = 2;

// Unit (sequence b, KV head) holding global tile x: cum[b] <= x < cum[b+1].
__device__ __forceinline__ int gqa_unit_of(const int *cum, int batch, int hkv, long long x) {
    int lo = 0, hi = batch;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cum[mid] <= x) lo = mid; else hi = mid;
    }
    const int per_head = (cum[lo + 1] - cum[lo]) / hkv;
    return lo * hkv + static_cast<int>((x - cum[lo]) / per_head);
}

// Weighted concatenation of the balanced split: unit u (n_u tiles, starting
// at tile x_u) occupies positions [x_u + kGqaUnitCost u, x_u + kGqaUnitCost
// (u + 1) + n_u), its virtual tiles first, so real tile x of unit u sits at
// x + kGqaUnitCost (u + 1).  The real tile a position y < T_w maps to (a
// position in a virtual block: the unit's first tile).
__device__ __forceinline__ long long gqa_tile_of_position(const int *cum, int batch, int hkv,
                                                          long long y) {
    const long long per_seq = static_cast<long long>(kGqaUnitCost) * hkv;
    int lo = 0, hi = batch;   // sequence b: cum[b] + per_seq b <= y
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cum[mid] + per_seq * mid <= y) lo = mid; else hi = mid;
    }
    const long long n = (cum[lo + 1] - cum[lo]) / hkv;   // tiles per unit of sequence lo
    const long long off = y - (cum[lo] + per_seq * lo);
    const long long h = off / (n + kGqaUnitCost);
    const long long o = off - h * (n + kGqaUnitCost) - kGqaUnitCost;
    return cum[lo] + h * n + min(max(o, 0LL), n);
}

// Balanced split: this CTA's tile range and units.  CTA c of C' = min(grid,
// tiles) takes the weighted positions [c T_w / C', (c + 1) T_w / C'), i.e.
// the real tiles from the image of its first position up to the next
// CTA's; CTAs past C' take none, and a range inside one virtual block is
// empty.
__device__ __forceinline__ GqaWalk gqa_balanced_walk(const GqaParams &p, const int *cum, int hkv) {
    GqaWalk w;
    w.first = 0;
    w.stride = 1;
    w.tiles = cum[p.batch];
    w.wtiles = w.tiles + static_cast<long long>(kGqaUnitCost) * hkv * p.batch;
    w.ctas = min(static_cast<long long>(gridDim.x), w.tiles);
    const long long c = blockIdx.x;
    w.count = 0;
    w.u0 = 0;
    w.x0 = w.x1 = 0;
    if (c < w.ctas) {
        w.x0 = gqa_tile_of_position(cum, p.batch, hkv, c * w.wtiles / w.ctas);
        w.x1 = c + 1 == w.ctas
                   ? w.tiles
                   : gqa_tile_of_position(cum, p.batch, hkv, (c + 1) * w.wtiles / w.ctas);
        if (w.x1 > w.x0) {
            w.u0 = gqa_unit_of(cum, p.batch, hkv, w.x0);
            w.count = gqa_unit_of(cum, p.batch, hkv, w.x1 - 1) - w.u0 + 1;
        }
    }
    return w;
}

// Item j of a balanced walk: the piece of unit u0 + j inside [x0, x1).
__device__ __forceinline__ GqaItem gqa_balanced_item(const GqaParams &p, const int *cum, int hkv,
                                                     const GqaWalk &w, int j) {
    GqaItem it;
    it.unit = w.u0 + j;
    it.b = it.unit / hkv;
    it.kvh = it.unit - it.b * hkv;
    it.unit_tiles = (cum[it.b + 1] - cum[it.b]) / hkv;
    it.unit_x = cum[it.b] + it.kvh * it.unit_tiles;
    const long long tb = max(w.x0 - it.unit_x, 0LL);
    const long long te = min(w.x1 - it.unit_x, static_cast<long long>(it.unit_tiles));
    const uint32_t cap = uint32_t(p.num_partitions) * uint32_t(p.chunk);
    it.L = static_cast<int>(min(p.kv_len[it.b], cap));
    it.start = static_cast<int>(tb) * kGqaTcTileKeys;
    it.end = min(static_cast<int>(te) * kGqaTcTileKeys, it.L);
    it.ntiles = it.start < it.end ? (it.end - it.start + kGqaTcTileKeys - 1) / kGqaTcTileKeys : 0;
    it.first = tb == 0;
    it.direct = tb == 0 && te == it.unit_tiles;
    it.part = static_cast<int>(blockIdx.x) + it.unit;   // partial slot
    return it;
}

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
    it.unit = lo * hkv + it.kvh;
    it.unit_x = 0;
    it.unit_tiles = 0;
    it.first = false;
    return it;
}

}  // namespace attn
