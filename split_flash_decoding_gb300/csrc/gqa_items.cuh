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

// Balanced split: this CTA's tile range [x0, x1), the first of its units
// and their count, and the totals the slot table needs; found by the warp
// that builds the item table (gqa_build_items) and read by every role.
struct GqaRange {
    int x0, x1, u0, count, tiles, wtiles, ctas;
};

// Balanced split: this CTA's walk from its range.
__device__ __forceinline__ GqaWalk gqa_balanced_walk(const GqaRange &rg) {
    GqaWalk w;
    w.first = 0;
    w.stride = 1;
    w.count = rg.count;
    w.x0 = rg.x0;
    w.x1 = rg.x1;
    w.u0 = rg.u0;
    w.tiles = rg.tiles;
    w.wtiles = rg.wtiles;
    w.ctas = rg.ctas;
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

// Build cum[0..batch] with one warp (all 32 lanes must call): lane l sums
// the tiles of sequences [l m, (l+1) m), a warp scan gives the chunk starts.
// Under the balanced split the same warp also finds this CTA's range (into
// *rg): in the weighted concatenation unit u (n_u tiles from tile x_u)
// occupies positions [x_u + kGqaUnitCost u, x_u + kGqaUnitCost (u + 1) +
// n_u), its virtual tiles first; CTA c of C' = min(grid, tiles) takes the
// positions [c T_w / C', (c + 1) T_w / C'), i.e. the real tiles from the image
// of its first position (a position in a virtual block maps to the unit's
// first tile) up to the next CTA's; CTAs past C' take none, and a range
// inside one virtual block is empty.  The lane whose chunk holds a range end
// finds its sequence, unit and tile.
__device__ __forceinline__ void gqa_build_items(const GqaParams &p, int hkv, int *cum, int lane,
                                                GqaRange *rg) {
    const uint32_t cap = uint32_t(p.num_partitions) * uint32_t(p.chunk);
    const int per_lane = (p.batch + 31) / 32;
    const int b0 = min(lane * per_lane, p.batch), b1 = min(b0 + per_lane, p.batch);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
        const uint32_t len_in = p.kv_len[b];
        if (len_in > cap && blockIdx.x == 0) atomicOr(p.err, kErrBadLength);
        const uint32_t L = min(len_in, cap);
        const int ns = static_cast<int>((L + p.chunk - 1) / p.chunk);
        local += max(ns, 1) * hkv;
    }
    int incl = local;  // inclusive warp scan of the per-lane sums
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int b = b0; b < b1; ++b) {
        cum[b] = run;
        const uint32_t L = min(p.kv_len[b], cap);
        const int ns = static_cast<int>((L + p.chunk - 1) / p.chunk);
        run += max(ns, 1) * hkv;
    }
    if (lane == 31) cum[p.batch] = incl;
    if (!p.balanced) return;

    const long long per_seq = static_cast<long long>(kGqaUnitCost) * hkv;
    const long long T = __shfl_sync(0xffffffffu, incl, 31);
    const long long Tw = T + per_seq * p.batch;
    const long long C = min(static_cast<long long>(gridDim.x), T);
    const long long c = blockIdx.x;
    const long long w_lo = (incl - local) + per_seq * b0, w_hi = incl + per_seq * b1;
    // Real tile of weighted position y: {x, unit, x is the unit's first tile}.
    auto locate = [&](long long y, int &unit, bool &at_first) -> long long {
        const bool mine = w_lo <= y && y < w_hi;
        const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
        long long x = 0;
        int u = 0, f = 0;
        if (lane == src) {
            long long xs = incl - local, ws = w_lo;   // the chunk's first tile / position
            for (int b = b0; b < b1; ++b) {
                const uint32_t L = min(p.kv_len[b], cap);
                const long long n = max(static_cast<int>((L + p.chunk - 1) / p.chunk), 1);
                const long long span = hkv * (n + kGqaUnitCost);
                if (y < ws + span) {
                    const long long off = y - ws;
                    const long long h = off / (n + kGqaUnitCost);
                    const long long o = off - h * (n + kGqaUnitCost) - kGqaUnitCost;
                    x = xs + h * n + min(max(o, 0LL), n);
                    u = b * hkv + static_cast<int>(h);
                    f = o <= 0;
                    break;
                }
                xs += hkv * n;
                ws += span;
            }
        }
        unit = __shfl_sync(0xffffffffu, u, src);
        at_first = __shfl_sync(0xffffffffu, f, src) != 0;
        return __shfl_sync(0xffffffffu, x, src);
    };
    GqaRange r;
    r.x0 = r.x1 = r.u0 = r.count = 0;
    r.tiles = static_cast<int>(T);
    r.wtiles = static_cast<int>(Tw);
    r.ctas = static_cast<int>(C);
    if (c < C) {
        int u0, u1;
        bool f0, f1;
        r.x0 = static_cast<int>(locate(c * Tw / C, u0, f0));
        int u_last;
        if (c + 1 == C) {
            r.x1 = static_cast<int>(T);
            u_last = p.batch * hkv - 1;
        } else {
            r.x1 = static_cast<int>(locate((c + 1) * Tw / C, u1, f1));
            u_last = f1 ? u1 - 1 : u1;   // x1 - 1 lies in the unit before when x1 opens one
        }
        r.u0 = u0;
        r.count = r.x1 > r.x0 ? u_last - u0 + 1 : 0;
    }
    if (lane == 0) *rg = r;
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
