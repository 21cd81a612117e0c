// gqa_decode_tc.cu -- split-K flash-decoding for grouped-query attention with
// head_dim 128 on the 5th-generation tensor cores.
//
// Same work list as the CUDA-core kernel (gqa_items.cuh: one item = one
// (sequence, KV head, key slice), persistent grid, one CTA per SM), but the
// two contractions of a 128-key tile run as tcgen05 MMAs with the keys / the
// channels on the 128-row M dimension and the folded query heads of the group
// on N (padded to 16):
//
//   S^T [128 keys x 16]  = K_tile [128 keys x 128 ch] . Q^T    (K-major A, B)
//   O^T [128 ch x 16]   += V_tile^T [128 ch x 128 keys] . P^T  (MN-major A)
//
// so the per-key work left to the SIMT threads is the softmax only (thread =
// key of the tile = TMEM lane), and the kernel stays bound by HBM.  The group
// makes Q.K' and P.V dense contractions of depth 128 over 128 keys; only the
// N side is padded.
//
// Few-token decode (n <= 16 / group query rows per sequence, e.g. draft
// tokens) folds the rows onto N as well: column c = (row i = c / group, head
// h = c % group), one TMA box of (64 channels x group heads x n rows) per Q
// half, and a per-column causal limit (row i of n sees keys j <= L - n + i).
// An item still covers all keys of a slice once for all the rows.
//
// Warp roles (224 threads): warps 0-3 softmax and epilogue, warp 4 streams
// K tiles and the item's Q (TMA), warp 5 streams V tiles (TMA), warp 6 owns
// TMEM and issues the MMAs.  Rings: 3 K stages and 3 V stages of 32 KB, each
// consumed in order by the single MMA thread, so parity waits never alias.
//
// Balanced split (up to 8 units per SM): the 128-key tiles of every (sequence, KV
// head) unit, concatenated, are dealt out in contiguous ranges of equal cost
// (tiles plus a fixed cost per unit opened), one per CTA, so ragged lengths
// cannot leave SMs idle; a CTA walks the pieces of the
// units its range meets, writes the units it holds whole and leaves a
// 16-column partial in slot (CTA + unit) for each piece of a cut unit; the
// CTA holding a unit's first tile publishes the unit's slot range for the
// split-K reduce.
//
// Small P, merged on chip: with 2 or 4 partitions the kernel can run as
// clusters of that many CTAs instead.  A cluster takes one (sequence, KV
// head) unit at a time and CTA r of the cluster covers the r-th of equal key
// slices of it; at the end of the unit every CTA leaves its partial (O^T, m,
// l per column) in its own shared memory, signals every CTA of the cluster
// through a cluster-scope mbarrier arrive, and then merges its share of the
// output channels by reading the partials of all CTAs over distributed
// shared memory -- no workspace and no reduce launch.  The merge buffers are
// double-buffered by unit parity: a CTA writes a buffer again only after the
// next unit's signal from every peer, which follows the peers' reads.
//
// Per tile: the MMA thread issues S(t) into one of two TMEM score buffers as
// soon as K(t) has landed; the softmax warps take the tile max per head
// across the four warps (shared memory), update the running max m and sums
// l, rescale O^T in TMEM when m moved, and write P^T (bf16) to shared memory;
// the MMA thread then accumulates O^T += V(t)^T P(t)^T.  Scores are scaled
// in fp32 after the MMA (q enters the MMA unscaled and exact).  Two sums are
// kept: of the fp32 weights (lse) and of the bf16 weights the MMA used
// (normalisation of O).  Keys past the sequence end are masked in S and
// zeroed in the V stage before the P.V MMA reads it.
#include "gqa_items.cuh"
#include "launch.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace attn {
namespace {

constexpr int kD = 128;
constexpr int kBK = kGqaTcTileKeys;          // 128 keys per tile
constexpr int kStages = 3;
constexpr int kBox = 128 * 128;              // 128 rows x 128 B
constexpr int kTileBytes = 2 * kBox;         // 128 keys x 128 channels, bf16
constexpr int kNRows = 16;                   // N of both MMAs (query heads, padded)
constexpr int kNBox = kNRows * 128;          // 16 rows x 128 B
constexpr int kNBytes = 2 * kNBox;           // 16 rows x 128 channels / keys
// Threads: softmax warps (4, or 8 for the 16-column fold: two groups of four
// sharing the TMEM lanes, each taking 8 of the 16 columns) + K producer + V
// producer + MMA.
__host__ __device__ constexpr int softmax_groups(int nc) { return nc > 8 ? 2 : 1; }
__host__ __device__ constexpr int threads_for(int nc) { return 32 * (4 * softmax_groups(nc) + 3); }
constexpr uint32_t kTmemCols = 64;
constexpr uint32_t kTmemS = 0;               // two 16-column score buffers
constexpr uint32_t kTmemO = 32;              // 16-column output accumulator

// 3-D tiled TMA load (Q: channel, head, query row).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
        : "memory");
}

// N consecutive TMEM columns of the thread's lane (N = 1, 2, 4, 8 or 16).
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
    if constexpr (N == 16) {
        float a[8], b[8];
        tc::tmem_ld_n<8>(taddr, a);
        tc::tmem_ld_n<8>(taddr + 8, b);
#pragma unroll
        for (int i = 0; i < 8; ++i) { v[i] = a[i]; v[8 + i] = b[i]; }
    } else {
        tc::tmem_ld_n<N>(taddr, v);
    }
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const float (&v)[N]) {
    if constexpr (N == 16) {
        float a[8], b[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) { a[i] = v[i]; b[i] = v[8 + i]; }
        tc::tmem_st_n<8>(taddr, a);
        tc::tmem_st_n<8>(taddr + 8, b);
    } else {
        tc::tmem_st_n<N>(taddr, v);
    }
}

// Maximum over the 32 lanes of the warp in one instruction (-inf is the
// identity; every lane gets the result).
__device__ __forceinline__ float warp_max_redux(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// First query row and row count of sequence b.
__device__ __forceinline__ void seq_rows(const GqaParams &p, int b, int &row0, int &nrows) {
    if (p.q_row_offsets) {
        row0 = int(p.q_row_offsets[b]);
        nrows = int(p.q_row_offsets[b + 1]) - row0;
    } else {
        row0 = b;
        nrows = 1;
    }
}

struct Smem {
    static constexpr int kring = 0;
    static constexpr int vring = kring + kStages * kTileBytes;
    static constexpr int q = vring + kStages * kTileBytes;     // [2] Q^T buffers
    static constexpr int p = q + 2 * kNBytes;                   // P^T
    static constexpr int red = p + kNBytes;                     // float [2][4][16] tile max
    static constexpr int lred = red + 2 * 4 * 16 * 4;           // float [2][4][2][16] row sums
    static constexpr int mrg = lred + 2 * 4 * 2 * 16 * 4;       // [2] merge buffers (clusters)
};
// One merge buffer: O^T partial [16 columns][128 channels] fp32, then m[16], l[16].
constexpr int kMrgO = 16 * 128 * 4;
constexpr int kMrgBytes = kMrgO + 2 * 16 * 4;
template <int C>
struct Tail {
    static constexpr int bars = Smem::mrg + (C > 1 ? 2 * kMrgBytes : 0);
    static constexpr int items = bars + 256;
};

// The balanced split's GqaRange sits after the barriers and the TMEM slot.
constexpr int kRangeOffset = 208;

enum Bar {
    kKFull = 0, kKEmpty = 3, kVFull = 6, kVEmpty = 9,   // [3] each
    kQFull = 12, kQEmpty = 14,                          // [2] each
    kSFull = 16, kSFree = 18,                           // [2] each
    kPFull = 20, kODone = 21,
    kMrgFull = 22,                                      // [2] clusters: partials in place
    kNumBars = 24
};
static_assert(kNumBars * 8 + 4 <= kRangeOffset && kRangeOffset + int(sizeof(GqaRange)) <= 256,
              "barriers, TMEM slot and range fit the 256-byte tail");

// Dynamic shared memory: the item table (one int per sequence) only without
// clusters.
template <int C>
size_t tc_smem_bytes(int batch) {
    return 1024 + size_t(Tail<C>::items) + (C > 1 ? 0 : sizeof(int) * size_t(batch + 1));
}

// Work walk of one CTA.  Without clusters: items (sequence, KV head, slice)
// j = blockIdx.x, blockIdx.x + gridDim.x, ...; under the balanced split the
// pieces of the units that meet the CTA's tile range, in order.  With
// clusters of C: units (sequence, KV head) j = cluster, cluster + clusters,
// ..., this CTA taking the slice of its rank.
template <int C>
__device__ __forceinline__ GqaWalk make_walk(const GqaParams &p, const int *cum, int hkv,
                                             const GqaRange &rg) {
    GqaWalk w;
    if (C == 1 && p.balanced) return gqa_balanced_walk(rg);
    w.first = C > 1 ? int(blockIdx.x) / C : int(blockIdx.x);
    w.stride = C > 1 ? int(gridDim.x) / C : int(gridDim.x);
    w.count = C > 1 ? p.batch * hkv : cum[p.batch];
    w.x0 = w.x1 = w.tiles = w.wtiles = w.ctas = 0;
    w.u0 = 0;
    return w;
}

template <int C>
__device__ __forceinline__ GqaItem walk_item(const GqaParams &p, const int *cum, int j, int hkv,
                                             const GqaWalk &w) {
    if constexpr (C == 1) {
        return p.balanced ? gqa_balanced_item(p, cum, hkv, w, j) : gqa_item<kBK>(p, cum, j, hkv);
    } else {
        GqaItem it;
        it.b = j / hkv;
        it.kvh = j - it.b * hkv;
        it.part = static_cast<int>(cluster_ctarank());
        const uint32_t cap = uint32_t(C) * uint32_t(p.chunk);
        const uint32_t len_in = p.kv_len[it.b];
        if (len_in > cap && it.kvh == 0 && it.part == 0 && threadIdx.x == 0)
            atomicOr(p.err, kErrBadLength);
        it.L = static_cast<int>(min(len_in, cap));
        // equal slices of this sequence, whole tiles
        const int cs = ((it.L + C - 1) / C + kBK - 1) / kBK * kBK;
        it.start = min(it.part * cs, it.L);
        it.end = min(it.start + cs, it.L);
        it.ntiles = it.start < it.end ? (it.end - it.start + kBK - 1) / kBK : 0;
        it.direct = false;
        it.unit = j;
        it.unit_x = it.unit_tiles = 0;
        it.first = false;
        return it;
    }
}

// Position of element (row r, column c) of a 16-row operand stored as two
// 128-byte-swizzled column boxes of 64 bf16 each.
__device__ __forceinline__ uint32_t n_operand_offset(int r, int c) {
    const int box = c >> 6, chunk = (c & 63) >> 3;
    return uint32_t(box * kNBox + r * 128 + ((chunk ^ (r & 7)) << 4) + (c & 7) * 2);
}

// Producer loop shared by the K (+Q) and V warps: walks this CTA's items and
// tiles, resolves pages lane-parallel (32 row boxes at a time) and lets lane
// 0 issue the boxes of each tile into the ring.
template <bool kIsK, int C>
__device__ __forceinline__ void produce(const GqaParams &p, const int *cum, const GqaWalk &w,
                                        int hkv, uint8_t *smem, uint64_t *bar, int lane) {
    const CUtensorMap *map = kIsK ? &p.k_map : &p.v_map;
    uint64_t *full = bar + (kIsK ? kKFull : kVFull);
    uint64_t *empty = bar + (kIsK ? kKEmpty : kVEmpty);
    uint8_t *ring = smem + (kIsK ? Smem::kring : Smem::vring);
    if (lane == 0) {
        prefetch_tensormap(map);
        if (kIsK) prefetch_tensormap(&p.q_map);
    }
    const int G = p.group;
    const int box_rows = p.box_rows;        // 128, 64, 32, 16 or 8
    const int nb = kBK / box_rows;          // row boxes per tile
    const uint32_t box_bytes = uint32_t(box_rows) * 128u;
    int g = 0, itq = 0;
    bool aborted = false;
    for (int j = w.first; j < w.count && !aborted; j += w.stride) {
        const GqaItem it = walk_item<C>(p, cum, j, hkv, w);
        if (it.ntiles == 0) continue;
        if (kIsK && lane == 0) {
            const int qb = itq & 1;
            if (itq >= 2 && !mbar_wait(&bar[kQEmpty + qb], ((itq >> 1) - 1) & 1, p.err)) {
                aborted = true;
            } else {
                // rows past the sequence (or the tensor) are masked columns
                int row0, nrows;
                seq_rows(p, it.b, row0, nrows);
                mbar_arrive_expect_tx(&bar[kQFull + qb],
                                      2u * uint32_t(G) * uint32_t(p.max_q_len) * 128u);
                uint8_t *qs = smem + Smem::q + qb * kNBytes;
                for (int cb = 0; cb < 2; ++cb)
                    tma_load_3d(qs + cb * kNBox, &p.q_map, &bar[kQFull + qb], cb * 64,
                                it.kvh * G, row0);
            }
        }
        aborted = __shfl_sync(0xffffffffu, aborted, 0);
        int cached = -1, my_page = -1, my_slot = 0;
        for (int t = 0; t < it.ntiles && !aborted; ++t) {
            const int gg = g + t;
            const int s = gg % kStages;
            const int key0 = it.start + t * kBK;
            const int live = min(nb, (it.L - key0 + box_rows - 1) / box_rows);
            if (lane == 0) {
                if (gg >= kStages && !mbar_wait(&empty[s], ((gg / kStages) - 1) & 1, p.err))
                    aborted = true;
                else
                    mbar_arrive_expect_tx(&full[s], uint32_t(live) * 2u * box_bytes);
            }
            aborted = __shfl_sync(0xffffffffu, aborted, 0);
            if (aborted) break;
            uint8_t *dst = ring + s * kTileBytes;
            for (int r = 0; r < live; ++r) {
                const int gb = (key0 - it.start) / box_rows + r;   // box index in the item
                if ((gb >> 5) != cached) {                          // warp-uniform refill
                    cached = gb >> 5;
                    const int tk = it.start + ((cached << 5) + lane) * box_rows;
                    my_page = -1;
                    my_slot = 0;
                    if (tk < it.L) {
                        if (p.page_table) {
                            const int pidx = tk / p.page_size;
                            int e = pidx < p.max_pages
                                        ? p.page_table[size_t(it.b) * p.max_pages + pidx] : -1;
                            if (e < 0 || e >= p.num_pages) {
                                if (kIsK) atomicOr(p.err, kErrBadPage);
                                e = -1;
                            }
                            my_page = e;
                            my_slot = tk % p.page_size;
                        } else {
                            my_page = it.b;
                            my_slot = tk;
                        }
                    }
                }
                const int page = __shfl_sync(0xffffffffu, my_page, gb & 31);
                const int slot = __shfl_sync(0xffffffffu, my_slot, gb & 31);
                if (lane == 0) {
                    if (page < 0) {
                        mbar_complete_tx(&full[s], 2u * box_bytes);   // skipped bad page
                    } else {
#pragma unroll
                        for (int cb = 0; cb < 2; ++cb)
                            tma_load_4d(dst + cb * kBox + r * box_rows * 128, map, &full[s],
                                        cb * 64, slot, it.kvh, page);
                    }
                }
            }
        }
        g += it.ntiles;
        ++itq;
    }
    // Every copy this warp issued must land before the CTA may leave.
    if (lane == 0) {
        for (int i = max(0, g - kStages); i < g; ++i)
            mbar_wait(&full[i % kStages], (i / kStages) & 1, p.err);
        if (kIsK)
            for (int i = max(0, itq - 2); i < itq; ++i)
                mbar_wait(&bar[kQFull + (i & 1)], (i >> 1) & 1, p.err);
    }
}

// G: query heads per KV head; NC: score columns (G for one row per sequence,
// 16 for the few-token fold).
template <int G, int NC, int C>
__global__ void __launch_bounds__(threads_for(NC), 1)
gqa_decode_tc_kernel(const __grid_constant__ GqaParams p) {
    constexpr int kGroups = softmax_groups(NC);   // softmax warp groups
    constexpr int NW = NC / kGroups;              // score columns per group
    constexpr int kWarpK = 4 * kGroups, kWarpV = kWarpK + 1, kWarpMma = kWarpK + 2;
    constexpr int kThreads = threads_for(NC);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Tail<C>::bars);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Tail<C>::bars + kNumBars * 8);
    int *cum = reinterpret_cast<int *>(smem + Tail<C>::items);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int hkv = p.num_q_heads / G;

    GqaRange *range = reinterpret_cast<GqaRange *>(smem + Tail<C>::bars + kRangeOffset);
    if (C == 1 && warp == 0) gqa_build_items(p, hkv, cum, lane, range);
    if (threadIdx.x == 32) {
        for (int i = 0; i < kNumBars; ++i) {
            const bool per_warp = (i == kSFree || i == kSFree + 1 || i == kPFull);
            const bool merge = i == kMrgFull || i == kMrgFull + 1;
            mbar_init(&bar[i], merge ? 4u * kGroups * C : (per_warp ? 4u * kGroups : 1u));
        }
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    // Padding rows of the Q^T and P^T operands (columns past the loaded
    // rows) stay zero.
    for (int i = threadIdx.x; i < (3 * kNBytes) / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem + Smem::q)[i] = make_uint4(0u, 0u, 0u, 0u);
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if constexpr (C > 1) cluster_sync();   // every CTA's barriers exist before a remote arrive
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const GqaWalk walk = make_walk<C>(p, cum, hkv, *range);

    if (warp == kWarpK) {
        produce<true, C>(p, cum, walk, hkv, smem, bar, lane);
    } else if (warp == kWarpV) {
        produce<false, C>(p, cum, walk, hkv, smem, bar, lane);
    } else if (warp == kWarpMma) {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc_s = tc::idesc_bf16_f32(128, kNRows, 0, 0);
            constexpr uint32_t idesc_o = tc::idesc_bf16_f32(128, kNRows, 1, 0);
            const uint32_t k_base = smem_addr(smem + Smem::kring);
            const uint32_t v_base = smem_addr(smem + Smem::vring);
            const uint32_t q_base = smem_addr(smem + Smem::q);
            const uint32_t p_base = smem_addr(smem + Smem::p);
            int g = 0, itq = 0;
            bool ok = true;
            for (int j = walk.first; ok && j < walk.count; j += walk.stride) {
                const GqaItem it = walk_item<C>(p, cum, j, hkv, walk);
                if (it.ntiles == 0) continue;
                const int qb = itq & 1;
                ok = mbar_wait(&bar[kQFull + qb], (itq >> 1) & 1, p.err);
                for (int t = 0; ok && t <= it.ntiles; ++t) {
                    if (t < it.ntiles) {
                        const int gg = g + t;
                        const int ks = gg % kStages;
                        const int sb = gg & 1;
                        ok = mbar_wait(&bar[kKFull + ks], (gg / kStages) & 1, p.err);
                        if (ok && gg >= 2)
                            ok = mbar_wait(&bar[kSFree + sb], ((gg >> 1) - 1) & 1, p.err);
                        if (!ok) break;
                        tc::fence_after_sync();
                        const uint32_t kst = k_base + ks * kTileBytes;
                        const uint32_t qst = q_base + qb * kNBytes;
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk) {
                            const uint32_t ka = kst + (kk >> 2) * kBox + (kk & 3) * 32;
                            const uint32_t qa = qst + (kk >> 2) * kNBox + (kk & 3) * 32;
                            tc::mma_bf16(tmem + kTmemS + sb * kNRows,
                                         tc::smem_desc_sw128(ka, 16, 1024),
                                         tc::smem_desc_sw128(qa, 16, 1024), idesc_s, kk > 0);
                        }
                        tc::mma_commit(&bar[kSFull + sb]);
                        tc::mma_commit(&bar[kKEmpty + ks]);
                    }
                    if (t >= 1) {
                        const int gp = g + t - 1;
                        const int vs = gp % kStages;
                        ok = mbar_wait(&bar[kPFull], gp & 1, p.err);
                        if (ok) ok = mbar_wait(&bar[kVFull + vs], (gp / kStages) & 1, p.err);
                        if (!ok) break;
                        tc::fence_after_sync();
                        const uint32_t vst = v_base + vs * kTileBytes;
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            const uint32_t pa = p_base + (kk >> 2) * kNBox + (kk & 3) * 32;
                            // V^T as the MN-major A operand: channel blocks of 64
                            // are the two 16 KB column boxes, 8-key groups 1 KB apart.
                            tc::mma_bf16(tmem + kTmemO,
                                         tc::smem_desc_sw128(vst + kk * 16 * 128, kBox, 1024),
                                         tc::smem_desc_sw128(pa, 16, 1024), idesc_o,
                                         t > 1 || kk > 0);
                        }
                        tc::mma_commit(&bar[kODone]);
                        tc::mma_commit(&bar[kVEmpty + vs]);
                    }
                }
                tc::mma_commit(&bar[kQEmpty + qb]);
                g += it.ntiles;
                ++itq;
            }
        }
    } else {
        // ---------------------------------------------------- softmax + epilogue
        const int kw = warp & 3;                     // key warp: TMEM lanes 32 kw ..
        const int grp = warp >> 2;                   // column group: columns grp * NW ..
        const int cg0 = grp * NW;
        const int k = kw * 32 + lane;                // key of the tile == TMEM lane
        const uint32_t lane_base = uint32_t(kw * 32) << 16;
        float *red = reinterpret_cast<float *>(smem + Smem::red);     // [2][4][16]
        float *lred = reinterpret_cast<float *>(smem + Smem::lred);   // [2][4][16]
        uint8_t *pbuf = smem + Smem::p;
        int g = 0, iter = 0;
        bool ok = true;
        for (int j = walk.first; j < walk.count; j += walk.stride, ++iter) {
            const GqaItem it = walk_item<C>(p, cum, j, hkv, walk);
            int row0, nrows;
            seq_rows(p, it.b, row0, nrows);
            // Column cg = (row cg / G, head cg % G): keys j < lim visible.
            // This group's columns: cg = cg0 + c, c < NW.
            int lim[NW];
#pragma unroll
            for (int c = 0; c < NW; ++c) {
                const int i = (cg0 + c) / G;
                lim[c] = i >= nrows ? 0 : (p.causal ? it.L - nrows + i + 1 : it.L);
            }
            float m[NW], l[NW], lr[NW];
#pragma unroll
            for (int c = 0; c < NW; ++c) {
                m[c] = -INFINITY;
                l[c] = 0.f;
                lr[c] = 0.f;
            }
            // Every warp runs every named barrier of every tile, even after a
            // wait gave up (ok == false), so no warp can strand the others.
            for (int t = 0; t < it.ntiles; ++t) {
                const int gg = g + t;
                const int sb = gg & 1;
                const int t0 = it.start + t * kBK;
                const int nvalid = min(kBK, it.end - t0);
                ok = ok && mbar_wait(&bar[kSFull + sb], (gg >> 1) & 1, p.err);
                tc::fence_after_sync();
                float s[NW];
                tmem_ld_cols<NW>(tmem + lane_base + kTmemS + sb * kNRows + cg0, s);
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[kSFree + sb]);

                // ---- tile max per column across the four warps ---------------
                const bool valid = k < nvalid;
                float *rb = red + (gg & 1) * 64;
#pragma unroll
                for (int c = 0; c < NW; ++c) {
                    s[c] = valid && t0 + k < lim[c] ? s[c] * p.qk_scale_log2 : -INFINITY;
                    const float wm = warp_max_redux(s[c]);
                    if (lane == 0) rb[kw * 16 + cg0 + c] = wm;
                }
                named_sync(1 + grp, 128);
                float alpha[NW];
                bool moved = false;
#pragma unroll
                for (int c = 0; c < NW; ++c) {
                    const int cg = cg0 + c;
                    const float tmax =
                        fmaxf(fmaxf(rb[cg], rb[16 + cg]), fmaxf(rb[32 + cg], rb[48 + cg]));
                    const float mn = fmaxf(m[c], tmax);
                    // A column with no visible key so far keeps m = -inf and
                    // weights 0 (its alpha is irrelevant: l and O are 0).
                    alpha[c] = mn == -INFINITY ? 1.f : fast_exp2(m[c] - mn);   // 0 on the first
                    moved |= mn != m[c];
                    m[c] = mn;
                }
                uint16_t pb[NW];
#pragma unroll
                for (int c = 0; c < NW; ++c) {
                    const float pv = s[c] != -INFINITY ? fast_exp2(s[c] - m[c]) : 0.f;
                    const uint32_t packed = pack_bf16x2(pv, 0.f);
                    pb[c] = static_cast<uint16_t>(packed & 0xffffu);
                    l[c] = l[c] * alpha[c] + pv;
                    lr[c] = lr[c] * alpha[c] + bf16_lo(packed);
                }
                if (t >= 1) {
                    // O^T(t-1) is complete: P^T may be overwritten and O^T
                    // rescaled (thread = channel lane, columns = heads).
                    ok = ok && mbar_wait(&bar[kODone], (gg - 1) & 1, p.err);
                    tc::fence_after_sync();
                    if (moved) {   // identical in every thread of the group
                        float o[NW];
                        tmem_ld_cols<NW>(tmem + lane_base + kTmemO + cg0, o);
#pragma unroll
                        for (int c = 0; c < NW; ++c) o[c] *= alpha[c];
                        tmem_st_cols<NW>(tmem + lane_base + kTmemO + cg0, o);
                        tc::tmem_wait_st();
                    }
                }
#pragma unroll
                for (int c = 0; c < NW; ++c)
                    *reinterpret_cast<uint16_t *>(pbuf + n_operand_offset(cg0 + c, k)) = pb[c];
                if (grp == 0 && t0 + kBK > it.L) {
                    // Slots past the sequence end may hold anything (even NaN):
                    // zero them in the V stage before P.V reads it.
                    const int vs = gg % kStages;
                    ok = ok && mbar_wait(&bar[kVFull + vs], (gg / kStages) & 1, p.err);
                    uint8_t *vst = smem + Smem::vring + vs * kTileBytes;
                    const int first = it.L - t0;               // first invalid key
                    const int nz = (kBK - first) * 8;          // 16-B chunks per box
                    for (int i = k; i < 2 * nz; i += 128) {
                        const int box = i / nz, rem = i - (i / nz) * nz;
                        *reinterpret_cast<uint4 *>(vst + box * kBox + (first + rem / 8) * 128 +
                                                   (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                tc::fence_async_smem();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[kPFull]);
            }

            // ---- item epilogue ----------------------------------------------------
            // The row sums first: they do not need O, so their exchange runs
            // while the last P.V is still in flight.
            float lsum[NW], lrsum[NW];
            {
                float *lb = lred + (iter & 1) * 128;   // [4 key warps][2][16 columns]
#pragma unroll
                for (int c = 0; c < NW; ++c) {
                    const float a = warp_sum(l[c]);
                    const float b2 = warp_sum(lr[c]);
                    if (lane == 0) {
                        lb[kw * 32 + cg0 + c] = a;
                        lb[kw * 32 + 16 + cg0 + c] = b2;
                    }
                }
                named_sync(1 + grp, 128);
#pragma unroll
                for (int c = 0; c < NW; ++c) {
                    const int cg = cg0 + c;
                    lsum[c] = (lb[cg] + lb[32 + cg]) + (lb[64 + cg] + lb[96 + cg]);
                    lrsum[c] = (lb[16 + cg] + lb[48 + cg]) + (lb[80 + cg] + lb[112 + cg]);
                }
            }
            if (ok && it.ntiles > 0) {
                ok = mbar_wait(&bar[kODone], (g + it.ntiles - 1) & 1, p.err);
                tc::fence_after_sync();
            }
            float o[NW];
            if (ok && it.ntiles > 0) {
                tmem_ld_cols<NW>(tmem + lane_base + kTmemO + cg0, o);
            } else {
#pragma unroll
                for (int c = 0; c < NW; ++c) o[c] = 0.f;
            }
            tc::fence_before_sync();
            if constexpr (C == 1) {
                const int ch = k;   // output channel of this thread
#pragma unroll
                for (int c = 0; c < NW; ++c) {
                    const int i = (cg0 + c) / G, h = (cg0 + c) % G;
                    if (i >= nrows) continue;
                    const int hq = it.kvh * G + h;
                    const size_t row = size_t(row0 + i);
                    if (it.direct) {
                        const float t2 = p.sink ? p.sink[hq] * kLog2e : -INFINITY;
                        const float Mf = fmaxf(m[c], t2);
                        float Z = 0.f, Zr = 0.f, so = 0.f;
                        if (Mf != -INFINITY) {
                            so = fast_exp2(m[c] - Mf);     // 0 when m = -inf
                            const float st = fast_exp2(t2 - Mf);
                            Z = lsum[c] * so + st;
                            Zr = lrsum[c] * so + st;
                        }
                        const float scale_o = Zr > 0.f ? so / Zr : 0.f;
                        const uint32_t packed = pack_bf16x2(o[c] * scale_o, 0.f);
                        p.out[(row * p.num_q_heads + hq) * kD + ch] =
                            static_cast<uint16_t>(packed & 0xffffu);
                        if (ch == 0 && p.lse)
                            p.lse[row * p.num_q_heads + hq] =
                                Z > 0.f ? (Mf + fast_log2(Z)) * kLn2 : -INFINITY;
                    } else {
                        // partition part: [P][rows][heads]; balanced-split slot:
                        // [slots][16 columns]
                        const size_t base =
                            p.balanced ? size_t(it.part) * kGqaSlotCols + (cg0 + c)
                                       : (size_t(it.part) * p.num_q_rows + row) * p.num_q_heads + hq;
                        const float scale_o = lrsum[c] > 0.f ? lsum[c] / lrsum[c] : 0.f;
                        p.ws_o[base * kD + ch] = o[c] * scale_o;
                        if (ch == 0) {
                            p.ws_m[base] = m[c] * kLn2;
                            p.ws_l[base] = lsum[c];
                        }
                    }
                }
                if (p.balanced && it.first && threadIdx.x == 0) {
                    // The CTA holding the unit's first tile publishes where its
                    // pieces are: slots c + unit for the CTAs c holding its
                    // first through last tile (CTA ((y + 1) C' - 1) / T_w holds
                    // weighted position y; tile x of unit u sits at y = x +
                    // kGqaUnitCost (u + 1)).
                    const long long last = it.unit_x + it.unit_tiles - 1 +
                                           static_cast<long long>(kGqaUnitCost) * (it.unit + 1);
                    const int c_last =
                        static_cast<int>(((last + 1) * walk.ctas - 1) / walk.wtiles);
                    const int c_first = static_cast<int>(blockIdx.x);
                    p.unit_slots[it.unit] = make_int2(c_first + it.unit, c_last - c_first + 1);
                }
            } else {
                // ---- on-chip merge of the cluster's partials -----------------
                const int buf = iter & 1;
                const int rank = it.part;
                uint8_t *mb = smem + Smem::mrg + buf * kMrgBytes;
                float *mo = reinterpret_cast<float *>(mb);                 // [16][128]
                float *mml = reinterpret_cast<float *>(mb + kMrgO);        // m[16], l[16]
#pragma unroll
                for (int c = 0; c < NW; ++c) {
                    // normalised to the fp32 weight sum, as a workspace partial
                    const float scale_o = lrsum[c] > 0.f ? lsum[c] / lrsum[c] : 0.f;
                    mo[(cg0 + c) * 128 + k] = o[c] * scale_o;
                }
                if (k == 0) {
#pragma unroll
                    for (int c = 0; c < NW; ++c) {
                        mml[cg0 + c] = m[c];        // base 2
                        mml[16 + cg0 + c] = lsum[c];
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    const uint32_t local = smem_addr(&bar[kMrgFull + buf]);
#pragma unroll
                    for (int q = 0; q < C; ++q) mbar_arrive_cluster(mapa_shared(local, q));
                }
                ok = mbar_wait_cluster(&bar[kMrgFull + buf], (iter >> 1) & 1, p.err) && ok;
                // this CTA's output channels [rank * 128 / C, (rank + 1) * 128 / C)
                constexpr int kChs = 128 / C;
                const uint32_t mb_local = smem_addr(mb);
                for (int idx = grp * 128 + k; idx < NC * kChs; idx += 128 * kGroups) {
                    const int c = idx / kChs;
                    const int chl = rank * kChs + (idx - c * kChs);
                    const int i = c / G, h = c % G;
                    if (i >= nrows) continue;
                    const int hq = it.kvh * G + h;
                    const size_t row = size_t(row0 + i);
                    float mq[C], lq[C], oq[C];
#pragma unroll
                    for (int q = 0; q < C; ++q) {
                        const uint32_t base = mapa_shared(mb_local, q);
                        mq[q] = ld_cluster_f32(base + uint32_t(kMrgO + 4 * c));
                        lq[q] = ld_cluster_f32(base + uint32_t(kMrgO + 64 + 4 * c));
                        oq[q] = ld_cluster_f32(base + uint32_t(4 * (c * 128 + chl)));
                    }
                    const float t2 = p.sink ? p.sink[hq] * kLog2e : -INFINITY;
                    float Mf = t2;
#pragma unroll
                    for (int q = 0; q < C; ++q) Mf = fmaxf(Mf, mq[q]);
                    float Z = 0.f, acc = 0.f;
                    if (Mf != -INFINITY) {
                        Z = fast_exp2(t2 - Mf);
#pragma unroll
                        for (int q = 0; q < C; ++q) {
                            const float w = mq[q] == -INFINITY ? 0.f : fast_exp2(mq[q] - Mf);
                            Z += w * lq[q];
                            acc += w * oq[q];
                        }
                    }
                    const uint32_t packed = pack_bf16x2(Z > 0.f ? acc / Z : 0.f, 0.f);
                    p.out[(row * p.num_q_heads + hq) * kD + chl] =
                        static_cast<uint16_t>(packed & 0xffffu);
                    if (chl == 0 && p.lse)
                        p.lse[row * p.num_q_heads + hq] =
                            Z > 0.f ? (Mf + fast_log2(Z)) * kLn2 : -INFINITY;
                }
            }
            g += it.ntiles;
        }
        pdl_launch_dependents();
    }

    tc::fence_before_sync();
    __syncthreads();
    if constexpr (C > 1) cluster_sync();   // no CTA leaves while a peer may read its partials
    if (warp == kWarpMma) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

int g_num_sms_tc[64];
int g_max_clusters_tc[64][2];   // clusters of 2 / 4 that fit at once, per device

template <int G, int NC, int C>
cudaError_t launch_g(const GqaParams &p, cudaStream_t stream) {
    const size_t smem = tc_smem_bytes<C>(p.batch);
    auto kern = gqa_decode_tc_kernel<G, NC, C>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (g_num_sms_tc[dev] == 0) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_num_sms_tc[dev] = n;
    }
    const long long units = static_cast<long long>(p.batch) * (p.num_q_heads / G);
    if constexpr (C == 1) {
        long long grid = g_num_sms_tc[dev];   // one resident CTA per SM
        const long long max_items = units * p.num_partitions;
        if (grid > max_items && !p.balanced) grid = max_items;
        if (grid < 1) grid = 1;
        kern<<<dim3(static_cast<unsigned>(grid)), threads_for(NC), smem, stream>>>(p);
        return cudaGetLastError();
    } else {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(threads_for(NC));
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int &max_clusters = g_max_clusters_tc[dev][C == 2 ? 0 : 1];
        if (max_clusters == 0) {
            cfg.gridDim = dim3(static_cast<unsigned>(g_num_sms_tc[dev] / C * C));
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
            if (e != cudaSuccess) return e;
            max_clusters = n > 0 ? n : 1;
        }
        long long clusters = max_clusters;   // persistent: one wave of clusters
        if (clusters > units) clusters = units;
        if (clusters < 1) clusters = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(clusters * C));
        e = cudaLaunchKernelEx(&cfg, kern, p);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
}

template <int G, int NC>
cudaError_t launch_c(const GqaParams &p, cudaStream_t stream) {
    switch (p.cluster) {
        case 0:
        case 1: return launch_g<G, NC, 1>(p, stream);
        case 2: return launch_g<G, NC, 2>(p, stream);
        case 4: return launch_g<G, NC, 4>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gqa_decode_tc(const GqaParams &p, cudaStream_t stream) {
    if (p.head_dim != kD || p.max_q_len < 1 || p.max_q_len * p.group > kNRows)
        return cudaErrorInvalidValue;
    const bool fold = p.max_q_len > 1;
    switch (p.group) {
        case 1: return fold ? launch_c<1, 16>(p, stream) : launch_c<1, 1>(p, stream);
        case 2: return fold ? launch_c<2, 16>(p, stream) : launch_c<2, 2>(p, stream);
        case 4: return fold ? launch_c<4, 16>(p, stream) : launch_c<4, 4>(p, stream);
        case 8: return fold ? launch_c<8, 16>(p, stream) : launch_c<8, 8>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
