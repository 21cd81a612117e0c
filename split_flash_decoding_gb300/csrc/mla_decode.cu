// mla_decode.cu -- split-K MLA decode on the 5th-generation tensor cores.
//
// Multi-head latent attention decode: 128 query heads attend to one KV head
// whose rows are 576 channels (512 latent + 64 rope), and V is the first 512
// channels of K, which is never fetched a second time (one KV head and V
// taken from K: flare_mla_decoding_dispatch, Parameters: kv_num_heads and
// Args: k).
//
// Work: clusters of two CTAs.  Fixed split (num_partitions P >= 1): one
// cluster per (key slice p, query row).  Balanced split (P = 0): one wave of
// clusters, cluster c taking a contiguous range of equal cost (tiles plus a
// fixed cost per row it opens) of the concatenated 64-key tiles of all query
// rows, found by the cluster from the lengths and walked as runs of
// consecutive tiles of one row; a run that is a whole row writes the output,
// a run cut by a range end writes a partial that the split-K reduce merges.  The 128 heads are the MMA's M dimension.
// The two CTAs of a cluster split the 576 channels evenly:
//
//   rank 0 loads channels [0, 256)   (its half of V) + rope [512, 544),
//   rank 1 loads channels [256, 512) (its half of V) + rope [544, 576),
//
// as four 64-channel TMA boxes (128-byte swizzle) and one 32-channel box
// (64-byte swizzle) per row group, so every byte of a K row is fetched from
// HBM exactly once per cluster and both CTAs issue 18 score MMA steps.
// Per 64-key tile each CTA computes a partial score S_r = Q[:, ch_r] K[:, ch_r]^T
// with tcgen05.mma into TMEM, the two CTAs swap partials through distributed
// shared memory and add them (fp32 addition is commutative, so both hold the
// identical full S), run the same online softmax, and each accumulates its
// half of the output, O_r += P V[:, 256 r : 256 r + 256], in TMEM.
//
// The partial-score exchange is the critical resource (32 KB each way per
// tile over the SM-to-SM network), so it is kept busy: the softmax warps
// work one tile ahead, staging tile t+1's partial scores for the copy
// before they run the softmax of tile t, which then overlaps the copy of
// tile t+1; and the receive side has three key-half slots, so the copy of
// a half never waits for the peer to finish reading the previous tile.
//
// Warp roles (352 threads per CTA):
//   warps 0-7  softmax: warps w and w+4 share head rows 32(w%4).. (their
//              TMEM lanes); warp half w/4 owns keys [32 half, 32 half + 32)
//              of every tile.  Per tile t: read the partial S(t+1) from TMEM
//              and stage it for the copy, add the peer's partial of S(t),
//              online softmax (row maxima of the two halves combined through
//              shared memory), P(t) (bf16 pairs) into TMEM, where the P.V MMA
//              takes it as the A operand.  They also copy this CTA's Q
//              channels into TMEM.
//   warp 8     TMA producer (K tiles into a 4-stage ring)
//   warp 9     TMEM allocation and MMA issue (one thread), order
//              S0 S1 S2 O0 S3 O1 ...: the score MMA of tile t+2 is issued
//              as soon as S(t+1) has been read, ahead of O(t)
//   warp 10    exchange: two bulk copies per tile, one per key half
//              (cp.async.bulk, shared::cta to the peer's shared::cluster,
//              complete-tx on the peer's barrier of the receiving slot),
//              16 KB each; a half is staged while the other half is on the
//              wire.  Half i = 2 t + half of the CTA's tile sequence lands
//              in receive slot i % 3.
//
// Q is the A operand of the score MMA straight from TMEM, so shared memory
// holds only the K ring and the exchange buffers.  TMEM columns: Q [0, 144)
// (bf16 pairs: 256 V channels, then 32 rope channels), P [160, 192), S
// [192, 256), O half [256, 512).
// The running max is kept lazily: P = exp2(s - m_ref) with m_ref raised (and
// O rescaled) only when a tile's max exceeds m_ref by more than 8 (base 2),
// so P <= 256 and O/l stay finite in fp32.
#include "launch.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace attn {
namespace {

constexpr int kBN = kMlaTileKeys;          // 64 keys per tile
constexpr int kStages = 4;
constexpr int kVBoxes = 4;                 // 64-channel boxes: this CTA's 256 V channels
constexpr int kKBoxBytes = kBN * 128;      // 64 rows x 128 B
constexpr int kRopeBoxBytes = kBN * 2 * kMlaRopeBoxCh;   // 64 rows x 64 B
constexpr int kStageBytes = kVBoxes * kKBoxBytes + kRopeBoxBytes;   // 36 KB
constexpr int kScoreSteps = (kVBoxes * 64 + kMlaRopeBoxCh) / 16;   // 18 MMAs of K = 16
constexpr int kSoftmaxThreads = 256;   // warps 0-7

// Warp roles.  Dense (paged or contiguous) caches: 352 threads, one TMA
// producer warp (8), MMA warp 9, exchange warp 10.  Sparse top-k: 512 threads,
// six TMA gather4 producer warps (8-11, 14, 15), MMA warp 12, exchange warp 13;
// the softmax warpgroups raise their register budget to 152 and the other
// two lower theirs to 104 (256 x 152 + 256 x 104 = 512 x 128 launched).
template <bool kSparse>
struct Layout {
    static constexpr int kThreads = kSparse ? 512 : 352;
    static constexpr int kMmaWarp = kSparse ? 12 : 9;
    static constexpr int kXchgWarp = kSparse ? 13 : 10;
    static constexpr int kProducers = kSparse ? 6 : 1;
    // producer index of a warp, or -1
    static __device__ __forceinline__ int producer(int warp) {
        if (!kSparse) return warp == 8 ? 0 : -1;
        if (warp >= 8 && warp < 12) return warp - 8;
        return warp >= 14 ? warp - 10 : -1;
    }
};
constexpr int kBarPair = 2;            // + (warp & 3): the two softmax warps of a row quarter
constexpr uint32_t kXBytes = 128u * kMlaTileKeys * 4u;   // one tile of fp32 partial scores
constexpr uint32_t kXHalfBytes = kXBytes / 2;            // one key half (32 keys)
constexpr int kXSlots = 3;                               // receive slots of key halves
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemQ = 0;             // 144 columns of packed bf16 pairs
constexpr uint32_t kTmemP = 160;           // 32 columns: P of one tile as bf16 pairs
constexpr uint32_t kTmemS = 192;           // 64-column S buffer
constexpr uint32_t kTmemO = 256;           // 256-column O half
constexpr float kRescaleThreshold = 8.0f;  // base-2 units

// V (B operand of O = P V) is MN-major: 4 boxes of 64 channels x 64 keys.
constexpr uint32_t kVLbo = kKBoxBytes;     // stride between 64-channel blocks
constexpr uint32_t kVSbo = 1024;           // stride between 8-key groups

struct Smem {
    static constexpr int kv = 0;
    static constexpr int x_in = kv + kStages * kStageBytes;           // 144 KB
    static constexpr int x_out = x_in + kXSlots * int(kXHalfBytes);   // +48 KB (peer's partials)
    static constexpr int red = x_out + int(kXBytes);                  // +32 KB (own partial)
    static constexpr int bars = red + 2 * 128 * 4;                    // +1 KB (row maxima)
    static constexpr int range = bars + 192;                          // balanced: MlaRange
    static constexpr int total = range + 64;
};
constexpr size_t kSmemBytes = Smem::total + 1024;

enum Bar {
    kKvFull = 0,                // [kStages]
    kKvEmpty = kStages,         // [kStages]
    kQFull = 2 * kStages,
    kSFull,       // partial S of a tile in TMEM (MMA commit)
    kSFree,       // the softmax warps have read it (4 arrivals)
    kPFull,       // P of a tile in TMEM, V tail cleared (4 arrivals)
    kODone,       // O MMA of a tile finished (commit)
    // [kXSlots] each: one per receive slot
    kXFull,                           // peer's half landed in the slot (own expect_tx + copy bytes)
    kXPeerFree = kXFull + kXSlots,    // the peer has read the slot (its 4 warps of that half)
    // [2] each: one per key half of x_out
    kXoReady = kXPeerFree + kXSlots,  // own 4 softmax warps of the half staged x_out
    kXoFree = kXoReady + 2,           // the bulk copy finished reading the half of x_out
    kXEnd = kXoFree + 2,
    kNumBars = kXEnd
};

// Partial score row h of one key half (32 keys, 128 B) in slot k of an
// exchange buffer: 16-B chunk c at a row-dependent rotation, so the 8 rows of
// a quarter-warp access hit all 32 banks.
__device__ __forceinline__ uint32_t x_half_off(int k, int h, int c) {
    return uint32_t(k) * kXHalfBytes + uint32_t(h * 128 + (((c + h) & 7) << 4));
}

// Row r (0..31), 16-byte chunk k of a warp's 4 KB slice of x_out, with the
// same rotation: both a lane per row and eight lanes per row are free of
// bank conflicts.
__device__ __forceinline__ uint32_t xw_off(int r, int k) {
    return uint32_t(r * 128 + (((k + r) & 7) << 4));
}

// One run of consecutive key tiles of one query row: keys [start, end) of
// row qrow (sequence b).  direct: the run is the whole row, so the final
// output is written; otherwise the partial goes to workspace slot ws.
struct MlaSeg {
    int qrow, b, start, end, ntiles, ws;
    bool direct;
};

// Fixed split: key slice `part` of query row qrow of sequence b (one row per
// sequence, or several given by row offsets, each with its own causal
// limit).  Every row of a sequence uses the same key slices; a row that sees
// none of a slice leaves an empty partial.  Returns false for a slice past
// the sequence end (no work at all).
template <bool kSparse>
__device__ __forceinline__ bool fixed_slice(const MlaParams &p, MlaSeg &s, bool report) {
    const int part = blockIdx.x >> 1;
    const int qrow = blockIdx.y;
    int b = qrow, n_rows = 1, i_row = 0;
    if (p.q_row_offsets) {
        int lo = 0, hi = p.batch;   // off[lo] <= qrow < off[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (static_cast<int>(p.q_row_offsets[mid]) <= qrow) lo = mid;
            else hi = mid;
        }
        b = lo;
        i_row = qrow - static_cast<int>(p.q_row_offsets[b]);
        n_rows = static_cast<int>(p.q_row_offsets[b + 1]) - static_cast<int>(p.q_row_offsets[b]);
    }
    uint32_t cap = uint32_t(p.num_partitions) * uint32_t(p.chunk);
    if (kSparse) cap = min(cap, uint32_t(p.indices_stride));   // keys a sequence can name
    const uint32_t len_in = p.kv_len[b];
    if (report && len_in > cap && part == 0) atomicOr(p.err, kErrBadLength);
    const int L = static_cast<int>(min(len_in, cap));
    const int start = part * p.chunk;
    const int nslices = (L + p.chunk - 1) / p.chunk;
    s.direct = nslices <= 1;
    if (start >= L && !(s.direct && part == 0)) return false;
    // keys j <= L - n + i for row i of n when causal
    const int L_vis = p.causal ? max(0, min(L, L - n_rows + i_row + 1)) : L;
    const int end = min(min(start + p.chunk, L), L_vis);
    s.qrow = qrow;
    s.b = b;
    s.start = start;
    s.end = end;
    s.ntiles = start < end ? (end - start + kBN - 1) / kBN : 0;
    s.ws = part * p.num_q_rows + qrow;
    return true;
}

// Balanced split: a cluster's time is
// its tiles plus a fixed cost for every run it opens (the row's Q into TMEM
// and the pipeline refill, then the epilogue: about kRunCost tiles' worth),
// so the split deals out a weighted concatenation in which every row with
// tiles is preceded by kRunCost virtual tiles: row r (n_r tiles from tile
// cum_r) occupies weighted positions [W_r, W_r + kRunCost + n_r), its real
// tile x at y(x) = x - cum_r + W_r + kRunCost.  Cluster c of C = min(clusters,
// T) takes the weighted positions [c T_w / C, (c+1) T_w / C) of the T_w in
// all, i.e. the real tiles from the image of its first position (a position
// inside a virtual block maps to the row's first tile) up to the next
// cluster's; a range inside one virtual block is empty.  A cluster whose
// range meets more rows so gets fewer tiles.
constexpr int kRunCost = 8;

// The rows of sequence b: first row r0, count nr (clipped to [0, rows)), and
// its visible length L (at most cap).
struct MlaSeqRows {
    int r0, nr, L;
};
__device__ __forceinline__ MlaSeqRows mla_seq_rows(const MlaParams &p, int b, uint32_t cap) {
    MlaSeqRows q;
    q.L = static_cast<int>(min(p.kv_len[b], cap));
    q.r0 = p.q_row_offsets ? static_cast<int>(p.q_row_offsets[b]) : b;
    q.nr = p.q_row_offsets ? static_cast<int>(p.q_row_offsets[b + 1]) - q.r0 : 1;
    q.nr = max(0, min(q.nr, p.num_q_rows - q.r0));   // rows outside [0, rows) are skipped
    if (q.r0 < 0) q.nr = 0;
    return q;
}
// Row i of n of a sequence of length L sees keys j <= L - n + i when causal.
__device__ __forceinline__ int mla_row_vis(const MlaParams &p, int L, int nr, int i) {
    return p.causal ? max(0, min(L, L - nr + i + 1)) : L;
}

// The runs a cluster processes, in order.  Fixed split: the one key slice of
// the cluster's grid position.  Balanced split: the rows that meet the
// cluster's tile range [x0, x1) of the concatenated row tiles, computed from
// the lengths as the walk goes (row i of sequence b, whose first tile is
// cum).  Every role walks the same list on its own.
template <bool kSparse>
struct SegWalk {
    int x0, x1;   // balanced: the cluster's tiles
    int b, i;     // balanced: the next row is row i of sequence b; fixed split: b = 0
                  // while the slice is still to come
    int cum;      // balanced: the next row's first tile

    __device__ __forceinline__ bool next(const MlaParams &p, MlaSeg &s) {
        if (!p.balanced) {
            if (b != 0) return false;
            b = 1;
            return fixed_slice<kSparse>(p, s, false);
        }
        const uint32_t cap = uint32_t(p.len_cap);
        while (b < p.batch) {
            int vis, row, seq;
            if constexpr (kSparse) {
                // one query row per sequence, every listed key visible
                seq = row = b++;
                vis = static_cast<int>(min(p.kv_len[seq], cap));
            } else {
                const MlaSeqRows sq = mla_seq_rows(p, b, cap);
                if (i >= sq.nr) {
                    ++b;
                    i = 0;
                    continue;
                }
                seq = b;
                vis = mla_row_vis(p, sq.L, sq.nr, i);
                row = sq.r0 + i;
                ++i;
            }
            const int n = (vis + kBN - 1) / kBN;
            const int first = cum;
            cum += n;
            if (first >= x1) {
                b = p.batch;   // past the range: the walk is over
                break;
            }
            const int tb = max(x0 - first, 0);
            const int te = min(x1 - first, n);
            if (tb >= te) continue;   // an empty row
            s.qrow = row;
            s.b = seq;
            s.start = tb * kBN;
            s.end = min(te * kBN, vis);
            s.ntiles = te - tb;
            s.direct = tb == 0 && te == n;
            s.ws = static_cast<int>(blockIdx.x >> 1) + row;
            return true;
        }
        return false;
    }
    // Row of the run after the one next() returned last, if there may be one
    // in the same sequence (balanced split).
    __device__ __forceinline__ int peek_row(const MlaParams &p) const {
        if (b >= p.batch || cum >= x1) return -1;
        if constexpr (kSparse) return b;
        const MlaSeqRows sq = mla_seq_rows(p, b, uint32_t(p.len_cap));
        return i < sq.nr ? sq.r0 + i : -1;
    }
};

// Balanced split: this cluster's range and the walk's first row, from the
// lengths, by one warp (all 32 lanes call; every lane gets the result).
// Lane l sums the tiles and weighted tiles of sequences [l m, (l+1) m); a
// warp scan gives every lane its first position; the lane whose weighted
// positions hold the cluster's first (the next cluster's first) position
// finds the row and the real tile.  With mark_empty, the reduce's entry of
// every row without tiles is written ({0, 0}: an empty row).
struct MlaRange {
    int x0, x1;      // the cluster's real tiles
    int b, i, cum;   // its first row (row i of sequence b) and that row's first tile
    int w;           // that row's first weighted position
    int tw, c;       // weighted positions in all, clusters taking part
};
__device__ __forceinline__ int4 mla_locate(const MlaParams &p, uint32_t cap, int b_lo, int b_hi,
                                           long long cum, long long W, long long y) {
    // {first tile, sequence b, row i in it, first weighted position} of the
    // row holding weighted position y, searched in sequences [b_lo, b_hi)
    // whose first row starts at tile cum and weighted position W.
    for (int b = b_lo; b < b_hi; ++b) {
        const MlaSeqRows q = mla_seq_rows(p, b, cap);
        for (int i = 0; i < q.nr; ++i) {
            const int n = (mla_row_vis(p, q.L, q.nr, i) + kBN - 1) / kBN;
            if (n > 0 && y < W + kRunCost + n)
                return make_int4(static_cast<int>(cum), b, i,
                                 static_cast<int>(W));
            cum += n;
            W += n > 0 ? n + kRunCost : 0;
        }
    }
    return make_int4(0, b_hi, 0, 0);
}
__device__ __forceinline__ MlaRange mla_balanced_range(const MlaParams &p, int lane, bool mark_empty) {
    const uint32_t cap = uint32_t(p.len_cap);
    const int per_lane = (p.batch + 31) / 32;
    const int b_lo = min(lane * per_lane, p.batch), b_hi = min(b_lo + per_lane, p.batch);
    long long tl = 0, wl = 0;
    for (int b = b_lo; b < b_hi; ++b) {
        if (mark_empty && p.kv_len[b] > cap) atomicOr(p.err, kErrBadLength);
        const MlaSeqRows q = mla_seq_rows(p, b, cap);
        for (int i = 0; i < q.nr; ++i) {
            const int n = (mla_row_vis(p, q.L, q.nr, i) + kBN - 1) / kBN;
            tl += n;
            wl += n > 0 ? n + kRunCost : 0;
            if (mark_empty && n == 0) p.plan_slots[q.r0 + i] = make_int2(0, 0);
        }
    }
    long long ti = tl, wi = wl;   // inclusive scans
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long u = __shfl_up_sync(0xffffffffu, ti, o);
        const long long v = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) {
            ti += u;
            wi += v;
        }
    }
    const long long T = __shfl_sync(0xffffffffu, ti, 31), Tw = __shfl_sync(0xffffffffu, wi, 31);
    const long long C = min(static_cast<long long>(p.num_clusters), T);
    const long long c = blockIdx.x >> 1;
    MlaRange r;
    r.x0 = r.x1 = r.cum = r.i = r.w = 0;
    r.b = p.batch;   // no rows
    r.tw = static_cast<int>(Tw);
    r.c = static_cast<int>(C);
    if (c < C) {
        for (int k = 0; k < 2; ++k) {
            if (k == 1 && c + 1 == C) {
                r.x1 = static_cast<int>(T);
                break;
            }
            const long long y = (c + k) * Tw / C;
            const bool mine = wi - wl <= y && y < wi;
            const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
            int4 e = make_int4(0, 0, 0, 0);
            int x = 0;
            if (lane == src) {
                e = mla_locate(p, cap, b_lo, b_hi, ti - tl, wi - wl, y);
                const MlaSeqRows q = mla_seq_rows(p, e.y, cap);
                const int n = (mla_row_vis(p, q.L, q.nr, e.z) + kBN - 1) / kBN;
                x = e.x + static_cast<int>(min(max(y - e.w - kRunCost, 0LL),
                                               static_cast<long long>(n)));
            }
            x = __shfl_sync(0xffffffffu, x, src);
            if (k == 0) {
                r.x0 = x;
                r.cum = __shfl_sync(0xffffffffu, e.x, src);
                r.b = __shfl_sync(0xffffffffu, e.y, src);
                r.i = __shfl_sync(0xffffffffu, e.z, src);
                r.w = __shfl_sync(0xffffffffu, e.w, src);
            } else {
                r.x1 = x;
            }
        }
    }
    return r;
}

// Balanced split, the reduce's table: for every row whose first tile this
// cluster holds, {first slot, partials}.  Cluster c writes row r's partial
// to slot c + r, and the cluster holding weighted position y is
// ((y + 1) C - 1) / T_w, so a row's partials are consecutive slots.
__device__ __forceinline__ void mla_write_slots(const MlaParams &p, const MlaRange &g) {
    const uint32_t cap = uint32_t(p.len_cap);
    const int c = static_cast<int>(blockIdx.x >> 1);
    long long cum = g.cum, W = g.w;
    int i = g.i;
    for (int b = g.b; b < p.batch; ++b, i = 0) {
        const MlaSeqRows q = mla_seq_rows(p, b, cap);
        for (; i < q.nr; ++i) {
            if (cum >= g.x1) return;
            const int n = (mla_row_vis(p, q.L, q.nr, i) + kBN - 1) / kBN;
            if (n > 0 && cum >= g.x0) {
                const long long wl = W + kRunCost + n - 1;   // weighted last tile
                const int cl = static_cast<int>(((wl + 1) * g.c - 1) / g.tw);
                p.plan_slots[q.r0 + i] = make_int2(c + q.r0 + i, cl - c + 1);
            }
            cum += n;
            W += n > 0 ? n + kRunCost : 0;
        }
    }
}

template <bool kSparse>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Layout<kSparse>::kThreads, 1)
mla_decode_kernel(const __grid_constant__ MlaParams p) {
    using Roles = Layout<kSparse>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Smem::bars);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Smem::bars + kNumBars * 8);

    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int col0 = int(rank) * (kMlaDimV / 2);                 // this CTA's V channels
    const int rope_col = kMlaDimV + int(rank) * kMlaRopeBoxCh;  // and rope channels

    SegWalk<kSparse> walk;
    walk.x0 = walk.x1 = walk.cum = walk.i = walk.b = 0;
    if (!p.balanced) {
        MlaSeg s0;
        if (!fixed_slice<kSparse>(p, s0, threadIdx.x == 0 && rank == 0))
            return;   // uniform over the cluster
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&bar[kKvFull + i], Roles::kProducers);
            mbar_init(&bar[kKvEmpty + i], 1);
        }
        mbar_init(&bar[kQFull], 8);   // the eight softmax warps, after Q is in TMEM
        mbar_init(&bar[kSFull], 1);
        mbar_init(&bar[kSFree], 8);
        mbar_init(&bar[kPFull], 8);
        mbar_init(&bar[kODone], 1);
        for (int i = 0; i < kXSlots; ++i) {
            mbar_init(&bar[kXFull + i], 1);
            mbar_init(&bar[kXPeerFree + i], 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar[kXoReady + i], 4);
            mbar_init(&bar[kXoFree + i], 1);
        }
        fence_mbar_init();
    }
    if (warp == Roles::kMmaWarp) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    MlaRange *range = reinterpret_cast<MlaRange *>(smem + Smem::range);
    if (p.balanced && warp == 0) {
        // The cluster's range, from the lengths (both CTAs find the same);
        // the first CTA also marks the rows without tiles for the reduce.
        const MlaRange r = mla_balanced_range(p, lane, blockIdx.x == 0);
        if (lane == 0) *range = r;
    }
    tc::fence_before_sync();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any remote arrive
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    if (p.balanced) {
        walk.x0 = range->x0;
        walk.x1 = range->x1;
        walk.cum = range->cum;
        walk.b = range->b;
        walk.i = range->i;
    }

    const int pidx = Roles::producer(warp);
    if (warp >= 8) {
        if constexpr (kSparse) setmaxnreg_dec<104>();   // same instruction for both warpgroups
        if (pidx >= 0) {
            // ------------------------------------------------------------ producer
            // Tile i of the CTA's whole run list goes to stage i % kStages, so
            // the ring runs on across the runs' boundaries.
            SegWalk<kSparse> w = walk;
            MlaSeg sg;
            int issued = 0;   // tiles of every run so far
            if (lane == 0) {
                prefetch_tensormap(&p.kv_map);
                prefetch_tensormap(&p.rope_map);
            }
            if constexpr (kSparse) {
                // Sparse top-k: key j of the sequence is cache row indices[b][j]
                // (rows at a uniform stride).  Rows are scattered, so a tile
                // arrives as gather4 copies (four rows x one box, swizzled like
                // a tiled load: 512 bytes for a 64-channel box, 256 for the
                // 32 rope channels): 16 row groups x 5 boxes per tile, spread
                // over the six producer warps, one copy per lane (warp w,
                // lane l takes copy w + 6 l).  Each warp
                // posts the bytes of its own copies on the stage barrier, so
                // the stage is full when all six warps' copies have landed and
                // the producers run up to kStages tiles ahead, as for a dense
                // cache.  A key past the run end, or an index outside the
                // cache (reported), reads row 0 in its place; the softmax
                // masks the former and the error word reports the latter.
                // The indices of tile i + 1 are loaded while tile i waits for
                // its stage.
                constexpr int kCopies = kVBoxes + 1;      // boxes per row group
                const int nq = 16 * kCopies;
                const int q = pidx + Roles::kProducers * lane;
                const bool mine = q < nq;
                const int g = mine ? q / kCopies : 0;        // rows 4g .. 4g + 3 of the tile
                const int cb = mine ? q - g * kCopies : 0;   // box; kVBoxes = the rope box
                bool run = true;
                while (run && w.next(p, sg)) {
                    const int32_t *idx = p.indices + size_t(sg.b) * size_t(p.indices_stride);
                    auto load4 = [&](int tile, int (&r)[4]) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int t = sg.start + tile * kBN + 4 * g + u;
                            r[u] = (mine && tile < sg.ntiles && t < sg.end) ? __ldg(idx + t) : 0;
                        }
                    };
                    int cur[4], nxt[4];
                    load4(0, cur);
                    for (int i = 0; i < sg.ntiles; ++i) {
                        load4(i + 1, nxt);
                        const int gi = issued;
                        const int s = gi % kStages;
                        bool ok = true;
                        if (lane == 0 && gi >= kStages)
                            ok = mbar_wait(&bar[kKvEmpty + s], ((gi / kStages) - 1) & 1, p.err);
                        if (!__shfl_sync(0xffffffffu, ok, 0)) {
                            run = false;
                            break;
                        }
                        const int t_g = sg.start + i * kBN + 4 * g;
                        const bool live = mine && t_g < sg.end;
                        bool bad = false;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if (cur[u] < 0 || static_cast<long long>(cur[u]) >= p.num_rows) {
                                bad = true;
                                cur[u] = 0;
                            }
                        }
                        if (live && bad) atomicOr(p.err, kErrBadPage);
                        const uint32_t bytes =
                            __reduce_add_sync(0xffffffffu, live ? (cb < kVBoxes ? 512u : 256u) : 0u);
                        if (lane == 0) mbar_arrive_expect_tx(&bar[kKvFull + s], bytes);
                        __syncwarp();   // the expected bytes are posted before any copy lands
                        uint8_t *st = smem + Smem::kv + s * kStageBytes;
                        if (live && cb < kVBoxes)
                            tma_gather4(st + cb * kKBoxBytes + g * 512, &p.kv_map,
                                        &bar[kKvFull + s], col0 + cb * 64, cur[0], cur[1], cur[2],
                                        cur[3]);
                        else if (live)
                            tma_gather4(st + kVBoxes * kKBoxBytes + g * 256, &p.rope_map,
                                        &bar[kKvFull + s], rope_col, cur[0], cur[1], cur[2],
                                        cur[3]);
                        issued = gi + 1;
#pragma unroll
                        for (int u = 0; u < 4; ++u) cur[u] = nxt[u];
                    }
                }
            } else {
                const int box_rows = p.box_rows;
                const int boxes_per_tile = kBN / box_rows;   // 1..8
                bool aborted = false;
                while (!aborted && w.next(p, sg)) {
                    const int G = issued;
                    for (int base = 0; base < sg.ntiles && !aborted; base += 32) {
                        // lane i resolves the pages of tile base + i (up to 8 row boxes)
                        int pg[8], sl[8];
#pragma unroll
                        for (int r = 0; r < 8; ++r) { pg[r] = -1; sl[r] = 0; }
                        const int my_tile = base + lane;
                        if (my_tile < sg.ntiles) {
                            const int t0 = sg.start + my_tile * kBN;
#pragma unroll
                            for (int r = 0; r < 8; ++r) {
                                const int t = t0 + r * box_rows;
                                if (r >= boxes_per_tile || t >= sg.end) continue;
                                if (p.page_table) {
                                    const int pi = t / p.page_size;
                                    int e = pi < p.max_pages
                                                ? p.page_table[size_t(sg.b) * p.max_pages + pi] : -1;
                                    if (e < 0 || e >= p.num_pages) {
                                        atomicOr(p.err, kErrBadPage);
                                        e = -1;
                                    }
                                    pg[r] = e;
                                    sl[r] = t % p.page_size;
                                } else {
                                    pg[r] = sg.b;
                                    sl[r] = t;
                                }
                            }
                        }
                        const int lim = min(base + 32, sg.ntiles);
                        for (int i = base; i < lim; ++i) {
                            int pages[8], slots[8];
#pragma unroll
                            for (int r = 0; r < 8; ++r) {
                                pages[r] = __shfl_sync(0xffffffffu, pg[r], i - base);
                                slots[r] = __shfl_sync(0xffffffffu, sl[r], i - base);
                            }
                            const int gi = G + i;
                            if (lane == 0) {
                                const int s = gi % kStages;
                                if (gi >= kStages &&
                                    !mbar_wait(&bar[kKvEmpty + s], ((gi / kStages) - 1) & 1, p.err)) {
                                    aborted = true;
                                } else {
                                    uint32_t nrow = 0;
#pragma unroll
                                    for (int r = 0; r < 8; ++r) nrow += pages[r] >= 0 ? 1u : 0u;
                                    mbar_arrive_expect_tx(
                                        &bar[kKvFull + s],
                                        nrow * uint32_t(box_rows) * uint32_t(kVBoxes * 128 + 2 * kMlaRopeBoxCh));
                                    uint8_t *st = smem + Smem::kv + s * kStageBytes;
#pragma unroll
                                    for (int r = 0; r < 8; ++r) {
                                        if (pages[r] < 0) continue;
#pragma unroll
                                        for (int cb = 0; cb < kVBoxes; ++cb)
                                            tma_load_4d(st + cb * kKBoxBytes + r * box_rows * 128,
                                                        &p.kv_map, &bar[kKvFull + s], col0 + cb * 64,
                                                        slots[r], 0, pages[r]);
                                        tma_load_4d(st + kVBoxes * kKBoxBytes + r * box_rows * 2 * kMlaRopeBoxCh,
                                                    &p.rope_map, &bar[kKvFull + s], rope_col, slots[r],
                                                    0, pages[r]);
                                    }
                                }
                            }
                            aborted = __shfl_sync(0xffffffffu, aborted, 0);
                            if (aborted) break;
                            issued = gi + 1;
                        }
                    }
                }
            }
            // every copy this warp issued must land before the CTA may leave
            if (lane == 0) {
                for (int i = max(0, issued - kStages); i < issued; ++i)
                    mbar_wait(&bar[kKvFull + i % kStages], (i / kStages) & 1, p.err);
            }
        } else if (warp == Roles::kMmaWarp) {
            // ------------------------------------------------------------ MMA issue
            if (lane == 0) {
                constexpr uint32_t idesc_s = tc::idesc_bf16_f32(128, kBN, 0, 0);
                constexpr uint32_t idesc_o = tc::idesc_bf16_f32(128, 256, 0, 1);
                const uint32_t kv_base = smem_addr(smem + Smem::kv);
                // S(g) = Q K^T over this CTA's channels for tile g of the run
                // list.  Descriptors advance by byte offset / 16 in their start
                // field; the loops are unrolled so issue is not bound by
                // descriptor arithmetic.
                auto issue_s = [&](int g) -> bool {
                    const int s = g % kStages;
                    if (!mbar_wait(&bar[kKvFull + s], (g / kStages) & 1, p.err)) return false;
                    if (g >= 1 && !mbar_wait(&bar[kSFree], (g - 1) & 1, p.err)) return false;
                    tc::fence_after_sync();
                    const uint64_t b0 = tc::smem_desc_sw128(kv_base + s * kStageBytes, 16, 1024);
                    const uint64_t br = tc::smem_desc_sw64(
                        kv_base + s * kStageBytes + kVBoxes * kKBoxBytes, 16, 512);
#pragma unroll
                    for (int ks = 0; ks < 4 * kVBoxes; ++ks)
                        // A = Q from TMEM: 16 channels = 8 columns of bf16 pairs per step
                        tc::mma_bf16_tmem_a(tmem + kTmemS, tmem + kTmemQ + ks * 8,
                                            b0 + uint64_t(((ks >> 2) * kKBoxBytes + (ks & 3) * 32) >> 4),
                                            idesc_s, ks > 0);
#pragma unroll
                    for (int ks = 4 * kVBoxes; ks < kScoreSteps; ++ks)
                        // the rope box: 64-byte rows, two steps of 32 bytes
                        tc::mma_bf16_tmem_a(tmem + kTmemS, tmem + kTmemQ + ks * 8,
                                            br + uint64_t(((ks - 4 * kVBoxes) * 32) >> 4), idesc_s,
                                            true);
                    tc::mma_commit(&bar[kSFull]);
                    return true;
                };
                SegWalk<kSparse> w = walk;
                MlaSeg sg;
                int G = 0, runs = 0;
                bool ok = true;
                while (ok && w.next(p, sg)) {
                    const int n = sg.ntiles;
                    if (n == 0) continue;
                    // Q of this run is in TMEM (the softmax warps finished the last run)
                    ok = mbar_wait(&bar[kQFull], runs & 1, p.err);
                    ++runs;
                    if (ok) ok = issue_s(G);
                    if (ok && n > 1) ok = issue_s(G + 1);
                    for (int t = 0; ok && t < n; ++t) {
                        const int g = G + t;
                        if (t + 2 < n && !(ok = issue_s(g + 2))) break;
                        ok = mbar_wait(&bar[kPFull], g & 1, p.err);
                        if (!ok) break;
                        tc::fence_after_sync();
                        const uint64_t v0 = tc::smem_desc_sw128(
                            kv_base + (g % kStages) * kStageBytes, kVLbo, kVSbo);
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            // A = P from TMEM: 16 keys = 8 columns of bf16 pairs per step
                            tc::mma_bf16_tmem_a(tmem + kTmemO, tmem + kTmemP + kk * 8,
                                                v0 + uint64_t((kk * 16 * 128) >> 4), idesc_o,
                                                t > 0 || kk > 0);
                        tc::mma_commit(&bar[kODone]);
                        tc::mma_commit(&bar[kKvEmpty + (g % kStages)]);
                    }
                    G += n;
                }
            }
        } else if (warp == Roles::kXchgWarp) {
            // ------------------------------------------------------------ exchange
            if (lane == 0) {
                const uint32_t dst = mapa_shared(smem_addr(smem + Smem::x_in), peer);
                const uint32_t dst_bar = mapa_shared(smem_addr(&bar[kXFull]), peer);
                const uint32_t src = smem_addr(smem + Smem::x_out);
                // The two key halves go one after the other, so one half is
                // staged while the other is on the wire; half i = 2 g + hf
                // goes to the peer's slot i % 3 once the peer has read that
                // slot's previous half, i - 3.
                SegWalk<kSparse> w = walk;
                MlaSeg sg;
                int G = 0;
                bool run = true;
                while (run && w.next(p, sg)) {
                    for (int t = 0; run && t < sg.ntiles; ++t) {
                        const int g = G + t;
                        for (int hf = 0; hf < 2; ++hf) {
                            const int i = 2 * g + hf, slot = i % kXSlots, use = i / kXSlots;
                            if (!mbar_wait(&bar[kXoReady + hf], g & 1, p.err) ||
                                (use >= 1 && !mbar_wait_cluster(&bar[kXPeerFree + slot],
                                                                (use - 1) & 1, p.err))) {
                                run = false;
                                break;
                            }
                            bulk_copy_to_peer(dst + slot * kXHalfBytes, src + hf * kXHalfBytes,
                                              kXHalfBytes, dst_bar + 8u * slot);
                            bulk_wait_read();
                            mbar_arrive(&bar[kXoFree + hf]);
                        }
                    }
                    G += sg.ntiles;
                }
            }
        }
    } else {
        if constexpr (kSparse) setmaxnreg_inc<152>();
        // ------------------------------------------------------------ softmax
        const int h = (warp & 3) * 32 + lane;    // head row == TMEM lane
        const int half = warp >> 2;              // keys [32 half, 32 half + 32)
        const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
        uint8_t *x_in = smem + Smem::x_in;
        uint8_t *x_out = smem + Smem::x_out;
        // This warp's 4 KB of x_out: rows h of its key half, the rows it
        // stages for the exchange; also its transpose buffer for the Q load
        // and the epilogue stores (row r, 16-byte chunk k at xw_off(r, k)).
        uint8_t *xw = x_out + x_half_off(half, (warp & 3) * 32, 0);
        float *red = reinterpret_cast<float *>(smem + Smem::red);
        const uint32_t peer_xfree = mapa_shared(smem_addr(&bar[kXPeerFree]), peer);
        const uint32_t s_col = kTmemS + 32u * half;
        SegWalk<kSparse> w = walk;
        MlaSeg sg;
        bool ok = true;   // no wait of this warp has failed
        int G = 0;        // tiles of the runs before this one
        while (w.next(p, sg)) {
            const int ntiles = sg.ntiles;
            const int start = sg.start, end = sg.end;
            const int next_row = p.balanced ? w.peek_row(p) : -1;
            if (next_row >= 0) {
                // The next run is likely that row: bring its Q lines of this
                // CTA into L2 now, so the refill after this run reads them
                // from there.
                const uint16_t *qr = p.q + (size_t(next_row) * kMlaHeads + h) * kMlaDimQK;
                const uint8_t *qn = reinterpret_cast<const uint8_t *>(qr + col0);
                for (int cb = half; cb < kVBoxes; cb += 2)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(qn + cb * 128));
                if (half == 1) asm volatile("prefetch.global.L2 [%0];" ::"l"(qr + rope_col));
            }
            float m_ref = -INFINITY;
            float l = 0.f, l_r = 0.f;   // this half's share of the row sums
            bool live = ok && ntiles > 0;
            float s_own[32];
            if (live) {
                // This CTA's Q channels of head row h into TMEM lane h: 64
                // channels (32 columns of bf16 pairs) per store, boxes split
                // over the halves, then the 32 rope channels (16 columns).
                // The last run's MMAs have all finished.  The warp reads its
                // 32 rows a 128-byte line per 8 lanes into its slice of x_out
                // (free: the last copy has read it, waited for in the last
                // run's epilogue) and each lane takes its row back out.
                const uint8_t *qw = reinterpret_cast<const uint8_t *>(
                    p.q + (size_t(sg.qrow) * kMlaHeads + (warp & 3) * 32) * kMlaDimQK);
                // Every line the warp needs requested up front (lane = row:
                // its two boxes and, for half 1, the rope channels), so the
                // boxes' loads below overlap their latencies.
                {
                    const uint8_t *mine = qw + size_t(lane) * kMlaDimQK * 2;
                    asm volatile("prefetch.global.L1 [%0];" ::"l"(mine + col0 * 2 + half * 128));
                    asm volatile("prefetch.global.L1 [%0];" ::"l"(mine + col0 * 2 + (half + 2) * 128));
                    if (half == 1) asm volatile("prefetch.global.L1 [%0];" ::"l"(mine + rope_col * 2));
                }
                for (int cb = half; cb < kVBoxes; cb += 2) {
                    uint4 ld[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = 4 * i + (lane >> 3);
                        ld[i] = *reinterpret_cast<const uint4 *>(
                            qw + size_t(r) * kMlaDimQK * 2 + (col0 + cb * 64) * 2 + (lane & 7) * 16);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<uint4 *>(xw + xw_off(4 * i + (lane >> 3), lane & 7)) = ld[i];
                    __syncwarp();
                    float v[32];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint4 wq = *reinterpret_cast<const uint4 *>(xw + xw_off(lane, k));
                        v[4 * k] = __uint_as_float(wq.x);
                        v[4 * k + 1] = __uint_as_float(wq.y);
                        v[4 * k + 2] = __uint_as_float(wq.z);
                        v[4 * k + 3] = __uint_as_float(wq.w);
                    }
                    __syncwarp();
                    tc::tmem_st32(tmem + lane_base + kTmemQ + cb * 32, v);
                }
                if (half == 1) {
                    uint4 lr[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = 8 * i + (lane >> 2);
                        lr[i] = *reinterpret_cast<const uint4 *>(
                            qw + size_t(r) * kMlaDimQK * 2 + rope_col * 2 + (lane & 3) * 16);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = 8 * i + (lane >> 2);
                        *reinterpret_cast<uint4 *>(xw + xw_off(r, lane & 3)) = lr[i];
                    }
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const uint4 a = *reinterpret_cast<const uint4 *>(xw + xw_off(lane, 2 * k));
                        const uint4 b = *reinterpret_cast<const uint4 *>(xw + xw_off(lane, 2 * k + 1));
                        const float v[8] = {__uint_as_float(a.x), __uint_as_float(a.y),
                                            __uint_as_float(a.z), __uint_as_float(a.w),
                                            __uint_as_float(b.x), __uint_as_float(b.y),
                                            __uint_as_float(b.z), __uint_as_float(b.w)};
                        tc::tmem_st_n<8>(tmem + lane_base + kTmemQ + 4 * kVBoxes * 8 + 8 * k, v);
                    }
                    __syncwarp();
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[kQFull]);

                // The run's first partial: read this half and stage it for the
                // copy once the copy of the last run's final tile has read x_out.
                live = __all_sync(0xffffffffu, mbar_wait(&bar[kSFull], G & 1, p.err));
                if (live) {
                    tc::fence_after_sync();
                    tc::tmem_ld32(tmem + lane_base + s_col, s_own);
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar[kSFree]);
                    if (G >= 1)
                        live = __all_sync(0xffffffffu,
                                          mbar_wait(&bar[kXoFree + half], (G - 1) & 1, p.err));
                }
                if (live) {
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<float4 *>(x_out + x_half_off(half, h, c)) =
                            make_float4(s_own[4 * c], s_own[4 * c + 1], s_own[4 * c + 2],
                                        s_own[4 * c + 3]);
                    tc::fence_async_smem();   // generic writes -> the bulk copy engine
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar[kXoReady + half]);
                }
            }
            // The loop never breaks: every softmax warp reaches the named
            // barriers of every tile; after a failed wait the rest is skipped.
            for (int t = 0; t < ntiles; ++t) {
                const int g = G + t;   // tile of the CTA's run list
                const int t0 = start + t * kBN;
                const int nvalid = min(kBN, end - t0) - 32 * half;   // this half's valid keys
                const int xi = 2 * g + half;             // this half's receive slot and use
                const int xslot = xi % kXSlots;
                if (live && h == 0) mbar_arrive_expect_tx(&bar[kXFull + xslot], kXHalfBytes);

                // ---- one tile ahead: partial S(g+1) out of TMEM, staged for the copy
                float s_next[32];
                const bool more = t + 1 < ntiles;
                if (live && more) {
                    live = __all_sync(0xffffffffu, mbar_wait(&bar[kSFull], (g + 1) & 1, p.err));
                    if (live) {
                        tc::fence_after_sync();
                        tc::tmem_ld32(tmem + lane_base + s_col, s_next);
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bar[kSFree]);
                        // copy(g) has read x_out
                        live = __all_sync(0xffffffffu,
                                          mbar_wait(&bar[kXoFree + half], g & 1, p.err));
                    }
                    if (live) {
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<float4 *>(x_out + x_half_off(half, h, c)) =
                                make_float4(s_next[4 * c], s_next[4 * c + 1], s_next[4 * c + 2],
                                            s_next[4 * c + 3]);
                        tc::fence_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bar[kXoReady + half]);
                    }
                }

                // ---- full S(g) = own partial + the peer's ------------------------
                if (live)
                    live = __all_sync(0xffffffffu, mbar_wait_cluster(&bar[kXFull + xslot],
                                                                     (xi / kXSlots) & 1, p.err));
                float mloc = -INFINITY;
                if (live) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float4 o =
                            *reinterpret_cast<const float4 *>(x_in + x_half_off(xslot, h, c));
                        const float2 a = __fadd2_rn(make_float2(s_own[4 * c], s_own[4 * c + 1]),
                                                    make_float2(o.x, o.y));
                        const float2 b = __fadd2_rn(make_float2(s_own[4 * c + 2], s_own[4 * c + 3]),
                                                    make_float2(o.z, o.w));
                        s_own[4 * c] = a.x;
                        s_own[4 * c + 1] = a.y;
                        s_own[4 * c + 2] = b.x;
                        s_own[4 * c + 3] = b.y;
                    }
                    __syncwarp();   // the warp's reads of x_in happen before the release
                    // The values read from x_in are already consumed (added into
                    // s_own) when the arrive issues, so a relaxed arrive suffices.
                    if (lane == 0)
                        asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];"
                                     ::"r"(peer_xfree + 8u * uint32_t(xslot)) : "memory");
                    if (p.qk_scale_log2 > 0.f) {
                        // Raw scores stay in s_own (keys past the run end -inf);
                        // the scale goes into the exponent's FMA and, being
                        // positive, commutes with the max (a tree of 3-input maxima).
                        if (nvalid < 32) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) s_own[j] = j < nvalid ? s_own[j] : -INFINITY;
                        }
                        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                        for (int j = 0; j < 32; j += 2)
                            m4[(j >> 1) & 3] = fmax3(m4[(j >> 1) & 3], s_own[j], s_own[j + 1]);
                        mloc = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.qk_scale_log2;
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            s_own[j] = j < nvalid ? s_own[j] * p.qk_scale_log2 : -INFINITY;
                            mloc = fmaxf(mloc, s_own[j]);
                        }
                    }
                }
                // ---- row max over both halves --------------------------------
                // the two warps of this row quarter (same SM sub-partition)
                named_sync(kBarPair + (warp & 3), 64);   // the last reads of red are done
                red[half * 128 + h] = mloc;
                named_sync(kBarPair + (warp & 3), 64);
                const float mt = fmaxf(mloc, red[(half ^ 1) * 128 + h]);

                if (live) {
                    // ---- online softmax in base 2, lazy max ----------------------
                    const bool raise = mt > m_ref + kRescaleThreshold;   // always on the first tile
                    float alpha = 1.f;
                    if (raise) {
                        alpha = fast_exp2(m_ref - mt);                  // 0 when m_ref = -inf
                        m_ref = mt;
                    }
                    // Two row sums: of the fp32 weights (for lse) and of the bf16-
                    // rounded weights the MMA multiplies V by (to normalise O).
                    // Key pairs go through the packed fp32x2 FMA (score times the
                    // folded scale minus m_ref: m_ref is finite here, every tile
                    // having a visible key in its first half) and adds.
                    const float sc_mul = p.qk_scale_log2 > 0.f ? p.qk_scale_log2 : 1.f;
                    const float2 mul2 = make_float2(sc_mul, sc_mul);
                    const float2 neg2 = make_float2(-m_ref, -m_ref);
                    float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    float2 rr[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    float pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float2 e =
                            __ffma2_rn(make_float2(s_own[2 * j], s_own[2 * j + 1]), mul2, neg2);
                        const float p0 = fast_exp2(e.x);
                        const float p1 = fast_exp2(e.y);
                        const uint32_t wp = pack_bf16x2(p0, p1);
                        pk[j] = __uint_as_float(wp);
                        rs[j & 1] = __fadd2_rn(rs[j & 1], make_float2(p0, p1));
                        add_bf16x2_f32(rr[j & 1], wp);
                    }
                    const float rowsum = (rs[0].x + rs[1].x) + (rs[0].y + rs[1].y);
                    const float rowsum_r = (rr[0].x + rr[1].x) + (rr[0].y + rr[1].y);
                    l = l * alpha + rowsum;
                    l_r = l_r * alpha + rowsum_r;

                    // O(g-1) has read P(g-1) and must be finished before O is rescaled.
                    if (t >= 1) {
                        live = __all_sync(0xffffffffu,
                                          mbar_wait(&bar[kODone], (g - 1) & 1, p.err));
                        tc::fence_after_sync();
                        if (live && __any_sync(0xffffffffu, raise)) {
                            // 8 columns at a time: both score arrays are live here
#pragma unroll 1
                            for (int c = 0; c < 128; c += 8) {
                                float v[8];
                                const uint32_t oc = kTmemO + 128u * half + c;
                                tc::tmem_ld_n<8>(tmem + lane_base + oc, v);
#pragma unroll
                                for (int j = 0; j < 8; ++j) v[j] *= alpha;
                                tc::tmem_st_n<8>(tmem + lane_base + oc, v);
                            }
                        }
                    }
                    if (live) {
                        float p8[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) p8[j] = pk[j];
                        tc::tmem_st_n<8>(tmem + lane_base + kTmemP + 16u * half, p8);
#pragma unroll
                        for (int j = 0; j < 8; ++j) p8[j] = pk[8 + j];
                        tc::tmem_st_n<8>(tmem + lane_base + kTmemP + 16u * half + 8, p8);
                        const int nv = min(kBN, end - t0);
                        if (nv < kBN) {
                            // Rows past the run end may hold anything (even NaN):
                            // zero them in the V part of the stage so 0 * V stays 0.
                            uint8_t *st = smem + Smem::kv + (g % kStages) * kStageBytes;
                            const int nz = (kBN - nv) * 4 * 8;   // 16-B chunks in 4 boxes
                            for (int i = threadIdx.x; i < nz; i += kSoftmaxThreads) {
                                const int box = i / ((kBN - nv) * 8);
                                const int rem = i - box * ((kBN - nv) * 8);
                                const int row = nv + rem / 8;
                                const int ch = rem & 7;
                                *reinterpret_cast<uint4 *>(st + box * kKBoxBytes + row * 128 +
                                                           ch * 16) = make_uint4(0u, 0u, 0u, 0u);
                            }
                            tc::fence_async_smem();
                        }
                        tc::tmem_wait_st();
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bar[kPFull]);   // one arrival per softmax warp
                    }
                }
                if (more) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) s_own[j] = s_next[j];
                }
            }

            // ---- run epilogue ---------------------------------------------------
            // Row sums of the two halves (same m_ref), one after the other
            // through the row-max buffer, while the last P.V is in flight.
            named_sync(kBarPair + (warp & 3), 64);
            red[half * 128 + h] = l;
            named_sync(kBarPair + (warp & 3), 64);
            const float l_other = red[(half ^ 1) * 128 + h];
            named_sync(kBarPair + (warp & 3), 64);
            red[half * 128 + h] = l_r;
            named_sync(kBarPair + (warp & 3), 64);
            l_r += red[(half ^ 1) * 128 + h];
            l += l_other;
            if (live) {
                live = __all_sync(0xffffffffu,
                                  mbar_wait(&bar[kODone], (G + ntiles - 1) & 1, p.err));
                tc::fence_after_sync();
            }
            // O was accumulated with the rounded weights: normalise it by their
            // sum (direct), or rescale it to the fp32 sum l kept for the merge.
            float scale_o = 0.f, Mf = -INFINITY, Z = 0.f;
            if (sg.direct) {
                const float t2 = p.sink ? p.sink[h] * kLog2e : -INFINITY;
                Mf = fmaxf(m_ref, t2);
                float so = 0.f, Zr = 0.f;
                if (Mf != -INFINITY) {
                    so = fast_exp2(m_ref - Mf);
                    const float st = fast_exp2(t2 - Mf);
                    Z = l * so + st;
                    Zr = l_r * so + st;
                }
                scale_o = Zr > 0.f ? so / Zr : 0.f;
            } else {
                scale_o = l_r > 0.f ? l / l_r : 0.f;
            }
            const size_t row = size_t(sg.qrow) * kMlaHeads + h;
            const size_t wrow = size_t(sg.ws) * kMlaHeads + h;
            const int ch0 = rank * 256 + half * 128;   // this warp's output channels
            // The rows go out through the warp's slice of x_out, eight lanes
            // a row (whole 128-byte lines), once the copy of the CTA's last
            // staged partial has read it.
            const int g_last = G + ntiles - 1;
            if (ok && g_last >= 0 &&
                !__all_sync(0xffffffffu, mbar_wait(&bar[kXoFree + half], g_last & 1, p.err))) {
                ok = false;   // sticks: the end of the run keeps a failed wait
                live = false;
            }
            const size_t row0 = size_t(sg.direct ? sg.qrow : sg.ws) * kMlaHeads + (warp & 3) * 32;
#pragma unroll 1
            for (int c = 0; c < 128; c += 32) {
                float v[32];
                if (live) {
                    tc::tmem_ld32(tmem + lane_base + kTmemO + 128u * half + c, v);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.f;
                }
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    *reinterpret_cast<float4 *>(xw + xw_off(lane, k)) =
                        make_float4(v[4 * k] * scale_o, v[4 * k + 1] * scale_o,
                                    v[4 * k + 2] * scale_o, v[4 * k + 3] * scale_o);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = 4 * i + (lane >> 3), k = lane & 7;
                    const float4 f = *reinterpret_cast<const float4 *>(xw + xw_off(r, k));
                    const size_t at = (row0 + r) * kMlaDimV + ch0 + c + 4 * k;
                    if (sg.direct)
                        *reinterpret_cast<uint2 *>(p.out + at) =
                            make_uint2(pack_bf16x2(f.x, f.y), pack_bf16x2(f.z, f.w));
                    else
                        *reinterpret_cast<float4 *>(p.ws_o + at) = f;
                }
                __syncwarp();
            }
            if (rank == 0 && half == 0) {
                if (sg.direct) {
                    if (p.lse) p.lse[row] = Z > 0.f ? (Mf + fast_log2(Z)) * kLn2 : -INFINITY;
                } else {
                    p.ws_m[wrow] = m_ref * kLn2;
                    p.ws_l[wrow] = l;
                }
            }
            if (ntiles > 0) ok = live;
            G += ntiles;
        }
        // The reduce's entries of the rows whose first tile this cluster holds.
        if (p.balanced && rank == 0 && warp == 0 && lane == 0) mla_write_slots(p, *range);
        pdl_launch_dependents();
    }

    tc::fence_before_sync();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still touch its smem
    if (warp == Roles::kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool kSparse>
cudaError_t launch_layout(const MlaParams &p, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel<kSparse>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kSmemBytes));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = p.balanced ? dim3(2 * p.num_clusters, 1) : dim3(2 * p.num_partitions, p.num_q_rows);
    cfg.blockDim = dim3(Layout<kSparse>::kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, mla_decode_kernel<kSparse>, p);
}

template <bool kSparse>
int cluster_slots(int num_sms) {
    static int cached = 0;
    if (cached > 0) return cached;
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2 > 0 ? num_sms / 2 : 1));
    cfg.blockDim = dim3(Layout<kSparse>::kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    if (cudaFuncSetAttribute(mla_decode_kernel<kSparse>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmemBytes)) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, mla_decode_kernel<kSparse>, &cfg) != cudaSuccess ||
        n <= 0) {
        (void)cudaGetLastError();
        n = num_sms / 2;
    }
    cached = n < num_sms / 2 ? n : num_sms / 2;
    if (cached < 1) cached = 1;
    return cached;
}

}  // namespace

cudaError_t launch_mla_decode(const MlaParams &p, cudaStream_t stream) {
    return p.sparse ? launch_layout<true>(p, stream) : launch_layout<false>(p, stream);
}


int mla_cluster_slots(int num_sms, bool sparse) {
    return sparse ? cluster_slots<true>(num_sms) : cluster_slots<false>(num_sms);
}

}  // namespace attn
