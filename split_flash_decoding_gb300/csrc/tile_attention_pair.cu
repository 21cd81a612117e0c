// tile_attention_pair.cu -- the tile path with two Q tiles per CTA pair
// (the 2Q configuration: mha_sm100_dispatch, summary, chooses between one
// and two Q tiles by occupancy and prompt length).
//
// A cluster of two CTAs takes two adjacent 128-row Q tiles of one
// (sequence, KV head); CTA r holds tile 2 u + r (its rows are (128 / group)
// tokens x the group's heads, as in the one-tile kernel) and runs the
// softmax of its own rows.  Both tiles share every K/V tile through the
// 5th-generation tensor cores' CTA-pair MMA (tcgen05.mma.cta_group::2, M =
// 256 rows across the pair): the pair's A operand is each CTA's own Q (or
// P), and the B operand is split between the two CTAs' shared memory --
//
//   S = Q K^T:  N = 128 keys;  CTA r holds keys [64 r, 64 r + 64) of the
//               tile, all 128 channels (K-major);
//   O += P V:   N = 128 channels;  CTA r holds channels [64 r, 64 r + 64)
//               of V, all 128 keys (MN-major);
//
// and each CTA's TMEM receives its 128 rows x all N columns.  Every byte of
// a K/V tile is loaded once per pair for 256 query rows, and each SM reads
// half of each MMA's B operand from its own shared memory: half the load
// traffic and 3/4 of the operand reads per row of the one-tile kernel.
//
// The even CTA's MMA thread issues every MMA of the pair and commits to
// both CTAs' barriers (multicast).  It must know that the odd CTA's halves
// have landed: that CTA's MMA warp, idle otherwise, relays its Q, K and V
// arrivals to the even CTA (lane 0: Q and K, lane 1: V), and so, once per
// tile, the completion of its softmax warps' S-free and P-full barriers
// (lanes 2 and 3); the softmax warps themselves only arrive locally.
// The softmax, masks, lazy running max and epilogue are those of the
// one-tile kernel (tile_attention.cu).
//
// Warp roles (352 threads per CTA): 0-7 softmax/epilogue, 8 TMA producer of
// Q and the K half, 9 TMA producer of the V half, 10 TMEM allocation and
// (even CTA) MMA issue, lane 0 the score MMAs and lane 1 the P.V MMAs / (odd
// CTA) arrival relay.
#include <type_traits>

#include "launch.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace attn {
namespace {

constexpr int kD = 128;
constexpr int kBN = kTileKeys;               // keys per tile (128)
constexpr int kStages = 4;
constexpr int kQBoxBytes = 128 * 128;        // 128 rows x 128 B (64 channels)
constexpr int kQBytes = 2 * kQBoxBytes;      // the Q tile: 128 rows x 128 channels
constexpr int kKBoxBytes = 64 * 128;         // 64 keys x 64 channels
constexpr int kHalfBytes = 2 * kKBoxBytes;   // a K half (64 keys x 128 ch) or V half (128 keys x 64 ch)
constexpr int kThreads = 352;
constexpr int kSoftmaxThreads = 256;         // warps 0-7
constexpr int kBarPair = 2;                  // named barriers 2..5: the two warps of a row quarter
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;               // S buffers at 0 and 128
constexpr uint32_t kTmemO = 256;
constexpr uint32_t kTmemP = 384;             // P buffers at 384 and 448 (64 columns each)
constexpr float kRescaleThreshold = 8.0f;

struct Smem {
    static constexpr int q = 0;                                  // 32 KB
    static constexpr int k = q + kQBytes;                        // K halves, 4 x 16 KB
    static constexpr int v = k + kStages * kHalfBytes;           // V halves, 4 x 16 KB
    static constexpr int red = v + kStages * kHalfBytes;
    static constexpr int bars = red + 2 * 128 * 4;               // +1 KB (row maxima)
    static constexpr int total = bars + 384;
};
constexpr size_t kSmemBytes = Smem::total + 1024;

enum Bar {
    kKFull = 0,                   // [kStages] own K half landed
    kKEmpty = kStages,            // [kStages] the pair's S MMA has read the stage (multicast)
    kVFull = 2 * kStages,         // [kStages] own V half landed
    kVEmpty = 3 * kStages,        // [kStages] the pair's P.V MMA has read the stage (multicast)
    kKPeer = 4 * kStages,         // [kStages] even CTA: the odd CTA's K half landed (relay)
    kVPeer = 5 * kStages,         // [kStages] even CTA: the odd CTA's V half landed (relay)
    kQFull = 6 * kStages,
    kQPeer = kQFull + 1,          // even CTA: the odd CTA's Q landed (relay)
    kSFull = kQPeer + 1,          // [2] S of a tile in TMEM (multicast commit)
    kSFree = kSFull + 2,          // [2] S buffer read: in the even CTA its 8 softmax warps + the
                                  // odd CTA's relay (9); in the odd CTA its 8 softmax warps
    kPFull = kSFree + 2,          // [2] P of a tile with this parity in TMEM, V tail cleared:
                                  // counted the same way
    kODone = kPFull + 2,          // [2] the pair's P.V MMA of a tile with this parity finished
                                  // (multicast commit)
    kNumBars = kODone + 2
};

// ---- CTA-pair tcgen05 forms (every tcgen05 instruction of this kernel
// names cta_group::2) -----------------------------------------------------------
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D[tmem] (+)= A[smem] * B[smem] over the pair (A rows and B columns split
// between the CTAs at the same shared-memory offsets).
__device__ __forceinline__ void mma_pair_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc ? 1u : 0u)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem] over the pair.
__device__ __forceinline__ void mma_pair_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                            bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc ? 1u : 0u)
        : "memory");
}
// Arrive on the mbarrier at this offset in both CTAs once every pair MMA
// issued so far by this thread is done.
__device__ __forceinline__ void commit_pair(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;" ::"r"(smem_addr(bar)),
        "h"(uint16_t(3))
        : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
tile_attention_pair_kernel(const __grid_constant__ TileParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Smem::bars);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Smem::bars + kNumBars * 8);

    const uint32_t rank = cluster_ctarank();
    const int G = p.group;
    const int T = kTileRows / G;                 // tokens per tile
    const int pairs = (p.tiles_per_seq + 1) / 2;
    // Longest pairs first: blockIdx.x / 2 counts down the pairs of a sequence.
    const int unit = pairs - 1 - static_cast<int>(blockIdx.x >> 1);
    const int tile = 2 * unit + static_cast<int>(rank);
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int q_off = static_cast<int>(p.q_row_offsets[b]);
    const int n = static_cast<int>(p.q_row_offsets[b + 1]) - q_off;
    const int L = static_cast<int>(p.kv_len[b]);
    if (2 * unit * T >= n) return;               // uniform over the cluster: no rows at all
    const int t0 = tile * T;
    // Keys any row of the pair can see (the odd tile's last row).
    const int pair_end = min(2 * unit * T + 2 * T, n);
    int kmax = p.causal ? L - n + pair_end : L;
    kmax = max(0, min(kmax, L));
    const int ntiles = (kmax + kBN - 1) / kBN;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const uint32_t cnt = (i >= kSFree && i < kPFull + 2) ? (rank == 0 ? 9u : 8u) : 1u;
            mbar_init(&bar[i], cnt);
        }
        fence_mbar_init();
    }
    if (warp == 10) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc::fence_before_sync();
    __syncthreads();
    cluster_sync();   // both CTAs' barriers and TMEM exist before any remote arrive or MMA
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8 || warp == 9) {
        // ------------------------------------------------------------ producers
        // warp 8: Q, then the K half (keys [64 rank, 64 rank + 64) of each
        // tile, both 64-channel boxes); warp 9: the V half (every key of the
        // tile, channels [64 rank, 64 rank + 64)).
        const bool is_k = warp == 8;
        const CUtensorMap *map = is_k ? &p.k_map : &p.v_map;
        uint8_t *ring = smem + (is_k ? Smem::k : Smem::v);
        uint64_t *full = &bar[is_k ? kKFull : kVFull];
        uint64_t *empty = &bar[is_k ? kKEmpty : kVEmpty];
        if (ntiles > 0) {
            if (lane == 0) {
                prefetch_tensormap(map);
                if (is_k) {
                    prefetch_tensormap(&p.q_map);
                    mbar_arrive_expect_tx(&bar[kQFull], kQBytes);
                    for (int cb = 0; cb < 2; ++cb)
                        tma_load_4d(smem + Smem::q + cb * kQBoxBytes, &p.q_map, &bar[kQFull],
                                    cb * 64, 0, kvh, q_off + t0);
                }
            }
            const int box_rows = is_k ? p.box_rows : p.box_rows_v;
            const int span = is_k ? 64 : kBN;              // keys of the tile this CTA loads
            const int key_lo = is_k ? 64 * static_cast<int>(rank) : 0;
            const int nb = span / box_rows;                // boxes per tile
            const int nch = is_k ? 2 : 1;                  // 64-channel boxes per row box
            const int ch0 = is_k ? 0 : 64 * static_cast<int>(rank);
            int cached = -1, my_page = -1, my_slot = 0;
            bool aborted = false;
            int issued = 0;
            for (int i = 0; i < ntiles && !aborted; ++i) {
                const int key0 = i * kBN + key_lo;
                const int live = max(0, min(nb, (L - key0 + box_rows - 1) / box_rows));
                const int s = i % kStages;
                if (lane == 0) {
                    if (i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1, p.err))
                        aborted = true;
                    else
                        mbar_arrive_expect_tx(&full[s], uint32_t(live) * uint32_t(nch) *
                                                            uint32_t(box_rows) * 128u);
                }
                aborted = __shfl_sync(0xffffffffu, aborted, 0);
                if (aborted) break;
                uint8_t *st = ring + s * kHalfBytes;
                for (int r = 0; r < live; ++r) {
                    const int g = i * nb + r;      // box index among this CTA's boxes
                    if ((g >> 5) != cached) {      // warp-uniform refill of 32 lookups
                        cached = g >> 5;
                        const int gi = (cached << 5) + lane;
                        const int t = (gi / nb) * kBN + key_lo + (gi % nb) * box_rows;
                        my_page = -1;
                        my_slot = 0;
                        if (t < L) {
                            if (p.page_table) {
                                const int pidx = t / p.page_size;
                                int e = pidx < p.max_pages
                                            ? p.page_table[size_t(b) * p.max_pages + pidx] : -1;
                                if (e < 0 || e >= p.num_pages) {
                                    atomicOr(p.err, kErrBadPage);
                                    e = -1;
                                }
                                my_page = e;
                                my_slot = t % p.page_size;
                            } else {
                                my_page = b;
                                my_slot = t;
                            }
                        }
                    }
                    const int page = __shfl_sync(0xffffffffu, my_page, g & 31);
                    const int slot = __shfl_sync(0xffffffffu, my_slot, g & 31);
                    if (lane == 0) {
                        if (page < 0) {
                            // a skipped (bad-page) box: retire its expected bytes
                            mbar_complete_tx(&full[s], uint32_t(nch) * uint32_t(box_rows) * 128u);
                        } else {
                            for (int cb = 0; cb < nch; ++cb)
                                tma_load_4d(st + cb * kKBoxBytes + r * box_rows * 128, map,
                                            &full[s], ch0 + cb * 64, slot, kvh, page);
                        }
                    }
                }
                issued = i + 1;
            }
            // every copy this warp issued must land before the CTA may leave
            if (lane == 0) {
                if (is_k) mbar_wait(&bar[kQFull], 0, p.err);
                for (int i = max(0, issued - kStages); i < issued; ++i)
                    mbar_wait(&full[i % kStages], (i / kStages) & 1, p.err);
            }
        }
    } else if (warp == 10) {
        if (rank == 1) {
            // ------------------------------------------------------------ relay
            // The odd CTA tells the even CTA's MMA thread what its own barriers
            // say, one cluster-scope arrive per event (a release across SMs is
            // slow; the softmax warps only arrive locally): lane 0 when its Q
            // and K halves land, lane 1 its V halves, lane 2 when its softmax
            // warps have read an S buffer, lane 3 when they have written P.
            if (lane < 4 && ntiles > 0) {
                bool ok = true;
                if (lane < 2) {
                    const bool is_k = lane == 0;
                    uint64_t *full = &bar[is_k ? kKFull : kVFull];
                    uint64_t *peer = &bar[is_k ? kKPeer : kVPeer];
                    if (is_k) {
                        ok = mbar_wait(&bar[kQFull], 0, p.err);
                        if (ok) mbar_arrive_cluster(mapa_shared(smem_addr(&bar[kQPeer]), 0));
                    }
                    for (int i = 0; ok && i < ntiles; ++i) {
                        ok = mbar_wait(&full[i % kStages], (i / kStages) & 1, p.err);
                        if (ok) mbar_arrive_cluster(mapa_shared(smem_addr(&peer[i % kStages]), 0));
                    }
                } else {
                    // Each local barrier advances once per two tiles (one per
                    // buffer), so phase (t >> 1) of buffer t % 2 is tile t.
                    uint64_t *local = &bar[lane == 2 ? kSFree : kPFull];
                    for (int t = 0; ok && t < ntiles; ++t) {
                        ok = mbar_wait(&local[t & 1], (t >> 1) & 1, p.err);
                        if (ok) mbar_arrive_cluster(mapa_shared(smem_addr(&local[t & 1]), 0));
                    }
                }
            }
        } else if (ntiles > 0 && lane == 0) {
            // ------------------------------------------------------------ MMA issue
            // Two issuing threads of the even CTA, each committing only its own
            // MMAs (to both CTAs): lane 0 the score MMAs, lane 1 the P.V MMAs,
            // so a score MMA never waits behind a P.V that waits for the
            // softmax of either CTA.  M = 256 over the pair; each instruction
            // covers 16 of K.
            constexpr uint32_t idesc_s = tc::idesc_bf16_f32(256, kBN, 0, 0);
            const uint32_t q_base = smem_addr(smem + Smem::q);
            const uint32_t k_base = smem_addr(smem + Smem::k);
            bool ok = mbar_wait(&bar[kQFull], 0, p.err);
            if (ok) ok = mbar_wait_cluster(&bar[kQPeer], 0, p.err);
            for (int t = 0; ok && t < ntiles; ++t) {
                const int s = t % kStages;
                const int sb = t & 1;
                ok = mbar_wait(&bar[kKFull + s], (t / kStages) & 1, p.err);
                if (ok) ok = mbar_wait_cluster(&bar[kKPeer + s], (t / kStages) & 1, p.err);
                if (ok && t >= 2)
                    ok = mbar_wait_cluster(&bar[kSFree + sb], ((t >> 1) - 1) & 1, p.err);
                if (!ok) break;
                tc::fence_after_sync();
                // S = Q K^T: A = this CTA's Q (two 128-row boxes of 64
                // channels), B = the K halves (two 64-key boxes of 64
                // channels); descriptors advance by byte offset / 16.
                const uint64_t qd = tc::smem_desc_sw128(q_base, 16, 1024);
                const uint64_t kd = tc::smem_desc_sw128(k_base + s * kHalfBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint64_t qo = uint64_t(((kk >> 2) * kQBoxBytes + (kk & 3) * 32) >> 4);
                    const uint64_t ko = uint64_t(((kk >> 2) * kKBoxBytes + (kk & 3) * 32) >> 4);
                    mma_pair_ss(tmem + kTmemS + sb * kBN, qd + qo, kd + ko, idesc_s, kk > 0);
                }
                commit_pair(&bar[kSFull + sb]);
                commit_pair(&bar[kKEmpty + s]);
            }
        } else if (ntiles > 0 && lane == 1) {
            constexpr uint32_t idesc_o = tc::idesc_bf16_f32(256, kD, 0, 1);
            const uint32_t v_base = smem_addr(smem + Smem::v);
            bool ok = true;
            for (int t = 0; ok && t < ntiles; ++t) {
                const int s = t % kStages;
                ok = mbar_wait_cluster(&bar[kPFull + (t & 1)], (t >> 1) & 1, p.err);
                if (ok) ok = mbar_wait(&bar[kVFull + s], (t / kStages) & 1, p.err);
                if (ok) ok = mbar_wait_cluster(&bar[kVPeer + s], (t / kStages) & 1, p.err);
                if (!ok) break;
                tc::fence_after_sync();
                // O += P V: A = P buffer t % 2 from TMEM (16 keys = 8
                // columns of bf16 pairs per step), B = the V halves
                // (MN-major, 8-key groups 1 KB apart).
                const uint64_t vd = tc::smem_desc_sw128(v_base + s * kHalfBytes, 16, 1024);
                const uint32_t pb = kTmemP + 64u * uint32_t(t & 1);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_pair_ts(tmem + kTmemO, tmem + pb + kk * 8,
                                vd + uint64_t((kk * 16 * 128) >> 4), idesc_o, t > 0 || kk > 0);
                commit_pair(&bar[kODone + (t & 1)]);
                commit_pair(&bar[kVEmpty + s]);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax
        // As in the one-tile kernel, for this CTA's rows; S-free and P-full
        // arrivals go to the even CTA, whose MMA thread issues for the pair.
        const int r = (warp & 3) * 32 + lane;    // MMA row == TMEM lane
        const int half = warp >> 2;              // keys [64 half, 64 half + 64) of a tile
        const int tok = t0 + r / G;              // token index inside the sequence
        const bool row_valid = tok < n;
        const int lim = p.causal ? min(L, L - n + tok + 1) : L;   // keys [0, lim)
        const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
        float *red = reinterpret_cast<float *>(smem + Smem::red);
        float m_ref = -INFINITY;
        float l = 0.f, l_r = 0.f;   // this half's share of the row sums
        bool ok = true;
        // The loop never breaks: every softmax warp reaches the named barriers
        // of every tile; after a failed wait the remaining work is skipped.
        for (int t = 0; t < ntiles; ++t) {
            const int sb = t & 1;
            const int key0 = t * kBN + 64 * half;
            float sc[64];
            float mloc = -INFINITY;
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar[kSFull + sb], (t >> 1) & 1, p.err));
            if (ok) {
                tc::fence_after_sync();
#pragma unroll
                for (int c = 0; c < 64; c += 32) {
                    float v[32];
                    tc::tmem_ld32(tmem + lane_base + kTmemS + sb * kBN + 64 * half + c, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) sc[c + j] = v[j];
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[kSFree + sb]);   // the odd CTA's is relayed
                const int nvis = lim - key0;         // keys of this half the row sees
                if (p.qk_scale_log2 > 0.f) {
                    // Raw scores stay in sc (masked keys -inf); the scale goes
                    // into the exponent's FMA and, being positive, commutes
                    // with the max.  Only tiles some row sees partly are masked.
                    if (!__all_sync(0xffffffffu, nvis >= 64)) {
#pragma unroll
                        for (int j = 0; j < 64; ++j) sc[j] = j < nvis ? sc[j] : -INFINITY;
                    }
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int j = 0; j < 64; j += 2)
                        m4[(j >> 1) & 3] = fmax3(m4[(j >> 1) & 3], sc[j], sc[j + 1]);
                    mloc = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.qk_scale_log2;
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        sc[j] = j < nvis ? sc[j] * p.qk_scale_log2 : -INFINITY;
                        mloc = fmaxf(mloc, sc[j]);
                    }
                }
            }
            // ---- row max over both halves (warps w and w + 4 only) --------------
            named_sync(kBarPair + (warp & 3), 64);   // the partner read the last tile's
            red[half * 128 + r] = mloc;
            named_sync(kBarPair + (warp & 3), 64);
            const float mt = fmaxf(mloc, red[(half ^ 1) * 128 + r]);
            if (!ok) continue;

            const bool raise = mt > m_ref + kRescaleThreshold;
            float alpha = 1.f;
            if (raise) {
                alpha = fast_exp2(m_ref - mt);
                m_ref = mt;
            }
            // A row that has seen no key yet has m_ref = -inf and only -inf
            // scores: exp2 of them against 0 gives the weights 0.
            const float m_use = m_ref != -INFINITY ? m_ref : 0.f;
            // Folded scale: raw scores times scale (positive) minus m_ref;
            // otherwise sc already holds the scaled scores.
            const float sc_mul = p.qk_scale_log2 > 0.f ? p.qk_scale_log2 : 1.f;
            // Two row sums: of the fp32 weights (for lse) and of the bf16-
            // rounded weights the MMA multiplies V by (to normalise O).
            const float2 mul2 = make_float2(sc_mul, sc_mul);
            const float2 neg2 = make_float2(-m_use, -m_use);
            float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            float2 rr[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            float pk[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float2 e = __ffma2_rn(make_float2(sc[2 * j], sc[2 * j + 1]), mul2, neg2);
                const float p0 = fast_exp2(e.x);
                const float p1 = fast_exp2(e.y);
                const uint32_t w = pack_bf16x2(p0, p1);
                pk[j] = __uint_as_float(w);
                rs[j & 1] = __fadd2_rn(rs[j & 1], make_float2(p0, p1));
                add_bf16x2_f32(rr[j & 1], w);
            }
            const float rowsum = (rs[0].x + rs[1].x) + (rs[0].y + rs[1].y);
            const float rowsum_r = (rr[0].x + rr[1].x) + (rr[0].y + rr[1].y);
            l = l * alpha + rowsum;
            l_r = l_r * alpha + rowsum_r;

            // P is double-buffered: P(t) overwrites the buffer that P.V(t-2)
            // read, so that is the MMA to wait for -- unless O must be
            // rescaled, which needs P.V(t-1) finished.  Each buffer has its
            // own P-full and P.V-done barriers, one phase per use: a warp can
            // only arrive for tile t+2 after P.V(t), which needs every arrival
            // for tile t, so no arrival lands in another tile's phase, and no
            // wait can mistake a later phase for its own (P.V(t) and P.V(t+1)
            // need P(t), which is not written yet).
            const bool rescale = __any_sync(0xffffffffu, raise) && t >= 1;
            if (rescale) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&bar[kODone + ((t - 1) & 1)], ((t - 1) >> 1) & 1, p.err));
            } else if (t >= 2) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&bar[kODone + (t & 1)], ((t - 2) >> 1) & 1, p.err));
            }
            if (!ok) continue;
            if (t >= 1) {
                tc::fence_after_sync();
                if (rescale) {
#pragma unroll 1
                    for (int c = 0; c < 64; c += 32) {
                        float v[32];
                        const uint32_t oc = kTmemO + 64u * half + c;
                        tc::tmem_ld32(tmem + lane_base + oc, v);
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] *= alpha;
                        tc::tmem_st32(tmem + lane_base + oc, v);
                    }
                }
            }
            // P row r, keys of this half: 32 columns of bf16 pairs.
            tc::tmem_st32(tmem + lane_base + kTmemP + 64u * uint32_t(t & 1) + 32u * half, pk);
            const int nkeys = min(kBN, L - t * kBN);
            if (nkeys < kBN) {
                // Slots past the sequence end may hold anything: zero them in
                // this CTA's V half, once it has landed.
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&bar[kVFull + t % kStages], (t / kStages) & 1, p.err));
                if (!ok) continue;
                uint8_t *vs = smem + Smem::v + (t % kStages) * kHalfBytes;
                const int chunks = (kBN - nkeys) * 8;           // 16-B chunks of one box
                for (int i = threadIdx.x; i < chunks; i += kSoftmaxThreads)
                    *reinterpret_cast<uint4 *>(vs + (nkeys + i / 8) * 128 + (i & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                tc::fence_async_smem();
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[kPFull + (t & 1)]);   // the odd CTA's is relayed
        }

        // ---- epilogue ---------------------------------------------------------
        if (ok && ntiles > 0) {
            // the last P.V (its commit covers every earlier MMA)
            ok = __all_sync(0xffffffffu, mbar_wait(&bar[kODone + ((ntiles - 1) & 1)],
                                                   ((ntiles - 1) >> 1) & 1, p.err));
            tc::fence_after_sync();
        }
        // Row sums of the two halves (same m_ref), through the Q buffer, which
        // no MMA reads any more.
        float *sums = reinterpret_cast<float *>(smem + Smem::q);
        named_sync(kBarPair + (warp & 3), 64);
        sums[half * 256 + r] = l;
        sums[half * 256 + 128 + r] = l_r;
        named_sync(kBarPair + (warp & 3), 64);
        l += sums[(half ^ 1) * 256 + r];
        l_r += sums[(half ^ 1) * 256 + 128 + r];
        const int h = kvh * G + (r % G);
        const float t2 = p.sink ? p.sink[h] * kLog2e : -INFINITY;
        const float Mf = fmaxf(m_ref, t2);
        float so = 0.f, Z = 0.f, Zr = 0.f;
        if (Mf != -INFINITY) {
            so = fast_exp2(m_ref - Mf);
            const float st = fast_exp2(t2 - Mf);
            Z = l * so + st;        // exact weights: lse
            Zr = l_r * so + st;     // the weights O was built with: output
        }
        const float scale_o = Zr > 0.f ? so / Zr : 0.f;
        const size_t row = size_t(q_off) + tok;
        uint16_t *dst = p.out + (row * p.num_q_heads + h) * kD + 64 * half;
#pragma unroll 1
        for (int c = 0; c < 64; c += 32) {
            float v[32];
            if (ntiles > 0 && ok) {
                tc::tmem_ld32(tmem + lane_base + kTmemO + 64u * half + c, v);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
            if (row_valid) {
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    uint4 w;
                    w.x = pack_bf16x2(v[j] * scale_o, v[j + 1] * scale_o);
                    w.y = pack_bf16x2(v[j + 2] * scale_o, v[j + 3] * scale_o);
                    w.z = pack_bf16x2(v[j + 4] * scale_o, v[j + 5] * scale_o);
                    w.w = pack_bf16x2(v[j + 6] * scale_o, v[j + 7] * scale_o);
                    *reinterpret_cast<uint4 *>(dst + c + j) = w;
                }
            }
        }
        if (row_valid && p.lse && half == 0)
            p.lse[row * p.num_q_heads + h] = Z > 0.f ? (Mf + fast_log2(Z)) * kLn2 : -INFINITY;
    }

    tc::fence_before_sync();
    __syncthreads();
    cluster_sync();   // no CTA leaves while the pair's MMAs may read its shared memory
    if (warp == 10) {
        tc::fence_after_sync();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_tile_attention_pair(const TileParams &p, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(tile_attention_pair_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kSmemBytes));
    if (e != cudaSuccess) return e;
    dim3 grid(2 * ((p.tiles_per_seq + 1) / 2), p.num_q_heads / p.group, p.batch);
    tile_attention_pair_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace attn
