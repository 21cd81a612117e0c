// tile_attention.cu -- tensor-core (tcgen05) attention tiles for batches
// whose sequences carry several query rows (ragged prefill mixed with
// decode), with a causal mask aligned to the end of the cache.
//
// Decode takes no route of its own here: one-token decode is handled as the
// degenerate case of prefill (mha_sm100_dispatch, summary), so every sequence of the
// batch, single-row ones included, is cut into tiles of 128 MMA rows.  A tile
// holds T = 128 / group consecutive tokens x the group's query heads of one
// KV head, so each K/V tile fetched serves all heads of the group.  Row r is
// token r / group, head r % group -- exactly the memory order of q, so one
// 4-D TMA box (64 channels x group heads x 1 KV head x T tokens) loads it.
//
// Per 128-key tile: S = Q K^T (M=128, N=128, K=128) into a double-buffered
// TMEM accumulator, online softmax by eight warps (two per row: warps w and
// w+4 share TMEM lanes 32(w%4).. and split the 128 keys; causal and length
// masks applied per element; the two halves' row maxima combined through
// shared memory, synchronising only the two warps of a row quarter, which
// share an SM sub-partition), P (bf16 pairs) into TMEM, then O += P V (M=128, N=128,
// K=128) with P as the A operand from TMEM.  The running max is lazy: it is
// raised, and O rescaled, only when a tile's max exceeds it by more than 8
// (base 2).  No split-K: each CTA covers all keys its rows can see.
//
// K and V have rings of their own (three 32 KB stages each): a K stage is
// free again as soon as its score MMA is done, so the next K tiles load
// while the softmax and P.V of earlier tiles run, and V tiles arrive for the
// P.V MMA later.
//
// Warp roles (352 threads): 0-7 softmax/epilogue, 8 TMA producer of Q and K,
// 9 TMA producer of V, 10 TMEM allocation + MMA issue.
#include "launch.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace attn {
namespace {

constexpr int kD = 128;
constexpr int kBN = kTileKeys;               // keys per tile
constexpr int kStages = 3;
constexpr int kBoxBytes = 128 * 128;         // 128 rows x 128 B (64 channels)
constexpr int kTileBytes = 2 * kBoxBytes;    // 128 rows x 128 channels
constexpr int kThreads = 352;
constexpr int kSoftmaxThreads = 256;         // warps 0-7
constexpr int kBarPair = 2;                  // named barriers 2..5: the two warps of a row quarter
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;               // S buffers at 0 and 128
constexpr uint32_t kTmemO = 256;
constexpr uint32_t kTmemP = 384;             // 64 columns: P of one tile as bf16 pairs
constexpr float kRescaleThreshold = 8.0f;

// V as the MN-major B operand: two 64-channel blocks 16 KB apart, 8-key
// groups 1 KB apart.
constexpr uint32_t kVLbo = kBoxBytes;
constexpr uint32_t kVSbo = 1024;

struct Smem {
    static constexpr int q = 0;                                  // 32 KB
    static constexpr int k = q + kTileBytes;                     // K ring, 96 KB
    static constexpr int v = k + kStages * kTileBytes;           // V ring, 96 KB
    static constexpr int red = v + kStages * kTileBytes;
    static constexpr int bars = red + 2 * 128 * 4;               // +1 KB (row maxima)
    static constexpr int total = bars + 256;
};
constexpr size_t kSmemBytes = Smem::total + 1024;

enum Bar {
    kKFull = 0,                   // [kStages]
    kKEmpty = kStages,            // [kStages]
    kVFull = 2 * kStages,         // [kStages]
    kVEmpty = 3 * kStages,        // [kStages]
    kQFull = 4 * kStages,
    kSFull = kQFull + 1,          // [2]
    kSFree = kSFull + 2,          // [2]
    kPFull = kSFree + 2,
    kODone = kPFull + 1,
    kNumBars = kODone + 1
};

__global__ void __launch_bounds__(kThreads, 1)
tile_attention_kernel(const __grid_constant__ TileParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Smem::bars);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Smem::bars + kNumBars * 8);

    const int G = p.group;
    const int T = kTileRows / G;                 // tokens per tile
    // Longest tiles first: blockIdx.x counts down the tiles of a sequence.
    const int tile = p.tiles_per_seq - 1 - static_cast<int>(blockIdx.x);
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int q_off = static_cast<int>(p.q_row_offsets[b]);
    const int n = static_cast<int>(p.q_row_offsets[b + 1]) - q_off;
    const int L = static_cast<int>(p.kv_len[b]);
    const int t0 = tile * T;
    if (t0 >= n) return;                         // uniform over the CTA
    const int t_end = min(t0 + T, n);
    // Keys any row of this tile can see.
    int kmax = p.causal ? L - n + t_end : L;
    kmax = max(0, min(kmax, L));
    const int ntiles = (kmax + kBN - 1) / kBN;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const uint32_t cnt = (i == kSFree || i == kSFree + 1 || i == kPFull) ? 8u : 1u;
            mbar_init(&bar[i], cnt);
        }
        fence_mbar_init();
    }
    if (warp == 10) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8 || warp == 9) {
        // ------------------------------------------------------------ producers
        // warp 8: Q, then the K ring; warp 9: the V ring.
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
                    mbar_arrive_expect_tx(&bar[kQFull], kTileBytes);
                    for (int cb = 0; cb < 2; ++cb)
                        tma_load_4d(smem + Smem::q + cb * kBoxBytes, &p.q_map, &bar[kQFull],
                                    cb * 64, 0, kvh, q_off + t0);
                }
            }
            const int box_rows = p.box_rows;       // 128, 64, 32, 16 or 8
            const int nb = kBN / box_rows;         // row boxes per key tile
            int cached = -1, my_page = -1, my_slot = 0;
            bool aborted = false;
            int issued = 0;
            for (int i = 0; i < ntiles && !aborted; ++i) {
                const int key0 = i * kBN;
                const int live = min(nb, (L - key0 + box_rows - 1) / box_rows);
                const int s = i % kStages;
                if (lane == 0) {
                    if (i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1, p.err))
                        aborted = true;
                    else
                        mbar_arrive_expect_tx(&full[s],
                                              uint32_t(live) * 2u * uint32_t(box_rows) * 128u);
                }
                aborted = __shfl_sync(0xffffffffu, aborted, 0);
                if (aborted) break;
                uint8_t *st = ring + s * kTileBytes;
                for (int r = 0; r < live; ++r) {
                    const int g = i * nb + r;      // box index within the sequence
                    if ((g >> 5) != cached) {      // warp-uniform refill of 32 lookups
                        cached = g >> 5;
                        const int t = ((cached << 5) + lane) * box_rows;
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
                            mbar_complete_tx(&full[s], 2u * uint32_t(box_rows) * 128u);
                        } else {
#pragma unroll
                            for (int cb = 0; cb < 2; ++cb)
                                tma_load_4d(st + cb * kBoxBytes + r * box_rows * 128, map, &full[s],
                                            cb * 64, slot, kvh, page);
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
        // ------------------------------------------------------------ MMA issue
        if (ntiles > 0 && lane == 0) {
            constexpr uint32_t idesc_s = tc::idesc_bf16_f32(128, kBN, 0, 0);
            constexpr uint32_t idesc_o = tc::idesc_bf16_f32(128, kD, 0, 1);
            const uint32_t q_base = smem_addr(smem + Smem::q);
            const uint32_t k_base = smem_addr(smem + Smem::k);
            const uint32_t v_base = smem_addr(smem + Smem::v);
            bool ok = mbar_wait(&bar[kQFull], 0, p.err);
            for (int t = 0; ok && t <= ntiles; ++t) {
                if (t < ntiles) {
                    const int s = t % kStages;
                    const int sb = t & 1;
                    ok = mbar_wait(&bar[kKFull + s], (t / kStages) & 1, p.err);
                    if (ok && t >= 2) ok = mbar_wait(&bar[kSFree + sb], ((t >> 1) - 1) & 1, p.err);
                    if (!ok) break;
                    tc::fence_after_sync();
                    // Descriptors advance by byte offset / 16 in their start
                    // field; unrolled so issue is not bound by descriptor math.
                    const uint64_t qd = tc::smem_desc_sw128(q_base, 16, 1024);
                    const uint64_t kd = tc::smem_desc_sw128(k_base + s * kTileBytes, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint64_t off = uint64_t(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
                        tc::mma_bf16(tmem + kTmemS + sb * kBN, qd + off, kd + off, idesc_s, kk > 0);
                    }
                    tc::mma_commit(&bar[kSFull + sb]);
                    tc::mma_commit(&bar[kKEmpty + s]);
                }
                if (t >= 1) {
                    const int tp = t - 1;
                    ok = mbar_wait(&bar[kPFull], tp & 1, p.err);
                    if (ok) ok = mbar_wait(&bar[kVFull + tp % kStages], (tp / kStages) & 1, p.err);
                    if (!ok) break;
                    tc::fence_after_sync();
                    const uint64_t vd = tc::smem_desc_sw128(v_base + (tp % kStages) * kTileBytes,
                                                            kVLbo, kVSbo);
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        // A = P from TMEM: 16 keys = 8 columns of bf16 pairs per step
                        tc::mma_bf16_tmem_a(tmem + kTmemO, tmem + kTmemP + kk * 8,
                                            vd + uint64_t((kk * 16 * 128) >> 4), idesc_o,
                                            tp > 0 || kk > 0);
                    tc::mma_commit(&bar[kODone]);
                    tc::mma_commit(&bar[kVEmpty + (tp % kStages)]);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ softmax
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
                if (lane == 0) mbar_arrive(&bar[kSFree + sb]);
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
            const bool folded = p.qk_scale_log2 > 0.f;
            const float sc_mul = folded ? p.qk_scale_log2 : 1.f;
            // Two row sums: of the fp32 weights (for lse) and of the bf16-
            // rounded weights the MMA multiplies V by (to normalise O).
            // Pairs of keys go through the packed fp32x2 FMA and adds.
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

            // O(t-1) has read P(t-1) and must be finished before P is
            // overwritten or O rescaled.
            if (t >= 1) {
                ok = __all_sync(0xffffffffu, mbar_wait(&bar[kODone], (t - 1) & 1, p.err));
                if (!ok) continue;
                tc::fence_after_sync();
                if (__any_sync(0xffffffffu, raise)) {
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
            tc::tmem_st32(tmem + lane_base + kTmemP + 32u * half, pk);
            const int nkeys = min(kBN, L - t * kBN);
            if (nkeys < kBN) {
                // Slots past the sequence end may hold anything: zero them in V,
                // once the V tile has landed.
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&bar[kVFull + t % kStages], (t / kStages) & 1, p.err));
                if (!ok) continue;
                uint8_t *vs = smem + Smem::v + (t % kStages) * kTileBytes;
                const int per_box = (kBN - nkeys) * 8;          // 16-B chunks
                for (int i = threadIdx.x; i < 2 * per_box; i += kSoftmaxThreads) {
                    const int box = i / per_box;
                    const int rem = i - box * per_box;
                    *reinterpret_cast<uint4 *>(vs + box * kBoxBytes + (nkeys + rem / 8) * 128 +
                                               (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                tc::fence_async_smem();
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[kPFull]);
        }

        // ---- epilogue ---------------------------------------------------------
        // Row sums of the two halves (same m_ref), through the Q buffer, which
        // no MMA reads any more (the last score MMA was done when its S was
        // read), while the last P.V is still in flight.
        float *sums = reinterpret_cast<float *>(smem + Smem::q);
        named_sync(kBarPair + (warp & 3), 64);
        sums[half * 256 + r] = l;
        sums[half * 256 + 128 + r] = l_r;
        named_sync(kBarPair + (warp & 3), 64);
        l += sums[(half ^ 1) * 256 + r];
        l_r += sums[(half ^ 1) * 256 + 128 + r];
        if (ok && ntiles > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bar[kODone], (ntiles - 1) & 1, p.err));
            tc::fence_after_sync();
        }
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
        // The warp's 32 rows x 64 channels (bf16) go out through 4 KB of the K
        // ring, which no MMA reads any more: a lane writes its row, then eight
        // lanes a row store whole 128-byte lines.
        uint8_t *tw = smem + Smem::k + warp * 4096;
#pragma unroll 1
        for (int c = 0; c < 64; c += 32) {
            float v[32];
            if (ntiles > 0 && ok) {
                tc::tmem_ld32(tmem + lane_base + kTmemO + 64u * half + c, v);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                uint4 w;
                w.x = pack_bf16x2(v[j] * scale_o, v[j + 1] * scale_o);
                w.y = pack_bf16x2(v[j + 2] * scale_o, v[j + 3] * scale_o);
                w.z = pack_bf16x2(v[j + 4] * scale_o, v[j + 5] * scale_o);
                w.w = pack_bf16x2(v[j + 6] * scale_o, v[j + 7] * scale_o);
                const int k = (c + j) >> 3;          // 16-byte chunk of the row
                *reinterpret_cast<uint4 *>(tw + lane * 128 + (((k + lane) & 7) << 4)) = w;
            }
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + (lane >> 3), k = lane & 7;
            const int r2 = (warp & 3) * 32 + rr;     // MMA row of that line
            const int tok2 = t0 + r2 / G;
            if (tok2 < n) {
                const uint4 w = *reinterpret_cast<const uint4 *>(tw + rr * 128 + (((k + rr) & 7) << 4));
                const size_t orow = (size_t(q_off) + tok2) * p.num_q_heads + kvh * G + (r2 % G);
                *reinterpret_cast<uint4 *>(p.out + orow * kD + 64 * half + 8 * k) = w;
            }
        }
        if (row_valid && p.lse && half == 0)
            p.lse[row * p.num_q_heads + h] = Z > 0.f ? (Mf + fast_log2(Z)) * kLn2 : -INFINITY;
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 10) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_tile_attention(const TileParams &p, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(tile_attention_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kSmemBytes));
    if (e != cudaSuccess) return e;
    dim3 grid(p.tiles_per_seq, p.num_q_heads / p.group, p.batch);
    tile_attention_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace attn
