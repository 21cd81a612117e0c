// gqa_decode.cu -- split-K flash-decoding kernel for grouped-query attention
// over a paged (or contiguous) bf16 KV cache.
//
// Work item: one (sequence b, KV head, key slice p).  The `group` query heads
// that share the KV head are folded into the item's rows, so every K/V byte
// is read from HBM once per call.  The kernel is persistent: a grid of two
// CTAs per SM walks the list of non-empty items in a fixed round-robin order
// (item j goes to CTA j mod grid), so the TMA pipeline never drains between
// items and slices past a sequence's end cost nothing.  Inside a CTA:
//
//   * two producer warps stream 32-key K tiles and V tiles with TMA
//     (cp.async.bulk.tensor, 128-byte swizzle) into two rings of shared-
//     memory stages, translating logical token -> (page, slot) through the
//     page table; they run ahead across item boundaries, K and V each at
//     their own pace, so the K of a warp's next tile lands while it is still
//     busy with the V of the current one;
//   * four consumer warps take the tiles round-robin (tile g -> warp g % 4).
//     Both ring sizes are multiples of 4, so every stage is always consumed
//     by the same warp, in order: a waiter is never more than one phase
//     behind its barrier and the parity wait cannot alias an older phase.
//     Each warp keeps its own online-softmax state (running max m, exp-sum l,
//     unnormalised O) -- a warp-level split of the slice
//     ("decoding_warp_split_k", mha_decoding_single_batch_pipelined,
//     Parameters) -- merged at the end of the item;
//   * scores: lane j owns key j of the tile and dots it with all group rows
//     of q (fp32, packed FFMA2); softmax statistics use warp-shuffle max;
//     P.V: lane owns head_dim/32 channels of every row.
//
// An item's result is either the final output (its sequence needs at most
// one slice) or the partial (O, m, l) for the split-K reduce (a slice leaves
// its exponential sum and running maximum for the reduce pass,
// mha_decoding_single_batch_pipelined, summary).  Scores are kept in base-2
// units internally (q is pre-scaled by scale*log2 e); the partial max written
// to the workspace is in natural-log units.
//
// The arithmetic order depends only on logical token indices, so a paged
// cache and a contiguous cache holding the same tokens give bit-identical
// results.
#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kTile = kGqaTileKeys;  // keys per stage
constexpr int kConsumers = 4;        // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;

constexpr int kThreadsAll = kThreads + 32;  // + the V producer warp

// Ring sizes are multiples of kConsumers (stage ownership, see above) and keep
// two CTAs (<= ~112 KB each) resident per SM.
template <int D, int G>
struct GqaShape {
    static constexpr int kBoxes = D / 64;                 // 64-channel (128 B) column boxes
    static constexpr int kTileBytes = kTile * D * 2;      // one K or V tile
    static constexpr int kKStages = D == 128 ? (G >= 8 ? 4 : 8) : 8;
    static constexpr int kVStages = 4;
    static constexpr int kDpl = D / 32;                   // P.V channels per lane
    static_assert(kKStages % kConsumers == 0 && kVStages % kConsumers == 0,
                  "every stage must have a single consumer warp");
};

// Shared-memory layout (byte offsets from the 1024-aligned base).
template <int D, int G>
struct GqaSmem {
    using S = GqaShape<D, G>;
    static constexpr int kring = 0;
    static constexpr int vring = kring + S::kKStages * S::kTileBytes;
    static constexpr int q = vring + S::kVStages * S::kTileBytes;        // fp32 [2][G][D]
    static constexpr int p = q + 2 * G * D * 4;                          // fp32 [4][32][G]
    static constexpr int mrg = p + kConsumers * kTile * G * 4;           // merge buffer
    static constexpr int mrg_bytes = (2 * kConsumers * G + kConsumers * G * D) * 4;
    static constexpr int bars = mrg + mrg_bytes;                         // kfull, kempty, vfull, vempty
    static constexpr int items = bars + 2 * (S::kKStages + S::kVStages) * 8;  // int [batch + 1]
    static constexpr int fixed = items;
};

template <int D, int G>
size_t gqa_smem_bytes(int batch) {
    return 1024 + size_t(GqaSmem<D, G>::fixed) + sizeof(int) * size_t(batch + 1);
}

// Item j -> (b, kvh, p) through the prefix sums cum[b] = number of items of
// sequences < b (each sequence has num_kv_heads * n_b items, n_b >= 1).
struct Item {
    int b, kvh, part, L, start, end, ntiles;
    bool direct;
};

__device__ __forceinline__ Item decode_item(const GqaParams &p, const int *cum, int j, int hkv) {
    int lo = 0, hi = p.batch;  // find b: cum[b] <= j < cum[b+1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cum[mid] <= j) lo = mid; else hi = mid;
    }
    Item it;
    it.b = lo;
    const int per_head = (cum[lo + 1] - cum[lo]) / hkv;   // n_b
    const int r = j - cum[lo];
    it.kvh = r / per_head;
    it.part = r - it.kvh * per_head;
    const uint32_t cap = uint32_t(p.num_partitions) * uint32_t(p.chunk);
    it.L = static_cast<int>(min(p.kv_len[lo], cap));
    it.start = it.part * p.chunk;
    it.end = min(it.start + p.chunk, it.L);
    it.ntiles = it.start < it.end ? (it.end - it.start + kTile - 1) / kTile : 0;
    it.direct = per_head <= 1 && (it.L + p.chunk - 1) / p.chunk <= 1;
    return it;
}

template <int D, int G>
__global__ void __launch_bounds__(kThreadsAll, 2)
gqa_decode_kernel(const __grid_constant__ GqaParams p) {
    using S = GqaShape<D, G>;
    using M = GqaSmem<D, G>;
    constexpr int kKStages = S::kKStages;
    constexpr int kVStages = S::kVStages;
    constexpr int kDpl = S::kDpl;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *kfull = reinterpret_cast<uint64_t *>(smem + M::bars);
    uint64_t *kempty = kfull + kKStages;
    uint64_t *vfull = kempty + kKStages;
    uint64_t *vempty = vfull + kVStages;
    int *cum = reinterpret_cast<int *>(smem + M::items);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int hkv = p.num_q_heads / G;
    const uint32_t cap = uint32_t(p.num_partitions) * uint32_t(p.chunk);

    // ---- item table: n_b = max(1, slices of b); cum = prefix sums * hkv ----
    if (warp == 0) {
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
    if (threadIdx.x == 32) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&kfull[s], 1);
            mbar_init(&kempty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&vfull[s], 1);
            mbar_init(&vempty[s], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    const int num_items = cum[p.batch];

    if (warp >= kConsumers) {
        // ------------------------------------------------------------------
        // Producer warps: warp 4 streams K, warp 5 streams V.  Page-table
        // lookups by all lanes, TMA issue by lane 0.
        // ------------------------------------------------------------------
        const bool is_k = warp == kConsumers;
        const CUtensorMap *map = is_k ? &p.k_map : &p.v_map;
        const int nst = is_k ? kKStages : kVStages;
        uint64_t *full = is_k ? kfull : vfull;
        uint64_t *empty = is_k ? kempty : vempty;
        uint8_t *ring = smem + (is_k ? M::kring : M::vring);
        if (lane == 0) prefetch_tensormap(map);
        const int box_rows = p.box_rows;  // 32, 16 or 8
        const int boxes_per_tile = kTile / box_rows;
        const uint32_t box_bytes = uint32_t(box_rows) * 128u;
        bool aborted = false;
        int g = 0;  // tiles issued by this warp so far
        for (int j = blockIdx.x; j < num_items && !aborted; j += gridDim.x) {
            const Item it = decode_item(p, cum, j, hkv);
            for (int base = 0; base < it.ntiles && !aborted; base += 32) {
                int pg[4] = {-1, -1, -1, -1};
                int sl[4] = {0, 0, 0, 0};
                const int my_tile = base + lane;
                if (my_tile < it.ntiles) {
                    const int t0 = it.start + my_tile * kTile;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int t = t0 + r * box_rows;
                        if (r >= boxes_per_tile || t >= it.L) continue;
                        if (p.page_table) {
                            const int pidx = t / p.page_size;
                            int e = pidx < p.max_pages
                                        ? p.page_table[size_t(it.b) * p.max_pages + pidx] : -1;
                            if (e < 0 || e >= p.num_pages) {
                                if (is_k) atomicOr(p.err, kErrBadPage);
                                e = -1;
                            }
                            pg[r] = e;
                            sl[r] = t % p.page_size;
                        } else {
                            pg[r] = it.b;
                            sl[r] = t;
                        }
                    }
                }
                const int lim = min(base + 32, it.ntiles);
                for (int i = base; i < lim; ++i) {
                    int pages[4], slots[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        pages[r] = __shfl_sync(0xffffffffu, pg[r], i - base);
                        slots[r] = __shfl_sync(0xffffffffu, sl[r], i - base);
                    }
                    if (lane == 0) {
                        const int s = g % nst;
                        if (g >= nst && !mbar_wait(&empty[s], ((g / nst) - 1) & 1, p.err)) {
                            aborted = true;
                        } else {
                            uint32_t nbox = 0;
#pragma unroll
                            for (int r = 0; r < 4; ++r) nbox += pages[r] >= 0 ? 1u : 0u;
                            mbar_arrive_expect_tx(&full[s], S::kBoxes * nbox * box_bytes);
                            uint8_t *dst = ring + s * S::kTileBytes;
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                if (pages[r] < 0) continue;
#pragma unroll
                                for (int cb = 0; cb < S::kBoxes; ++cb)
                                    tma_load_4d(dst + cb * kTile * 128 + r * box_rows * 128, map,
                                                &full[s], cb * 64, slots[r], it.kvh, pages[r]);
                            }
                        }
                    }
                    aborted = __shfl_sync(0xffffffffu, aborted, 0);
                    if (aborted) break;
                    ++g;
                }
            }
        }
        // Before the warp leaves, every copy it issued must have landed
        // (normally the consumers already saw these phases complete).
        if (lane == 0)
            for (int i = max(0, g - nst); i < g; ++i)
                mbar_wait(&full[i % nst], (i / nst) & 1, p.err);
        return;
    }

    // ----------------------------------------------------------------------
    // Consumer warps (threads 0..127).
    // ----------------------------------------------------------------------
    const int tid = threadIdx.x;
    // P.V addressing: this lane's kDpl channels inside the swizzled V rows.
    const int pv_col = lane * kDpl;
    const int pv_box = pv_col / 64;
    const int pv_byte = (pv_col % 64) * 2;
    const int pv_chunk = pv_byte >> 4;
    const int pv_inner = pv_byte & 15;
    float *p_w = reinterpret_cast<float *>(smem + M::p) + warp * kTile * G;

    // q of the next item, prefetched into registers.
    constexpr int kQPer = (G * D + kConsumers * 32 - 1) / (kConsumers * 32);
    uint16_t q_next[kQPer];
    auto load_q = [&](int j) {
        if (j < num_items) {
            const Item it = decode_item(p, cum, j, hkv);
            const uint16_t *src = p.q + (size_t(it.b) * p.num_q_heads + it.kvh * G) * D;
#pragma unroll
            for (int k = 0; k < kQPer; ++k) {
                const int idx = tid + k * kConsumers * 32;
                q_next[k] = idx < G * D ? src[idx] : uint16_t(0);
            }
        }
    };
    load_q(blockIdx.x);

    bool ok = true;
    int g_base = 0;  // tiles of this CTA before the current item
    int iter = 0;
    for (int j = blockIdx.x; j < num_items; j += gridDim.x, ++iter) {
        const Item it = decode_item(p, cum, j, hkv);
        float *q_s = reinterpret_cast<float *>(smem + M::q) + (iter & 1) * G * D;
#pragma unroll
        for (int k = 0; k < kQPer; ++k) {
            const int idx = tid + k * kConsumers * 32;
            if (idx < G * D)
                q_s[idx] = __uint_as_float(uint32_t(q_next[k]) << 16) * p.qk_scale_log2;
        }
        load_q(j + gridDim.x);
        // q_s ready; every consumer has also finished reading the merge
        // buffer of the previous item.
        named_sync(1, kConsumers * 32);

        float m_run[G], l_lane[G], o_acc[G][kDpl];
#pragma unroll
        for (int r = 0; r < G; ++r) {
            m_run[r] = -INFINITY;
            l_lane[r] = 0.f;
#pragma unroll
            for (int d = 0; d < kDpl; ++d) o_acc[r][d] = 0.f;
        }

        // This warp's tiles of the item: item-local t with (g_base + t) % 4 == warp.
        const int t_first = (warp - g_base % kConsumers + kConsumers) % kConsumers;
        for (int t = t_first; ok && t < it.ntiles; t += kConsumers) {
            const int g = g_base + t;
            const int sk = g % kKStages;
            const int sv = g % kVStages;
            if (!mbar_wait(&kfull[sk], (g / kKStages) & 1, p.err)) {
                ok = false;
                break;
            }
            const uint8_t *ks = smem + M::kring + sk * S::kTileBytes;
            const uint8_t *vs = smem + M::vring + sv * S::kTileBytes;
            const int t0 = it.start + t * kTile;
            const int nvalid = min(kTile, it.end - t0);

            // ---- scores: lane j <-> key j ----------------------------------
            float2 acc[G];
#pragma unroll
            for (int r = 0; r < G; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll
            for (int cb = 0; cb < S::kBoxes; ++cb) {
                const uint8_t *krow = ks + cb * kTile * 128 + lane * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint4 kw =
                        *reinterpret_cast<const uint4 *>(krow + ((ch ^ (lane & 7)) << 4));
                    const float2 k01 = bf16x2_to_float2(kw.x);
                    const float2 k23 = bf16x2_to_float2(kw.y);
                    const float2 k45 = bf16x2_to_float2(kw.z);
                    const float2 k67 = bf16x2_to_float2(kw.w);
                    const float *qc = q_s + cb * 64 + ch * 8;
#pragma unroll
                    for (int r = 0; r < G; ++r) {
                        const float4 qa = *reinterpret_cast<const float4 *>(qc + r * D);
                        const float4 qb = *reinterpret_cast<const float4 *>(qc + r * D + 4);
                        acc[r] = __ffma2_rn(make_float2(qa.x, qa.y), k01, acc[r]);
                        acc[r] = __ffma2_rn(make_float2(qa.z, qa.w), k23, acc[r]);
                        acc[r] = __ffma2_rn(make_float2(qb.x, qb.y), k45, acc[r]);
                        acc[r] = __ffma2_rn(make_float2(qb.z, qb.w), k67, acc[r]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&kempty[sk]);   // K tile no longer needed

            // ---- online softmax (base 2) -----------------------------------
            const bool valid = lane < nvalid;
            float pr[G], alpha[G];
#pragma unroll
            for (int r = 0; r < G; ++r) {
                const float sc = valid ? acc[r].x + acc[r].y : -INFINITY;
                const float mt = warp_max(sc);          // finite: key 0 of the tile is valid
                const float mn = fmaxf(m_run[r], mt);
                alpha[r] = fast_exp2(m_run[r] - mn);    // 0 on the first tile
                pr[r] = fast_exp2(sc - mn);             // 0 for masked keys
                m_run[r] = mn;
                l_lane[r] = l_lane[r] * alpha[r] + pr[r];
            }
            if constexpr (G == 4) {
                *reinterpret_cast<float4 *>(p_w + lane * 4) =
                    make_float4(pr[0], pr[1], pr[2], pr[3]);
            } else if constexpr (G == 2) {
                *reinterpret_cast<float2 *>(p_w + lane * 2) = make_float2(pr[0], pr[1]);
            } else {
#pragma unroll
                for (int r = 0; r < G; ++r) p_w[lane * G + r] = pr[r];
            }
            __syncwarp();
#pragma unroll
            for (int r = 0; r < G; ++r)
#pragma unroll
                for (int d = 0; d < kDpl; ++d) o_acc[r][d] *= alpha[r];

            // ---- P.V: lane owns kDpl channels of every row -----------------
            if (!mbar_wait(&vfull[sv], (g / kVStages) & 1, p.err)) {
                ok = false;
                break;
            }
            const uint8_t *vbase = vs + pv_box * kTile * 128 + pv_inner;
            for (int jj = 0; jj < nvalid; ++jj) {
                const uint8_t *vr = vbase + jj * 128 + ((pv_chunk ^ (jj & 7)) << 4);
                float2 v01, v23;
                if constexpr (kDpl == 4) {
                    const uint2 vw = *reinterpret_cast<const uint2 *>(vr);
                    v01 = bf16x2_to_float2(vw.x);
                    v23 = bf16x2_to_float2(vw.y);
                } else {
                    v01 = bf16x2_to_float2(*reinterpret_cast<const uint32_t *>(vr));
                }
                float pj[G];
                if constexpr (G == 4) {
                    const float4 tq = *reinterpret_cast<const float4 *>(p_w + jj * 4);
                    pj[0] = tq.x; pj[1] = tq.y; pj[2] = tq.z; pj[3] = tq.w;
                } else {
#pragma unroll
                    for (int r = 0; r < G; ++r) pj[r] = p_w[jj * G + r];
                }
#pragma unroll
                for (int r = 0; r < G; ++r) {
                    float2 o01 = make_float2(o_acc[r][0], o_acc[r][1]);
                    o01 = __ffma2_rn(make_float2(pj[r], pj[r]), v01, o01);
                    o_acc[r][0] = o01.x;
                    o_acc[r][1] = o01.y;
                    if constexpr (kDpl == 4) {
                        float2 o23 = make_float2(o_acc[r][2], o_acc[r][3]);
                        o23 = __ffma2_rn(make_float2(pj[r], pj[r]), v23, o23);
                        o_acc[r][2] = o23.x;
                        o_acc[r][3] = o23.y;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&vempty[sv]);
        }
        g_base += it.ntiles;

        // ---- merge the consumer warps' states and write the item --------------
        float *mb = reinterpret_cast<float *>(smem + M::mrg);
        float *m_s = mb;                          // [consumer][row]
        float *l_s = mb + kConsumers * G;
        float *o_s = mb + 2 * kConsumers * G;     // [consumer][row][D]
#pragma unroll
        for (int r = 0; r < G; ++r) {
            const float l = warp_sum(l_lane[r]);
            if (lane == 0) {
                m_s[warp * G + r] = m_run[r];
                l_s[warp * G + r] = l;
            }
#pragma unroll
            for (int d = 0; d < kDpl; ++d) o_s[(warp * G + r) * D + pv_col + d] = o_acc[r][d];
        }
        named_sync(1, kConsumers * 32);

        const int h0 = it.kvh * G;
        constexpr int kVec = 4;
        for (int idx = tid; idx < G * D / kVec; idx += kConsumers * 32) {
            const int r = idx / (D / kVec);
            const int c0 = (idx - r * (D / kVec)) * kVec;
            float Mx = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) Mx = fmaxf(Mx, m_s[w * G + r]);
            float l = 0.f;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) {
                const float mw = m_s[w * G + r];
                if (mw == -INFINITY) continue;
                const float sc = fast_exp2(mw - Mx);
                l += sc * l_s[w * G + r];
                const float4 ow = *reinterpret_cast<const float4 *>(o_s + (w * G + r) * D + c0);
                o.x += sc * ow.x; o.y += sc * ow.y; o.z += sc * ow.z; o.w += sc * ow.w;
            }
            const int h = h0 + r;
            if (it.direct) {
                const float t2 = p.sink ? p.sink[h] * kLog2e : -INFINITY;
                const float Mf = fmaxf(Mx, t2);
                float Z = 0.f, so = 0.f;
                if (Mf != -INFINITY) {
                    so = fast_exp2(Mx - Mf);
                    Z = l * so + fast_exp2(t2 - Mf);
                }
                const float inv = Z > 0.f ? so / Z : 0.f;
                uint2 packed;
                packed.x = pack_bf16x2(o.x * inv, o.y * inv);
                packed.y = pack_bf16x2(o.z * inv, o.w * inv);
                *reinterpret_cast<uint2 *>(p.out + (size_t(it.b) * p.num_q_heads + h) * D + c0) =
                    packed;
                if (c0 == 0 && p.lse)
                    p.lse[size_t(it.b) * p.num_q_heads + h] =
                        Z > 0.f ? (Mf + fast_log2(Z)) * kLn2 : -INFINITY;
            } else {
                const size_t base = (size_t(it.part) * p.batch + it.b) * p.num_q_heads + h;
                *reinterpret_cast<float4 *>(p.ws_o + base * D + c0) = o;
                if (c0 == 0) {
                    p.ws_m[base] = Mx * kLn2;
                    p.ws_l[base] = l;
                }
            }
        }
    }
    pdl_launch_dependents();
}

int g_num_sms[64];

template <int D, int G>
cudaError_t launch_t(const GqaParams &p, cudaStream_t stream) {
    const size_t smem = gqa_smem_bytes<D, G>(p.batch);
    auto kern = gqa_decode_kernel<D, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (g_num_sms[dev] == 0) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_num_sms[dev] = n;
    }
    // Two resident CTAs per SM; never more CTAs than the largest item count.
    long long grid = 2LL * g_num_sms[dev];
    const long long max_items = static_cast<long long>(p.batch) * (p.num_q_heads / G) *
                                p.num_partitions;
    if (grid > max_items) grid = max_items;
    if (grid < 1) grid = 1;
    kern<<<dim3(static_cast<unsigned>(grid)), kThreadsAll, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const GqaParams &p, cudaStream_t stream) {
    switch (p.group) {
        case 1: return launch_t<D, 1>(p, stream);
        case 2: return launch_t<D, 2>(p, stream);
        case 4: return launch_t<D, 4>(p, stream);
        case 8: return launch_t<D, 8>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gqa_decode(const GqaParams &p, cudaStream_t stream) {
    switch (p.head_dim) {
        case 64: return launch_d<64>(p, stream);
        case 128: return launch_d<128>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
