// gqa_decode.cu -- split-K flash-decoding partition kernel for grouped-query
// attention over a paged (or contiguous) bf16 KV cache.
//
// One CTA handles one (key slice p, KV head, sequence b).  The `group` query
// heads that share the KV head are folded into the CTA's rows, so every K/V
// byte is read from HBM once per call.  Inside the CTA:
//
//   * one producer warp streams 32-key K and V tiles with TMA
//     (cp.async.bulk.tensor, 128-byte swizzle) into a ring of shared-memory
//     stages, translating logical token -> (page, slot) through the page
//     table for every tile;
//   * four consumer warps take the tiles round-robin.  Each keeps its own
//     online-softmax state (running max m, exp-sum l, unnormalised O) --
//     a warp-level split of the slice ("decoding_warp_split_k",
//     mha_decoding_single_batch_pipelined, Parameters) -- and the four are
//     merged at the end;
//   * scores: lane j owns key j of the tile and dots it with all group rows
//     of q (fp32, packed FFMA2); softmax statistics use warp-shuffle max;
//     P.V: lane owns head_dim/32 channels of every row.
//
// The slice's result is either the final output (the sequence needs at most
// one slice) or the partial (O, m, l) for the split-K reduce ("writes partial
// exp_sum and qk_max statistics for a subsequent mha_splitk_reduce pass",
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

template <int D>
struct GqaShape {
    static constexpr int kBoxes = D / 64;                 // 64-channel (128 B) column boxes
    static constexpr int kTileBytes = kTile * D * 2;      // one K or V tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStages = D == 128 ? 6 : 10;
    static constexpr int kDpl = D / 32;                   // P.V channels per lane
};

template <int D, int G>
constexpr size_t gqa_smem_bytes() {
    using S = GqaShape<D>;
    return 1024 /* alignment slack */ + size_t(S::kStages) * S::kStageBytes +
           sizeof(float) * (G * D + kConsumers * kTile * G + 2 * kConsumers * G +
                            kConsumers * G * D) +
           sizeof(uint64_t) * 2 * S::kStages;
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 2)
gqa_decode_kernel(const __grid_constant__ GqaParams p) {
    using S = GqaShape<D>;
    constexpr int kStages = S::kStages;
    constexpr int kDpl = S::kDpl;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *q_s = reinterpret_cast<float *>(smem + kStages * S::kStageBytes);
    float *p_s = q_s + G * D;                  // [consumer][key][row]
    float *m_s = p_s + kConsumers * kTile * G;  // [consumer][row]
    float *l_s = m_s + kConsumers * G;
    float *o_s = l_s + kConsumers * G;         // [consumer][row][D]
    uint64_t *full = reinterpret_cast<uint64_t *>(o_s + kConsumers * G * D);
    uint64_t *empty = full + kStages;

    const int part = blockIdx.x;
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // A length above the planned capacity P * chunk is a caller error: flag
    // it and attend to the first P * chunk keys only.
    const uint32_t cap = uint32_t(p.num_partitions) * uint32_t(p.chunk);
    const uint32_t len_in = p.kv_len[b];
    if (len_in > cap && part == 0 && threadIdx.x == 0) atomicOr(p.err, kErrBadLength);
    const int L = static_cast<int>(min(len_in, cap));
    const int start = part * p.chunk;
    const int end = min(start + p.chunk, L);
    const int nslices = (L + p.chunk - 1) / p.chunk;
    const bool direct = nslices <= 1;  // this CTA (part 0) writes the final rows
    if (start >= L && !(direct && part == 0)) return;
    const int ntiles = start < end ? (end - start + kTile - 1) / kTile : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumers) {
        // ------------------------------------------------------------------
        // Producer warp: page-table lookups by all lanes, TMA issue by lane 0.
        // ------------------------------------------------------------------
        if (lane == 0) {
            prefetch_tensormap(&p.k_map);
            prefetch_tensormap(&p.v_map);
        }
        const int box_rows = p.box_rows;            // 32, 16 or 8
        const int boxes_per_tile = kTile / box_rows;
        const uint32_t box_bytes = uint32_t(box_rows) * 128u;
        bool aborted = false;
        int issued = 0;
        for (int base = 0; base < ntiles && !aborted; base += 32) {
            int pg[4] = {-1, -1, -1, -1};
            int sl[4] = {0, 0, 0, 0};
            const int my_tile = base + lane;
            if (my_tile < ntiles) {
                const int t0 = start + my_tile * kTile;
                for (int r = 0; r < boxes_per_tile; ++r) {
                    const int t = t0 + r * box_rows;
                    if (t >= L) break;
                    if (p.page_table) {
                        const int pidx = t / p.page_size;
                        int e = pidx < p.max_pages
                                    ? p.page_table[size_t(b) * p.max_pages + pidx] : -1;
                        if (e < 0 || e >= p.num_pages) {
                            atomicOr(p.err, kErrBadPage);
                            e = -1;
                        }
                        pg[r] = e;
                        sl[r] = t % p.page_size;
                    } else {
                        pg[r] = b;
                        sl[r] = t;
                    }
                }
            }
            const int lim = min(base + 32, ntiles);
            for (int i = base; i < lim; ++i) {
                int pages[4], slots[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    pages[r] = __shfl_sync(0xffffffffu, pg[r], i - base);
                    slots[r] = __shfl_sync(0xffffffffu, sl[r], i - base);
                }
                if (lane == 0) {
                    const int s = i % kStages;
                    if (i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1, p.err)) {
                        aborted = true;
                    } else {
                        uint32_t nbox = 0;
                        for (int r = 0; r < boxes_per_tile; ++r) nbox += pages[r] >= 0 ? 1u : 0u;
                        // every box is loaded for K and V, in kBoxes column blocks
                        mbar_arrive_expect_tx(&full[s], 2u * S::kBoxes * nbox * box_bytes);
                        uint8_t *ks = smem + s * S::kStageBytes;
                        uint8_t *vs = ks + S::kTileBytes;
                        for (int r = 0; r < boxes_per_tile; ++r) {
                            if (pages[r] < 0) continue;
#pragma unroll
                            for (int cb = 0; cb < S::kBoxes; ++cb) {
                                const int off = cb * kTile * 128 + r * box_rows * 128;
                                tma_load_4d(ks + off, &p.k_map, &full[s], cb * 64, slots[r], kvh,
                                            pages[r]);
                                tma_load_4d(vs + off, &p.v_map, &full[s], cb * 64, slots[r], kvh,
                                            pages[r]);
                            }
                        }
                    }
                }
                aborted = __shfl_sync(0xffffffffu, aborted, 0);
                if (aborted) break;
                issued = i + 1;
            }
        }
        // Before the warp leaves, every copy it issued must have landed
        // (normally the consumers already saw these phases complete).
        if (lane == 0)
            for (int i = max(0, issued - kStages); i < issued; ++i)
                mbar_wait(&full[i % kStages], (i / kStages) & 1, p.err);
        return;
    }

    // ----------------------------------------------------------------------
    // Consumer warps.
    // ----------------------------------------------------------------------
    const int h0 = kvh * G;  // first query head of this KV head's group
    for (int i = threadIdx.x; i < G * D; i += kConsumers * 32) {
        const int r = i / D, c = i - (i / D) * D;
        const uint16_t bits = p.q[(size_t(b) * p.num_q_heads + h0 + r) * D + c];
        q_s[i] = __uint_as_float(uint32_t(bits) << 16) * p.qk_scale_log2;
    }
    named_sync(1, kConsumers * 32);

    float m_run[G], l_lane[G], o_acc[G][kDpl];
#pragma unroll
    for (int r = 0; r < G; ++r) {
        m_run[r] = -INFINITY;
        l_lane[r] = 0.f;
#pragma unroll
        for (int d = 0; d < kDpl; ++d) o_acc[r][d] = 0.f;
    }

    // P.V addressing: this lane's kDpl channels inside the swizzled V rows.
    const int pv_col = lane * kDpl;
    const int pv_box = pv_col / 64;
    const int pv_byte = (pv_col % 64) * 2;
    const int pv_chunk = pv_byte >> 4;
    const int pv_inner = pv_byte & 15;
    float *p_w = p_s + warp * kTile * G;

    for (int i = warp; i < ntiles; i += kConsumers) {
        const int s = i % kStages;
        if (!mbar_wait(&full[s], (i / kStages) & 1, p.err)) break;
        const uint8_t *ks = smem + s * S::kStageBytes;
        const uint8_t *vs = ks + S::kTileBytes;
        const int t0 = start + i * kTile;
        const int nvalid = min(kTile, end - t0);

        // ---- scores: lane j <-> key j --------------------------------------
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

        // ---- online softmax (base 2) ---------------------------------------
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
            *reinterpret_cast<float4 *>(p_w + lane * 4) = make_float4(pr[0], pr[1], pr[2], pr[3]);
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

        // ---- P.V: lane owns kDpl channels of every row ---------------------
        const uint8_t *vbase = vs + pv_box * kTile * 128 + pv_inner;
        for (int j = 0; j < nvalid; ++j) {
            const uint8_t *vr = vbase + j * 128 + ((pv_chunk ^ (j & 7)) << 4);
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
                const float4 t = *reinterpret_cast<const float4 *>(p_w + j * 4);
                pj[0] = t.x; pj[1] = t.y; pj[2] = t.z; pj[3] = t.w;
            } else {
#pragma unroll
                for (int r = 0; r < G; ++r) pj[r] = p_w[j * G + r];
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
        if (lane == 0) mbar_arrive(&empty[s]);
    }

    pdl_launch_dependents();

    // ---- merge the consumer warps' states ---------------------------------
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

    constexpr int kVec = 4;
    for (int idx = threadIdx.x; idx < G * D / kVec; idx += kConsumers * 32) {
        const int r = idx / (D / kVec);
        const int c0 = (idx - r * (D / kVec)) * kVec;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, m_s[w * G + r]);
        float l = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) {
            const float mw = m_s[w * G + r];
            if (mw == -INFINITY) continue;
            const float sc = fast_exp2(mw - M);
            l += sc * l_s[w * G + r];
            const float4 ow = *reinterpret_cast<const float4 *>(o_s + (w * G + r) * D + c0);
            o.x += sc * ow.x; o.y += sc * ow.y; o.z += sc * ow.z; o.w += sc * ow.w;
        }
        const int h = h0 + r;
        if (direct) {
            const float t2 = p.sink ? p.sink[h] * kLog2e : -INFINITY;
            const float Mf = fmaxf(M, t2);
            float Z = 0.f, so = 0.f;
            if (Mf != -INFINITY) {
                so = fast_exp2(M - Mf);
                Z = l * so + fast_exp2(t2 - Mf);
            }
            const float inv = Z > 0.f ? so / Z : 0.f;
            uint2 packed;
            packed.x = pack_bf16x2(o.x * inv, o.y * inv);
            packed.y = pack_bf16x2(o.z * inv, o.w * inv);
            *reinterpret_cast<uint2 *>(p.out + (size_t(b) * p.num_q_heads + h) * D + c0) = packed;
            if (c0 == 0 && p.lse)
                p.lse[size_t(b) * p.num_q_heads + h] =
                    Z > 0.f ? (Mf + fast_log2(Z)) * kLn2 : -INFINITY;
        } else {
            const size_t base = (size_t(part) * p.batch + b) * p.num_q_heads + h;
            *reinterpret_cast<float4 *>(p.ws_o + base * D + c0) = o;
            if (c0 == 0) {
                p.ws_m[base] = M * kLn2;
                p.ws_l[base] = l;
            }
        }
    }
}

template <int D, int G>
cudaError_t launch_t(const GqaParams &p, cudaStream_t stream) {
    constexpr size_t smem = gqa_smem_bytes<D, G>();
    auto kern = gqa_decode_kernel<D, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_partitions, p.num_q_heads / G, p.batch);
    kern<<<grid, kThreads, smem, stream>>>(p);
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
