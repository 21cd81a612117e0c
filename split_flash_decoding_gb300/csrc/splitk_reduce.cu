// splitk_reduce.cu -- log-sum-exp merge of split-K partials
// (mha_splitk_reduce / mla_splitk_reduce, mha_decoding_single_batch_pipelined
// summary and flare_mla_decoding_dispatch summary).
//
// Two shapes: for many (row, head) items, one warp per item (eight per CTA);
// for few items (a long-context batch of one), one CTA of eight warps per
// item with the partitions split across the warps.  For partials (O_p unnormalised,
// m_p natural-log max, l_p exp-sum relative to m_p) and an optional sink
// logit t:
//   M = max(max_p m_p, t), w_p = exp(m_p - M), Z = sum_p w_p l_p + exp(t - M),
//   out = sum_p w_p O_p / Z,  lse = M + ln Z.
// Lanes read the partition statistics in parallel, the weights go to the
// warp's slice of shared memory, and then each lane accumulates 4 channels
// per 128-channel stripe over all partitions with independent, unrolled
// loads.  Partitions with m_p = -inf (empty slices) get weight 0 and their
// O_p is never read.  The kernel is latency-bound (a few dependent rounds of
// global loads), so it issues everything it can at once.
#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxP = 1024;   // ATTN_MAX_PARTITIONS
constexpr int kFastP = 8;     // partitions merged in one round trip

// Sequence of query row `row`: the row itself, or found in the row offsets.
__device__ __forceinline__ int row_sequence(const ReduceParams &p, int row) {
    if (!p.q_row_offsets) return row;
    int lo = 0, hi = p.batch;   // off[lo] <= row < off[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (int(p.q_row_offsets[mid]) <= row) lo = mid; else hi = mid;
    }
    return lo;
}

// Where the partials of (row, h) are: returns their count P (-1: the row was
// finished by the partition kernel), the distance between consecutive
// partials and the index of the first, in units of one (row, head) entry.
__device__ __forceinline__ int locate_partials(const ReduceParams &p, int row, int h,
                                               size_t &stride_p, size_t &widx0) {
    int P = p.num_partitions;
    stride_p = static_cast<size_t>(p.rows) * p.num_q_heads;   // per partition
    widx0 = static_cast<size_t>(row) * p.num_q_heads + h;
    if (p.slots) {
        // Balanced MLA split: the row's partials sit in consecutive slots.
        const int2 e = p.slots[row];
        if (e.y == 1) return -1;   // finished by the decode kernel
        stride_p = p.num_q_heads;
        if (e.x < 0 || e.y < 0 || e.y > p.num_slots - e.x) return 0;
        widx0 = static_cast<size_t>(e.x) * p.num_q_heads + h;
        return e.y;                // 0: an empty row, written from the sink alone
    }
    if (p.unit_slots) {
        // Balanced GQA split: the unit's partials sit in consecutive slots of
        // 16 columns (query row within the sequence x head within the group).
        const int b = row_sequence(p, row);
        const int first_row = p.q_row_offsets ? int(p.q_row_offsets[b]) : b;
        const int2 e = p.unit_slots[b * p.hkv + h / p.group];
        if (e.y == 1) return -1;
        stride_p = kGqaSlotCols;
        widx0 = static_cast<size_t>(e.x) * kGqaSlotCols + (row - first_row) * p.group + h % p.group;
        return e.y;
    }
    if (p.kv_len) {
        // Rows that fit in one slice were finished by the partition kernel.
        uint32_t cap = uint32_t(p.num_partitions) * uint32_t(p.chunk);
        if (p.len_cap > 0) cap = min(cap, uint32_t(p.len_cap));
        const uint32_t L = min(p.kv_len[row_sequence(p, row)], cap);
        const int ns = static_cast<int>((L + p.chunk - 1) / p.chunk);
        return ns < 2 ? -1 : ns;
    }
    return P;
}

__global__ void __launch_bounds__(kWarps * 32)
splitk_reduce_kernel(const __grid_constant__ ReduceParams p) {
    // With programmatic dependent launch this grid may start while the
    // partition kernel is still running: wait for its writes first.
    pdl_wait_primary();

    __shared__ float w_s[kWarps][kMaxP / 4];   // weights, up to 256 partitions per warp
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long item = static_cast<long long>(blockIdx.x) * kWarps + warp;
    if (item >= static_cast<long long>(p.rows) * p.num_q_heads) return;
    const int row = static_cast<int>(item / p.num_q_heads);
    const int h = static_cast<int>(item - static_cast<long long>(row) * p.num_q_heads);

    const size_t idx0 = static_cast<size_t>(row) * p.num_q_heads + h;  // out / lse
    size_t stride_p, widx0;                                            // workspace
    const int P = locate_partials(p, row, h, stride_p, widx0);
    if (P < 0) return;   // uniform over the warp

    if (P <= kFastP) {
        // Few partitions: the O partials of the first channel block, m and l
        // are all requested at once (one round trip), and lane q's weight
        // reaches the other lanes by shuffle.
        const float m_lane = lane < P ? p.ws_m[lane * stride_p + widx0] : -INFINITY;
        const float l_lane = lane < P ? p.ws_l[lane * stride_p + widx0] : 0.f;
        const float *src0 = p.ws_o + widx0 * p.dim_v + lane * 4;
        const size_t step = stride_p * p.dim_v;
        float4 o[kFastP];
#pragma unroll
        for (int q = 0; q < kFastP; ++q)
            if (q < P && lane * 4 < p.dim_v)
                o[q] = *reinterpret_cast<const float4 *>(src0 + q * step);
        const float t = p.sink ? p.sink[h] : -INFINITY;
        const float Mf = fmaxf(warp_max(m_lane), t);
        const float w_lane = m_lane == -INFINITY ? 0.f : fast_exp2((m_lane - Mf) * kLog2e);
        float Z = warp_sum(w_lane * l_lane);
        if (Mf != -INFINITY) Z += fast_exp2((t - Mf) * kLog2e);
        const float inv = Z > 0.f ? 1.f / Z : 0.f;
        for (int c = lane * 4; c < p.dim_v; c += 128) {
            if (c != lane * 4) {
#pragma unroll
                for (int q = 0; q < kFastP; ++q)
                    if (q < P) o[q] = *reinterpret_cast<const float4 *>(src0 + (c - lane * 4) + q * step);
            }
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < kFastP; ++q) {
                const float w = __shfl_sync(0xffffffffu, w_lane, q);
                if (q < P && w != 0.f) {
                    acc.x += w * o[q].x; acc.y += w * o[q].y;
                    acc.z += w * o[q].z; acc.w += w * o[q].w;
                }
            }
            uint2 packed;
            packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
            packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2 *>(p.out + idx0 * p.dim_v + c) = packed;
        }
        if (lane == 0 && p.lse) p.lse[idx0] = Z > 0.f ? Mf + fast_log2(Z) * kLn2 : -INFINITY;
        return;
    }

    float mloc = -INFINITY;
    for (int q = lane; q < P; q += 32) mloc = fmaxf(mloc, p.ws_m[q * stride_p + widx0]);
    const float M = warp_max(mloc);
    const float t = p.sink ? p.sink[h] : -INFINITY;
    const float Mf = fmaxf(M, t);

    // Weights: kept in shared memory when P fits the warp's slice, otherwise
    // recomputed in the channel loop.
    const bool cached = P <= kMaxP / 4;
    float zloc = 0.f;
    for (int q = lane; q < P; q += 32) {
        const float m = p.ws_m[q * stride_p + widx0];
        float w = 0.f;
        if (m != -INFINITY) {
            w = fast_exp2((m - Mf) * kLog2e);
            zloc += w * p.ws_l[q * stride_p + widx0];
        }
        if (cached) w_s[warp][q] = w;
    }
    __syncwarp();
    float Z = warp_sum(zloc);
    if (Mf != -INFINITY) Z += fast_exp2((t - Mf) * kLog2e);
    const float inv = Z > 0.f ? 1.f / Z : 0.f;

    for (int c = lane * 4; c < p.dim_v; c += 128) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float *src = p.ws_o + widx0 * p.dim_v + c;
#pragma unroll 8
        for (int q = 0; q < P; ++q) {
            float w;
            if (cached) {
                w = w_s[warp][q];
            } else {
                const float m = p.ws_m[q * stride_p + widx0];
                w = m == -INFINITY ? 0.f : fast_exp2((m - Mf) * kLog2e);
            }
            if (w == 0.f) continue;
            const float4 o = *reinterpret_cast<const float4 *>(src + q * stride_p * p.dim_v);
            acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
        }
        uint2 packed;
        packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2 *>(p.out + idx0 * p.dim_v + c) = packed;
    }
    if (lane == 0 && p.lse) p.lse[idx0] = Z > 0.f ? Mf + fast_log2(Z) * kLn2 : -INFINITY;
}

// Few items: CTA per (row, head); warp w takes partitions q = w, w + 8, ...
__global__ void __launch_bounds__(kWarps * 32)
splitk_reduce_wide_kernel(const __grid_constant__ ReduceParams p) {
    pdl_wait_primary();

    __shared__ float w_s[kMaxP];
    __shared__ float red[kWarps];
    __shared__ float4 part[kWarps][32];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tid = threadIdx.x;
    const int row = blockIdx.x / p.num_q_heads;
    const int h = blockIdx.x - row * p.num_q_heads;

    const size_t idx0 = static_cast<size_t>(row) * p.num_q_heads + h;
    size_t stride_p, widx0;
    const int P = locate_partials(p, row, h, stride_p, widx0);
    if (P < 0) return;   // uniform over the CTA

    float mloc = -INFINITY;
    for (int q = tid; q < P; q += kWarps * 32) mloc = fmaxf(mloc, p.ws_m[q * stride_p + widx0]);
    mloc = warp_max(mloc);
    if (lane == 0) red[warp] = mloc;
    __syncthreads();
    float M = red[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) M = fmaxf(M, red[i]);
    __syncthreads();
    const float t = p.sink ? p.sink[h] : -INFINITY;
    const float Mf = fmaxf(M, t);

    float zloc = 0.f;
    for (int q = tid; q < P; q += kWarps * 32) {
        const float m = p.ws_m[q * stride_p + widx0];
        float w = 0.f;
        if (m != -INFINITY) {
            w = fast_exp2((m - Mf) * kLog2e);
            zloc += w * p.ws_l[q * stride_p + widx0];
        }
        w_s[q] = w;
    }
    zloc = warp_sum(zloc);
    if (lane == 0) red[warp] = zloc;
    __syncthreads();   // also publishes w_s
    float Z = 0.f;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) Z += red[i];
    if (Mf != -INFINITY) Z += fast_exp2((t - Mf) * kLog2e);
    const float inv = Z > 0.f ? 1.f / Z : 0.f;

    for (int c0 = 0; c0 < p.dim_v; c0 += 128) {
        const int c = c0 + lane * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < p.dim_v) {
            const float *src = p.ws_o + widx0 * p.dim_v + c;
#pragma unroll 4
            for (int q = warp; q < P; q += kWarps) {
                const float w = w_s[q];
                if (w == 0.f) continue;
                const float4 o = *reinterpret_cast<const float4 *>(src + q * stride_p * p.dim_v);
                acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
            }
        }
        part[warp][lane] = acc;
        __syncthreads();
        if (warp == 0 && c < p.dim_v) {
            for (int k = 1; k < kWarps; ++k) {
                const float4 o = part[k][lane];
                acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
            }
            uint2 packed;
            packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
            packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2 *>(p.out + idx0 * p.dim_v + c) = packed;
        }
        __syncthreads();
    }
    if (tid == 0 && p.lse) p.lse[idx0] = Z > 0.f ? Mf + fast_log2(Z) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_splitk_reduce(const ReduceParams &p, cudaStream_t stream, bool pdl) {
    const long long items = static_cast<long long>(p.rows) * p.num_q_heads;
    if (items == 0) return cudaSuccess;
    if (p.num_partitions > kMaxP) return cudaErrorInvalidValue;
    // Fewer items than about two warps per SM: spread each item over a CTA.
    const bool wide = items <= 256;
    const long long blocks = wide ? items : (items + kWarps - 1) / kWarps;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return wide ? cudaLaunchKernelEx(&cfg, splitk_reduce_wide_kernel, p)
                : cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, p);
}

}  // namespace attn
