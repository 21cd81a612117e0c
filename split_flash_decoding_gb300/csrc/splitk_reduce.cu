// splitk_reduce.cu -- log-sum-exp merge of split-K partials
// (mha_splitk_reduce / mla_splitk_reduce, mha_decoding_single_batch_pipelined
// summary and flare_mla_decoding_dispatch summary).
//
// One warp per (row, head).  For partials (O_p unnormalised, m_p natural-log
// max, l_p exp-sum relative to m_p) and an optional sink logit t:
//   M = max(max_p m_p, t), w_p = exp(m_p - M), Z = sum_p w_p l_p + exp(t - M),
//   out = sum_p w_p O_p / Z,  lse = M + ln Z.
// Lanes own 4 consecutive channels per 128-channel stripe; partitions with
// m_p = -inf (empty slices) are skipped, so their O_p is never read.
#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kWarps = 4;

__global__ void __launch_bounds__(kWarps * 32)
splitk_reduce_kernel(const __grid_constant__ ReduceParams p) {
    // With programmatic dependent launch this grid may start while the
    // partition kernel is still running: wait for its writes first.
    pdl_wait_primary();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long item = static_cast<long long>(blockIdx.x) * kWarps + warp;
    if (item >= static_cast<long long>(p.rows) * p.num_q_heads) return;
    const int row = static_cast<int>(item / p.num_q_heads);
    const int h = static_cast<int>(item - static_cast<long long>(row) * p.num_q_heads);

    int P = p.num_partitions;
    if (p.kv_len) {
        // Rows that fit in one slice were finished by the partition kernel.
        const uint32_t cap = uint32_t(p.num_partitions) * uint32_t(p.chunk);
        const uint32_t L = min(p.kv_len[row], cap);
        const int ns = static_cast<int>((L + p.chunk - 1) / p.chunk);
        if (ns < 2) return;
        P = ns;
    }
    const size_t stride_p = static_cast<size_t>(p.rows) * p.num_q_heads;  // per partition
    const size_t idx0 = static_cast<size_t>(row) * p.num_q_heads + h;

    float M = -INFINITY;
    for (int q = lane; q < P; q += 32) M = fmaxf(M, p.ws_m[q * stride_p + idx0]);
    M = warp_max(M);
    const float t = p.sink ? p.sink[h] : -INFINITY;
    const float Mf = fmaxf(M, t);

    float Z = 0.f;
    if (Mf != -INFINITY) {
        for (int q = lane; q < P; q += 32) {
            const float m = p.ws_m[q * stride_p + idx0];
            if (m != -INFINITY) Z += fast_exp2((m - Mf) * kLog2e) * p.ws_l[q * stride_p + idx0];
        }
    }
    Z = warp_sum(Z);
    if (Mf != -INFINITY) Z += fast_exp2((t - Mf) * kLog2e);
    const float inv = Z > 0.f ? 1.f / Z : 0.f;

    for (int c0 = lane * 4; c0 < p.dim_v; c0 += 128) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (Mf != -INFINITY) {
            for (int q = 0; q < P; ++q) {
                const float m = p.ws_m[q * stride_p + idx0];
                if (m == -INFINITY) continue;
                const float w = fast_exp2((m - Mf) * kLog2e);
                const float4 o = *reinterpret_cast<const float4 *>(
                    p.ws_o + (q * stride_p + idx0) * p.dim_v + c0);
                acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
            }
        }
        uint2 packed;
        packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2 *>(p.out + idx0 * p.dim_v + c0) = packed;
    }
    if (lane == 0 && p.lse) p.lse[idx0] = Z > 0.f ? Mf + fast_log2(Z) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_splitk_reduce(const ReduceParams &p, cudaStream_t stream, bool pdl) {
    const long long items = static_cast<long long>(p.rows) * p.num_q_heads;
    if (items == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((items + kWarps - 1) / kWarps));
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, p);
}

}  // namespace attn
