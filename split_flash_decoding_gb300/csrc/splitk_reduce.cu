// splitk_reduce.cu -- log-sum-exp merge of split-K partials
// (mha_splitk_reduce / mla_splitk_reduce, mha_decoding_single_batch_pipelined
// summary and flare_mla_decoding_dispatch summary).
//
// One CTA of 256 threads per (row, head).  For partials (O_p unnormalised,
// m_p natural-log max, l_p exp-sum relative to m_p) and an optional sink
// logit t:
//   M = max(max_p m_p, t), w_p = exp(m_p - M), Z = sum_p w_p l_p + exp(t - M),
//   out = sum_p w_p O_p / Z,  lse = M + ln Z.
// The weights are computed once into shared memory; then thread t owns
// channel vector t % V (V = dv / 4 vectors, at most 256) of the partitions
// congruent to t / V, and the 256 / V partial sums are added in shared
// memory.  Partitions with m_p = -inf (empty slices) get weight 0 and their
// O_p is never read.
#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxP = 1024;   // ATTN_MAX_PARTITIONS

__device__ __forceinline__ float block_max(float v, float *red) {
    v = warp_max(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    v = red[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) v = fmaxf(v, red[i]);
    __syncthreads();
    return v;
}

__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    v = red[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) v += red[i];
    __syncthreads();
    return v;
}

__global__ void __launch_bounds__(kThreads)
splitk_reduce_kernel(const __grid_constant__ ReduceParams p) {
    // With programmatic dependent launch this grid may start while the
    // partition kernel is still running: wait for its writes first.
    pdl_wait_primary();

    __shared__ float w_s[kMaxP];
    __shared__ float red[kWarps];
    __shared__ float4 part[kThreads];

    const int row = blockIdx.x / p.num_q_heads;
    const int h = blockIdx.x - row * p.num_q_heads;
    const int tid = threadIdx.x;

    int P = p.num_partitions;
    if (p.kv_len) {
        // Rows that fit in one slice were finished by the partition kernel.
        const uint32_t cap = uint32_t(p.num_partitions) * uint32_t(p.chunk);
        const uint32_t L = min(p.kv_len[row], cap);
        const int ns = static_cast<int>((L + p.chunk - 1) / p.chunk);
        if (ns < 2) return;  // uniform over the CTA
        P = ns;
    }
    const size_t stride_p = static_cast<size_t>(p.rows) * p.num_q_heads;  // per partition
    const size_t idx0 = static_cast<size_t>(row) * p.num_q_heads + h;

    float mloc = -INFINITY;
    for (int q = tid; q < P; q += kThreads) mloc = fmaxf(mloc, p.ws_m[q * stride_p + idx0]);
    const float M = block_max(mloc, red);
    const float t = p.sink ? p.sink[h] : -INFINITY;
    const float Mf = fmaxf(M, t);

    float zloc = 0.f;
    for (int q = tid; q < P; q += kThreads) {
        const float m = p.ws_m[q * stride_p + idx0];
        float w = 0.f;
        if (m != -INFINITY) {
            w = fast_exp2((m - Mf) * kLog2e);
            zloc += w * p.ws_l[q * stride_p + idx0];
        }
        w_s[q] = w;
    }
    float Z = block_sum(zloc, red);   // also publishes w_s
    if (Mf != -INFINITY) Z += fast_exp2((t - Mf) * kLog2e);
    const float inv = Z > 0.f ? 1.f / Z : 0.f;

    const int V = min(p.dim_v / 4, kThreads);   // channel vectors handled at once
    const int lanes = kThreads / V;             // partition lanes
    const int v = tid % V;
    const int pl = tid / V;
    for (int c0 = 0; c0 < p.dim_v; c0 += V * 4) {
        const int c = c0 + v * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (pl < lanes && c < p.dim_v) {
#pragma unroll 4
            for (int q = pl; q < P; q += lanes) {
                const float w = w_s[q];
                if (w == 0.f) continue;
                const float4 o = *reinterpret_cast<const float4 *>(
                    p.ws_o + (q * stride_p + idx0) * p.dim_v + c);
                acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
            }
        }
        part[tid] = acc;
        __syncthreads();
        if (pl == 0 && c < p.dim_v) {
            for (int k = 1; k < lanes; ++k) {
                const float4 o = part[k * V + v];
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
    if (p.num_partitions > kMaxP || items > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(items));
    cfg.blockDim = dim3(kThreads);
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
