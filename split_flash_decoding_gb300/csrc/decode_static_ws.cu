// decode_static_ws.cu -- attn_decode_noalloc: attn_decode with its split-K
// workspace taken from a fixed array inside the library instead of from
// the caller.
//
// Who needs it: callers that cannot allocate device memory themselves --
// an inference-engine plugin that runs under a memory plan fixed at start-up,
// or a plain C program with no allocator at hand -- yet want split-K decode,
// whose partial results need scratch space.  The library holds that scratch
// in a file-scope __device__ array, so the call itself allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "attn_decode.h"

namespace {

// 32 MiB of split-K scratch: enough for batch 64 x 32 heads x head_dim 128
// with 16 partitions (about 17 MB).  Every GPU that loads the library holds
// this array until the process exits.
constexpr size_t kScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];

// Device address of g_scratch on the current device.  In host code the name
// g_scratch is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress, once per device, with that device current.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr)
            return ATTN_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return ATTN_OK;
}

}  // namespace

extern "C" int attn_decode_noalloc(const void *q, const attn_kv_t *k, const attn_kv_t *v,
                                   const uint32_t *kv_len, const uint32_t *q_row_offsets,
                                   int batch, int num_q_rows, int num_q_heads, int group,
                                   int head_dim, int max_q_len, int max_kv_len, float scale,
                                   const float *sink, int causal, int num_partitions, void *out,
                                   float *lse, attn_stream_t stream) {
    if (num_partitions < 0 || group <= 0 || num_q_heads <= 0 || num_q_heads % group)
        return ATTN_ERR_INVALID_ARG;
    int P = num_partitions;
    size_t need = 0;
    if (max_q_len > 1) {
        P = 1;  // the multi-row tile path does not split
    } else {
        // The planner only does arithmetic (and, for P = 0, reads the SM
        // count); it allocates nothing.
        const int st = attn_plan_partitions(0, batch, num_q_rows, num_q_heads,
                                            num_q_heads / group, head_dim, max_kv_len, P, &P,
                                            &need);
        if (st != ATTN_OK) return st;
    }
    if (need > kScratchBytes) return ATTN_ERR_WORKSPACE;  // beyond the fixed scratch
    void *scratch = nullptr;
    if (need > 0) {
        const int st = scratch_address(&scratch);
        if (st != ATTN_OK) return st;
    }
    return attn_decode(q, k, v, kv_len, q_row_offsets, batch, num_q_rows, num_q_heads, group,
                       head_dim, max_q_len, max_kv_len, scale, sink, causal, P, scratch, need,
                       out, lse, stream);
}
