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

#include "attn_decode.h"

namespace {

// 32 MiB of split-K scratch: enough for batch 64 x 32 heads x head_dim 128
// with 16 partitions (about 17 MB).  Every GPU that loads the library holds
// this array until the process exits.
constexpr size_t kScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch in the current device's context.  In host
// code the name g_scratch is only a host-side stand-in, so the address is
// looked up with cudaGetSymbolAddress, with that device current.  It is
// looked up on every call (a host-side table lookup), so a device reset or
// a new primary context never leaves a stale address behind.
int scratch_address(void **out) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr)
        return ATTN_ERR_CUDA;
    *out = ptr;
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
    // The planner routes the call exactly as attn_decode does: single rows and
    // the few-row fold keep split-K (a non-zero P is taken as given, 0 plans
    // it), and longer row runs take the tile kernel, which does not split
    // (there a P above 1 is rejected).  It only does arithmetic (and, for
    // P = 0, reads the SM count); it allocates nothing.
    int P = 0;
    size_t need = 0;
    const int st = attn_plan_partitions(0, batch, num_q_rows, max_q_len, num_q_heads,
                                        num_q_heads / group, head_dim, max_kv_len,
                                        num_partitions, &P, &need);
    if (st != ATTN_OK) return st;
    if (need > kScratchBytes) return ATTN_ERR_WORKSPACE;  // beyond the fixed scratch
    void *scratch = nullptr;
    if (need > 0) {
        const int sa = scratch_address(&scratch);
        if (sa != ATTN_OK) return sa;
    }
    return attn_decode(q, k, v, kv_len, q_row_offsets, batch, num_q_rows, num_q_heads, group,
                       head_dim, max_q_len, max_kv_len, scale, sink, causal, P, scratch, need,
                       out, lse, stream);
}
