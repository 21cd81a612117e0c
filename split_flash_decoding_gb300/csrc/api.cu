// api.cu -- the extern "C" entry points of libattn.so (declared in
// include/attn_decode.h): host-side validation, the split-K partition
// planner, TMA tensor-map encoding and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn_decode.h"
#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace {

// Device error word written by kernels instead of trapping or hanging.
__device__ unsigned g_error_word;

// Address of g_error_word in the current device's context.  Looked up on
// every call (a host-side table lookup, far cheaper than a launch), so a
// device reset or a new primary context never leaves a stale address behind.
int error_word(unsigned **out) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_error_word) != cudaSuccess || ptr == nullptr)
        return ATTN_ERR_CUDA;
    *out = static_cast<unsigned *>(ptr);
    return ATTN_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 4-D map over a cache operand: (channel, slot in page, kv head, page) with a
// box of box_ch channels x box_rows slots x 1 x 1: 64 channels (128 B) with
// the 128-byte swizzle, or 32 channels (64 B) with the 64-byte swizzle.
int encode_kv_map(CUtensorMap *map, const attn_kv_t &kv, int dim, int num_kv_heads,
                  int box_rows, int box_ch = 64) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return ATTN_ERR_CUDA;
    cuuint64_t gdim[4] = {cuuint64_t(dim), cuuint64_t(kv.page_size), cuuint64_t(num_kv_heads),
                          cuuint64_t(kv.num_pages)};
    cuuint64_t gstride[3] = {cuuint64_t(kv.token_stride) * 2, cuuint64_t(kv.head_stride) * 2,
                             cuuint64_t(kv.page_stride) * 2};
    cuuint32_t box[4] = {cuuint32_t(box_ch), cuuint32_t(box_rows), 1, 1};
    cuuint32_t estride[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(kv.base), gdim,
                    gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    box_ch == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_UNSUPPORTED;
}

bool is_pow2(long long x) { return x > 0 && (x & (x - 1)) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// GQA decode on the tensor cores (head_dim 128) with 2 or 4 partitions
// merges them on chip (a cluster of P CTAs) and needs no workspace.
bool merges_on_chip(int P, int head_dim) { return head_dim == 128 && (P == 2 || P == 4); }

// A few query rows per sequence (head_dim 128, max_q_len * group <= 16)
// fold onto the N side of the tensor-core decode kernel, next to the group's
// heads, and keep its split-K; longer row runs take the tile kernel.
bool folds_rows(int max_q_len, int head_dim, int group, int batch) {
    return max_q_len > 1 && head_dim == 128 && max_q_len * group <= 16 && batch <= kGqaMaxBatch;
}

// Workspace layout for P partitions: ws_o | ws_m | ws_l, each 256-B aligned.
size_t workspace_layout(int P, long long rows, int hq, int dv, size_t *off_m, size_t *off_l) {
    if (P <= 1) {
        if (off_m) *off_m = 0;
        if (off_l) *off_l = 0;
        return 0;
    }
    const size_t n = size_t(P) * size_t(rows) * size_t(hq);
    const size_t o_bytes = align256(n * size_t(dv) * sizeof(float));
    const size_t m_bytes = align256(n * sizeof(float));
    if (off_m) *off_m = o_bytes;
    if (off_l) *off_l = o_bytes + m_bytes;
    return o_bytes + 2 * m_bytes;
}

// Balanced MLA split: fp32 partials for clusters + rows slots, then the
// reduce's table (per row: its first slot and partials).
size_t mla_balanced_layout(int clusters, long long rows, size_t *off_m, size_t *off_l,
                           size_t *off_plan) {
    const size_t n = (size_t(clusters) + size_t(rows)) * size_t(kMlaHeads);
    const size_t o_bytes = align256(n * size_t(kMlaDimV) * sizeof(float));
    const size_t m_bytes = align256(n * sizeof(float));
    if (off_m) *off_m = o_bytes;
    if (off_l) *off_l = o_bytes + m_bytes;
    if (off_plan) *off_plan = o_bytes + 2 * m_bytes;
    return o_bytes + 2 * m_bytes + align256(size_t(rows) * 8);
}

// Balanced GQA split: partial slots (CTAs + units) of 16 columns x 128
// channels, m and l per column, then the unit table {first slot, pieces}.
size_t gqa_balanced_layout(int ctas, long long units, size_t *off_m, size_t *off_l,
                           size_t *off_table) {
    const size_t n = (size_t(ctas) + size_t(units)) * size_t(kGqaSlotCols);
    const size_t o_bytes = align256(n * 128 * sizeof(float));
    const size_t m_bytes = align256(n * sizeof(float));
    if (off_m) *off_m = o_bytes;
    if (off_l) *off_l = o_bytes + m_bytes;
    if (off_table) *off_table = o_bytes + 2 * m_bytes;
    return o_bytes + 2 * m_bytes + align256(size_t(units) * 8);
}

int chunk_for(int max_kv_len, int P, int tile) {
    long long per = (static_cast<long long>(max_kv_len) + P - 1) / P;
    if (per < 1) per = 1;
    per = (per + tile - 1) / tile * tile;
    return static_cast<int>(per);
}

// Validate one cache operand.  contiguous (no page table) means page b is
// sequence b and page_size bounds every length.
int check_kv(const attn_kv_t *kv, int batch, int dim, int max_kv_len) {
    if (!kv || !kv->base) return ATTN_ERR_INVALID_ARG;
    if (kv->reserved != 0) return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(kv->base) % 16) return ATTN_ERR_INVALID_ARG;
    if (kv->page_size <= 0 || kv->num_pages <= 0) return ATTN_ERR_INVALID_ARG;
    if (kv->token_stride <= 0 || kv->head_stride <= 0 || kv->page_stride <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (kv->token_stride % 8 || kv->head_stride % 8 || kv->page_stride % 8)
        return ATTN_ERR_INVALID_ARG;
    if (kv->head_stride < dim && kv->token_stride < dim) return ATTN_ERR_INVALID_ARG;
    if (kv->page_table) {
        if (!is_pow2(kv->page_size) || kv->page_size < 8) return ATTN_ERR_UNSUPPORTED;
        if (kv->max_pages <= 0) return ATTN_ERR_INVALID_ARG;
        const long long need = (static_cast<long long>(max_kv_len) + kv->page_size - 1) /
                               kv->page_size;
        if (need > kv->max_pages) return ATTN_ERR_INVALID_ARG;
    } else {
        if (kv->page_size < max_kv_len) return ATTN_ERR_INVALID_ARG;
        if (kv->num_pages < batch) return ATTN_ERR_INVALID_ARG;
    }
    return ATTN_OK;
}

int map_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

// Failure-path self-test: an mbarrier that nothing ever arrives on, waited on
// with the same bounded wait the kernels use.  The wait gives up after its
// time limit and sets the timeout bit of the error word; the kernel then
// returns normally.
__global__ void selftest_wait_kernel(unsigned *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, err);
}

int prefill_path(const void *q, const attn_kv_t *k, const attn_kv_t *v, const uint32_t *kv_len,
                 const uint32_t *q_row_offsets, int batch, int num_q_rows, int num_q_heads,
                 int group, int head_dim, int max_q_len, int max_kv_len, float scale,
                 const float *sink, int causal, int num_partitions, void *out, float *lse,
                 attn_stream_t stream);

}  // namespace
}  // namespace attn


namespace attn {
namespace {

int prefill_path(const void *q, const attn_kv_t *k, const attn_kv_t *v, const uint32_t *kv_len,
                 const uint32_t *q_row_offsets, int batch, int num_q_rows, int num_q_heads,
                 int group, int head_dim, int max_q_len, int max_kv_len, float scale,
                 const float *sink, int causal, int num_partitions, void *out, float *lse,
                 attn_stream_t stream) {
    if (head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    if (group != 1 && group != 2 && group != 4 && group != 8) return ATTN_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(out) % 16 || reinterpret_cast<uintptr_t>(q) % 16)
        return ATTN_ERR_INVALID_ARG;
    const int hkv = num_q_heads / group;
    int st = check_kv(k, batch, head_dim, max_kv_len);
    if (st) return st;
    st = check_kv(v, batch, head_dim, max_kv_len);
    if (st) return st;
    if (k->page_table != v->page_table || k->page_size != v->page_size ||
        k->max_pages != v->max_pages || k->num_pages != v->num_pages)
        return ATTN_ERR_UNSUPPORTED;

    // num_partitions 0 (automatic) and 1 take one Q tile per CTA, measured
    // faster than two Q tiles per CTA pair on every shape tried (1.43-1.51x:
    // the pair runs each tile in lockstep across two SMs);
    // ATTN_PARTITIONS_TILE_PAIR asks for the pair.
    const bool pair = num_partitions == ATTN_PARTITIONS_TILE_PAIR;
    TileParams p;
    std::memset(&p, 0, sizeof(p));
    const int ps = k->page_table ? k->page_size : kTileKeys;
    p.box_rows = ps < kTileKeys ? ps : kTileKeys;
    p.box_rows_v = p.box_rows;
    if (pair) p.box_rows = ps < 64 ? ps : 64;   // the K half of a pair: 64 keys
    st = encode_kv_map(&p.k_map, *k, head_dim, hkv, p.box_rows);
    if (st) return st;
    st = encode_kv_map(&p.v_map, *v, head_dim, hkv, p.box_rows_v);
    if (st) return st;
    const int tokens = kTileRows / group;
    {
        EncodeTiledFn fn = encode_fn();
        if (!fn) return ATTN_ERR_CUDA;
        cuuint64_t gdim[4] = {128, cuuint64_t(group), cuuint64_t(hkv), cuuint64_t(num_q_rows)};
        cuuint64_t gstride[3] = {128 * 2, cuuint64_t(group) * 128 * 2,
                                 cuuint64_t(num_q_heads) * 128 * 2};
        cuuint32_t box[4] = {64, cuuint32_t(group), 1, cuuint32_t(tokens)};
        cuuint32_t estride[4] = {1, 1, 1, 1};
        CUresult r = fn(&p.q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(q),
                        gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return ATTN_ERR_UNSUPPORTED;
    }
    st = error_word(&p.err);
    if (st) return st;
    p.kv_len = kv_len;
    p.q_row_offsets = q_row_offsets;
    p.page_table = k->page_table;
    p.sink = sink;
    p.out = static_cast<uint16_t *>(out);
    p.lse = lse;
    p.batch = batch;
    p.num_q_rows = num_q_rows;
    p.num_q_heads = num_q_heads;
    p.group = group;
    p.max_pages = k->max_pages;
    p.page_size = k->page_size;
    p.num_pages = k->num_pages;
    p.causal = causal ? 1 : 0;
    p.tiles_per_seq = (max_q_len + tokens - 1) / tokens;
    p.qk_scale_log2 = scale * 1.4426950408889634f;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return map_cuda(pair ? launch_tile_attention_pair(p, s) : launch_tile_attention(p, s));
}

}  // namespace
}  // namespace attn

using namespace attn;

namespace attn {
namespace {

// The partition plan behind attn_plan_partitions and the automatic choice of
// attn_decode (num_partitions 0).  The one place that decides which GQA
// kernel a call with max_q_len rows per sequence takes: single rows and the
// few-row fold run split-K on the decode kernel, longer row runs take the
// tile kernel, which does not split (P = 1, no workspace).
int plan_impl(int num_sms, int batch, int num_q_rows, int max_q_len, int num_q_heads,
              int num_kv_heads, int head_dim_v, int max_kv_len, int requested,
              int *num_partitions, size_t *workspace_bytes) {
    if (!num_partitions || !workspace_bytes) return ATTN_ERR_INVALID_ARG;
    if (batch < 0 || num_q_rows < 0 || max_q_len < 1 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        head_dim_v <= 0 || max_kv_len < 0 || requested < ATTN_PARTITIONS_TILE_PAIR)
        return ATTN_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads) return ATTN_ERR_INVALID_ARG;
    if (requested > ATTN_MAX_PARTITIONS) return ATTN_ERR_INVALID_ARG;
    const bool mla_shape = num_kv_heads == 1 && head_dim_v == kMlaDimV;
    const bool tile_path = !mla_shape && max_q_len > 1 &&
                           !folds_rows(max_q_len, head_dim_v, num_q_heads / num_kv_heads, batch);
    // the split-K route on the tensor cores (head_dim 128): single rows and
    // the few-row fold
    const bool gqa_tc = !mla_shape && !tile_path && head_dim_v == 128;
    if (requested == ATTN_PARTITIONS_BALANCED && !mla_shape && !gqa_tc)
        return ATTN_ERR_INVALID_ARG;
    if (requested == ATTN_PARTITIONS_TILE_PAIR && !tile_path) return ATTN_ERR_INVALID_ARG;
    if (tile_path) {
        // the tile kernels: every row run in one pass, no split-K; one Q tile
        // per CTA unless two per CTA pair are asked for
        if (requested > 1) return ATTN_ERR_UNSUPPORTED;
        *num_partitions = requested == ATTN_PARTITIONS_TILE_PAIR ? requested : 1;
        *workspace_bytes = 0;
        return ATTN_OK;
    }
    if (requested <= 0 && num_sms <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    const long long gqa_units = static_cast<long long>(batch > 0 ? batch : 1) * num_kv_heads;
    if (requested == ATTN_PARTITIONS_BALANCED && gqa_tc) {
        *num_partitions = ATTN_PARTITIONS_BALANCED;
        *workspace_bytes = gqa_balanced_layout(num_sms, gqa_units, nullptr, nullptr, nullptr);
        return ATTN_OK;
    }
    if (requested == ATTN_PARTITIONS_BALANCED) {
        *num_partitions = 0;
        *workspace_bytes = mla_balanced_layout(num_sms / 2 > 0 ? num_sms / 2 : 1,
                                               num_q_rows > 0 ? num_q_rows : 1, nullptr, nullptr,
                                               nullptr);
        return ATTN_OK;
    }
    if (requested == 0 && gqa_tc && gqa_units <= 8LL * num_sms &&
        max_kv_len > kGqaTcTileKeys) {
        // Up to eight (sequence, KV head) units per SM: every unit's 128-key
        // tiles, concatenated, are dealt out in contiguous ranges of equal
        // cost, one per SM, so ragged lengths cannot leave SMs idle and only the units a
        // range end cuts leave partials for the reduce (measured faster than
        // the slice plans at 16 to 64 sequences of Llama-3-8B shapes, single
        // or a few rows).  The workspace grows by ~8 KB per unit, so larger
        // batches keep the slice plans below.
        *num_partitions = ATTN_PARTITIONS_BALANCED;
        *workspace_bytes = gqa_balanced_layout(num_sms, gqa_units, nullptr, nullptr, nullptr);
        return ATTN_OK;
    }
    int P = requested;
    if (P == 0) {
        // GQA runs a persistent grid over (sequence, KV head, slice) items,
        // one CTA per SM for head_dim 128 (tensor cores) and two for
        // head_dim 64.  GQA with fewer (sequence, KV head) units than CTAs
        // gets one slice per CTA (one wave), as if every sequence had
        // max_kv_len keys.  Otherwise P is at least what gives every CTA four
        // items at full length and at least max_kv_len / 1024, which keeps a
        // ragged batch balanced; when it does not cost more than doubling P,
        // P is rounded up so that units * P is a multiple of the CTA count.
        // MLA: the fixed-slice count P' is the larger of ~4096 keys per slice
        // and as many slices per row as one wave of two-CTA clusters holds.
        // It only decides whether to split: P' = 1 keeps one unsplit slice
        // per row (no partials, no reduce), and anything larger becomes the
        // balanced split (P = 0), which deals all rows' tiles out evenly to
        // one wave of clusters instead of P' slices per row.
        const bool mla = num_kv_heads == 1 && head_dim_v == kMlaDimV;
        const bool tc = !mla && head_dim_v == 128;   // tensor-core decode: one CTA per SM
        // MLA runs a cluster per query row; GQA folds a sequence's rows
        const long long units =
            mla ? (num_q_rows > 0 ? num_q_rows : 1)
                : static_cast<long long>(batch > 0 ? batch : 1) * num_kv_heads;
        const long long ctas = mla ? (num_sms / 2 > 0 ? num_sms / 2 : 1)
                                   : (tc ? num_sms : 2LL * num_sms);
        // MLA: ~4096 keys per slice and query row, so a sequence with n rows
        // (n clusters per slice) gets n times longer slices
        const long long rows_per_seq =
            batch > 0 && num_q_rows > batch ? (num_q_rows + batch - 1) / batch : 1;
        const long long target = mla ? 4096 * rows_per_seq : 1024;
        long long p;
        if (mla) {
            const long long p_fill = ctas / units > 0 ? ctas / units : 1;
            const long long p_len = (static_cast<long long>(max_kv_len) + target - 1) / target;
            p = p_fill > p_len ? p_fill : p_len;
        } else if (tc && max_q_len > 1 && units >= 2 * ctas) {
            // A few query rows per sequence fold onto 16 score columns.  With
            // two units per CTA or more the split buys little (the memory
            // streams are already spread over every SM) and costs a
            // workspace and a reduce: one slice per unit.  With fewer units
            // the folded items are long, and the many-item rule below (not
            // one wave of slices) keeps a ragged batch balanced.
            p = 1;
        } else if (units < ctas && !(tc && max_q_len > 1)) {
            p = (ctas + units - 1) / units;
        } else {
            const long long p_fill = (4 * ctas + units - 1) / units;
            const long long p_len = (static_cast<long long>(max_kv_len) + target - 1) / target;
            p = p_fill > p_len ? p_fill : p_len;
            long long g = ctas, u = units;   // q = ctas / gcd(ctas, units)
            while (u) { const long long r = g % u; g = u; u = r; }
            const long long q = ctas / g;
            const long long aligned = (p + q - 1) / q * q;
            if (aligned <= 2 * p) p = aligned;
        }
        const long long tile = mla ? kMlaTileKeys : (tc ? kGqaTcTileKeys : kGqaTileKeys);
        const long long p_max_useful = (static_cast<long long>(max_kv_len) + tile - 1) / tile;
        if (p > p_max_useful) p = p_max_useful;
        if (p < 1) p = 1;
        if (p > ATTN_MAX_PARTITIONS) p = ATTN_MAX_PARTITIONS;
        P = static_cast<int>(p);
        if (mla && P > 1) {
            // MLA keys that need splitting at all take the balanced split over
            // one wave of two-CTA clusters instead of P slices per row.
            *num_partitions = 0;
            *workspace_bytes = mla_balanced_layout(num_sms / 2 > 0 ? num_sms / 2 : 1,
                                                   num_q_rows > 0 ? num_q_rows : 1, nullptr,
                                                   nullptr, nullptr);
            return ATTN_OK;
        }
    }
    *num_partitions = P;
    const bool gqa = !(num_kv_heads == 1 && head_dim_v == kMlaDimV);
    *workspace_bytes = gqa && merges_on_chip(P, head_dim_v)
                           ? 0
                           : workspace_layout(P, num_q_rows, num_q_heads, head_dim_v, nullptr,
                                              nullptr);
    return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" int attn_plan_partitions(int num_sms, int batch, int num_q_rows, int max_q_len,
                                    int num_q_heads, int num_kv_heads, int head_dim_v,
                                    int max_kv_len, int requested, int *num_partitions,
                                    size_t *workspace_bytes) {
    return plan_impl(num_sms, batch, num_q_rows, max_q_len, num_q_heads, num_kv_heads,
                     head_dim_v, max_kv_len, requested, num_partitions, workspace_bytes);
}

extern "C" int attn_decode(const void *q, const attn_kv_t *k, const attn_kv_t *v,
                           const uint32_t *kv_len, const uint32_t *q_row_offsets, int batch,
                           int num_q_rows, int num_q_heads, int group, int head_dim,
                           int max_q_len, int max_kv_len, float scale, const float *sink,
                           int causal, int num_partitions, void *workspace,
                           size_t workspace_bytes, void *out, float *lse, attn_stream_t stream) {
    if (batch < 0 || num_q_rows < 0 || num_q_heads <= 0 || group <= 0 || max_kv_len < 0 ||
        max_q_len < 1)
        return ATTN_ERR_INVALID_ARG;
    if (num_q_heads % group) return ATTN_ERR_INVALID_ARG;
    if ((num_partitions < 0 && num_partitions != ATTN_PARTITIONS_TILE_PAIR &&
         num_partitions != ATTN_PARTITIONS_BALANCED) ||
        num_partitions > ATTN_MAX_PARTITIONS)
        return ATTN_ERR_INVALID_ARG;
    if (!(scale == scale)) return ATTN_ERR_INVALID_ARG;
    if (!q_row_offsets && (num_q_rows != batch || max_q_len != 1)) return ATTN_ERR_INVALID_ARG;
    if (batch == 0 || num_q_rows == 0) return ATTN_OK;
    if (!q || !kv_len || !out) return ATTN_ERR_INVALID_ARG;
    // A few rows per sequence fold onto the N side of the tensor-core decode
    // kernel, split-K included; longer row runs take the tile path (not split).
    const bool fold = folds_rows(max_q_len, head_dim, group, batch);
    if (num_partitions == ATTN_PARTITIONS_TILE_PAIR && !(max_q_len > 1 && !fold))
        return ATTN_ERR_INVALID_ARG;   // the pair of Q tiles is a tile-path request
    if (num_partitions == ATTN_PARTITIONS_BALANCED && ((max_q_len > 1 && !fold) || head_dim != 128))
        return ATTN_ERR_INVALID_ARG;   // the balanced split is a split-K route on the tensor cores
    if (max_q_len > 1 && !fold) {
        if (num_partitions > 1) return ATTN_ERR_UNSUPPORTED;
        return prefill_path(q, k, v, kv_len, q_row_offsets, batch, num_q_rows, num_q_heads,
                            group, head_dim, max_q_len, max_kv_len, scale, sink, causal,
                            num_partitions, out, lse, stream);
    }
    if (num_partitions == 0) {
        // automatic: the planner's choice for this shape on the current device
        size_t planned = 0;
        const int st = plan_impl(0, batch, num_q_rows, max_q_len, num_q_heads,
                                 num_q_heads / group, head_dim, max_kv_len, 0, &num_partitions,
                                 &planned);
        if (st) return st;
    }
    if (!fold && q_row_offsets && num_q_rows != batch) return ATTN_ERR_INVALID_ARG;
    if (batch > kGqaMaxBatch) return ATTN_ERR_UNSUPPORTED;
    if (group != 1 && group != 2 && group != 4 && group != 8) return ATTN_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(out) % 16 || reinterpret_cast<uintptr_t>(q) % 16)
        return ATTN_ERR_INVALID_ARG;
    const int hkv = num_q_heads / group;
    int st = check_kv(k, batch, head_dim, max_kv_len);
    if (st) return st;
    st = check_kv(v, batch, head_dim, max_kv_len);
    if (st) return st;
    if (k->page_table != v->page_table || k->page_size != v->page_size ||
        k->max_pages != v->max_pages || k->num_pages != v->num_pages)
        return ATTN_ERR_UNSUPPORTED;

    // head_dim 128 runs on the tensor cores (128-key tiles), head_dim 64 on
    // the CUDA cores (32-key tiles).  On the tensor cores a split into 2 or 4
    // partitions is merged on chip by a cluster of that many CTAs.
    const bool tc = head_dim == 128;
    const bool balanced = num_partitions == ATTN_PARTITIONS_BALANCED;
    const bool on_chip = !balanced && merges_on_chip(num_partitions, head_dim);
    size_t off_m = 0, off_l = 0, off_table = 0;
    int ctas = 0;
    size_t need;
    if (balanced) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&ctas, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        need = gqa_balanced_layout(ctas, static_cast<long long>(batch) * hkv, &off_m, &off_l,
                                   &off_table);
    } else {
        need = workspace_layout(num_partitions, num_q_rows, num_q_heads, head_dim, &off_m,
                                &off_l);
    }
    if (balanced || (num_partitions > 1 && !on_chip)) {
        if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) % 256) return ATTN_ERR_WORKSPACE;
    }
    const int tile = tc ? kGqaTcTileKeys : kGqaTileKeys;
    GqaParams p;
    std::memset(&p, 0, sizeof(p));
    p.box_rows = k->page_table ? (k->page_size < tile ? k->page_size : tile) : tile;
    st = encode_kv_map(&p.k_map, *k, head_dim, hkv, p.box_rows);
    if (st) return st;
    st = encode_kv_map(&p.v_map, *v, head_dim, hkv, p.box_rows);
    if (st) return st;
    if (tc) {
        // Q as (channel, head, query row); one box = the group's heads of
        // max_q_len consecutive rows (rows past the tensor read as zero).
        EncodeTiledFn fn = encode_fn();
        if (!fn) return ATTN_ERR_CUDA;
        cuuint64_t gdim[3] = {128, cuuint64_t(num_q_heads), cuuint64_t(num_q_rows)};
        cuuint64_t gstride[2] = {128 * 2, cuuint64_t(num_q_heads) * 128 * 2};
        cuuint32_t box[3] = {64, cuuint32_t(group), cuuint32_t(max_q_len)};
        cuuint32_t estride[3] = {1, 1, 1};
        CUresult r = fn(&p.q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q),
                        gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return ATTN_ERR_UNSUPPORTED;
    }
    st = error_word(&p.err);
    if (st) return st;

    p.q = static_cast<const uint16_t *>(q);
    p.kv_len = kv_len;
    p.q_row_offsets = fold ? q_row_offsets : nullptr;
    p.page_table = k->page_table;
    p.sink = sink;
    if (balanced || (num_partitions > 1 && !on_chip)) {
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        p.ws_o = reinterpret_cast<float *>(ws);
        p.ws_m = reinterpret_cast<float *>(ws + off_m);
        p.ws_l = reinterpret_cast<float *>(ws + off_l);
        if (balanced) p.unit_slots = reinterpret_cast<int2 *>(ws + off_table);
    }
    p.cluster = on_chip ? num_partitions : 0;
    p.out = static_cast<uint16_t *>(out);
    p.lse = lse;
    p.batch = batch;
    p.num_q_rows = fold ? num_q_rows : batch;
    p.max_q_len = fold ? max_q_len : 1;
    p.causal = causal ? 1 : 0;
    p.num_q_heads = num_q_heads;
    p.group = group;
    p.head_dim = head_dim;
    p.max_pages = k->max_pages;
    p.page_size = k->page_size;
    p.num_pages = k->num_pages;
    p.num_partitions = num_partitions;
    p.chunk = chunk_for(max_kv_len, num_partitions, tile);
    if (balanced) {
        // the item table counts 128-key tiles of every unit
        p.balanced = 1;
        p.chunk = kGqaTcTileKeys;
        p.num_partitions = max_kv_len > 0 ? (max_kv_len + kGqaTcTileKeys - 1) / kGqaTcTileKeys : 1;
    }
    p.qk_scale_log2 = scale * 1.4426950408889634f;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = map_cuda(tc ? launch_gqa_decode_tc(p, s) : launch_gqa_decode(p, s));
    if (st || num_partitions == 1 || on_chip) return st;
    if (balanced) {
        ReduceParams r;
        std::memset(&r, 0, sizeof(r));
        r.ws_o = p.ws_o;
        r.ws_m = p.ws_m;
        r.ws_l = p.ws_l;
        r.sink = sink;
        r.out = p.out;
        r.lse = lse;
        r.q_row_offsets = p.q_row_offsets;
        r.batch = batch;
        r.num_partitions = ctas;   // the most pieces a unit can have
        r.rows = p.num_q_rows;
        r.num_q_heads = num_q_heads;
        r.dim_v = head_dim;
        r.unit_slots = p.unit_slots;
        r.group = group;
        r.hkv = hkv;
        return map_cuda(launch_splitk_reduce(r, s, /*pdl=*/true));
    }

    ReduceParams r;
    std::memset(&r, 0, sizeof(r));
    r.ws_o = p.ws_o;
    r.ws_m = p.ws_m;
    r.ws_l = p.ws_l;
    r.sink = sink;
    r.out = p.out;
    r.lse = lse;
    r.kv_len = kv_len;
    r.q_row_offsets = p.q_row_offsets;
    r.batch = batch;
    r.num_partitions = num_partitions;
    r.rows = p.num_q_rows;
    r.num_q_heads = num_q_heads;
    r.dim_v = head_dim;
    r.chunk = p.chunk;
    return map_cuda(launch_splitk_reduce(r, s, /*pdl=*/true));
}

namespace {

// A cache read as rows for sparse top-k: row r is slot r % page_size of page
// r / page_size, so any page size (1 included) and any page order work.
int check_kv_rows(const attn_kv_t *kv, int dim) {
    if (!kv || !kv->base) return ATTN_ERR_INVALID_ARG;
    if (kv->reserved != 0 || kv->page_table) return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(kv->base) % 16) return ATTN_ERR_INVALID_ARG;
    if (kv->page_size <= 0 || kv->num_pages <= 0) return ATTN_ERR_INVALID_ARG;
    if (kv->token_stride <= 0 || kv->head_stride <= 0 || kv->page_stride <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (kv->token_stride % 8 || kv->head_stride % 8 || kv->page_stride % 8)
        return ATTN_ERR_INVALID_ARG;
    if (kv->head_stride < dim && kv->token_stride < dim) return ATTN_ERR_INVALID_ARG;
    // rows at one uniform stride (a contiguous pool of pages)
    if (kv->page_stride != static_cast<int64_t>(kv->page_size) * kv->token_stride)
        return ATTN_ERR_UNSUPPORTED;
    if (kv->token_stride < dim) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

// The cache as a 2-D row array (channel, row) for gather4: box box_ch
// channels x one row, 128-byte swizzle for 64 channels, 64-byte for 32.
int encode_rows_map(CUtensorMap *map, const attn_kv_t &kv, int dim, int box_ch = 64) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return ATTN_ERR_CUDA;
    const long long rows = static_cast<long long>(kv.num_pages) * kv.page_size;
    cuuint64_t gdim[2] = {cuuint64_t(dim), cuuint64_t(rows)};
    cuuint64_t gstride[1] = {cuuint64_t(kv.token_stride) * 2};
    cuuint32_t box[2] = {cuuint32_t(box_ch), 1};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(kv.base), gdim,
                    gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    box_ch == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_UNSUPPORTED;
}

// Shared body of the dense (paged or contiguous) and sparse MLA entry points.
int mla_decode_impl(const void *q, const attn_kv_t *kv, const uint32_t *kv_len,
                    const uint32_t *q_row_offsets, int num_q_rows, int causal, bool sparse,
                    const int32_t *indices, int indices_stride, int batch, int num_q_heads,
                    int dim_qk, int dim_v, int max_kv_len, float scale, const float *sink,
                    int num_partitions, void *workspace, size_t workspace_bytes, void *out,
                    float *lse, attn_stream_t stream) {
    if (batch < 0 || num_q_rows < 0 || num_q_heads <= 0 || dim_qk <= 0 || dim_v <= 0 ||
        max_kv_len < 0)
        return ATTN_ERR_INVALID_ARG;
    if (!q_row_offsets && num_q_rows != batch) return ATTN_ERR_INVALID_ARG;
    if (num_partitions < 0 || num_partitions > ATTN_MAX_PARTITIONS) return ATTN_ERR_INVALID_ARG;
    if (!(scale == scale)) return ATTN_ERR_INVALID_ARG;
    if (batch == 0 || num_q_rows == 0) return ATTN_OK;
    if (!q || !kv_len || !out) return ATTN_ERR_INVALID_ARG;
    if (num_q_heads != kMlaHeads || dim_qk != kMlaDimQK || dim_v != kMlaDimV)
        return ATTN_ERR_UNSUPPORTED;
    const bool balanced = num_partitions == 0;
    if (num_partitions != 1 && !workspace) return ATTN_ERR_WORKSPACE;
    // Balanced split: tile counts and starts are int (rows x tiles per row).
    if (balanced &&
        static_cast<long long>(num_q_rows) * ((static_cast<long long>(max_kv_len) + kMlaTileKeys - 1) /
                                              kMlaTileKeys) >= (1LL << 31))
        return ATTN_ERR_UNSUPPORTED;
    if (num_q_rows > 65535) return ATTN_ERR_UNSUPPORTED;   // grid rows
    if (reinterpret_cast<uintptr_t>(out) % 16 || reinterpret_cast<uintptr_t>(q) % 16)
        return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(indices) % 4) return ATTN_ERR_INVALID_ARG;
    int st = sparse ? check_kv_rows(kv, dim_qk) : check_kv(kv, batch, dim_qk, max_kv_len);
    if (st) return st;
    size_t off_m = 0, off_l = 0, off_plan = 0;
    int clusters = 0;
    size_t need;
    if (balanced) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        clusters = mla_cluster_slots(sms, sparse);
        need = mla_balanced_layout(clusters, num_q_rows, &off_m, &off_l, &off_plan);
    } else {
        need = workspace_layout(num_partitions, num_q_rows, num_q_heads, dim_v, &off_m, &off_l);
    }
    if (num_partitions != 1) {
        if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) % 256) return ATTN_ERR_WORKSPACE;
    }

    MlaParams p;
    std::memset(&p, 0, sizeof(p));
    p.box_rows = sparse ? 1
                 : kv->page_table ? (kv->page_size < kMlaTileKeys ? kv->page_size : kMlaTileKeys)
                                  : kMlaTileKeys;
    st = sparse ? encode_rows_map(&p.kv_map, *kv, dim_qk)
                : encode_kv_map(&p.kv_map, *kv, dim_qk, 1, p.box_rows);
    if (st) return st;
    st = sparse ? encode_rows_map(&p.rope_map, *kv, dim_qk, kMlaRopeBoxCh)
                : encode_kv_map(&p.rope_map, *kv, dim_qk, 1, p.box_rows, kMlaRopeBoxCh);
    if (st) return st;
    p.q = static_cast<const uint16_t *>(q);
    st = error_word(&p.err);
    if (st) return st;
    p.kv_len = kv_len;
    p.q_row_offsets = q_row_offsets;
    p.num_q_rows = num_q_rows;
    p.causal = causal ? 1 : 0;
    p.page_table = kv->page_table;
    p.sparse = sparse ? 1 : 0;
    p.indices = indices;
    p.indices_stride = indices_stride;
    p.num_rows = static_cast<long long>(kv->num_pages) * kv->page_size;
    p.sink = sink;
    if (num_partitions != 1) {
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        p.ws_o = reinterpret_cast<float *>(ws);
        p.ws_m = reinterpret_cast<float *>(ws + off_m);
        p.ws_l = reinterpret_cast<float *>(ws + off_l);
    }
    if (balanced) {
        p.plan_slots = reinterpret_cast<int2 *>(static_cast<uint8_t *>(workspace) + off_plan);
        p.balanced = 1;
        p.num_clusters = clusters;
        p.len_cap = max_kv_len;
    }
    p.out = static_cast<uint16_t *>(out);
    p.lse = lse;
    p.batch = batch;
    p.max_pages = kv->max_pages;
    p.page_size = kv->page_size;
    p.num_pages = kv->num_pages;
    p.num_partitions = num_partitions;
    p.chunk = balanced ? kMlaTileKeys : chunk_for(max_kv_len, num_partitions, kMlaTileKeys);
    p.qk_scale_log2 = scale * 1.4426950408889634f;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = map_cuda(launch_mla_decode(p, s));
    if (st || num_partitions == 1) return st;

    ReduceParams r;
    std::memset(&r, 0, sizeof(r));
    r.ws_o = p.ws_o;
    r.ws_m = p.ws_m;
    r.ws_l = p.ws_l;
    r.sink = sink;
    r.out = p.out;
    r.lse = lse;
    r.kv_len = kv_len;
    r.q_row_offsets = q_row_offsets;
    r.batch = batch;
    r.num_partitions = num_partitions;
    r.rows = num_q_rows;
    r.num_q_heads = num_q_heads;
    r.dim_v = dim_v;
    r.chunk = p.chunk;
    r.len_cap = sparse ? indices_stride : 0;
    if (balanced) {
        r.slots = p.plan_slots;
        r.num_slots = clusters + num_q_rows;
        r.kv_len = nullptr;
        r.q_row_offsets = nullptr;
        r.num_partitions = clusters;   // the most partials a row can have
    }
    return map_cuda(launch_splitk_reduce(r, s, /*pdl=*/true));
}

}  // namespace

extern "C" int attn_mla_decode(const void *q, const attn_kv_t *kv, const uint32_t *kv_len,
                               int batch, int num_q_heads, int dim_qk, int dim_v, int max_kv_len,
                               float scale, const float *sink, int num_partitions,
                               void *workspace, size_t workspace_bytes, void *out, float *lse,
                               attn_stream_t stream) {
    return mla_decode_impl(q, kv, kv_len, nullptr, batch, 0, false, nullptr, 0, batch,
                           num_q_heads, dim_qk, dim_v, max_kv_len, scale, sink, num_partitions,
                           workspace, workspace_bytes, out, lse, stream);
}

extern "C" int attn_mla_decode_rows(const void *q, const attn_kv_t *kv, const uint32_t *kv_len,
                                    const uint32_t *q_row_offsets, int batch, int num_q_rows,
                                    int num_q_heads, int dim_qk, int dim_v, int max_kv_len,
                                    float scale, const float *sink, int causal,
                                    int num_partitions, void *workspace, size_t workspace_bytes,
                                    void *out, float *lse, attn_stream_t stream) {
    if (batch > 0 && num_q_rows > 0 && !q_row_offsets) return ATTN_ERR_INVALID_ARG;
    if (num_q_rows < 0 || batch < 0) return ATTN_ERR_INVALID_ARG;
    return mla_decode_impl(q, kv, kv_len, q_row_offsets, num_q_rows, causal, false, nullptr, 0,
                           batch, num_q_heads, dim_qk, dim_v, max_kv_len, scale, sink,
                           num_partitions, workspace, workspace_bytes, out, lse, stream);
}

extern "C" int attn_mla_decode_sparse(const void *q, const attn_kv_t *kv,
                                      const int32_t *indices, int indices_stride,
                                      const int32_t *topk_lengths, int batch, int num_q_heads,
                                      int dim_qk, int dim_v, float scale, const float *sink,
                                      int num_partitions, void *workspace,
                                      size_t workspace_bytes, void *out, float *lse,
                                      attn_stream_t stream) {
    if (indices_stride < 0) return ATTN_ERR_INVALID_ARG;
    if (batch > 0 && indices_stride > 0 && !indices) return ATTN_ERR_INVALID_ARG;
    if (batch > 0 && !topk_lengths) return ATTN_ERR_INVALID_ARG;
    // topk_lengths is read as unsigned: a negative count is above any cap and
    // is reported as a length error.
    return mla_decode_impl(q, kv, reinterpret_cast<const uint32_t *>(topk_lengths), nullptr,
                           batch, 0, true, indices, indices_stride, batch, num_q_heads, dim_qk, dim_v, indices_stride,
                           scale, sink, num_partitions, workspace, workspace_bytes, out, lse,
                           stream);
}

extern "C" int attn_splitk_reduce(const float *ws_o, const float *ws_m, const float *ws_l,
                                  int num_partitions, int rows, int num_q_heads, int dim_v,
                                  const float *sink, void *out, float *lse,
                                  attn_stream_t stream) {
    if (num_partitions < 1 || num_partitions > ATTN_MAX_PARTITIONS || rows < 0 ||
        num_q_heads <= 0 || dim_v <= 0 || dim_v % 4 || dim_v > 1024)
        return ATTN_ERR_INVALID_ARG;
    if (rows == 0) return ATTN_OK;
    if (!ws_o || !ws_m || !ws_l || !out) return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws_o) % 16 || reinterpret_cast<uintptr_t>(out) % 8)
        return ATTN_ERR_INVALID_ARG;
    ReduceParams r;
    std::memset(&r, 0, sizeof(r));
    r.ws_o = ws_o;
    r.ws_m = ws_m;
    r.ws_l = ws_l;
    r.sink = sink;
    r.out = static_cast<uint16_t *>(out);
    r.lse = lse;
    r.num_partitions = num_partitions;
    r.rows = rows;
    r.num_q_heads = num_q_heads;
    r.dim_v = dim_v;
    return map_cuda(launch_splitk_reduce(r, reinterpret_cast<cudaStream_t>(stream), false));
}

extern "C" int attn_selftest_wait_timeout(attn_stream_t stream) {
    unsigned *err = nullptr;
    const int st = error_word(&err);
    if (st) return st;
    selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err);
    return map_cuda(cudaGetLastError());
}

extern "C" int attn_device_error_flags(unsigned int *flags, int clear) {
    if (!flags) return ATTN_ERR_INVALID_ARG;
    unsigned *ptr = nullptr;
    int st = error_word(&ptr);
    if (st) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemcpy(flags, ptr, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (clear && cudaMemset(ptr, 0, sizeof(unsigned)) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}
