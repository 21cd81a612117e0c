// launch.h -- parameter blocks passed from the C-ABI layer (api.cu) to the
// kernel launchers.  Everything here is already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// Keys per pipeline stage and per consumer warp pass in the GQA kernel;
// partition slices are multiples of it.
constexpr int kGqaTileKeys = 32;
// Keys per tile of the tensor-core GQA decode kernel (head_dim 128); its
// partition slices are multiples of it.
constexpr int kGqaTcTileKeys = 128;
// The single-token decode kernel keeps a per-sequence item table in shared
// memory; batches above this size are rejected.
constexpr int kGqaMaxBatch = 2048;

struct GqaParams {
    CUtensorMap k_map;            // 4-D: (channel, slot, kv head, page)
    CUtensorMap v_map;
    CUtensorMap q_map;            // 3-D: (channel, head, query row), box (64, group,
                                  // max_q_len); tensor-core kernel only
    const uint16_t *q;            // bf16 [rows][Hq][D]
    const uint32_t *kv_len;       // [batch]
    const uint32_t *q_row_offsets;  // [batch + 1], or nullptr: row b is sequence b
    const int32_t *page_table;    // [batch][max_pages] or nullptr
    const float *sink;            // [Hq] or nullptr
    float *ws_o;                  // [P][rows][Hq][D]
    float *ws_m;                  // [P][rows][Hq]
    float *ws_l;                  // [P][rows][Hq]
    uint16_t *out;                // bf16 [rows][Hq][D]
    float *lse;                   // [rows][Hq] or nullptr
    unsigned *err;                // device error word
    int batch, num_q_rows, num_q_heads, group, head_dim;
    int max_q_len;                // rows of any sequence (tensor-core kernel: * group <= 16)
    int causal;                   // rows of a sequence see keys j <= L - n + i
    int max_pages, page_size, num_pages;
    int box_rows;                 // tokens per TMA box (min(tile, page size))
    int num_partitions;           // P (grid.x)
    int chunk;                    // keys per partition slice, multiple of kGqaTileKeys
    int cluster;                  // tensor-core kernel: 2 or 4 = P CTAs of a cluster split a
                                  // unit and merge on chip (no workspace); 0 = off
    // Balanced split (tensor-core kernel): the 128-key tiles of every
    // (sequence, KV head) unit, concatenated, in equal contiguous ranges per
    // CTA (num_partitions = ceil(max_kv_len / 128), chunk = 128, so the item
    // table counts tiles).  A unit cut by a range end leaves one partial per
    // piece in slot (CTA + unit): ws_o [slots][16 columns][128], ws_m / ws_l
    // [slots][16]; unit_slots[unit] = {first slot, pieces} for the reduce.
    int balanced;
    int2 *unit_slots;             // [batch * num_kv_heads]
    float qk_scale_log2;          // scale * log2(e)
};
// Columns of one balanced-split partial slot (the N side of the tensor-core
// decode kernel: query rows x heads of a group).
constexpr int kGqaSlotCols = 16;

// Keys per tile in the MLA kernel; its partition slices are multiples of it.
constexpr int kMlaTileKeys = 64;
constexpr int kMlaHeads = 128;
constexpr int kMlaDimQK = 576;
constexpr int kMlaDimV = 512;
constexpr int kMlaRopeBoxCh = 32;   // rope channels each CTA of an MLA pair loads

struct MlaParams {
    CUtensorMap kv_map;           // 4-D: (channel 576, slot, head 1, page); sparse:
                                  // 2-D (channel 576, row), box height 1; 64-channel boxes
    CUtensorMap rope_map;         // the same cache with 32-channel boxes (64-byte swizzle)
    const uint16_t *q;            // bf16 [rows][128][576]
    const uint32_t *kv_len;       // [batch]
    const int32_t *page_table;    // [batch][max_pages] or nullptr
    const int32_t *indices;       // sparse: [batch][indices_stride] cache rows
    long long num_rows;           // sparse: rows in the cache (num_pages * page_size)
    int sparse;                   // 1: keys are named by indices, kv_len = top-k counts
    int indices_stride;
    const uint32_t *q_row_offsets;  // [batch + 1] or nullptr (one query row per sequence)
    int num_q_rows;               // rows of q / out (= batch without row offsets)
    int causal;                   // rows of a sequence end at its last key (row offsets only)
    const float *sink;            // [128] or nullptr
    float *ws_o;                  // [P][rows][128][512]
    float *ws_m;                  // [P][rows][128]
    float *ws_l;
    uint16_t *out;                // bf16 [rows][128][512]
    float *lse;                   // [rows][128] or nullptr
    unsigned *err;
    int batch, max_pages, page_size, num_pages;
    int box_rows;                 // tokens per TMA box (min(64, page size))
    int num_partitions, chunk;    // chunk: multiple of kMlaTileKeys
    float qk_scale_log2;
    // Balanced split (num_partitions 0): cluster c takes tiles [x0, x1) of the
    // concatenation of every query row's key tiles, found by the cluster from
    // the lengths.  Partials go to slot c + row; the cluster holding a row's
    // first tile writes its entry of the table below (cluster 0 those of the
    // rows without tiles) for the reduce.
    int balanced;
    int num_clusters;
    int len_cap;                  // kv_len above it is clamped (error bit 2)
    int2 *plan_slots;             // [num_q_rows] {first slot, partials} for the reduce
};

// Multi-row (prefill-shaped) tile kernel: 128 MMA rows = (128 / group)
// tokens x group heads of one KV head; 128-key tiles.
constexpr int kTileRows = 128;
constexpr int kTileKeys = 128;

struct TileParams {
    CUtensorMap q_map;            // 4-D: (channel, head in group, kv head, row)
    CUtensorMap k_map;            // 4-D: (channel, slot, kv head, page)
    CUtensorMap v_map;
    const uint32_t *kv_len;       // [batch]
    const uint32_t *q_row_offsets;  // [batch + 1]
    const int32_t *page_table;    // [batch][max_pages] or nullptr
    const float *sink;            // [Hq] or nullptr
    uint16_t *out;                // bf16 [rows][Hq][128]
    float *lse;                   // [rows][Hq] or nullptr
    unsigned *err;
    int batch, num_q_rows, num_q_heads, group;
    int max_pages, page_size, num_pages, box_rows;
    int box_rows_v;               // two-Q-tile kernel: tokens per V box (K boxes: box_rows)
    int causal;
    int tiles_per_seq;            // Q tiles of the longest sequence: ceil(max_q_len / (128 / group))
    float qk_scale_log2;
};

struct ReduceParams {
    const float *ws_o, *ws_m, *ws_l;
    const float *sink;            // [Hq] or nullptr
    uint16_t *out;                // bf16 [rows][Hq][dv]
    float *lse;                   // [rows][Hq] or nullptr
    const uint32_t *kv_len;       // optional: rows whose kv_len needs < 2 slices are skipped
    const uint32_t *q_row_offsets;  // optional: kv_len is per sequence, row r of sequence b
                                    // has off[b] <= r < off[b+1]
    int batch;
    int num_partitions, rows, num_q_heads, dim_v;
    int chunk;                    // slice length when kv_len is given
    int len_cap;                  // > 0: kv_len is clamped to it as well as to P * chunk
    // Balanced MLA split: row r's partials are slots e.x .. e.x + e.y - 1 of
    // the workspace (e = slots[r]); e.y == 1 rows were finished by the
    // decode kernel, e.y == 0 rows are empty.  An entry outside the
    // num_slots slots (a row no sequence owns) is read as an empty row.
    const int2 *slots;
    int num_slots;
    // Balanced GQA split: (row r, head h) of sequence b belongs to unit u =
    // b * hkv + h / group, whose partials are slots e.x .. e.x + e.y - 1
    // (e = unit_slots[u]) of [slots][kGqaSlotCols][dim_v], at column
    // (r - first row of b) * group + h % group; e.y == 1: finished by the
    // decode kernel.
    const int2 *unit_slots;
    int group, hkv;
};

cudaError_t launch_gqa_decode(const GqaParams &p, cudaStream_t stream);
cudaError_t launch_gqa_decode_tc(const GqaParams &p, cudaStream_t stream);
cudaError_t launch_mla_decode(const MlaParams &p, cudaStream_t stream);
// Two-CTA MLA clusters that run at once on num_sms SMs (at most num_sms / 2).
int mla_cluster_slots(int num_sms, bool sparse);
cudaError_t launch_tile_attention(const TileParams &p, cudaStream_t stream);
// Two adjacent Q tiles per CTA pair sharing each K/V tile (K boxes of
// min(64, page size) tokens, V boxes of min(128, page size)).
cudaError_t launch_tile_attention_pair(const TileParams &p, cudaStream_t stream);
cudaError_t launch_splitk_reduce(const ReduceParams &p, cudaStream_t stream, bool pdl);

}  // namespace attn
