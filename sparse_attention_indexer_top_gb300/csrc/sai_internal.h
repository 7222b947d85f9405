// Internal launch interface between the C-ABI layer (sai_api.cu) and the
// kernel translation units. Not part of the public header.
#pragma once
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace sai {

// Device status bits (OR-ed into the library's device status word).
enum DevStatusBits : int {
  kDevBadRowMeta = 1,      // a row's seq_len / row_start / row_to_batch was out of range
  kDevWaitTimeout = 2,     // a pipeline wait gave up (the affected rows are undefined)
  kDevBadPage = 4,         // a block-table entry was out of range (fused path)
};

struct TopkLaunch {
  const float* scores;
  long long stride;
  int rows;
  const int* row_starts;
  const int* seq_lens;
  const int* page_tables;
  long long pt_rows, pt_stride;
  const int* row_to_batch;
  int page_size;
  int* out_slots;
  int* out_idx;
  int chunks;      // work units per row (1 = one unit per row)
  int chunk_len;   // window elements per unit when chunks > 1
  uint32_t* part_key;  // [rows*chunks, 512] when chunks > 1
  int32_t* part_idx;
  int* part_cnt;       // [rows*chunks]
  int* work;           // unit counter, zero at launch (null: fixed unit order)
  int* status;
  int block_size;      // out_blocks: per-row ascending distinct blocks of the slots
  int* out_blocks;     // [rows, 512] or null
  int* out_counts;     // [rows] or null
};

// Bytes at the start of a topk_transform workspace: the unit counter.
constexpr size_t kTopkWorkHeader = 256;

// How a topk_transform call is split; shared by the workspace query and the
// launcher so both always agree.
struct TopkPlan {
  int chunks;
  int chunk_len;
  size_t workspace_bytes;
};

TopkPlan topk_plan(long long rows, long long max_window, int num_sms);
cudaError_t launch_topk_transform(const TopkLaunch& p, int num_sms, cudaStream_t stream);

// Final merge of per-unit candidate lists (also used by the fused path).
struct MergeLaunch {
  int rows;
  int units_per_row;
  const uint32_t* part_key;
  const int32_t* part_idx;
  const int* part_cnt;
  const int* seq_lens;         // for the padding count (may be null: use candidates)
  const int* page_tables;
  long long pt_rows, pt_stride;
  const int* row_to_batch;
  int page_size;
  int* out_slots;
  int* out_idx;
  float* out_scores;           // optional: scores of the selected (fused path)
  int* status;
  int block_size;              // out_blocks: per-row ascending distinct blocks of the slots
  int* out_blocks;             // [rows, 512] or null
  int* out_counts;             // [rows] or null
};
cudaError_t launch_merge(const MergeLaunch& p, cudaStream_t stream);

// Per-row distinct blocks of top-k slots (sparse_blocks.cu).
cudaError_t launch_sparse_blocks(const int32_t* slots, int rows, int k, int block_size, int32_t* out_blocks,
                                 int32_t* out_counts, cudaStream_t stream);

struct FusedLaunch {
  const void* q;           // [rows, 64, 128] e4m3 codes or bf16
  const float* w;          // [rows, 64]
  const float* kscale;     // [num_blocks, 128], or null (scale 1; bf16 cache only)
  long long num_blocks;
  const int* block_table;  // [bt_rows, bt_stride]
  long long bt_rows, bt_stride;
  const int* row_to_batch;
  const int* seq_lens;
  int rows;
  int max_len;       // caller's bound on seq_lens (checked per row)
  int chunks;        // work units per row group
  int chunk_blocks;  // KV blocks per unit
  uint32_t* part_key;
  int32_t* part_idx;
  int* part_cnt;     // [rows * chunks]
  float* dense;      // dense modes: [rows, dense_stride] or [rows, 64, dense_stride]
  int sign_w;        // per-head mode: use sign(w_h) for w_h (same order per (row, head), comparable scales)
  long long dense_stride;
  int* status;
  int stall_unit;    // test hook: this work unit streams no key tiles (-1: none)
};
struct FusedPlan {
  int group;         // query rows per CTA (1 or 4)
  int chunks;        // KV chunks per row group
  int chunk_blocks;  // KV blocks per chunk
  size_t workspace_bytes;
};
FusedPlan fused_plan(long long rows, int max_seq_len, int group_rows, int num_sms);
// What a fused launch writes: per-(row, chunk) partial top-k lists, dense
// head-summed scores [rows, dense_stride], or dense per-head scores
// [rows, 64, dense_stride].
enum class FusedOut { kTopk, kDense, kPerHead };
cudaError_t launch_fused(const FusedLaunch& p, int group, FusedOut out, bool bf16, const void* kcache,
                         cudaStream_t stream);
// Per-(row, head) lengths and block-table rows of the per-head top-k:
// n = seq_lens[row] (0 for a row the fused kernel would reject), batch =
// row_to_batch ? row_to_batch[row] : row.
cudaError_t launch_per_head_expand(const int* seq_lens, const int* row_to_batch, int rows, int max_len,
                                   long long bt_rows, long long bt_stride, int* out_lens, int* out_batch,
                                   cudaStream_t stream);

}  // namespace sai
