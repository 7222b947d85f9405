// Per-index-head top-k: metadata for the top-k over per-head score rows.
//
// The fused decode kernel of ROCm/ATOM PR #1473 "enable minimax m3 fp8 index
// cache and fuse index_score_kernel with partial_topk kernel" is launched
// over (query, index head, key chunk) (review diff of index_topk.py), which
// admits one selection per index head. The library computes each head's
// score densely (the fused kernel's per-head mode, [rows, 64, stride]) and
// selects with the top-k kernel over rows x 64 score rows; this kernel gives
// score row (row, h) its length and block-table row.
#include <cuda_runtime.h>

#include "sai_internal.h"

namespace sai {

namespace {

constexpr int kHeads = 64;

__global__ void per_head_expand_kernel(const int* seq_lens, const int* row_to_batch, int rows, int max_len,
                                       long long bt_rows, long long bt_stride, int* out_lens, int* out_batch) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)rows * kHeads) return;
  const int row = static_cast<int>(e / kHeads);
  int n = seq_lens[row];
  int b = row_to_batch ? row_to_batch[row] : row;
  // the fused kernel empties (and flags) such a row: it has no scores
  const bool bad = b < 0 || b >= bt_rows || n < 0 || n > max_len || (long long)(n + 127) / 128 > bt_stride;
  out_lens[e] = bad ? 0 : n;
  out_batch[e] = bad ? 0 : b;
}

}  // namespace

cudaError_t launch_per_head_expand(const int* seq_lens, const int* row_to_batch, int rows, int max_len,
                                   long long bt_rows, long long bt_stride, int* out_lens, int* out_batch,
                                   cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const long long n = (long long)rows * kHeads;
  const int threads = 256;
  const int grid = static_cast<int>((n + threads - 1) / threads);
  per_head_expand_kernel<<<grid, threads, 0, stream>>>(seq_lens, row_to_batch, rows, max_len, bt_rows, bt_stride,
                                                       out_lens, out_batch);
  return cudaGetLastError();
}

}  // namespace sai
