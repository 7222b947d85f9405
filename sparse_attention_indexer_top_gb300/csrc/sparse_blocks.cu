// sparse_blocks: per-row distinct KV blocks of the top-k slots.
//
// ROCm/ATOM PR #1282 "merge build sparse block into topk" (title and
// Motivation): the sparse attention that follows the indexer reads KV
// blocks, so each row's selected physical slots become the list of the
// distinct blocks (slot / block_size) they fall in. Slots < 0 are padding.
// The list is ascending, -1 padded to k, with its length per row.
//
// GB300 design: four rows per CTA, 128 threads per row, up to 512 slots per
// row (4 per thread). When a row's blocks span at most 16384 ids (a KV
// pool's blocks, or a 2M-token window) they are set as bits of a shared
// bitmap and read back in ascending order with a popcount scan (a handful
// of barriers). Wider rows are compacted (a block scan), sorted ascending
// with the bitonic network of the top-k finalize, and first occurrences are
// marked against the previous sorted entry and compacted with a second
// scan. Bound: HBM (k slots read and k blocks written per row).
#include <cuda_runtime.h>

#include <cstdint>

#include "sai_blocks.cuh"
#include "sai_internal.h"

namespace sai {
namespace {

constexpr int kRowsPerCta = 4;

__global__ void __launch_bounds__(kRowsPerCta * kBlockThreads)
    sparse_blocks_kernel(const int32_t* __restrict__ slots, int rows, int k, int block_size,
                         int32_t* __restrict__ out_blocks, int32_t* __restrict__ out_counts) {
  extern __shared__ unsigned char smem_raw[];
  const int g = threadIdx.x / kBlockThreads, t = threadIdx.x % kBlockThreads;
  BlockScratch& S = reinterpret_cast<BlockScratch*>(smem_raw)[g];
  const long long row = (long long)blockIdx.x * kRowsPerCta + g;
  const bool live = row < rows;
  int32_t sl[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int j = 4 * t + e;
    sl[e] = (live && j < k) ? slots[row * k + j] : -1;
  }
  row_blocks128(sl, k, block_size, out_blocks + (live ? row * k : 0), out_counts ? out_counts + (live ? row : 0) : nullptr,
                S, t, 1 + g, live);
}

}  // namespace

cudaError_t launch_sparse_blocks(const int32_t* slots, int rows, int k, int block_size, int32_t* out_blocks,
                                 int32_t* out_counts, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int grid = (rows + kRowsPerCta - 1) / kRowsPerCta;
  sparse_blocks_kernel<<<grid, kRowsPerCta * kBlockThreads, kRowsPerCta * sizeof(BlockScratch), stream>>>(
      slots, rows, k, block_size, out_blocks, out_counts);
  return cudaGetLastError();
}

}  // namespace sai
