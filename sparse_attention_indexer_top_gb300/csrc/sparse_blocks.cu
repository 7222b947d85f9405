// sparse_blocks: per-row distinct KV blocks of the top-k slots.
//
// ROCm/ATOM PR #1282 "merge build sparse block into topk" (title and
// Motivation): the sparse attention that follows the indexer reads KV
// blocks, so each row's selected physical slots become the list of the
// distinct blocks (slot / block_size) they fall in. Slots < 0 are padding.
// The list is ascending, -1 padded to k, with its length per row.
//
// GB300 design: four rows per CTA, 128 threads per row, up to 512 slots per
// row (4 per thread). The valid slots' blocks are compacted into shared
// memory (a block scan), sorted ascending with the bitonic network of the
// top-k finalize (registers, warp shuffles, three shared-memory stages),
// first occurrences marked against the previous sorted entry and compacted
// with a second scan. Bound: HBM (k slots read and k blocks written per
// row; a few microseconds for 16384 rows).
#include <cuda_runtime.h>

#include <cstdint>

#include "sai_internal.h"
#include "sai_ptx.cuh"
#include "sai_select.cuh"

namespace sai {
namespace {

constexpr int kRowsPerCta = 4;
constexpr int kRowThreads = 128;

struct __align__(16) BlockRowSmem {
  uint32_t key[kTopK];  // ~block, so the descending sort gives ascending blocks
  int32_t idx[kTopK];
  unsigned long long sortbuf[kTopK];
  uint32_t wsum[32];
  int32_t last[4];  // each warp's last sorted block
};

__global__ void __launch_bounds__(kRowsPerCta * kRowThreads)
    sparse_blocks_kernel(const int32_t* __restrict__ slots, int rows, int k, int block_size,
                         int32_t* __restrict__ out_blocks, int32_t* __restrict__ out_counts) {
  extern __shared__ unsigned char smem_raw[];
  const int g = threadIdx.x / kRowThreads, t = threadIdx.x % kRowThreads;
  const int lane = t & 31, warp = t >> 5;
  BlockRowSmem& S = reinterpret_cast<BlockRowSmem*>(smem_raw)[g];
  const long long row = (long long)blockIdx.x * kRowsPerCta + g;
  const int bar = 1 + g;
  const bool live = row < rows;

  // 1. blocks of the valid slots, compacted
  int32_t b[4];
  int c = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int j = 4 * t + e;
    const int32_t s = (live && j < k) ? slots[row * k + j] : -1;
    if (s >= 0) b[c++] = s / block_size;
  }
  int total;
  int pos = block_exscan<kRowThreads>(c, &total, S.wsum, t, bar);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (e < c) {
      S.key[pos] = ~static_cast<uint32_t>(b[e]);
      S.idx[pos] = pos;
      ++pos;
    }
  }
  named_bar(bar, kRowThreads);

  // 2. ascending blocks: sorted position 4t + e holds blk[e] (-1: padding)
  unsigned long long v[4];
  bitonic_sort512_128(S.key, S.idx, total, S.sortbuf, v, t, bar);
  int32_t blk[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) blk[e] = v[e] ? static_cast<int32_t>(~static_cast<uint32_t>(v[e] >> 32)) : -1;

  // 3. first occurrences: compare with the previous sorted entry
  if (lane == 31) S.last[warp] = blk[3];
  named_bar(bar, kRowThreads);
  int32_t prev = __shfl_up_sync(0xFFFFFFFFu, blk[3], 1);
  if (lane == 0) prev = warp > 0 ? S.last[warp - 1] : -1;
  bool first[4];
  int nf = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int32_t before = e == 0 ? prev : blk[e - 1];
    first[e] = blk[e] >= 0 && (4 * t + e == 0 || blk[e] != before);
    nf += first[e] ? 1 : 0;
  }
  int count;
  int out = block_exscan<kRowThreads>(nf, &count, S.wsum, t, bar);
  if (!live) return;

  // 4. write, -1 padded to k
  const long long o = row * k;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (first[e]) out_blocks[o + out++] = blk[e];
  }
  for (int j = count + t; j < k; j += kRowThreads) out_blocks[o + j] = -1;
  if (out_counts && t == 0) out_counts[row] = count;
}

}  // namespace

cudaError_t launch_sparse_blocks(const int32_t* slots, int rows, int k, int block_size, int32_t* out_blocks,
                                 int32_t* out_counts, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int grid = (rows + kRowsPerCta - 1) / kRowsPerCta;
  sparse_blocks_kernel<<<grid, kRowsPerCta * kRowThreads, kRowsPerCta * sizeof(BlockRowSmem), stream>>>(
      slots, rows, k, block_size, out_blocks, out_counts);
  return cudaGetLastError();
}

}  // namespace sai
