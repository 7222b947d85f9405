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

#include "sai_internal.h"
#include "sai_ptx.cuh"
#include "sai_select.cuh"

namespace sai {
namespace {

constexpr int kRowsPerCta = 4;
constexpr int kRowThreads = 128;
constexpr int kBitmapWords = 512;  // 16384 block ids per row

struct __align__(16) BlockRowSmem {
  union {
    struct {
      uint32_t key[kTopK];  // ~block, so the descending sort gives ascending blocks
      int32_t idx[kTopK];
      unsigned long long sortbuf[kTopK];
    } s;
    uint32_t bitmap[kBitmapWords];
  } u;
  uint32_t wsum[32];
  int32_t last[4];  // each warp's last sorted block
  int32_t wmin[4], wmax[4];
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

  int32_t b[4];
  bool v4[4];
  int32_t lmin = 0x7FFFFFFF, lmax = -1;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int j = 4 * t + e;
    const int32_t s = (live && j < k) ? slots[row * k + j] : -1;
    v4[e] = s >= 0;
    b[e] = v4[e] ? s / block_size : 0;
    if (v4[e]) {
      lmin = min(lmin, b[e]);
      lmax = max(lmax, b[e]);
    }
  }
  lmin = __reduce_min_sync(0xFFFFFFFFu, lmin);
  lmax = __reduce_max_sync(0xFFFFFFFFu, lmax);
  if (lane == 0) {
    S.wmin[warp] = lmin;
    S.wmax[warp] = lmax;
  }
  named_bar(bar, kRowThreads);
  int32_t bmin = S.wmin[0], bmax = S.wmax[0];
#pragma unroll
  for (int w = 1; w < kRowThreads / 32; ++w) {
    bmin = min(bmin, S.wmin[w]);
    bmax = max(bmax, S.wmax[w]);
  }
  const long long o = row * k;
  if (bmax < 0 || (long long)bmax - bmin < 32LL * kBitmapWords) {
    // ---- bitmap: bit (block - bmin) of the row's 512 words
    const int words = bmax < 0 ? 0 : (bmax - bmin) / 32 + 1;
    for (int w = t; w < words; w += kRowThreads) S.u.bitmap[w] = 0u;
    named_bar(bar, kRowThreads);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (v4[e]) atomicOr(&S.u.bitmap[(b[e] - bmin) >> 5], 1u << ((b[e] - bmin) & 31));
    }
    named_bar(bar, kRowThreads);
    // thread t owns words 4t .. 4t+3
    uint32_t wv[4];
    int nf = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int w = 4 * t + e;
      wv[e] = w < words ? S.u.bitmap[w] : 0u;
      nf += __popc(wv[e]);
    }
    int count;
    int out = block_exscan<kRowThreads>(nf, &count, S.wsum, t, bar);
    if (!live) return;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t m = wv[e];
      while (m) {
        const int bit = __ffs(m) - 1;
        m &= m - 1u;
        out_blocks[o + out++] = bmin + 32 * (4 * t + e) + bit;
      }
    }
    for (int j = count + t; j < k; j += kRowThreads) out_blocks[o + j] = -1;
    if (out_counts && t == 0) out_counts[row] = count;
    return;
  }

  // ---- sort: blocks of the valid slots compacted, sorted, first
  // occurrences kept
  int c = 0;
  int32_t bc[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (v4[e]) bc[c++] = b[e];
  int total;
  int pos = block_exscan<kRowThreads>(c, &total, S.wsum, t, bar);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (e < c) {
      S.u.s.key[pos] = ~static_cast<uint32_t>(bc[e]);
      S.u.s.idx[pos] = pos;
      ++pos;
    }
  }
  named_bar(bar, kRowThreads);
  // ascending blocks: sorted position 4t + e holds blk[e] (-1: padding)
  unsigned long long v[4];
  bitonic_sort512_128(S.u.s.key, S.u.s.idx, total, S.u.s.sortbuf, v, t, bar);
  int32_t blk[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) blk[e] = v[e] ? static_cast<int32_t>(~static_cast<uint32_t>(v[e] >> 32)) : -1;
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
