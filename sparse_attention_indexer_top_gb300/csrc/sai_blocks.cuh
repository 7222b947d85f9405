// Distinct KV blocks of one row's selected slots, for a group of 128
// threads holding 4 slots each.
//
// ROCm/ATOM PR #1282 "merge build sparse block into topk" (title and
// Motivation): the sparse attention that follows the indexer reads KV
// blocks, so each row's selected physical slots become the list of the
// distinct blocks (slot / block_size) they fall in. Slots < 0 are padding.
// The list is ascending, -1 padded to k, with its length.
//
// Used by the sparse_blocks kernel (slots read back from memory) and by the
// last stage of every top-k path (slots still in registers), so the block
// lists come out of the same kernel that picks the slots.
//   * When the row's blocks span at most 16384 ids (a KV pool's blocks, or a
//     2M-token window) they are set as bits of a shared bitmap and read back
//     in ascending order with a popcount scan.
//   * Wider rows are compacted, sorted ascending with the 128-thread bitonic
//     network, and first occurrences kept.
#pragma once
#include <cstdint>

#include "sai_ptx.cuh"
#include "sai_select.cuh"

namespace sai {

constexpr int kBlockThreads = 128;
constexpr int kBitmapWords = 512;  // 16384 block ids per row

struct __align__(16) BlockScratch {
  union {
    struct {
      uint32_t key[kTopK];  // ~block, so the descending sort gives ascending blocks
      int32_t idx[kTopK];
      unsigned long long sortbuf[kTopK];
    } s;
    uint32_t bitmap[kBitmapWords];
  } u;
  uint32_t wsum[32];
  unsigned long long wtot[4];  // each warp's packed word counts (bitmap path)
  int32_t last[4];             // each warp's last sorted block
  int32_t wmin[4], wmax[4];
};

// The 128 threads t of a group (named barrier `bar`) each pass 4 slots;
// writes the row's ascending distinct blocks to out_blocks[0, k) (-1 padded)
// and their number to *out_count (if not null). Every thread of the group
// must call it; `live` false computes but writes nothing.
__device__ __forceinline__ void row_blocks128(const int32_t (&slot)[4], int k, int block_size, int32_t* out_blocks,
                                              int32_t* out_count, BlockScratch& S, int t, int bar, bool live) {
  const int lane = t & 31, warp = t >> 5;
  int32_t b[4];
  bool v4[4];
  int32_t lmin = 0x7FFFFFFF, lmax = -1;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v4[e] = slot[e] >= 0;
    b[e] = v4[e] ? slot[e] / block_size : 0;
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
  named_bar(bar, kBlockThreads);
  int32_t bmin = S.wmin[0], bmax = S.wmax[0];
#pragma unroll
  for (int w = 1; w < kBlockThreads / 32; ++w) {
    bmin = min(bmin, S.wmin[w]);
    bmax = max(bmax, S.wmax[w]);
  }
  if (bmax < 0 || (long long)bmax - bmin < 32LL * kBitmapWords) {
    // ---- bitmap: bit (block - bmin) of the row's 512 words
    const int words = bmax < 0 ? 0 : (bmax - bmin) / 32 + 1;
    for (int w = t; w < words; w += kBlockThreads) S.u.bitmap[w] = 0u;
    named_bar(bar, kBlockThreads);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (v4[e]) atomicOr(&S.u.bitmap[(b[e] - bmin) >> 5], 1u << ((b[e] - bmin) & 31));
    }
    named_bar(bar, kBlockThreads);
    // Thread t owns words t + 128e (e = 0..3), so a row spanning few words
    // spreads its set bits over many threads. Its four word counts travel
    // as 16-bit fields of one 64-bit value through a single scan: the first
    // word of field e lands after every word of the fields before it, then
    // after the same field's words of lower threads (ascending word order).
    uint32_t wv[4];
    unsigned long long packed = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int w = t + kBlockThreads * e;
      wv[e] = w < words ? S.u.bitmap[w] : 0u;
      packed |= static_cast<unsigned long long>(__popc(wv[e])) << (16 * e);
    }
    unsigned long long incl = packed;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const unsigned long long o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= d) incl += o;
    }
    if (lane == 31) S.wtot[warp] = incl;
    named_bar(bar, kBlockThreads);
    unsigned long long before = incl - packed, total = 0;
#pragma unroll
    for (int w = 0; w < kBlockThreads / 32; ++w) {
      const unsigned long long v = S.wtot[w];
      before += w < warp ? v : 0ull;
      total += v;
    }
    named_bar(bar, kBlockThreads);  // the scratch is read before the group reuses it
    if (!live) return;
    int count = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int out = count + static_cast<int>((before >> (16 * e)) & 0xFFFFu);
      count += static_cast<int>((total >> (16 * e)) & 0xFFFFu);
      uint32_t m = wv[e];
      while (m) {
        const int bit = __ffs(m) - 1;
        m &= m - 1u;
        out_blocks[out++] = bmin + 32 * (t + kBlockThreads * e) + bit;
      }
    }
    for (int j = count + t; j < k; j += kBlockThreads) out_blocks[j] = -1;
    if (out_count && t == 0) *out_count = count;
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
  int pos = block_exscan<kBlockThreads>(c, &total, S.wsum, t, bar);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (e < c) {
      S.u.s.key[pos] = ~static_cast<uint32_t>(bc[e]);
      S.u.s.idx[pos] = pos;
      ++pos;
    }
  }
  named_bar(bar, kBlockThreads);
  // ascending blocks: sorted position 4t + e holds blk[e] (-1: padding)
  unsigned long long v[4];
  bitonic_sort512_128(S.u.s.key, S.u.s.idx, total, S.u.s.sortbuf, v, t, bar);
  int32_t blk[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) blk[e] = v[e] ? static_cast<int32_t>(~static_cast<uint32_t>(v[e] >> 32)) : -1;
  if (lane == 31) S.last[warp] = blk[3];
  named_bar(bar, kBlockThreads);
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
  int out = block_exscan<kBlockThreads>(nf, &count, S.wsum, t, bar);
  named_bar(bar, kBlockThreads);  // the scratch is read before the group reuses it
  if (!live) return;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (first[e]) out_blocks[out++] = blk[e];
  }
  for (int j = count + t; j < k; j += kBlockThreads) out_blocks[j] = -1;
  if (out_count && t == 0) *out_count = count;
}

}  // namespace sai
