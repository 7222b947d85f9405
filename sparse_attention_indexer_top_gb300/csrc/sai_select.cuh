// Shared-memory top-k building blocks used by every selection kernel:
//   * order_key: fp32 -> uint32 key whose unsigned order is the score order;
//   * append: warp-aggregated append of (key, index) candidates;
//   * select_topk: exact top-K of a candidate list by (key desc, index asc)
//     with range-based radix passes over 8-bit digits in shared memory;
//   * bitonic_desc512: sort 512 (key, index) pairs, one per thread.
//
// The ordering rule (higher score first, equal scores to the lower row-local
// index) is the deterministic order the library exposes; the pages of
// sglang PR #37889 "[AMD] Enable GLM DSA prefill top-k to the v2 kernel"
// define the window and page-table addressing (Modifications) but not the
// order among the k outputs.
#pragma once
#include <cstdint>

#include "sai_ptx.cuh"

namespace sai {

constexpr int kTopK = 512;

// -0.0 is folded into +0.0 first (the two compare equal as scores).
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(__fadd_rn(x, 0.0f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

struct SelectScratch {
  uint32_t hist[256];
  uint32_t wmin[32], wmax[32], wcnt[32];
  uint32_t vmin, vmax, nact;
  uint32_t bin, need_after, bin_count;
  int out_cnt;
  uint32_t tau;
};

// Result of a threshold search over a set of uint32 values: the selected
// values are those whose offset (v - base) >> lo is > prefix, plus, among
// the ones equal to prefix, either all of them (all_eq) or `need` of them.
struct Threshold {
  uint32_t base, prefix, need;
  int lo;
  bool all_eq;
};

__device__ __forceinline__ uint32_t shr64(uint32_t o, int lo) {
  return static_cast<uint32_t>(static_cast<uint64_t>(o) >> lo);
}

// Find the threshold bin of the `need` largest values among the active
// values of the group. Each thread visits its own share through
// `each(fn)`, which calls fn(v) once per active value v of the thread. All
// NT threads of the group call it; `bar` is the group's named barrier id.
// `need` must not exceed the number of active values.
template <int NT, typename Each>
__device__ Threshold radix_refine(Threshold t, SelectScratch& sc, int tid, int bar, Each each);

template <int NT, typename Each>
__device__ Threshold radix_threshold_each(uint32_t need, SelectScratch& sc, int tid, int bar, Each each) {
  constexpr int NW = NT / 32;
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t lmin = 0xFFFFFFFFu, lmax = 0u, lcnt = 0u;
  each([&](uint32_t v) {
    lmin = min(lmin, v);
    lmax = max(lmax, v);
    ++lcnt;
  });
  lmin = __reduce_min_sync(0xFFFFFFFFu, lmin);
  lmax = __reduce_max_sync(0xFFFFFFFFu, lmax);
  lcnt = __reduce_add_sync(0xFFFFFFFFu, lcnt);
  if (lane == 0) {
    sc.wmin[warp] = lmin;
    sc.wmax[warp] = lmax;
    sc.wcnt[warp] = lcnt;
  }
  named_bar(bar, NT);
  if (warp == 0) {
    uint32_t a = lane < NW ? sc.wmin[lane] : 0xFFFFFFFFu;
    uint32_t b = lane < NW ? sc.wmax[lane] : 0u;
    uint32_t c = lane < NW ? sc.wcnt[lane] : 0u;
    a = __reduce_min_sync(0xFFFFFFFFu, a);
    b = __reduce_max_sync(0xFFFFFFFFu, b);
    c = __reduce_add_sync(0xFFFFFFFFu, c);
    if (lane == 0) {
      sc.vmin = a;
      sc.vmax = b;
      sc.nact = c;
    }
  }
  named_bar(bar, NT);
  Threshold t;
  t.base = sc.vmin;
  const uint32_t span = sc.vmax - sc.vmin;
  t.lo = span ? 32 - __clz(span) : 0;
  t.prefix = 0;
  t.need = need;
  t.all_eq = (sc.nact == need);
  return radix_refine<NT>(t, sc, tid, bar, each);
}

// Narrow a threshold 8 bits at a time: among the values whose bits above t.lo
// (relative to t.base) equal t.prefix, find the t.need-th largest.
template <int NT, typename Each>
__device__ Threshold radix_refine(Threshold t, SelectScratch& sc, int tid, int bar, Each each) {
  const int lane = tid & 31, warp = tid >> 5;
  while (t.lo > 0 && !t.all_eq) {
    const int dlo = t.lo > 8 ? t.lo - 8 : 0;
    const int dbits = t.lo - dlo;
    const uint32_t dmask = (1u << dbits) - 1u;
    for (int i = tid; i < 256; i += NT) sc.hist[i] = 0;
    named_bar(bar, NT);
    each([&](uint32_t v) {
      const uint32_t o = v - t.base;
      if (shr64(o, t.lo) == t.prefix) atomicAdd(&sc.hist[(o >> dlo) & dmask], 1u);
    });
    named_bar(bar, NT);
    if (warp == 0) {
      // Lane l owns bins [8l, 8l+8); scan from the top bin down.
      uint32_t h[8];
      uint32_t tot = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        h[i] = sc.hist[lane * 8 + i];
        tot += h[i];
      }
      // inclusive suffix sum over lanes (lane 31 holds the highest bins)
      uint32_t suf = tot;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_down_sync(0xFFFFFFFFu, suf, d);
        if (lane + d < 32) suf += o;
      }
      uint32_t above = suf - tot;  // count in bins of higher lanes
      const uint32_t nd = t.need;
      if (above < nd && nd <= suf) {
#pragma unroll
        for (int i = 7; i >= 0; --i) {
          if (above < nd && nd <= above + h[i]) {
            sc.bin = lane * 8 + i;
            sc.need_after = nd - above;
            sc.bin_count = h[i];
          }
          above += h[i];
        }
      }
    }
    named_bar(bar, NT);
    t.prefix = (t.prefix << dbits) | sc.bin;
    t.need = sc.need_after;
    t.all_eq = (sc.bin_count == t.need);
    t.lo = dlo;
  }
  return t;
}

// radix_threshold_each with a wider first step: the values are counted in
// up to 512 bins fitted to [vmin, vmax] (`bins`: 512 words of scratch), and
// when the bin that holds the need-th largest value then holds at most 32
// values, one warp ranks them directly, so no further pass over the values
// is made; otherwise the 8-bit passes continue inside that bin.
template <int NT, typename Each>
__device__ Threshold radix_threshold_fast(uint32_t need, SelectScratch& sc, uint32_t* bins, int tid, int bar,
                                          Each each) {
  constexpr int NW = NT / 32;
  constexpr int kBins = 512;
  constexpr int BPT = kBins / NT;  // bins per thread in the scan
  static_assert(kBins % NT == 0, "whole bins per thread");
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t lmin = 0xFFFFFFFFu, lmax = 0u, lcnt = 0u;
  each([&](uint32_t v) {
    lmin = min(lmin, v);
    lmax = max(lmax, v);
    ++lcnt;
  });
  lmin = __reduce_min_sync(0xFFFFFFFFu, lmin);
  lmax = __reduce_max_sync(0xFFFFFFFFu, lmax);
  lcnt = __reduce_add_sync(0xFFFFFFFFu, lcnt);
  if (lane == 0) {
    sc.wmin[warp] = lmin;
    sc.wmax[warp] = lmax;
    sc.wcnt[warp] = lcnt;
  }
#pragma unroll
  for (int i = 0; i < BPT; ++i) bins[BPT * tid + i] = 0u;
  if (tid == 0) sc.out_cnt = 0;
  named_bar(bar, NT);
  uint32_t vmin = sc.wmin[0], vmax = sc.wmax[0], nact = sc.wcnt[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) {
    vmin = min(vmin, sc.wmin[w]);
    vmax = max(vmax, sc.wmax[w]);
    nact += sc.wcnt[w];
  }
  Threshold t;
  t.base = vmin;
  const uint32_t span = vmax - vmin;
  t.lo = span ? 32 - __clz(span) : 0;
  t.prefix = 0;
  t.need = need;
  t.all_eq = (nact == need);
  if (t.lo == 0 || t.all_eq) return t;  // (uniform: every thread read the same partials)
  const int dlo = t.lo > 9 ? t.lo - 9 : 0;
  each([&](uint32_t v) { atomicAdd(&bins[(v - t.base) >> dlo], 1u); });
  named_bar(bar, NT);  // also: every thread has read the pass-0 partials
  // bin holding the need-th largest value; thread tid owns bins [BPT*tid, BPT*tid + BPT)
  uint32_t h[BPT];
  uint32_t tot = 0;
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    h[i] = bins[BPT * tid + i];
    tot += h[i];
  }
  uint32_t suf = tot;  // inclusive suffix sum over lanes (higher lanes own higher bins)
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_down_sync(0xFFFFFFFFu, suf, d);
    if (lane + d < 32) suf += o;
  }
  if (lane == 0) sc.wcnt[warp] = suf;  // warp total
  named_bar(bar, NT);
  uint32_t above = suf - tot;
#pragma unroll
  for (int w = 0; w < NW; ++w) above += w > warp ? sc.wcnt[w] : 0u;
  if (above < need && need <= above + tot) {
#pragma unroll
    for (int i = BPT - 1; i >= 0; --i) {
      if (above < need && need <= above + h[i]) {
        sc.bin = BPT * tid + i;
        sc.need_after = need - above;
        sc.bin_count = h[i];
      }
      above += h[i];
    }
  }
  named_bar(bar, NT);
  const uint32_t B = sc.bin, nb = sc.need_after, cb = sc.bin_count;
  t.prefix = B;
  t.need = nb;
  t.all_eq = (cb == nb);
  t.lo = dlo;
  if (t.all_eq || dlo == 0) return t;
  if (cb > 32) return radix_refine<NT>(t, sc, tid, bar, each);
  // few values in the bin: collect them (sc.wmin holds 32) and rank them in one warp
  each([&](uint32_t v) {
    if (((v - t.base) >> dlo) == B) sc.wmin[atomicAdd(&sc.out_cnt, 1)] = v;
  });
  named_bar(bar, NT);
  if (warp == 0) {
    const uint32_t x = lane < (int)cb ? sc.wmin[lane] : 0u;
    uint32_t gt = 0, eq = 0;
    for (uint32_t j = 0; j < cb; ++j) {
      const uint32_t y = sc.wmin[j];
      gt += y > x ? 1u : 0u;
      eq += y == x ? 1u : 0u;
    }
    // the nb-th largest of the bin (lanes holding the same value write the same)
    if (lane < (int)cb && gt < nb && nb <= gt + eq) {
      sc.tau = x;
      sc.need_after = nb - gt;
      sc.bin_count = eq;
    }
  }
  named_bar(bar, NT);
  t.prefix = sc.tau - t.base;
  t.lo = 0;
  t.need = sc.need_after;
  t.all_eq = (sc.bin_count == t.need);
  return t;
}

// The same over the entries j in [0, n) of the group, thread tid taking
// j = tid, tid + NT, ...; entry j is active with value v when get(j, v).
template <int NT, typename Get>
__device__ Threshold radix_threshold(int n, uint32_t need, SelectScratch& sc, int tid, int bar, Get get) {
  return radix_threshold_each<NT>(need, sc, tid, bar, [&](auto fn) {
    for (int j = tid; j < n; j += NT) {
      uint32_t v;
      if (get(j, v)) fn(v);
    }
  });
}

__device__ __forceinline__ int thr_cmp(const Threshold& t, uint32_t v) {
  const uint32_t hi = shr64(v - t.base, t.lo);
  return hi > t.prefix ? 1 : (hi == t.prefix ? 0 : -1);
}

// Keep the top K of ckey/cidx[0, n) by (key desc, index asc); the survivors
// are moved to [0, K) (in no particular order) through `aux_key/aux_idx`
// (K entries). Returns a valid strict filter threshold: every entry not
// kept, and every later entry (larger index) with key <= the returned
// value, is outside the top K. Requires n > K.
template <int NT>
__device__ uint32_t select_topk(uint32_t* ckey, int32_t* cidx, int n, int K, uint32_t* aux_key,
                                int32_t* aux_idx, SelectScratch& sc, int tid, int bar) {
  const Threshold t = radix_threshold<NT>(n, (uint32_t)K, sc, tid, bar, [&](int j, uint32_t& v) {
    v = ckey[j];
    return true;
  });
  Threshold ti{};
  bool ties = !t.all_eq;
  if (ties) {
    // All tied entries carry the same key; take the t.need lowest indices.
    ti = radix_threshold<NT>(n, t.need, sc, tid, bar, [&](int j, uint32_t& v) {
      v = 0x7FFFFFFFu - static_cast<uint32_t>(cidx[j]);
      return thr_cmp(t, ckey[j]) == 0;
    });
  }
  if (tid == 0) sc.out_cnt = 0;
  named_bar(bar, NT);
  const int lane = tid & 31;
  for (int j0 = 0; j0 < n; j0 += NT) {
    const int j = j0 + tid;
    bool sel = false;
    uint32_t key = 0;
    int32_t idx = 0;
    if (j < n) {
      key = ckey[j];
      idx = cidx[j];
      const int c = thr_cmp(t, key);
      sel = c > 0 || (c == 0 && (!ties || thr_cmp(ti, 0x7FFFFFFFu - static_cast<uint32_t>(idx)) >= 0));
    }
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, sel);
    if (m) {
      int base = 0;
      if (lane == 0) base = atomicAdd(&sc.out_cnt, __popc(m));
      base = __shfl_sync(0xFFFFFFFFu, base, 0);
      if (sel) {
        const int pos = base + __popc(m & ((1u << lane) - 1u));
        if (pos < K) {  // exactly K are selected; the guard only bounds the buffer
          aux_key[pos] = key;
          aux_idx[pos] = idx;
        }
      }
    }
  }
  named_bar(bar, NT);
  for (int j = tid; j < K; j += NT) {
    ckey[j] = aux_key[j];
    cidx[j] = aux_idx[j];
  }
  // lowest key of the threshold bin: <= the K-th key
  const uint32_t tau = t.base + static_cast<uint32_t>(static_cast<uint64_t>(t.prefix) << t.lo);
  named_bar(bar, NT);
  return tau;
}

// Composite sort key: key in the high word, bit-inverted index in the low
// word, so a larger composite means higher score, then lower index. Padding
// entries use 0, which sorts after every real entry.
__device__ __forceinline__ unsigned long long composite(uint32_t key, int32_t idx) {
  return (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(idx));
}


// ------------------------------------------------------------------------
// Block-wide helpers for a 512-thread group (named barrier `bar`).

// Exclusive prefix sum of `c` over the group; *total receives the sum.
__device__ __forceinline__ int block_exscan512(int c, int* total, uint32_t* wsum, int tid, int bar) {
  const int lane = tid & 31, warp = tid >> 5;
  int incl = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) wsum[warp] = (uint32_t)incl;
  named_bar(bar, 512);
  int off = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < 16; ++w) {
    const int v = (int)wsum[w];
    off += w < warp ? v : 0;
    tot += v;
  }
  *total = tot;
  return off + incl - c;
}

// Threshold bin over a 4096-bin histogram of key >> 20 (8 bins per thread):
// the bin B with count(bins > B) < need <= count(bins >= B). Returns -1 if
// the histogram holds fewer than `need`. *need_in_bin / *bin_count describe
// the cut inside B. Two barriers; `wsum` needs 16 words.
struct BinCut {
  int bin;
  uint32_t need_in_bin;
  uint32_t bin_count;
};

__device__ __forceinline__ BinCut hist_cut4096(const uint32_t* hist, uint32_t need, uint32_t* wsum, uint32_t* bcast,
                                               int tid, int bar) {
  const int lane = tid & 31, warp = tid >> 5;
  const uint4 a = reinterpret_cast<const uint4*>(hist)[2 * tid];
  const uint4 b = reinterpret_cast<const uint4*>(hist)[2 * tid + 1];
  const uint32_t h[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += h[i];
  // inclusive suffix sum across lanes (higher lanes own higher bins)
  uint32_t suf = s;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_down_sync(0xFFFFFFFFu, suf, d);
    if (lane + d < 32) suf += o;
  }
  if (lane == 0) wsum[warp] = suf;  // warp total
  if (tid == 0) bcast[0] = 0xFFFFFFFFu;
  named_bar(bar, 512);
  uint32_t above_w = 0;
#pragma unroll
  for (int w = 0; w < 16; ++w) above_w += w > warp ? wsum[w] : 0u;
  uint32_t above = above_w + suf - s;
  if (above < need && need <= above + s) {
#pragma unroll
    for (int i = 7; i >= 0; --i) {
      if (above < need && need <= above + h[i]) {
        bcast[0] = (uint32_t)(8 * tid + i);
        bcast[1] = need - above;
        bcast[2] = h[i];
      }
      above += h[i];
    }
  }
  named_bar(bar, 512);
  BinCut c;
  c.bin = bcast[0] == 0xFFFFFFFFu ? -1 : (int)bcast[0];
  c.need_in_bin = bcast[1];
  c.bin_count = bcast[2];
  return c;
}

// Exact top-K (K = 512) of ckey/cidx[0, n), n > K, by (key desc, index asc),
// written to aux_key/aux_idx[0, K). Keys are counted in 4096 bins,
// bin = (key - kmin) >> shift, which must be < 4096 for every key (kmin <=
// every key); bins fitted to the keys' range leave few keys in the bin that
// holds the K-th. `hist` (4096 words) is scratch and is left zeroed. CAPT
// bounds n.
template <int CAPT>
__device__ void fast_select512(const uint32_t* ckey, const int32_t* cidx, int n, uint32_t kmin, int shift,
                               uint32_t* hist, uint32_t* aux_key, int32_t* aux_idx, SelectScratch& sc,
                               uint32_t* bcast, int tid, int bar) {
  constexpr int K = kTopK;
  constexpr int M = (CAPT + 511) / 512;
  auto bin_of = [&](uint32_t key) { return (key - kmin) >> shift; };
  for (int j = tid; j < n; j += 512) atomicAdd(&hist[bin_of(ckey[j])], 1u);
  named_bar(bar, 512);
  const BinCut cut = hist_cut4096(hist, K, sc.wmin, bcast, tid, bar);
  const uint32_t B = (uint32_t)cut.bin;
  // inside the threshold bin: exact cut by key, then by index for ties
  Threshold t{};
  t.all_eq = cut.bin_count == cut.need_in_bin;
  Threshold ti{};
  bool ties = false;
  if (!t.all_eq) {
    t = radix_threshold<512>(n, cut.need_in_bin, sc, tid, bar, [&](int j, uint32_t& v) {
      v = ckey[j];
      return bin_of(v) == B;
    });
    ties = !t.all_eq;
    if (ties) {
      ti = radix_threshold<512>(n, t.need, sc, tid, bar, [&](int j, uint32_t& v) {
        v = 0x7FFFFFFFu - static_cast<uint32_t>(cidx[j]);
        return bin_of(ckey[j]) == B && thr_cmp(t, ckey[j]) == 0;
      });
    }
  }
  // clear the histogram for the next user (8 words per thread)
  reinterpret_cast<uint4*>(hist)[2 * tid] = make_uint4(0, 0, 0, 0);
  reinterpret_cast<uint4*>(hist)[2 * tid + 1] = make_uint4(0, 0, 0, 0);
  uint32_t selm = 0;
  int c = 0;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int j = tid + 512 * m;
    if (j < n) {
      const uint32_t key = ckey[j];
      const uint32_t hb = bin_of(key);
      bool sel = hb > B;
      if (hb == B) {
        if (cut.bin_count == cut.need_in_bin) {
          sel = true;
        } else {
          const int cc = thr_cmp(t, key);
          sel = cc > 0 ||
                (cc == 0 && (!ties || thr_cmp(ti, 0x7FFFFFFFu - static_cast<uint32_t>(cidx[j])) >= 0));
        }
      }
      if (sel) {
        selm |= 1u << m;
        ++c;
      }
    }
  }
  int total;
  int pos = block_exscan512(c, &total, sc.wcnt, tid, bar);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    if (selm & (1u << m)) {
      const int j = tid + 512 * m;
      if (pos < K) {
        aux_key[pos] = ckey[j];
        aux_idx[pos] = cidx[j];
      }
      ++pos;
    }
  }
  named_bar(bar, 512);
}

// Float threshold equivalent to "order key >= tau" for every non-NaN x.
__device__ __forceinline__ float tau_float(uint32_t tau) {
  if (tau <= 0x007FFFFFu) return __int_as_float(0xFF800000);  // -inf: everything passes
  return key_to_float(tau);
}

// ------------------------------------------------------------------------
// Helpers for a group of NT threads (NT a multiple of 32, NT <= 512).

template <int NT>
__device__ __forceinline__ int block_exscan(int c, int* total, uint32_t* wsum, int tid, int bar) {
  constexpr int NW = NT / 32;
  const int lane = tid & 31, warp = tid >> 5;
  int incl = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) wsum[warp] = (uint32_t)incl;
  named_bar(bar, NT);
  int off = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const int v = (int)wsum[w];
    off += w < warp ? v : 0;
    tot += v;
  }
  *total = tot;
  return off + incl - c;
}

// Sort the `cnt` (<= 512) entries of aux_key/aux_idx by (key desc, index
// asc): 16 runs of 32 are sorted by warp shuffles, then each entry's rank is
// its place in its run plus, for every other run, the number of entries
// before it (binary search over the run's 32-bit keys: a run spans the 32
// banks once, so the search is conflict-free; equal keys are then ordered
// by index). Thread tid handles runs warp, warp+NW, ...; for each, k/ix[e]
// is its entry (ix = -1: padding) and rank[e] its output position.
// `runs_key` / `runs_idx` need 512 entries each.
template <int NT>
__device__ __forceinline__ void rank_sort(const uint32_t* aux_key, const int32_t* aux_idx, int cnt,
                                          uint32_t* runs_key, int32_t* runs_idx, uint32_t (&k)[kTopK / NT],
                                          int32_t (&ix)[kTopK / NT], int (&rank)[kTopK / NT], int tid, int bar) {
  constexpr int NW = NT / 32;
  constexpr int E = kTopK / NT;
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int r = warp + NW * e;
    const int j = 32 * r + lane;
    unsigned long long x = j < cnt ? composite(aux_key[j], aux_idx[j]) : 0ull;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
      const bool asc = (lane & size) != 0;
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const unsigned long long p = __shfl_xor_sync(0xFFFFFFFFu, x, stride);
        const bool lower = (lane & stride) == 0;
        x = (lower != asc) ? (x > p ? x : p) : (x < p ? x : p);
      }
    }
    k[e] = static_cast<uint32_t>(x >> 32);
    ix[e] = x ? static_cast<int32_t>(~static_cast<uint32_t>(x & 0xFFFFFFFFull)) : -1;
    runs_key[j] = k[e];
    runs_idx[j] = ix[e];
  }
  named_bar(bar, NT);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int r0 = warp + NW * e;
    int rk = lane;
    const uint32_t xk = k[e];
    const int32_t xi = ix[e];
#pragma unroll 4
    for (int r = 0; r < 16; ++r) {
      if (r == r0) continue;
      const uint32_t* run = runs_key + 32 * r;
      int pos = run[31] > xk ? 32 : 0;
#pragma unroll
      for (int s = 16; s > 0; s >>= 1)
        if (pos + s <= 31 && run[pos + s - 1] > xk) pos += s;
      // padding entries (key 0, index -1) never precede a real entry
      while (pos < 32 && run[pos] == xk && runs_idx[32 * r + pos] >= 0 && runs_idx[32 * r + pos] < xi) ++pos;
      rk += pos;
    }
    rank[e] = rk;
  }
  named_bar(bar, NT);
}

// Exact top-K (K = 512) over W sub-lists, one per warp of the group:
// sub-list w holds counts[w] <= SUB entries at key/idx[w * SUB ...] and is
// walked by warp w alone, so every pass touches only filled entries. Writes
// the top K by (key desc, index asc) to aux_key/aux_idx[0, K) (unordered).
// Requires the total to exceed K. Returns the lowest key of the final
// threshold bin (<= the K-th key).
template <int NT, int W, int SUB>
__device__ uint32_t select512_sub_to_aux(const uint32_t* key, const int32_t* idx, const int (&counts)[W],
                                         uint32_t* aux_key, int32_t* aux_idx, SelectScratch& sc, int tid, int bar) {
  static_assert(NT == 32 * W, "one warp per sub-list");
  constexpr int K = kTopK;
  constexpr int M = SUB / 32;
  static_assert(SUB % 32 == 0 && M <= 32, "entries per lane fit a 32-bit mask");
  const int lane = tid & 31, w = tid >> 5;
  int c = counts[0];
#pragma unroll
  for (int u = 1; u < W; ++u) c = w == u ? counts[u] : c;  // no dynamic index: keeps counts in registers
  const uint32_t* const mk = key + w * SUB;
  const int32_t* const mi = idx + w * SUB;
  // aux_key is this call's output and free until the end: it serves as bins
  const Threshold t = radix_threshold_fast<NT>((uint32_t)K, sc, aux_key, tid, bar, [&](auto fn) {
    for (int j = lane; j < c; j += 32) fn(mk[j]);
  });
  Threshold ti{};
  const bool ties = !t.all_eq;
  if (ties) {
    ti = radix_threshold_each<NT>(t.need, sc, tid, bar, [&](auto fn) {
      for (int j = lane; j < c; j += 32)
        if (thr_cmp(t, mk[j]) == 0) fn(0x7FFFFFFFu - static_cast<uint32_t>(mi[j]));
    });
  }
  uint32_t selm = 0;
  int cs = 0;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int j = lane + 32 * m;
    if (j < c) {
      const int cc = thr_cmp(t, mk[j]);
      const bool sel = cc > 0 || (cc == 0 && (!ties || thr_cmp(ti, 0x7FFFFFFFu - static_cast<uint32_t>(mi[j])) >= 0));
      if (sel) {
        selm |= 1u << m;
        ++cs;
      }
    }
  }
  int total;
  int pos = block_exscan<NT>(cs, &total, sc.wcnt, tid, bar);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    if (selm & (1u << m)) {
      const int j = lane + 32 * m;
      if (pos < K) {
        aux_key[pos] = mk[j];
        aux_idx[pos] = mi[j];
      }
      ++pos;
    }
  }
  named_bar(bar, NT);
  return t.base + static_cast<uint32_t>(static_cast<uint64_t>(t.prefix) << t.lo);
}

// Sort cnt (<= 512) entries of aux_key/aux_idx by (key desc, index asc)
// with a bitonic network over 128 threads, 4 entries per thread: thread t
// holds virtual positions 4t .. 4t+3, so strides 1-2 stay in registers,
// strides 4-64 use warp shuffles and strides 128-256 go through `buf`
// (512 entries). On return v[j] is the entry of output rank 4t + j
// (composite key, 0 = padding).
__device__ __forceinline__ void bitonic_sort512_128(const uint32_t* aux_key, const int32_t* aux_idx, int cnt,
                                                    unsigned long long* buf, unsigned long long (&v)[4], int tid,
                                                    int bar) {
  const int lane = tid & 31;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = tid + 128 * j;  // any placement works: everything gets sorted
    v[j] = e < cnt ? composite(aux_key[e], aux_idx[e]) : 0ull;
  }
#pragma unroll
  for (int size = 2; size <= 512; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride < 4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (j & stride) continue;
          const int j2 = j | stride;
          const bool asc = ((4 * tid + j) & size) != 0;
          const unsigned long long x = v[j], y = v[j2];
          const unsigned long long hi = x > y ? x : y, lo = x > y ? y : x;
          v[j] = asc ? lo : hi;
          v[j2] = asc ? hi : lo;
        }
      } else if (stride < 128) {
        const int d = stride >> 2;  // lane distance
        const bool lower = (lane & d) == 0;
        const bool asc = ((4 * tid) & size) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const unsigned long long p = __shfl_xor_sync(0xFFFFFFFFu, v[j], d);
          v[j] = (lower != asc) ? (v[j] > p ? v[j] : p) : (v[j] < p ? v[j] : p);
        }
      } else {
        const int d = stride >> 2;  // thread distance
        const bool lower = (tid & d) == 0;
        const bool asc = ((4 * tid) & size) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) buf[4 * tid + j] = v[j];
        named_bar(bar, 128);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const unsigned long long p = buf[4 * (tid ^ d) + j];
          v[j] = (lower != asc) ? (v[j] > p ? v[j] : p) : (v[j] < p ? v[j] : p);
        }
        named_bar(bar, 128);
      }
    }
  }
}

// Exact output ranks of the cnt (<= 512) entries of aux_key/aux_idx under
// (key desc, index asc), without a sorting network. Keys are binned into
// 1024 bins over [kmin, kmax] (bin 0 holds the highest keys), the bins are
// counted and prefix-summed, and an entry's rank is its bin's offset plus
// the number of entries of its own bin that precede it, found by comparing
// with each of them (a bin holds one or two entries on typical data).
// Thread tid handles entries j = tid + NT*e: k/ix[e] is the entry (ix = -1:
// none) and rank[e] its output position. `hist` needs 1024 words and
// `bucket` 512 halfwords, both free for the call. Returns false, leaving
// aux untouched, when some bin holds more than 16 entries (heavy ties or a
// very uneven range); the caller then sorts another way.
template <int NT>
__device__ bool bucket_rank512(const uint32_t* aux_key, const int32_t* aux_idx, int cnt, uint32_t* hist,
                               uint16_t* bucket, SelectScratch& sc, uint32_t (&k)[kTopK / NT],
                               int32_t (&ix)[kTopK / NT], int (&rank)[kTopK / NT], int tid, int bar) {
  constexpr int E = kTopK / NT;
  constexpr int NW = NT / 32;
  constexpr int kBins = 1024;
  constexpr int B = kBins / NT;  // bins per thread in the scan
  constexpr int kMaxBin = 16;
  static_assert(B % 4 == 0, "bins per thread in whole uint4s");
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t lmin = 0xFFFFFFFFu, lmax = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = tid + NT * e;
    const bool v = j < cnt;
    k[e] = v ? aux_key[j] : 0u;
    ix[e] = v ? aux_idx[j] : -1;
    rank[e] = j;
    if (v) {
      lmin = min(lmin, k[e]);
      lmax = max(lmax, k[e]);
    }
  }
  lmin = __reduce_min_sync(0xFFFFFFFFu, lmin);
  lmax = __reduce_max_sync(0xFFFFFFFFu, lmax);
  if (lane == 0) {
    sc.wmin[warp] = lmin;
    sc.wmax[warp] = lmax;
  }
#pragma unroll
  for (int i = 0; i < B / 4; ++i) reinterpret_cast<uint4*>(hist)[tid * (B / 4) + i] = make_uint4(0u, 0u, 0u, 0u);
  named_bar(bar, NT);
  uint32_t kmin = sc.wmin[0], kmax = sc.wmax[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) {
    kmin = min(kmin, sc.wmin[w]);
    kmax = max(kmax, sc.wmax[w]);
  }
  const uint32_t span = kmax - kmin;
  const int shift = span >= (uint32_t)kBins ? (32 - __clz(span)) - 10 : 0;
  int bin[E], slot[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    bin[e] = (int)((kmax - k[e]) >> shift);
    slot[e] = ix[e] >= 0 ? (int)atomicAdd(&hist[bin[e]], 1u) : 0;
  }
  named_bar(bar, NT);
  // exclusive prefix sum of the bins in place; thread tid owns B bins
  uint32_t h[B];
#pragma unroll
  for (int i = 0; i < B / 4; ++i) {
    const uint4 q = reinterpret_cast<const uint4*>(hist)[tid * (B / 4) + i];
    h[4 * i] = q.x;
    h[4 * i + 1] = q.y;
    h[4 * i + 2] = q.z;
    h[4 * i + 3] = q.w;
  }
  uint32_t tot = 0;
#pragma unroll
  for (int i = 0; i < B; ++i) {
    const uint32_t c = h[i];
    h[i] = tot;
    tot += c;
  }
  uint32_t incl = tot;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) sc.wcnt[warp] = incl;
  named_bar(bar, NT);
  uint32_t off = incl - tot;
#pragma unroll
  for (int w = 0; w < NW; ++w) off += w < warp ? sc.wcnt[w] : 0u;
#pragma unroll
  for (int i = 0; i < B / 4; ++i)
    reinterpret_cast<uint4*>(hist)[tid * (B / 4) + i] =
        make_uint4(h[4 * i] + off, h[4 * i + 1] + off, h[4 * i + 2] + off, h[4 * i + 3] + off);
  named_bar(bar, NT);
  int start[E], size[E];
  bool heavy = false;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    start[e] = 0;
    size[e] = 0;
    if (ix[e] >= 0) {
      start[e] = (int)hist[bin[e]];
      size[e] = (bin[e] < kBins - 1 ? (int)hist[bin[e] + 1] : cnt) - start[e];
      bucket[start[e] + slot[e]] = static_cast<uint16_t>(tid + NT * e);
      heavy = heavy || size[e] > kMaxBin;
    }
  }
  if (named_bar_or(bar, NT, heavy)) return false;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    int r = 0;
    if (size[e] > 1) {
      for (int m = 0; m < size[e]; ++m) {
        const int o = bucket[start[e] + m];
        const uint32_t ko = aux_key[o];
        const int32_t io = aux_idx[o];
        r += (ko > k[e] || (ko == k[e] && io < ix[e])) ? 1 : 0;
      }
    }
    rank[e] = start[e] + r;
  }
  return true;
}

}  // namespace sai
