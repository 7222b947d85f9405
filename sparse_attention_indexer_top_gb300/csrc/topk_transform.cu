// topk_transform: per-row window top-512 + page-table transform.
//
// Contract (sglang PR #37889 "[AMD] Enable GLM DSA prefill top-k to the v2
// kernel", Modifications): row i reads scores[i, row_starts[i] :
// row_starts[i] + seq_lens[i]] (row_starts optional -> 0), picks the top-k
// row-local positions and maps them through page_tables[row_to_batch[i]]
// (row_to_batch optional -> i) to physical KV slots. Building the physical
// addressing inside the top-k kernel is the "merge build sparse block into
// topk" step of ROCm/ATOM PR #1282.
//
// GB300 design: one warp owns one work unit (a row, or a chunk of a long
// row) at a time, with no synchronisation beyond the warp, so an SM runs a
// dozen fully independent streams and hides each one's latency with the
// others.
//   * Each warp (a one-warp CTA) keeps its own ring of six 1 KB shared-memory
//     stages filled with 1-D bulk TMA copies (cp.async.bulk + mbarrier
//     complete_tx, evict-first in L2: every score is read once). The
//     16-byte-aligned interior of each window goes through TMA; its <= 3
//     leading and <= 3 trailing elements (any row stride, any row start) are
//     read with scalar loads. This is the scalar path the pages require for
//     strides that are not a multiple of 4, folded into every row instead of
//     a separate fallback kernel.
//   * Each lane compares its 8 scores of a stage against the running
//     threshold tau and the warp appends the survivors (order key, row-local
//     index) to its candidate list with one ballot per element slot. When
//     the list is nearly full it is cut to the exact top 512 (warp radix
//     select in shared memory) and tau rises to that cut, so the filter
//     stays exact: every dropped element is beaten by 512 kept ones.
//   * A unit starts from a threshold extrapolated from the warp's previous
//     unit. Whether it was low enough is checked exactly at the unit end (at
//     least min(n, 512) elements must have passed); if not, the unit is redone
//     from global memory with no threshold.
//   * At the end of a unit the candidates are cut to 512, sorted by
//     (score desc, index asc) with a 512-element warp bitonic network (16 per
//     lane, registers and shuffles), page-transformed and written (one unit
//     per row), or written as a partial list for the merge kernel (split
//     rows).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "sai_internal.h"
#include "sai_ptx.cuh"
#include "sai_select.cuh"

namespace sai {
namespace {

constexpr int kWS = 256;                         // floats per stage (1 KB): two float4 per lane
constexpr int kNS = 6;                           // stages in flight per warp
constexpr int kWCap = 1024;                      // candidate list per warp
constexpr int kMaxExtra = 8;                     // scalar head/tail elements of a window
constexpr int kPruneAt = kWCap - kWS - kMaxExtra;

static_assert(kPruneAt >= kTopK, "room to keep the top 512 and append one stage");
static_assert(kWCap % 32 == 0, "whole warp chunks");

struct SlotInfo {
  int unit;  // -1: no more work
  int row, batch;
  int base, nvec;  // row-local index of stage element 0; TMA elements (multiple of 4)
  int flags;       // 1: first stage of the unit, 2: last stage of the unit
  int lo, len;     // the unit's range of the window: [lo, lo + len)
  int nextra;      // scalar elements (first stage only)
  int pad_;
  long long woff;  // element offset of the row's window start in `scores`
  int extra_idx[kMaxExtra];
  float extra_val[kMaxExtra];
};

struct __align__(128) WarpSmem {
  float stage[kNS][kWS];
  uint32_t ckey[kWCap];
  int32_t cidx[kWCap];
  uint32_t hist[256];
  SlotInfo info[kNS];
  uint64_t full[kNS];
};

constexpr size_t kSmemBytes = sizeof(WarpSmem) + 128;  // + alignment slack

__device__ __forceinline__ WarpSmem& smem_ref(unsigned char* raw) {
  uintptr_t a = reinterpret_cast<uintptr_t>(raw);
  a = (a + 127) & ~static_cast<uintptr_t>(127);
  return *reinterpret_cast<WarpSmem*>(a);
}

// The warp's walk over its work units (warp-uniform registers).
struct Cursor {
  int unit, s, nst;
  int row, batch, lo, head, body, tail;
  long long woff;
};

__device__ void cursor_load(const TopkLaunch& p, Cursor& c) {
  const int units = p.rows * p.chunks;
  c.s = 0;
  if (c.unit >= units) return;
  const int row = c.unit / p.chunks;
  const int ch = c.unit - row * p.chunks;
  int n = p.seq_lens[row];
  const long long start = p.row_starts ? p.row_starts[row] : 0;
  int b = p.row_to_batch ? p.row_to_batch[row] : row;
  bool bad = n < 0 || start < 0 || start + n > p.stride;
  if (p.page_tables)
    bad = bad || b < 0 || b >= p.pt_rows || (n > 0 && (long long)(n - 1) / p.page_size >= p.pt_stride);
  if (bad) {
    if ((threadIdx.x & 31) == 0) atomicOr(p.status, kDevBadRowMeta);
    n = 0;
    b = 0;
  }
  c.row = row;
  c.batch = b;
  c.woff = (long long)row * p.stride + (bad ? 0 : start);
  int lo = p.chunks > 1 ? ch * p.chunk_len : 0;
  const int hi = p.chunks > 1 ? min(n, lo + p.chunk_len) : n;
  if (lo > hi) lo = hi;
  const int len = hi - lo;
  int head = (int)(((16u - (reinterpret_cast<uintptr_t>(p.scores + c.woff + lo) & 15u)) & 15u) >> 2);
  int body = 0;
  if (len <= kMaxExtra || head > len) {
    head = len;
  } else {
    body = (len - head) & ~3;
  }
  c.lo = lo;
  c.head = head;
  c.body = body;
  c.tail = len - head - body;
  c.nst = max(1, (body + kWS - 1) / kWS);
}

// Issue the cursor's next stage into `slot` (whole warp) and advance.
// Returns false once the terminal descriptor has been issued.
__device__ bool issue_stage(const TopkLaunch& p, WarpSmem& S, Cursor& c, int slot, uint64_t policy, int lane) {
  const int units = p.rows * p.chunks;
  SlotInfo& d = S.info[slot];
  if (c.unit >= units) {
    __syncwarp();
    if (lane == 0) {
      d.unit = -1;
      mbar_arrive(&S.full[slot]);
    }
    return false;
  }
  const int base = c.lo + c.head + c.s * kWS;
  const int nvec = min(kWS, c.body - c.s * kWS);
  const int nextra = c.s == 0 ? c.head + c.tail : 0;
  if (lane < nextra) {
    const int j = lane < c.head ? c.lo + lane : c.lo + c.head + c.body + (lane - c.head);
    d.extra_idx[lane] = j;
    d.extra_val[lane] = __ldg(p.scores + c.woff + j);
  }
  if (lane == 0) {
    d.unit = c.unit;
    d.row = c.row;
    d.batch = c.batch;
    d.base = base;
    d.nvec = nvec;
    d.flags = (c.s == 0 ? 1 : 0) | (c.s == c.nst - 1 ? 2 : 0);
    d.lo = c.lo;
    d.len = c.head + c.body + c.tail;
    d.nextra = nextra;
    d.woff = c.woff;
  }
  __syncwarp();
  if (lane == 0) {
    if (nvec > 0) {
      mbar_arrive_expect_tx(&S.full[slot], (uint32_t)nvec * 4u);
      bulk_g2s_stream(S.stage[slot], p.scores + c.woff + base, (uint32_t)nvec * 4u, &S.full[slot], policy);
    } else {
      mbar_arrive(&S.full[slot]);
    }
  }
  if (++c.s >= c.nst) {
    c.unit += gridDim.x;
    cursor_load(p, c);
  }
  return true;
}

// ---------------------------------------------------------------- warp select
// Threshold bin of the `need` largest values among the active entries j in
// [0, n) (active/value from `get(j, v)`), by 8-bit radix digits over the
// value range, for one warp. `need` must not exceed the active count.
template <typename Get>
__device__ Threshold warp_threshold(int n, uint32_t need, uint32_t* hist, int lane, Get get) {
  uint32_t lmin = 0xFFFFFFFFu, lmax = 0u, lcnt = 0u;
  for (int j = lane; j < n; j += 32) {
    uint32_t v;
    if (get(j, v)) {
      lmin = min(lmin, v);
      lmax = max(lmax, v);
      ++lcnt;
    }
  }
  Threshold t;
  t.base = __reduce_min_sync(0xFFFFFFFFu, lmin);
  const uint32_t span = __reduce_max_sync(0xFFFFFFFFu, lmax) - t.base;
  const uint32_t nact = __reduce_add_sync(0xFFFFFFFFu, lcnt);
  t.lo = span ? 32 - __clz(span) : 0;
  t.prefix = 0;
  t.need = need;
  t.all_eq = (nact == need);
  while (t.lo > 0 && !t.all_eq) {
    const int dlo = t.lo > 8 ? t.lo - 8 : 0;
    const int dbits = t.lo - dlo;
    const uint32_t dmask = (1u << dbits) - 1u;
    reinterpret_cast<uint4*>(hist)[2 * lane] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(hist)[2 * lane + 1] = make_uint4(0, 0, 0, 0);
    __syncwarp();
    for (int j = lane; j < n; j += 32) {
      uint32_t v;
      if (get(j, v)) {
        const uint32_t o = v - t.base;
        if (shr64(o, t.lo) == t.prefix) atomicAdd(&hist[(o >> dlo) & dmask], 1u);
      }
    }
    __syncwarp();
    const uint4 a = reinterpret_cast<const uint4*>(hist)[2 * lane];
    const uint4 b = reinterpret_cast<const uint4*>(hist)[2 * lane + 1];
    const uint32_t h[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t tot = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) tot += h[i];
    uint32_t suf = tot;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_down_sync(0xFFFFFFFFu, suf, d);
      if (lane + d < 32) suf += o;
    }
    uint32_t above = suf - tot;
    const uint32_t nd = t.need;
    uint32_t bin = 0, need_after = 0, bcount = 0;
    const bool mine = above < nd && nd <= suf;
    if (mine) {
#pragma unroll
      for (int i = 7; i >= 0; --i) {
        if (above < nd && nd <= above + h[i]) {
          bin = lane * 8 + i;
          need_after = nd - above;
          bcount = h[i];
        }
        above += h[i];
      }
    }
    const int src = __ffs(__ballot_sync(0xFFFFFFFFu, mine)) - 1;
    bin = __shfl_sync(0xFFFFFFFFu, bin, src);
    need_after = __shfl_sync(0xFFFFFFFFu, need_after, src);
    bcount = __shfl_sync(0xFFFFFFFFu, bcount, src);
    t.prefix = (t.prefix << dbits) | bin;
    t.need = need_after;
    t.all_eq = (bcount == t.need);
    t.lo = dlo;
    __syncwarp();
  }
  return t;
}

// Cut the warp's list ckey/cidx[0, n), n > 512, to its top 512 by (key
// desc, index asc), compacted in place to [0, 512). Returns the lowest key
// of the final threshold bin (<= the 512th key): "key >= returned value" is
// a valid filter for later elements.
__device__ uint32_t warp_select512(WarpSmem& S, int n, int lane) {
  uint32_t* const ckey = S.ckey;
  int32_t* const cidx = S.cidx;
  const Threshold t = warp_threshold(n, (uint32_t)kTopK, S.hist, lane, [&](int j, uint32_t& v) {
    v = ckey[j];
    return true;
  });
  Threshold ti{};
  const bool ties = !t.all_eq;
  if (ties) {
    ti = warp_threshold(n, t.need, S.hist, lane, [&](int j, uint32_t& v) {
      v = 0x7FFFFFFFu - static_cast<uint32_t>(cidx[j]);
      return thr_cmp(t, ckey[j]) == 0;
    });
  }
  // In-place compaction: chunk c is read before any of its selected entries
  // is written, and a write position never exceeds its read position.
  int out = 0;
  const uint32_t lt = (1u << lane) - 1u;
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    bool sel = false;
    uint32_t key = 0;
    int32_t idx = 0;
    if (j < n) {
      key = ckey[j];
      idx = cidx[j];
      const int cc = thr_cmp(t, key);
      sel = cc > 0 || (cc == 0 && (!ties || thr_cmp(ti, 0x7FFFFFFFu - static_cast<uint32_t>(idx)) >= 0));
    }
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, sel);
    __syncwarp();
    if (sel) {
      const int pos = out + __popc(bal & lt);
      if (pos < kTopK) {
        ckey[pos] = key;
        cidx[pos] = idx;
      }
    }
    out += __popc(bal);
    __syncwarp();
  }
  return t.base + static_cast<uint32_t>(static_cast<uint64_t>(t.prefix) << t.lo);
}

// Sort the warp's list ckey/cidx[0, cnt), cnt <= 512, by (key desc, index
// asc): bitonic network over the virtual index vi = 16*lane + s, so that on
// return v[s] holds the entry of output rank 16*lane + s (0 = padding).
__device__ __forceinline__ void warp_sort512(const WarpSmem& S, int cnt, unsigned long long (&v)[16], int lane) {
#pragma unroll
  for (int s = 0; s < 16; ++s) {
    const int e = 32 * s + lane;  // any placement works: everything gets sorted
    v[s] = e < cnt ? composite(S.ckey[e], S.cidx[e]) : 0ull;
  }
#pragma unroll
  for (int size = 2; size <= 512; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride < 16) {
#pragma unroll
        for (int s = 0; s < 16; ++s) {
          if (s & stride) continue;
          const int s2 = s | stride;
          const bool asc = ((16 * lane + s) & size) != 0;
          const unsigned long long x = v[s], y = v[s2];
          const unsigned long long hi = x > y ? x : y, lo = x > y ? y : x;
          v[s] = asc ? lo : hi;
          v[s2] = asc ? hi : lo;
        }
      } else {
        const int d = stride >> 4;
        const bool lower = (lane & d) == 0;
        const bool asc = (lane & (size >> 4)) != 0;
#pragma unroll
        for (int s = 0; s < 16; ++s) {
          const unsigned long long p = __shfl_xor_sync(0xFFFFFFFFu, v[s], d);
          v[s] = (lower != asc) ? (v[s] > p ? v[s] : p) : (v[s] < p ? v[s] : p);
        }
      }
    }
  }
}

__device__ __forceinline__ uint32_t pass4(const float4& v, float tf) {
  return (v.x >= tf ? 1u : 0u) | (v.y >= tf ? 2u : 0u) | (v.z >= tf ? 4u : 0u) | (v.w >= tf ? 8u : 0u);
}

// Append the elements whose bit is set in `mask` to the warp's list: lane
// holds a = elements base+4*lane+0..3, b = elements base+128+4*lane+0..3 and
// one scalar element x at index xi. One ballot per element slot.
__device__ __forceinline__ int warp_append(WarpSmem& S, const float4& a, const float4& b, float x, int xi, int base,
                                           uint32_t mask, int wcnt, int lane) {
  if (!__any_sync(0xFFFFFFFFu, mask != 0)) return wcnt;
  const uint32_t lt = (1u << lane) - 1u;
  int pos = wcnt;
  const int i0 = base + 4 * lane, i1 = base + 128 + 4 * lane;
#define SAI_PUT(I, V, IDX)                                  \
  {                                                         \
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, (mask >> (I)) & 1u); \
    if (bal) {                                              \
      if ((mask >> (I)) & 1u) {                             \
        const int q = pos + __popc(bal & lt);               \
        S.ckey[q] = order_key(V);                           \
        S.cidx[q] = (IDX);                                  \
      }                                                     \
      pos += __popc(bal);                                   \
    }                                                       \
  }
  SAI_PUT(0, a.x, i0 + 0)
  SAI_PUT(1, a.y, i0 + 1)
  SAI_PUT(2, a.z, i0 + 2)
  SAI_PUT(3, a.w, i0 + 3)
  SAI_PUT(4, b.x, i1 + 0)
  SAI_PUT(5, b.y, i1 + 1)
  SAI_PUT(6, b.z, i1 + 2)
  SAI_PUT(7, b.w, i1 + 3)
  SAI_PUT(8, x, xi)
#undef SAI_PUT
  __syncwarp();
  return pos;
}

// ---------------------------------------------------------------- kernel
__global__ void __launch_bounds__(32) topk_stream_kernel(const __grid_constant__ TopkLaunch p) {
  extern __shared__ unsigned char smem_raw[];
  WarpSmem& S = smem_ref(smem_raw);
  const int lane = threadIdx.x;
  if (lane == 0) {
    for (int i = 0; i < kNS; ++i) mbar_init(&S.full[i], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t policy = l2_policy_evict_first();
  Cursor cur{};
  cur.unit = blockIdx.x;
  cursor_load(p, cur);
  bool issuing = true;
  for (int i = 0; i < kNS && issuing; ++i) issuing = issue_stage(p, S, cur, i, policy, lane);

  uint32_t it = 0;
  int wcnt = 0;        // entries in the candidate list
  int wapp = 0;        // elements that passed the filter in this unit
  uint32_t tau = 0;    // keep elements whose order key >= tau
  uint32_t spec = 0;   // starting threshold for the next unit (0: none)
  uint32_t spec_used = 0;
  while (true) {
    const int slot = it % kNS;
    const uint32_t ph = (it / kNS) & 1u;
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&S.full[slot], ph))) {
      if (lane == 0) {
        atomicOr(p.status, kDevWaitTimeout);
        // let copies already issued land before the CTA exits (bounded)
        for (int k = 1; k < kNS; ++k) mbar_wait(&S.full[(it + k) % kNS], ((it + k) / kNS) & 1u);
      }
      break;
    }
    const SlotInfo& d = S.info[slot];
    const int unit = d.unit;
    if (unit < 0) break;
    const int flags = d.flags, nvec = d.nvec, base = d.base, row = d.row, batch = d.batch;
    const int lo = d.lo, len = d.len, nextra = d.nextra;
    const long long woff = d.woff;
    if (flags & 1) {
      wcnt = 0;
      wapp = 0;
      tau = spec;
      spec_used = spec;
    }
    const float tf = tau_float(tau);
    float4 va = make_float4(0.f, 0.f, 0.f, 0.f), vb = va;
    float vx = 0.f;
    int xi = 0;
    uint32_t mask = 0;
    if (4 * lane < nvec) {
      va = reinterpret_cast<const float4*>(S.stage[slot])[lane];
      mask = pass4(va, tf);
    }
    if (4 * (lane + 32) < nvec) {
      vb = reinterpret_cast<const float4*>(S.stage[slot])[lane + 32];
      mask |= pass4(vb, tf) << 4;
    }
    if (lane < nextra) {
      xi = d.extra_idx[lane];
      vx = d.extra_val[lane];
      mask |= (vx >= tf ? 1u : 0u) << 8;
    }
    __syncwarp();
    if (issuing) {  // the slot's data is in registers: refill it
      if (lane == 0) fence_proxy_async_smem();
      issuing = issue_stage(p, S, cur, slot, policy, lane);
    }
    const int nw = warp_append(S, va, vb, vx, xi, base, mask, wcnt, lane);
    wapp += nw - wcnt;
    wcnt = nw;
    if (wcnt > kPruneAt) {
      tau = max(tau, warp_select512(S, wcnt, lane));
      wcnt = kTopK;
    }
    if (flags & 2) {
      if (spec_used && wapp < min(len, kTopK)) {
        // The starting threshold was too high for this unit: redo it from
        // global memory with no threshold (exact again, just slower).
        wcnt = 0;
        wapp = 0;
        tau = 0;
        for (int b0 = 0; b0 < len; b0 += kWS) {
          const float tf0 = tau_float(tau);
          const float* src = p.scores + woff + lo + b0;
          float r[8];
          uint32_t rm = 0;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int j = k < 4 ? 4 * lane + k : 128 + 4 * lane + (k - 4);
            r[k] = 0.f;
            if (b0 + j < len) {
              r[k] = __ldg(src + j);
              rm |= (r[k] >= tf0 ? 1u : 0u) << k;
            }
          }
          const int nw2 = warp_append(S, make_float4(r[0], r[1], r[2], r[3]), make_float4(r[4], r[5], r[6], r[7]),
                                      0.f, 0, lo + b0, rm, wcnt, lane);
          wapp += nw2 - wcnt;
          wcnt = nw2;
          if (wcnt > kPruneAt) {
            tau = max(tau, warp_select512(S, wcnt, lane));
            wcnt = kTopK;
          }
        }
        spec_used = 0;
      }
      if (wcnt > kTopK) {
        warp_select512(S, wcnt, lane);
        wcnt = kTopK;
      }
      unsigned long long v[16];
      warp_sort512(S, wcnt, v, lane);
      __syncwarp();
      if (p.chunks == 1) {
        const long long o = (long long)row * kTopK + 16 * lane;
        int oi[16], os[16];
#pragma unroll
        for (int s = 0; s < 16; ++s) {
          const bool real = 16 * lane + s < wcnt;
          const int idx = real ? static_cast<int>(~static_cast<uint32_t>(v[s] & 0xFFFFFFFFull)) : -1;
          oi[s] = idx;
          os[s] = -1;
          if (real && p.page_tables) {
            const int ps = p.page_size;
            const long long page = p.page_tables[(long long)batch * p.pt_stride + (ps == 1 ? idx : idx / ps)];
            os[s] = static_cast<int>(ps == 1 ? page : page * ps + idx % ps);
          }
        }
        const bool vec = ((reinterpret_cast<uintptr_t>(p.out_idx) | reinterpret_cast<uintptr_t>(p.out_slots)) & 15u) == 0;
        if (p.out_idx) {
          if (vec) {
            int4* dst = reinterpret_cast<int4*>(p.out_idx + o);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_int4(oi[4 * q], oi[4 * q + 1], oi[4 * q + 2], oi[4 * q + 3]);
          } else {
#pragma unroll
            for (int s = 0; s < 16; ++s) p.out_idx[o + s] = oi[s];
          }
        }
        if (p.out_slots) {
          if (vec) {
            int4* dst = reinterpret_cast<int4*>(p.out_slots + o);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_int4(os[4 * q], os[4 * q + 1], os[4 * q + 2], os[4 * q + 3]);
          } else {
#pragma unroll
            for (int s = 0; s < 16; ++s) p.out_slots[o + s] = os[s];
          }
        }
      } else {
        const long long o = (long long)unit * kTopK + 16 * lane;
#pragma unroll
        for (int s = 0; s < 16; ++s) {
          if (16 * lane + s < wcnt) {
            p.part_key[o + s] = static_cast<uint32_t>(v[s] >> 32);
            p.part_idx[o + s] = static_cast<int32_t>(~static_cast<uint32_t>(v[s] & 0xFFFFFFFFull));
          }
        }
        if (lane == 0) p.part_cnt[unit] = wcnt;
      }
      // Next unit's starting threshold: extrapolate the tail one octave of
      // rank down, t = 2*v(512) - v(256), which keeps about twice the
      // needed count when neighbouring rows look alike.
      spec = 0;
      const uint32_t k256 = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v[15] >> 32), 15);
      const uint32_t k512 = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v[15] >> 32), 31);
      if (wcnt >= kTopK && k512 != 0) {
        const float t = 2.0f * key_to_float(k512) - key_to_float(k256);
        if (isfinite(t) && isfinite(key_to_float(k256)) && isfinite(key_to_float(k512))) spec = order_key(t);
      }
      wcnt = 0;
    }
    ++it;
  }
}

// ---------------------------------------------------------------- merge
constexpr int kMergeUnits = 12;
constexpr int kMergeCap = kMergeUnits * kTopK;

struct __align__(16) MergeSmem {
  union {
    struct {
      uint32_t key[kMergeCap];
      int32_t idx[kMergeCap];
    } c;
    struct {
      uint32_t key[kTopK];
      int32_t idx[kTopK];
    } runs;
  } cand;
  uint32_t hist[4096];
  uint32_t aux_key[kTopK];
  int32_t aux_idx[kTopK];
  SelectScratch sc;
  uint32_t bcast[4];
};

__global__ void __launch_bounds__(kTopK, 1) merge_kernel(const __grid_constant__ MergeLaunch p) {
  extern __shared__ unsigned char smem_raw[];
  MergeSmem& S = *reinterpret_cast<MergeSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const long long row = blockIdx.x;
  reinterpret_cast<uint4*>(S.hist)[2 * tid] = make_uint4(0, 0, 0, 0);
  reinterpret_cast<uint4*>(S.hist)[2 * tid + 1] = make_uint4(0, 0, 0, 0);
  int total = 0;
  for (int c = 0; c < p.units_per_row; ++c) {
    const long long unit = row * p.units_per_row + c;
    const int n = min(p.part_cnt[unit], kTopK);
    if (tid < n) {
      S.cand.c.key[total + tid] = p.part_key[unit * kTopK + tid];
      S.cand.c.idx[total + tid] = p.part_idx[unit * kTopK + tid];
    }
    total += n;
  }
  __syncthreads();
  int cnt = total;
  if (cnt > kTopK) {
    fast_select512<kMergeCap>(S.cand.c.key, S.cand.c.idx, cnt, S.hist, S.aux_key, S.aux_idx, S.sc, S.bcast, tid, 1);
    cnt = kTopK;
  } else {
    if (tid < cnt) {
      S.aux_key[tid] = S.cand.c.key[tid];
      S.aux_idx[tid] = S.cand.c.idx[tid];
    }
    __syncthreads();
  }
  uint32_t k[1];
  int32_t ix[1];
  int rk[1];
  rank_sort<kTopK>(S.aux_key, S.aux_idx, cnt, S.cand.runs.key, S.cand.runs.idx, k, ix, rk, tid, 1);
  const long long o = row * kTopK;
  if (ix[0] >= 0) {
    if (p.out_idx) p.out_idx[o + rk[0]] = ix[0];
    if (p.out_scores) p.out_scores[o + rk[0]] = key_to_float(k[0]);
    if (p.out_slots) {
      const int batch = p.row_to_batch ? p.row_to_batch[row] : (int)row;
      const int ps = p.page_size;
      const long long page = p.page_tables[(long long)batch * p.pt_stride + (ps == 1 ? ix[0] : ix[0] / ps)];
      p.out_slots[o + rk[0]] = static_cast<int>(ps == 1 ? page : page * ps + ix[0] % ps);
    }
  }
  if (tid >= cnt) {
    if (p.out_idx) p.out_idx[o + tid] = -1;
    if (p.out_slots) p.out_slots[o + tid] = -1;
    if (p.out_scores) p.out_scores[o + tid] = __int_as_float(0x7FC00000);
  }
}

bool g_attr_done[64];
bool g_merge_attr_done[64];

}  // namespace

TopkPlan topk_plan(long long rows, long long max_window, int num_sms) {
  TopkPlan pl{1, 0, 0};
  if (rows <= 0 || max_window <= 0) return pl;
  const long long slots = 2LL * num_sms;
  constexpr long long kMinChunk = 4096;
  if (rows < slots && max_window > 2 * kMinChunk) {
    long long chunks = (max_window + kMinChunk - 1) / kMinChunk;
    chunks = std::min<long long>(chunks, kMergeUnits);
    long long len = (max_window + chunks - 1) / chunks;
    len = (len + 15) / 16 * 16;
    chunks = (max_window + len - 1) / len;
    pl.chunks = static_cast<int>(chunks);
    pl.chunk_len = static_cast<int>(len);
    const long long units = rows * chunks;
    pl.workspace_bytes = static_cast<size_t>(units) * kTopK * 8 + static_cast<size_t>(units) * 4 + 256;
  }
  return pl;
}

size_t merge_smem_bytes() { return sizeof(MergeSmem); }

cudaError_t launch_merge(const MergeLaunch& p, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !g_merge_attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(MergeSmem));
    if (e != cudaSuccess) return e;
    g_merge_attr_done[dev] = true;
  }
  merge_kernel<<<p.rows, kTopK, sizeof(MergeSmem), stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_topk_transform(const TopkLaunch& p, int num_sms, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !g_attr_done[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(topk_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    g_attr_done[dev] = true;
  }
  static int ctas_per_sm[64];
  if (dev < 64 && ctas_per_sm[dev] == 0) {
    int nb = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, topk_stream_kernel, 32, kSmemBytes);
    if (e != cudaSuccess) return e;
    ctas_per_sm[dev] = nb > 0 ? nb : 1;
  }
  const long long units = (long long)p.rows * p.chunks;
  const int grid = (int)std::min<long long>(units, (long long)(dev < 64 ? ctas_per_sm[dev] : 1) * num_sms);
  topk_stream_kernel<<<grid, 32, kSmemBytes, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.chunks == 1) return e;
  MergeLaunch m{};
  m.rows = p.rows;
  m.units_per_row = p.chunks;
  m.part_key = p.part_key;
  m.part_idx = p.part_idx;
  m.part_cnt = p.part_cnt;
  m.seq_lens = p.seq_lens;
  m.page_tables = p.page_tables;
  m.pt_rows = p.pt_rows;
  m.pt_stride = p.pt_stride;
  m.row_to_batch = p.row_to_batch;
  m.page_size = p.page_size;
  m.out_slots = p.out_slots;
  m.out_idx = p.out_idx;
  m.out_scores = nullptr;
  m.status = p.status;
  return launch_merge(m, stream);
}

}  // namespace sai
