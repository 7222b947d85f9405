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
// GB300 design: many small persistent CTAs (4 warps, ~43 KB of shared
// memory, five per SM), each streaming one work unit (a row, or a chunk of a
// long row) at a time, so that the serial latency of one CTA's
// stage -> filter -> barrier chain is hidden by the other CTAs on the SM.
// The kernel is bound by instruction issue, not by HBM, so each stage is
// large (12 KB, 24 scores per thread, two stages per CTA) to spread the
// per-stage cost (measured against 16 and 32 scores per thread, two and
// three stages, three to six CTAs per SM).
//   * Thread 0 keeps a ring of shared-memory stages filled with 1-D bulk TMA
//     copies (cp.async.bulk + mbarrier complete_tx, evict-first in L2: every
//     score is read once). The 16-byte-aligned interior of each window goes
//     through TMA; its <= 3 leading and <= 3 trailing elements (any row
//     stride, any row start) are read with scalar loads. This is the scalar
//     path the pages require for strides that are not a multiple of 4,
//     folded into every row instead of a separate fallback kernel.
//   * Each thread compares its 24 scores of a stage against the running
//     threshold tau (as a float) and appends the survivors (order key,
//     row-local index) to its warp's own candidate sub-list: a ballot prefix
//     inside the warp, no shared atomics. The one block barrier per stage
//     (it releases the stage for refill) also ORs "some warp's survivors do
//     not fit"; then all sub-lists are cut together to the exact top 512
//     (radix select in shared memory), dealt back 128 per warp, tau rises to
//     that cut and the stage is appended a quarter at a time. The filter
//     stays exact: every dropped element is beaten by 512 kept ones.
//   * At the end of a unit the candidates are cut to 512, sorted by
//     (score desc, index asc), page-transformed and written (one unit per
//     row), or written as a partial list for the merge kernel (split rows).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "sai_blocks.cuh"
#include "sai_internal.h"
#include "sai_ptx.cuh"
#include "sai_select.cuh"

namespace sai {
namespace {

constexpr int kThreads = 128;                    // 4 warps per CTA
#ifndef SAI_TOPK_VEC
#define SAI_TOPK_VEC 6
#endif
#ifndef SAI_TOPK_MIN_CHUNK
// Shortest window piece of a split row: rows of up to twice this stay on one
// CTA (measured on 128 decode rows of 8K-32K scores: 0.048 ms unsplit, 0.069
// in pieces of 8192 and 0.096 in pieces of 4096, the merge of the pieces'
// lists taking ~20 us).
#define SAI_TOPK_MIN_CHUNK 16384
#endif
#ifndef SAI_TOPK_CTAS
#define SAI_TOPK_CTAS 5
#endif
constexpr int kVec = SAI_TOPK_VEC;               // float4 loads per thread per stage
constexpr int kStage = kVec * 4 * kThreads;      // floats per stage (12 KB)
#ifndef SAI_TOPK_NSTAGE
#define SAI_TOPK_NSTAGE 2
#endif
constexpr int kNStage = SAI_TOPK_NSTAGE;         // 24 KB in flight per CTA
#ifndef SAI_TOPK_DEEP_STAGES
#define SAI_TOPK_DEEP_STAGES 16
#endif
constexpr int kDeepStages = SAI_TOPK_DEEP_STAGES;  // ring of a call whose units all fit on the SMs at once
constexpr int kWarps = kThreads / 32;
constexpr int kCap = 1536;                       // candidate capacity (all warps)
constexpr int kSub = kCap / kWarps;              // one candidate sub-list per warp
constexpr int kMaxExtra = 8;                     // scalar head/tail elements of a window
constexpr int kPartWarp = 4 * 32 + kMaxExtra;    // most entries a warp appends from one float4 per lane
constexpr int kSubCutAt = kSub - kPartWarp;      // slow path: cut before a part that might not fit
constexpr int kBar = 1;                          // named barrier id (all 128 threads)
constexpr int kCtasPerSm = SAI_TOPK_CTAS;
static_assert(4 * kVec <= 32, "one mask bit per score of a thread's stage");

static_assert(kSubCutAt >= kTopK / kWarps, "a dealt-back sub-list must take one more part");

// What a unit's first and last stage need besides the stage itself.
struct UnitInfo {
  int row;
  int batch;         // page-table row
  int head, tail;    // scalar elements: [lo, lo+head) and [tail_at, tail_at+tail)
  int lo, tail_at;
  int len;           // elements of the unit's window range [lo, lo+len)
  int pad;
  long long woff;    // element offset of the row's window start in `scores`
};

// Per-slot descriptor written by the issuing thread: `hot` = {unit (-1: no
// more work), row-local index of the stage's element 0, TMA elements in the
// stage (a multiple of 4), flags (1: first stage of the unit, 2: last)} is
// read every stage; `u` is written and read only when flags != 0.
struct StageDesc {
  int4 hot;
  UnitInfo u;
};

// Thread 0's walk over its work units (the issue side of the ring).
struct Cursor {
  int unit;          // current unit (>= units: done)
  int s, nst;        // stage index within the unit, stage count
  int base;          // row-local index of the next stage's element 0
  int body_left;     // TMA elements not issued yet
  const float* src;  // global address of the next stage
  UnitInfo u;
};

template <int NS>
struct __align__(128) SmemT {
  float stage[NS][kStage];
  union {
    struct {
      uint32_t key[kCap];
      int32_t idx[kCap];
    } c;
    unsigned long long sortbuf[kTopK];  // final sort (the list is dead by then)
    struct {
      uint32_t hist[1024];
      uint16_t bucket[kTopK];
    } rank;                             // final ranking (likewise)
    BlockScratch blocks;                // block lists of the output (likewise)
  } cand;
  uint32_t aux_key[kTopK];
  int32_t aux_idx[kTopK];
  StageDesc desc[NS];
  uint64_t full[NS];
  SelectScratch sc;
  uint32_t spec_keys[2];  // keys at ranks 256 and 512 of the last finished unit
  int wcnt[kWarps];       // sub-list sizes, published before a cut
  int wapp[kWarps];       // per-warp appends of the unit, published at its end
  int timeout;            // set by a thread whose stage wait gave up
  Cursor cur;
};

template <int NS>
constexpr size_t smem_bytes() {
  return sizeof(SmemT<NS>) + 128;  // + alignment slack
}

template <int NS>
__device__ __forceinline__ SmemT<NS>& smem_ref(unsigned char* raw) {
  uintptr_t a = reinterpret_cast<uintptr_t>(raw);
  a = (a + 127) & ~static_cast<uintptr_t>(127);
  return *reinterpret_cast<SmemT<NS>*>(a);
}

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
    atomicOr(p.status, kDevBadRowMeta);
    n = 0;
    b = 0;
  }
  const long long woff = (long long)row * p.stride + (bad ? 0 : start);
  int lo = p.chunks > 1 ? ch * p.chunk_len : 0;
  const int hi = p.chunks > 1 ? min(n, lo + p.chunk_len) : n;
  if (lo > hi) lo = hi;
  const int len = hi - lo;
  int head = (int)(((16u - (reinterpret_cast<uintptr_t>(p.scores + woff + lo) & 15u)) & 15u) >> 2);
  int body = 0;
  if (len <= kMaxExtra || head > len) {
    head = len;
  } else {
    body = (len - head) & ~3;
  }
  c.u.row = row;
  c.u.batch = b;
  c.u.head = head;
  c.u.tail = len - head - body;
  c.u.lo = lo;
  c.u.tail_at = lo + head + body;
  c.u.len = len;
  c.u.woff = woff;
  c.nst = max(1, (body + kStage - 1) / kStage);
  c.base = lo + head;
  c.body_left = body;
  c.src = p.scores + woff + lo + head;
}

// Issue the cursor's next stage into `slot` (thread 0 only) and advance.
// Returns false once the terminal descriptor has been issued.
template <int NS>
__device__ bool issue_stage(const TopkLaunch& p, SmemT<NS>& S, int slot, uint64_t policy) {
  Cursor& c = S.cur;
  StageDesc& d = S.desc[slot];
  if (c.unit >= p.rows * p.chunks) {
    d.hot = make_int4(-1, 0, 0, 0);
    mbar_arrive(&S.full[slot]);
    return false;
  }
  const int s = c.s, nst = c.nst;
  const int flags = (s == 0 ? 1 : 0) | (s == nst - 1 ? 2 : 0);
  const int nvec = min(kStage, c.body_left);
  d.hot = make_int4(c.unit, c.base, nvec, flags);
  if (flags) d.u = c.u;
  if (nvec > 0) {
    mbar_arrive_expect_tx(&S.full[slot], (uint32_t)nvec * 4u);
    bulk_g2s_stream(S.stage[slot], c.src, (uint32_t)nvec * 4u, &S.full[slot], policy);
  } else {
    mbar_arrive(&S.full[slot]);
  }
  if (s + 1 >= nst) {
    // Units after each CTA's first come from a shared counter when there is
    // one, so that CTAs that drew short rows (or no redo) take more of them.
    c.unit = p.work ? static_cast<int>(gridDim.x) + atomicAdd(p.work, 1) : c.unit + static_cast<int>(gridDim.x);
    cursor_load(p, c);
  } else {
    c.s = s + 1;
    c.base += kStage;
    c.body_left -= nvec;
    c.src += kStage;
  }
  return true;
}

// Offsets of this lane's survivors in its warp's sub-list: bit i of `mask`
// marks a surviving score of the lane's stage data, `xs` a surviving scalar
// end element (at most 4*kVec + 1 per lane). Survivors are rare (about 1%
// of a row), so the common case is one survivor on a few lanes and one
// ballot gives every lane its offset; only when some lane has several does
// the warp ballot the bits of the per-lane counts. Returns the warp total
// (warp-uniform) and this lane's first offset in *pos.
__device__ __forceinline__ int warp_offsets(uint32_t mask, bool xs, int lane, int* pos) {
  const uint32_t m = __popc(mask) + (xs ? 1u : 0u);
  const uint32_t any = __ballot_sync(0xFFFFFFFFu, m != 0);
  const uint32_t lt = (1u << lane) - 1u;
  *pos = 0;
  if (any == 0) return 0;
  const uint32_t multi = __ballot_sync(0xFFFFFFFFu, m > 1);
  if (multi == 0) {
    *pos = __popc(any & lt);
    return __popc(any);
  }
  int off = 0, total = 0;
#pragma unroll
  for (int k = 0; k < 6; ++k) {
    const uint32_t bk = __ballot_sync(0xFFFFFFFFu, (m >> k) & 1u);
    off += __popc(bk & lt) << k;
    total += __popc(bk) << k;
  }
  *pos = off;
  return total;
}

// Write this lane's survivors (order key, row-local index) from position
// pos of its warp's sub-list on. a[q] holds elements base + 4*(q*kThreads +
// tid) + 0..3 (mask bits 4q..4q+3); x is one scalar element at index xi
// (kept when xs). Each lane walks only its set bits.
__device__ __forceinline__ void write_survivors(uint32_t* key, int32_t* idx, int pos, const float4 (&a)[kVec],
                                                float x, int xi, int base, uint32_t mask, bool xs, int tid) {
#pragma unroll
  for (int q = 0; q < kVec; ++q) {
    uint32_t m = (mask >> (4 * q)) & 0xFu;
    while (m) {
      const int r = __ffs(m) - 1;
      m &= m - 1u;
      const float v = r == 0 ? a[q].x : (r == 1 ? a[q].y : (r == 2 ? a[q].z : a[q].w));
      key[pos] = order_key(v);
      idx[pos] = base + 4 * (q * kThreads + tid) + r;
      ++pos;
    }
  }
  if (xs) {
    key[pos] = order_key(x);
    idx[pos] = xi;
  }
}

// write_survivors for a stage still held in shared memory: the value of
// mask bit i (a score of this thread's float4 i/4) is re-read from the stage
// buffer, so a lane's loop is one load and two stores per survivor whichever
// float4 it sits in.
__device__ __forceinline__ void write_survivors_smem(uint32_t* key, int32_t* idx, int pos, const float* stage,
                                                     float x, int xi, int base, uint32_t mask, bool xs, int tid) {
  uint32_t m = mask;
  while (m) {
    const int i = __ffs(m) - 1;
    m &= m - 1u;
    const int off = ((i >> 2) * kThreads + tid) * 4 + (i & 3);
    key[pos] = order_key(stage[off]);
    idx[pos] = base + off;
    ++pos;
  }
  if (xs) {
    key[pos] = order_key(x);
    idx[pos] = xi;
  }
}

// Starting threshold for a unit that has no estimate carried from the CTA's
// previous unit (a CTA's first unit): the m-th largest of 1024 scores
// sampled evenly over the window, m = twice the expected number of samples
// above the window's 512th score plus 8, so that it lies below the 512th
// score except with negligible probability (the unit end checks this
// exactly and redoes the unit otherwise); about 1024 + len/128 scores then
// pass. 0 (no threshold) for windows under 4096. Out of line: it runs once
// per CTA or so, and stays out of the stream loop's registers.
template <int NS>
__device__ __noinline__ uint32_t sample_tau(const float* win, int len, SmemT<NS>& S, int tid) {
  constexpr int kSamples = 1024, kPer = kSamples / kThreads;
  if (len < 4096) return 0u;
  const uint32_t expect = static_cast<uint32_t>(((long long)kSamples * kTopK + len - 1) / len);
  const uint32_t m = 2u * expect + 8u;
  if (m >= static_cast<uint32_t>(kSamples)) return 0u;
  uint32_t v[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const long long j = tid + kThreads * e;
    v[e] = order_key(__ldg(win + ((2 * j + 1) * len) / (2 * kSamples)));
  }
  const Threshold t = radix_threshold_each<kThreads>(m, S.sc, tid, kBar, [&](auto fn) {
#pragma unroll
    for (int e = 0; e < kPer; ++e) fn(v[e]);
  });
  return t.base + static_cast<uint32_t>(static_cast<uint64_t>(t.prefix) << t.lo);
}

// Gather every warp's sub-list into aux: the exact top 512 of their union
// when it holds more (tau rises to the cut), else all of it. All threads
// call this with their warp's wcnt; returns the number in aux.
template <int NS>
__device__ int gather_to_aux(SmemT<NS>& S, int wcnt, uint32_t& tau, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  if (lane == 0) S.wcnt[warp] = wcnt;
  named_bar(kBar, kThreads);
  int counts[kWarps];
  int total = 0, off = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    counts[w] = S.wcnt[w];
    off += w < warp ? counts[w] : 0;
    total += counts[w];
  }
  if (total > kTopK) {
    tau = max(tau, select512_sub_to_aux<kThreads, kWarps, kSub>(S.cand.c.key, S.cand.c.idx, counts, S.aux_key,
                                                                S.aux_idx, S.sc, tid, kBar));
    return kTopK;
  }
  const uint32_t* key = S.cand.c.key + warp * kSub;
  const int32_t* idx = S.cand.c.idx + warp * kSub;
  for (int j = lane; j < wcnt; j += 32) {
    S.aux_key[off + j] = key[j];
    S.aux_idx[off + j] = idx[j];
  }
  named_bar(kBar, kThreads);
  return total;
}

// Cut all sub-lists together (gather_to_aux) and deal the kept entries back,
// 128 per warp. Returns the warp's new sub-list size.
template <int NS>
__device__ __forceinline__ int prune(SmemT<NS>& S, int wcnt, uint32_t& tau, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  const int total = gather_to_aux(S, wcnt, tau, tid);
  constexpr int kShare = kTopK / kWarps;
  const int mine = min(max(total - kShare * warp, 0), kShare);
  uint32_t* key = S.cand.c.key + warp * kSub;
  int32_t* idx = S.cand.c.idx + warp * kSub;
  for (int j = lane; j < mine; j += 32) {
    key[j] = S.aux_key[kShare * warp + j];
    idx[j] = S.aux_idx[kShare * warp + j];
  }
  __syncwarp();
  return mine;
}

__device__ __forceinline__ uint32_t pass4(const float4& v, float tf) {
  return (v.x >= tf ? 1u : 0u) | (v.y >= tf ? 2u : 0u) | (v.z >= tf ? 4u : 0u) | (v.w >= tf ? 8u : 0u);
}

// Filter mask of a thread's stage data against tf: bits 4q..4q+3 for a[q]
// (only the float4s that lie inside the stage's nvec elements).
__device__ __forceinline__ uint32_t stage_mask(const float4 (&a)[kVec], int nvec, float tf, int tid) {
  uint32_t mask = 0;
#pragma unroll
  for (int q = 0; q < kVec; ++q)
    if (4 * (q * kThreads + tid) < nvec) mask |= pass4(a[q], tf) << (4 * q);
  return mask;
}

// kBlocks: this launch builds block lists in the single-unit row ends (the
// instantiation without it carries none of that code, so the stream loop
// keeps its registers when no block lists are asked for).
template <bool kBlocks, int NS, int CPS>
__global__ void __launch_bounds__(kThreads, CPS) topk_stream_kernel(const __grid_constant__ TopkLaunch p) {
  extern __shared__ unsigned char smem_raw[];
  SmemT<NS>& S = smem_ref<NS>(smem_raw);
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  pdl_trigger();  // the merge may be scheduled now; it waits for this grid to finish
  uint32_t* const wkey = S.cand.c.key + warp * kSub;  // this warp's sub-list
  int32_t* const widx = S.cand.c.idx + warp * kSub;
  uint64_t policy = 0;
  bool issuing = false;
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&S.full[i], 1);
    S.timeout = 0;
    fence_mbar_init();
    policy = l2_policy_evict_first();
    S.cur.unit = blockIdx.x;
    cursor_load(p, S.cur);
    issuing = true;
    for (int i = 0; i < NS && issuing; ++i) issuing = issue_stage(p, S, i, policy);
  }
  __syncthreads();
  uint32_t it = 0;
  int wcnt = 0;       // entries in this warp's sub-list (warp-uniform)
  int appended = 0;   // elements this warp let through the filter in this unit
  uint32_t tau = 0;   // keep elements whose order key >= tau
  // the previous unit's 512th score, its gap to the 256th, and its length
  // (spec_len 0: no estimate), from which the next unit's start is taken
  float spec_v512 = 0.f, spec_gap = 0.f;
  int spec_len = 0;
  uint32_t spec_used = 0;
  // Slow path of a stage (or of a redo step) in which some warp's survivors
  // did not fit its sub-list: cut all sub-lists, then the warps whose
  // survivors did not fit (!fits) append their data one float4 per lane at
  // a time, filtered against the raised threshold, with a cut before any
  // part that might not fit. Returns how many this warp appended.
  auto append_parts = [&](const float4(&a)[kVec], int nvec, float x, int xi, bool has_x, int base, bool fits) {
    int added = 0;
    wcnt = prune(S, wcnt, tau, tid);
#pragma unroll
    for (int q = 0; q < kVec; ++q) {
      if (q > 0 && named_bar_or(kBar, kThreads, wcnt > kSubCutAt)) wcnt = prune(S, wcnt, tau, tid);
      const float tf = tau_float(tau);
      uint32_t mq = 0;
      if (!fits && 4 * (q * kThreads + tid) < nvec) mq = pass4(a[q], tf) << (4 * q);
      const bool xq = !fits && q == 0 && has_x && x >= tf;
      int pq;
      const int tq = warp_offsets(mq, xq, lane, &pq);
      write_survivors(wkey, widx, wcnt + pq, a, x, xi, base, mq, xq, tid);
      wcnt += tq;
      added += tq;
    }
    return added;
  };
  while (true) {
    const int slot = it % NS;
    const uint32_t ph = (it / NS) & 1u;
    const bool ok = mbar_wait(&S.full[slot], ph);
    // after a timeout the descriptor is not trusted: process nothing, then
    // leave together at the barrier below
    const int4 hot = S.desc[slot].hot;
    const int unit = ok ? hot.x : 0;
    if (unit < 0) break;
    const int base = hot.y, nvec = ok ? hot.z : 0, flags = ok ? hot.w : 0;
    UnitInfo u{};
    if (flags) u = S.desc[slot].u;  // read before the slot is handed back
    const int row = u.row, batch = u.batch, lo = u.lo, len = u.len;
    const long long woff = u.woff;
    if (flags & 1) {
      wcnt = 0;
      appended = 0;
      // Start from a threshold extrapolated from the previous unit (or a
      // sampled one); whether it was low enough is checked exactly when the
      // unit ends. The previous unit's 256th and 512th scores are two points
      // of the score tail at quantiles 256/n' and 512/n'; the start is put
      // at quantile 1.4 * 512 / n on the line through them in log-quantile
      // (t = v512 - (v256 - v512) * log2(1.4 n' / n)), which keeps about
      // 1.4x the needed count when rows look alike, whatever their lengths.
      uint32_t est = 0;
      if (spec_len > 0 && len > 0) {
        const float t = spec_v512 - spec_gap * log2f(1.4f * static_cast<float>(spec_len) / static_cast<float>(len));
        if (isfinite(t)) est = order_key(t);
      }
      tau = est ? est : sample_tau(p.scores + woff + lo, len, S, tid);
      spec_used = tau;
    }
    float4 a[kVec];
#pragma unroll
    for (int q = 0; q < kVec; ++q) {
      a[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (4 * (q * kThreads + tid) < nvec) a[q] = reinterpret_cast<const float4*>(S.stage[slot])[q * kThreads + tid];
    }
    // scalar ends of the window (first stage of a unit)
    const bool has_x = (flags & 1) && tid < u.head + u.tail;
    float x = 0.f;
    int xi = 0;
    if (has_x) {
      xi = tid < u.head ? lo + tid : u.tail_at + (tid - u.head);
      x = __ldg(p.scores + woff + xi);
    }
    const float tf0 = tau_float(tau);
    const uint32_t mask = stage_mask(a, nvec, tf0, tid);
    const bool xs = has_x && x >= tf0;
    int pos;
    const int total = warp_offsets(mask, xs, lane, &pos);
    // A warp whose survivors fit appends them now, while the stage is still
    // in shared memory; one whose survivors do not fit defers them to the
    // slow path below (its registers still hold the stage).
    const bool fits = wcnt + total <= kSub;
    if (fits) {
      write_survivors_smem(wkey, widx, wcnt + pos, S.stage[slot], x, xi, base, mask, xs, tid);
      wcnt += total;
      appended += total;
    }
    if (!ok) S.timeout = 1;
    // Everyone is done with the stage, so the slot can be refilled. The same
    // barrier tells whether some warp deferred its survivors.
    const bool any = named_bar_or(kBar, kThreads, !ok || !fits);
    if (any && S.timeout) {
      if (tid == 0) {
        atomicOr(p.status, kDevWaitTimeout);
        // let the copies already issued land before the CTA exits (bounded)
        for (int k = 1; k < NS; ++k) mbar_wait(&S.full[(it + k) % NS], ((it + k) / NS) & 1u);
      }
      break;
    }
    if (tid == 0 && issuing) {
      fence_proxy_async_smem();
      issuing = issue_stage(p, S, slot, policy);
    }
    // The threshold is far below this stage's scores (e.g. the first unit of
    // a CTA, or a rising row) and some warp deferred its survivors.
    if (any) appended += append_parts(a, nvec, x, xi, has_x, base, fits);
    if (flags & 2) {
      if (lane == 0) S.wapp[warp] = appended;
      named_bar(kBar, kThreads);
      int passed = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) passed += S.wapp[w];
      if (spec_used && passed < min(len, kTopK)) {
        // The starting threshold was too high for this unit: redo it from
        // global memory with no threshold (exact again): the window's
        // 16-byte-aligned body in steps of kStage scores (float4 loads), its
        // scalar ends in the first step, with the stream's fit check and
        // slow path.
        wcnt = 0;
        tau = 0;
        const int body = len - u.head - u.tail;
        const float4* bsrc = reinterpret_cast<const float4*>(p.scores + woff + lo + u.head);
        for (int b0 = 0; b0 == 0 || b0 < body; b0 += kStage) {
          float4 r[kVec];
#pragma unroll
          for (int q = 0; q < kVec; ++q) {
            const int v4 = q * kThreads + tid;
            r[q] = 4 * v4 < body - b0 ? __ldg(bsrc + b0 / 4 + v4) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          const bool hx = b0 == 0 && tid < u.head + u.tail;
          float xr = 0.f;
          int xir = 0;
          if (hx) {
            xir = tid < u.head ? lo + tid : u.tail_at + (tid - u.head);
            xr = __ldg(p.scores + woff + xir);
          }
          const float tfr = tau_float(tau);
          const uint32_t rm = stage_mask(r, body - b0, tfr, tid);
          const bool rx = hx && xr >= tfr;
          int pr;
          const int tr = warp_offsets(rm, rx, lane, &pr);
          const bool rfits = wcnt + tr <= kSub;
          if (rfits) {
            write_survivors(wkey, widx, wcnt + pr, r, xr, xir, lo + u.head + b0, rm, rx, tid);
            wcnt += tr;
          }
          if (named_bar_or(kBar, kThreads, !rfits)) append_parts(r, body - b0, xr, xir, hx, lo + u.head + b0, rfits);
        }
        spec_used = 0;
      }
      const int cnt = gather_to_aux(S, wcnt, tau, tid);
      // entry e of this thread: key k[e], row-local index ix[e] (-1: none),
      // output rank rk[e]
      uint32_t k[4];
      int32_t ix[4];
      int rk[4];
      if (!bucket_rank512<kThreads>(S.aux_key, S.aux_idx, cnt, S.cand.rank.hist, S.cand.rank.bucket, S.sc, k, ix, rk,
                                    tid, kBar)) {
        unsigned long long v[4];
        bitonic_sort512_128(S.aux_key, S.aux_idx, cnt, S.cand.sortbuf, v, tid, kBar);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          k[e] = static_cast<uint32_t>(v[e] >> 32);
          ix[e] = v[e] ? static_cast<int32_t>(~static_cast<uint32_t>(v[e] & 0xFFFFFFFFull)) : -1;
          rk[e] = 4 * tid + e;
        }
      }
      if (tid == 0) S.spec_keys[0] = S.spec_keys[1] = 0;
      named_bar(kBar, kThreads);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (ix[e] >= 0 && rk[e] == kTopK / 2 - 1) S.spec_keys[0] = k[e];
        if (ix[e] >= 0 && rk[e] == kTopK - 1) S.spec_keys[1] = k[e];
      }
      if (p.chunks == 1) {
        const long long o = (long long)row * kTopK;
        int32_t sl[kTopK / kThreads];  // this thread's slots, for the block lists
#pragma unroll
        for (int e = 0; e < kTopK / kThreads; ++e) {
          sl[e] = -1;
          if (ix[e] < 0) continue;
          if (p.out_idx) p.out_idx[o + rk[e]] = ix[e];
          if (p.out_slots || (kBlocks && p.out_blocks)) {
            const int ps = p.page_size;
            const long long page = p.page_tables[(long long)batch * p.pt_stride + (ps == 1 ? ix[e] : ix[e] / ps)];
            sl[e] = static_cast<int>(ps == 1 ? page : page * ps + ix[e] % ps);
            if (p.out_slots) p.out_slots[o + rk[e]] = sl[e];
          }
        }
        for (int j = cnt + tid; j < kTopK; j += kThreads) {
          if (p.out_idx) p.out_idx[o + j] = -1;
          if (p.out_slots) p.out_slots[o + j] = -1;
        }
        if (kBlocks && p.out_blocks) {
          // the distinct blocks of the row's slots, built here from the
          // slots in registers (the ranking's scratch is free once read)
          named_bar(kBar, kThreads);
          row_blocks128(sl, kTopK, p.block_size, p.out_blocks + o, p.out_counts ? p.out_counts + row : nullptr,
                        S.cand.blocks, tid, kBar, true);
        }
      } else {
        const long long o = (long long)unit * kTopK;
#pragma unroll
        for (int e = 0; e < kTopK / kThreads; ++e) {
          if (ix[e] < 0) continue;
          p.part_key[o + rk[e]] = k[e];
          p.part_idx[o + rk[e]] = ix[e];
        }
        if (tid == 0) p.part_cnt[unit] = cnt;
      }
      named_bar(kBar, kThreads);
      // The tail points the next unit's starting threshold comes from.
      spec_len = 0;
      if (S.spec_keys[1] != 0) {
        const float v256 = key_to_float(S.spec_keys[0]), v512 = key_to_float(S.spec_keys[1]);
        if (isfinite(v256) && isfinite(v512)) {
          spec_v512 = v512;
          spec_gap = v256 - v512;
          spec_len = len;
        }
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
  uint32_t umin[kMergeUnits];  // lowest key of each full partial list
  uint32_t kmin, kmax;         // range of the kept candidates
  int32_t slot_s[kTopK];       // the row's slots, for its block list
  BlockScratch blocks;
};

__global__ void __launch_bounds__(kTopK, 1) merge_kernel(const __grid_constant__ MergeLaunch p) {
  extern __shared__ unsigned char smem_raw[];
  MergeSmem& S = *reinterpret_cast<MergeSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31;
  const long long row = blockIdx.x;
  const int U = p.units_per_row;  // <= kMergeUnits
  reinterpret_cast<uint4*>(S.hist)[2 * tid] = make_uint4(0, 0, 0, 0);
  reinterpret_cast<uint4*>(S.hist)[2 * tid + 1] = make_uint4(0, 0, 0, 0);
  if (tid < kMergeUnits) S.umin[tid] = 0xFFFFFFFFu;
  S.slot_s[tid] = -1;
  if (tid == 0) {
    S.kmin = 0xFFFFFFFFu;
    S.kmax = 0u;
  }
  pdl_wait();  // the partial lists come from the grid launched just before
  // entry tid of every partial list of the row, all loads in flight at once
  const long long base = row * U;
  int n[kMergeUnits];
  uint32_t kv[kMergeUnits];
  int32_t iv[kMergeUnits];
#pragma unroll
  for (int c = 0; c < kMergeUnits; ++c) n[c] = c < U ? min(max(p.part_cnt[base + c], 0), kTopK) : 0;
#pragma unroll
  for (int c = 0; c < kMergeUnits; ++c) {
    kv[c] = 0;
    iv[c] = -1;
    if (tid < n[c]) {
      kv[c] = p.part_key[(base + c) * kTopK + tid];
      iv[c] = p.part_idx[(base + c) * kTopK + tid];
    }
  }
  __syncthreads();
  // A full list holds the exact top 512 of its range, so its lowest key is
  // at most the row's 512th key: entries below the largest such bound cannot
  // be selected, and at least 512 entries reach it.
#pragma unroll
  for (int c = 0; c < kMergeUnits; ++c) {
    if (n[c] == kTopK) {  // the same for the whole block
      const uint32_t m = __reduce_min_sync(0xFFFFFFFFu, kv[c]);
      if (lane == 0) atomicMin(&S.umin[c], m);
    }
  }
  __syncthreads();
  uint32_t bound = 0;
#pragma unroll
  for (int c = 0; c < kMergeUnits; ++c)
    if (n[c] == kTopK) bound = max(bound, S.umin[c]);
  uint32_t selm = 0;
  int mine = 0;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
  for (int c = 0; c < kMergeUnits; ++c) {
    if (tid < n[c] && kv[c] >= bound) {
      selm |= 1u << c;
      ++mine;
      lo = min(lo, kv[c]);
      hi = max(hi, kv[c]);
    }
  }
  lo = __reduce_min_sync(0xFFFFFFFFu, lo);
  hi = __reduce_max_sync(0xFFFFFFFFu, hi);
  if (lane == 0) {
    atomicMin(&S.kmin, lo);
    atomicMax(&S.kmax, hi);
  }
  int total;
  int pos = block_exscan512(mine, &total, S.sc.wcnt, tid, 1);
#pragma unroll
  for (int c = 0; c < kMergeUnits; ++c) {
    if (selm & (1u << c)) {
      S.cand.c.key[pos] = kv[c];
      S.cand.c.idx[pos] = iv[c];
      ++pos;
    }
  }
  __syncthreads();
  int cnt = total;
  if (cnt > kTopK) {
    // 4096 bins over the candidates' key range
    const uint32_t span = S.kmax - S.kmin;
    const int shift = span >= 4096u ? (32 - __clz(span)) - 12 : 0;
    fast_select512<kMergeCap>(S.cand.c.key, S.cand.c.idx, cnt, S.kmin, shift, S.hist, S.aux_key, S.aux_idx, S.sc,
                              S.bcast, tid, 1);
    cnt = kTopK;
  } else {
    if (tid < cnt) {
      S.aux_key[tid] = S.cand.c.key[tid];
      S.aux_idx[tid] = S.cand.c.idx[tid];
    }
    __syncthreads();
  }
  // output order: rank the 512 by bucketing (half the threads, two entries
  // each), or with the sorting ranks when a bucket is too full
  const long long o = row * kTopK;
  const int batch = p.row_to_batch ? p.row_to_batch[row] : (int)row;
  auto emit = [&](uint32_t key, int32_t ix, int rk) {
    if (p.out_idx) p.out_idx[o + rk] = ix;
    if (p.out_scores) p.out_scores[o + rk] = key_to_float(key);
    if (p.out_slots || p.out_blocks) {
      const int ps = p.page_size;
      const long long page = p.page_tables[(long long)batch * p.pt_stride + (ps == 1 ? ix : ix / ps)];
      const int slot = static_cast<int>(ps == 1 ? page : page * ps + ix % ps);
      if (p.out_slots) p.out_slots[o + rk] = slot;
      S.slot_s[rk] = slot;
    }
  };
  uint32_t k2[2];
  int32_t i2[2];
  int r2[2];
  if (tid < kTopK / 2) {
    const bool ok = bucket_rank512<kTopK / 2>(S.aux_key, S.aux_idx, cnt, S.hist,
                                              reinterpret_cast<uint16_t*>(S.hist + 1024), S.sc, k2, i2, r2, tid, 2);
    if (tid == 0) S.bcast[0] = ok ? 1u : 0u;
  }
  __syncthreads();
  if (S.bcast[0]) {
    if (tid < kTopK / 2) {
#pragma unroll
      for (int e = 0; e < 2; ++e)
        if (i2[e] >= 0) emit(k2[e], i2[e], r2[e]);
    }
  } else {
    uint32_t k[1];
    int32_t ix[1];
    int rk[1];
    rank_sort<kTopK>(S.aux_key, S.aux_idx, cnt, S.cand.runs.key, S.cand.runs.idx, k, ix, rk, tid, 1);
    if (ix[0] >= 0) emit(k[0], ix[0], rk[0]);
  }
  if (tid >= cnt) {
    if (p.out_idx) p.out_idx[o + tid] = -1;
    if (p.out_slots) p.out_slots[o + tid] = -1;
    if (p.out_scores) p.out_scores[o + tid] = __int_as_float(0x7FC00000);
  }
  if (p.out_blocks) {  // the distinct blocks of the row's slots, by the first 128 threads
    __syncthreads();
    if (tid < kBlockThreads) {
      int32_t sl[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) sl[e] = S.slot_s[4 * tid + e];
      row_blocks128(sl, kTopK, p.block_size, p.out_blocks + o, p.out_counts ? p.out_counts + row : nullptr, S.blocks,
                    tid, 3, true);
    }
  }
}

// ---------------------------------------------------------------- rank
// When every row has a single partial list (the fused path with one KV
// chunk per row), that list already is the row's exact top 512: only the
// output order and the page transform remain. Four rows per CTA, 128
// threads each: load the list, rank it by bucketing (a bitonic network for
// heavy bins), write indices, slots and scores by rank.
constexpr int kRankRows = 4;

struct __align__(16) RankRowSmem {
  union {
    struct {
      uint32_t aux_key[kTopK];
      int32_t aux_idx[kTopK];
      union {
        struct {
          uint32_t hist[1024];
          uint16_t bucket[kTopK];
        } r;
        unsigned long long sortbuf[kTopK];
      } s;
      SelectScratch sc;
    } k;
    BlockScratch blocks;  // the row's block list, once its ranks are in registers
  } u;
};

__global__ void __launch_bounds__(kRankRows * 128) rank_kernel(const __grid_constant__ MergeLaunch p) {
  extern __shared__ unsigned char smem_raw[];
  const int g = threadIdx.x >> 7, t = threadIdx.x & 127;
  RankRowSmem& S = reinterpret_cast<RankRowSmem*>(smem_raw)[g];
  const long long row = (long long)blockIdx.x * kRankRows + g;
  const int bar = 1 + g;
  const bool live = row < p.rows;
  pdl_wait();  // the lists come from the grid launched just before
  const int cnt = live ? min(max(p.part_cnt[row], 0), kTopK) : 0;
  for (int j = t; j < cnt; j += 128) {
    S.u.k.aux_key[j] = p.part_key[row * kTopK + j];
    S.u.k.aux_idx[j] = p.part_idx[row * kTopK + j];
  }
  named_bar(bar, 128);
  uint32_t k4[4];
  int32_t i4[4];
  int rk4[4];
  if (!bucket_rank512<128>(S.u.k.aux_key, S.u.k.aux_idx, cnt, S.u.k.s.r.hist, S.u.k.s.r.bucket, S.u.k.sc, k4, i4,
                           rk4, t, bar)) {
    unsigned long long v[4];
    bitonic_sort512_128(S.u.k.aux_key, S.u.k.aux_idx, cnt, S.u.k.s.sortbuf, v, t, bar);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      k4[e] = static_cast<uint32_t>(v[e] >> 32);
      i4[e] = v[e] ? static_cast<int32_t>(~static_cast<uint32_t>(v[e] & 0xFFFFFFFFull)) : -1;
      rk4[e] = 4 * t + e;
    }
  }
  if (!live) return;
  const long long o = row * kTopK;
  const int batch = p.row_to_batch ? p.row_to_batch[row] : (int)row;
  const int ps = p.page_size;
  int32_t sl[4];  // this thread's slots, for the block list
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    sl[e] = -1;
    if (i4[e] < 0) continue;
    if (p.out_idx) p.out_idx[o + rk4[e]] = i4[e];
    if (p.out_scores) p.out_scores[o + rk4[e]] = key_to_float(k4[e]);
    if (p.out_slots || p.out_blocks) {
      const long long page = p.page_tables[(long long)batch * p.pt_stride + (ps == 1 ? i4[e] : i4[e] / ps)];
      sl[e] = static_cast<int>(ps == 1 ? page : page * ps + i4[e] % ps);
      if (p.out_slots) p.out_slots[o + rk4[e]] = sl[e];
    }
  }
  for (int j = cnt + t; j < kTopK; j += 128) {
    if (p.out_idx) p.out_idx[o + j] = -1;
    if (p.out_slots) p.out_slots[o + j] = -1;
    if (p.out_scores) p.out_scores[o + j] = __int_as_float(0x7FC00000);
  }
  if (p.out_blocks) {
    named_bar(bar, 128);  // the ranking's scratch is read; the block list reuses it
    row_blocks128(sl, kTopK, p.block_size, p.out_blocks + o, p.out_counts ? p.out_counts + row : nullptr, S.u.blocks,
                  t, bar, true);
  }
}

bool g_merge_attr_done[64];
bool g_rank_attr_done[64];

}  // namespace

TopkPlan topk_plan(long long rows, long long max_window, int num_sms) {
  TopkPlan pl{1, 0, kTopkWorkHeader};
  if (rows <= 0 || max_window <= 0) return TopkPlan{1, 0, 0};
  const long long slots = 2LL * num_sms;
  constexpr long long kMinChunk = SAI_TOPK_MIN_CHUNK;
  if (rows < slots && max_window > 2 * kMinChunk) {
    long long chunks = (max_window + kMinChunk - 1) / kMinChunk;
    chunks = std::min<long long>(chunks, kMergeUnits);
    long long len = (max_window + chunks - 1) / chunks;
    len = (len + 15) / 16 * 16;
    chunks = (max_window + len - 1) / len;
    pl.chunks = static_cast<int>(chunks);
    pl.chunk_len = static_cast<int>(len);
    const long long units = rows * chunks;
    pl.workspace_bytes =
        kTopkWorkHeader + static_cast<size_t>(units) * kTopK * 8 + static_cast<size_t>(units) * 4 + 256;
  }
  return pl;
}

size_t merge_smem_bytes() { return sizeof(MergeSmem); }

// Launch a kernel that starts with pdl_wait() so that it may be scheduled
// while the grid before it on the stream finishes.
template <typename Kernel>
cudaError_t launch_dependent(Kernel kernel, int grid, int block, size_t smem, cudaStream_t stream,
                             const MergeLaunch& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t launch_merge(const MergeLaunch& p, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  if (p.units_per_row < 1 || p.units_per_row > kMergeUnits) return cudaErrorInvalidValue;
  int dev = 0;
  cudaGetDevice(&dev);
  if (p.units_per_row == 1) {
    if (dev < 64 && !g_rank_attr_done[dev]) {
      cudaError_t e = cudaFuncSetAttribute(rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)(kRankRows * sizeof(RankRowSmem)));
      if (e != cudaSuccess) return e;
      g_rank_attr_done[dev] = true;
    }
    const int grid = (p.rows + kRankRows - 1) / kRankRows;
    return launch_dependent(rank_kernel, grid, kRankRows * 128, kRankRows * sizeof(RankRowSmem), stream, p);
  }
  if (dev < 64 && !g_merge_attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(MergeSmem));
    if (e != cudaSuccess) return e;
    g_merge_attr_done[dev] = true;
  }
  return launch_dependent(merge_kernel, p.rows, kTopK, sizeof(MergeSmem), stream, p);
}

template <bool kBlocks, int NS, int CPS>
static cudaError_t launch_stream(const TopkLaunch& p, int num_sms, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  constexpr size_t kBytes = smem_bytes<NS>();
  static bool attr_done[64];
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(topk_stream_kernel<kBlocks, NS, CPS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  static int ctas_per_sm[64];
  if (dev < 64 && ctas_per_sm[dev] == 0) {
    int nb = 0;
    cudaError_t e =
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, topk_stream_kernel<kBlocks, NS, CPS>, kThreads, kBytes);
    if (e != cudaSuccess) return e;
    ctas_per_sm[dev] = nb > 0 ? nb : 1;
  }
  const long long units = (long long)p.rows * p.chunks;
  const int grid = (int)std::min<long long>(units, (long long)(dev < 64 ? ctas_per_sm[dev] : 1) * num_sms);
  topk_stream_kernel<kBlocks, NS, CPS><<<grid, kThreads, kBytes, stream>>>(p);
  return cudaGetLastError();
}

// Stream kernel instance for a call: a call whose units all fit on the SMs
// at once runs one CTA per SM with a deep ring (nothing else shares the SM,
// so its stream is not limited by a two-stage pipeline); otherwise five CTAs
// per SM with two stages each. Block lists come from the stream kernel only
// when it ends the rows itself (one unit per row); split rows get theirs
// from the merge.
template <bool kBlocks>
static cudaError_t launch_stream_for(const TopkLaunch& p, int num_sms, cudaStream_t stream) {
  if ((long long)p.rows * p.chunks <= num_sms) return launch_stream<kBlocks, kDeepStages, 1>(p, num_sms, stream);
  return launch_stream<kBlocks, kNStage, kCtasPerSm>(p, num_sms, stream);
}

cudaError_t launch_topk_transform(const TopkLaunch& p, int num_sms, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  cudaError_t e = p.out_blocks && p.chunks == 1 ? launch_stream_for<true>(p, num_sms, stream)
                                                : launch_stream_for<false>(p, num_sms, stream);
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
  m.block_size = p.block_size;
  m.out_blocks = p.out_blocks;
  m.out_counts = p.out_counts;
  return launch_merge(m, stream);
}

}  // namespace sai
