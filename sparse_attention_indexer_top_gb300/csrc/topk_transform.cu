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
// GB300 design. One persistent CTA processes a strided list of work units
// (a whole row, or one chunk of a long row). Inside the CTA:
//   * a producer warp streams each unit's window into a ring of shared-memory
//     stages with 1-D bulk TMA copies (cp.async.bulk + mbarrier
//     complete_tx), evict-first in L2 since each score is read once. The
//     16-byte-aligned interior of the window goes through TMA; the <= 3
//     leading and <= 3 trailing elements (any row stride or row start) are
//     read by the producer with plain loads and handed over in the stage
//     descriptor. This is the scalar path the pages require when the stride
//     is not a multiple of 4, folded into every row instead of a fallback;
//   * 16 consumer warps turn each stage into order keys and keep a running
//     threshold tau: only keys > tau are appended (warp-aggregated) to a
//     shared candidate buffer. When the buffer nears capacity it is cut back
//     to the exact top 512 (radix select in shared memory) and tau rises.
//     Every later element has a larger index than all kept ones, so the
//     strict filter never drops a winner;
//   * at the end of a unit the candidates are cut to 512, bitonic-sorted by
//     (score desc, index asc), page-transformed and written (one unit per
//     row), or written as a partial list for the merge kernel (split rows).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "sai_internal.h"
#include "sai_ptx.cuh"
#include "sai_select.cuh"

namespace sai {
namespace {

constexpr int kConsumers = 512;                 // 16 consumer warps
constexpr int kThreads = kConsumers + 32;       // + 1 producer warp
constexpr int kStage = 2048;                    // floats per stage (8 KB): one float4 per consumer
constexpr int kNStage = 5;                      // 40 KB in flight per CTA
constexpr int kExtra = 8;                       // scalar elements per descriptor
constexpr int kPruneAt = 2048;                  // prune the candidate list above this size
constexpr int kCap = 4352;                      // >= kPruneAt + kStage + kExtra
constexpr int kScanEvery = 256;                 // raise the threshold after this many appends
constexpr int kBarConsumers = 1;                // named barrier id

static_assert(kTopK == kConsumers, "the final sort keeps one entry per consumer thread");
static_assert(kCap >= kPruneAt + kStage + kExtra, "candidate list overflow");
static_assert(kStage == 4 * kConsumers, "one float4 per consumer per stage");

struct StageDesc {
  int unit;   // -1: no more work
  int row;
  int base;   // row-local index of stage element 0
  int nvec;   // TMA elements in this stage (multiple of 4)
  int nextra;
  int flags;  // 1: first stage of the unit, 2: last stage of the unit
  int batch;  // page-table row
  int pad_;
  int extra_idx[kExtra];
  float extra_val[kExtra];
};

struct __align__(128) Smem {
  float stage[kNStage][kStage];
  union {
    struct {
      uint32_t key[kCap];
      int32_t idx[kCap];
    } c;
    unsigned long long runs[kTopK];  // final sort (the list is dead by then)
  } cand;
  uint32_t hist[4096];  // running histogram of key >> 20 of every appended element
  uint32_t aux_key[kTopK];
  int32_t aux_idx[kTopK];
  StageDesc desc[kNStage];
  uint64_t full[kNStage];
  uint64_t empty[kNStage];
  SelectScratch sc;
  uint32_t bcast[4];
  int add[3];
};

constexpr size_t kSmemBytes = sizeof(Smem) + 128;  // + alignment slack

__device__ __forceinline__ Smem& smem_ref(unsigned char* raw) {
  uintptr_t a = reinterpret_cast<uintptr_t>(raw);
  a = (a + 127) & ~static_cast<uintptr_t>(127);
  return *reinterpret_cast<Smem*>(a);
}

// ---------------------------------------------------------------- producer
__device__ void producer(const TopkLaunch& p, Smem& S) {
  const uint64_t policy = l2_policy_evict_first();
  const int units = p.rows * p.chunks;
  uint32_t it = 0;
  for (int u = blockIdx.x;; u += gridDim.x) {
    const bool done = u >= units;
    int row = 0, b = 0, lo = 0, hi = 0;
    const float* win = p.scores;
    if (!done) {
      row = u / p.chunks;
      const int ch = u - row * p.chunks;
      int n = p.seq_lens[row];
      const long long start = p.row_starts ? p.row_starts[row] : 0;
      b = p.row_to_batch ? p.row_to_batch[row] : row;
      bool bad = n < 0 || start < 0 || start + n > p.stride;
      if (p.page_tables) {
        bad = bad || b < 0 || b >= p.pt_rows || (n > 0 && (long long)(n - 1) / p.page_size >= p.pt_stride);
      }
      if (bad) {
        atomicOr(p.status, kDevBadRowMeta);
        n = 0;
        b = 0;
      }
      win = p.scores + (long long)row * p.stride + (bad ? 0 : start);
      lo = p.chunks > 1 ? ch * p.chunk_len : 0;
      hi = p.chunks > 1 ? min(n, lo + p.chunk_len) : n;
      if (lo > hi) lo = hi;
    }
    // split [lo, hi) into scalar head, 16-byte aligned body, scalar tail
    const int len = hi - lo;
    int head = (int)(((16u - (reinterpret_cast<uintptr_t>(win + lo) & 15u)) & 15u) >> 2);
    int body = 0;
    if (len <= kExtra || head > len) {
      head = len;
    } else {
      body = (len - head) & ~3;
    }
    const int tail = len - head - body;
    const int nst = done ? 1 : max(1, (body + kStage - 1) / kStage);
    for (int s = 0; s < nst; ++s, ++it) {
      const int slot = it % kNStage;
      const uint32_t ph = (it / kNStage) & 1u;
      if (!mbar_wait(&S.empty[slot], ph ^ 1u)) {
        atomicOr(p.status, kDevWaitTimeout);
        return;  // consumers time out on the full barrier and stop too
      }
      StageDesc& d = S.desc[slot];
      if (done) {
        d.unit = -1;
        mbar_arrive(&S.full[slot]);
        return;
      }
      d.unit = u;
      d.row = row;
      d.batch = b;
      d.flags = (s == 0 ? 1 : 0) | (s == nst - 1 ? 2 : 0);
      d.base = lo + head + s * kStage;
      d.nvec = min(kStage, body - s * kStage);
      d.nextra = 0;
      if (s == 0) {
        int e = 0;
        for (int i = 0; i < head; ++i, ++e) {
          d.extra_idx[e] = lo + i;
          d.extra_val[e] = __ldg(win + lo + i);
        }
        for (int i = 0; i < tail; ++i, ++e) {
          const int j = lo + head + body + i;
          d.extra_idx[e] = j;
          d.extra_val[e] = __ldg(win + j);
        }
        d.nextra = e;
      }
      if (d.nvec > 0) {
        mbar_arrive_expect_tx(&S.full[slot], (uint32_t)d.nvec * 4u);
        bulk_g2s_stream(S.stage[slot], win + d.base, (uint32_t)d.nvec * 4u, &S.full[slot], policy);
      } else {
        mbar_arrive(&S.full[slot]);
      }
    }
  }
}

// ---------------------------------------------------------------- consumers
// Append the elements whose bit is set in `mask` (order keys computed here)
// and count them in the running histogram; one shared atomic per warp for
// the positions.
__device__ __forceinline__ void append_pass(uint32_t* ckey, int32_t* cidx, uint32_t* hist, int base, int* counter,
                                            const float (&vals)[5], const int32_t (&idxs)[5], uint32_t mask,
                                            int lane) {
  const int m = __popc(mask);
  if (!__any_sync(0xFFFFFFFFu, m > 0)) return;
  int incl = m;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += o;
  }
  int start = 0;
  if (lane == 31) start = atomicAdd(counter, incl);
  int pos = __shfl_sync(0xFFFFFFFFu, start, 31) + base + incl - m;
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    if (mask & (1u << i)) {
      const uint32_t key = order_key(vals[i]);
      ckey[pos] = key;
      cidx[pos] = idxs[i];
      atomicAdd(&hist[key >> 20], 1u);
      ++pos;
    }
  }
}

// Write one row's output: entry of composite v goes to position `rank`;
// threads tid >= cnt write the -1 padding at position tid.
__device__ __forceinline__ void emit_ranked(long long row, int batch, unsigned long long v, int rank, int cnt,
                                            int tid, const int* pt, long long pt_stride, int ps, int* out_slots,
                                            int* out_idx, float* out_scores) {
  const long long o = row * kTopK;
  if (v != 0ull) {
    const int idx = static_cast<int>(~static_cast<uint32_t>(v & 0xFFFFFFFFull));
    if (out_idx) out_idx[o + rank] = idx;
    if (out_scores) out_scores[o + rank] = key_to_float(static_cast<uint32_t>(v >> 32));
    if (out_slots) {
      int slot = -1;
      if (pt) {
        const long long page = pt[(long long)batch * pt_stride + (ps == 1 ? idx : idx / ps)];
        slot = static_cast<int>(ps == 1 ? page : page * ps + idx % ps);
      }
      out_slots[o + rank] = slot;
    }
  }
  if (tid >= cnt) {
    if (out_idx) out_idx[o + tid] = -1;
    if (out_slots) out_slots[o + tid] = -1;
    if (out_scores) out_scores[o + tid] = __int_as_float(0x7FC00000);
  }
}

__device__ void consumers(const TopkLaunch& p, Smem& S, int tid) {
  const int lane = tid & 31;
  uint32_t* const ckey = S.cand.c.key;
  int32_t* const cidx = S.cand.c.idx;
  uint32_t it = 0;
  int cnt = 0;       // candidates held before the current stage (uniform)
  int since = 0;     // appends since the last threshold update
  uint32_t tau = 0;  // keep elements whose order key >= tau
  while (true) {
    const int slot = it % kNStage;
    const uint32_t ph = (it / kNStage) & 1u;
    // One thread polls the mbarrier; the others wait in the named barrier,
    // which also publishes the stage (and any timeout) to all consumers.
    const bool ok = named_bar_and(kBarConsumers, kConsumers, tid == 0 ? mbar_wait(&S.full[slot], ph) : true);
    if (!ok) {
      if (tid == 0) atomicOr(p.status, kDevWaitTimeout);
      return;
    }
    const StageDesc& d = S.desc[slot];
    const int unit = d.unit;
    if (unit < 0) return;
    const int flags = d.flags, nvec = d.nvec, nextra = d.nextra, base = d.base, row = d.row, batch = d.batch;
    if (flags & 1) {
      cnt = 0;
      since = 0;
      tau = 0;
    }
    const float tf = tau_float(tau);
    float vals[5];
    int32_t idxs[5];
    uint32_t mask = 0;
    if (4 * tid < nvec) {
      const float4 v = reinterpret_cast<const float4*>(S.stage[slot])[tid];
      vals[0] = v.x;
      vals[1] = v.y;
      vals[2] = v.z;
      vals[3] = v.w;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        idxs[i] = base + 4 * tid + i;
        mask |= (vals[i] >= tf ? 1u : 0u) << i;
      }
    }
    if (tid < nextra) {
      vals[4] = d.extra_val[tid];
      idxs[4] = d.extra_idx[tid];
      mask |= (vals[4] >= tf ? 1u : 0u) << 4;
    }
    append_pass(ckey, cidx, S.hist, cnt, &S.add[it % 3], vals, idxs, mask, lane);
    named_bar(kBarConsumers, kConsumers);
    if (tid == 0) {
      mbar_arrive(&S.empty[slot]);  // stage data and descriptor are no longer read
      S.add[(it + 2) % 3] = 0;      // counter of stage it+2; last read before this barrier
    }
    const int added = S.add[it % 3];
    cnt += added;
    since += added;
    if (since >= kScanEvery || cnt > kPruneAt) {
      since = 0;
      const BinCut c = hist_cut4096(S.hist, kTopK, S.sc.wmin, S.bcast, tid, kBarConsumers);
      if (c.bin >= 0) tau = max(tau, static_cast<uint32_t>(c.bin) << 20);
      if (cnt > kPruneAt) {
        cnt = compact_ge<kCap>(ckey, cidx, cnt, tau, S.sc.wcnt, tid, kBarConsumers);
        if (cnt > kPruneAt) {  // the threshold bin alone is too full: exact cut
          const uint32_t t2 = select_topk<kConsumers>(ckey, cidx, cnt, kTopK, S.aux_key, S.aux_idx, S.sc, tid,
                                                      kBarConsumers);
          tau = max(tau, t2);
          cnt = kTopK;
        }
      }
    }
    if (flags & 2) {
      // the running histogram counts pruned elements too: start a fresh one
      reinterpret_cast<uint4*>(S.hist)[2 * tid] = make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4*>(S.hist)[2 * tid + 1] = make_uint4(0, 0, 0, 0);
      named_bar(kBarConsumers, kConsumers);
      if (cnt > kTopK) {
        fast_select512<kCap>(ckey, cidx, cnt, S.hist, S.aux_key, S.aux_idx, S.sc, S.bcast, tid, kBarConsumers);
        cnt = kTopK;
      } else {
        if (tid < cnt) {
          S.aux_key[tid] = ckey[tid];
          S.aux_idx[tid] = cidx[tid];
        }
        named_bar(kBarConsumers, kConsumers);
      }
      if (p.chunks == 1) {
        unsigned long long v;
        const int rank = rank_sort512(S.aux_key, S.aux_idx, cnt, S.cand.runs, &v, tid, kBarConsumers);
        emit_ranked(row, batch, v, rank, cnt, tid, p.page_tables, p.pt_stride, p.page_size, p.out_slots, p.out_idx,
                    nullptr);
      } else {
        const long long o = (long long)unit * kTopK;
        if (tid < cnt) {
          p.part_key[o + tid] = S.aux_key[tid];
          p.part_idx[o + tid] = S.aux_idx[tid];
        }
        if (tid == 0) p.part_cnt[unit] = cnt;
        named_bar(kBarConsumers, kConsumers);
      }
      cnt = 0;
    }
    ++it;
  }
}

__global__ void __launch_bounds__(kThreads, 2) topk_stream_kernel(const __grid_constant__ TopkLaunch p) {
  extern __shared__ unsigned char smem_raw[];
  Smem& S = smem_ref(smem_raw);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < kNStage; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], 1);
    }
    S.add[0] = S.add[1] = S.add[2] = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < 4096; i += kThreads) S.hist[i] = 0;
  __syncthreads();
  if (tid >= kConsumers) {
    if (tid == kConsumers) producer(p, S);
    return;
  }
  consumers(p, S, tid);
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
    unsigned long long runs[kTopK];
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
  unsigned long long v;
  const int rank = rank_sort512(S.aux_key, S.aux_idx, cnt, S.cand.runs, &v, tid, 1);
  const int batch = cnt > 0 ? (p.row_to_batch ? p.row_to_batch[row] : (int)row) : 0;
  emit_ranked(row, batch, v, rank, cnt, tid, p.page_tables, p.pt_stride, p.page_size, p.out_slots, p.out_idx,
              p.out_scores);
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
  const long long units = (long long)p.rows * p.chunks;
  const int grid = (int)std::min<long long>(units, 2LL * num_sms);
  topk_stream_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p);
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
