// index_score_topk: FP8 index scores + top-512 in one pass, no score buffer.
//
// What is computed (ROCm/ATOM PR #1473 "enable minimax m3 fp8 index cache
// and fuse index_score_kernel with partial_topk kernel": pull request
// overview "Changes", the fused decode kernel over (query, index head, key
// chunk) and its paged block loop in the review diff of index_topk.py):
//
//   score(i, t) = kscale[p, o] * sum_h w[i, h] * relu( q[i, h, :] . k[p, o, :] )
//
// with p = block_table[b][t / 128], o = t % 128, b = row_to_batch[i] (or i),
// for every key t < seq_lens[i] (the causal length), then the top-512 keys
// by (score desc, index asc), mapped to physical slots p*128 + o. The pages
// name the fused kernel and its FP8 index cache but print no formula; this
// is the formula the library adopts (scale outside the relu, no 1/sqrt(d)).
//
// GB300 design. A work unit is a group of R query rows (R = 1 for decode,
// R = 4 for packed prefill, whose rows come in groups of 4 sharing one
// request) and a chunk of that request's KV blocks; one CTA per unit (the
// kernel can also walk several units with its barrier phases carried over).
// Roles:
//   * warp 4R streams each 128-token key block [128 keys x 128 dims]
//     through a shared-memory ring with 2-D TMA tensor loads (128-byte
//     swizzle; the paged gather is just the block's row coordinate);
//   * warp 4R+1 issues tcgen05.mma kind::f8f6f4 with the keys as M = 128 and
//     the group's R x 64 (row, head) query vectors as N, K = 128 dims in four
//     K = 32 steps, accumulating in FP32 in tensor memory, double-buffered;
//   * warps 4r..4r+3 are row r's epilogue, one TMEM lane quadrant (32 keys)
//     each: 16x256b tcgen05.ld gives a lane 4 keys x 16 heads, so the lane
//     keeps its 16 head weights in registers; relu (an exact saturating
//     multiply), the weighted head sum (f32x2 FMAs), a 4-lane reduce-scatter
//     to one key per lane, the key's scale, and the row's running top-k
//     filter.
//
// Running top-k. Each epilogue warp keeps its own candidate list and never
// waits for the row's other warps while the unit streams: when its list is
// about to overflow it cuts it, alone, to its own exact top 512 (every
// dropped key is beaten by 512 keys of the same warp). The row's warps meet
// twice per unit. (1) The unit's tiles are streamed starting from its middle
// tile (then wrapping around); after the first kSampleTiles tiles every
// key of those tiles is a candidate, and the row sets a start threshold at
// the m-th largest of those sampled scores, m about four standard
// deviations above the number of samples expected among the unit's top 512
// (so fewer than 512 keys reach it only rarely). (2) At the
// unit end the row's candidates are cut to its top 512. The start threshold
// is a guess: if fewer than 512 candidates reached it, keys above the true
// 512th may have been dropped, so the unit is streamed again (TMA, MMA and
// epilogue all replay it) without a start threshold. With at least 512
// candidates at or above the threshold, the 512th key is at or above it and
// nothing that belongs to the top 512 was dropped.
//
// The per-(row, chunk) candidate lists go to a workspace; the merge kernel
// of topk_transform.cu then selects, sorts and page-transforms each row.
//
// bf16 index cache (the "auto" cache type of the same pull request, i.e. the
// model dtype): q and the keys are bf16, the MMA is kind::f16 (K = 16 per
// instruction) and a 256-byte key row is staged as two 128-byte-swizzled
// halves of 64 dims (one TMA box each), so the MMA walks 2 x 4 K-steps; the
// relu is s + |s| (bf16 dot products have no fixed range), and the key
// scale may be absent (scale 1). Everything else is shared with the FP8 path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "sai_internal.h"
#include "sai_ptx.cuh"
#include "sai_select.cuh"

namespace sai {


namespace {

constexpr int kH = 64;        // index heads
constexpr int kD = 128;       // head dim (elements per row)
constexpr int kSwB = 128;     // bytes per row of one 128-byte-swizzled region
constexpr int kBlk = 128;     // tokens per KV block = MMA M
// K-tile ring slots and resident CTAs per SM: single rows (decode) run three
// small CTAs per SM with a 2-slot ring; groups of four rows (prefill, MMA
// N = 256, both accumulator buffers filling the SM's 512 TMEM columns) run
// one CTA per SM with a 4-slot ring (3 for bf16, whose query tile is twice
// as large). A ring slot is one 16 KB 128-byte-swizzled region of a key
// tile: an FP8 tile is one region, a bf16 tile two (dims 0-63, 64-127).
template <int R, bool BF16 = false>
__host__ __device__ constexpr int fused_stages() {
  return R == 1 ? 2 : (BF16 ? 3 : 4);
}
template <int R, bool BF16 = false>
__host__ __device__ constexpr int fused_ctas_per_sm() {
  return R == 1 ? 3 : 1;
}
template <bool BF16>
__host__ __device__ constexpr int elem_bytes() {
  return BF16 ? 2 : 1;
}
// 128-byte-swizzled regions per 128-dim row: 1 for FP8, 2 for bf16
template <bool BF16>
__host__ __device__ constexpr int sw_regions() {
  return kD * elem_bytes<BF16>() / kSwB;
}
// Candidate list per epilogue warp: a warp appends at most 32 per tile, and
// cuts its list to 512 when the next tile might not fit.
constexpr int kSub = 640;
static_assert(kSub >= kTopK + 32 && kSub % 32 == 0 && kSub / 32 <= 32, "sub-list size");
constexpr int kEpiRow = 128;       // epilogue threads per query row (4 warps, one TMEM lane quadrant each)
constexpr int kSampleTiles = 8;    // tiles sampled, spread over the unit, before the start threshold
constexpr int kSpecMinKeys = 2048; // a row's unit needs this many keys to start from a sampled threshold

template <int R, bool BF16>
struct __align__(1024) FusedSmem {
  // a ring slot is one region of a key tile, [128 keys x 128 bytes]; the
  // query tile is sw_regions() regions of [R*64 rows x 128 bytes]
  uint8_t kst[fused_stages<R, BF16>()][kBlk * kSwB];  // 16 KB each, 1024-aligned
  uint8_t q[R * kH * kD * elem_bytes<BF16>()];
  uint32_t ckey[R][4 * kSub];  // row r: four per-warp candidate lists
  int32_t cidx[R][4 * kSub];
  // the row's cut output; between the row's two meetings, each warp's 1 KB
  // quarter of it is that warp's histogram for cutting its own list
  uint32_t aux_key[R][kTopK];
  int32_t aux_idx[R][kTopK];
  SelectScratch sc[R];
  uint64_t full[fused_stages<R, BF16>()], empty[fused_stages<R, BF16>()], tfull[2], tempty[2];
  uint64_t qfull, qempty, verdict;
  uint32_t tmem_base;
  int wcnt[R][4];       // per-warp list sizes at a meeting of the row
  int row_fail[2][R];   // rows whose start threshold was too high, by pass parity
  int replay;           // the verdict of the last pass: 1 = stream the unit again
};

template <int R, bool BF16>
constexpr size_t fused_smem_bytes() {
  return sizeof(FusedSmem<R, BF16>) + 1024;
}

static_assert(3 * (fused_smem_bytes<1, false>() + 1024) <= 228 * 1024, "three single-row CTAs per SM");
static_assert(3 * (fused_smem_bytes<1, true>() + 1024) <= 228 * 1024, "three single-row bf16 CTAs per SM");
static_assert(fused_smem_bytes<4, false>() <= 227 * 1024, "one four-row CTA per SM");
static_assert(fused_smem_bytes<4, true>() <= 227 * 1024, "one four-row bf16 CTA per SM");

template <int R, bool BF16>
__device__ __forceinline__ FusedSmem<R, BF16>& fused_smem(unsigned char* raw) {
  uintptr_t a = reinterpret_cast<uintptr_t>(raw);
  a = (a + 1023) & ~static_cast<uintptr_t>(1023);
  return *reinterpret_cast<FusedSmem<R, BF16>*>(a);
}

// Row group metadata, recomputed identically by every thread.
struct GroupMeta {
  int row0, nrows;  // rows [row0, row0 + nrows)
  int batch;
  int nblk;         // blocks to visit for the group (max over its rows)
  int blk0, blk1;   // this unit's block range
};

template <int R>
__device__ GroupMeta group_meta(const FusedLaunch& p, int g, int c, int (&n)[R], bool report) {
  GroupMeta m;
  m.row0 = g * R;
  m.nrows = min(R, p.rows - m.row0);
  m.batch = p.row_to_batch ? p.row_to_batch[m.row0] : m.row0;
  bool bad_batch = m.batch < 0 || m.batch >= p.bt_rows;
  int nmax = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    n[r] = 0;
    if (r < m.nrows) {
      const int row = m.row0 + r;
      int nr = p.seq_lens[row];
      const int br = p.row_to_batch ? p.row_to_batch[row] : row;
      const bool bad = bad_batch || nr < 0 || nr > p.max_len || br != m.batch ||
                       (long long)(nr + kBlk - 1) / kBlk > p.bt_stride;
      if (bad) {
        if (report) atomicOr(p.status, kDevBadRowMeta);
        nr = 0;
      }
      n[r] = nr;
      nmax = max(nmax, nr);
    }
  }
  if (bad_batch) m.batch = 0;
  m.nblk = (nmax + kBlk - 1) / kBlk;
  m.blk0 = min(m.nblk, c * p.chunk_blocks);
  m.blk1 = min(m.nblk, m.blk0 + p.chunk_blocks);
  return m;
}

// The order in which a unit's T tiles are streamed (every role walks the
// same one): position i holds tile (i + T/2) mod T when the unit has at
// least 2 x kSampleTiles tiles, so the kSampleTiles tiles sampled for the
// start threshold come from the middle of the unit (not its first tokens,
// which can score high for every query, nor its most recent ones); shorter
// units stream in ascending order.
__device__ __forceinline__ int tile_at(int i, int T) {
  if (T < 2 * kSampleTiles) return i;
  const int t = i + (T >> 1);
  return t < T ? t : t - T;
}

// relu(s) * 2^-64 for an FP32 dot product s of two 128-element e4m3 rows:
// s * 2^-64 saturated to [0, 1]. Exact: |s| <= 128 * 448^2 < 2^64, so the
// clamp at 1 never acts, and s is a multiple of 2^-18, so s * 2^-64 is a
// normal float (no rounding); negatives and -0 give +0.
__device__ __forceinline__ float relu_lo(uint32_t s_bits) {
  float r;
  asm("mul.rn.sat.f32 %0, %1, 0f1F800000;" : "=f"(r) : "f"(__uint_as_float(s_bits)));
  return r;
}

// relu of an FP32 accumulator, on the FMA pipe (the ALU pipe is the busier
// one): FP8 keeps it scaled by 2^-64 (exact, see above); bf16 products have
// no such bound, so there it is s + |s| = 2 relu(s), exact for |s| < 2^127,
// with the 1/2 folded into the weights.
template <bool BF16>
__device__ __forceinline__ float relu_of(uint32_t s_bits) {
  if constexpr (BF16) {
    const float s = __uint_as_float(s_bits);
    return __fadd_rn(s, fabsf(s));
  } else {
    return relu_lo(s_bits);
  }
}

// ---- one warp's candidate list

// Keep, in place and in order, the entries of key/idx[0, n) for which
// keep(key, idx) holds; returns how many.
template <typename Keep>
__device__ __forceinline__ int warp_compact(uint32_t* key, int32_t* idx, int n, int lane, Keep keep) {
  int out = 0;
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    uint32_t k = 0;
    int32_t x = 0;
    bool kp = false;
    if (j < n) {
      k = key[j];
      x = idx[j];
      kp = keep(k, x);
    }
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, kp);
    __syncwarp();  // every lane has read its entry before any is overwritten (writes go to positions <= j)
    if (kp) {
      const int o = out + __popc(b & ((1u << lane) - 1u));
      key[o] = k;
      idx[o] = x;
    }
    out += __popc(b);
  }
  __syncwarp();
  return out;
}

// The need-th largest of the values v(j) (j < n, taken where get(j, v)
// holds) by four 8-bit radix passes over a 256-word histogram: on return
// `value` is that value and `need` how many of the entries equal to it are
// among the need largest (>= 1). Requires need <= the number of entries.
template <typename Get>
__device__ void warp_radix_select(int n, uint32_t& value, uint32_t& need, uint32_t* hist, int lane, Get get) {
  uint32_t prefix = 0, mask = 0;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = lane; b < 256; b += 32) hist[b] = 0u;
    __syncwarp();
    for (int j = lane; j < n; j += 32) {
      uint32_t v;
      if (get(j, v) && (v & mask) == prefix) atomicAdd(&hist[(v >> shift) & 255u], 1u);
    }
    __syncwarp();
    uint32_t h[8], tot = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      h[i] = hist[8 * lane + i];
      tot += h[i];
    }
    uint32_t suf = tot;  // inclusive suffix sum over lanes (lane l holds bins 8l .. 8l+7)
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_down_sync(0xFFFFFFFFu, suf, d);
      if (lane + d < 32) suf += o;
    }
    uint32_t above = suf - tot;
    int pick = -1;
    uint32_t pick_above = 0;
    if (above < need && need <= suf) {
#pragma unroll
      for (int i = 7; i >= 0; --i) {
        if (pick < 0 && above < need && need <= above + h[i]) {
          pick = 8 * lane + i;
          pick_above = above;
        }
        above += h[i];
      }
    }
    const int src = __ffs(__ballot_sync(0xFFFFFFFFu, pick >= 0)) - 1;
    pick = __shfl_sync(0xFFFFFFFFu, pick, src);
    pick_above = __shfl_sync(0xFFFFFFFFu, pick_above, src);
    prefix |= static_cast<uint32_t>(pick) << shift;
    mask |= 0xFFu << shift;
    need -= pick_above;
    __syncwarp();  // the histogram is read before the next pass clears it
  }
  value = prefix;
}

// Cut one warp's list key/idx[0, n), n > 512, in place to its top 512 by
// (key desc, index asc). Returns the 512th key: every dropped entry is below
// it or equal to it with a larger index.
__device__ __noinline__ uint32_t warp_cut512(uint32_t* key, int32_t* idx, int n, uint32_t* hist, int lane) {
  uint32_t kv, need = kTopK;
  warp_radix_select(n, kv, need, hist, lane, [&](int j, uint32_t& v) {
    v = key[j];
    return true;
  });
  uint32_t eq = 0;
  for (int j = lane; j < n; j += 32) eq += key[j] == kv ? 1u : 0u;
  eq = __reduce_add_sync(0xFFFFFFFFu, eq);
  // among the entries equal to kv, the `need` lowest indices stay
  uint32_t iv = 0;
  if (eq > need) {
    uint32_t need_i = need;
    warp_radix_select(n, iv, need_i, hist, lane, [&](int j, uint32_t& v) {
      v = 0x7FFFFFFFu - static_cast<uint32_t>(idx[j]);
      return key[j] == kv;
    });
  }
  const int kept = warp_compact(key, idx, n, lane, [&](uint32_t k, int32_t x) {
    return k > kv || (k == kv && 0x7FFFFFFFu - static_cast<uint32_t>(x) >= iv);
  });
  (void)kept;  // == 512
  return kv;
}

// The row's start threshold after its sample tiles (all 128 threads of the
// row, named barrier `bar`): the m-th largest of the row's sampled scores,
// as the lowest key of the radix bin that holds it (at least m sampled keys
// reach it); each warp then keeps only its list's entries at or above it.
// Of the `sampled` keys, about e = 512 x sampled / n_unit are expected
// among the unit's top 512 (a count with a standard deviation of at most
// sqrt(e)); m = e + 4 sqrt(e) + 2, so the threshold lies above the unit's
// 512th key (and the unit is replayed) only when that count runs four
// standard deviations high. The unit then keeps about 512 m / e candidates:
// ~680 for a decode unit sampling a third of its keys, ~1100 for a prefill
// unit sampling a thirtieth. Returns {threshold (0: none set),
// this warp's new list size}. `bins` (512 words) is the row's aux array.
__device__ __forceinline__ uint2 spec_threshold(int* wcnt, SelectScratch& sc, uint32_t* bins, uint32_t* my_key,
                                             int32_t* my_idx, int wc, int n_unit, int quad, int et, int lane,
                                             int bar) {
  __syncwarp();
  if (lane == 0) wcnt[quad] = wc;
  named_bar(bar, kEpiRow);
  int counts[4];
  int sampled = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    counts[q] = wcnt[q];
    sampled += counts[q];
  }
  uint32_t ts = 0;
  const float e = static_cast<float>(kTopK) * static_cast<float>(sampled) / static_cast<float>(n_unit);
  const long long mm = static_cast<long long>(ceilf(e + 4.f * sqrtf(e) + 2.f));
  if (mm >= 1 && mm < sampled) {
    const int cq = counts[quad];
    const Threshold th = radix_threshold_fast<kEpiRow>((uint32_t)mm, sc, bins, et, bar, [&](auto fn) {
      for (int j = lane; j < cq; j += 32) fn(my_key[j]);
    });
    ts = th.base + static_cast<uint32_t>(static_cast<uint64_t>(th.prefix) << th.lo);
    wc = warp_compact(my_key, my_idx, wc, lane, [&](uint32_t k, int32_t) { return k >= ts; });
    ts = max(ts, 1u);  // (a key of 0 would pass everything anyway)
  }
  named_bar(bar, kEpiRow);  // everyone has read the counts; aux is free again
  return make_uint2(ts, static_cast<uint32_t>(wc));
}

template <int R>
__host__ __device__ constexpr int fused_threads() {
  return R * kEpiRow + 64;  // R row groups of 4 epilogue warps, a TMA warp, an MMA warp
}

// What the epilogue produces: the running top-k (partial lists), the dense
// head-summed scores, or the dense per-head scores (each head's summand).
constexpr int kModeTopk = 0, kModeDense = 1, kModePerHead = 2;

// Work units are walked last to first: a packed prefill batch's later
// rows see the most keys, so its longest units start in the first wave and
// the shortest fill the last one.
__device__ __forceinline__ int unit_at(int i, int units) { return units - 1 - i; }

template <int R, int MODE, bool BF16>
__global__ void __launch_bounds__(fused_threads<R>(), (fused_ctas_per_sm<R, BF16>()))
    fused_score_topk_kernel(const __grid_constant__ FusedLaunch p, const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ unsigned char smem_raw[];
  FusedSmem<R, BF16>& S = fused_smem<R, BF16>(smem_raw);
  constexpr int N = R * kH;          // MMA N
  constexpr uint32_t kCols = 2 * N;  // two accumulator buffers
  constexpr uint32_t kIdesc = BF16 ? umma_idesc_bf16(kBlk, N) : umma_idesc_e4m3(kBlk, N);
  constexpr int kRegions = sw_regions<BF16>();
  constexpr uint32_t kSlotBytes = kBlk * kSwB;  // one region of a key tile
  constexpr uint32_t kQTileBytes = N * kD * elem_bytes<BF16>();
  constexpr int kEpiWarps = 4 * R;
  constexpr int kTmaWarp = kEpiWarps, kMmaWarp = kEpiWarps + 1;
  constexpr int kNSf = fused_stages<R, BF16>();
  constexpr int kEpiBar = 1 + R;  // named barrier of all epilogue threads (rows use 1 .. R)
  // only the top-k mode can replay a unit (the dense modes set no start threshold)
  constexpr bool kTopkMode = MODE == kModeTopk;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int units = ((p.rows + R - 1) / R) * p.chunks;

  if (tid == 0) {
    for (int i = 0; i < kNSf; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.tfull[i], 1);
      mbar_init(&S.tempty[i], kEpiWarps * 32);  // every epilogue thread arrives (no lane-0 branch)
    }
    mbar_init(&S.qfull, 1);
    mbar_init(&S.qempty, 1);
    mbar_init(&S.verdict, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&S.tmem_base, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  if constexpr (MODE == kModeTopk) pdl_trigger();  // the merge may be scheduled now; it waits for this grid to finish

  // Every role walks the same units (blockIdx.x, + gridDim.x, ..., mapped
  // by unit_at) and passes (a unit is streamed again when the epilogue's
  // verdict says so) and derives the same tile counts, so the barrier phases
  // below (counted over all tiles, passes and units of this CTA) stay in step.
  if (warp == kTmaWarp) {
    // ---------------- TMA producer: the unit's query tile, then its key
    // blocks through the ring; the block ids come straight from the table
    if (lane == 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&qmap);
      const uint64_t keep = l2_policy_evict_last();  // q and K are re-read by other CTAs
      uint32_t it = 0, qn = 0, vn = 0;
      bool run = true;
      for (int iu = blockIdx.x; iu < units && run; iu += gridDim.x) {
        const int u = unit_at(iu, units);
        int n[R];
        const GroupMeta m = group_meta<R>(p, u / p.chunks, u % p.chunks, n, false);
        const int ntiles = m.blk1 - m.blk0;
        if (ntiles == 0) continue;
        const int32_t* bt = p.block_table + (long long)m.batch * p.bt_stride + m.blk0;
        run = mbar_wait(&S.qempty, (qn & 1u) ^ 1u);
        if (!run) break;
        mbar_arrive_expect_tx(&S.qfull, kQTileBytes);
#pragma unroll
        for (int h = 0; h < kRegions; ++h)  // region h: dims [64h, 64h + 64) of a bf16 row
          tma_load_2d(S.q + h * N * kSwB, &qmap, h * (kSwB / elem_bytes<BF16>()), m.row0 * kH, &S.qfull, keep);
        ++qn;
        bool again = true;
        while (again && run) {
          int page_next = __ldg(bt + tile_at(0, ntiles));
          // (test hook: a stalled unit streams no key tiles, so every wait
          // for them runs out)
          for (int i = 0; i < ntiles && run && u != p.stall_unit; ++i) {
            int page = page_next;
            if (i + 1 < ntiles) page_next = __ldg(bt + tile_at(i + 1, ntiles));
            if (page < 0 || page >= p.num_blocks) page = 0;  // the epilogue masks this block
#pragma unroll
            for (int h = 0; h < kRegions; ++h, ++it) {  // region h: dims [64h, 64h + 64) of a bf16 key
              const int s = it % kNSf;
              if (!(run = mbar_wait(&S.empty[s], ((it / kNSf) & 1u) ^ 1u))) break;
              mbar_arrive_expect_tx(&S.full[s], kSlotBytes);
              tma_load_2d(S.kst[s], &kmap, h * (kSwB / elem_bytes<BF16>()), page * kBlk, &S.full[s], keep);
            }
          }
          again = false;
          if (kTopkMode && run) {  // the epilogue's verdict on this pass
            if (!(run = mbar_wait(&S.verdict, vn & 1u))) break;
            ++vn;
            again = *reinterpret_cast<volatile int*>(&S.replay) != 0;
          }
        }
      }
      if (!run) atomicOr(p.status, kDevWaitTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, rs = 0, qn = 0, vn = 0;  // tiles (accumulator buffers), ring slots, query tiles, verdicts
      bool run = true;
      for (int iu = blockIdx.x; iu < units && run; iu += gridDim.x) {
        const int u = unit_at(iu, units);
        int n[R];
        const GroupMeta m = group_meta<R>(p, u / p.chunks, u % p.chunks, n, false);
        const int ntiles = m.blk1 - m.blk0;
        if (ntiles == 0) continue;
        if (!(run = mbar_wait(&S.qfull, qn & 1u))) break;
        ++qn;
        const uint64_t bdesc = umma_desc_sw128_kmajor(smem_u32(S.q));
        bool again = true;
        while (again && run) {
          for (int i = 0; i < ntiles && run; ++i, ++it) {
            const int buf = it & 1;
            if (!(run = mbar_wait(&S.tempty[buf], ((it >> 1) & 1u) ^ 1u))) break;
            // each instruction takes 32 bytes of K (32 FP8 or 16 bf16 dims):
            // four per region (ring slot); the descriptor start field counts 16 B
#pragma unroll
            for (int h = 0; h < kRegions; ++h, ++rs) {
              const int s = rs % kNSf;
              if (!(run = mbar_wait(&S.full[s], (rs / kNSf) & 1u))) break;
              tc_fence_after();
              const uint64_t adesc = umma_desc_sw128_kmajor(smem_u32(S.kst[s]));
#pragma unroll
              for (int k = 0; k < kSwB / 32; ++k) {
                const uint64_t ad = adesc + (uint64_t)(2 * k);
                const uint64_t bd = bdesc + (uint64_t)(h * N * kSwB / 16 + 2 * k);
                const uint32_t acc = (h > 0 || k > 0) ? 1u : 0u;
                if constexpr (BF16)
                  umma_bf16(tmem + buf * N, ad, bd, kIdesc, acc);
                else
                  umma_f8(tmem + buf * N, ad, bd, kIdesc, acc);
              }
              umma_commit(&S.empty[s]);
            }
            if (!run) break;
            umma_commit(&S.tfull[buf]);
          }
          again = false;
          if (kTopkMode && run) {
            if (!(run = mbar_wait(&S.verdict, vn & 1u))) break;
            ++vn;
            again = *reinterpret_cast<volatile int*>(&S.replay) != 0;
          }
        }
        umma_commit(&S.qempty);  // the query tile is free once this unit's MMAs are done
      }
      if (!run) atomicOr(p.status, kDevWaitTimeout);
    }
  } else {
    // ---------------- epilogue: row r = warp / 4 of the group; TMEM lanes
    // quad*32 .. quad*32+31 (the warp's quadrant) are its 32 keys
    const int r = warp >> 2, quad = warp & 3, et = tid - r * kEpiRow;  // et = thread within the row's 128
    const int bar = 1 + r;
    uint32_t* const ckey = S.ckey[r];
    int32_t* const cidx = S.cidx[r];
    uint32_t* const my_key = ckey + quad * kSub;
    const uint32_t lt_mask = (1u << lane) - 1u;
    int32_t* const my_idx = cidx + quad * kSub;
    // this warp's histogram for cutting its own list: its quarter of aux
    uint32_t* const whist = quad < 2 ? S.aux_key[r] + 256 * quad : reinterpret_cast<uint32_t*>(S.aux_idx[r]) + 256 * (quad - 2);
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    // TMEM is read in the 16x256b shape: a warp loads its 32 keys as two
    // 16-lane halves, and lane l gets keys l/4 and l/4 + 8 of each half at
    // heads 8j + 2(l%4) + {0, 1}, j < 8. So a lane needs only those 16 head
    // weights (kept in registers) and holds partial sums for 4 keys; a
    // reduce-scatter over the 4 lanes sharing l/4 leaves each lane the full
    // score of one key, key kl of the block.
    const int kl = quad * 32 + (lane >> 2) + 8 * ((lane >> 1) & 1) + 16 * (lane & 1);
    constexpr float kWScale = BF16 ? 0.5f : 0x1p64f;  // undoes relu_of's scaling
    bool ok = true;     // false after a pipeline wait gave up (then nothing more is waited for)
    uint32_t tt = 0;    // tiles so far (accumulator buffer and phase)
    uint32_t vn = 0;    // verdicts so far (passes over units)
    for (int iu = blockIdx.x; iu < units; iu += gridDim.x) {
      const int u = unit_at(iu, units);
      const int g = u / p.chunks, c = u - g * p.chunks;
      int n[R];
      const GroupMeta m = group_meta<R>(p, g, c, n, et == 0 && r == 0 && c == 0);
      const int ntiles = m.blk1 - m.blk0;
      if (ntiles == 0) {
        // nothing streamed: an empty partial list per row
        if (kTopkMode && r < m.nrows && et == 0) p.part_cnt[(long long)(m.row0 + r) * p.chunks + c] = 0;
        continue;
      }
      const bool row_live = r < m.nrows;
      const int nr = row_live ? n[r] : 0;
      const int32_t* bt = p.block_table + (long long)m.batch * p.bt_stride + m.blk0;
      // keys of this row in this unit
      const int n_unit = row_live ? max(0, min(nr - m.blk0 * kBlk, ntiles * kBlk)) : 0;
      float2 w2[8];
      const float* wr = p.w + (long long)(row_live ? m.row0 + r : 0) * kH + 2 * (lane & 3);
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // FP8: scaled by 2^64, see relu_lo below
        float wa = row_live ? __ldg(wr + 8 * j) : 0.f, wb = row_live ? __ldg(wr + 8 * j + 1) : 0.f;
        if (MODE == kModePerHead && p.sign_w) {
          wa = static_cast<float>((wa > 0.f) - (wa < 0.f));
          wb = static_cast<float>((wb > 0.f) - (wb < 0.f));
        }
        w2[j] = make_float2(wa * kWScale, wb * kWScale);
      }
      // the key scale of the next tile is fetched one tile ahead (1 when the
      // cache has no scales)
      auto key_scale = [&](int page) -> float {
        return p.kscale ? __ldg(p.kscale + (long long)page * kBlk + kl) : 1.f;
      };
      bool row_done = !row_live || !kTopkMode;  // this row's partial list is written
      for (int pass = 0;; ++pass) {
        // a row streams its keys on the first pass, and again on a replay
        // if its start threshold failed; a done row only drains the tiles
        const bool active = !row_done || !kTopkMode;
        // the start threshold is sampled on the first pass only
        const bool spec = kTopkMode && active && pass == 0 && ntiles >= 2 * kSampleTiles && n_unit >= kSpecMinKeys;
        int wc = 0;         // entries in this warp's list
        uint32_t tau = 0;   // keep keys whose order key >= tau
        float tf = tau_float(0);
        bool spec_used = false;
        // position i of the walk holds tile `cur` of the unit (rotated to
        // start in the middle, see tile_at); `nxt` is position i + 1's
        int nxt = tile_at(0, ntiles);
        int page_next = __ldg(bt + nxt);
        bool ok_next = static_cast<unsigned>(page_next) < static_cast<unsigned>(p.num_blocks);
        float ks_next = ok_next ? key_scale(page_next) : 0.f;
        if (!active) {
          // drain: free each accumulator buffer of the pass (a done row of a
          // group whose other rows stream the unit again)
          for (int i = 0; i < ntiles; ++i, ++tt) {
            const int buf = tt & 1;
            ok = ok && __all_sync(0xFFFFFFFFu, mbar_wait(&S.tfull[buf], (tt >> 1) & 1u));
            tc_fence_after();
            tc_fence_before();
            if (ok) mbar_arrive(&S.tempty[buf]);
          }
        }
        bool bad_page = false;  // reported once, after the pass
        for (int i = 0; active && i < ntiles; ++i, ++tt) {
          const int cur = nxt, buf = tt & 1;
          nxt = cur + 1 == ntiles ? 0 : cur + 1;
          const int blk = m.blk0 + cur;
          const int t = blk * kBlk + kl;
          const bool page_ok = ok_next;
          const float ks = ks_next;
          const int page = page_next;
          // (after the last position nxt wraps to a tile already read: in range)
          page_next = __ldg(bt + nxt);
          ok_next = static_cast<unsigned>(page_next) < static_cast<unsigned>(p.num_blocks);
          ks_next = ok_next ? key_scale(page_next) : 0.f;
          bad_page |= !page_ok;
          if (ok && !__all_sync(0xFFFFFFFFu, mbar_try_wait(&S.tfull[buf], (tt >> 1) & 1u)))
            ok = __all_sync(0xFFFFFFFFu, mbar_wait_slow(&S.tfull[buf], (tt >> 1) & 1u));
          float score = 0.f;
          if (ok) {
            tc_fence_after();
            const uint32_t col = tmem + lane_base + static_cast<uint32_t>(buf * N + r * kH);
            // sum_h w_h relu(s_h) = sum_h (w_h 2^64) relu_lo(s_h): the relu
            // is one saturating multiply on the FMA pipe (the ALU pipe, where
            // a max would go, is the busier one), then packed f32x2 FMAs; the
            // power-of-two scalings are exact, so every product is w_h relu(s_h).
            // acc[k] = this lane's partial for keys l/4, l/4+8, 16+l/4, 24+l/4
            float2 acc[4];  // set by the first head pair's multiply
            // per-head mode: the scales of this lane's 4 keys, and its row's
            // [64, dense_stride] block of the output
            float ksq[4] = {0.f, 0.f, 0.f, 0.f};
            float* const ph_out = p.dense + (long long)(m.row0 + (row_live ? r : 0)) * kH * p.dense_stride;
            if constexpr (MODE == kModePerHead) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int key = quad * 32 + (lane >> 2) + 8 * (e & 1) + 16 * (e >> 1);
                ksq[e] = page_ok ? (p.kscale ? __ldg(p.kscale + (long long)page * kBlk + key) : 1.f)
                                 : __int_as_float(0xFF800000);  // a key on a bad block scores -inf
              }
            }
            // The 32 keys x 64 heads come in four 16-lane x 32-column loads
            // (half = keys 0-15 / 16-31 of the quadrant, hq = heads 0-31 /
            // 32-63); with one CTA per SM (groups of four rows) each is
            // issued before the math of the one before it, so the TMEM
            // latency hides behind the FMA work. Load (half, hq)
            // gives lane l keys l/4 and l/4 + 8 of the half at heads
            // 32 hq + 8j + 2(l%4) + {0, 1}, j < 4: weights w2[4 hq + j].
            auto math = [&](const uint32_t (&a)[16], int half, int hq) {
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const int j = 4 * hq + jj;
                const float2 x0 = make_float2(relu_of<BF16>(a[4 * jj]), relu_of<BF16>(a[4 * jj + 1]));
                const float2 x1 = make_float2(relu_of<BF16>(a[4 * jj + 2]), relu_of<BF16>(a[4 * jj + 3]));
                if constexpr (MODE == kModePerHead) {
                  // heads h0, h0 + 1 of keys key0 and key0 + 8: w_h relu(s_h) x scale
                  const int h0 = 8 * j + 2 * (lane & 3);
                  const int key0 = quad * 32 + 16 * half + (lane >> 2);
                  const int t0 = blk * kBlk + key0, t1 = t0 + 8;
                  float* const o0 = ph_out + (long long)h0 * p.dense_stride;
                  float* const o1 = o0 + p.dense_stride;
                  if (row_live && t0 < nr) {
                    const float sc = ksq[2 * half];
                    o0[t0] = page_ok ? x0.x * w2[j].x * sc : sc;
                    o1[t0] = page_ok ? x0.y * w2[j].y * sc : sc;
                  }
                  if (row_live && t1 < nr) {
                    const float sc = ksq[2 * half + 1];
                    o0[t1] = page_ok ? x1.x * w2[j].x * sc : sc;
                    o1[t1] = page_ok ? x1.y * w2[j].y * sc : sc;
                  }
                } else if (j == 0) {
                  acc[2 * half] = __fmul2_rn(x0, w2[j]);
                  acc[2 * half + 1] = __fmul2_rn(x1, w2[j]);
                } else {
                  acc[2 * half] = __ffma2_rn(x0, w2[j], acc[2 * half]);
                  acc[2 * half + 1] = __ffma2_rn(x1, w2[j], acc[2 * half + 1]);
                }
              }
            };
            auto taddr = [&](int half, int hq) {
              return col + (static_cast<uint32_t>(16 * half) << 16) + static_cast<uint32_t>(32 * hq);
            };
            if constexpr (R >= 4) {
              uint32_t b0[16], b1[16];
              tmem_ld16x256_x4(taddr(0, 0), b0);
              tmem_ld_wait16(b0);
              tmem_ld16x256_x4(taddr(0, 1), b1);
              math(b0, 0, 0);
              tmem_ld_wait16(b1);
              tmem_ld16x256_x4(taddr(1, 0), b0);
              math(b1, 0, 1);
              tmem_ld_wait16(b0);
              tmem_ld16x256_x4(taddr(1, 1), b1);
              math(b0, 1, 0);
              tmem_ld_wait16(b1);
              // the accumulator buffer is free once all its loads are in registers
              tc_fence_before();
              mbar_arrive(&S.tempty[buf]);
              math(b1, 1, 1);
            } else {
              // single rows (three CTAs per SM hide the latency): one
              // 16-lane x 64-column load per half
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                uint32_t a[32];
                tmem_ld16x256_x8(col + (static_cast<uint32_t>(16 * half) << 16), a);
                tmem_ld_wait();
                if (half == 1) {  // the accumulator buffer is free once both halves are in registers
                  tc_fence_before();
                  mbar_arrive(&S.tempty[buf]);
                }
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                  // registers 16 hq .. 16 hq + 15 are the head quarter hq
                  const uint32_t(&aq)[16] = *reinterpret_cast<const uint32_t(*)[16]>(a + 16 * hq);
                  math(aq, half, hq);
                }
              }
            }
            const float p0 = acc[0].x + acc[0].y, p1 = acc[1].x + acc[1].y;
            const float p2 = acc[2].x + acc[2].y, p3 = acc[3].x + acc[3].y;
            // reduce-scatter over lanes 4g..4g+3: after the xor-1 step a lane
            // holds two keys (l/4 and l/4 + 8 if l is even, else 16 + l/4 and
            // 24 + l/4), after the xor-2 step one (the second of them if l & 2)
            const bool odd = lane & 1, hi = lane & 2;
            float k0 = odd ? p2 : p0, k1 = odd ? p3 : p1;
            k0 += __shfl_xor_sync(0xFFFFFFFFu, odd ? p0 : p2, 1);
            k1 += __shfl_xor_sync(0xFFFFFFFFu, odd ? p1 : p3, 1);
            const float keep = hi ? k1 : k0;
            score = (keep + __shfl_xor_sync(0xFFFFFFFFu, hi ? k0 : k1, 2)) * ks;
          }
          const bool live = ok && page_ok && t < nr;  // (nr = 0 for a row past the group's end)
          if constexpr (MODE == kModeDense) {
            if (live) p.dense[(long long)(m.row0 + r) * p.dense_stride + t] = score;
          } else if constexpr (MODE == kModeTopk) {
            // running top-k filter: cut this warp's list if the tile's
            // survivors might not fit, then append them
            const bool pass_ = live && score >= tf;
            const uint32_t bal = __ballot_sync(0xFFFFFFFFu, pass_);
            if (bal) {
              // cut this warp's list first if the survivors might not fit
              // (they passed the old threshold: keeping them is still exact)
              if (wc > kSub - 32) {
                tau = max(tau, warp_cut512(my_key, my_idx, wc, whist, lane));
                tf = tau_float(tau);
                wc = kTopK;
              }
              const int pos = wc + __popc(bal & lt_mask);
              st_shared_if(pass_, my_key + pos, order_key(score));
              st_shared_if(pass_, reinterpret_cast<uint32_t*>(my_idx) + pos, static_cast<uint32_t>(t));
              wc += __popc(bal);
            }
            if (spec && i == kSampleTiles - 1) {
              // the sample tiles are in: the row's start threshold
              const uint2 sw = spec_threshold(S.wcnt[r], S.sc[r], S.aux_key[r], my_key, my_idx, wc, n_unit, quad, et,
                                              lane, bar);
              wc = static_cast<int>(sw.y);
              if (sw.x != 0u) {
                tau = max(tau, sw.x);
                tf = tau_float(tau);
                spec_used = true;
              }
            }
          }
        }
        if (bad_page && et == 0 && r == 0 && pass == 0) atomicOr(p.status, kDevBadPage);
        bool row_failed = false;
        if constexpr (MODE == kModeTopk) {
          if (active) {
            // unit end: cut the row's candidates to 512
            __syncwarp();
            if (lane == 0) S.wcnt[r][quad] = wc;
            const bool all_ok = named_bar_and(bar, kEpiRow, ok);
            int counts[4];
            int total = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              counts[q] = S.wcnt[r][q];
              total += counts[q];
            }
            int kept = 0;  // after a timeout the lists are not trusted: an empty list
            if (all_ok && total > kTopK) {
              select512_sub_to_aux<kEpiRow, 4, kSub>(ckey, cidx, counts, S.aux_key[r], S.aux_idx[r], S.sc[r], et,
                                                     bar);
              kept = kTopK;
            } else if (all_ok) {
              kept = total;
              int before = 0;
#pragma unroll
              for (int q = 0; q < 4; ++q) before += q < quad ? counts[q] : 0;
              for (int j = lane; j < wc; j += 32) {
                S.aux_key[r][before + j] = my_key[j];
                S.aux_idx[r][before + j] = my_idx[j];
              }
              named_bar(bar, kEpiRow);
            }
            // too high a start threshold: fewer than 512 keys reached it
            row_failed = all_ok && spec_used && total < kTopK;
            if (!row_failed && row_live) {
              const long long pu = (long long)(m.row0 + r) * p.chunks + c;
              const int cr = kept;
              for (int j = et; j < cr; j += kEpiRow) {
                p.part_key[pu * kTopK + j] = S.aux_key[r][j];
                p.part_idx[pu * kTopK + j] = S.aux_idx[r][j];
              }
              if (et == 0) p.part_cnt[pu] = cr;
            }
          }
          // the verdict of this pass: stream the unit again if a row failed
          if (et == 0) S.row_fail[vn & 1][r] = row_failed ? 1 : 0;
          named_bar(kEpiBar, R * kEpiRow);
          bool any = false;
#pragma unroll
          for (int q = 0; q < R; ++q) any = any || S.row_fail[vn & 1][q] != 0;
          if (tid == 0) {
            S.replay = any ? 1 : 0;
            mbar_arrive(&S.verdict);  // releases the replay flag to the TMA and MMA threads
          }
          ++vn;
          if (active && !row_failed) row_done = true;
          if (!any) break;
          // (aux and the lists are rewritten only after the row's next
          // barrier, which every thread of the row reaches after reading them)
        } else {
          break;
        }
      }
    }
    if (!ok && et == 0) atomicOr(p.status, kDevWaitTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 2-D map over [rows, 128] elements (uint8 FP8 codes or bf16) with a box of
// box_rows rows x 128 bytes (all 128 FP8 dims, or 64 bf16 dims), 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, long long rows, int box_rows, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int eb = bf16 ? 2 : 1;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD * eb)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kSwB / eb), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base),
            dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int R, int MODE, bool BF16>
cudaError_t launch_fused_t(const FusedLaunch& p, const void* kcache, cudaStream_t stream) {
  CUtensorMap kmap, qmap;
  if (!make_map(&kmap, kcache, p.num_blocks * kBlk, kBlk, BF16)) return cudaErrorInvalidValue;
  if (!make_map(&qmap, p.q, (long long)p.rows * kH, R * kH, BF16)) return cudaErrorInvalidValue;
  static bool attr_done[64];
  int dev = 0;
  cudaGetDevice(&dev);
  constexpr size_t smem = fused_smem_bytes<R, BF16>();
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(fused_score_topk_kernel<R, MODE, BF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  // One CTA per unit: decode units differ in length (row lengths vary), and
  // the hardware's CTA scheduler balances them better than a fixed
  // assignment of units to resident CTAs (measured); the kernel's unit loop
  // then runs once per CTA.
  const long long units = (long long)((p.rows + R - 1) / R) * p.chunks;
  const int grid = (int)units;
  fused_score_topk_kernel<R, MODE, BF16><<<grid, fused_threads<R>(), smem, stream>>>(p, kmap, qmap);
  return cudaGetLastError();
}

}  // namespace

#ifndef SAI_FUSED_UNITS_PER_SM
#define SAI_FUSED_UNITS_PER_SM 4  // work units per SM the plan aims at
#endif

FusedPlan fused_plan(long long rows, int max_seq_len, int group_rows, int num_sms) {
  FusedPlan pl{1, 1, 1, 0};
  // Packed prefill rows come in groups of 4 sharing a request; the kernel
  // takes each group in one CTA (MMA N = 256, one CTA per SM: each key tile
  // is staged once for four rows; measured faster than pairs of rows with
  // N = 128 and two CTAs per SM).
  pl.group = group_rows == 4 ? 4 : 1;
  const long long max_blocks = std::max<long long>(1, ((long long)max_seq_len + kBlk - 1) / kBlk);
  const long long groups = (rows + pl.group - 1) / pl.group;
  // about four units per SM (a little over one wave of three resident
  // single-row CTAs): measured against 2, 3, 5, 6 and 8 per SM on the
  // decode workload
  const long long target = (long long)SAI_FUSED_UNITS_PER_SM * num_sms;
  long long chunks = groups > 0 ? (target + groups - 1) / groups : 1;
  chunks = std::max<long long>(1, std::min<long long>({chunks, 12LL, max_blocks}));
  const long long cb = (max_blocks + chunks - 1) / chunks;
  pl.chunk_blocks = static_cast<int>(cb);
  pl.chunks = static_cast<int>((max_blocks + cb - 1) / cb);
  pl.workspace_bytes = static_cast<size_t>(rows) * pl.chunks * (kTopK * 8 + 4) + 256;
  return pl;
}

template <int MODE>
cudaError_t launch_fused_m(const FusedLaunch& p, int group, bool bf16, const void* kcache, cudaStream_t stream) {
  if (bf16)
    return group == 4 ? launch_fused_t<4, MODE, true>(p, kcache, stream) : launch_fused_t<1, MODE, true>(p, kcache, stream);
  return group == 4 ? launch_fused_t<4, MODE, false>(p, kcache, stream) : launch_fused_t<1, MODE, false>(p, kcache, stream);
}

cudaError_t launch_fused(const FusedLaunch& p, int group, FusedOut out, bool bf16, const void* kcache,
                         cudaStream_t stream) {
  switch (out) {
    case FusedOut::kTopk: return launch_fused_m<kModeTopk>(p, group, bf16, kcache, stream);
    case FusedOut::kDense: return launch_fused_m<kModeDense>(p, group, bf16, kcache, stream);
    case FusedOut::kPerHead: return launch_fused_m<kModePerHead>(p, group, bf16, kcache, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace sai
