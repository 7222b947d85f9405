// C-ABI layer of libsai: argument validation, workspace planning, device
// status word, launch on the caller's stream. See include/sai.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <mutex>

#include "../../include/sai.h"
#include "sai_internal.h"

namespace {

__device__ int g_device_status;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];
std::mutex g_mu;

// Per-device set-up, done once with that device current.
bool device_setup(int* dev_out, int** status, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return false;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return false;
    g_num_sms[dev] = n;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  *dev_out = dev;
  *status = g_status_ptr[dev];
  *sms = g_num_sms[dev];
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

thread_local const char* t_last_error = "";
thread_local int t_stall_unit = -1;  // test hook, consumed by the thread's next fused top-k call

// Map a CUDA error to a status, remembering its text for sai_last_error.
int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return SAI_OK;
  t_last_error = cudaGetErrorString(e);
  return SAI_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* sai_last_error(void) { return t_last_error; }

void sai_test_stall_next_fused(int32_t unit) { t_stall_unit = unit < 0 ? -1 : unit; }

const char* sai_status_string(int status) {
  switch (status) {
    case SAI_OK: return "ok";
    case SAI_ERR_NULL: return "a required pointer is NULL";
    case SAI_ERR_SHAPE: return "a size or count is out of range";
    case SAI_ERR_UNSUPPORTED: return "unsupported configuration";
    case SAI_ERR_WORKSPACE: return "workspace too small or misaligned";
    case SAI_ERR_CUDA: return "CUDA runtime or launch failure";
    case SAI_ERR_DEVICE_CHECK: return "a kernel flagged bad device-side metadata";
    case SAI_ERR_ALIGN: return "misaligned pointer";
    default: return "unknown status";
  }
}

int sai_device_status(int* out_bits, int clear, sai_stream_t stream) {
  if (!out_bits) return SAI_ERR_NULL;
  int dev, sms;
  int* st;
  if (!device_setup(&dev, &st, &sms)) return SAI_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int bits = 0;
  if (cudaMemcpyAsync(&bits, st, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return SAI_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SAI_ERR_CUDA;
  if (clear && bits) {
    if (cudaMemsetAsync(st, 0, sizeof(int), s) != cudaSuccess) return SAI_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SAI_ERR_CUDA;
  }
  *out_bits = bits;
  return bits ? SAI_ERR_DEVICE_CHECK : SAI_OK;
}

size_t sai_topk_transform_workspace(int64_t rows, int64_t score_stride, int32_t k) {
  if (rows <= 0 || score_stride <= 0 || k != SAI_TOPK) return 0;
  int dev, sms;
  int* st;
  if (!device_setup(&dev, &st, &sms)) return 0;
  return sai::topk_plan(rows, score_stride, sms).workspace_bytes;
}

int sai_topk_transform(const float* scores, int64_t rows, int64_t score_stride, const int32_t* row_starts,
                       const int32_t* seq_lens, const int32_t* page_tables, int64_t pt_rows, int64_t pt_stride,
                       const int32_t* row_to_batch, int32_t page_size, int32_t k, int32_t* out_slots,
                       int32_t* out_indices, int32_t block_size, int32_t* out_blocks, int32_t* out_counts,
                       void* workspace, size_t workspace_bytes, sai_stream_t stream) {
  if (k <= 0 || rows < 0) return SAI_ERR_SHAPE;
  if (k != SAI_TOPK) return SAI_ERR_UNSUPPORTED;
  if (rows > INT_MAX / 16) return SAI_ERR_SHAPE;
  if (!out_slots && !out_indices && !out_blocks) return SAI_ERR_NULL;
  if (out_counts && !out_blocks) return SAI_ERR_NULL;
  if (out_blocks && block_size < 1) return SAI_ERR_SHAPE;
  if (rows == 0) return SAI_OK;
  if (!scores || !seq_lens) return SAI_ERR_NULL;
  if (score_stride < 1) return SAI_ERR_SHAPE;
  if ((out_slots || out_blocks) && !page_tables) return SAI_ERR_NULL;
  if (page_tables) {
    if (page_size < 1 || pt_rows < 1 || pt_stride < 1) return SAI_ERR_SHAPE;
    if (!row_to_batch && pt_rows < rows) return SAI_ERR_SHAPE;
  }
  if (!aligned(scores, 4) || !aligned(seq_lens, 4) || (row_starts && !aligned(row_starts, 4)) ||
      (page_tables && !aligned(page_tables, 4)) || (row_to_batch && !aligned(row_to_batch, 4)) ||
      (out_slots && !aligned(out_slots, 4)) || (out_indices && !aligned(out_indices, 4)) ||
      (out_blocks && !aligned(out_blocks, 4)) || (out_counts && !aligned(out_counts, 4)))
    return SAI_ERR_ALIGN;
  int dev, sms;
  int* st;
  if (!device_setup(&dev, &st, &sms)) return SAI_ERR_CUDA;

  sai::TopkPlan plan = sai::topk_plan(rows, score_stride, sms);
  const bool have_ws = workspace && workspace_bytes >= sai::kTopkWorkHeader && aligned(workspace, 16);
  if (plan.chunks > 1 && (!have_ws || workspace_bytes < plan.workspace_bytes)) plan = sai::TopkPlan{1, 0, 0};

  sai::TopkLaunch p{};
  p.scores = scores;
  p.stride = score_stride;
  p.rows = static_cast<int>(rows);
  p.row_starts = row_starts;
  p.seq_lens = seq_lens;
  p.page_tables = page_tables;
  p.pt_rows = page_tables ? pt_rows : 0;
  p.pt_stride = page_tables ? pt_stride : 0;
  p.row_to_batch = row_to_batch;
  p.page_size = page_tables ? page_size : 1;
  p.out_slots = out_slots;
  p.out_idx = out_indices;
  p.block_size = out_blocks ? block_size : 1;
  p.out_blocks = out_blocks;
  p.out_counts = out_counts;
  p.chunks = plan.chunks;
  p.chunk_len = plan.chunk_len;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (have_ws) {
    p.work = static_cast<int*>(workspace);
    cudaError_t e = cudaMemsetAsync(p.work, 0, sizeof(int), cs);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (plan.chunks > 1) {
    const size_t units = static_cast<size_t>(rows) * plan.chunks;
    char* w = static_cast<char*>(workspace) + sai::kTopkWorkHeader;
    p.part_key = reinterpret_cast<uint32_t*>(w);
    p.part_idx = reinterpret_cast<int32_t*>(w + units * SAI_TOPK * 4);
    p.part_cnt = reinterpret_cast<int*>(w + units * SAI_TOPK * 8);
  }
  p.status = st;
  return cuda_status(sai::launch_topk_transform(p, sms, cs));
}

}  // extern "C"

namespace {

// Shared argument checks of the fused-score entry points. The FP8 cache needs
// its per-key scales; a bf16 cache may have none (kscale null = scale 1).
int check_fused_args(const void* q, const float* w, const void* kcache, const float* kscale, bool bf16,
                     int64_t num_blocks, const int32_t* block_table, int64_t bt_rows, int64_t bt_stride,
                     const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows, int32_t heads,
                     int32_t dim, int32_t block_size, int32_t max_seq_len, int32_t group_rows) {
  if (rows < 0 || max_seq_len < 0 || num_blocks < 0 || bt_rows < 0 || bt_stride < 0) return SAI_ERR_SHAPE;
  if (heads != 64 || dim != 128 || block_size != 128) return SAI_ERR_UNSUPPORTED;
  if (group_rows != 1 && group_rows != 4) return SAI_ERR_UNSUPPORTED;
  if (rows == 0) return SAI_OK;
  if (!q || !w || !kcache || (!kscale && !bf16) || !block_table || !seq_lens) return SAI_ERR_NULL;
  if (num_blocks < 1 || bt_rows < 1 || bt_stride < 1) return SAI_ERR_SHAPE;
  if (num_blocks * 128 > INT_MAX || rows * 64 > INT_MAX || rows > INT_MAX / 16) return SAI_ERR_SHAPE;
  if (!row_to_batch && bt_rows < rows) return SAI_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(kcache, 16) || !aligned(w, 16) || (kscale && !aligned(kscale, 4)) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || (row_to_batch && !aligned(row_to_batch, 4)))
    return SAI_ERR_ALIGN;
  return SAI_OK;
}

sai::FusedLaunch fused_launch(const void* q, const float* w, const float* kscale, int64_t num_blocks,
                              const int32_t* block_table, int64_t bt_rows, int64_t bt_stride,
                              const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows,
                              int32_t max_seq_len, const sai::FusedPlan& plan, int* st) {
  sai::FusedLaunch p{};
  p.stall_unit = -1;
  p.q = q;
  p.w = w;
  p.kscale = kscale;
  p.num_blocks = num_blocks;
  p.block_table = block_table;
  p.bt_rows = bt_rows;
  p.bt_stride = bt_stride;
  p.row_to_batch = row_to_batch;
  p.seq_lens = seq_lens;
  p.rows = static_cast<int>(rows);
  p.max_len = max_seq_len;
  p.chunks = plan.chunks;
  p.chunk_blocks = plan.chunk_blocks;
  p.status = st;
  return p;
}

int fused_topk(const void* q, const float* w, const void* kcache, const float* kscale, bool bf16, int64_t num_blocks,
               const int32_t* block_table, int64_t bt_rows, int64_t bt_stride, const int32_t* row_to_batch,
               const int32_t* seq_lens, int64_t rows, int32_t heads, int32_t dim, int32_t block_size,
               int32_t max_seq_len, int32_t group_rows, int32_t k, int32_t* out_slots, int32_t* out_indices,
               float* out_scores, int32_t list_block_size, int32_t* out_blocks, int32_t* out_counts,
               void* workspace, size_t workspace_bytes, sai_stream_t stream) {
  if (k <= 0) return SAI_ERR_SHAPE;
  if (k != SAI_TOPK) return SAI_ERR_UNSUPPORTED;
  if (!out_slots && !out_indices && !out_scores && !out_blocks) return SAI_ERR_NULL;
  if (out_counts && !out_blocks) return SAI_ERR_NULL;
  if (out_blocks && list_block_size < 1) return SAI_ERR_SHAPE;
  int st_arg = check_fused_args(q, w, kcache, kscale, bf16, num_blocks, block_table, bt_rows, bt_stride,
                                row_to_batch, seq_lens, rows, heads, dim, block_size, max_seq_len, group_rows);
  if (st_arg != SAI_OK || rows == 0) return st_arg;
  if ((out_slots && !aligned(out_slots, 4)) || (out_indices && !aligned(out_indices, 4)) ||
      (out_scores && !aligned(out_scores, 4)) || (out_blocks && !aligned(out_blocks, 4)) ||
      (out_counts && !aligned(out_counts, 4)))
    return SAI_ERR_ALIGN;
  int dev, sms;
  int* st;
  if (!device_setup(&dev, &st, &sms)) return SAI_ERR_CUDA;
  const sai::FusedPlan plan = sai::fused_plan(rows, max_seq_len, group_rows, sms);
  if (!workspace || workspace_bytes < plan.workspace_bytes || !aligned(workspace, 16)) return SAI_ERR_WORKSPACE;
  const size_t units = static_cast<size_t>(rows) * plan.chunks;
  char* ws = static_cast<char*>(workspace);
  sai::FusedLaunch p = fused_launch(q, w, kscale, num_blocks, block_table, bt_rows, bt_stride, row_to_batch,
                                    seq_lens, rows, max_seq_len, plan, st);
  p.part_key = reinterpret_cast<uint32_t*>(ws);
  p.part_idx = reinterpret_cast<int32_t*>(ws + units * SAI_TOPK * 4);
  p.part_cnt = reinterpret_cast<int*>(ws + units * SAI_TOPK * 8);
  p.stall_unit = t_stall_unit;
  t_stall_unit = -1;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = sai::launch_fused(p, plan.group, sai::FusedOut::kTopk, bf16, kcache, s);
  if (e != cudaSuccess) return cuda_status(e);
  sai::MergeLaunch m{};
  m.rows = static_cast<int>(rows);
  m.units_per_row = plan.chunks;
  m.part_key = p.part_key;
  m.part_idx = p.part_idx;
  m.part_cnt = p.part_cnt;
  m.seq_lens = seq_lens;
  m.page_tables = block_table;
  m.pt_rows = bt_rows;
  m.pt_stride = bt_stride;
  m.row_to_batch = row_to_batch;
  m.page_size = 128;
  m.out_slots = out_slots;
  m.out_idx = out_indices;
  m.out_scores = out_scores;
  m.status = st;
  m.block_size = out_blocks ? list_block_size : 1;
  m.out_blocks = out_blocks;
  m.out_counts = out_counts;
  return cuda_status(sai::launch_merge(m, s));
}

int fused_dense(const void* q, const float* w, const void* kcache, const float* kscale, bool bf16, int64_t num_blocks,
                const int32_t* block_table, int64_t bt_rows, int64_t bt_stride, const int32_t* row_to_batch,
                const int32_t* seq_lens, int64_t rows, int32_t heads, int32_t dim, int32_t block_size,
                int32_t max_seq_len, int32_t group_rows, float* out_scores, int64_t out_stride, sai_stream_t stream) {
  int st_arg = check_fused_args(q, w, kcache, kscale, bf16, num_blocks, block_table, bt_rows, bt_stride,
                                row_to_batch, seq_lens, rows, heads, dim, block_size, max_seq_len, group_rows);
  if (st_arg != SAI_OK || rows == 0) return st_arg;
  if (!out_scores) return SAI_ERR_NULL;
  if (out_stride < max_seq_len) return SAI_ERR_SHAPE;
  if (!aligned(out_scores, 4)) return SAI_ERR_ALIGN;
  int dev, sms;
  int* st;
  if (!device_setup(&dev, &st, &sms)) return SAI_ERR_CUDA;
  const sai::FusedPlan plan = sai::fused_plan(rows, max_seq_len, group_rows, sms);
  sai::FusedLaunch p = fused_launch(q, w, kscale, num_blocks, block_table, bt_rows, bt_stride, row_to_batch,
                                    seq_lens, rows, max_seq_len, plan, st);
  p.dense = out_scores;
  p.dense_stride = out_stride;
  return cuda_status(
      sai::launch_fused(p, plan.group, sai::FusedOut::kDense, bf16, kcache, reinterpret_cast<cudaStream_t>(stream)));
}

// Per-head top-k workspace: dense per-head scores [rows * 64, stride], the
// per-(row, head) lengths and block-table rows, then the top-k workspace.
struct PerHeadLayout {
  long long stride;
  size_t lens_off, batch_off, topk_off, topk_bytes, total;
};

bool per_head_layout(int64_t rows, int32_t max_seq_len, int sms, PerHeadLayout* L) {
  if (rows <= 0 || max_seq_len < 0 || rows > INT_MAX / (16 * 64)) return false;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const long long hr = rows * 64;
  L->stride = std::max<long long>(4, (static_cast<long long>(max_seq_len) + 3) / 4 * 4);
  const size_t dense = static_cast<size_t>(hr) * L->stride * sizeof(float);
  L->lens_off = up(dense);
  L->batch_off = L->lens_off + up(static_cast<size_t>(hr) * 4);
  L->topk_off = L->batch_off + up(static_cast<size_t>(hr) * 4);
  L->topk_bytes = sai::topk_plan(hr, L->stride, sms).workspace_bytes;
  L->total = L->topk_off + up(std::max<size_t>(L->topk_bytes, 256));
  return true;
}

int fused_per_head_dense(const void* q, const float* w, const void* kcache, const float* kscale, bool bf16,
                         int64_t num_blocks, const int32_t* block_table, int64_t bt_rows, int64_t bt_stride,
                         const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows, int32_t heads,
                         int32_t dim, int32_t block_size, int32_t max_seq_len, float* out_scores, int64_t out_stride,
                         sai_stream_t stream) {
  int st_arg = check_fused_args(q, w, kcache, kscale, bf16, num_blocks, block_table, bt_rows, bt_stride,
                                row_to_batch, seq_lens, rows, heads, dim, block_size, max_seq_len, 1);
  if (st_arg != SAI_OK || rows == 0) return st_arg;
  if (!out_scores) return SAI_ERR_NULL;
  if (out_stride < max_seq_len) return SAI_ERR_SHAPE;
  if (!aligned(out_scores, 4)) return SAI_ERR_ALIGN;
  int dev, sms;
  int* st;
  if (!device_setup(&dev, &st, &sms)) return SAI_ERR_CUDA;
  const sai::FusedPlan plan = sai::fused_plan(rows, max_seq_len, 1, sms);
  sai::FusedLaunch p = fused_launch(q, w, kscale, num_blocks, block_table, bt_rows, bt_stride, row_to_batch,
                                    seq_lens, rows, max_seq_len, plan, st);
  p.dense = out_scores;
  p.dense_stride = out_stride;
  return cuda_status(
      sai::launch_fused(p, plan.group, sai::FusedOut::kPerHead, bf16, kcache, reinterpret_cast<cudaStream_t>(stream)));
}

int fused_per_head_topk(const void* q, const float* w, const void* kcache, const float* kscale, bool bf16,
                        int64_t num_blocks, const int32_t* block_table, int64_t bt_rows, int64_t bt_stride,
                        const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows, int32_t heads,
                        int32_t dim, int32_t block_size, int32_t max_seq_len, int32_t k, int32_t* out_slots,
                        int32_t* out_indices, void* workspace, size_t workspace_bytes, sai_stream_t stream) {
  if (k <= 0) return SAI_ERR_SHAPE;
  if (k != SAI_TOPK) return SAI_ERR_UNSUPPORTED;
  if (!out_slots && !out_indices) return SAI_ERR_NULL;
  int st_arg = check_fused_args(q, w, kcache, kscale, bf16, num_blocks, block_table, bt_rows, bt_stride,
                                row_to_batch, seq_lens, rows, heads, dim, block_size, max_seq_len, 1);
  if (st_arg != SAI_OK || rows == 0) return st_arg;
  if ((out_slots && !aligned(out_slots, 4)) || (out_indices && !aligned(out_indices, 4))) return SAI_ERR_ALIGN;
  int dev, sms;
  int* st;
  if (!device_setup(&dev, &st, &sms)) return SAI_ERR_CUDA;
  PerHeadLayout L;
  if (!per_head_layout(rows, max_seq_len, sms, &L)) return SAI_ERR_SHAPE;
  if (!workspace || workspace_bytes < L.total || !aligned(workspace, 256)) return SAI_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  float* dense = reinterpret_cast<float*>(ws);
  int* lens = reinterpret_cast<int*>(ws + L.lens_off);
  int* batch = reinterpret_cast<int*>(ws + L.batch_off);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = sai::launch_per_head_expand(seq_lens, row_to_batch, static_cast<int>(rows), max_seq_len, bt_rows,
                                              bt_stride, lens, batch, s);
  if (e != cudaSuccess) return cuda_status(e);
  const sai::FusedPlan plan = sai::fused_plan(rows, max_seq_len, 1, sms);
  sai::FusedLaunch p = fused_launch(q, w, kscale, num_blocks, block_table, bt_rows, bt_stride, row_to_batch,
                                    seq_lens, rows, max_seq_len, plan, st);
  p.dense = dense;
  p.dense_stride = L.stride;
  // a positive factor per (row, head) does not change that row's selection;
  // without |w_h| the score rows have comparable scales, which the top-k
  // kernel's threshold carried from row to row relies on
  p.sign_w = 1;
  e = sai::launch_fused(p, plan.group, sai::FusedOut::kPerHead, bf16, kcache, s);
  if (e != cudaSuccess) return cuda_status(e);
  return sai_topk_transform(dense, rows * 64, L.stride, nullptr, lens, block_table, bt_rows, bt_stride, batch, 128,
                            SAI_TOPK, out_slots, out_indices, 0, nullptr, nullptr, ws + L.topk_off, L.topk_bytes,
                            stream);
}

}  // namespace

extern "C" {

size_t sai_index_score_topk_workspace(int64_t rows, int32_t max_seq_len, int32_t group_rows, int32_t k) {
  if (rows <= 0 || max_seq_len < 0 || k != SAI_TOPK || (group_rows != 1 && group_rows != 4)) return 0;
  int dev, sms;
  int* st;
  if (!device_setup(&dev, &st, &sms)) return 0;
  return sai::fused_plan(rows, max_seq_len, group_rows, sms).workspace_bytes;
}

int sai_index_score_topk(const uint8_t* q_fp8, const float* w, const uint8_t* kcache_fp8, const float* kscale,
                         int64_t num_blocks, const int32_t* block_table, int64_t bt_rows, int64_t bt_stride,
                         const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows, int32_t heads,
                         int32_t dim, int32_t block_size, int32_t max_seq_len, int32_t group_rows, int32_t k,
                         int32_t* out_slots, int32_t* out_indices, float* out_scores, int32_t list_block_size,
                         int32_t* out_blocks, int32_t* out_counts, void* workspace, size_t workspace_bytes,
                         sai_stream_t stream) {
  return fused_topk(q_fp8, w, kcache_fp8, kscale, false, num_blocks, block_table, bt_rows, bt_stride, row_to_batch,
                    seq_lens, rows, heads, dim, block_size, max_seq_len, group_rows, k, out_slots, out_indices,
                    out_scores, list_block_size, out_blocks, out_counts, workspace, workspace_bytes, stream);
}

int sai_index_score_topk_bf16(const uint16_t* q_bf16, const float* w, const uint16_t* kcache_bf16,
                              const float* kscale, int64_t num_blocks, const int32_t* block_table, int64_t bt_rows,
                              int64_t bt_stride, const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows,
                              int32_t heads, int32_t dim, int32_t block_size, int32_t max_seq_len, int32_t group_rows,
                              int32_t k, int32_t* out_slots, int32_t* out_indices, float* out_scores,
                              int32_t list_block_size, int32_t* out_blocks, int32_t* out_counts, void* workspace,
                              size_t workspace_bytes, sai_stream_t stream) {
  return fused_topk(q_bf16, w, kcache_bf16, kscale, true, num_blocks, block_table, bt_rows, bt_stride, row_to_batch,
                    seq_lens, rows, heads, dim, block_size, max_seq_len, group_rows, k, out_slots, out_indices,
                    out_scores, list_block_size, out_blocks, out_counts, workspace, workspace_bytes, stream);
}

int sai_index_score(const uint8_t* q_fp8, const float* w, const uint8_t* kcache_fp8, const float* kscale,
                    int64_t num_blocks, const int32_t* block_table, int64_t bt_rows, int64_t bt_stride,
                    const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows, int32_t heads, int32_t dim,
                    int32_t block_size, int32_t max_seq_len, int32_t group_rows, float* out_scores,
                    int64_t out_stride, sai_stream_t stream) {
  return fused_dense(q_fp8, w, kcache_fp8, kscale, false, num_blocks, block_table, bt_rows, bt_stride, row_to_batch,
                     seq_lens, rows, heads, dim, block_size, max_seq_len, group_rows, out_scores, out_stride, stream);
}

int sai_index_score_bf16(const uint16_t* q_bf16, const float* w, const uint16_t* kcache_bf16, const float* kscale,
                         int64_t num_blocks, const int32_t* block_table, int64_t bt_rows, int64_t bt_stride,
                         const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows, int32_t heads,
                         int32_t dim, int32_t block_size, int32_t max_seq_len, int32_t group_rows, float* out_scores,
                         int64_t out_stride, sai_stream_t stream) {
  return fused_dense(q_bf16, w, kcache_bf16, kscale, true, num_blocks, block_table, bt_rows, bt_stride, row_to_batch,
                     seq_lens, rows, heads, dim, block_size, max_seq_len, group_rows, out_scores, out_stride, stream);
}

size_t sai_index_score_topk_per_head_workspace(int64_t rows, int32_t max_seq_len, int32_t k) {
  if (k != SAI_TOPK || rows <= 0 || max_seq_len < 0) return 0;
  int dev, sms;
  int* st;
  if (!device_setup(&dev, &st, &sms)) return 0;
  PerHeadLayout L;
  return per_head_layout(rows, max_seq_len, sms, &L) ? L.total : 0;
}

int sai_index_score_per_head(const uint8_t* q_fp8, const float* w, const uint8_t* kcache_fp8, const float* kscale,
                             int64_t num_blocks, const int32_t* block_table, int64_t bt_rows, int64_t bt_stride,
                             const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows, int32_t heads,
                             int32_t dim, int32_t block_size, int32_t max_seq_len, float* out_scores,
                             int64_t out_stride, sai_stream_t stream) {
  return fused_per_head_dense(q_fp8, w, kcache_fp8, kscale, false, num_blocks, block_table, bt_rows, bt_stride,
                              row_to_batch, seq_lens, rows, heads, dim, block_size, max_seq_len, out_scores,
                              out_stride, stream);
}

int sai_index_score_per_head_bf16(const uint16_t* q_bf16, const float* w, const uint16_t* kcache_bf16,
                                  const float* kscale, int64_t num_blocks, const int32_t* block_table,
                                  int64_t bt_rows, int64_t bt_stride, const int32_t* row_to_batch,
                                  const int32_t* seq_lens, int64_t rows, int32_t heads, int32_t dim,
                                  int32_t block_size, int32_t max_seq_len, float* out_scores, int64_t out_stride,
                                  sai_stream_t stream) {
  return fused_per_head_dense(q_bf16, w, kcache_bf16, kscale, true, num_blocks, block_table, bt_rows, bt_stride,
                              row_to_batch, seq_lens, rows, heads, dim, block_size, max_seq_len, out_scores,
                              out_stride, stream);
}

int sai_index_score_topk_per_head(const uint8_t* q_fp8, const float* w, const uint8_t* kcache_fp8,
                                  const float* kscale, int64_t num_blocks, const int32_t* block_table,
                                  int64_t bt_rows, int64_t bt_stride, const int32_t* row_to_batch,
                                  const int32_t* seq_lens, int64_t rows, int32_t heads, int32_t dim,
                                  int32_t block_size, int32_t max_seq_len, int32_t k, int32_t* out_slots,
                                  int32_t* out_indices, void* workspace, size_t workspace_bytes,
                                  sai_stream_t stream) {
  return fused_per_head_topk(q_fp8, w, kcache_fp8, kscale, false, num_blocks, block_table, bt_rows, bt_stride,
                             row_to_batch, seq_lens, rows, heads, dim, block_size, max_seq_len, k, out_slots,
                             out_indices, workspace, workspace_bytes, stream);
}

int sai_index_score_topk_per_head_bf16(const uint16_t* q_bf16, const float* w, const uint16_t* kcache_bf16,
                                       const float* kscale, int64_t num_blocks, const int32_t* block_table,
                                       int64_t bt_rows, int64_t bt_stride, const int32_t* row_to_batch,
                                       const int32_t* seq_lens, int64_t rows, int32_t heads, int32_t dim,
                                       int32_t block_size, int32_t max_seq_len, int32_t k, int32_t* out_slots,
                                       int32_t* out_indices, void* workspace, size_t workspace_bytes,
                                       sai_stream_t stream) {
  return fused_per_head_topk(q_bf16, w, kcache_bf16, kscale, true, num_blocks, block_table, bt_rows, bt_stride,
                             row_to_batch, seq_lens, rows, heads, dim, block_size, max_seq_len, k, out_slots,
                             out_indices, workspace, workspace_bytes, stream);
}

int sai_sparse_blocks(const int32_t* slots, int64_t rows, int32_t k, int32_t block_size, int32_t* out_blocks,
                      int32_t* out_counts, sai_stream_t stream) {
  if (rows < 0 || k < 1 || k > SAI_TOPK || block_size < 1 || rows > INT_MAX / SAI_TOPK) return SAI_ERR_SHAPE;
  if (rows == 0) return SAI_OK;
  if (!slots || !out_blocks) return SAI_ERR_NULL;
  if (!aligned(slots, 4) || !aligned(out_blocks, 4) || (out_counts && !aligned(out_counts, 4))) return SAI_ERR_ALIGN;
  int dev, sms;
  int* st;
  if (!device_setup(&dev, &st, &sms)) return SAI_ERR_CUDA;
  return cuda_status(sai::launch_sparse_blocks(slots, static_cast<int>(rows), k, block_size, out_blocks, out_counts,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
