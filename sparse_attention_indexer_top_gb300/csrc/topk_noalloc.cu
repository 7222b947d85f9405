// Allocation-free entry point for topk_transform.
//
// Some callers cannot allocate device memory at the point where they need a
// top-k: code running inside a region that forbids allocation (an
// allocator's own callbacks, a memory-pool owner that has handed all its
// memory out, a host thread that must not take the allocator lock), or a
// caller with no allocator at all beyond its fixed input and output
// buffers. sai_topk_transform_noalloc serves them: the split path's partial
// top-k lists live in one fixed array of device memory that this library
// owns, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable of SAI_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits. Its
// name in host code is only a host-side stand-in, so the device address is
// looked up once per device (with that device current) through
// cudaGetSymbolAddress and passed to the kernels as a plain pointer.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/sai.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SAI_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device; nullptr on error.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int sai_topk_transform_noalloc(const float* scores, int64_t rows, int64_t score_stride,
                                          const int32_t* row_starts, const int32_t* seq_lens,
                                          const int32_t* page_tables, int64_t pt_rows, int64_t pt_stride,
                                          const int32_t* row_to_batch, int32_t page_size, int32_t k,
                                          int32_t* out_slots, int32_t* out_indices, sai_stream_t stream) {
  // Scratch these sizes want: the 256-byte header with the row work counter
  // for every valid call (also when each row is one CTA's unit), plus the
  // partial lists when long rows are split; 0 only for invalid arguments,
  // which the call below reports.
  const size_t need = sai_topk_transform_workspace(rows, score_stride, k);
  if (need > SAI_NOALLOC_SCRATCH_BYTES) return SAI_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = scratch_on_current_device();
    if (!scratch) return SAI_ERR_CUDA;
  }
  // Only the work counter has to start at zero, and sai_topk_transform
  // clears it on the stream before its launch; every work unit writes its
  // candidate count and entries before the merge kernel reads them.
  return sai_topk_transform(scores, rows, score_stride, row_starts, seq_lens, page_tables, pt_rows, pt_stride,
                            row_to_batch, page_size, k, out_slots, out_indices, 0, nullptr, nullptr, scratch,
                            scratch ? static_cast<size_t>(SAI_NOALLOC_SCRATCH_BYTES) : 0, stream);
}
