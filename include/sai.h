/*
 * sai.h -- C ABI of libsai, the GB300 (sm_103a) sparse-attention indexer
 * top-k library.
 *
 * Conventions for every entry point
 * ---------------------------------
 * - All array pointers are DEVICE pointers on the calling thread's current
 *   CUDA device, owned by the caller. The library allocates nothing; where
 *   scratch memory helps, the caller passes a workspace sized by the matching
 *   *_workspace query (same arguments, same device).
 * - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *   legacy default stream). No entry point synchronizes, except
 *   sai_device_status.
 * - Host-visible argument errors are reported before anything is launched.
 *   Row metadata that lives on the device (seq_lens, row_starts,
 *   row_to_batch, page/block ids) is checked by the kernels: an out-of-range
 *   row is treated as empty (all -1 outputs) and a bit is set in the
 *   library's device status word, read with sai_device_status. No kernel
 *   ever reads outside the extents the caller declares.
 * - Row-local index order of the k outputs: higher score first, equal scores
 *   to the lower row-local index (-0.0 == +0.0; +-inf are ordinary values;
 *   NaN scores are not admissible). Positions [min(seq_len, k), k) are -1.
 * - No C++ exception crosses this boundary.
 */
#ifndef SAI_H_
#define SAI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so users need no CUDA headers. */
typedef struct CUstream_st* sai_stream_t;

typedef enum {
  SAI_OK = 0,
  SAI_ERR_NULL = -1,        /* a required pointer is NULL */
  SAI_ERR_SHAPE = -2,       /* a size or count is out of range */
  SAI_ERR_UNSUPPORTED = -3, /* valid but not implemented (e.g. k != 512) */
  SAI_ERR_WORKSPACE = -4,   /* workspace too small or misaligned */
  SAI_ERR_CUDA = -5,        /* a CUDA runtime call or launch failed */
  SAI_ERR_DEVICE_CHECK = -6,/* a kernel flagged bad device-side metadata */
  SAI_ERR_ALIGN = -7        /* a pointer lacks the alignment its type needs */
} sai_status;

/* Fixed top-k of this library (the "512" of topk_transform_512_v2). */
#define SAI_TOPK 512

/* Human-readable name of a status code (static storage). */
const char* sai_status_string(int status);

/*
 * Text of the CUDA error behind the calling thread's most recent
 * SAI_ERR_CUDA ("" if none); valid until that thread's next call.
 */
const char* sai_last_error(void);

/*
 * Read (and optionally clear) the device status word of the current device
 * after synchronizing `stream`. *out_bits receives the OR of the bits set by
 * kernels since the last clear: 1 = bad row metadata, 2 = an internal
 * pipeline wait gave up, 4 = a block id out of range. Returns
 * SAI_ERR_DEVICE_CHECK if any bit was set, else SAI_OK.
 */
int sai_device_status(int* out_bits, int clear, sai_stream_t stream);

/*
 * Test hook for the bounded waits (not part of the computation; the paper
 * has no counterpart). Every pipeline wait inside the kernels gives up after
 * about two seconds, sets status bit 2 and lets the launch finish, so a lost
 * arrival can never hang the GPU. To exercise that exit, the next
 * sai_index_score_topk / sai_index_score_topk_bf16 call made by this host
 * thread streams no key tiles for its work unit `unit` (a unit is a group of
 * query rows and a chunk of their KV blocks; unit 0 holds the first rows'
 * first chunk): that unit's waits run out, the call completes with status
 * bit 2 set, and the rows of that unit are undefined. -1 clears the hook;
 * the call consumes it either way.
 */
void sai_test_stall_next_fused(int32_t unit);

/*
 * Workspace bytes that sai_topk_transform wants for these sizes on the
 * current device: a 256-byte header (a work counter that lets CTAs take
 * rows as they finish, zeroed by the call on its stream), plus, when long
 * rows on few rows are split over several CTAs, their partial top-k lists.
 */
size_t sai_topk_transform_workspace(int64_t rows, int64_t score_stride, int32_t k);

/*
 * sai_topk_transform -- per-row window top-k and page-table transform.
 *
 * Follows sglang PR #37889 "[AMD] Enable GLM DSA prefill top-k to the v2
 * kernel" (Modifications: the two optional (rows,) int32 indirections of
 * topk_transform_512_v2) and ROCm/ATOM PR #1282 "merge build sparse block
 * into topk" (the physical addressing is produced by the top-k kernel).
 *
 * For each row i in [0, rows):
 *   n      = seq_lens[i]
 *   start  = row_starts ? row_starts[i] : 0
 *   window = scores[i*score_stride + start + t], t in [0, n)
 *   b      = row_to_batch ? row_to_batch[i] : i
 *   idx[j] = row-local position of the j-th best score (j < min(n, k))
 *   slot[j]= page_tables[b*pt_stride + idx[j]/page_size]*page_size
 *            + idx[j]%page_size
 *
 * scores       fp32 [rows, score_stride], 4-byte aligned; any stride and any
 *              row start work (the 16-byte-aligned interior of each window
 *              is streamed with bulk TMA copies, the ragged ends with scalar
 *              loads).
 * row_starts   int32 [rows] or NULL. The caller guarantees
 *              start + n <= score_stride (checked on device).
 * seq_lens     int32 [rows], >= 0.
 * page_tables  int32 [pt_rows, pt_stride]; required when out_slots or
 *              out_blocks is given.
 *              Without row_to_batch, pt_rows >= rows is checked here; with
 *              it, 0 <= row_to_batch[i] < pt_rows is checked on device.
 * page_size    >= 1 (1 = one slot per token, the "wide" table).
 * k            must be 512 (SAI_ERR_UNSUPPORTED otherwise).
 * out_slots    int32 [rows, 512] or NULL; out_indices int32 [rows, 512] or
 *              NULL (row-local positions).
 * out_blocks   int32 [rows, 512] or NULL: the row's selected slots as the
 *              ascending distinct blocks slot / block_size, -1 padded, built
 *              by the same call from the slots it picks (ROCm/ATOM PR #1282
 *              "merge build sparse block into topk": the block list comes out
 *              of the top-k, not out of a second pass over the slots); needs
 *              page_tables. block_size >= 1 when out_blocks is given (128:
 *              a 128-token KV block; ignored otherwise). out_counts int32
 *              [rows] or NULL: each row's number of blocks (only with
 *              out_blocks). At least one of out_slots, out_indices and
 *              out_blocks must be given.
 * workspace    device memory of workspace_bytes (16-byte aligned) or NULL.
 *              If it is smaller than sai_topk_transform_workspace asks for,
 *              every row is processed by a single CTA (correct, slower for
 *              few long rows); below 256 bytes (or NULL) the CTAs also take
 *              rows in a fixed order instead of from the work counter.
 *              Calls that share a workspace must not overlap on the GPU.
 */
int sai_topk_transform(const float* scores, int64_t rows, int64_t score_stride, const int32_t* row_starts,
                       const int32_t* seq_lens, const int32_t* page_tables, int64_t pt_rows, int64_t pt_stride,
                       const int32_t* row_to_batch, int32_t page_size, int32_t k, int32_t* out_slots,
                       int32_t* out_indices, int32_t block_size, int32_t* out_blocks, int32_t* out_counts,
                       void* workspace, size_t workspace_bytes, sai_stream_t stream);

/*
 * Workspace bytes that sai_index_score_topk needs for these sizes on the
 * current device (the per-(row, KV chunk) candidate lists).
 */
size_t sai_index_score_topk_workspace(int64_t rows, int32_t max_seq_len, int32_t group_rows, int32_t k);

/*
 * sai_index_score_topk -- FP8 index scores and top-k in one pass.
 *
 * Follows ROCm/ATOM PR #1473 "enable minimax m3 fp8 index cache and fuse
 * index_score_kernel with partial_topk kernel" (pull request overview: FP8
 * index cache, the score computed in FP8, index score and partial top-k fused
 * so that no score tensor is written; the fused decode kernel walks the
 * request's block table and masks keys at or beyond the causal length).
 * For each query row i, with b = row_to_batch ? row_to_batch[i] : i and
 * n = seq_lens[i]:
 *   score(t) = kscale[p*128 + o] * sum_h w[i*64 + h] * relu(sum_d q[i,h,d] k[p,o,d])
 *   for t < n, p = block_table[b*bt_stride + t/128], o = t % 128;
 * then the top-k keys by (score desc, index asc):
 *   out_indices[i*512 + j] = t_j, out_slots[...] = p_j*128 + o_j,
 *   out_scores[...] = score(t_j) (fp32), padded with -1 / NaN;
 *   optionally out_blocks[i*512 + j] = the row's ascending distinct
 *   out_slots / list_block_size (-1 padded) and out_counts[i] their number,
 *   as for sai_topk_transform (list_block_size 128 gives the block ids p_j).
 *
 * q_fp8       e4m3fn [rows, heads, dim], 16-byte aligned.
 * w           fp32 [rows, heads].
 * kcache_fp8  e4m3fn [num_blocks, block_size, dim], 16-byte aligned.
 * kscale      fp32 [num_blocks, block_size].
 * block_table int32 [bt_rows, bt_stride]; block ids outside [0, num_blocks)
 *             mask their keys and set status bit 4.
 * seq_lens    int32 [rows], 0 <= n <= max_seq_len and ceil(n/128) <= bt_stride
 *             (checked on device; a bad row is emptied and sets bit 1).
 * heads = 64, dim = 128, block_size = 128, k = 512 (else SAI_ERR_UNSUPPORTED).
 * group_rows  1, or 4 when every 4 consecutive rows share one row_to_batch
 *             value (packed prefill): the kernel then scores the rows in
 *             pairs, each key block once per pair. A pair whose rows differ
 *             is emptied and sets bit 1.
 * out_*       any of out_slots, out_indices, out_scores, out_blocks may be
 *             NULL, not all; out_counts only with out_blocks, which needs
 *             list_block_size >= 1.
 * workspace   at least sai_index_score_topk_workspace(...) bytes, 16-byte aligned.
 */
int sai_index_score_topk(const uint8_t* q_fp8, const float* w, const uint8_t* kcache_fp8, const float* kscale,
                         int64_t num_blocks, const int32_t* block_table, int64_t bt_rows, int64_t bt_stride,
                         const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows, int32_t heads,
                         int32_t dim, int32_t block_size, int32_t max_seq_len, int32_t group_rows, int32_t k,
                         int32_t* out_slots, int32_t* out_indices, float* out_scores, int32_t list_block_size,
                         int32_t* out_blocks, int32_t* out_counts, void* workspace, size_t workspace_bytes,
                         sai_stream_t stream);

/*
 * sai_index_score -- the same FP8 index scores written densely (for tests):
 * out_scores[i*out_stride + t] = score(i, t) for t < seq_lens[i]; other
 * cells are not written. out_stride >= max_seq_len. Same argument rules.
 */
int sai_index_score(const uint8_t* q_fp8, const float* w, const uint8_t* kcache_fp8, const float* kscale,
                    int64_t num_blocks, const int32_t* block_table, int64_t bt_rows, int64_t bt_stride,
                    const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows, int32_t heads, int32_t dim,
                    int32_t block_size, int32_t max_seq_len, int32_t group_rows, float* out_scores,
                    int64_t out_stride, sai_stream_t stream);

/*
 * sai_index_score_topk_bf16 / sai_index_score_bf16 -- the same two calls for
 * a bf16 index cache.
 *
 * The index cache may be kept at the model dtype instead of FP8 (ROCm/ATOM PR
 * #1473: the index-cache type option whose default "auto" is the model dtype,
 * and its commit "convert auto for bf16 type"; FP8 only when the KV cache
 * dtype is an fp8 one). Then q and the keys are bfloat16 bit patterns and the
 * dot products run in bf16 with fp32 accumulation; the score, selection,
 * outputs, workspace (sai_index_score_topk_workspace) and status bits are those
 * of the FP8 calls.
 *
 * q_bf16       bf16 [rows, heads, dim], 16-byte aligned.
 * kcache_bf16  bf16 [num_blocks, block_size, dim], 16-byte aligned.
 * kscale       fp32 [num_blocks, block_size], or NULL: the pages give a bf16
 *              cache no per-key scale, and NULL means scale 1.
 * Other arguments as for sai_index_score_topk / sai_index_score.
 */
int sai_index_score_topk_bf16(const uint16_t* q_bf16, const float* w, const uint16_t* kcache_bf16,
                              const float* kscale, int64_t num_blocks, const int32_t* block_table, int64_t bt_rows,
                              int64_t bt_stride, const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows,
                              int32_t heads, int32_t dim, int32_t block_size, int32_t max_seq_len, int32_t group_rows,
                              int32_t k, int32_t* out_slots, int32_t* out_indices, float* out_scores,
                              int32_t list_block_size, int32_t* out_blocks, int32_t* out_counts, void* workspace,
                              size_t workspace_bytes, sai_stream_t stream);
int sai_index_score_bf16(const uint16_t* q_bf16, const float* w, const uint16_t* kcache_bf16, const float* kscale,
                         int64_t num_blocks, const int32_t* block_table, int64_t bt_rows, int64_t bt_stride,
                         const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows, int32_t heads,
                         int32_t dim, int32_t block_size, int32_t max_seq_len, int32_t group_rows, float* out_scores,
                         int64_t out_stride, sai_stream_t stream);

/*
 * Per-index-head top-k: one selection per (query row, index head).
 *
 * The fused decode kernel of ROCm/ATOM PR #1473 is launched over (query,
 * index head, key chunk) (review diff of index_topk.py), which admits a
 * selection per index head. Head h's score is its summand of the
 * head-summed score:
 *   score_h(t) = kscale[p*128 + o] * w[i*64 + h] * relu(sum_d q[i,h,d] k[p,o,d])
 * (p, o, n, b as for sai_index_score_topk), and each (i, h) takes its top-k
 * keys by (score desc, index asc).
 *
 * sai_index_score_per_head[_bf16] writes the scores densely:
 *   out_scores[(i*64 + h)*out_stride + t] = score_h(t) for t < seq_lens[i]
 * (other cells untouched; a key on a block id outside [0, num_blocks) gets
 * -inf and sets status bit 4). out_stride >= max_seq_len.
 *
 * sai_index_score_topk_per_head[_bf16] computes those scores into its
 * workspace and selects with the top-k kernel:
 *   out_indices[(i*64 + h)*512 + j] = t_j, out_slots[...] = p_j*128 + o_j
 * (-1 padded; either output may be NULL, not both). The workspace holds
 * rows*64 score rows of max_seq_len floats (rounded up to 4) plus metadata:
 * sai_index_score_topk_per_head_workspace(...) bytes, 256-byte aligned
 * (about 17 MB per decode row of 32768 keys).
 *
 * Arguments as for sai_index_score_topk (FP8) / sai_index_score_topk_bf16
 * (bf16, kscale may be NULL), without group_rows (rows are scored one per
 * unit). Same host errors; bad rows are emptied and flagged as there.
 */
size_t sai_index_score_topk_per_head_workspace(int64_t rows, int32_t max_seq_len, int32_t k);
int sai_index_score_per_head(const uint8_t* q_fp8, const float* w, const uint8_t* kcache_fp8, const float* kscale,
                             int64_t num_blocks, const int32_t* block_table, int64_t bt_rows, int64_t bt_stride,
                             const int32_t* row_to_batch, const int32_t* seq_lens, int64_t rows, int32_t heads,
                             int32_t dim, int32_t block_size, int32_t max_seq_len, float* out_scores,
                             int64_t out_stride, sai_stream_t stream);
int sai_index_score_per_head_bf16(const uint16_t* q_bf16, const float* w, const uint16_t* kcache_bf16,
                                  const float* kscale, int64_t num_blocks, const int32_t* block_table,
                                  int64_t bt_rows, int64_t bt_stride, const int32_t* row_to_batch,
                                  const int32_t* seq_lens, int64_t rows, int32_t heads, int32_t dim,
                                  int32_t block_size, int32_t max_seq_len, float* out_scores, int64_t out_stride,
                                  sai_stream_t stream);
int sai_index_score_topk_per_head(const uint8_t* q_fp8, const float* w, const uint8_t* kcache_fp8,
                                  const float* kscale, int64_t num_blocks, const int32_t* block_table,
                                  int64_t bt_rows, int64_t bt_stride, const int32_t* row_to_batch,
                                  const int32_t* seq_lens, int64_t rows, int32_t heads, int32_t dim,
                                  int32_t block_size, int32_t max_seq_len, int32_t k, int32_t* out_slots,
                                  int32_t* out_indices, void* workspace, size_t workspace_bytes,
                                  sai_stream_t stream);
int sai_index_score_topk_per_head_bf16(const uint16_t* q_bf16, const float* w, const uint16_t* kcache_bf16,
                                       const float* kscale, int64_t num_blocks, const int32_t* block_table,
                                       int64_t bt_rows, int64_t bt_stride, const int32_t* row_to_batch,
                                       const int32_t* seq_lens, int64_t rows, int32_t heads, int32_t dim,
                                       int32_t block_size, int32_t max_seq_len, int32_t k, int32_t* out_slots,
                                       int32_t* out_indices, void* workspace, size_t workspace_bytes,
                                       sai_stream_t stream);

/*
 * sai_sparse_blocks -- per-row distinct KV blocks of top-k slots.
 *
 * For callers that already hold slots; the top-k entry points above build
 * the same lists in their last stage when given out_blocks.
 * Follows ROCm/ATOM PR #1282 "merge build sparse block into topk" (title and
 * Motivation): the sparse attention after the indexer reads KV blocks, so
 * each row's selected physical slots (the out_slots of sai_topk_transform
 * or sai_index_score_topk) become the list of distinct blocks they fall in.
 * For each row i:
 *   B_i = ascending distinct values of slots[i*k + j] / block_size over the
 *         j in [0, k) with slots[i*k + j] >= 0 (negative slots are padding)
 *   out_blocks[i*k + t] = B_i[t] for t < |B_i|, -1 for |B_i| <= t < k
 *   out_counts[i] = |B_i|
 *
 * slots       int32 [rows, k], 4-byte aligned; k in [1, 512].
 * block_size  >= 1 (128: the KV block of the fused path; a slot of the
 *             page_size=1 top-k is a token slot, so its block is slot / 128).
 * out_blocks  int32 [rows, k]; out_counts int32 [rows] or NULL.
 * Errors: NULL pointers, k outside [1, 512] or block_size < 1 are reported
 * before anything is launched.
 */
int sai_sparse_blocks(const int32_t* slots, int64_t rows, int32_t k, int32_t block_size, int32_t* out_blocks,
                      int32_t* out_counts, sai_stream_t stream);

/*
 * Size of the library-owned device scratch used by
 * sai_topk_transform_noalloc: 8 MiB, held on every GPU that loads the
 * library until the process exits.
 */
#define SAI_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * sai_topk_transform_noalloc -- sai_topk_transform without a workspace
 * argument, for callers that cannot allocate device memory where they need
 * the top-k (inside an allocator callback or a region that forbids
 * allocation, a pool owner whose memory is all handed out, or code with no
 * allocator beyond its fixed input and output buffers). The paper has no
 * counterpart: this entry point exists only for such callers.
 *
 * Arguments, outputs, ordering and errors are those of sai_topk_transform
 * without the block-list outputs. Instead of a caller workspace, every call
 * uses a fixed library-owned
 * device array of SAI_NOALLOC_SCRATCH_BYTES: its first 256 bytes hold the
 * work counter from which the CTAs take rows (reset to zero by each call on
 * its stream), and the split path for few long rows also keeps its partial
 * top-k lists there. Calls whose sizes need more scratch than that (as
 * reported by sai_topk_transform_workspace) are rejected with
 * SAI_ERR_WORKSPACE before anything is launched. Nothing is allocated: no
 * cudaMalloc, no cudaFree.
 *
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture. All calls
 * on a device share the one array and it keeps the previous call's contents
 * (the counter is the only part that must start at zero, and each call
 * clears it). Any two calls that can overlap on the GPU (different streams
 * without ordering between them), short rows or long, race on the work
 * counter and, when split, on the partial lists: rows can be skipped and
 * outputs left unwritten. The caller must serialize them.
 */
int sai_topk_transform_noalloc(const float* scores, int64_t rows, int64_t score_stride, const int32_t* row_starts,
                               const int32_t* seq_lens, const int32_t* page_tables, int64_t pt_rows,
                               int64_t pt_stride, const int32_t* row_to_batch, int32_t page_size, int32_t k,
                               int32_t* out_slots, int32_t* out_indices, sai_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SAI_H_ */
