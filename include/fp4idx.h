/*
 * fp4idx.h -- C ABI of the GB300 FP4 indexer library (libfp4idx.so).
 *
 * The DeepSeek-V4 sparse-attention indexer, as described on three SGLang pull
 * request pages:
 *   [P1] "dsv4.1-amd: KV cache layouts, FP4 indexer, compressor and router kernels"
 *   [P2] "[AMD] Enable FP4 indexer for Deepseek V4"
 *   [P3] "[AMD] DeepSeek-V4.1-Flash on MI350X (gfx950)"
 * Write side: each compressed bf16 index-K row of 128 goes through RMSNorm, RoPE
 * (dims 0..63), a 128-point Hadamard rotation and e2m1 quantisation with one
 * UE8M0 scale per 32 elements, into a paged cache split into a 64-byte payload
 * tensor and a 4-byte scale tensor.  Read side: paged-MQA logits
 *   logits[t,s] = sum_h w[t,h] * ReLU(q_fp4[t,h] . k_fp4[s]),  s < context_lens[t],
 * then a per-row top-k of compressed-token indices, ascending.
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers (cudaMalloc / torch CUDA memory on the current
 *     device) unless marked "host".  Arrays are dense, row-major, 16-byte aligned.
 *   - bf16 values are passed as uint16_t bit patterns.
 *   - Ownership stays with the caller.  The library never allocates, frees or
 *     synchronises; every call only enqueues kernels on `stream` (a cudaStream_t,
 *     NULL = the legacy default stream) and returns.  Calls are safe inside CUDA
 *     graph capture.
 *   - Return value: FP4IDX_OK, or an fp4idx_status for a problem the host can see
 *     (null pointer, bad size, misalignment, unsupported shape, too small a
 *     workspace, a failed launch).  Nothing is enqueued when a call fails.
 *   - status_dev (nullable, one int32 in device memory, zero it before use): the
 *     kernels record the first data-dependent error they meet (a page id outside
 *     [0, num_pages), a slot past the cache, a position outside the RoPE table, a
 *     context length above the stated maximum, a pipeline wait that ran out).
 *     They skip the offending access and never trap.
 *   - Fixed shapes: head_dim 128, 64 indexer heads, 64 tokens per cache page.
 *   - Devices: calls run on the current device.  The first call of a kernel on each
 *     device sets that kernel's shared-memory size attribute there (once per device,
 *     thread-safe), so make the first call of each entry point on a device outside
 *     stream capture.
 *
 * Cache layout (split, [P2] Motivation): per physical page p and token j < 64,
 *   payload[p][c][j][0..15]  (uint8, [num_pages,4,64,16]; 64 B per token)
 *   scale  [p][c][j]         (uint8, [num_pages,4,64];    4 B per token)
 * c = 32-element block (element 32c+2b in the low nibble of byte b, 32c+2b+1 in
 * the high nibble), scale byte = e + 127 where the block is e2m1(x * 2^-e).
 * Slot of token j on page p: p*64 + j.
 * Query layout (this library's own, shaped like one K page with heads in place
 * of tokens): q_payload[t][c][h][0..15] ([T,4,64,16]), q_scale[t][c][h] ([T,4,64]).
 */
#ifndef FP4IDX_H
#define FP4IDX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP4IDX_HEAD_DIM 128
#define FP4IDX_NUM_HEADS 64
#define FP4IDX_PAGE_TOKENS 64
#define FP4IDX_FP8_PAGE_BYTES (64 * 128 + 64 * 4)
#define FP4IDX_MAX_TOPK 4096
#define FP4IDX_MAX_CONTEXT 65536
#define FP4IDX_MAX_HIDDEN 16384 /* hidden size limit of fp4idx_quant_q_w */
#define FP4IDX_TOPK_NOALLOC_MAX_BYTES (16u * 1024u * 1024u) /* fixed scratch of fp4idx_topk_noalloc */

typedef enum {
  FP4IDX_OK = 0,
  FP4IDX_ERR_INVALID_ARG = 1,  /* null pointer, negative size, misaligned pointer, k out of range */
  FP4IDX_ERR_UNSUPPORTED = 2,  /* a shape the kernels do not implement (heads != 64, ...) */
  FP4IDX_ERR_CUDA = 3,         /* a CUDA launch or attribute call failed */
  FP4IDX_ERR_WORKSPACE = 4,    /* schedule/workspace buffer smaller than the size query says */
  FP4IDX_ERR_BAD_PAGE = 5,     /* device: page id / slot outside the cache */
  FP4IDX_ERR_TIMEOUT = 6,      /* device: a pipeline wait exceeded its iteration limit */
  FP4IDX_ERR_BAD_POSITION = 7, /* device: RoPE position outside [0, max_pos) */
  FP4IDX_ERR_BAD_LENGTH = 8,   /* device: context length < 0 or above max_context / page-table width */
  FP4IDX_ERR_SCHEDULE = 9,     /* schedule built for another row count or grid, or its selection
                                  counters were left non-zero by a call that failed: rebuild it */
  FP4IDX_ERR_SCRATCH_LIMIT = 10 /* fp4idx_topk_noalloc: the call needs more than its fixed scratch */
} fp4idx_status;

/* Human-readable name of a status code (static string). */
const char* fp4idx_status_string(int status);

/* Number of SMs of the current device (host out-pointer). */
int fp4idx_num_sms(int32_t* num_sms_out);

/*
 * K store -- the fused writer of [P2] Modifications / FP4 kernel adapters
 * ("fused RMSNorm, RoPE, Hadamard, FP4 quantization, and paged cache writes")
 * into the split layout of [P2] Motivation; round-to-nearest-even per [P1] Summary.
 *   k          [n_rows,128] bf16   compressed index-K rows
 *   positions  [n_rows] int32      RoPE position of each row, in [0, max_pos)
 *   slots      [n_rows] int32      destination slot page*64+j; slot < 0 = padding, skipped
 *   norm_w     [128] bf16          RMSNorm weight ([P2] compressor.py BF16 mirror)
 *   eps                            RMSNorm epsilon (1e-6 for DeepSeek-V4)
 *   cos_sin    [max_pos,64] bf16   row p: cos(p f_i) for i<32, then sin(p f_i)
 *   payload    [num_pages,4,64,16] uint8, scale [num_pages,4,64] uint8 (written)
 * Device errors: BAD_PAGE (slot >= num_pages*64), BAD_POSITION; the row is skipped.
 */
int fp4idx_store_k(const uint16_t* k, int64_t n_rows, const int32_t* positions, const int32_t* slots,
                   const uint16_t* norm_w, float eps, const uint16_t* cos_sin, int32_t max_pos,
                   uint8_t* payload, uint8_t* scale, int64_t num_pages, int32_t* status_dev, void* stream);

/*
 * K store into the FP8 "fused" indexer layout, 132 bytes per token ([P2] Device
 * memory and sizing: the FP8 footprint the FP4 entry replaces).  Same chain up to
 * the Hadamard, then one fp32 scale per token s = amax/448 (1 if amax = 0) and
 * e4m3 = RNE-satfinite(x / s).  Page layout (fp8_pages, [num_pages, 8448] uint8):
 * bytes [j*128, j*128+128) = token j's e4m3 values, bytes [8192 + 4j, 8192 + 4j + 4)
 * = its fp32 scale.  Arguments and errors as fp4idx_store_k.
 */
int fp4idx_store_k_fp8(const uint16_t* k, int64_t n_rows, const int32_t* positions, const int32_t* slots,
                       const uint16_t* norm_w, float eps, const uint16_t* cos_sin, int32_t max_pos,
                       uint8_t* fp8_pages, int64_t num_pages, int32_t* status_dev, void* stream);

/*
 * Q quant -- [P2] Modifications / fp4_indexer_hip.py "Q RoPE/Hadamard/FP4
 * quantization" and [P1] Summary's query packer: RoPE at q_positions[t], Hadamard,
 * e2m1 + UE8M0/32.  No RMSNorm on the query side.
 *   q [n_rows, n_heads, 128] bf16;  q_positions [n_rows] int32
 *   q_payload [n_rows,4,64,16] uint8, q_scale [n_rows,4,64] uint8 (written)
 * n_heads must be 64 (UNSUPPORTED otherwise).  Device error: BAD_POSITION.
 */
int fp4idx_quant_q(const uint16_t* q, int64_t n_rows, int32_t n_heads, const int32_t* q_positions,
                   const uint16_t* cos_sin, int32_t max_pos, uint8_t* q_payload, uint8_t* q_scale,
                   int32_t* status_dev, void* stream);

/*
 * FP8 query pack -- the query side of the FP8 comparison path ([P2] Device memory and
 * sizing: the 132 B/token FP8 entry the FP4 entry replaces).  RoPE and the Hadamard as in
 * fp4idx_quant_q, then the K side's FP8 rule per (row, head): s = amax/448 (1 if amax = 0),
 * e4m3 = RNE-satfinite(x / s).  The pages give only the K entry; this rule for the query is
 * a reading.
 *   q8 [n_rows,8,64,16] uint8: q8[t][c][h][i] = element 16c + i of head h (written)
 *   q8_scale [n_rows,64] fp32 (written)
 * n_heads must be 64.  Device error: BAD_POSITION.
 */
int fp4idx_quant_q_fp8(const uint16_t* q, int64_t n_rows, int32_t n_heads, const int32_t* q_positions,
                       const uint16_t* cos_sin, int32_t max_pos, uint8_t* q8, float* q8_scale, int32_t* status_dev,
                       void* stream);

/*
 * Q quant and head weights in one launch -- [P1] Summary: "a one-launch index-Q pack +
 * head weights", where indexer_head_weights runs a batch-invariant split-K bf16 GEMV whose
 * result stays in fp32.  The queries are packed exactly as fp4idx_quant_q packs them
 * (same arguments, same bytes); beside them
 *   w_out[t][h] = w_scale * sum_d hidden[t][d] * w_proj[h][d]      (fp32, [n_rows, 64])
 *   hidden [n_rows, hidden_dim] bf16; w_proj [64, hidden_dim] bf16 (row h: head h)
 *   hidden_dim a multiple of 256, at most FP4IDX_MAX_HIDDEN (UNSUPPORTED otherwise)
 * The pages give neither the hidden size nor a scale: any constant factor goes into
 * w_scale.  Order of the sum (the same for every batch, so a row's weights do not depend
 * on the rows beside it): the hidden dimension is cut into M = hidden_dim/256 chunks of
 * 256 and the chunks into 8 runs [wM/8, (w+1)M/8); in run w, lane l of 32 adds the products
 * d = 256m + 8l + i, m then i ascending, one fp32 rounding per addition (bf16 products are
 * exact in fp32); then the 32 lane sums pairwise at lane distances 16, 8, 4, 2, 1; then the
 * 8 run sums in run order; then one rounding for w_scale.  A product meets at most
 * 8*ceil(M/8) + 12 <= hidden_dim/256 + 19 roundings, so the result is within
 * (hidden_dim/256 + 20) * 2^-24 * |w_scale| * sum_d |hidden*w_proj| of the exact value.
 */
int fp4idx_quant_q_w(const uint16_t* q, int64_t n_rows, int32_t n_heads, const int32_t* q_positions,
                     const uint16_t* cos_sin, int32_t max_pos, const uint16_t* hidden, int32_t hidden_dim,
                     const uint16_t* w_proj, float w_scale, uint8_t* q_payload, uint8_t* q_scale, float* w_out,
                     int32_t* status_dev, void* stream);

/*
 * Schedule -- the length-balanced split of the logits work over the GPU
 * ([P1] Summary: an in-tree decode schedule whose registers do not grow with the
 * row count; [P2] Attention runtime: schedules built during graph capture and
 * reused across all C4 layers of a forward).  One small device kernel: no host
 * sync, capturable, a pure function of (context_lens, row_seq, n_rows, num_ctas),
 * so a schedule built once serves every layer of the same batch.
 *   context_lens [n_rows] int32  visible compressed tokens of each query row
 *                                (padded rows: 0; prefill rows: floor((p+1)/4))
 *   row_seq      [n_rows] int32  sequence (page-table row) of each query row; rows
 *                                of one sequence that are adjacent share K tiles
 *   num_ctas                     grid the logits kernel will use (0 = SM count)
 *   schedule     device buffer of at least fp4idx_schedule_workspace_bytes(n_rows, num_ctas)
 * Besides the work split, the schedule holds one counter per row that the fused
 * selection of fp4idx_logits_topk_fused counts up and puts back to zero; the build
 * zeroes them.
 */
size_t fp4idx_schedule_workspace_bytes(int64_t max_rows, int32_t num_ctas);
int fp4idx_build_schedule(const int32_t* context_lens, const int32_t* row_seq, int64_t n_rows,
                          int32_t num_ctas, void* schedule, size_t schedule_bytes, void* stream);

/*
 * The decode step's preparation in one launch: the work of fp4idx_build_schedule,
 * fp4idx_store_k and fp4idx_quant_q, with the same arguments and the same results
 * (bit for bit), in one grid -- [P2] Attention runtime (the schedule is built in the
 * captured step) and Modifications (the fused K writer and the Q packer).  One block builds
 * the schedule, the others store the n_new K rows and pack the n_rows query rows; they
 * run side by side, and the whole grid allows the logits launch that follows on the
 * stream (fp4idx_logits_topk, fp4idx_logits) to start its own set-up before the grid ends.
 * Arguments as in the three calls; q_positions, context_lens and row_seq describe the
 * n_rows query rows, k, positions and slots the n_new K rows (n_new may be 0).
 * Device errors: those of the three calls.
 */
int fp4idx_prepare_step(const uint16_t* k, int64_t n_new, const int32_t* positions, const int32_t* slots,
                        const uint16_t* norm_w, float eps, const uint16_t* q, int64_t n_rows, int32_t n_heads,
                        const int32_t* q_positions, const uint16_t* cos_sin, int32_t max_pos, uint8_t* payload,
                        uint8_t* scale, int64_t num_pages, uint8_t* q_payload, uint8_t* q_scale,
                        const int32_t* context_lens, const int32_t* row_seq, int32_t num_ctas, void* schedule,
                        size_t schedule_bytes, int32_t* status_dev, void* stream);

/*
 * Paged-MQA logits + top-k -- [P2] Modifications: "Dispatch decode and prefill
 * FP4 paged-MQA logits" over the split cache through a guarded page table; padded
 * rows keep context length 0 ([P2] Attention runtime); the selection is sorted
 * and ordered by position ([P3] Changes, Historical results).
 *   q_payload/q_scale   output of fp4idx_quant_q for the n_rows rows
 *   w                   [n_rows,64] fp32 head weights
 *   payload/scale       the split K cache, num_pages pages
 *   page_table          [num_seqs, max_pages] int32 physical page of logical page i
 *   row_seq, context_lens  as given to fp4idx_build_schedule (same arrays)
 *   max_context         host-known upper bound of context_lens (<= FP4IDX_MAX_CONTEXT)
 *   k                   1..FP4IDX_MAX_TOPK
 *   schedule            built by fp4idx_build_schedule for these rows (read only here)
 *   workspace           >= fp4idx_logits_workspace_bytes(n_rows, max_context, k) bytes:
 *                       a logits buffer (unused when logits_out is given) and the
 *                       selection's scratch; nothing in it needs to be initialised
 *   topk_idx  [n_rows,k] int32 (written): the k highest-logit token indices of each
 *             row in ascending order; all of them when context_len <= k; -1 pads.
 *   logits_out [n_rows, logits_stride] fp32 (nullable): when given, receives
 *             logits[t,s] for s < context_lens[t] (the rest is not written).
 * Two launches: the logits kernel, then the top-k kernel (one CTA, or a pair of CTAs
 * in a cluster, per row).
 * Device errors: BAD_PAGE (page id out of range: the tile is skipped),
 * BAD_LENGTH, TIMEOUT, SCHEDULE.
 */
size_t fp4idx_logits_workspace_bytes(int64_t max_rows, int32_t max_context, int32_t k);
int fp4idx_logits_topk(const uint8_t* q_payload, const uint8_t* q_scale, const float* w, int64_t n_rows,
                       int32_t n_heads, const uint8_t* payload, const uint8_t* scale, int64_t num_pages,
                       const int32_t* page_table, int64_t num_seqs, int32_t max_pages, const int32_t* row_seq,
                       const int32_t* context_lens, int32_t max_context, int32_t k, const void* schedule,
                       size_t schedule_bytes, void* workspace, size_t workspace_bytes, int32_t* topk_idx,
                       float* logits_out, int64_t logits_stride, int32_t* status_dev, void* stream);

/*
 * fp4idx_logits_topk in one launch ([P3] Changes: "sorted top-k selection"; the
 * selection is folded into the logits kernel).  Same arguments, result and errors, with
 * one difference: `schedule` is written.  When n_rows is at most the device's SM count,
 * the epilogue warps count, per row, the pieces of its logits they have written (a
 * release add on a counter in the schedule); after its own work the CTA of each row --
 * or a pair of CTAs in a cluster, when the grid holds two for every row -- waits for all
 * of the row's pieces (bounded) and selects the row from the logits in L2.  The launch
 * is cooperative (every CTA resident at once).  The counters go back to zero, so calls
 * that share a schedule must be ordered (one stream), and after a call that reported an
 * error the schedule must be built again.  Larger batches run the two launches of
 * fp4idx_logits_topk.  Both give the same selection.  Inside a CUDA graph, where the
 * second launch of fp4idx_logits_topk costs little, that call is the faster of the two on
 * GB300; this one saves the launch where launches are not overlapped.
 */
int fp4idx_logits_topk_fused(const uint8_t* q_payload, const uint8_t* q_scale, const float* w, int64_t n_rows,
                             int32_t n_heads, const uint8_t* payload, const uint8_t* scale, int64_t num_pages,
                             const int32_t* page_table, int64_t num_seqs, int32_t max_pages, const int32_t* row_seq,
                             const int32_t* context_lens, int32_t max_context, int32_t k, void* schedule,
                             size_t schedule_bytes, void* workspace, size_t workspace_bytes, int32_t* topk_idx,
                             float* logits_out, int64_t logits_stride, int32_t* status_dev, void* stream);

/*
 * The two halves of fp4idx_logits_topk, for callers that want the logits themselves or
 * select elsewhere.  fp4idx_logits writes logits_out[t][s] for s < context_lens[t]
 * (logits_stride >= max_context; the rest of each row is not written).  fp4idx_topk
 * selects from such a buffer: topk_idx[t] = the k largest of logits[t][0..L_t), ascending
 * positions, -1 padding; ties at the k-th value go to the lower positions.  Its scratch
 * (per row, the sort keys of the positions past the first 32,768, which do not fit in
 * shared memory; at least 256 bytes even when max_context <= 32768) lives in `workspace`,
 * at least fp4idx_topk_workspace_bytes(n_rows, max_context) bytes, 16-byte aligned;
 * nothing in it needs to be initialised.
 */
int fp4idx_logits(const uint8_t* q_payload, const uint8_t* q_scale, const float* w, int64_t n_rows, int32_t n_heads,
                  const uint8_t* payload, const uint8_t* scale, int64_t num_pages, const int32_t* page_table,
                  int64_t num_seqs, int32_t max_pages, const int32_t* row_seq, const int32_t* context_lens,
                  int32_t max_context, const void* schedule, size_t schedule_bytes, float* logits_out,
                  int64_t logits_stride, int32_t* status_dev, void* stream);
size_t fp4idx_topk_workspace_bytes(int64_t max_rows, int32_t max_context);
int fp4idx_topk(const float* logits, int64_t logits_stride, const int32_t* context_lens, int64_t n_rows,
                int32_t max_context, int32_t k, void* workspace, size_t workspace_bytes, int32_t* topk_idx,
                int32_t* status_dev, void* stream);

/*
 * FP8 logits -- the read side of the FP8 comparison path ([P2] Device memory and sizing:
 * the fused 132 B/token FP8 entry that the 68 B FP4 entry replaces), over the pages of
 * fp4idx_store_k_fp8 and the queries of fp4idx_quant_q_fp8:
 *   logits[t,s] = sum_h w[t,h] * ReLU(q[t,h] . k[s]),  s < context_lens[t],
 * with q = e4m3(q8[t,.,h,.]) * q8_scale[t,h] and k = e4m3(token s's 128 bytes) * its fp32
 * scale.  Tensor-core kernel (e4m3 x e4m3 -> f32); the two scales are applied in fp32
 * after the dot products.
 *   q8 [n_rows,8,64,16] uint8, q8_scale [n_rows,64] fp32, w [n_rows,64] fp32
 *   fp8_pages [num_pages, 8448] uint8 (1 <= num_pages <= INT32_MAX)
 *   page_table, row_seq, context_lens, max_context, schedule: as fp4idx_logits (the same
 *   schedule serves both formats)
 *   logits_out [n_rows, logits_stride] fp32: written for s < context_lens[t], NaN where
 *   the token's page id is out of range; the rest of each row is not written.
 * All pointers 16-byte aligned except page_table, row_seq, context_lens, logits_out and
 * status_dev (4-byte).  Device errors: BAD_PAGE, BAD_LENGTH, TIMEOUT, SCHEDULE.
 */
int fp4idx_logits_fp8(const uint8_t* q8, const float* q8_scale, const float* w, int64_t n_rows, int32_t n_heads,
                      const uint8_t* fp8_pages, int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                      int32_t max_pages, const int32_t* row_seq, const int32_t* context_lens, int32_t max_context,
                      const void* schedule, size_t schedule_bytes, float* logits_out, int64_t logits_stride,
                      int32_t* status_dev, void* stream);

/*
 * FP8 logits + top-k in one call: fp4idx_logits_fp8 into a logits buffer, then the
 * selection of fp4idx_topk.  Workspace, k, topk_idx and logits_out (nullable) as in
 * fp4idx_logits_topk; the other arguments as in fp4idx_logits_fp8.  A token on an
 * out-of-range page has a NaN logit (status BAD_PAGE), and its place in the selection is
 * then unspecified.
 */
int fp4idx_logits_topk_fp8(const uint8_t* q8, const float* q8_scale, const float* w, int64_t n_rows, int32_t n_heads,
                           const uint8_t* fp8_pages, int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                           int32_t max_pages, const int32_t* row_seq, const int32_t* context_lens,
                           int32_t max_context, int32_t k, const void* schedule, size_t schedule_bytes,
                           void* workspace, size_t workspace_bytes, int32_t* topk_idx, float* logits_out,
                           int64_t logits_stride, int32_t* status_dev, void* stream);

/*
 * fp4idx_topk_noalloc -- fp4idx_topk for callers that may not allocate device memory.
 * The pages this library follows have no counterpart: it is an interface addition.
 * A serving runtime that gives all of its memory to its own pool at start-up, or a
 * plug-in host that passes a library only a stream and the call's tensors, cannot hand
 * fp4idx_topk a workspace; this entry point takes none.
 *
 * Same arguments and result as fp4idx_topk, without workspace/workspace_bytes.  The
 * top-k scratch is a fixed array of the library's device code,
 * FP4IDX_TOPK_NOALLOC_MAX_BYTES per device; no call allocates or frees anything
 * itself (but see the set-up below).
 *   - Limit: fp4idx_topk_workspace_bytes(n_rows, max_context) must not exceed
 *     FP4IDX_TOPK_NOALLOC_MAX_BYTES (any row count fits at max_context <= 32768, up to
 *     128 rows at 65536); a larger call returns FP4IDX_ERR_SCRATCH_LIMIT and enqueues
 *     nothing.
 *   - Setup: the first valid call on each device (with that device current) looks up
 *     the array's address once.  Under CUDA's default lazy module loading that is also
 *     when the array's memory is committed on the device, so the first call can fail
 *     for lack of memory and may synchronise: make it at start-up, before a memory pool
 *     reserves the device's memory and before any stream capture begins.  A call with
 *     n_rows = 0 (other pointers may then be null) does the set-up and nothing else.
 *     Argument errors are reported before the set-up is attempted.  The address is
 *     kept for the life of the process; after cudaDeviceReset the entry point must not
 *     be used on that device again.  Of the conventions at the top of this file, the
 *     one on graph capture is not stated for this entry point.
 *   - Nothing in the array needs to start at zero: a call writes every key it
 *     reads back.
 *   - All calls on a device share the array: calls whose kernels may overlap (unordered
 *     streams, concurrent host threads) race on it.  Order them on one stream.
 */
int fp4idx_topk_noalloc(const float* logits, int64_t logits_stride, const int32_t* context_lens, int64_t n_rows,
                        int32_t max_context, int32_t k, int32_t* topk_idx, int32_t* status_dev, void* stream);

/*
 * Whole pages of the split cache -- [P1] Summary (dequantize_k_cache_paged serves the
 * V4.1 layouts) and [P2] Device memory and sizing / HiCache integration (page-row views
 * of the separately allocated payload and scale buffers; FP4 indexer rows move to and
 * from host memory as whole pages, payload and scale as separate regions).
 *   page_ids  [n_pages] int32  pages to process; an id < 0 is padding (skipped, its
 *                              output untouched); an id >= num_pages records BAD_PAGE
 *                              in status_dev and is skipped.
 * fp4idx_dequant_pages: out [n_pages,64,128] fp32 (written), out[i][j][d] = the
 *   e2m1 value of element d of token j of page page_ids[i] times 2^(scale byte - 127),
 *   exact in fp32 (values past the fp32 range, possible only for scale bytes >= 253,
 *   become +-inf).
 * fp4idx_export_pages: rows_payload [n_pages,4096] uint8 and rows_scale [n_pages,256]
 *   uint8 (written) = the payload and scale bytes of page page_ids[i], unchanged: page
 *   rows ready for one host copy each region.
 * fp4idx_import_pages: the reverse, writing page page_ids[i] of payload/scale from row
 *   i.  The ids of one call must be distinct (two rows into one page race).
 * rows_* and out are 16-byte aligned device buffers owned by the caller.
 */
int fp4idx_dequant_pages(const uint8_t* payload, const uint8_t* scale, int64_t num_pages, const int32_t* page_ids,
                         int64_t n_pages, float* out, int32_t* status_dev, void* stream);
int fp4idx_export_pages(const uint8_t* payload, const uint8_t* scale, int64_t num_pages, const int32_t* page_ids,
                        int64_t n_pages, uint8_t* rows_payload, uint8_t* rows_scale, int32_t* status_dev,
                        void* stream);
int fp4idx_import_pages(const uint8_t* rows_payload, const uint8_t* rows_scale, const int32_t* page_ids,
                        int64_t n_pages, uint8_t* payload, uint8_t* scale, int64_t num_pages, int32_t* status_dev,
                        void* stream);

/*
 * Context-parallel top-k -- [P3] the context-parallel runs (one long sequence's
 * compressed tokens sharded over GPUs): each shard scores its own token range and keeps
 * its top-k; the row's selection is the top-k of the gathered (value, index)
 * candidates.  The merge is exact: every token of the row's top-k is in its shard's
 * top-k, ties included (both sides give equal values to the lower position).
 * fp4idx_topk_values: values[t][i] = logits[t][topk_idx[t][i]] (the values of a
 *   selection made by fp4idx_topk on the same buffer); -inf where topk_idx is -1.
 *   n_rows <= 65535.
 * fp4idx_topk_merge: cand_values/cand_idx [n_rows, n_shards, k] fp32/int32: per row and
 *   shard, the shard's selection as GLOBAL positions (ascending, -1 padding at the end)
 *   with their values; shards in ascending position order (every position of shard s
 *   below every position of shard s+1).  topk_idx [n_rows, k] (written): the k largest
 *   candidates of the row, equal values to the lower position, ascending, -1 padding --
 *   the same selection fp4idx_topk makes on the whole row.  n_shards * k <=
 *   FP4IDX_MAX_CONTEXT, n_shards <= 1024, n_rows <= 65535; workspace of at least
 *   fp4idx_topk_merge_workspace_bytes(n_rows, n_shards, k) bytes, 16-byte aligned,
 *   nothing in it needs to be initialised.  Device errors as fp4idx_topk.
 */
size_t fp4idx_topk_merge_workspace_bytes(int64_t max_rows, int32_t n_shards, int32_t k);
int fp4idx_topk_values(const float* logits, int64_t logits_stride, const int32_t* topk_idx, int64_t n_rows, int32_t k,
                       float* values, void* stream);
int fp4idx_topk_merge(const float* cand_values, const int32_t* cand_idx, int64_t n_rows, int32_t n_shards, int32_t k,
                      void* workspace, size_t workspace_bytes, int32_t* topk_idx, int32_t* status_dev, void* stream);

/*
 * Test support for the logits kernels' bounded waits (failure detection), with no
 * counterpart on the pages.  Every wait of a logits pipeline gives up after
 * wait_limit_ns (0 restores the default, 2 s): the CTA then records FP4IDX_ERR_TIMEOUT
 * in status_dev, lets the copies it issued land, frees its tensor memory and returns,
 * and the context stays usable.  idle_producers != 0 tells the producer warps of
 * later logits launches to issue nothing, so that every launch ends in that timeout;
 * a test sets it with a short limit, checks the status, and calls
 * fp4idx_test_pipeline_waits(0, 0) to restore normal operation.  Process-wide; host
 * only (takes effect at the next launch).
 */
int fp4idx_test_pipeline_waits(int32_t idle_producers, int64_t wait_limit_ns);

/* Copy the device status word to *host_out (host pointer).  Synchronises `stream`:
 * a test/diagnostic helper, not for the hot path. */
int fp4idx_read_status(const int32_t* status_dev, int32_t* host_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP4IDX_H */
