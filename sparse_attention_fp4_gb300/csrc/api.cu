// C ABI of libfp4idx.so: argument validation, then kernel launches on the caller's
// stream.  No allocation, no synchronisation (except fp4idx_read_status).
#include <cstdio>

#include "launchers.cuh"
#include "schedule.cuh"

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline int from_cuda(cudaError_t e) { return e == cudaSuccess ? FP4IDX_OK : FP4IDX_ERR_CUDA; }

int device_sms(int32_t* n) { return fp4idx_num_sms(n); }

inline int64_t logits_row_stride(int32_t max_context) { return ((int64_t)max_context + 3) / 4 * 4; }

int check_store_args(const uint16_t* k, int64_t n_rows, const int32_t* positions, const int32_t* slots,
                     const uint16_t* norm_w, const uint16_t* cos_sin, int32_t max_pos, int64_t num_pages) {
  if (n_rows < 0 || num_pages < 0 || max_pos <= 0) return FP4IDX_ERR_INVALID_ARG;
  if (num_pages > (int64_t)INT32_MAX / fp4idx::kPage) return FP4IDX_ERR_UNSUPPORTED;  // slots are int32
  if (n_rows == 0) return FP4IDX_OK;
  if (!k || !positions || !slots || !norm_w || !cos_sin) return FP4IDX_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(norm_w) || !aligned16(cos_sin) || !aligned4(positions) || !aligned4(slots))
    return FP4IDX_ERR_INVALID_ARG;
  return FP4IDX_OK;
}

}  // namespace

extern "C" {

const char* fp4idx_status_string(int status) {
  switch (status) {
    case FP4IDX_OK: return "ok";
    case FP4IDX_ERR_INVALID_ARG: return "invalid argument";
    case FP4IDX_ERR_UNSUPPORTED: return "unsupported shape";
    case FP4IDX_ERR_CUDA: return "CUDA error";
    case FP4IDX_ERR_WORKSPACE: return "workspace too small";
    case FP4IDX_ERR_BAD_PAGE: return "page id or slot outside the cache";
    case FP4IDX_ERR_TIMEOUT: return "pipeline wait timed out";
    case FP4IDX_ERR_BAD_POSITION: return "RoPE position outside the table";
    case FP4IDX_ERR_BAD_LENGTH: return "context length out of range";
    case FP4IDX_ERR_SCHEDULE: return "schedule does not match the call";
    case FP4IDX_ERR_SCRATCH_LIMIT: return "call needs more than the fixed top-k scratch";
    default: return "unknown status";
  }
}

int fp4idx_num_sms(int32_t* num_sms_out) {
  if (!num_sms_out) return FP4IDX_ERR_INVALID_ARG;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP4IDX_ERR_CUDA;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FP4IDX_ERR_CUDA;
  *num_sms_out = n;
  return FP4IDX_OK;
}

int fp4idx_store_k(const uint16_t* k, int64_t n_rows, const int32_t* positions, const int32_t* slots,
                   const uint16_t* norm_w, float eps, const uint16_t* cos_sin, int32_t max_pos,
                   uint8_t* payload, uint8_t* scale, int64_t num_pages, int32_t* status_dev, void* stream) {
  int st = check_store_args(k, n_rows, positions, slots, norm_w, cos_sin, max_pos, num_pages);
  if (st != FP4IDX_OK || n_rows == 0) return st;
  if (!payload || !scale || !aligned16(payload)) return FP4IDX_ERR_INVALID_ARG;
  if (status_dev && !aligned4(status_dev)) return FP4IDX_ERR_INVALID_ARG;
  return from_cuda(fp4idx::launch_store_k(k, n_rows, positions, slots, norm_w, eps, cos_sin, max_pos, payload,
                                          scale, num_pages, status_dev, as_stream(stream)));
}

int fp4idx_store_k_fp8(const uint16_t* k, int64_t n_rows, const int32_t* positions, const int32_t* slots,
                       const uint16_t* norm_w, float eps, const uint16_t* cos_sin, int32_t max_pos,
                       uint8_t* fp8_pages, int64_t num_pages, int32_t* status_dev, void* stream) {
  int st = check_store_args(k, n_rows, positions, slots, norm_w, cos_sin, max_pos, num_pages);
  if (st != FP4IDX_OK || n_rows == 0) return st;
  if (!fp8_pages || !aligned16(fp8_pages)) return FP4IDX_ERR_INVALID_ARG;
  if (status_dev && !aligned4(status_dev)) return FP4IDX_ERR_INVALID_ARG;
  return from_cuda(fp4idx::launch_store_k_fp8(k, n_rows, positions, slots, norm_w, eps, cos_sin, max_pos,
                                              fp8_pages, num_pages, status_dev, as_stream(stream)));
}

int fp4idx_quant_q(const uint16_t* q, int64_t n_rows, int32_t n_heads, const int32_t* q_positions,
                   const uint16_t* cos_sin, int32_t max_pos, uint8_t* q_payload, uint8_t* q_scale,
                   int32_t* status_dev, void* stream) {
  if (n_rows < 0 || max_pos <= 0) return FP4IDX_ERR_INVALID_ARG;
  if (n_heads != fp4idx::kHeads) return FP4IDX_ERR_UNSUPPORTED;
  if (n_rows == 0) return FP4IDX_OK;
  if (!q || !q_positions || !cos_sin || !q_payload || !q_scale) return FP4IDX_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(cos_sin) || !aligned16(q_payload) || !aligned4(q_positions))
    return FP4IDX_ERR_INVALID_ARG;
  if (status_dev && !aligned4(status_dev)) return FP4IDX_ERR_INVALID_ARG;
  return from_cuda(fp4idx::launch_quant_q(q, n_rows, q_positions, cos_sin, max_pos, q_payload, q_scale, status_dev,
                                          as_stream(stream)));
}

int fp4idx_quant_q_fp8(const uint16_t* q, int64_t n_rows, int32_t n_heads, const int32_t* q_positions,
                       const uint16_t* cos_sin, int32_t max_pos, uint8_t* q8, float* q8_scale, int32_t* status_dev,
                       void* stream) {
  if (n_rows < 0 || max_pos <= 0) return FP4IDX_ERR_INVALID_ARG;
  if (n_heads != fp4idx::kHeads) return FP4IDX_ERR_UNSUPPORTED;
  if (n_rows == 0) return FP4IDX_OK;
  if (!q || !q_positions || !cos_sin || !q8 || !q8_scale) return FP4IDX_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(cos_sin) || !aligned16(q8) || !aligned4(q_positions) || !aligned4(q8_scale))
    return FP4IDX_ERR_INVALID_ARG;
  if (status_dev && !aligned4(status_dev)) return FP4IDX_ERR_INVALID_ARG;
  return from_cuda(fp4idx::launch_quant_q_fp8(q, n_rows, q_positions, cos_sin, max_pos, q8, q8_scale, status_dev,
                                              as_stream(stream)));
}

int fp4idx_quant_q_w(const uint16_t* q, int64_t n_rows, int32_t n_heads, const int32_t* q_positions,
                     const uint16_t* cos_sin, int32_t max_pos, const uint16_t* hidden, int32_t hidden_dim,
                     const uint16_t* w_proj, float w_scale, uint8_t* q_payload, uint8_t* q_scale, float* w_out,
                     int32_t* status_dev, void* stream) {
  if (n_rows < 0 || max_pos <= 0 || hidden_dim <= 0) return FP4IDX_ERR_INVALID_ARG;
  if (n_heads != fp4idx::kHeads) return FP4IDX_ERR_UNSUPPORTED;
  if (hidden_dim % 256 != 0 || hidden_dim > FP4IDX_MAX_HIDDEN) return FP4IDX_ERR_UNSUPPORTED;
  if (n_rows > (int64_t)INT32_MAX / 12) return FP4IDX_ERR_UNSUPPORTED;  // 4 quant blocks and 8 weight blocks a row
  if (n_rows == 0) return FP4IDX_OK;
  if (!q || !q_positions || !cos_sin || !q_payload || !q_scale || !hidden || !w_proj || !w_out)
    return FP4IDX_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(cos_sin) || !aligned16(q_payload) || !aligned4(q_positions) || !aligned16(hidden) ||
      !aligned16(w_proj) || !aligned4(w_out))
    return FP4IDX_ERR_INVALID_ARG;
  if (status_dev && !aligned4(status_dev)) return FP4IDX_ERR_INVALID_ARG;
  return from_cuda(fp4idx::launch_quant_q_w(q, n_rows, q_positions, cos_sin, max_pos, q_payload, q_scale, hidden,
                                            hidden_dim, w_proj, w_scale, w_out, status_dev, as_stream(stream)));
}

size_t fp4idx_schedule_workspace_bytes(int64_t max_rows, int32_t num_ctas) {
  if (max_rows < 0 || max_rows > INT32_MAX - 1 || num_ctas < 0) return 0;
  if (num_ctas == 0 && device_sms(&num_ctas) != FP4IDX_OK) return 0;
  return fp4idx::sched_bytes(max_rows, num_ctas);
}

int fp4idx_build_schedule(const int32_t* context_lens, const int32_t* row_seq, int64_t n_rows, int32_t num_ctas,
                          void* schedule, size_t schedule_bytes, void* stream) {
  if (n_rows < 0 || n_rows > INT32_MAX - 1 || num_ctas < 0) return FP4IDX_ERR_INVALID_ARG;
  if (!schedule || !aligned16(schedule)) return FP4IDX_ERR_INVALID_ARG;
  if (n_rows > 0 && (!context_lens || !row_seq || !aligned4(context_lens) || !aligned4(row_seq)))
    return FP4IDX_ERR_INVALID_ARG;
  if (num_ctas == 0) {
    int st = device_sms(&num_ctas);
    if (st != FP4IDX_OK) return st;
  }
  if (schedule_bytes < fp4idx::sched_bytes(n_rows, num_ctas)) return FP4IDX_ERR_WORKSPACE;
  return from_cuda(fp4idx::launch_build_schedule(context_lens, row_seq, (int32_t)n_rows, num_ctas, schedule,
                                                 as_stream(stream)));
}

int fp4idx_prepare_step(const uint16_t* k, int64_t n_new, const int32_t* positions, const int32_t* slots,
                        const uint16_t* norm_w, float eps, const uint16_t* q, int64_t n_rows, int32_t n_heads,
                        const int32_t* q_positions, const uint16_t* cos_sin, int32_t max_pos, uint8_t* payload,
                        uint8_t* scale, int64_t num_pages, uint8_t* q_payload, uint8_t* q_scale,
                        const int32_t* context_lens, const int32_t* row_seq, int32_t num_ctas, void* schedule,
                        size_t schedule_bytes, int32_t* status_dev, void* stream) {
  // the checks of fp4idx_store_k, fp4idx_quant_q and fp4idx_build_schedule
  int st = check_store_args(k, n_new, positions, slots, norm_w, cos_sin, max_pos, num_pages);
  if (st != FP4IDX_OK) return st;
  if (n_new > 0 && (!payload || !scale || !aligned16(payload))) return FP4IDX_ERR_INVALID_ARG;
  if (n_rows < 0 || n_rows > INT32_MAX - 1 || num_ctas < 0) return FP4IDX_ERR_INVALID_ARG;
  if (n_heads != fp4idx::kHeads) return FP4IDX_ERR_UNSUPPORTED;
  if (n_rows > 0) {
    if (!q || !q_positions || !cos_sin || !q_payload || !q_scale || !context_lens || !row_seq) return FP4IDX_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(cos_sin) || !aligned16(q_payload) || !aligned4(q_positions) ||
        !aligned4(context_lens) || !aligned4(row_seq))
      return FP4IDX_ERR_INVALID_ARG;
  }
  if (!schedule || !aligned16(schedule)) return FP4IDX_ERR_INVALID_ARG;
  if (status_dev && !aligned4(status_dev)) return FP4IDX_ERR_INVALID_ARG;
  if (num_ctas == 0) {
    st = device_sms(&num_ctas);
    if (st != FP4IDX_OK) return st;
  }
  if (schedule_bytes < fp4idx::sched_bytes(n_rows, num_ctas)) return FP4IDX_ERR_WORKSPACE;
  return from_cuda(fp4idx::launch_prepare_step(k, n_new, positions, slots, norm_w, eps, q, n_rows, q_positions,
                                               cos_sin, max_pos, payload, scale, num_pages, q_payload, q_scale,
                                               context_lens, row_seq, num_ctas, schedule, status_dev,
                                               as_stream(stream)));
}

// Layout of the logits + top-k workspace: [logits buffer][top-k scratch].
inline size_t logits_region_bytes(int64_t rows, int32_t max_context) {
  return ((size_t)rows * (size_t)logits_row_stride(max_context) * sizeof(float) + 255) & ~(size_t)255;
}

size_t fp4idx_topk_workspace_bytes(int64_t max_rows, int32_t max_context) {
  if (max_rows < 0 || max_context < 0) return 0;
  return fp4idx::topk_workspace_bytes(max_rows, max_context);
}

// Scratch after the logits region: the top-k kernel's (separate selection) or the fused
// selection's (the sort keys of positions past what a CTA keeps in shared memory).
inline size_t select_scratch_bytes(int64_t rows, int32_t max_context) {
  const size_t a = fp4idx::topk_workspace_bytes(rows, max_context);
  const size_t b = fp4idx::logits_select_spill_bytes(rows, max_context);
  return a > b ? a : b;
}

size_t fp4idx_logits_workspace_bytes(int64_t max_rows, int32_t max_context, int32_t k) {
  (void)k;
  if (max_rows < 0 || max_context < 0) return 0;
  return logits_region_bytes(max_rows, max_context) + select_scratch_bytes(max_rows, max_context);
}

namespace {

int check_logits_args(const uint8_t* q_payload, const uint8_t* q_scale, const float* w, int64_t n_rows,
                      int32_t n_heads, const uint8_t* payload, const uint8_t* scale, int64_t num_pages,
                      const int32_t* page_table, int64_t num_seqs, int32_t max_pages, const int32_t* row_seq,
                      const int32_t* context_lens, int32_t max_context, const void* schedule, size_t schedule_bytes,
                      int32_t* status_dev) {
  if (n_rows < 0 || n_rows > INT32_MAX - 1 || num_pages < 0 || num_seqs < 0 || max_pages < 0 || max_context < 0)
    return FP4IDX_ERR_INVALID_ARG;
  if (n_heads != fp4idx::kHeads) return FP4IDX_ERR_UNSUPPORTED;
  if (max_context > FP4IDX_MAX_CONTEXT) return FP4IDX_ERR_UNSUPPORTED;
  if (n_rows == 0) return FP4IDX_OK;
  if (!q_payload || !q_scale || !w || !payload || !scale || !page_table || !row_seq || !context_lens || !schedule)
    return FP4IDX_ERR_INVALID_ARG;
  if (!aligned16(q_payload) || !aligned16(q_scale) || !aligned16(w) || !aligned16(payload) || !aligned16(scale) ||
      !aligned4(page_table) || !aligned4(row_seq) || !aligned4(context_lens) || !aligned16(schedule))
    return FP4IDX_ERR_INVALID_ARG;
  if (status_dev && !aligned4(status_dev)) return FP4IDX_ERR_INVALID_ARG;
  int32_t sms = 0;
  if (device_sms(&sms) != FP4IDX_OK) return FP4IDX_ERR_CUDA;
  if (schedule_bytes < fp4idx::sched_bytes(n_rows, sms)) return FP4IDX_ERR_WORKSPACE;
  return FP4IDX_OK;
}

int launch_logits_checked(const uint8_t* q_payload, const uint8_t* q_scale, const float* w, int64_t n_rows,
                          const uint8_t* payload, const uint8_t* scale, int64_t num_pages, const int32_t* page_table,
                          int64_t num_seqs, int32_t max_pages, const int32_t* row_seq, const int32_t* context_lens,
                          int32_t max_context, const void* schedule, float* buf, int64_t stride, int32_t k,
                          int32_t* topk_idx, void* spill, int32_t* status_dev, cudaStream_t s) {
  int32_t grid = 0;
  int st = device_sms(&grid);
  if (st != FP4IDX_OK) return st;
  return from_cuda(fp4idx::launch_logits_mxf4(q_payload, q_scale, w, (int32_t)n_rows, payload, scale, num_pages,
                                              page_table, num_seqs, max_pages, row_seq, context_lens, max_context,
                                              schedule, grid, buf, stride, k, topk_idx, spill, status_dev, s));
}

}  // namespace

int fp4idx_logits(const uint8_t* q_payload, const uint8_t* q_scale, const float* w, int64_t n_rows, int32_t n_heads,
                  const uint8_t* payload, const uint8_t* scale, int64_t num_pages, const int32_t* page_table,
                  int64_t num_seqs, int32_t max_pages, const int32_t* row_seq, const int32_t* context_lens,
                  int32_t max_context, const void* schedule, size_t schedule_bytes, float* logits_out,
                  int64_t logits_stride, int32_t* status_dev, void* stream) {
  int st = check_logits_args(q_payload, q_scale, w, n_rows, n_heads, payload, scale, num_pages, page_table, num_seqs,
                             max_pages, row_seq, context_lens, max_context, schedule, schedule_bytes, status_dev);
  if (st != FP4IDX_OK || n_rows == 0) return st;
  if (!logits_out || !aligned4(logits_out) || logits_stride < max_context) return FP4IDX_ERR_INVALID_ARG;
  return launch_logits_checked(q_payload, q_scale, w, n_rows, payload, scale, num_pages, page_table, num_seqs,
                               max_pages, row_seq, context_lens, max_context, schedule, logits_out, logits_stride, 0,
                               nullptr, nullptr, status_dev, as_stream(stream));
}

int fp4idx_logits_fp8(const uint8_t* q8, const float* q8_scale, const float* w, int64_t n_rows, int32_t n_heads,
                      const uint8_t* fp8_pages, int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                      int32_t max_pages, const int32_t* row_seq, const int32_t* context_lens, int32_t max_context,
                      const void* schedule, size_t schedule_bytes, float* logits_out, int64_t logits_stride,
                      int32_t* status_dev, void* stream) {
  // the FP8 operands take the places of the FP4 ones in the common checks (all 16-byte aligned)
  int st = check_logits_args(q8, reinterpret_cast<const uint8_t*>(q8_scale), w, n_rows, n_heads, fp8_pages, fp8_pages,
                             num_pages, page_table, num_seqs, max_pages, row_seq, context_lens, max_context, schedule,
                             schedule_bytes, status_dev);
  if (st != FP4IDX_OK || n_rows == 0) return st;
  if (!logits_out || !aligned4(logits_out) || logits_stride < max_context) return FP4IDX_ERR_INVALID_ARG;
  if (num_pages < 1 || num_pages > INT32_MAX) return FP4IDX_ERR_INVALID_ARG;
  int32_t grid = 0;
  st = device_sms(&grid);
  if (st != FP4IDX_OK) return st;
  return from_cuda(fp4idx::launch_logits_fp8(q8, q8_scale, w, (int32_t)n_rows, fp8_pages, num_pages, page_table,
                                             num_seqs, max_pages, context_lens, max_context, schedule, grid,
                                             logits_out, logits_stride, status_dev, as_stream(stream)));
}

int fp4idx_topk(const float* logits, int64_t logits_stride, const int32_t* context_lens, int64_t n_rows,
                int32_t max_context, int32_t k, void* workspace, size_t workspace_bytes, int32_t* topk_idx,
                int32_t* status_dev, void* stream) {
  if (n_rows < 0 || n_rows > INT32_MAX - 1 || max_context < 0 || k < 1 || k > FP4IDX_MAX_TOPK)
    return FP4IDX_ERR_INVALID_ARG;
  if (max_context > FP4IDX_MAX_CONTEXT) return FP4IDX_ERR_UNSUPPORTED;
  if (n_rows == 0) return FP4IDX_OK;
  if (!logits || !context_lens || !topk_idx || !aligned4(logits) || !aligned4(context_lens) || !aligned4(topk_idx) ||
      logits_stride < max_context)
    return FP4IDX_ERR_INVALID_ARG;
  if (status_dev && !aligned4(status_dev)) return FP4IDX_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return FP4IDX_ERR_INVALID_ARG;
  if (workspace_bytes < fp4idx::topk_workspace_bytes(n_rows, max_context)) return FP4IDX_ERR_WORKSPACE;
  return from_cuda(fp4idx::launch_topk(logits, logits_stride, context_lens, (int32_t)n_rows, max_context, k,
                                       workspace, topk_idx, status_dev, as_stream(stream)));
}

namespace {

// fp4idx_logits_topk and fp4idx_logits_topk_fused: the same checks and buffers; `fused`
// asks for the selection inside the logits launch where the grid has a CTA for every row.
int logits_topk_impl(const uint8_t* q_payload, const uint8_t* q_scale, const float* w, int64_t n_rows,
                     int32_t n_heads, const uint8_t* payload, const uint8_t* scale, int64_t num_pages,
                     const int32_t* page_table, int64_t num_seqs, int32_t max_pages, const int32_t* row_seq,
                     const int32_t* context_lens, int32_t max_context, int32_t k, void* schedule,
                     size_t schedule_bytes, void* workspace, size_t workspace_bytes, int32_t* topk_idx,
                     float* logits_out, int64_t logits_stride, int32_t* status_dev, void* stream, bool fused) {
  int st = check_logits_args(q_payload, q_scale, w, n_rows, n_heads, payload, scale, num_pages, page_table, num_seqs,
                             max_pages, row_seq, context_lens, max_context, schedule, schedule_bytes, status_dev);
  if (st != FP4IDX_OK) return st;
  if (k < 1 || k > FP4IDX_MAX_TOPK) return FP4IDX_ERR_INVALID_ARG;
  if (n_rows == 0) return FP4IDX_OK;
  if (!topk_idx || !aligned4(topk_idx)) return FP4IDX_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return FP4IDX_ERR_INVALID_ARG;
  if (workspace_bytes < fp4idx_logits_workspace_bytes(n_rows, max_context, k)) return FP4IDX_ERR_WORKSPACE;
  float* buf;
  int64_t stride;
  if (logits_out) {
    if (logits_stride < max_context || !aligned4(logits_out)) return FP4IDX_ERR_INVALID_ARG;
    buf = logits_out;
    stride = logits_stride;
  } else {
    stride = logits_row_stride(max_context);
    buf = reinterpret_cast<float*>(workspace);
  }
  void* topk_ws = reinterpret_cast<uint8_t*>(workspace) + logits_region_bytes(n_rows, max_context);
  cudaStream_t s = as_stream(stream);
  int32_t sms = 0;
  st = device_sms(&sms);
  if (st != FP4IDX_OK) return st;
  if (fused && n_rows <= sms) {
    // the CTA (pair) of each row selects it from the logits the launch wrote
    return launch_logits_checked(q_payload, q_scale, w, n_rows, payload, scale, num_pages, page_table, num_seqs,
                                 max_pages, row_seq, context_lens, max_context, schedule, buf, stride, k, topk_idx,
                                 topk_ws, status_dev, s);
  }
  // the logits launch, then the top-k launch (one CTA, or a pair of CTAs, per row)
  st = launch_logits_checked(q_payload, q_scale, w, n_rows, payload, scale, num_pages, page_table, num_seqs, max_pages,
                             row_seq, context_lens, max_context, schedule, buf, stride, 0, nullptr, nullptr,
                             status_dev, s);
  if (st != FP4IDX_OK) return st;
  return from_cuda(fp4idx::launch_topk(buf, stride, context_lens, (int32_t)n_rows, max_context, k, topk_ws,
                                       topk_idx, status_dev, s));
}

}  // namespace

int fp4idx_logits_topk(const uint8_t* q_payload, const uint8_t* q_scale, const float* w, int64_t n_rows,
                       int32_t n_heads, const uint8_t* payload, const uint8_t* scale, int64_t num_pages,
                       const int32_t* page_table, int64_t num_seqs, int32_t max_pages, const int32_t* row_seq,
                       const int32_t* context_lens, int32_t max_context, int32_t k, const void* schedule,
                       size_t schedule_bytes, void* workspace, size_t workspace_bytes, int32_t* topk_idx,
                       float* logits_out, int64_t logits_stride, int32_t* status_dev, void* stream) {
  return logits_topk_impl(q_payload, q_scale, w, n_rows, n_heads, payload, scale, num_pages, page_table, num_seqs,
                          max_pages, row_seq, context_lens, max_context, k, const_cast<void*>(schedule),
                          schedule_bytes, workspace, workspace_bytes, topk_idx, logits_out, logits_stride, status_dev,
                          stream, false);
}

int fp4idx_logits_topk_fused(const uint8_t* q_payload, const uint8_t* q_scale, const float* w, int64_t n_rows,
                             int32_t n_heads, const uint8_t* payload, const uint8_t* scale, int64_t num_pages,
                             const int32_t* page_table, int64_t num_seqs, int32_t max_pages, const int32_t* row_seq,
                             const int32_t* context_lens, int32_t max_context, int32_t k, void* schedule,
                             size_t schedule_bytes, void* workspace, size_t workspace_bytes, int32_t* topk_idx,
                             float* logits_out, int64_t logits_stride, int32_t* status_dev, void* stream) {
  return logits_topk_impl(q_payload, q_scale, w, n_rows, n_heads, payload, scale, num_pages, page_table, num_seqs,
                          max_pages, row_seq, context_lens, max_context, k, schedule, schedule_bytes, workspace,
                          workspace_bytes, topk_idx, logits_out, logits_stride, status_dev, stream, true);
}

int fp4idx_logits_topk_fp8(const uint8_t* q8, const float* q8_scale, const float* w, int64_t n_rows, int32_t n_heads,
                           const uint8_t* fp8_pages, int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                           int32_t max_pages, const int32_t* row_seq, const int32_t* context_lens,
                           int32_t max_context, int32_t k, const void* schedule, size_t schedule_bytes,
                           void* workspace, size_t workspace_bytes, int32_t* topk_idx, float* logits_out,
                           int64_t logits_stride, int32_t* status_dev, void* stream) {
  int st = check_logits_args(q8, reinterpret_cast<const uint8_t*>(q8_scale), w, n_rows, n_heads, fp8_pages, fp8_pages,
                             num_pages, page_table, num_seqs, max_pages, row_seq, context_lens, max_context, schedule,
                             schedule_bytes, status_dev);
  if (st != FP4IDX_OK) return st;
  if (k < 1 || k > FP4IDX_MAX_TOPK) return FP4IDX_ERR_INVALID_ARG;
  if (n_rows == 0) return FP4IDX_OK;
  if (num_pages < 1 || num_pages > INT32_MAX) return FP4IDX_ERR_INVALID_ARG;
  if (!topk_idx || !aligned4(topk_idx)) return FP4IDX_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return FP4IDX_ERR_INVALID_ARG;
  if (workspace_bytes < fp4idx_logits_workspace_bytes(n_rows, max_context, k)) return FP4IDX_ERR_WORKSPACE;
  float* buf;
  int64_t stride;
  if (logits_out) {
    if (logits_stride < max_context || !aligned4(logits_out)) return FP4IDX_ERR_INVALID_ARG;
    buf = logits_out;
    stride = logits_stride;
  } else {
    stride = logits_row_stride(max_context);
    buf = reinterpret_cast<float*>(workspace);
  }
  void* topk_ws = reinterpret_cast<uint8_t*>(workspace) + logits_region_bytes(n_rows, max_context);
  cudaStream_t s = as_stream(stream);
  int32_t grid = 0;
  st = device_sms(&grid);
  if (st != FP4IDX_OK) return st;
  st = from_cuda(fp4idx::launch_logits_fp8(q8, q8_scale, w, (int32_t)n_rows, fp8_pages, num_pages, page_table,
                                           num_seqs, max_pages, context_lens, max_context, schedule, grid, buf,
                                           stride, status_dev, s));
  if (st != FP4IDX_OK) return st;
  return from_cuda(fp4idx::launch_topk(buf, stride, context_lens, (int32_t)n_rows, max_context, k, topk_ws,
                                       topk_idx, status_dev, s));
}

namespace {

int check_page_args(const void* payload, const void* scale, int64_t num_pages, const int32_t* page_ids,
                    int64_t n_pages, const void* rows_a, const void* rows_b, int32_t* status_dev) {
  if (num_pages < 0 || n_pages < 0 || n_pages > INT32_MAX) return FP4IDX_ERR_INVALID_ARG;
  if (n_pages == 0) return FP4IDX_OK;
  if (!payload || !scale || !page_ids || !rows_a || !rows_b) return FP4IDX_ERR_INVALID_ARG;
  if (!aligned16(payload) || !aligned16(scale) || !aligned4(page_ids) || !aligned16(rows_a) || !aligned16(rows_b))
    return FP4IDX_ERR_INVALID_ARG;
  if (status_dev && !aligned4(status_dev)) return FP4IDX_ERR_INVALID_ARG;
  return FP4IDX_OK;
}

}  // namespace

int fp4idx_dequant_pages(const uint8_t* payload, const uint8_t* scale, int64_t num_pages, const int32_t* page_ids,
                         int64_t n_pages, float* out, int32_t* status_dev, void* stream) {
  const int st = check_page_args(payload, scale, num_pages, page_ids, n_pages, out, out, status_dev);
  if (st != FP4IDX_OK || n_pages == 0) return st;
  return from_cuda(fp4idx::launch_dequant_pages(payload, scale, num_pages, page_ids, n_pages, out, status_dev,
                                                as_stream(stream)));
}

int fp4idx_export_pages(const uint8_t* payload, const uint8_t* scale, int64_t num_pages, const int32_t* page_ids,
                        int64_t n_pages, uint8_t* rows_payload, uint8_t* rows_scale, int32_t* status_dev,
                        void* stream) {
  const int st = check_page_args(payload, scale, num_pages, page_ids, n_pages, rows_payload, rows_scale, status_dev);
  if (st != FP4IDX_OK || n_pages == 0) return st;
  return from_cuda(fp4idx::launch_copy_pages(const_cast<uint8_t*>(payload), const_cast<uint8_t*>(scale), num_pages,
                                             page_ids, n_pages, rows_payload, rows_scale, true, status_dev,
                                             as_stream(stream)));
}

int fp4idx_import_pages(const uint8_t* rows_payload, const uint8_t* rows_scale, const int32_t* page_ids,
                        int64_t n_pages, uint8_t* payload, uint8_t* scale, int64_t num_pages, int32_t* status_dev,
                        void* stream) {
  const int st = check_page_args(payload, scale, num_pages, page_ids, n_pages, rows_payload, rows_scale, status_dev);
  if (st != FP4IDX_OK || n_pages == 0) return st;
  return from_cuda(fp4idx::launch_copy_pages(payload, scale, num_pages, page_ids, n_pages,
                                             const_cast<uint8_t*>(rows_payload), const_cast<uint8_t*>(rows_scale),
                                             false, status_dev, as_stream(stream)));
}

size_t fp4idx_topk_merge_workspace_bytes(int64_t max_rows, int32_t n_shards, int32_t k) {
  if (max_rows < 0 || n_shards < 1 || k < 1 || (int64_t)n_shards * k > FP4IDX_MAX_CONTEXT) return 0;
  return fp4idx::merge_workspace_bytes(max_rows, n_shards, k);
}

int fp4idx_topk_values(const float* logits, int64_t logits_stride, const int32_t* topk_idx, int64_t n_rows, int32_t k,
                       float* values, void* stream) {
  if (n_rows < 0 || n_rows > 65535 || k < 1 || k > FP4IDX_MAX_TOPK || logits_stride < 1) return FP4IDX_ERR_INVALID_ARG;
  if (n_rows == 0) return FP4IDX_OK;
  if (!logits || !topk_idx || !values || !aligned4(logits) || !aligned4(topk_idx) || !aligned4(values))
    return FP4IDX_ERR_INVALID_ARG;
  return from_cuda(fp4idx::launch_gather_values(logits, logits_stride, topk_idx, (int32_t)n_rows, k, values,
                                                as_stream(stream)));
}

int fp4idx_topk_merge(const float* cand_values, const int32_t* cand_idx, int64_t n_rows, int32_t n_shards, int32_t k,
                      void* workspace, size_t workspace_bytes, int32_t* topk_idx, int32_t* status_dev, void* stream) {
  if (n_rows < 0 || n_rows > 65535 || k < 1 || k > FP4IDX_MAX_TOPK || n_shards < 1 || n_shards > 1024 ||
      (int64_t)n_shards * k > FP4IDX_MAX_CONTEXT)
    return FP4IDX_ERR_INVALID_ARG;
  if (n_rows == 0) return FP4IDX_OK;
  if (!cand_values || !cand_idx || !topk_idx || !workspace || !aligned4(cand_values) || !aligned4(cand_idx) ||
      !aligned4(topk_idx) || !aligned16(workspace))
    return FP4IDX_ERR_INVALID_ARG;
  if (status_dev && !aligned4(status_dev)) return FP4IDX_ERR_INVALID_ARG;
  if (workspace_bytes < fp4idx::merge_workspace_bytes(n_rows, n_shards, k)) return FP4IDX_ERR_WORKSPACE;
  return from_cuda(fp4idx::launch_topk_merge(cand_values, cand_idx, (int32_t)n_rows, n_shards, k, workspace,
                                             topk_idx, status_dev, as_stream(stream)));
}

int fp4idx_read_status(const int32_t* status_dev, int32_t* host_out, void* stream) {
  if (!status_dev || !host_out) return FP4IDX_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  if (cudaMemcpyAsync(host_out, status_dev, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FP4IDX_ERR_CUDA;
  return from_cuda(cudaStreamSynchronize(s));
}

}  // extern "C"
