// Host launchers of the kernels of libfp4idx.so, called by the C ABI (api.cu) and by
// launchers that compose others.
#pragma once

#include <cuda.h>

#include "fp4idx_internal.cuh"

namespace fp4idx {

// ---------------------------------------------------------------- shared host helpers (host_util.cu)
// cuTensorMapEncodeTiled, looked up once through the runtime.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();
// 2-D view of `rows` rows of `row_bytes` bytes as uint64 elements; box = one row.
bool encode_rows(CUtensorMap* map, const void* base, int64_t rows, uint32_t row_bytes);
// A kernel's dynamic shared-memory limit, set once per (kernel, device); thread-safe.
cudaError_t set_smem_attr_once(const void* kernel, size_t bytes);
// How many CTAs of `threads` threads and `smem` bytes of dynamic shared memory fit on the
// current device at once (SMs x CTAs per SM), computed once per (kernel, device).
cudaError_t resident_ctas(const void* kernel, int threads, size_t smem, int* out);
// How long one pipeline wait of the logits kernels may last before the kernel records
// FP4IDX_ERR_TIMEOUT and winds down, and whether their producers are told to issue
// nothing (a test switch, off by default: with it on, every launch ends in that timeout).
constexpr int64_t kDefaultWaitLimitNs = 2000000000;
uint64_t pipeline_wait_limit_ns();
bool pipeline_idle_producers();

// ---------------------------------------------------------------- launchers (host)
cudaError_t launch_store_k(const uint16_t* k, int64_t n_rows, const int32_t* positions, const int32_t* slots,
                           const uint16_t* norm_w, float eps, const uint16_t* cos_sin, int32_t max_pos,
                           uint8_t* payload, uint8_t* scale, int64_t num_pages, int32_t* status,
                           cudaStream_t stream);
cudaError_t launch_store_k_fp8(const uint16_t* k, int64_t n_rows, const int32_t* positions, const int32_t* slots,
                               const uint16_t* norm_w, float eps, const uint16_t* cos_sin, int32_t max_pos,
                               uint8_t* pages, int64_t num_pages, int32_t* status, cudaStream_t stream);
cudaError_t launch_quant_q(const uint16_t* q, int64_t n_rows, const int32_t* q_positions, const uint16_t* cos_sin,
                           int32_t max_pos, uint8_t* q_payload, uint8_t* q_scale, int32_t* status,
                           cudaStream_t stream);

cudaError_t launch_quant_q_fp8(const uint16_t* q, int64_t n_rows, const int32_t* q_positions, const uint16_t* cos_sin,
                               int32_t max_pos, uint8_t* q8, float* q8_scale, int32_t* status, cudaStream_t stream);
cudaError_t launch_quant_q_w(const uint16_t* q, int64_t n_rows, const int32_t* q_positions, const uint16_t* cos_sin,
                             int32_t max_pos, uint8_t* q_payload, uint8_t* q_scale, const uint16_t* hidden,
                             int32_t dim, const uint16_t* w_proj, float w_scale, float* w_out, int32_t* status,
                             cudaStream_t stream);

// The decode step's preparation (schedule, K store, Q quant) in one launch.
cudaError_t launch_prepare_step(const uint16_t* k, int64_t n_new, const int32_t* positions, const int32_t* slots,
                                const uint16_t* norm_w, float eps, const uint16_t* q, int64_t n_rows,
                                const int32_t* q_positions, const uint16_t* cos_sin, int32_t max_pos,
                                uint8_t* payload, uint8_t* scale, int64_t num_pages, uint8_t* q_payload,
                                uint8_t* q_scale, const int32_t* context_lens, const int32_t* row_seq,
                                int32_t num_ctas, void* schedule, int32_t* status, cudaStream_t stream);
cudaError_t launch_build_schedule(const int32_t* context_lens, const int32_t* row_seq, int32_t n_rows,
                                  int32_t num_ctas, void* ws, cudaStream_t stream);
cudaError_t launch_logits_mxf4(const uint8_t* q_payload, const uint8_t* q_scale, const float* w, int32_t n_rows,
                               const uint8_t* payload, const uint8_t* scale, int64_t num_pages,
                               const int32_t* page_table, int64_t num_seqs, int32_t max_pages,
                               const int32_t* row_seq, const int32_t* context_lens, int32_t max_context,
                               const void* schedule, int32_t num_ctas, float* out, int64_t out_stride,
                               int32_t k, int32_t* topk, void* spill, int32_t* status, cudaStream_t stream);
// Scratch of the fused selection (k > 0 in launch_logits_mxf4): the sort keys of row
// positions past what one CTA keeps in shared memory.  Nothing in it needs initialising.
size_t logits_select_spill_bytes(int64_t n_rows, int32_t max_context);
cudaError_t launch_logits_fp8(const uint8_t* q8, const float* q8_scale, const float* w, int32_t n_rows,
                              const uint8_t* pages, int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                              int32_t max_pages, const int32_t* context_lens, int32_t max_context,
                              const void* schedule, int32_t num_ctas, float* out, int64_t out_stride,
                              int32_t* status, cudaStream_t stream);
cudaError_t launch_dequant_pages(const uint8_t* payload, const uint8_t* scale, int64_t num_pages,
                                 const int32_t* page_ids, int64_t n_pages, float* out, int32_t* status,
                                 cudaStream_t stream);
cudaError_t launch_copy_pages(uint8_t* payload, uint8_t* scale, int64_t num_pages, const int32_t* page_ids,
                              int64_t n_pages, uint8_t* rows_payload, uint8_t* rows_scale, bool to_rows,
                              int32_t* status, cudaStream_t stream);
size_t merge_workspace_bytes(int64_t n_rows, int32_t n_shards, int32_t k);
cudaError_t launch_gather_values(const float* logits, int64_t stride, const int32_t* idx, int32_t n_rows, int32_t k,
                                 float* values, cudaStream_t stream);
cudaError_t launch_topk_merge(const float* cand_values, const int32_t* cand_idx, int32_t n_rows, int32_t n_shards,
                              int32_t k, void* workspace, int32_t* topk_idx, int32_t* status, cudaStream_t stream);
size_t topk_workspace_bytes(int64_t n_rows, int32_t max_context);
cudaError_t launch_topk(const float* logits, int64_t stride, const int32_t* context_lens, int32_t n_rows,
                        int32_t max_context, int32_t k, void* workspace, int32_t* out, int32_t* status,
                        cudaStream_t stream);

}  // namespace fp4idx
