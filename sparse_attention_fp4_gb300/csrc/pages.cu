// Whole-page access to the split FP4 index-K cache: dequantisation, and export to /
// import from contiguous page rows.
//
// dsv4.1-amd: KV cache layouts, FP4 indexer, compressor and router kernels -- Summary:
// dequantize_k_cache_paged serves the V4.1 layouts.  [AMD] Enable FP4 indexer for
// Deepseek V4 -- Device memory and sizing / HiCache integration: the pool exposes
// page-row views of the separately allocated payload and scale buffers, and host
// transfers of the FP4 indexer rows are whole-page only (payload and scale regions
// move as separate page-contiguous regions).
//
// One CTA of 256 threads per listed page.  A page is 4,096 payload bytes
// ([c][token][16 B]) and 256 scale bytes ([c][token]); thread t owns the 16-byte row
// (c, j) = (t / 64, t % 64) of the payload and, for t < 16, a 16-byte piece of the
// scales, so every global access is a coalesced 16-byte access.  Page ids < 0 are
// padding and skipped; ids >= num_pages record FP4IDX_ERR_BAD_PAGE and are skipped.
#include "launchers.cuh"

namespace fp4idx {
namespace {

constexpr int kPageThreads = 256;  // 4 blocks x 64 tokens
constexpr uint32_t kPagePayload = 4096, kPageScale = 256;

// Page id of list entry i, or -1 when the entry is padding or out of range (recorded).
__device__ __forceinline__ int64_t page_of(const int32_t* page_ids, int64_t i, int64_t num_pages, int32_t* status) {
  const int32_t p = __ldg(page_ids + i);
  if (p < 0) return -1;
  if ((int64_t)p >= num_pages) {
    if (threadIdx.x == 0) record_error(status, FP4IDX_ERR_BAD_PAGE);
    return -1;
  }
  return p;
}

// Value of an e2m1 code (OCP MX: 1 sign, 2 exponent, 1 mantissa bit; no inf/NaN):
// magnitudes 0, 0.5 (subnormal), then 2^(m/2 - 1) * (1 + (m & 1) / 2) = 1, 1.5, 2, 3,
// 4, 6 for m = 2..7; bit 3 is the sign.
__device__ __forceinline__ float e2m1_value(uint32_t code) {
  const uint32_t m = code & 7u;
  const float mag = m < 2u ? 0.5f * (float)m : (float)(1u << ((m >> 1) - 1u)) * (1.0f + 0.5f * (float)(m & 1u));
  return (code & 8u) ? -mag : mag;
}

// out[i][j][32c + e] = e2m1(element 32c + e of token j) * 2^(scale[c][j] - 127), fp32.
// A page's 32 KB of output is staged in shared memory (rows padded to 132 floats, so
// the 16-byte stores of a quarter warp fall in distinct banks) and written out as one
// contiguous run of 16-byte stores.
constexpr int kOutPitch = 128 + 4;

__global__ void __launch_bounds__(kPageThreads) dequant_pages_kernel(const uint8_t* __restrict__ payload,
                                                                     const uint8_t* __restrict__ scale,
                                                                     int64_t num_pages,
                                                                     const int32_t* __restrict__ page_ids,
                                                                     float* __restrict__ out, int32_t* status) {
  __shared__ __align__(16) float tile[64 * kOutPitch];
  const int64_t i = blockIdx.x;
  const int64_t p = page_of(page_ids, i, num_pages, status);
  if (p < 0) return;
  const int t = threadIdx.x, c = t >> 6, j = t & 63;
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(payload + p * kPagePayload) + t);  // row (c, j)
  const int e = (int)__ldg(scale + p * kPageScale + c * 64 + j) - 127;
  const float s = ldexpf(1.0f, e);  // exact power of two (subnormal below 2^-126)
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float4* st = reinterpret_cast<float4*>(tile + j * kOutPitch + 32 * c);
#pragma unroll
  for (int b = 0; b < 4; b++) {
    float v[8];
#pragma unroll
    for (int n = 0; n < 8; n++) v[n] = e2m1_value((w[b] >> (4 * n)) & 0xFu) * s;
    st[2 * b] = make_float4(v[0], v[1], v[2], v[3]);
    st[2 * b + 1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  __syncthreads();
  float4* dst = reinterpret_cast<float4*>(out + i * 64 * 128);
#pragma unroll
  for (int r = 0; r < 8; r++) {
    const int f = r * kPageThreads + t;  // float4 index in the page's [64][128] output
    const int row = f >> 5, col = f & 31;
    dst[f] = *reinterpret_cast<const float4*>(tile + row * kOutPitch + 4 * col);
  }
}

// Export (to_rows = true): rows_payload[i] = payload[page_ids[i]], rows_scale[i] =
// scale[page_ids[i]].  Import (to_rows = false): the reverse.
__global__ void __launch_bounds__(kPageThreads) copy_pages_kernel(uint8_t* payload, uint8_t* scale, int64_t num_pages,
                                                                  const int32_t* __restrict__ page_ids,
                                                                  uint8_t* rows_payload, uint8_t* rows_scale,
                                                                  bool to_rows, int32_t* status) {
  const int64_t i = blockIdx.x;
  const int64_t p = page_of(page_ids, i, num_pages, status);
  if (p < 0) return;
  const int t = threadIdx.x;
  uint4* cache_pay = reinterpret_cast<uint4*>(payload + p * kPagePayload);
  uint4* row_pay = reinterpret_cast<uint4*>(rows_payload + i * kPagePayload);
  if (to_rows)
    row_pay[t] = __ldg(cache_pay + t);
  else
    cache_pay[t] = __ldg(row_pay + t);
  if (t < (int)(kPageScale / 16)) {
    uint4* cache_sc = reinterpret_cast<uint4*>(scale + p * kPageScale);
    uint4* row_sc = reinterpret_cast<uint4*>(rows_scale + i * kPageScale);
    if (to_rows)
      row_sc[t] = __ldg(cache_sc + t);
    else
      cache_sc[t] = __ldg(row_sc + t);
  }
}

}  // namespace

cudaError_t launch_dequant_pages(const uint8_t* payload, const uint8_t* scale, int64_t num_pages,
                                 const int32_t* page_ids, int64_t n_pages, float* out, int32_t* status,
                                 cudaStream_t stream) {
  if (n_pages == 0) return cudaSuccess;
  dequant_pages_kernel<<<(unsigned)n_pages, kPageThreads, 0, stream>>>(payload, scale, num_pages, page_ids, out,
                                                                      status);
  return cudaGetLastError();
}

cudaError_t launch_copy_pages(uint8_t* payload, uint8_t* scale, int64_t num_pages, const int32_t* page_ids,
                              int64_t n_pages, uint8_t* rows_payload, uint8_t* rows_scale, bool to_rows,
                              int32_t* status, cudaStream_t stream) {
  if (n_pages == 0) return cudaSuccess;
  copy_pages_kernel<<<(unsigned)n_pages, kPageThreads, 0, stream>>>(payload, scale, num_pages, page_ids,
                                                                   rows_payload, rows_scale, to_rows, status);
  return cudaGetLastError();
}

}  // namespace fp4idx
