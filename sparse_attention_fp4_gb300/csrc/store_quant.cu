// K store (split FP4 and FP8 layouts) and query packing.
//
// [AMD] Enable FP4 indexer for Deepseek V4 -- Modifications, FP4 kernel adapters:
// the K writer is "fused RMSNorm, RoPE, Hadamard, FP4 quantization, and paged cache
// writes"; the query side is "Q RoPE/Hadamard/FP4 quantization".  Round to nearest
// even: dsv4.1-amd: KV cache layouts, FP4 indexer, compressor and router kernels --
// Summary.
//
// Mapping: a half-warp owns one 128-wide row, lane l (0..15) holds elements
// 8l..8l+7 (one 16-byte bf16 load).  Every floating-point operation is an explicit
// round-to-nearest intrinsic in a fixed order, so the bytes written do not depend
// on the compiler's contraction choices:
//   * RMSNorm: each lane sums its 8 squares left to right, the 16 partials are
//     combined by an xor butterfly (1,2,4,8), which is the pairwise tree in index
//     order; r = 1/sqrt(mean + eps) with IEEE sqrt and divide; y = (x*r)*w.
//   * RoPE on dims 0..63, pairs (i, i+32): lanes 0..3 hold the first halves, lanes
//     4..7 the second halves, exchanged with one xor-4 shuffle.
//   * Hadamard: stages h = 1,2,4 inside the lane, h = 8..64 across lanes (xor
//     1,2,4,8), then one multiply by fp32(1/sqrt(128)).
//   * UE8M0 per 32-element block (4 lanes): smallest e with 6*2^e >= amax, from the
//     exponent/mantissa bits of amax; e2m1 by the hardware RNE-satfinite convert,
//     the sign of zero taken from the input.
#include "launchers.cuh"
#include "schedule_build.cuh"

#include <atomic>

namespace fp4idx {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr uint32_t kInvSqrt128Bits = 0x3DB504F3u;  // fp32 nearest to 2^-3.5

__device__ __forceinline__ void unpack_bf16x8(uint4 u, float v[8]) {
  v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xFFFF0000u);
  v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xFFFF0000u);
  v[4] = __uint_as_float(u.z << 16); v[5] = __uint_as_float(u.z & 0xFFFF0000u);
  v[6] = __uint_as_float(u.w << 16); v[7] = __uint_as_float(u.w & 0xFFFF0000u);
}

__device__ __forceinline__ uint4 ldg16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// y <- RMSNorm(x) * w over the half-warp's row.
__device__ __forceinline__ void rmsnorm_row(float v[8], const float w[8], float eps) {
  float s = __fmul_rn(v[0], v[0]);
#pragma unroll
  for (int e = 1; e < 8; e++) s = __fadd_rn(s, __fmul_rn(v[e], v[e]));
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) s = __fadd_rn(s, __shfl_xor_sync(kFull, s, m));
  const float mean = __fmul_rn(s, 0.0078125f);
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
#pragma unroll
  for (int e = 0; e < 8; e++) v[e] = __fmul_rn(__fmul_rn(v[e], r), w[e]);
}

// RoPE on dims 0..63 with the bf16 table row at cs_row (cos 0..31 | sin 32..63).
__device__ __forceinline__ void rope_row(float v[8], const uint16_t* cs_row, int lh) {
  float p[8];
#pragma unroll
  for (int e = 0; e < 8; e++) p[e] = __shfl_xor_sync(kFull, v[e], 4);
  if (lh < 8) {
    float c[8], s[8];
    const int i0 = 8 * (lh & 3);
    unpack_bf16x8(ldg16(cs_row + i0), c);
    unpack_bf16x8(ldg16(cs_row + 32 + i0), s);
    if (lh < 4) {  // first half a: a*c - b*s
#pragma unroll
      for (int e = 0; e < 8; e++) v[e] = __fsub_rn(__fmul_rn(v[e], c[e]), __fmul_rn(p[e], s[e]));
    } else {       // second half b: b*c + a*s
#pragma unroll
      for (int e = 0; e < 8; e++) v[e] = __fadd_rn(__fmul_rn(v[e], c[e]), __fmul_rn(p[e], s[e]));
    }
  }
}

__device__ __forceinline__ void hadamard_row(float v[8], int lh) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int e = 0; e < 8; e++) {
      if (e & h) continue;
      const float a = v[e], b = v[e + h];
      v[e] = __fadd_rn(a, b);
      v[e + h] = __fsub_rn(a, b);
    }
  }
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
    const bool hi = (lh & m) != 0;
#pragma unroll
    for (int e = 0; e < 8; e++) {
      const float p = __shfl_xor_sync(kFull, v[e], m);
      v[e] = hi ? __fsub_rn(p, v[e]) : __fadd_rn(v[e], p);
    }
  }
  const float sc = __uint_as_float(kInvSqrt128Bits);
#pragma unroll
  for (int e = 0; e < 8; e++) v[e] = __fmul_rn(v[e], sc);
}

// UE8M0 byte (e + 127) of the smallest e with 6 * 2^e >= amax, e clamped to [-127, 127].
// amax = f * 2^E, f in [1,2): e = E - 2 + (f > 1.5); zero/subnormal amax -> byte 0.
__device__ __forceinline__ uint32_t ue8m0_byte(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int biased = (int)((b >> 23) & 0xFFu);
  if (biased == 0) return 0u;
  int byte = biased - 2 + (((b & 0x7FFFFFu) > 0x400000u) ? 1 : 0);
  byte = max(0, min(254, byte));
  return (uint32_t)byte;
}

// Two fp32 -> one byte of e2m1 (lo nibble = first), RNE, satfinite, sign of zero kept.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t out;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(out) : "f"(lo), "f"(hi));
  out &= 0x77u;
  out |= (__float_as_uint(lo) >> 31) << 3;
  out |= (__float_as_uint(hi) >> 31) << 7;
  return out;
}

// Two fp32 -> two bytes of e4m3 (byte 0 = first), RNE, satfinite, sign of zero kept.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t t;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(t) : "f"(lo), "f"(hi));
  uint32_t out = (uint32_t)t & 0x7F7Fu;
  out |= (__float_as_uint(lo) >> 31) << 7;
  out |= (__float_as_uint(hi) >> 31) << 15;
  return out;
}

// Quantise the half-warp's row (after the Hadamard) and return this lane's 4 payload
// bytes (elements 8l..8l+7) and its block's scale byte.
__device__ __forceinline__ uint32_t fp4_encode_lane(const float v[8], uint32_t& scale_byte) {
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; e++) amax = fmaxf(amax, fabsf(v[e]));
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
  scale_byte = ue8m0_byte(amax);
  const float inv = __uint_as_float((254u - scale_byte) << 23);  // 2^(127 - byte) = 2^-e
  uint32_t word = 0;
#pragma unroll
  for (int e = 0; e < 8; e += 2)
    word |= e2m1x2(__fmul_rn(v[e], inv), __fmul_rn(v[e + 1], inv)) << (4 * e);
  return word;
}

// ------------------------------------------------------------------ kernels
constexpr int kRowsPerBlock = 16;  // 256 threads, a half-warp per row

// K store of the 16 rows of block `block` (a half-warp per row).
__device__ __forceinline__ void store_k_block(int64_t block, const uint16_t* __restrict__ k, int64_t n_rows,
                                              const int32_t* __restrict__ positions,
                                              const int32_t* __restrict__ slots, const uint16_t* __restrict__ norm_w,
                                              float eps, const uint16_t* __restrict__ cos_sin, int32_t max_pos,
                                              uint8_t* __restrict__ payload, uint8_t* __restrict__ scale,
                                              int64_t num_pages, int32_t* status) {
  const int lh = threadIdx.x & 15;
  const int64_t n = block * kRowsPerBlock + (threadIdx.x >> 4);
  const bool in_range = n < n_rows;
  int32_t slot = -1, pos = 0;
  if (in_range) {
    slot = __ldg(slots + n);
    pos = __ldg(positions + n);
  }
  bool store = in_range && slot >= 0;
  if (store && (int64_t)slot >= num_pages * kPage) {
    if (lh == 0) record_error(status, FP4IDX_ERR_BAD_PAGE);
    store = false;
  }
  if (in_range && (pos < 0 || pos >= max_pos)) {
    if (lh == 0 && slot >= 0) record_error(status, FP4IDX_ERR_BAD_POSITION);
    store = false;
    pos = 0;
  }
  float v[8], w[8];
  if (in_range) unpack_bf16x8(ldg16(k + n * kHeadDim + 8 * lh), v);
  else {
#pragma unroll
    for (int e = 0; e < 8; e++) v[e] = 0.0f;
  }
  unpack_bf16x8(ldg16(norm_w + 8 * lh), w);
  rmsnorm_row(v, w, eps);
  rope_row(v, cos_sin + (int64_t)pos * kRope, lh);
  hadamard_row(v, lh);
  uint32_t sb;
  const uint32_t word = fp4_encode_lane(v, sb);
  if (store) {
    const int64_t page = slot >> 6;
    const int j = slot & 63;
    const int c = lh >> 2;
    uint8_t* dst = payload + ((page * 4 + c) * kPage + j) * 16 + (lh & 3) * 4;
    *reinterpret_cast<uint32_t*>(dst) = word;
    if ((lh & 3) == 0) scale[(page * 4 + c) * kPage + j] = (uint8_t)sb;
  }
}

__global__ void __launch_bounds__(256) store_k_kernel(
    const uint16_t* __restrict__ k, int64_t n_rows, const int32_t* __restrict__ positions,
    const int32_t* __restrict__ slots, const uint16_t* __restrict__ norm_w, float eps,
    const uint16_t* __restrict__ cos_sin, int32_t max_pos, uint8_t* __restrict__ payload,
    uint8_t* __restrict__ scale, int64_t num_pages, int32_t* status) {
  store_k_block(blockIdx.x, k, n_rows, positions, slots, norm_w, eps, cos_sin, max_pos, payload, scale, num_pages,
                status);
}

__global__ void __launch_bounds__(256) store_k_fp8_kernel(
    const uint16_t* __restrict__ k, int64_t n_rows, const int32_t* __restrict__ positions,
    const int32_t* __restrict__ slots, const uint16_t* __restrict__ norm_w, float eps,
    const uint16_t* __restrict__ cos_sin, int32_t max_pos, uint8_t* __restrict__ pages, int64_t num_pages,
    int32_t* status) {
  const int lh = threadIdx.x & 15;
  const int64_t n = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 4);
  const bool in_range = n < n_rows;
  int32_t slot = -1, pos = 0;
  if (in_range) {
    slot = __ldg(slots + n);
    pos = __ldg(positions + n);
  }
  bool store = in_range && slot >= 0;
  if (store && (int64_t)slot >= num_pages * kPage) {
    if (lh == 0) record_error(status, FP4IDX_ERR_BAD_PAGE);
    store = false;
  }
  if (in_range && (pos < 0 || pos >= max_pos)) {
    if (lh == 0 && slot >= 0) record_error(status, FP4IDX_ERR_BAD_POSITION);
    store = false;
    pos = 0;
  }
  float v[8], w[8];
  if (in_range) unpack_bf16x8(ldg16(k + n * kHeadDim + 8 * lh), v);
  else {
#pragma unroll
    for (int e = 0; e < 8; e++) v[e] = 0.0f;
  }
  unpack_bf16x8(ldg16(norm_w + 8 * lh), w);
  rmsnorm_row(v, w, eps);
  rope_row(v, cos_sin + (int64_t)pos * kRope, lh);
  hadamard_row(v, lh);
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; e++) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, m));
  const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  uint2 out;
  out.x = e4m3x2(__fdiv_rn(v[0], s), __fdiv_rn(v[1], s)) | (e4m3x2(__fdiv_rn(v[2], s), __fdiv_rn(v[3], s)) << 16);
  out.y = e4m3x2(__fdiv_rn(v[4], s), __fdiv_rn(v[5], s)) | (e4m3x2(__fdiv_rn(v[6], s), __fdiv_rn(v[7], s)) << 16);
  if (store) {
    const int64_t page = slot >> 6;
    const int j = slot & 63;
    uint8_t* base = pages + page * (int64_t)FP4IDX_FP8_PAGE_BYTES;
    *reinterpret_cast<uint2*>(base + j * kHeadDim + lh * 8) = out;
    if (lh == 0) *reinterpret_cast<float*>(base + kPage * kHeadDim + j * 4) = s;
  }
}

// Q quant of the 16 (row, head) vectors of block `block`.
__device__ __forceinline__ void quant_q_block(int64_t block, const uint16_t* __restrict__ q, int64_t n_rows,
                                              const int32_t* __restrict__ q_positions,
                                              const uint16_t* __restrict__ cos_sin, int32_t max_pos,
                                              uint8_t* __restrict__ q_payload, uint8_t* __restrict__ q_scale,
                                              int32_t* status) {
  // one "row" per (query row t, head h); 64 heads
  const int lh = threadIdx.x & 15;
  const int64_t th = block * kRowsPerBlock + (threadIdx.x >> 4);
  const int64_t total = n_rows * kHeads;
  const bool in_range = th < total;
  const int64_t t = th >> 6;
  const int h = (int)(th & 63);
  int32_t pos = in_range ? __ldg(q_positions + t) : 0;
  bool store = in_range;
  if (in_range && (pos < 0 || pos >= max_pos)) {
    if (lh == 0 && h == 0) record_error(status, FP4IDX_ERR_BAD_POSITION);
    store = false;
    pos = 0;
  }
  float v[8];
  if (in_range) unpack_bf16x8(ldg16(q + th * kHeadDim + 8 * lh), v);
  else {
#pragma unroll
    for (int e = 0; e < 8; e++) v[e] = 0.0f;
  }
  rope_row(v, cos_sin + (int64_t)pos * kRope, lh);
  hadamard_row(v, lh);
  uint32_t sb;
  const uint32_t word = fp4_encode_lane(v, sb);
  if (store) {
    const int c = lh >> 2;
    uint8_t* dst = q_payload + ((t * 4 + c) * kHeads + h) * 16 + (lh & 3) * 4;
    *reinterpret_cast<uint32_t*>(dst) = word;
    if ((lh & 3) == 0) q_scale[(t * 4 + c) * kHeads + h] = (uint8_t)sb;
  }
}

__global__ void __launch_bounds__(256) quant_q_kernel(
    const uint16_t* __restrict__ q, int64_t n_rows, const int32_t* __restrict__ q_positions,
    const uint16_t* __restrict__ cos_sin, int32_t max_pos, uint8_t* __restrict__ q_payload,
    uint8_t* __restrict__ q_scale, int32_t* status) {
  quant_q_block(blockIdx.x, q, n_rows, q_positions, cos_sin, max_pos, q_payload, q_scale, status);
}

// The decode step's preparation in one launch: block 0 builds the logits schedule (the
// build of schedule_build.cuh with 256 threads), the next kb blocks store the new K rows,
// the rest pack the queries -- the launches of fp4idx_build_schedule, fp4idx_store_k and
// fp4idx_quant_q, doing the same work, with the same results, in one grid.  Every block
// signals at its start that a programmatic dependent launch (the logits kernel) may
// begin its own set-up; that launch waits for this grid's results before reading them.
struct PrepareParams {
  const uint16_t* k;
  int64_t n_new;
  const int32_t* positions;
  const int32_t* slots;
  const uint16_t* norm_w;
  float eps;
  const uint16_t* q;
  int64_t n_rows;
  const int32_t* q_positions;
  const uint16_t* cos_sin;
  int32_t max_pos;
  uint8_t* payload;
  uint8_t* scale;
  int64_t num_pages;
  uint8_t* q_payload;
  uint8_t* q_scale;
  const int32_t* context_lens;
  const int32_t* row_seq;
  int32_t num_ctas;
  void* schedule;
  int32_t* status;
  int64_t kb;  // blocks of the K store
};

__global__ void __launch_bounds__(256) prepare_step_kernel(const PrepareParams p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == 0) {
    build_schedule_block<256>(p.context_lens, p.row_seq, (int32_t)p.n_rows, p.num_ctas, p.schedule);
  } else if ((int64_t)blockIdx.x <= p.kb) {
    store_k_block(blockIdx.x - 1, p.k, p.n_new, p.positions, p.slots, p.norm_w, p.eps, p.cos_sin, p.max_pos,
                  p.payload, p.scale, p.num_pages, p.status);
  } else {
    quant_q_block(blockIdx.x - 1 - p.kb, p.q, p.n_rows, p.q_positions, p.cos_sin, p.max_pos, p.q_payload,
                  p.q_scale, p.status);
  }
}

// FP8 query pack (the comparison path of the 132 B/token layout): per (row t, head h), RoPE
// and the Hadamard as for the FP4 pack, then the K side's FP8 rule -- one fp32 scale
// s = amax / 448 (1 when amax = 0) and e4m3 = RNE-satfinite(x / s).  Layout q8[t][c][h][16]
// (chunk c = elements 16c .. 16c + 15), q8_scale[t][h].
__global__ void __launch_bounds__(256) quant_q_fp8_kernel(
    const uint16_t* __restrict__ q, int64_t n_rows, const int32_t* __restrict__ q_positions,
    const uint16_t* __restrict__ cos_sin, int32_t max_pos, uint8_t* __restrict__ q8, float* __restrict__ q8_scale,
    int32_t* status) {
  const int lh = threadIdx.x & 15;
  const int64_t th = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 4);
  const bool in_range = th < n_rows * kHeads;
  const int64_t t = th >> 6;
  const int h = (int)(th & 63);
  int32_t pos = in_range ? __ldg(q_positions + t) : 0;
  bool store = in_range;
  if (in_range && (pos < 0 || pos >= max_pos)) {
    if (lh == 0 && h == 0) record_error(status, FP4IDX_ERR_BAD_POSITION);
    store = false;
    pos = 0;
  }
  float v[8];
  if (in_range) unpack_bf16x8(ldg16(q + th * kHeadDim + 8 * lh), v);
  else {
#pragma unroll
    for (int e = 0; e < 8; e++) v[e] = 0.0f;
  }
  rope_row(v, cos_sin + (int64_t)pos * kRope, lh);
  hadamard_row(v, lh);
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; e++) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, m));
  const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  uint2 out;
  out.x = e4m3x2(__fdiv_rn(v[0], s), __fdiv_rn(v[1], s)) | (e4m3x2(__fdiv_rn(v[2], s), __fdiv_rn(v[3], s)) << 16);
  out.y = e4m3x2(__fdiv_rn(v[4], s), __fdiv_rn(v[5], s)) | (e4m3x2(__fdiv_rn(v[6], s), __fdiv_rn(v[7], s)) << 16);
  if (store) {
    // elements 8 lh .. 8 lh + 7: chunk lh / 2, bytes 8 (lh & 1) .. of that chunk's 16
    *reinterpret_cast<uint2*>(q8 + ((t * 8 + (lh >> 1)) * kHeads + h) * 16 + 8 * (lh & 1)) = out;
    if (lh == 0) q8_scale[t * kHeads + h] = s;
  }
}

// Head weights of query row t: w[t][h] = w_scale * sum_d hidden[t][d] * w_proj[h][d], bf16
// inputs, fp32 accumulation ([P1] Summary: indexer_head_weights runs a batch-invariant
// split-K bf16 GEMV whose result stays in fp32).  A CTA takes row t and heads 8g .. 8g+7;
// its 8 warps split the hidden dimension: with M = hidden_dim / 256 chunks, warp w takes
// chunks [w M / 8, (w + 1) M / 8).  Fixed order, whatever the batch: lane l of warp w adds
// the products d = 256 m + 8 l + i of its chunks, m then i ascending (every bf16 product is
// exact in fp32, one rounding per addition); then the 32 lanes pairwise at distances 16, 8,
// 4, 2, 1; then the 8 warp sums in warp order; then one rounding for the scale.  Each warp
// keeps four heads' sums side by side, so that their weight loads are in flight together.
__device__ __forceinline__ void head_weights_part(int64_t t, int g, const uint16_t* __restrict__ hidden, int32_t dim,
                                                  const uint16_t* __restrict__ w_proj, float w_scale,
                                                  float* __restrict__ w_out, uint16_t* hs, float* part) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint4* src = reinterpret_cast<const uint4*>(hidden + t * dim);
  for (int i = threadIdx.x; i < dim / 8; i += 256) reinterpret_cast<uint4*>(hs)[i] = __ldg(src + i);
  __syncthreads();
  const int M = dim / 256;
  const int m0 = warp * M / 8, m1 = (warp + 1) * M / 8;
  float acc[8];
#pragma unroll
  for (int hp = 0; hp < 2; hp++) {
    const uint16_t* wr = w_proj + (int64_t)(8 * g + 4 * hp) * dim;
    float a4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
    for (int m = m0; m < m1; m++) {
      const int d = 256 * m + 8 * lane;
      uint4 wv[4];
#pragma unroll
      for (int j = 0; j < 4; j++) wv[j] = ldg16(wr + (int64_t)j * dim + d);
      float a[8];
      unpack_bf16x8(*reinterpret_cast<const uint4*>(hs + d), a);
#pragma unroll
      for (int j = 0; j < 4; j++) {
        float b[8];
        unpack_bf16x8(wv[j], b);
#pragma unroll
        for (int i = 0; i < 8; i++) a4[j] = __fadd_rn(a4[j], __fmul_rn(a[i], b[i]));
      }
    }
#pragma unroll
    for (int j = 0; j < 4; j++) acc[4 * hp + j] = a4[j];
  }
#pragma unroll
  for (int j = 0; j < 8; j++) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[j] = __fadd_rn(acc[j], __shfl_xor_sync(0xFFFFFFFFu, acc[j], o));
  }
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < 8; j++) part[warp * 8 + j] = acc[j];
  }
  __syncthreads();
  if (threadIdx.x < 8) {
    float sum = part[threadIdx.x];
    for (int w = 1; w < 8; w++) sum = __fadd_rn(sum, part[w * 8 + threadIdx.x]);
    w_out[t * kHeads + 8 * g + threadIdx.x] = __fmul_rn(sum, w_scale);
  }
}

// One launch: blocks [0, q_blocks) quantise the queries, blocks q_blocks + 8t + g compute
// row t's head weights 8g .. 8g + 7.
__global__ void __launch_bounds__(256) quant_q_w_kernel(
    const uint16_t* __restrict__ q, int64_t n_rows, const int32_t* __restrict__ q_positions,
    const uint16_t* __restrict__ cos_sin, int32_t max_pos, uint8_t* __restrict__ q_payload,
    uint8_t* __restrict__ q_scale, int64_t q_blocks, const uint16_t* __restrict__ hidden, int32_t dim,
    const uint16_t* __restrict__ w_proj, float w_scale, float* __restrict__ w_out, int32_t* status) {
  extern __shared__ __align__(16) uint16_t hidden_row[];
  __shared__ float part[64];
  if ((int64_t)blockIdx.x < q_blocks)
    quant_q_block(blockIdx.x, q, n_rows, q_positions, cos_sin, max_pos, q_payload, q_scale, status);
  else
    head_weights_part(((int64_t)blockIdx.x - q_blocks) >> 3, (int)(((int64_t)blockIdx.x - q_blocks) & 7), hidden, dim,
                      w_proj, w_scale, w_out, hidden_row, part);
}

inline unsigned grid_for(int64_t rows) { return (unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock); }

// These kernels need no shared memory, but they run just before the logits kernel, which
// needs nearly all of it: asking for the largest shared-memory carveout keeps the SMs in
// that configuration, so the logits CTAs launch without a carveout change.
template <class K>
cudaError_t prefer_max_shared(K kernel, std::atomic<bool>* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev].load()) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(true);
  return e;
}
std::atomic<bool> g_carve_store[64], g_carve_store_fp8[64], g_carve_quant[64], g_carve_quant_w[64];

}  // namespace

cudaError_t launch_store_k(const uint16_t* k, int64_t n_rows, const int32_t* positions, const int32_t* slots,
                           const uint16_t* norm_w, float eps, const uint16_t* cos_sin, int32_t max_pos,
                           uint8_t* payload, uint8_t* scale, int64_t num_pages, int32_t* status,
                           cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  cudaError_t e = prefer_max_shared(store_k_kernel, g_carve_store);
  if (e != cudaSuccess) return e;
  store_k_kernel<<<grid_for(n_rows), 256, 0, stream>>>(k, n_rows, positions, slots, norm_w, eps, cos_sin,
                                                        max_pos, payload, scale, num_pages, status);
  return cudaGetLastError();
}

cudaError_t launch_store_k_fp8(const uint16_t* k, int64_t n_rows, const int32_t* positions, const int32_t* slots,
                               const uint16_t* norm_w, float eps, const uint16_t* cos_sin, int32_t max_pos,
                               uint8_t* pages, int64_t num_pages, int32_t* status, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  cudaError_t e = prefer_max_shared(store_k_fp8_kernel, g_carve_store_fp8);
  if (e != cudaSuccess) return e;
  store_k_fp8_kernel<<<grid_for(n_rows), 256, 0, stream>>>(k, n_rows, positions, slots, norm_w, eps, cos_sin,
                                                            max_pos, pages, num_pages, status);
  return cudaGetLastError();
}

cudaError_t launch_quant_q(const uint16_t* q, int64_t n_rows, const int32_t* q_positions, const uint16_t* cos_sin,
                           int32_t max_pos, uint8_t* q_payload, uint8_t* q_scale, int32_t* status,
                           cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  cudaError_t e = prefer_max_shared(quant_q_kernel, g_carve_quant);
  if (e != cudaSuccess) return e;
  quant_q_kernel<<<grid_for(n_rows * kHeads), 256, 0, stream>>>(q, n_rows, q_positions, cos_sin, max_pos,
                                                                 q_payload, q_scale, status);
  return cudaGetLastError();
}

cudaError_t launch_prepare_step(const uint16_t* k, int64_t n_new, const int32_t* positions, const int32_t* slots,
                                const uint16_t* norm_w, float eps, const uint16_t* q, int64_t n_rows,
                                const int32_t* q_positions, const uint16_t* cos_sin, int32_t max_pos,
                                uint8_t* payload, uint8_t* scale, int64_t num_pages, uint8_t* q_payload,
                                uint8_t* q_scale, const int32_t* context_lens, const int32_t* row_seq,
                                int32_t num_ctas, void* schedule, int32_t* status, cudaStream_t stream) {
  static std::atomic<bool> done[64];
  cudaError_t e = prefer_max_shared(prepare_step_kernel, done);
  if (e != cudaSuccess) return e;
  PrepareParams p;
  p.k = k;
  p.n_new = n_new;
  p.positions = positions;
  p.slots = slots;
  p.norm_w = norm_w;
  p.eps = eps;
  p.q = q;
  p.n_rows = n_rows;
  p.q_positions = q_positions;
  p.cos_sin = cos_sin;
  p.max_pos = max_pos;
  p.payload = payload;
  p.scale = scale;
  p.num_pages = num_pages;
  p.q_payload = q_payload;
  p.q_scale = q_scale;
  p.context_lens = context_lens;
  p.row_seq = row_seq;
  p.num_ctas = num_ctas;
  p.schedule = schedule;
  p.status = status;
  p.kb = (n_new + kRowsPerBlock - 1) / kRowsPerBlock;
  const int64_t qb = (n_rows * kHeads + kRowsPerBlock - 1) / kRowsPerBlock;
  prepare_step_kernel<<<(unsigned)(1 + p.kb + qb), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quant_q_fp8(const uint16_t* q, int64_t n_rows, const int32_t* q_positions, const uint16_t* cos_sin,
                               int32_t max_pos, uint8_t* q8, float* q8_scale, int32_t* status, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  quant_q_fp8_kernel<<<grid_for(n_rows * kHeads), 256, 0, stream>>>(q, n_rows, q_positions, cos_sin, max_pos, q8,
                                                                   q8_scale, status);
  return cudaGetLastError();
}

cudaError_t launch_quant_q_w(const uint16_t* q, int64_t n_rows, const int32_t* q_positions, const uint16_t* cos_sin,
                             int32_t max_pos, uint8_t* q_payload, uint8_t* q_scale, const uint16_t* hidden,
                             int32_t dim, const uint16_t* w_proj, float w_scale, float* w_out, int32_t* status,
                             cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  cudaError_t e = prefer_max_shared(quant_q_w_kernel, g_carve_quant_w);
  if (e != cudaSuccess) return e;
  const int64_t q_blocks = grid_for(n_rows * kHeads);
  quant_q_w_kernel<<<(unsigned)(q_blocks + 8 * n_rows), 256, (size_t)dim * sizeof(uint16_t), stream>>>(
      q, n_rows, q_positions, cos_sin, max_pos, q_payload, q_scale, q_blocks, hidden, dim, w_proj, w_scale, w_out,
      status);
  return cudaGetLastError();
}

}  // namespace fp4idx
