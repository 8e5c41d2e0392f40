// K store (split FP4 and FP8 layouts) and query packing.
//
// [AMD] Enable FP4 indexer for Deepseek V4 -- Modifications, FP4 kernel adapters:
// the K writer is "fused RMSNorm, RoPE, Hadamard, FP4 quantization, and paged cache
// writes"; the query side is "Q RoPE/Hadamard/FP4 quantization".  Round to nearest
// even: dsv4.1-amd: KV cache layouts, FP4 indexer, compressor and router kernels --
// Summary.
//
// Two mappings of a 128-wide row onto lanes.  The query packers give a half-warp a row,
// lane l (0..15) holding elements 8l..8l+7 (one 16-byte bf16 load); the K stores give a
// quarter-warp a row (the qw helpers below), with fewer shuffles and redundant per-row
// steps per row.  Every floating-point operation is an explicit round-to-nearest
// intrinsic in a fixed order, so the bytes written do not depend on the compiler's
// contraction choices or on the mapping:
//   * RMSNorm: each group of 8 squares summed left to right, the 16 group sums combined
//     by the pairwise tree in index order; r = 1/sqrt(mean + eps) with IEEE sqrt and
//     divide; y = (x*r)*w.
//   * RoPE on dims 0..63, pairs (i, i+32): a' = a*c - b*s, b' = b*c + a*s, each product
//     rounded.
//   * Hadamard: stages h = 1, 2, 4, ..., 64 in that order, (a, b) -> (a+b, a-b), then one
//     multiply by fp32(1/sqrt(128)).
//   * UE8M0 per 32-element block: smallest e with 6*2^e >= amax, from the
//     exponent/mantissa bits of amax; e2m1 by the hardware RNE-satfinite convert,
//     which keeps the sign of a value that rounds to zero.
#include "launchers.cuh"
#include "schedule_build.cuh"

#include <algorithm>
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

// The converts below round to nearest even, saturate to the largest finite value, and
// keep the sign of an input that rounds to zero (e2m1 code 8, e4m3 byte 0x80), which is
// the encoding's rule for negative values too small for the grid.
// Eight fp32 -> one word of e2m1 (nibble i = value i).
__device__ __forceinline__ uint32_t e2m1x8(float v0, float v1, float v2, float v3, float v4, float v5, float v6,
                                           float v7) {
  uint32_t out;
  asm("{\n\t.reg .b8 a, b, c, d;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 a, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 d, %8, %7;\n\t"
      "mov.b32 %0, {a, b, c, d};\n\t}"
      : "=r"(out) : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return out;
}

// Two fp32 -> two bytes of e4m3 (byte 0 = first).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t t;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(t) : "f"(lo), "f"(hi));
  return (uint32_t)t;
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
  float y[8];
#pragma unroll
  for (int e = 0; e < 8; e++) y[e] = __fmul_rn(v[e], inv);
  return e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
}

// ------------------------------------------------------------------ quarter-warp row transform
// The K store maps a row to four lanes (eight rows a warp): lane l of the quarter holds the
// elements i = 32 m + 8 l + e (m = 0..3 its four 16-byte chunks, e = 0..7), as float pairs
// x[m][p] = (element 32 m + 8 l + 2 p, element 32 m + 8 l + 2 p + 1).  Index bits 0-2 and 5-6
// are in the lane's registers, bits 3-4 across the quarter, so that
//   * RoPE's pairs (i, i + 32) sit in one lane (chunks m = 0 and 1), and every lane rotates
//     eight of them with its own 16 bytes of cos and of sin;
//   * five of the seven Hadamard stages run inside the lane, two across it;
//   * the operations on pairs are the packed f32x2 forms (add/sub/mul/fma .rn), one
//     rounding per element as in the scalar chain, except where a product feeds a sum
//     (RoPE): there the scalar forms keep the two roundings apart.
// The order of every rounded operation is the one the half-warp helpers above follow:
// squares summed left to right within each group of eight, the sixteen group sums
// combined by the pairwise tree in index order, the Hadamard stages h = 1 .. 64 in turn.
namespace qw {

struct f2 {
  float x, y;
};

__device__ __forceinline__ uint64_t pk(f2 a) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
  return r;
}
__device__ __forceinline__ f2 upk(uint64_t r) {
  f2 a;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
  return a;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)));
  return upk(d);
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)));
  return upk(d);
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)));
  return upk(d);
}
// a * b + c with one rounding; with b = (+-1, +-1) it is the correctly rounded c +- a.
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)), "l"(pk(c)));
  return upk(d);
}

__device__ __forceinline__ void unpack(uint4 u, f2 v[4]) {
  v[0] = {__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u)};
  v[1] = {__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u)};
  v[2] = {__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xFFFF0000u)};
  v[3] = {__uint_as_float(u.w << 16), __uint_as_float(u.w & 0xFFFF0000u)};
}

// y <- RMSNorm(x) * w.
__device__ __forceinline__ void rmsnorm(f2 x[4][4], const f2 w[4][4], float eps) {
  float g[4];  // the sums of the lane's groups 4 m + l, left to right
#pragma unroll
  for (int m = 0; m < 4; m++) {
    const f2 a = mul2(x[m][0], x[m][0]), b = mul2(x[m][1], x[m][1]);
    const f2 c = mul2(x[m][2], x[m][2]), d = mul2(x[m][3], x[m][3]);
    float s = __fadd_rn(a.x, a.y);
    s = __fadd_rn(s, b.x); s = __fadd_rn(s, b.y);
    s = __fadd_rn(s, c.x); s = __fadd_rn(s, c.y);
    s = __fadd_rn(s, d.x); s = __fadd_rn(s, d.y);
    g[m] = s;
  }
  // tree levels 1 and 2 pair groups 4m+l with 4m+(l^1), then with 4m+(l^2): across the quarter
  f2 p = {g[0], g[1]}, q = {g[2], g[3]};
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    const f2 pp = {__shfl_xor_sync(kFull, p.x, o), __shfl_xor_sync(kFull, p.y, o)};
    const f2 qq = {__shfl_xor_sync(kFull, q.x, o), __shfl_xor_sync(kFull, q.y, o)};
    p = add2(p, pp);
    q = add2(q, qq);
  }
  // levels 3 and 4: (m0 + m1) + (m2 + m3), now inside the lane
  const float s = __fadd_rn(__fadd_rn(p.x, p.y), __fadd_rn(q.x, q.y));
  const float mean = __fmul_rn(s, 0.0078125f);
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
  const f2 rr = {r, r};
#pragma unroll
  for (int m = 0; m < 4; m++)
#pragma unroll
    for (int j = 0; j < 4; j++) x[m][j] = mul2(mul2(x[m][j], rr), w[m][j]);
}

// RoPE on dims 0..63: the lane's pairs (32 * 0 + 8 l + e, 32 * 1 + 8 l + e), with cos and
// sin of index 8 l + e from the bf16 table row.  Scalar operations: a packed product
// feeding a packed sum may be fused into one rounding by the code generator, which would
// change the result, so each product and each sum here is its own rounded instruction.
__device__ __forceinline__ void rope(f2 x[4][4], uint4 cos_raw, uint4 sin_raw) {
  f2 c[4], s[4];
  unpack(cos_raw, c);
  unpack(sin_raw, s);
#pragma unroll
  for (int j = 0; j < 4; j++) {
    const f2 a = x[0][j], b = x[1][j];
    x[0][j] = {__fsub_rn(__fmul_rn(a.x, c[j].x), __fmul_rn(b.x, s[j].x)),
               __fsub_rn(__fmul_rn(a.y, c[j].y), __fmul_rn(b.y, s[j].y))};
    x[1][j] = {__fadd_rn(__fmul_rn(b.x, c[j].x), __fmul_rn(a.x, s[j].x)),
               __fadd_rn(__fmul_rn(b.y, c[j].y), __fmul_rn(a.y, s[j].y))};
  }
}

__device__ __forceinline__ void hadamard(f2 x[4][4], int l) {
  // h = 1: inside each pair
#pragma unroll
  for (int m = 0; m < 4; m++)
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const float a = x[m][j].x, b = x[m][j].y;
      x[m][j] = {__fadd_rn(a, b), __fsub_rn(a, b)};
    }
  // h = 2, 4: pairs j and j + h/2
#pragma unroll
  for (int hj = 1; hj <= 2; hj <<= 1)
#pragma unroll
    for (int m = 0; m < 4; m++)
#pragma unroll
      for (int j = 0; j < 4; j++) {
        if (j & hj) continue;
        const f2 a = x[m][j], b = x[m][j + hj];
        x[m][j] = add2(a, b);
        x[m][j + hj] = sub2(a, b);
      }
  // h = 8, 16: lanes l and l ^ (h / 8); the lane with the bit set keeps partner - own
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    const float sg = (l & o) ? -1.0f : 1.0f;
    const f2 sgn = {sg, sg};
#pragma unroll
    for (int m = 0; m < 4; m++)
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const f2 p = {__shfl_xor_sync(kFull, x[m][j].x, o), __shfl_xor_sync(kFull, x[m][j].y, o)};
        x[m][j] = fma2(x[m][j], sgn, p);
      }
  }
  // h = 32, 64: chunks m and m + h/32
#pragma unroll
  for (int hm = 1; hm <= 2; hm <<= 1)
#pragma unroll
    for (int m = 0; m < 4; m++) {
      if (m & hm) continue;
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const f2 a = x[m][j], b = x[m + hm][j];
        x[m][j] = add2(a, b);
        x[m + hm][j] = sub2(a, b);
      }
    }
  const float sc = __uint_as_float(kInvSqrt128Bits);
  const f2 sc2 = {sc, sc};
#pragma unroll
  for (int m = 0; m < 4; m++)
#pragma unroll
    for (int j = 0; j < 4; j++) x[m][j] = mul2(x[m][j], sc2);
}

// FP4 encoding of block m (elements 32 m .. 32 m + 31, eight of them in each lane of the
// quarter): this lane's 4 payload bytes and the block's scale byte.
__device__ __forceinline__ uint32_t fp4_block(const f2 xm[4], uint32_t& scale_byte) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; j++) amax = fmaxf(amax, fmaxf(fabsf(xm[j].x), fabsf(xm[j].y)));
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
  scale_byte = ue8m0_byte(amax);
  const float inv = __uint_as_float((254u - scale_byte) << 23);  // 2^-e, exact scaling
  const f2 inv2 = {inv, inv};
  f2 y[4];
#pragma unroll
  for (int j = 0; j < 4; j++) y[j] = mul2(xm[j], inv2);
  return e2m1x8(y[0].x, y[0].y, y[1].x, y[1].y, y[2].x, y[2].y, y[3].x, y[3].y);
}

}  // namespace qw

// ------------------------------------------------------------------ K store kernels
constexpr int kRowsPerBlock = 16;        // half-warp mapping (query packing): 256 threads
constexpr int kStoreRowsPerBlock = 64;   // quarter-warp mapping (K store): 256 threads

// Checks of one K-store row: the row is written only with a slot in the cache and a
// position inside the table (a negative slot is padding and skipped silently).  Returns
// whether to write; `pos` is clamped to 0 for the table read of a rejected row.
__device__ __forceinline__ bool store_row_ok(bool in_range, int32_t slot, int32_t& pos, int64_t num_pages,
                                             int32_t max_pos, bool reporter, int32_t* status) {
  bool store = in_range && slot >= 0;
  if (store && (int64_t)slot >= num_pages * kPage) {
    if (reporter) record_error(status, FP4IDX_ERR_BAD_PAGE);
    store = false;
  }
  if (in_range && (pos < 0 || pos >= max_pos)) {
    if (reporter && slot >= 0) record_error(status, FP4IDX_ERR_BAD_POSITION);
    store = false;
  }
  if (!store) pos = 0;
  return store;
}

struct StoreArgs {
  const uint16_t* k;
  int64_t n_rows;
  const int32_t* positions;
  const int32_t* slots;
  const uint16_t* norm_w;
  float eps;
  const uint16_t* cos_sin;
  int32_t max_pos;
  int64_t num_pages;
  int32_t* status;
};

// The chain of one K row up to the Hadamard, on the quarter-warp mapping: x holds the
// lane's 32 values on return.  cs holds the lane's 8 cos and 8 sin of the row's position.
__device__ __forceinline__ void k_chain_qw(qw::f2 x[4][4], const uint4 raw[4], const qw::f2 w[4][4], float eps,
                                           const uint4 cs[2], int l) {
#pragma unroll
  for (int m = 0; m < 4; m++) qw::unpack(raw[m], x[m]);
  qw::rmsnorm(x, w, eps);
  qw::rope(x, cs[0], cs[1]);
  qw::hadamard(x, l);
}

__device__ __forceinline__ void load_cs(const uint16_t* cos_sin, int32_t pos, int l, uint4 cs[2]) {
  const uint16_t* row = cos_sin + (int64_t)pos * kRope;
  cs[0] = __ldg(reinterpret_cast<const uint4*>(row + 8 * l));
  cs[1] = __ldg(reinterpret_cast<const uint4*>(row + 32 + 8 * l));
}

// The lane's 32 norm weights (elements 32 m + 8 l + e) from the block's fp32 copy in
// shared memory: eight 16-byte loads, each a broadcast to the warp's eight rows.
__device__ __forceinline__ void norm_w_of_lane(const float* wsm, int l, qw::f2 w[4][4]) {
#pragma unroll
  for (int m = 0; m < 4; m++) {
    const float4 u0 = *reinterpret_cast<const float4*>(wsm + 32 * m + 8 * l);
    const float4 u1 = *reinterpret_cast<const float4*>(wsm + 32 * m + 8 * l + 4);
    w[m][0] = {u0.x, u0.y};
    w[m][1] = {u0.z, u0.w};
    w[m][2] = {u1.x, u1.y};
    w[m][3] = {u1.z, u1.w};
  }
}

// One row of the K store as a quarter-warp sees it: its raw K, cos/sin and destination.
struct StoreRow {
  uint4 raw[4];
  uint4 cs[2];
  int32_t slot;
  bool store;
};

// Loads of row n except the table (the position decides which table row): slot and
// position checked, raw K.  Rows past the end are not stored and read table row 0.
__device__ __forceinline__ int32_t load_row_head(const StoreArgs& a, int64_t n, int l, bool reporter, StoreRow& r) {
  const bool in_range = n < a.n_rows;
  int32_t pos = 0;
  r.slot = -1;
  if (in_range) {
    r.slot = __ldg(a.slots + n);
    pos = __ldg(a.positions + n);
    const uint16_t* row = a.k + n * kHeadDim + 8 * l;
#pragma unroll
    for (int m = 0; m < 4; m++) r.raw[m] = __ldg(reinterpret_cast<const uint4*>(row + 32 * m));
  } else {
#pragma unroll
    for (int m = 0; m < 4; m++) r.raw[m] = make_uint4(0u, 0u, 0u, 0u);
  }
  r.store = store_row_ok(in_range, r.slot, pos, a.num_pages, a.max_pos, reporter, a.status);
  return pos;
}

// Rows u * 8 + (lane / 4) for units u = first, first + stride, ...: every lane of a warp
// takes the same number of iterations, as the shuffles need.  Software pipeline, one row
// deep: while row i is computed, row i+1's K, slot and position are in flight, and its
// cos/sin load is issued once row i's Hadamard is done (the position has arrived by
// then).  The norm weight is kept in shared memory as fp32 and read per row (114
// registers a thread in the FP4 kernel, two CTAs an SM): on 65,536 rows after an L2 flush that measured
// 16.3-16.9 us a launch against 16.7-17.3 us with the weight held in 32 registers (124
// a thread), 18.0 us for a variant that streams two rows ahead into shared memory with
// cp.async at three CTAs an SM, and 21-22 us at three CTAs an SM with this pipeline
// (80 registers, spilling).
template <bool kFp8>
__device__ __forceinline__ void store_k_rows(const StoreArgs& a, int64_t first_unit, int64_t unit_stride,
                                             uint8_t* payload, uint8_t* scale, uint8_t* fp8_pages) {
  const int lane = threadIdx.x & 31, l = lane & 3;
  const int sub = lane >> 2;
  const bool reporter = l == 0;
  const int64_t n_units = (a.n_rows + 7) >> 3;
  int64_t u = first_unit;
  __shared__ __align__(16) float wsm[kHeadDim];  // the norm weight in fp32 (exact)
  if (threadIdx.x < kHeadDim) wsm[threadIdx.x] = __uint_as_float((uint32_t)__ldg(a.norm_w + threadIdx.x) << 16);
  __syncthreads();
  if (u >= n_units) return;  // uniform over the warp, after the block's barrier
  StoreRow cur;
  load_cs(a.cos_sin, load_row_head(a, u * 8 + sub, l, reporter, cur), l, cur.cs);
  for (;;) {
    const int64_t un = u + unit_stride;
    const bool more = un < n_units;
    StoreRow nxt;
    int32_t npos = 0;
    if (more) npos = load_row_head(a, un * 8 + sub, l, reporter, nxt);
    qw::f2 x[4][4], w[4][4];
    norm_w_of_lane(wsm, l, w);
    k_chain_qw(x, cur.raw, w, a.eps, cur.cs, l);
    if (more) load_cs(a.cos_sin, npos, l, nxt.cs);
    const int64_t page = cur.slot >> 6;
    const int j = cur.slot & 63;
    if constexpr (!kFp8) {
      uint32_t sb[4], word[4];
#pragma unroll
      for (int m = 0; m < 4; m++) word[m] = qw::fp4_block(x[m], sb[m]);
      if (cur.store) {
#pragma unroll
        for (int m = 0; m < 4; m++)
          *reinterpret_cast<uint32_t*>(payload + ((page * 4 + m) * kPage + j) * 16 + 4 * l) = word[m];
        const uint32_t mine = l == 0 ? sb[0] : l == 1 ? sb[1] : l == 2 ? sb[2] : sb[3];
        scale[(page * 4 + l) * kPage + j] = (uint8_t)mine;
      }
    } else {
      float amax = 0.0f;
#pragma unroll
      for (int m = 0; m < 4; m++)
#pragma unroll
        for (int jj = 0; jj < 4; jj++) amax = fmaxf(amax, fmaxf(fabsf(x[m][jj].x), fabsf(x[m][jj].y)));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
      const float sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
      uint8_t* base = fp8_pages + page * (int64_t)FP4IDX_FP8_PAGE_BYTES;
#pragma unroll
      for (int m = 0; m < 4; m++) {
        uint2 out;
        out.x = e4m3x2(__fdiv_rn(x[m][0].x, sc), __fdiv_rn(x[m][0].y, sc)) |
                (e4m3x2(__fdiv_rn(x[m][1].x, sc), __fdiv_rn(x[m][1].y, sc)) << 16);
        out.y = e4m3x2(__fdiv_rn(x[m][2].x, sc), __fdiv_rn(x[m][2].y, sc)) |
                (e4m3x2(__fdiv_rn(x[m][3].x, sc), __fdiv_rn(x[m][3].y, sc)) << 16);
        if (cur.store) *reinterpret_cast<uint2*>(base + j * kHeadDim + 32 * m + 8 * l) = out;
      }
      if (cur.store && l == 0) *reinterpret_cast<float*>(base + kPage * kHeadDim + j * 4) = sc;
    }
    if (!more) break;
    u = un;
    cur = nxt;
  }
}

__global__ void __launch_bounds__(256) store_k_kernel(const StoreArgs a, uint8_t* __restrict__ payload,
                                                      uint8_t* __restrict__ scale) {
  const int64_t warps = (int64_t)gridDim.x * 8;
  store_k_rows<false>(a, (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5), warps, payload, scale, nullptr);
}

__global__ void __launch_bounds__(256) store_k_fp8_kernel(const StoreArgs a, uint8_t* __restrict__ pages) {
  const int64_t warps = (int64_t)gridDim.x * 8;
  store_k_rows<true>(a, (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5), warps, nullptr, nullptr, pages);
}

// K store of the 16 rows of block `block` on the half-warp mapping (the query packers'),
// for the step preparation: its few new rows are latency-bound, and a half-warp's row
// chain is about a third as long as a quarter-warp's (8 elements a lane against 32).  Same
// arithmetic in the same order, so the same bytes.
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
  int64_t kb;  // blocks of the K store (16 rows each)
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

// The K stores run one pass over the rows with at most as many CTAs as fit on the GPU at
// once (each warp then loops over its share, loading its next row ahead of the arithmetic).
template <class Kern>
unsigned store_grid(Kern kernel, int64_t n_rows, cudaError_t* err) {
  const int64_t need = (n_rows + kStoreRowsPerBlock - 1) / kStoreRowsPerBlock;
  int fit = 0;
  *err = resident_ctas(reinterpret_cast<const void*>(kernel), 256, 0, &fit);
  return (unsigned)std::max<int64_t>(1, std::min<int64_t>(need, fit));
}

cudaError_t launch_store_k(const uint16_t* k, int64_t n_rows, const int32_t* positions, const int32_t* slots,
                           const uint16_t* norm_w, float eps, const uint16_t* cos_sin, int32_t max_pos,
                           uint8_t* payload, uint8_t* scale, int64_t num_pages, int32_t* status,
                           cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  cudaError_t e = prefer_max_shared(store_k_kernel, g_carve_store);
  if (e != cudaSuccess) return e;
  const unsigned grid = store_grid(store_k_kernel, n_rows, &e);
  if (e != cudaSuccess) return e;
  const StoreArgs a{k, n_rows, positions, slots, norm_w, eps, cos_sin, max_pos, num_pages, status};
  store_k_kernel<<<grid, 256, 0, stream>>>(a, payload, scale);
  return cudaGetLastError();
}

cudaError_t launch_store_k_fp8(const uint16_t* k, int64_t n_rows, const int32_t* positions, const int32_t* slots,
                               const uint16_t* norm_w, float eps, const uint16_t* cos_sin, int32_t max_pos,
                               uint8_t* pages, int64_t num_pages, int32_t* status, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  cudaError_t e = prefer_max_shared(store_k_fp8_kernel, g_carve_store_fp8);
  if (e != cudaSuccess) return e;
  const unsigned grid = store_grid(store_k_fp8_kernel, n_rows, &e);
  if (e != cudaSuccess) return e;
  const StoreArgs a{k, n_rows, positions, slots, norm_w, eps, cos_sin, max_pos, num_pages, status};
  store_k_fp8_kernel<<<grid, 256, 0, stream>>>(a, pages);
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
