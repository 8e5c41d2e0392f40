/*
 * fp4idx_ref.c -- CPU oracle for the DeepSeek-V4 FP4 indexer hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
 * statement of what the indexer computes.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg load it; the product path (the CUDA library
 * behind include/fp4idx.h) never calls, links or includes anything here, and
 * this file includes nothing of the product.
 *
 * Sources (three SGLang pull-request pages on the FP4 indexer):
 *   [P1] "dsv4.1-amd: KV cache layouts, FP4 indexer, compressor and router kernels"
 *   [P2] "[AMD] Enable FP4 indexer for Deepseek V4"
 *   [P3] "[AMD] DeepSeek-V4.1-Flash on MI350X (gfx950)"
 * What each function follows is cited beside it.  Where the pages leave a step
 * open (eps, RoPE pairing, Hadamard scale placement, UE8M0 rounding rule,
 * nibble order, reduction orders) the reading used is stated at the function;
 * the CUDA path implements the same readings independently.
 *
 * Floating point: every float operation is a separately rounded IEEE binary32
 * operation in the order written (build with -ffp-contract=off, no fast-math).
 * Logits are computed in binary64 from the dequantised operands.
 *
 * Parity status of each function: pinned by the CPU tests (closed forms,
 * exhaustive grids, brute force on tiny inputs, invariants), except where a
 * function's comment says "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define D 128          /* index-K / index-Q row width */
#define ROT 64         /* RoPE span: dims 0..63 */
#define BLK 32         /* elements per UE8M0 scale block */
#define NBLK 4         /* scale blocks per row */
#define PAGE 64        /* tokens per cache page */

enum { REF_OK = 0, REF_ERR_ARG = 1, REF_ERR_BAD_PAGE = 5 };

static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static float f32_from_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

void ref_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int ref_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ RMSNorm
 * [P2] Modifications / FP4 kernel adapters: the K writer runs "fused RMSNorm,
 * RoPE, Hadamard, FP4 quantization, and paged cache writes"; [P2] compressor.py
 * keeps a BF16 mirror of the indexer RMSNorm weight for that writer.
 * y_i = x_i / sqrt(mean(x^2) + eps) * w_i.
 * Reading (order of the sum of squares): partial sums over consecutive groups of
 * eight squares, each summed left to right; the sixteen partials combined by a
 * pairwise tree in index order.  r = 1/sqrt(mean+eps) with IEEE sqrt and divide;
 * y_i = (x_i * r) * w_i.  eps is an argument (1e-6 in the workloads). */
void ref_rmsnorm(const float x[D], const float w[D], float eps, float y[D]) {
  float part[16];
  for (int g = 0; g < 16; g++) {
    float s = 0.0f;
    for (int i = 0; i < 8; i++) {
      float xi = x[8 * g + i];
      float sq = xi * xi;
      s = s + sq;
    }
    part[g] = s;
  }
  float lvl[16];
  int n = 16;
  memcpy(lvl, part, sizeof(part));
  while (n > 1) {
    float nxt[8];
    for (int i = 0; i < n / 2; i++) nxt[i] = lvl[2 * i] + lvl[2 * i + 1];
    n /= 2;
    memcpy(lvl, nxt, sizeof(float) * (size_t)n);
  }
  float sumsq = lvl[0];
  float mean = sumsq * 0.0078125f; /* 1/128, exact */
  float r = 1.0f / sqrtf(mean + eps);
  for (int i = 0; i < D; i++) {
    float t = x[i] * r;
    y[i] = t * w[i];
  }
}

/* ------------------------------------------------------------------ RoPE
 * [P2] Modifications / deepseek_v4.py: Q and K transforms reuse the model-owned
 * BF16 RoPE cos/sin cache.  The rotary span is dims 0..63 of the 128.
 * Table row `pos` holds cos(pos*f_i) in columns 0..31, sin(pos*f_i) in 32..63.
 * Reading (pairing): half-split pairs (i, i+32), i < 32:
 *   a' = a*cos_i - b*sin_i,  b' = b*cos_i + a*sin_i   (each product rounded).
 * Dims 64..127 pass through. */
void ref_rope(float u[D], const uint16_t* cos_sin_row) {
  for (int i = 0; i < ROT / 2; i++) {
    float c = bf16_to_f32(cos_sin_row[i]);
    float s = bf16_to_f32(cos_sin_row[ROT / 2 + i]);
    float a = u[i];
    float b = u[i + ROT / 2];
    float ac = a * c, bs = b * s, bc = b * c, as = a * s;
    u[i] = ac - bs;
    u[i + ROT / 2] = bc + as;
  }
}

/* ------------------------------------------------------------------ Hadamard
 * [P2] Modifications: Q/K go through a Hadamard rotation before FP4.
 * 128-point Walsh-Hadamard in Sylvester order: stages with half-width
 * h = 1, 2, 4, ..., 64; in each, for every i with (i & h) == 0,
 *   (u_i, u_{i+h}) <- (u_i + u_{i+h}, u_i - u_{i+h}).
 * Then every element is multiplied once by the binary32 value of 1/sqrt(128)
 * (bit pattern 0x3DB504F3), so the rotation is orthonormal. */
void ref_hadamard128(float u[D]) {
  for (int h = 1; h < D; h <<= 1) {
    for (int i = 0; i < D; i++) {
      if (i & h) continue;
      float a = u[i], b = u[i + h];
      u[i] = a + b;
      u[i + h] = a - b;
    }
  }
  const float inv_sqrt128 = f32_from_bits(0x3DB504F3u);
  for (int i = 0; i < D; i++) u[i] = u[i] * inv_sqrt128;
}

/* ------------------------------------------------------------------ UE8M0 block scale
 * [P2] Motivation: one UE8M0 scale byte per 32 elements.
 * Reading (rounding rule): the block exponent e is the smallest integer with
 * 6 * 2^e >= amax (6 = largest e2m1 magnitude), so no element saturates;
 * clamped to [-127, 127]; amax = 0 gives -127.  Stored byte = e + 127. */
int ref_ue8m0_exponent(float amax) {
  if (!(amax > 0.0f)) return -127;
  int E;
  (void)frexpf(amax, &E);              /* amax = m * 2^E, 0.5 <= m < 1 */
  int e = E - 4;                       /* 6 * 2^(E-4) = 0.375 * 2^E < amax: below the answer */
  while (ldexp(6.0, e) < (double)amax) e++;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

int ref_ue8m0_byte(float amax) { return ref_ue8m0_exponent(amax) + 127; }

/* ------------------------------------------------------------------ e2m1
 * [P1] Summary: FP4 rows are quantised "with round-to-nearest-even".
 * e2m1 magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6} are codes 0..7; bit 3 is the sign.
 * Nearest grid value; a tie goes to the even code; magnitudes beyond 6 go to 6.
 * Reading: the sign bit is kept for values that round to zero (code 8 = -0). */
static const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double ref_e2m1_value(int code) {
  double m = kE2M1[code & 7];
  return (code & 8) ? -m : m;
}

int ref_e2m1_code(float v) {
  double mag = fabs((double)v);
  if (mag >= 6.0) return 7 | (signbit(v) ? 8 : 0); /* saturate */
  int best = 0;
  double bestd = fabs(mag - kE2M1[0]);
  for (int c = 1; c < 8; c++) {
    double d = fabs(mag - kE2M1[c]);
    if (d < bestd || (d == bestd && (c & 1) == 0)) {
      best = c;
      bestd = d;
    }
  }
  return best | (signbit(v) ? 8 : 0);
}

/* ------------------------------------------------------------------ e4m3 (FP8 layout)
 * [P2] Device memory and sizing: the FP8 indexer entry is 132 bytes per token
 * (128 e4m3 + a 4-byte scale).  e4m3 ("fn": no infinities, 0x7F/0xFF NaN),
 * finite maximum 448; round to nearest, ties to even code, saturating.
 * Reading: sign kept for values that round to zero. */
double ref_e4m3_value(int code) {
  int e = (code >> 3) & 15, m = code & 7;
  double v = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return (code & 0x80) ? -v : v;
}

int ref_e4m3_code(float v) {
  double mag = fabs((double)v);
  if (mag >= 448.0) return 0x7E | (signbit(v) ? 0x80 : 0); /* saturate */
  int best = 0;
  double bestd = mag;
  for (int c = 1; c <= 0x7E; c++) {
    double d = fabs(mag - ref_e4m3_value(c));
    if (d < bestd || (d == bestd && (c & 1) == 0)) {
      best = c;
      bestd = d;
    }
  }
  return best | (signbit(v) ? 0x80 : 0);
}

/* ------------------------------------------------------------------ the K / Q chains
 * [P2] Modifications: K: RMSNorm -> RoPE -> Hadamard -> FP4 -> paged write;
 * Q: RoPE -> Hadamard -> FP4 (no norm on the query side).
 * stage: 1 = after RMSNorm, 2 = after RoPE, 3 = after Hadamard (for the pins). */
void ref_k_chain(const uint16_t* k_row, int32_t pos, const uint16_t* norm_w, float eps,
                 const uint16_t* cos_sin, int stage, float out[D]) {
  float x[D], w[D], y[D];
  for (int i = 0; i < D; i++) {
    x[i] = bf16_to_f32(k_row[i]);
    w[i] = bf16_to_f32(norm_w[i]);
  }
  ref_rmsnorm(x, w, eps, y);
  if (stage >= 2) ref_rope(y, cos_sin + (size_t)pos * ROT);
  if (stage >= 3) ref_hadamard128(y);
  memcpy(out, y, sizeof(y));
}

void ref_q_chain(const uint16_t* q_row, int32_t pos, const uint16_t* cos_sin, int stage, float out[D]) {
  float y[D];
  for (int i = 0; i < D; i++) y[i] = bf16_to_f32(q_row[i]);
  if (stage >= 2) ref_rope(y, cos_sin + (size_t)pos * ROT);
  if (stage >= 3) ref_hadamard128(y);
  memcpy(out, y, sizeof(y));
}

/* FP4 encoding of one rotated row: per block c, scale byte sc[c] and 16 packed
 * bytes pk[c][b].  Reading (nibble order): byte b of block c holds element
 * 32c+2b in its low nibble and 32c+2b+1 in its high nibble. */
void ref_fp4_encode_row(const float z[D], uint8_t pk[NBLK][16], uint8_t sc[NBLK]) {
  for (int c = 0; c < NBLK; c++) {
    float amax = 0.0f;
    for (int i = 0; i < BLK; i++) {
      float a = fabsf(z[BLK * c + i]);
      if (a > amax) amax = a;
    }
    int e = ref_ue8m0_exponent(amax);
    sc[c] = (uint8_t)(e + 127);
    for (int b = 0; b < 16; b++) {
      float v0 = ldexpf(z[BLK * c + 2 * b], -e);
      float v1 = ldexpf(z[BLK * c + 2 * b + 1], -e);
      pk[c][b] = (uint8_t)(ref_e2m1_code(v0) | (ref_e2m1_code(v1) << 4));
    }
  }
}

/* ------------------------------------------------------------------ K store (split layout)
 * [P2] Motivation: per compressed token a 64-byte FP4 payload and a 4-byte
 * UE8M0 scale in separate tensors, payload [num_pages, 1, 4, 64, 16] and scale
 * [num_pages, 1, 4, 64] (64 tokens per page; the singleton dim is dropped here).
 * Reading of the "preshuffled" order: dim 1 is the 32-element block c, dim 2 the
 * token j within the page:  payload[page][c][j][0..15], scale[page][c][j].
 * slot = page*64 + j; rows with slot < 0 are padding and are skipped.
 * Returns REF_ERR_BAD_PAGE (and skips the row) for a slot past the cache. */
int ref_store_k(const uint16_t* k, int64_t n_rows, const int32_t* positions, const int32_t* slots,
                const uint16_t* norm_w, float eps, const uint16_t* cos_sin, int32_t max_pos,
                uint8_t* payload, uint8_t* scale, int64_t num_pages) {
  int status = REF_OK;
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < n_rows; n++) {
    int32_t slot = slots[n];
    if (slot < 0) continue;
    int64_t page = slot / PAGE, j = slot % PAGE;
    if (page >= num_pages || positions[n] < 0 || positions[n] >= max_pos) {
#pragma omp critical
      status = REF_ERR_BAD_PAGE;
      continue;
    }
    float z[D];
    uint8_t pk[NBLK][16], sc[NBLK];
    ref_k_chain(k + (size_t)n * D, positions[n], norm_w, eps, cos_sin, 3, z);
    ref_fp4_encode_row(z, pk, sc);
    for (int c = 0; c < NBLK; c++) {
      memcpy(payload + ((size_t)page * NBLK + c) * PAGE * 16 + (size_t)j * 16, pk[c], 16);
      scale[((size_t)page * NBLK + c) * PAGE + (size_t)j] = sc[c];
    }
  }
  return status;
}

/* ------------------------------------------------------------------ K store, FP8 fused layout
 * [P2] Device memory and sizing / HiCache integration: the FP8 indexer entry is
 * 132 bytes per token in a fused page.  Readings (the pages give only the size):
 * same chain up to the Hadamard; one fp32 scale per token = amax/448 (IEEE
 * divide; amax = 0 gives scale 1); element = e4m3(z/scale); page layout
 * [64 tokens x 128 B e4m3][64 tokens x 4 B fp32 scale] = 8,448 B. */
int ref_store_k_fp8(const uint16_t* k, int64_t n_rows, const int32_t* positions, const int32_t* slots,
                    const uint16_t* norm_w, float eps, const uint16_t* cos_sin, int32_t max_pos,
                    uint8_t* pages, int64_t num_pages) {
  int status = REF_OK;
  const size_t page_bytes = (size_t)PAGE * (D + 4);
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < n_rows; n++) {
    int32_t slot = slots[n];
    if (slot < 0) continue;
    int64_t page = slot / PAGE, j = slot % PAGE;
    if (page >= num_pages || positions[n] < 0 || positions[n] >= max_pos) {
#pragma omp critical
      status = REF_ERR_BAD_PAGE;
      continue;
    }
    float z[D];
    ref_k_chain(k + (size_t)n * D, positions[n], norm_w, eps, cos_sin, 3, z);
    float amax = 0.0f;
    for (int i = 0; i < D; i++) {
      float a = fabsf(z[i]);
      if (a > amax) amax = a;
    }
    float s = (amax > 0.0f) ? amax / 448.0f : 1.0f;
    uint8_t* base = pages + (size_t)page * page_bytes;
    for (int i = 0; i < D; i++) base[(size_t)j * D + i] = (uint8_t)ref_e4m3_code(z[i] / s);
    memcpy(base + (size_t)PAGE * D + (size_t)j * 4, &s, 4);
  }
  return status;
}

/* ------------------------------------------------------------------ Q quant
 * [P2] Modifications / fp4_indexer_hip.py: "Q RoPE/Hadamard/FP4 quantization";
 * [P1] Summary: the query packer.  Same FP4 encoding as K, no RMSNorm.
 * Output layout (this library's own query format, shaped like one K page with the
 * 64 heads in place of the 64 tokens): q_payload[t][c][h][16], q_scale[t][c][h]. */
int ref_quant_q(const uint16_t* q, int64_t T, int32_t H, const int32_t* q_positions,
                const uint16_t* cos_sin, int32_t max_pos, uint8_t* q_payload, uint8_t* q_scale) {
  int status = REF_OK;
#pragma omp parallel for schedule(static)
  for (int64_t th = 0; th < T * H; th++) {
    int64_t t = th / H, h = th % H;
    int32_t pos = q_positions[t];
    if (pos < 0 || pos >= max_pos) {
#pragma omp critical
      status = REF_ERR_ARG;
      continue;
    }
    float z[D];
    uint8_t pk[NBLK][16], sc[NBLK];
    ref_q_chain(q + (size_t)th * D, pos, cos_sin, 3, z);
    ref_fp4_encode_row(z, pk, sc);
    for (int c = 0; c < NBLK; c++) {
      memcpy(q_payload + (((size_t)t * NBLK + c) * H + (size_t)h) * 16, pk[c], 16);
      q_scale[((size_t)t * NBLK + c) * H + (size_t)h] = sc[c];
    }
  }
  return status;
}

/* ------------------------------------------------------------------ dequantisation
 * value = e2m1(code) * 2^(scale_byte - 127), in binary64 (exact). */
static void dequant_row(const uint8_t pk[NBLK][16], const uint8_t sc[NBLK], double out[D]) {
  for (int c = 0; c < NBLK; c++) {
    int e = (int)sc[c] - 127;
    for (int b = 0; b < 16; b++) {
      out[BLK * c + 2 * b] = ldexp(ref_e2m1_value(pk[c][b] & 15), e);
      out[BLK * c + 2 * b + 1] = ldexp(ref_e2m1_value(pk[c][b] >> 4), e);
    }
  }
}

/* dequantised K of one cached token (split layout) */
void ref_dequant_k_token(const uint8_t* payload, const uint8_t* scale, int64_t page, int32_t j, double out[D]) {
  uint8_t pk[NBLK][16], sc[NBLK];
  for (int c = 0; c < NBLK; c++) {
    memcpy(pk[c], payload + ((size_t)page * NBLK + c) * PAGE * 16 + (size_t)j * 16, 16);
    sc[c] = scale[((size_t)page * NBLK + c) * PAGE + (size_t)j];
  }
  dequant_row(pk, sc, out);
}

/* dequantised Q of one (row, head) */
void ref_dequant_q(const uint8_t* q_payload, const uint8_t* q_scale, int32_t H, int64_t t, int32_t h, double out[D]) {
  uint8_t pk[NBLK][16], sc[NBLK];
  for (int c = 0; c < NBLK; c++) {
    memcpy(pk[c], q_payload + (((size_t)t * NBLK + c) * H + (size_t)h) * 16, 16);
    sc[c] = q_scale[((size_t)t * NBLK + c) * H + (size_t)h];
  }
  dequant_row(pk, sc, out);
}

/* ------------------------------------------------------------------ paged-MQA logits
 * [P2] Modifications: decode and prefill "FP4 paged-MQA logits" read the split
 * payload/scale cache through the page table.  The pages do not write the formula;
 * this library reads it as (ReLU, head weights, no softmax or 1/sqrt(d))
 *   logits[t,s] = sum_h w[t,h] * ReLU(q_hat[t,h] . k_hat[s]),  s < context_lens[t],
 * with q_hat, k_hat the dequantised FP4 operands.  Token s of row t lives at
 * physical page page_table[row_seq[t]][s / 64], slot s % 64.
 * For each requested row (rows[0..n_req)), writes logits[r][s] for s < L (binary64)
 * and, when bound != NULL, bound[r][s] = sum_h |w| * sum_i |q_hat_i * k_hat_i|,
 * the scale of the rounding error any binary32 evaluation can make. */
int ref_logits(const uint8_t* q_payload, const uint8_t* q_scale, const float* w, int64_t T, int32_t H,
               const uint8_t* payload, const uint8_t* scale, int64_t num_pages,
               const int32_t* page_table, int32_t max_pages, const int32_t* row_seq,
               const int32_t* context_lens, const int64_t* rows, int64_t n_req, int64_t L_stride,
               double* logits, double* bound) {
  int status = REF_OK;
  for (int64_t r = 0; r < n_req; r++) {
    int64_t t = rows[r];
    if (t < 0 || t >= T) return REF_ERR_ARG;
    int32_t L = context_lens[t];
    if (L > L_stride) return REF_ERR_ARG;
    double* qh = (double*)malloc(sizeof(double) * (size_t)H * D);
    for (int32_t h = 0; h < H; h++) ref_dequant_q(q_payload, q_scale, H, t, h, qh + (size_t)h * D);
    const int32_t* pt = page_table + (size_t)row_seq[t] * max_pages;
#pragma omp parallel for schedule(static)
    for (int32_t s = 0; s < L; s++) {
      int32_t lp = s / PAGE;
      int64_t page = (lp < max_pages) ? pt[lp] : -1;
      if (page < 0 || page >= num_pages) {
#pragma omp critical
        status = REF_ERR_BAD_PAGE;
        logits[r * L_stride + s] = NAN;
        if (bound) bound[r * L_stride + s] = NAN;
        continue;
      }
      double kh[D];
      ref_dequant_k_token(payload, scale, page, s % PAGE, kh);
      double acc = 0.0, accb = 0.0;
      for (int32_t h = 0; h < H; h++) {
        const double* qv = qh + (size_t)h * D;
        double dot = 0.0, adot = 0.0;
        for (int i = 0; i < D; i++) {
          double p = qv[i] * kh[i];
          dot += p;
          adot += fabs(p);
        }
        double wh = (double)w[t * H + h];
        acc += wh * (dot > 0.0 ? dot : 0.0);
        accb += fabs(wh) * adot;
      }
      logits[r * L_stride + s] = acc;
      if (bound) bound[r * L_stride + s] = accb;
    }
    free(qh);
  }
  return status;
}

/* ------------------------------------------------------------------ FP8 comparison path
 * [P2] Device memory and sizing: the FP8 indexer entry that the FP4 entry replaces, 132 B
 * per token (128 e4m3 values and one fp32 scale).  Page layout as ref_store_k_fp8 writes it:
 * bytes [j*128, j*128+128) = token j's e4m3 values, bytes [8192 + 4j, 8192 + 4j + 4) = its
 * fp32 scale.  The query side follows the K side's rule (a reading: the pages give only the
 * K entry): after RoPE and the Hadamard, one fp32 scale s = amax/448 per (row, head), 1 when
 * amax = 0, and e4m3 = RNE-satfinite(z / s).  Query layout (this library's own):
 * q8[t][c][h][16] for the 8 chunks c of 16 values, q8_scale[t][h] fp32. */
int ref_quant_q_fp8(const uint16_t* q, int64_t T, int32_t H, const int32_t* q_positions, const uint16_t* cos_sin,
                    int32_t max_pos, uint8_t* q8, float* q8_scale) {
  int status = REF_OK;
#pragma omp parallel for schedule(static)
  for (int64_t th = 0; th < T * H; th++) {
    int64_t t = th / H;
    int32_t h = (int32_t)(th % H), pos = q_positions[t];
    if (pos < 0 || pos >= max_pos) {
#pragma omp critical
      status = REF_ERR_ARG;
      continue;
    }
    float z[D];
    ref_q_chain(q + (size_t)th * D, pos, cos_sin, 3, z);
    float amax = 0.0f;
    for (int i = 0; i < D; i++) {
      float a = fabsf(z[i]);
      if (a > amax) amax = a;
    }
    float sc = (amax > 0.0f) ? amax / 448.0f : 1.0f;
    for (int i = 0; i < D; i++)
      q8[((size_t)(t * 8 + i / 16) * H + h) * 16 + (i % 16)] = (uint8_t)ref_e4m3_code(z[i] / sc);
    q8_scale[t * H + h] = sc;
  }
  return status;
}

/* dequantised K of one token of an FP8 page */
void ref_dequant_k_fp8_token(const uint8_t* pages, int64_t page, int32_t j, double out[D]) {
  const uint8_t* base = pages + (size_t)page * PAGE * (D + 4);
  float sc;
  memcpy(&sc, base + (size_t)PAGE * D + (size_t)j * 4, 4);
  for (int i = 0; i < D; i++) out[i] = ref_e4m3_value(base[(size_t)j * D + i]) * (double)sc;
}

/* dequantised FP8 Q of one (row, head) */
void ref_dequant_q_fp8(const uint8_t* q8, const float* q8_scale, int32_t H, int64_t t, int32_t h, double out[D]) {
  double sc = (double)q8_scale[t * H + h];
  for (int i = 0; i < D; i++) out[i] = ref_e4m3_value(q8[((size_t)(t * 8 + i / 16) * H + h) * 16 + (i % 16)]) * sc;
}

/* logits[t,s] = sum_h w[t,h] * ReLU(q_hat[t,h] . k_hat[s]) over the FP8 operands, binary64,
 * with the same paging, masking and bound as ref_logits. */
int ref_logits_fp8(const uint8_t* q8, const float* q8_scale, const float* w, int64_t T, int32_t H,
                   const uint8_t* pages, int64_t num_pages, const int32_t* page_table, int32_t max_pages,
                   const int32_t* row_seq, const int32_t* context_lens, const int64_t* rows, int64_t n_req,
                   int64_t L_stride, double* logits, double* bound) {
  int status = REF_OK;
  for (int64_t r = 0; r < n_req; r++) {
    int64_t t = rows[r];
    if (t < 0 || t >= T) return REF_ERR_ARG;
    int32_t L = context_lens[t];
    if (L > L_stride) return REF_ERR_ARG;
    double* qh = (double*)malloc(sizeof(double) * (size_t)H * D);
    for (int32_t h = 0; h < H; h++) ref_dequant_q_fp8(q8, q8_scale, H, t, h, qh + (size_t)h * D);
    const int32_t* pt = page_table + (size_t)row_seq[t] * max_pages;
#pragma omp parallel for schedule(static)
    for (int32_t s = 0; s < L; s++) {
      int32_t lp = s / PAGE;
      int64_t page = (lp < max_pages) ? pt[lp] : -1;
      if (page < 0 || page >= num_pages) {
#pragma omp critical
        status = REF_ERR_BAD_PAGE;
        logits[r * L_stride + s] = NAN;
        if (bound) bound[r * L_stride + s] = NAN;
        continue;
      }
      double kh[D];
      ref_dequant_k_fp8_token(pages, page, s % PAGE, kh);
      double acc = 0.0, accb = 0.0;
      for (int32_t h = 0; h < H; h++) {
        const double* qv = qh + (size_t)h * D;
        double dot = 0.0, adot = 0.0;
        for (int i = 0; i < D; i++) {
          double p = qv[i] * kh[i];
          dot += p;
          adot += fabs(p);
        }
        double wh = (double)w[t * H + h];
        acc += wh * (dot > 0.0 ? dot : 0.0);
        accb += fabs(wh) * adot;
      }
      logits[r * L_stride + s] = acc;
      if (bound) bound[r * L_stride + s] = accb;
    }
    free(qh);
  }
  return status;
}

/* ------------------------------------------------------------------ top-k
 * Per query row, the k largest logits among s < L; [P3] Changes and
 * Historical results: the selection is sorted and "ordered by position, not KV
 * slot".  Candidates ordered by (logit descending, index ascending); the first
 * min(k, L) are kept and emitted in ascending index order; the rest is -1. */
typedef struct {
  double v;
  int32_t i;
} ref_cand;

static int cand_cmp(const void* a, const void* b) {
  const ref_cand* x = (const ref_cand*)a;
  const ref_cand* y = (const ref_cand*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->i > y->i) - (x->i < y->i);
}

static int int_cmp(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

int ref_topk(const double* logits, int64_t L, int32_t k, int32_t* out) {
  if (k <= 0 || L < 0) return REF_ERR_ARG;
  ref_cand* c = (ref_cand*)malloc(sizeof(ref_cand) * (size_t)(L > 0 ? L : 1));
  for (int64_t s = 0; s < L; s++) {
    c[s].v = logits[s];
    c[s].i = (int32_t)s;
  }
  qsort(c, (size_t)L, sizeof(ref_cand), cand_cmp);
  int64_t m = L < k ? L : k;
  for (int64_t i = 0; i < m; i++) out[i] = c[i].i;
  qsort(out, (size_t)m, sizeof(int32_t), int_cmp);
  for (int64_t i = m; i < k; i++) out[i] = -1;
  free(c);
  return REF_OK;
}

/* ------------------------------------------------------------------ array helpers for the pins */
void ref_e2m1_codes(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)ref_e2m1_code(v[i]);
}

void ref_e4m3_codes(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)ref_e4m3_code(v[i]);
}

void ref_ue8m0_bytes(const float* amax, int64_t n, int32_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = ref_ue8m0_byte(amax[i]);
}

void ref_fp4_encode_rows(const float* z, int64_t n, uint8_t* pk, uint8_t* sc) {
  for (int64_t r = 0; r < n; r++) ref_fp4_encode_row(z + r * D, (uint8_t(*)[16])(pk + r * 64), sc + r * 4);
}

void ref_fp4_decode_rows(const uint8_t* pk, const uint8_t* sc, int64_t n, double* out) {
  for (int64_t r = 0; r < n; r++) dequant_row((const uint8_t(*)[16])(pk + r * 64), sc + r * 4, out + r * D);
}
