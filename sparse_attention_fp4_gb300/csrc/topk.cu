// Per-row top-k of the logits, emitted as ascending compressed-token indices.
//
// [AMD] DeepSeek-V4.1-Flash on MI350X (gfx950) -- Changes: "sorted top-k selection";
// Historical results: the decode top-k is ordered by position, not by KV slot.
// [AMD] Enable FP4 indexer for Deepseek V4 -- Attention runtime: padded rows keep
// context length 0 (their selection is empty: all -1).
//
// Selection = the k largest logits of a row, ties at the k-th value to the lower
// positions, emitted in ascending position order.  Two launches:
//   filter (one CTA per row and 4,096-token chunk): every CTA of a row takes the same
//     fixed sample of 1,024 logits and derives the same conservative threshold bucket
//     (a linear 256-bucket histogram of the sample, cut about four standard deviations
//     beyond the expected position of the k-th largest), then writes the positions of
//     its chunk's logits at or above it, in order, into the chunk's own region of a
//     candidate buffer: no cross-CTA synchronisation;
//   select (one CTA per row): concatenates the chunk regions in order, gathers the
//     candidates' logits, finds the key of the k-th largest by radix select (11 + 11 + 10
//     bits) and emits the keys above it and the lowest-positioned keys equal to it.
// The sample decides speed, never the result: when fewer than k or more than kCapB
// logits pass, the select launch runs the exact path over the whole row (2048 buckets
// linear in value between the row's min and max, a refinement of a crowded bucket over
// its own range, the bucket's candidates ranked exactly, radix select when a bucket is
// all ties).
#include "fp4idx_internal.cuh"

namespace fp4idx {
namespace {

constexpr int kThreads = 512;          // select launch
constexpr int kFilterThreads = 256;    // filter launch
constexpr int kChunk = 4096;           // tokens per filter CTA (16 per thread)
constexpr int kCapB = 8192;            // candidates the select launch keeps in shared memory
constexpr int kMaxChunks = (FP4IDX_MAX_CONTEXT + kChunk - 1) / kChunk;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kThreads;
constexpr int kGather = 1024;
constexpr int kSample = 1024;    // sample for the filter threshold
constexpr int kSampleBins = 256;
constexpr unsigned kFull = 0xFFFFFFFFu;

// Order-preserving key; -0 maps to +0 so that equal values are equal keys.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = f == 0.0f ? 0u : __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Linear bucket of value x over [lo, lo + 2047/scale]; scale = 0 puts everything in bucket 0.
__device__ __forceinline__ int lin_bucket(float x, float lo, float scale) {
  const float v = (x - lo) * scale;
  if (!(v >= 0.0f)) return 0;  // also NaN
  return v >= (float)(kBins - 1) ? kBins - 1 : (int)v;
}

__device__ __forceinline__ float lin_scale(float lo, float hi) {
  const float range = hi - lo;
  return (range > 0.0f && range < INFINITY) ? (float)(kBins - 1) / range : 0.0f;
}

// Exclusive block scan of an int; `total` gets the block sum.
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += n;
    }
    if (lane < kWarps) scratch[lane] = w;
  }
  __syncthreads();
  const int before = (warp > 0 ? scratch[warp - 1] : 0) + x - v;
  total = scratch[kWarps - 1];
  __syncthreads();
  return before;
}

template <bool kMax>
__device__ __forceinline__ uint32_t block_reduce(uint32_t v, uint32_t* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t n = __shfl_xor_sync(kFull, v, o);
    v = kMax ? max(v, n) : min(v, n);
  }
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  uint32_t r = scratch[0];
  for (int i = 1; i < kWarps; i++) r = kMax ? max(r, scratch[i]) : min(r, scratch[i]);
  __syncthreads();
  return r;
}

// Thread whose run of histogram bins (taken from the top) contains the rem-th largest
// element writes (bin, rem - elements above the bin).
__device__ __forceinline__ void find_bin_from_top(const int* counts, int rem, int* scratch, int* out_bin,
                                                  int* out_rem) {
  const int tb = (kThreads - 1 - (int)threadIdx.x) * kBinsPerThread;
  int mine = 0;
#pragma unroll
  for (int j = 0; j < kBinsPerThread; j++) mine += counts[tb + j];
  int tot;
  const int above = block_excl_scan(mine, scratch, tot);
  if (above < rem && rem <= above + mine) {
    int acc = above;
    for (int j = kBinsPerThread - 1; j >= 0; j--) {
      const int c = counts[tb + j];
      if (acc < rem && rem <= acc + c) {
        *out_bin = tb + j;
        *out_rem = rem - acc;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// Radix select (11 + 11 + 10 bits, warp-aggregated shared-memory atomics) over the elements
// i < n with member(i): the key of the rem-th largest and how many elements equal to it a
// selection of rem must take.  Results in *tau, *take (shared).
template <class KeyFn, class MemberFn>
__device__ void radix_select(int n, KeyFn key_of, MemberFn member, int rem, int* hist, int* scratch, int* sh_bin,
                             int* sh_rem, uint32_t* tau, int* take) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0, pmask = 0;
  int r = rem;
#pragma unroll 1
  for (int pass = 0; pass < 3; pass++) {
    const int dshift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
    for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kThreads) {
      const int i = i0 + tid;
      bool in = false;
      uint32_t digit = 0;
      if (i < n && member(i)) {
        const uint32_t u = key_of(i);
        in = (u & pmask) == prefix;
        digit = (u >> dshift) & dmask;
      }
      const unsigned active = __ballot_sync(kFull, in);
      if (in) {
        const unsigned peers = __match_any_sync(active, digit);
        if ((__ffs(peers) - 1) == (tid & 31)) atomicAdd(&hist[digit], __popc(peers));
      }
    }
    __syncthreads();
    find_bin_from_top(hist, r, scratch, sh_bin, sh_rem);
    prefix |= (uint32_t)*sh_bin << dshift;
    pmask |= dmask << dshift;
    r = *sh_rem;
    __syncthreads();
  }
  if (tid == 0) {
    *tau = prefix;
    *take = r;
  }
  __syncthreads();
}

// Emit, in index order, every element i < n whose key is above tau and the first
// take_total (in index order) whose key equals tau: o[...] = pos_of(i).  Each thread owns a
// contiguous run of indices; two block scans give the output offsets.  Returns the count.
template <class KeyFn, class PosFn>
__device__ int emit_ordered(int n, KeyFn key_of, PosFn pos_of, uint32_t tau, int take_total, int32_t* o, int k,
                            int* scratch) {
  const int tid = threadIdx.x;
  const int run = ((n + kThreads - 1) / kThreads) | 1;  // odd stride: conflict-free reads
  const int i0 = min(n, tid * run), i1 = min(n, i0 + run);
  int gt = 0, eq = 0;
  for (int i = i0; i < i1; i++) {
    const uint32_t u = key_of(i);
    gt += u > tau;
    eq += u == tau;
  }
  int tot;
  const int eq_before = block_excl_scan(eq, scratch, tot);
  const int take_eq = max(0, min(eq, take_total - eq_before));
  int total;
  int w = block_excl_scan(gt + take_eq, scratch, total);
  int te = 0;
  for (int i = i0; i < i1 && w < k; i++) {
    const uint32_t u = key_of(i);
    if (u > tau || (u == tau && te++ < take_eq)) o[w++] = pos_of(i);
  }
  return total;
}


// Exclusive scan over a block of NT threads (any multiple of 32 up to 1024).
template <int NT>
__device__ __forceinline__ int scan_nt(int v, int* scratch, int& total) {
  constexpr int W = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < W ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += n;
    }
    if (lane < W) scratch[lane] = w;
  }
  __syncthreads();
  const int before = (warp > 0 ? scratch[warp - 1] : 0) + x - v;
  total = scratch[W - 1];
  __syncthreads();
  return before;
}

template <int NT, bool kMax>
__device__ __forceinline__ uint32_t reduce_nt(uint32_t v, uint32_t* scratch) {
  constexpr int W = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t n = __shfl_xor_sync(kFull, v, o);
    v = kMax ? max(v, n) : min(v, n);
  }
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  uint32_t r = scratch[0];
  for (int i = 1; i < W; i++) r = kMax ? max(r, scratch[i]) : min(r, scratch[i]);
  __syncthreads();
  return r;
}

// ------------------------------------------------------------------ filter launch
// grid (chunks, rows).  Writes cnt[row][c] and the chunk's candidate positions, in order,
// at cand[row][c * kChunk ...].
__global__ void __launch_bounds__(kFilterThreads) topk_filter_kernel(const float* __restrict__ logits,
                                                                     int64_t stride,
                                                                     const int32_t* __restrict__ context_lens,
                                                                     int32_t max_context, int32_t k,
                                                                     int32_t* __restrict__ cand, int64_t cstride,
                                                                     int32_t* __restrict__ cnt, int32_t nch) {
  constexpr int NT = kFilterThreads;
  constexpr int kPer = kChunk / NT;  // 16 consecutive tokens per thread
  __shared__ int hist[kSampleBins];
  __shared__ int scratch[NT / 32];
  __shared__ uint32_t uscratch[NT / 32];
  __shared__ int sh_blo;
  const int64_t row = blockIdx.y;
  const int c = blockIdx.x;
  const int tid = threadIdx.x;
  int32_t L = __ldg(context_lens + row);
  L = L < 0 ? 0 : (L > max_context ? max_context : L);
  const int c0 = c * kChunk;
  if (L <= k || c0 >= L) {
    if (tid == 0) cnt[row * nch + c] = 0;
    return;
  }
  const float* lg = logits + row * stride;
  // the row's fixed sample: positions floor(i * L / kSample)
  uint32_t sk[kSample / NT];
  uint32_t smin = 0xFFFFFFFFu, smax = 0u;
#pragma unroll
  for (int j = 0; j < kSample / NT; j++) {
    const int i = j * NT + tid;
    sk[j] = order_key(__ldg(lg + (int)(((int64_t)i * L) / kSample)));
    smin = min(smin, sk[j]);
    smax = max(smax, sk[j]);
  }
  // this thread's 16 tokens (issued now, used after the threshold is known)
  float x[kPer];
  const int t0 = c0 + tid * kPer;
  const bool vec = ((reinterpret_cast<uintptr_t>(lg + t0) & 15) == 0) && t0 + kPer <= L;
  if (vec) {
#pragma unroll
    for (int q = 0; q < kPer / 4; q++) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(lg + t0) + q);
      x[4 * q] = v.x;
      x[4 * q + 1] = v.y;
      x[4 * q + 2] = v.z;
      x[4 * q + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int q = 0; q < kPer; q++) x[q] = t0 + q < L ? __ldg(lg + t0 + q) : 0.f;
  }
  for (int b = tid; b < kSampleBins; b += NT) hist[b] = 0;
  smin = reduce_nt<NT, false>(smin, uscratch);
  smax = reduce_nt<NT, true>(smax, uscratch);
  const float lo = key_value(smin);
  const float sc = lin_scale(lo, key_value(smax)) * ((float)kSampleBins / (float)kBins);
  auto bucket = [&](float v) -> int {
    const int b = lin_bucket(v, lo, sc);
    return b >= kSampleBins ? kSampleBins - 1 : b;
  };
#pragma unroll
  for (int j = 0; j < kSample / NT; j++) atomicAdd(&hist[bucket(key_value(sk[j]))], 1);
  __syncthreads();
  // keep the expected share of k in the sample plus four standard deviations
  const float q = (float)k / (float)L;
  const float mean = q * (float)kSample;
  const int need = min(kSample, (int)ceilf(mean + 4.0f * sqrtf(mean * (1.0f - q)) + 8.0f));
  const int mine = hist[kSampleBins - 1 - tid];  // NT == kSampleBins
  int tot;
  const int above = scan_nt<NT>(mine, scratch, tot);
  if (above < need && need <= above + mine) sh_blo = kSampleBins - 1 - tid;
  __syncthreads();
  const int blo = sh_blo;
  // order-preserving compaction of this chunk's passing tokens
  unsigned flags = 0;
  int nmine = 0;
#pragma unroll
  for (int qq = 0; qq < kPer; qq++) {
    const bool in = t0 + qq < L && bucket(x[qq]) >= blo;
    flags |= (unsigned)in << qq;
    nmine += in;
  }
  int total;
  int w = scan_nt<NT>(nmine, scratch, total);
  int32_t* dst = cand + row * cstride + c0;
#pragma unroll
  for (int qq = 0; qq < kPer; qq++)
    if (flags & (1u << qq)) dst[w++] = t0 + qq;
  if (tid == 0) cnt[row * nch + c] = total;
}

// ------------------------------------------------------------------ select launch
__global__ void __launch_bounds__(kThreads, 2) topk_select_kernel(const float* __restrict__ logits, int64_t stride,
                                                                  const int32_t* __restrict__ context_lens,
                                                                  int32_t max_context, int32_t k,
                                                                  const int32_t* __restrict__ cand, int64_t cstride,
                                                                  const int32_t* __restrict__ cnt, int32_t nch,
                                                                  int32_t* __restrict__ out, int32_t* status) {
  extern __shared__ __align__(16) uint32_t dyn[];  // ckey[kCapB], then cpos[kCapB]
  __shared__ int hist[kBins];
  __shared__ uint32_t gkey[kGather];
  __shared__ int gidx[kGather];
  __shared__ int scratch[kWarps];
  __shared__ uint32_t uscratch[kWarps];
  __shared__ int coff[kMaxChunks + 1];
  __shared__ int sh_bin, sh_rem, sh_gcount;
  __shared__ uint32_t sh_key;
  __shared__ int sh_take;
  uint32_t* ckey = dyn;
  int* cpos = reinterpret_cast<int*>(dyn + kCapB);

  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x;
  int32_t L = __ldg(context_lens + row);
  if (L < 0 || L > max_context) {
    if (tid == 0) record_error(status, FP4IDX_ERR_BAD_LENGTH);
    L = L < 0 ? 0 : max_context;
  }
  int32_t* o = out + row * k;
  if (L <= k) {
    for (int i = tid; i < k; i += kThreads) o[i] = i < L ? i : -1;
    return;
  }
  const float* lg = logits + row * stride;
  if (tid < 32) {  // chunk offsets into the concatenated candidate list
    int run = 0;
    for (int c0 = 0; c0 < nch; c0 += 32) {
      const int c = c0 + tid;
      int v = c < nch ? __ldg(cnt + row * nch + c) : 0;
      int x = v;
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const int n = __shfl_up_sync(kFull, x, o2);
        if (tid >= o2) x += n;
      }
      if (c < nch) coff[c] = run + x - v;
      run += __shfl_sync(kFull, x, 31);
    }
    if (tid == 0) coff[nch] = run;
  }
  __syncthreads();
  const int m = coff[nch];
  if (m >= k && m <= kCapB) {
    // gather the candidates (positions in order, and their keys)
    for (int i = tid; i < m; i += kThreads) {
      int c = 0;
      while (coff[c + 1] <= i) c++;
      const int pos = __ldg(cand + row * cstride + (int64_t)c * kChunk + (i - coff[c]));
      cpos[i] = pos;
      ckey[i] = order_key(__ldg(lg + pos));
    }
    __syncthreads();
    auto ck = [&](int i) -> uint32_t { return ckey[i]; };
    radix_select(m, ck, [](int) { return true; }, k, hist, scratch, &sh_bin, &sh_rem, &sh_key, &sh_take);
    const int got = emit_ordered(m, ck, [&](int i) { return cpos[i]; }, sh_key, sh_take, o, k, scratch);
    for (int i = got + tid; i < k; i += kThreads) o[i] = -1;  // only rows with non-finite logits
    return;
  }

  // ---- exact path over the whole row, read from global memory (L2)
  auto key_at = [&](int s) -> uint32_t { return order_key(__ldg(lg + s)); };
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int s = tid; s < L; s += kThreads) {
    const uint32_t u = key_at(s);
    kmin = min(kmin, u);
    kmax = max(kmax, u);
  }
  kmin = block_reduce<false>(kmin, uscratch);
  kmax = block_reduce<true>(kmax, uscratch);
  const float lo1 = key_value(kmin), sc1 = lin_scale(lo1, key_value(kmax));
  for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
  if (tid == 0) sh_gcount = 0;
  __syncthreads();
  for (int s = tid; s < L; s += kThreads) atomicAdd(&hist[lin_bucket(key_value(key_at(s)), lo1, sc1)], 1);
  __syncthreads();
  find_bin_from_top(hist, k, scratch, &sh_bin, &sh_rem);
  const int b1 = sh_bin;
  int rem = sh_rem;
  int nb = hist[b1];
  __syncthreads();  // every thread has read nb before any path clears the histogram
  float lo2 = 0.0f, sc2 = 0.0f;
  int b2 = -1;
  if (nb > kGather) {  // refine a crowded bucket over its own value range
    uint32_t bmin = 0xFFFFFFFFu, bmax = 0u;
    for (int s = tid; s < L; s += kThreads) {
      const uint32_t u = key_at(s);
      if (lin_bucket(key_value(u), lo1, sc1) == b1) {
        bmin = min(bmin, u);
        bmax = max(bmax, u);
      }
    }
    bmin = block_reduce<false>(bmin, uscratch);
    bmax = block_reduce<true>(bmax, uscratch);
    lo2 = key_value(bmin);
    sc2 = lin_scale(lo2, key_value(bmax));
    for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int s = tid; s < L; s += kThreads) {
      const float x = key_value(key_at(s));
      if (lin_bucket(x, lo1, sc1) == b1) atomicAdd(&hist[lin_bucket(x, lo2, sc2)], 1);
    }
    __syncthreads();
    find_bin_from_top(hist, rem, scratch, &sh_bin, &sh_rem);
    b2 = sh_bin;
    rem = sh_rem;
    nb = hist[b2];
    __syncthreads();
  }
  auto in_bucket = [&](uint32_t u) -> bool {
    const float x = key_value(u);
    return lin_bucket(x, lo1, sc1) == b1 && (b2 < 0 || lin_bucket(x, lo2, sc2) == b2);
  };
  if (nb <= kGather) {
    for (int s = tid; s < L; s += kThreads) {
      const uint32_t u = key_at(s);
      if (in_bucket(u)) {
        const int slot = atomicAdd(&sh_gcount, 1);
        gkey[slot] = u;
        gidx[slot] = s;
      }
    }
    __syncthreads();
    for (int i = tid; i < nb; i += kThreads) {
      const uint32_t ki = gkey[i];
      const int ii = gidx[i];
      int rk = 0;
      for (int j = 0; j < nb; j++) {
        const uint32_t kj = gkey[j];
        rk += (kj > ki) || (kj == ki && gidx[j] < ii);
      }
      if (rk == rem - 1) {
        int gt = 0;
        for (int j = 0; j < nb; j++) gt += gkey[j] > ki;
        sh_key = ki;
        sh_take = rem - gt;
      }
    }
    __syncthreads();
  } else {
    radix_select(L, key_at, [&](int s) { return in_bucket(key_at(s)); }, rem, hist, scratch, &sh_bin, &sh_rem,
                 &sh_key, &sh_take);
  }
  const int got = emit_ordered(L, key_at, [](int s) { return s; }, sh_key, sh_take, o, k, scratch);
  for (int i = got + tid; i < k; i += kThreads) o[i] = -1;  // only rows with non-finite logits
}

inline int num_chunks(int32_t max_context) { return (max(max_context, 1) + kChunk - 1) / kChunk; }
inline int64_t cand_stride(int32_t max_context) { return ((int64_t)max(max_context, 1) + 3) / 4 * 4; }

}  // namespace

size_t topk_workspace_bytes(int64_t n_rows, int32_t max_context) {
  const size_t c = (size_t)n_rows * (size_t)cand_stride(max_context) * sizeof(int32_t);
  const size_t n = (size_t)n_rows * (size_t)num_chunks(max_context) * sizeof(int32_t);
  return ((c + 15) & ~(size_t)15) + ((n + 15) & ~(size_t)15);
}

cudaError_t launch_topk(const float* logits, int64_t stride, const int32_t* context_lens, int32_t n_rows,
                        int32_t max_context, int32_t k, void* workspace, int32_t* out, int32_t* status,
                        cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(2 * kCapB * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int nch = num_chunks(max_context);
  const int64_t cst = cand_stride(max_context);
  int32_t* cand = reinterpret_cast<int32_t*>(workspace);
  const size_t cbytes = (((size_t)n_rows * (size_t)cst * sizeof(int32_t)) + 15) & ~(size_t)15;
  int32_t* cnt = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(workspace) + cbytes);
  topk_filter_kernel<<<dim3(nch, n_rows), kFilterThreads, 0, stream>>>(logits, stride, context_lens, max_context, k,
                                                                       cand, cst, cnt, nch);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  topk_select_kernel<<<n_rows, kThreads, 2 * kCapB * sizeof(uint32_t), stream>>>(
      logits, stride, context_lens, max_context, k, cand, cst, cnt, nch, out, status);
  return cudaGetLastError();
}

}  // namespace fp4idx
