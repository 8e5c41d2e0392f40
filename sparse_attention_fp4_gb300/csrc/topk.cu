// Per-row top-k of the logits, emitted as ascending compressed-token indices.
//
// [AMD] DeepSeek-V4.1-Flash on MI350X (gfx950) -- Changes: "sorted top-k selection";
// Historical results: the decode top-k is ordered by position, not by KV slot.
// [AMD] Enable FP4 indexer for Deepseek V4 -- Attention runtime: padded rows keep
// context length 0 (their selection is empty: all -1).
//
// One CTA per query row; the row's logits are cached in shared memory as
// order-preserving 32-bit keys.  Selection = the k largest (ties at the k-th value to the
// lower positions), found in three steps:
//   1. bucket histogram: 2048 buckets linear in value between the row's min and max.
//      floor((x - min) * 2047/(max - min)) is non-decreasing in x, so every logit in a
//      higher bucket is larger than every logit in a lower one; values spread over the
//      buckets, so the shared-memory atomics rarely collide.  When the bucket holding the
//      k-th largest is crowded (heavy tails), a second linear histogram over that
//      bucket's own value range narrows it.
//   2. the candidates of the final bucket are gathered and ranked by (key desc, index
//      asc).  When more than kGather remain (many equal values), a radix select over the
//      exact keys with warp-aggregated atomics takes over.
//   3. one ordered pass keeps every key above the threshold key and the lowest-indexed
//      keys equal to it: each thread owns a contiguous run of positions, two block scans
//      give the output offsets, so the selection comes out sorted by position.
#include "fp4idx_internal.cuh"

namespace fp4idx {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kThreads;
constexpr int kGather = 1024;
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
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
// element writes (bin, rem - elements above the bin).  `counts` holds nbins bins.
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

__global__ void __launch_bounds__(kThreads) topk_kernel(const float* __restrict__ logits, int64_t stride,
                                                        const int32_t* __restrict__ context_lens, int32_t max_context,
                                                        int32_t k, int32_t* __restrict__ out, int32_t smem_cap,
                                                        int32_t* status) {
  extern __shared__ __align__(16) uint32_t keys[];
  __shared__ int hist[kBins];
  __shared__ uint32_t gkey[kGather];
  __shared__ int gidx[kGather];
  __shared__ int scratch[kWarps];
  __shared__ uint32_t uscratch[kWarps];
  __shared__ int sh_bin, sh_rem, sh_gcount;
  __shared__ uint32_t sh_kmin, sh_kmax;
  __shared__ uint32_t sh_key;
  __shared__ int sh_take;

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
  const bool cached = L <= smem_cap;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  auto take = [&](int s, float x) {
    const uint32_t u = order_key(x);
    kmin = min(kmin, u);
    kmax = max(kmax, u);
    if (cached) keys[s] = u;
  };
  // The row comes from L2 or HBM: keep four 16-byte loads in flight per thread.
  int s_done = 0;
  if ((stride & 3) == 0 && (reinterpret_cast<uintptr_t>(lg) & 15) == 0) {
    const float4* lg4 = reinterpret_cast<const float4*>(lg);
    const int L4 = L >> 2;
    for (int v0 = 0; v0 < L4; v0 += 4 * kThreads) {
      float4 x[4];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int v = v0 + u * kThreads + tid;
        x[u] = v < L4 ? __ldg(lg4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int v = v0 + u * kThreads + tid;
        if (v < L4) {
          take(4 * v, x[u].x);
          take(4 * v + 1, x[u].y);
          take(4 * v + 2, x[u].z);
          take(4 * v + 3, x[u].w);
        }
      }
    }
    s_done = L4 << 2;
  }
  for (int s0 = s_done; s0 < L; s0 += 4 * kThreads) {
    float x[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int s = s0 + u * kThreads + tid;
      x[u] = s < L ? __ldg(lg + s) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int s = s0 + u * kThreads + tid;
      if (s < L) take(s, x[u]);
    }
  }
  for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
  kmin = block_reduce<false>(kmin, uscratch);
  kmax = block_reduce<true>(kmax, uscratch);
  auto key_at = [&](int s) -> uint32_t { return cached ? keys[s] : order_key(__ldg(lg + s)); };

  // 1. bucket histogram over [min, max]
  const float lo1 = key_value(kmin), sc1 = lin_scale(lo1, key_value(kmax));
  for (int s = tid; s < L; s += kThreads) atomicAdd(&hist[lin_bucket(key_value(key_at(s)), lo1, sc1)], 1);
  if (tid == 0) {
    sh_gcount = 0;
    sh_kmin = 0xFFFFFFFFu;
    sh_kmax = 0u;
  }
  __syncthreads();
  find_bin_from_top(hist, k, scratch, &sh_bin, &sh_rem);
  const int b1 = sh_bin;
  int rem = sh_rem;
  int nb = hist[b1];
  __syncthreads();  // every thread has read nb before any path clears the histogram
  // optional refinement of a crowded bucket over its own value range
  float lo2 = 0.0f, sc2 = 0.0f;
  int b2 = -1;
  if (nb > kGather) {
    for (int s = tid; s < L; s += kThreads) {
      const uint32_t u = key_at(s);
      if (lin_bucket(key_value(u), lo1, sc1) == b1) {
        atomicMin(&sh_kmin, u);
        atomicMax(&sh_kmax, u);
      }
    }
    for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
    __syncthreads();
    lo2 = key_value(sh_kmin);
    sc2 = lin_scale(lo2, key_value(sh_kmax));
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
  // membership of the final candidate bucket
  auto in_bucket = [&](uint32_t u) -> bool {
    const float x = key_value(u);
    return lin_bucket(x, lo1, sc1) == b1 && (b2 < 0 || lin_bucket(x, lo2, sc2) == b2);
  };

  // 2. resolve the threshold bucket: threshold key tau and how many keys equal to tau to keep
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
      int rank = 0;
      for (int j = 0; j < nb; j++) {
        const uint32_t kj = gkey[j];
        rank += (kj > ki) || (kj == ki && gidx[j] < ii);
      }
      if (rank == rem - 1) {
        int gt = 0;
        for (int j = 0; j < nb; j++) gt += gkey[j] > ki;
        sh_key = ki;
        sh_take = rem - gt;
      }
    }
    __syncthreads();
  } else {
    // degenerate bucket: exact radix select over the keys inside it (11 + 11 + 10 bits)
    uint32_t prefix = 0, pmask = 0;
    int r = rem;
#pragma unroll 1
    for (int pass = 0; pass < 3; pass++) {
      const int dshift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
      for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
      __syncthreads();
      for (int s_base = 0; s_base < L; s_base += kThreads) {
        const int s = s_base + tid;
        bool take = false;
        uint32_t digit = 0;
        if (s < L) {
          const uint32_t u = key_at(s);
          take = in_bucket(u) && (u & pmask) == prefix;
          digit = (u >> dshift) & dmask;
        }
        const unsigned active = __ballot_sync(kFull, take);
        if (take) {
          const unsigned peers = __match_any_sync(active, digit);
          if ((__ffs(peers) - 1) == (tid & 31)) atomicAdd(&hist[digit], __popc(peers));
        }
      }
      __syncthreads();
      find_bin_from_top(hist, r, scratch, &sh_bin, &sh_rem);
      prefix |= (uint32_t)sh_bin << dshift;
      pmask |= dmask << dshift;
      r = sh_rem;
      __syncthreads();
    }
    if (tid == 0) {
      sh_key = prefix;
      sh_take = r;
    }
    __syncthreads();
  }
  const uint32_t tau = sh_key;
  const int take_total = sh_take;

  // 3. ordered output
  int chunk = (L + kThreads - 1) / kThreads;
  chunk |= 1;  // odd stride between threads' runs: conflict-free shared-memory reads
  const int s0 = min(L, tid * chunk), s1 = min(L, s0 + chunk);
  int gt = 0, eq = 0;
  for (int s = s0; s < s1; s++) {
    const uint32_t u = key_at(s);
    gt += u > tau;
    eq += u == tau;
  }
  int tot;
  const int eq_before = block_excl_scan(eq, scratch, tot);
  const int take_eq = max(0, min(eq, take_total - eq_before));
  const int pos = block_excl_scan(gt + take_eq, scratch, tot);
  int w = pos, te = 0;
  for (int s = s0; s < s1 && w < k; s++) {
    const uint32_t u = key_at(s);
    if (u > tau || (u == tau && te++ < take_eq)) o[w++] = s;
  }
  for (int i = tot + tid; i < k; i += kThreads) o[i] = -1;  // only for non-finite rows
}

}  // namespace

int32_t topk_smem_cap() { return 49152; }

cudaError_t launch_topk(const float* logits, int64_t stride, const int32_t* context_lens, int32_t n_rows,
                        int32_t max_context, int32_t k, int32_t* out, int32_t* status, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  const int32_t cap = min(max_context, topk_smem_cap());
  const size_t smem = (size_t)(cap > 0 ? cap : 1) * sizeof(uint32_t);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(topk_smem_cap() * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  topk_kernel<<<n_rows, kThreads, smem, stream>>>(logits, stride, context_lens, max_context, k, out, cap, status);
  return cudaGetLastError();
}

}  // namespace fp4idx
