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
//      buckets, so the shared-memory atomics rarely collide.
//   2. the bucket holding the k-th largest is resolved exactly: its few candidates are
//      gathered and ranked by (key desc, index asc).  When it holds more than kGather
//      candidates (a degenerate row: many equal values), a radix select over the exact
//      keys with warp-aggregated atomics takes over.
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

__device__ __forceinline__ int bucket_of(float x, float lo, float scale) {
  const float v = (x - lo) * scale;
  if (!(v >= 0.0f)) return 0;  // also NaN
  return v >= (float)(kBins - 1) ? kBins - 1 : (int)v;
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
__device__ __forceinline__ float block_reduce(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float n = __shfl_xor_sync(kFull, v, o);
    v = kMax ? fmaxf(v, n) : fminf(v, n);
  }
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float r = scratch[0];
  for (int i = 1; i < kWarps; i++) r = kMax ? fmaxf(r, scratch[i]) : fminf(r, scratch[i]);
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
  __shared__ float fscratch[kWarps];
  __shared__ int sh_bin, sh_rem, sh_gcount;
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
  float mn = INFINITY, mx = -INFINITY;
  for (int s = tid; s < L; s += kThreads) {
    const float x = __ldg(lg + s);
    mn = fminf(mn, x);
    mx = fmaxf(mx, x);
    if (cached) keys[s] = order_key(x);
  }
  for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
  mn = block_reduce<false>(mn, fscratch);
  mx = block_reduce<true>(mx, fscratch);
  const float range = mx - mn;
  const float scale = (range > 0.0f && range < INFINITY) ? (float)(kBins - 1) / range : 0.0f;
  auto key_at = [&](int s) -> uint32_t { return cached ? keys[s] : order_key(__ldg(lg + s)); };

  // 1. bucket histogram
  for (int s = tid; s < L; s += kThreads) atomicAdd(&hist[bucket_of(key_value(key_at(s)), mn, scale)], 1);
  if (tid == 0) sh_gcount = 0;
  __syncthreads();
  find_bin_from_top(hist, k, scratch, &sh_bin, &sh_rem);
  const int bstar = sh_bin;
  const int rem = sh_rem;
  const int nb = hist[bstar];

  // 2. resolve the threshold bucket: threshold key tau and how many keys equal to tau to keep
  if (nb <= kGather) {
    for (int s = tid; s < L; s += kThreads) {
      const uint32_t u = key_at(s);
      if (bucket_of(key_value(u), mn, scale) == bstar) {
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
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
      for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
      __syncthreads();
      for (int base = 0; base < L; base += kThreads) {
        const int s = base + tid;
        bool take = false;
        uint32_t digit = 0;
        if (s < L) {
          const uint32_t u = key_at(s);
          take = bucket_of(key_value(u), mn, scale) == bstar && (u & pmask) == prefix;
          digit = (u >> shift) & dmask;
        }
        const unsigned active = __ballot_sync(kFull, take);
        if (take) {
          const unsigned peers = __match_any_sync(active, digit);
          if ((__ffs(peers) - 1) == (tid & 31)) atomicAdd(&hist[digit], __popc(peers));
        }
      }
      __syncthreads();
      find_bin_from_top(hist, r, scratch, &sh_bin, &sh_rem);
      prefix |= (uint32_t)sh_bin << shift;
      pmask |= dmask << shift;
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
