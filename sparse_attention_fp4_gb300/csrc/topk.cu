// Per-row top-k of the logits, emitted as ascending compressed-token indices.
//
// [AMD] DeepSeek-V4.1-Flash on MI350X (gfx950) -- Changes: "sorted top-k selection";
// Historical results: the decode top-k is ordered by position, not by KV slot.
// [AMD] Enable FP4 indexer for Deepseek V4 -- Attention runtime: padded rows keep
// context length 0 (their selection is empty: all -1).
//
// One CTA per query row.  Logits become order-preserving 32-bit keys (cached in shared
// memory when the row fits); a three-pass radix select (11 + 11 + 10 bits, shared-memory
// histograms) finds the key of the k-th largest logit; a block scan in index order then
// keeps every key above it plus the lowest-indexed keys equal to it, which writes the
// selection already sorted by position.  Rows with context_len <= k keep all tokens.
#include "fp4idx_internal.cuh"

namespace fp4idx {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kThreads;
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block scan of an int; returns the prefix, `total` gets the block sum.
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

__global__ void __launch_bounds__(kThreads) topk_kernel(const float* __restrict__ logits, int64_t stride,
                                                        const int32_t* __restrict__ context_lens, int32_t max_context,
                                                        int32_t k, int32_t* __restrict__ out, int32_t smem_cap,
                                                        int32_t* status) {
  extern __shared__ __align__(16) uint32_t keys[];
  __shared__ int hist[kBins];
  __shared__ int scratch[kWarps];
  __shared__ uint32_t sel_prefix;
  __shared__ int sel_rem;

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
  if (cached)
    for (int s = tid; s < L; s += kThreads) keys[s] = order_key(__ldg(lg + s));
  __syncthreads();
  auto key_at = [&](int s) -> uint32_t { return cached ? keys[s] : order_key(__ldg(lg + s)); };

  uint32_t prefix = 0, pmask = 0;
  int rem = k;
#pragma unroll 1
  for (int pass = 0; pass < 3; pass++) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
    for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int s = tid; s < L; s += kThreads) {
      const uint32_t u = key_at(s);
      if ((u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & dmask], 1);
    }
    __syncthreads();
    // counts at or above each thread's bins, from the top bin down
    const int tb = (kThreads - 1 - tid) * kBinsPerThread;  // this thread's lowest bin, top first
    int mine = 0;
#pragma unroll
    for (int j = 0; j < kBinsPerThread; j++) mine += hist[tb + j];
    int tot;
    const int above = block_excl_scan(mine, scratch, tot);  // elements in bins above this thread's
    if (above < rem && rem <= above + mine) {
      int acc = above;
      for (int j = kBinsPerThread - 1; j >= 0; j--) {
        const int c = hist[tb + j];
        if (acc < rem && rem <= acc + c) {
          sel_prefix = prefix | ((uint32_t)(tb + j) << shift);
          sel_rem = rem - acc;
          break;
        }
        acc += c;
      }
    }
    __syncthreads();
    prefix = sel_prefix;
    rem = sel_rem;
    pmask |= dmask << shift;
    __syncthreads();
  }
  // prefix = key of the k-th largest; keep all keys above it and the first `rem` equal ones.
  const int chunk = (L + kThreads - 1) / kThreads;
  const int s0 = min(L, tid * chunk), s1 = min(L, s0 + chunk);
  int gt = 0, eq = 0;
  for (int s = s0; s < s1; s++) {
    const uint32_t u = key_at(s);
    gt += u > prefix;
    eq += u == prefix;
  }
  int tot;
  const int eq_before = block_excl_scan(eq, scratch, tot);
  const int take_eq = max(0, min(eq, rem - eq_before));
  const int pos = block_excl_scan(gt + take_eq, scratch, tot);
  int w = pos, te = 0;
  for (int s = s0; s < s1; s++) {
    const uint32_t u = key_at(s);
    if (u > prefix || (u == prefix && te++ < take_eq)) o[w++] = s;
  }
}

}  // namespace

int32_t topk_smem_cap() { return 49152; }

cudaError_t launch_topk(const float* logits, int64_t stride, const int32_t* context_lens, int32_t n_rows,
                        int32_t max_context, int32_t k, int32_t* out, int32_t* status, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  const int32_t cap = min(max_context, topk_smem_cap());
  const size_t smem = (size_t)(cap > 0 ? cap : 1) * sizeof(uint32_t);
  static size_t attr_bytes = 0;
  if (smem > attr_bytes) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(topk_smem_cap() * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    attr_bytes = topk_smem_cap() * sizeof(uint32_t);
  }
  topk_kernel<<<n_rows, kThreads, smem, stream>>>(logits, stride, context_lens, max_context, k, out, cap, status);
  return cudaGetLastError();
}

}  // namespace fp4idx
