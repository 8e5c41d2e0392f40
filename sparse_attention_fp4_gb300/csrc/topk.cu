// Per-row top-k of the logits, emitted as ascending compressed-token indices.
//
// [AMD] DeepSeek-V4.1-Flash on MI350X (gfx950) -- Changes: "sorted top-k selection";
// Historical results: the decode top-k is ordered by position, not by KV slot.
// [AMD] Enable FP4 indexer for Deepseek V4 -- Attention runtime: padded rows keep
// context length 0 (their selection is empty: all -1).
//
// Selection = the k largest logits of a row, ties at the k-th value to the lower
// positions, emitted in ascending position order.  One CTA of 512 threads per row and
// no communication between CTAs (every hand-off between CTAs -- a global candidate list,
// a fence and an arrival counter -- cost microseconds of latency on this path):
//   1. a fixed sample of 1,024 of the row's logits (128 runs of 8 adjacent logits) gives
//      a conservative threshold: a linear 256-bucket histogram of the sample, cut about
//      four standard deviations beyond the expected place of the k-th largest;
//   2. the row, 32 logits per thread held in registers (blocks of 16,384 tokens, read as
//      float4 groups interleaved across the threads so that loads coalesce), is compacted
//      in position order into the candidates at or above the threshold: in shared memory
//      when they fit (kCapB), else in the caller's workspace;
//   3. the candidates are bucketed linearly between their min and max (2,048 buckets),
//      the boundary bucket is ranked exactly (radix select when it is crowded with
//      ties), and the keys above the k-th plus the lowest-positioned equal ones are
//      emitted in order.
// The threshold is superset-closed (a value that passes lets every larger one pass), so
// with at least k candidates they hold the whole answer: the sample decides speed, never
// the result.  With fewer than k candidates the exact path runs over the whole row.
#include "fp4idx_internal.cuh"

#include <atomic>

namespace fp4idx {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kPer = 32;                      // logits a thread holds per block
constexpr int kBlockTokens = kThreads * kPer; // 32,768
constexpr int kCapB = 8192;                   // candidates kept in shared memory
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kThreads;
constexpr int kGather = 1024;                 // largest boundary bucket ranked by direct counting
constexpr int kSample = 1024;                 // logits per row behind the candidate threshold
constexpr int kSampleBins = 256;
constexpr size_t kDynSmem = kCapB * (sizeof(uint32_t) + sizeof(uint16_t)) + FP4IDX_MAX_TOPK * sizeof(int32_t);
constexpr int kSamplePer = kSample / kThreads;  // sample logits a thread loads
static_assert(kSampleBins <= kThreads && kSample % kThreads == 0 && kBins % kThreads == 0 && kPer % 8 == 0,
              "layout");
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
// Exclusive block scan of a 64-bit value; `total` gets the block sum.
__device__ __forceinline__ uint64_t block_excl_scan64(uint64_t v, uint64_t* scratch, uint64_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t n = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint64_t w = lane < kWarps ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t n = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += n;
    }
    if (lane < kWarps) scratch[lane] = w;
  }
  __syncthreads();
  const uint64_t before = (warp > 0 ? scratch[warp - 1] : 0) + x - v;
  total = scratch[kWarps - 1];
  __syncthreads();
  return before;
}

// Writes o[0..k): the selected positions in index order, then -1.  They are staged in
// shared memory (`stage`, k entries) and copied out with coalesced stores.
template <class KeyFn, class PosFn>
__device__ void emit_ordered(int n, KeyFn key_of, PosFn pos_of, uint32_t tau, int take_total, int32_t* o, int k,
                             uint64_t* scratch, int32_t* stage) {
  const int tid = threadIdx.x;
  const int run = ((n + kThreads - 1) / kThreads) | 1;  // odd stride: conflict-free reads
  const int i0 = min(n, tid * run), i1 = min(n, i0 + run);
  int gt = 0, eq = 0;
  for (int i = i0; i < i1; i++) {
    const uint32_t u = key_of(i);
    gt += u > tau;
    eq += u == tau;
  }
  // one scan of (greater, equal) counts: the equal keys are taken greedily in index
  // order, so the keys equal to tau taken before this thread's run are min(E, take)
  uint64_t tot;
  const uint64_t pre = block_excl_scan64(((uint64_t)gt << 32) | (uint32_t)eq, scratch, tot);
  const int G = (int)(pre >> 32), E = (int)(uint32_t)pre;
  const int take_eq = max(0, min(eq, take_total - E));
  int w = G + min(E, take_total);
  const int total = (int)(tot >> 32) + min((int)(uint32_t)tot, take_total);
  int te = 0;
  for (int i = i0; i < i1 && w < k; i++) {
    const uint32_t u = key_of(i);
    if (u > tau || (u == tau && te++ < take_eq)) stage[w++] = pos_of(i);
  }
  __syncthreads();
  const int got = min(total, k);  // below k only for rows with non-finite logits
  for (int i = threadIdx.x; i < k; i += kThreads) o[i] = i < got ? stage[i] : -1;
}

// Block-wide min and max of uint32 keys in one barrier round; scratch holds 2 * kWarps.
__device__ __forceinline__ void block_minmax(uint32_t& mn, uint32_t& mx, uint32_t* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(kFull, mn, o));
    mx = max(mx, __shfl_xor_sync(kFull, mx, o));
  }
  if (lane == 0) {
    scratch[warp] = mn;
    scratch[kWarps + warp] = mx;
  }
  __syncthreads();
  mn = scratch[0];
  mx = scratch[kWarps];
#pragma unroll
  for (int i = 1; i < kWarps; i++) {
    mn = min(mn, scratch[i]);
    mx = max(mx, scratch[kWarps + i]);
  }
  __syncthreads();
}

struct Shared {
  uint32_t wsum[kWarps][kPer / 8];
  uint32_t gsum[kPer / 8];
  uint64_t scratch64[kWarps];
  int hist[kBins];
  uint32_t gkey[kGather];
  int gidx[kGather];
  int scratch[kWarps];
  uint32_t uscratch[2 * kWarps];
  int bin, rem, gcount, take, blo, last;
  uint32_t key;
};

// Members of the boundary bucket (nb <= kGather of them, keys from key_of) ranked by
// direct counting: sets sh.key to the rem-th largest and sh.take to how many keys equal
// to it the selection takes.  `in_bucket(i)` says whether element i is a member.
template <class KeyFn, class InFn>
__device__ void rank_bucket(int n, KeyFn key_of, InFn in_bucket, int nb, int rem, Shared& sh) {
  const int tid = threadIdx.x;
  for (int i = tid; i < n; i += kThreads) {
    if (in_bucket(i)) {
      const int slot = atomicAdd(&sh.gcount, 1);
      sh.gkey[slot] = key_of(i);
      sh.gidx[slot] = i;
    }
  }
  __syncthreads();
  for (int i = tid; i < nb; i += kThreads) {
    const uint32_t ki = sh.gkey[i];
    const int ii = sh.gidx[i];
    int rk = 0, gt = 0;
    for (int j = 0; j < nb; j++) {
      const uint32_t kj = sh.gkey[j];
      gt += kj > ki;
      rk += (kj > ki) || (kj == ki && sh.gidx[j] < ii);
    }
    if (rk == rem - 1) {
      sh.key = ki;
      sh.take = rem - gt;
    }
  }
  __syncthreads();
}

// Exact selection over the whole row, read from global memory: the path for rows whose
// candidate set came out too small or too large.
__device__ void select_whole_row(const float* lg, int L, int k, int32_t* o, Shared& sh, int32_t* stage) {
  const int tid = threadIdx.x;
  auto key_at = [&](int s) -> uint32_t { return order_key(__ldg(lg + s)); };
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int s = tid; s < L; s += kThreads) {
    const uint32_t u = key_at(s);
    kmin = min(kmin, u);
    kmax = max(kmax, u);
  }
  for (int b = tid; b < kBins; b += kThreads) sh.hist[b] = 0;
  if (tid == 0) sh.gcount = 0;
  block_minmax(kmin, kmax, sh.uscratch);
  const float lo1 = key_value(kmin), sc1 = lin_scale(lo1, key_value(kmax));
  for (int s = tid; s < L; s += kThreads) atomicAdd(&sh.hist[lin_bucket(key_value(key_at(s)), lo1, sc1)], 1);
  __syncthreads();
  find_bin_from_top(sh.hist, k, sh.scratch, &sh.bin, &sh.rem);
  const int b1 = sh.bin;
  int rem = sh.rem;
  int nb = sh.hist[b1];
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
    for (int b = tid; b < kBins; b += kThreads) sh.hist[b] = 0;
    block_minmax(bmin, bmax, sh.uscratch);
    lo2 = key_value(bmin);
    sc2 = lin_scale(lo2, key_value(bmax));
    for (int s = tid; s < L; s += kThreads) {
      const float x = key_value(key_at(s));
      if (lin_bucket(x, lo1, sc1) == b1) atomicAdd(&sh.hist[lin_bucket(x, lo2, sc2)], 1);
    }
    __syncthreads();
    find_bin_from_top(sh.hist, rem, sh.scratch, &sh.bin, &sh.rem);
    b2 = sh.bin;
    rem = sh.rem;
    nb = sh.hist[b2];
    __syncthreads();
  }
  auto in_bucket = [&](int s) -> bool {
    const float x = key_value(key_at(s));
    return lin_bucket(x, lo1, sc1) == b1 && (b2 < 0 || lin_bucket(x, lo2, sc2) == b2);
  };
  if (nb <= kGather) {
    rank_bucket(L, key_at, in_bucket, nb, rem, sh);
  } else {
    radix_select(L, key_at, in_bucket, rem, sh.hist, sh.scratch, &sh.bin, &sh.rem, &sh.key, &sh.take);
  }
  emit_ordered(L, key_at, [](int s) { return s; }, sh.key, sh.take, o, k, sh.scratch64, stage);
}


constexpr int kGroups = kPer / 4;  // float4 groups a thread holds per block

// Position of element e of this thread's group j in a block starting at `base`: groups are
// interleaved across the threads (group j of thread t covers base + 4*(j*kThreads + t)),
// so each warp-wide 16-byte load reads 512 contiguous bytes.
__device__ __forceinline__ int elem_pos(int base, int j, int e) {
  return base + 4 * (j * kThreads + (int)threadIdx.x) + e;
}

// This thread's kPer logits of the block starting at `base`; past L reads nothing and
// yields 0.
__device__ __forceinline__ void load_block(const float* lg, int base, int L, float* x) {
  const bool vec = (reinterpret_cast<uintptr_t>(lg) & 15) == 0;
#pragma unroll
  for (int j = 0; j < kGroups; j++) {
    const int p0 = elem_pos(base, j, 0);
    if (vec && p0 + 4 <= L) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(lg + p0));
      x[4 * j] = v.x;
      x[4 * j + 1] = v.y;
      x[4 * j + 2] = v.z;
      x[4 * j + 3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; e++) x[4 * j + e] = p0 + e < L ? __ldg(lg + p0 + e) : 0.0f;
    }
  }
}

// Exclusive prefix, in (group, thread) order, of this thread's per-group counts c[j]
// (each at most 4): off[j] = sum of all counts of groups before j plus those of lower
// threads in group j.  Counts travel two to a register in 16-bit halves (a block total
// is at most 4 * kThreads = 4096).  Returns the block total.
__device__ __forceinline__ int group_scan(const int* c, int* off, uint32_t (*wsum)[kGroups / 2], uint32_t* gsum) {
  constexpr int P = kGroups / 2;
  static_assert(kWarps <= 32, "one warp scans the warp sums");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t v[P], x[P];
#pragma unroll
  for (int i = 0; i < P; i++) x[i] = v[i] = (uint32_t)c[2 * i] | ((uint32_t)c[2 * i + 1] << 16);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < P; i++) {
      const uint32_t n = __shfl_up_sync(kFull, x[i], o);
      if (lane >= o) x[i] += n;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int i = 0; i < P; i++) wsum[warp][i] = x[i];
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the kWarps warp sums; gsum = per-group block totals
    uint32_t y[P], z[P];
#pragma unroll
    for (int i = 0; i < P; i++) z[i] = y[i] = lane < kWarps ? wsum[lane][i] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
      for (int i = 0; i < P; i++) {
        const uint32_t n = __shfl_up_sync(kFull, z[i], o);
        if (lane >= o) z[i] += n;
      }
    }
#pragma unroll
    for (int i = 0; i < P; i++) {
      if (lane < kWarps) wsum[lane][i] = z[i] - y[i];
      if (lane == kWarps - 1) gsum[i] = z[i];
    }
  }
  __syncthreads();
  int base = 0;
#pragma unroll
  for (int i = 0; i < P; i++) {
    const uint32_t pre = x[i] - v[i] + wsum[warp][i];  // within-group exclusive prefix, packed
    const uint32_t tot = gsum[i];
    off[2 * i] = base + (int)(pre & 0xFFFFu);
    base += (int)(tot & 0xFFFFu);
    off[2 * i + 1] = base + (int)(pre >> 16);
    base += (int)(tot >> 16);
  }
  __syncthreads();  // wsum / gsum may be reused
  return base;
}

// One CTA per row.  cand_key/cand_pos + row * cstride: the row's region of the workspace,
// used when its candidates do not fit in shared memory.
__global__ void __launch_bounds__(kThreads, 1) topk_row_kernel(const float* __restrict__ logits, int64_t stride,
                                                               const int32_t* __restrict__ context_lens,
                                                               int32_t max_context, int32_t k, uint32_t* cand_key,
                                                               uint16_t* cand_pos, int64_t cstride,
                                                               int32_t* __restrict__ out, int32_t* status) {
  extern __shared__ __align__(16) uint32_t dyn[];  // ckey[kCapB], cpos[kCapB] (uint16), stage[k]
  __shared__ Shared sh;
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
  int32_t* const stage = reinterpret_cast<int32_t*>(dyn + kCapB + kCapB / 2);  // after ckey and cpos

  // ---- 1. threshold from the row's fixed sample: 128 runs of 8 adjacent logits starting
  // at floor(r * L / 128) rounded down to 8 (single logits at floor(i * L / 1024) for
  // rows shorter than 1024)
  float sv[kSamplePer];
#pragma unroll
  for (int j = 0; j < kSamplePer; j++) {
    const int i = j * kThreads + tid;
    const int sp = L >= kSample ? (((int)(((int64_t)(i >> 3) * L) / (kSample / 8)) & ~7) + (i & 7))
                                : (int)(((int64_t)i * L) / kSample);
    sv[j] = __ldg(lg + sp);
  }
  float x[kPer];
  load_block(lg, 0, L, x);  // issued before the threshold is known
  if (tid < kSampleBins) sh.hist[tid] = 0;
  uint32_t smin = 0xFFFFFFFFu, smax = 0u;
#pragma unroll
  for (int j = 0; j < kSamplePer; j++) {
    smin = min(smin, order_key(sv[j]));
    smax = max(smax, order_key(sv[j]));
  }
  block_minmax(smin, smax, sh.uscratch);  // its barriers also order the histogram clear
  const float lo = key_value(smin);
  const float sc = lin_scale(lo, key_value(smax)) * ((float)kSampleBins / (float)kBins);
  auto sbucket = [&](float v) -> int {
    const int b = lin_bucket(v, lo, sc);
    return b >= kSampleBins ? kSampleBins - 1 : b;
  };
#pragma unroll
  for (int j = 0; j < kSamplePer; j++) atomicAdd(&sh.hist[sbucket(sv[j])], 1);
  __syncthreads();
  // keep the sample's expected share of k plus four standard deviations
  const float q = (float)k / (float)L;
  const float mean = q * (float)kSample;
  const int need = min(kSample, (int)ceilf(mean + 4.0f * sqrtf(mean * (1.0f - q)) + 8.0f));
  const int mine = tid < kSampleBins ? sh.hist[kSampleBins - 1 - tid] : 0;
  int tot;
  const int above = block_excl_scan(mine, sh.scratch, tot);
  if (tid < kSampleBins && above < need && need <= above + mine) sh.blo = kSampleBins - 1 - tid;
  __syncthreads();
  const int blo = sh.blo;
  // the cut as a key: bucket blo starts at lo + blo / sc.  Any key threshold keeps the
  // candidate set superset-closed, so the rounding of this edge cannot change the result.
  const uint32_t kthr = (blo == 0 || !(sc > 0.0f)) ? 0u : order_key(lo + (float)blo / sc);

  // ---- 2. order-preserving compaction of the candidates, block by block.  Candidate i
  // lives in shared memory for i < kCapB and in the row's workspace region beyond.
  uint32_t* const ckey_s = dyn;
  uint16_t* const cpos_s = reinterpret_cast<uint16_t*>(dyn + kCapB);
  uint32_t* const ckey_g = cand_key + row * cstride;
  uint16_t* const cpos_g = cand_pos + row * cstride;
  const int nblocks = (L + kBlockTokens - 1) / kBlockTokens;
  int m = 0;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int blk = 0; blk < nblocks; blk++) {
    const int base = blk * kBlockTokens;
    if (blk > 0) load_block(lg, base, L, x);
    unsigned flags = 0;
    int cnt[kGroups], off[kGroups];
#pragma unroll
    for (int j = 0; j < kGroups; j++) {
      const int p0 = elem_pos(base, j, 0);
      cnt[j] = 0;
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const bool in = p0 + e < L && order_key(x[4 * j + e]) >= kthr;
        flags |= (unsigned)in << (4 * j + e);
        cnt[j] += in;
      }
    }
    const int total = group_scan(cnt, off, sh.wsum, sh.gsum);
    if (m + total <= kCapB) {  // the common case, uniform over the CTA: branch-free stores
#pragma unroll
      for (int j = 0; j < kGroups; j++) {
        int w = m + off[j];
        const int p0 = elem_pos(base, j, 0);
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const bool in = (flags >> (4 * j + e)) & 1u;
          const uint32_t u = order_key(x[4 * j + e]);
          if (in) {
            ckey_s[w] = u;
            cpos_s[w] = (uint16_t)(p0 + e);  // positions < FP4IDX_MAX_CONTEXT = 65536
          }
          kmin = min(kmin, in ? u : 0xFFFFFFFFu);
          kmax = max(kmax, in ? u : 0u);
          w += in;
        }
      }
    } else {  // candidates past kCapB go to the row's workspace region
#pragma unroll
      for (int j = 0; j < kGroups; j++) {
        int w = m + off[j];
        const int p0 = elem_pos(base, j, 0);
#pragma unroll
        for (int e = 0; e < 4; e++) {
          if (flags & (1u << (4 * j + e))) {
            const uint32_t u = order_key(x[4 * j + e]);
            if (w < kCapB) {
              ckey_s[w] = u;
              cpos_s[w] = (uint16_t)(p0 + e);
            } else {
              ckey_g[w] = u;
              cpos_g[w] = (uint16_t)(p0 + e);
            }
            kmin = min(kmin, u);
            kmax = max(kmax, u);
            w++;
          }
        }
      }
    }
    m += total;
  }
  if (m < k) {  // the threshold was too high for this row: exact path over the whole row
    select_whole_row(lg, L, k, o, sh, stage);
    return;
  }

  // ---- 3. selection among the candidates (m >= k)
  for (int b = tid; b < kBins; b += kThreads) sh.hist[b] = 0;
  if (tid == 0) sh.gcount = 0;
  block_minmax(kmin, kmax, sh.uscratch);  // its barriers also publish the candidates
  const float lo1 = key_value(kmin), sc1 = lin_scale(lo1, key_value(kmax));
  auto ck = [&](int i) -> uint32_t { return i < kCapB ? ckey_s[i] : __ldcg(ckey_g + i); };
  auto cpos = [&](int i) -> int { return i < kCapB ? (int)cpos_s[i] : (int)__ldcg(cpos_g + i); };
  for (int i = tid; i < m; i += kThreads) atomicAdd(&sh.hist[lin_bucket(key_value(ck(i)), lo1, sc1)], 1);
  __syncthreads();
  find_bin_from_top(sh.hist, k, sh.scratch, &sh.bin, &sh.rem);
  const int b1 = sh.bin, rem = sh.rem, nb = sh.hist[b1];
  __syncthreads();  // every thread has read nb before the radix path clears the histogram
  auto in_b1 = [&](int i) -> bool { return lin_bucket(key_value(ck(i)), lo1, sc1) == b1; };
  if (nb <= kGather) {
    rank_bucket(m, ck, in_b1, nb, rem, sh);
  } else {
    radix_select(m, ck, in_b1, rem, sh.hist, sh.scratch, &sh.bin, &sh.rem, &sh.key, &sh.take);
  }
  emit_ordered(m, ck, cpos, sh.key, sh.take, o, k, sh.scratch64, stage);
}

inline int64_t cand_stride(int32_t max_context) { return ((int64_t)max(max_context, 1) + 7) / 8 * 8; }
inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

std::atomic<bool> g_attr_done[64];

}  // namespace

// Workspace: per row, a spill region for its candidate keys (u32) and positions (u16).
size_t topk_workspace_bytes(int64_t n_rows, int32_t max_context) {
  const size_t cells = (size_t)n_rows * (size_t)cand_stride(max_context);
  return align256(cells * sizeof(uint32_t)) + align256(cells * sizeof(uint16_t));
}

cudaError_t launch_topk(const float* logits, int64_t stride, const int32_t* context_lens, int32_t n_rows,
                        int32_t max_context, int32_t k, void* workspace, int32_t* out, int32_t* status,
                        cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !g_attr_done[dev].load()) {
    e = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) g_attr_done[dev].store(true);
  }
  const size_t cells = (size_t)n_rows * (size_t)cand_stride(max_context);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  topk_row_kernel<<<(unsigned)n_rows, kThreads, kDynSmem, stream>>>(
      logits, stride, context_lens, max_context, k, reinterpret_cast<uint32_t*>(ws),
      reinterpret_cast<uint16_t*>(ws + align256(cells * sizeof(uint32_t))), cand_stride(max_context), out, status);
  return cudaGetLastError();
}

}  // namespace fp4idx
