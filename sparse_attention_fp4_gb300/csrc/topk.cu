// Per-row top-k of the logits, emitted as ascending compressed-token indices.
//
// [AMD] DeepSeek-V4.1-Flash on MI350X (gfx950) -- Changes: "sorted top-k selection";
// Historical results: the decode top-k is ordered by position, not by KV slot.
// [AMD] Enable FP4 indexer for Deepseek V4 -- Attention runtime: padded rows keep
// context length 0 (their selection is empty: all -1).
//
// Selection = the k largest logits of a row, ties at the k-th value to the lower
// positions, emitted in ascending position order.  One launch, grid (rows, chunks of
// 4,096 tokens):
//   every CTA of a row takes the same fixed sample of 1,024 of the row's logits and
//     derives the same conservative threshold (a linear 256-bucket histogram of the
//     sample, cut about four standard deviations beyond the expected place of the k-th
//     largest), then writes the keys and positions of its chunk's logits at or above it,
//     in order, into the chunk's own region of a candidate buffer;
//   the last CTA of the row to finish (a fence, then an arrival counter; nobody waits)
//     concatenates the regions in order, buckets the candidates linearly between their
//     min and max, ranks the boundary bucket's members exactly and emits the keys above
//     the k-th and the lowest-positioned ones equal to it.
// The threshold is superset-closed (a value that passes lets every larger one pass), so
// with at least k candidates the candidates hold the whole answer.  The sample decides
// speed, never the result: with fewer than k or more than kCapB candidates the last CTA
// runs the exact path over the whole row (2048 linear buckets between the row's min and
// max, a refinement of a crowded bucket over its own range, the bucket ranked exactly,
// radix select when a bucket is all ties).
#include "fp4idx_internal.cuh"

#include <atomic>

namespace fp4idx {
namespace {


constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 4096;                  // tokens per CTA: 8 per thread
constexpr int kPer = kChunk / kThreads;
constexpr int kCapB = 8192;                   // candidates the selecting CTA holds in shared memory
constexpr int kMaxChunks = (FP4IDX_MAX_CONTEXT + kChunk - 1) / kChunk;
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kThreads;
constexpr int kGather = 1024;                 // largest boundary bucket ranked by direct counting
constexpr int kSample = 1024;                 // logits per row behind the candidate threshold
constexpr int kSampleBins = 256;
constexpr size_t kDynSmem = kCapB * (sizeof(uint32_t) + sizeof(uint16_t));
static_assert(kSampleBins <= kThreads && kMaxChunks <= 32 && kSample % kThreads == 0, "layout");
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
  int hist[kBins];
  uint32_t gkey[kGather];
  int gidx[kGather];
  int scratch[kWarps];
  uint32_t uscratch[2 * kWarps];
  int coff[kMaxChunks + 1];
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
__device__ void select_whole_row(const float* lg, int L, int k, int32_t* o, Shared& sh) {
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
  const int got = emit_ordered(L, key_at, [](int s) { return s; }, sh.key, sh.take, o, k, sh.scratch);
  for (int i = got + tid; i < k; i += kThreads) o[i] = -1;  // only rows with non-finite logits
}

// grid (rows, chunks).  Candidate regions: cand_key/cand_pos[row * cstride + chunk * kChunk
// ...], counts cnt[row * nch + chunk], arrival counters arrivals[row] (zero at launch).
__global__ void __launch_bounds__(kThreads, 3) topk_kernel(const float* __restrict__ logits, int64_t stride,
                                                        const int32_t* __restrict__ context_lens, int32_t max_context,
                                                        int32_t k, uint32_t* cand_key, uint16_t* cand_pos,
                                                        int64_t cstride, int32_t* cnt, int32_t nch,
                                                        unsigned int* arrivals, int32_t* __restrict__ out,
                                                        int32_t* status) {
  extern __shared__ __align__(16) uint32_t dyn[];  // ckey[kCapB], then cpos[kCapB] (uint16)
  __shared__ Shared sh;
  const int64_t row = blockIdx.x;
  const int c = blockIdx.y;
  const int tid = threadIdx.x;
  int32_t L = __ldg(context_lens + row);
  if (L < 0 || L > max_context) {
    if (c == 0 && tid == 0) record_error(status, FP4IDX_ERR_BAD_LENGTH);
    L = L < 0 ? 0 : max_context;
  }
  int32_t* o = out + row * k;
  if (L <= k) {
    if (c == 0)
      for (int i = tid; i < k; i += kThreads) o[i] = i < L ? i : -1;
    return;
  }
  const int c0 = c * kChunk;
  if (c0 >= L) return;
  const int nrow = (L + kChunk - 1) / kChunk;  // CTAs of this row that take part
  const float* lg = logits + row * stride;

  // ---- the row's fixed sample and this CTA's tokens.  The sample is 128 runs of 8
  // adjacent logits starting at floor(r * L / 128) rounded down to 8 (two float4 loads a
  // run) when the row is 16-byte aligned and L >= 1024, else single logits at
  // floor(i * L / 1024).
  float sv[kSample / kThreads];
  if ((reinterpret_cast<uintptr_t>(lg) & 15) == 0 && L >= kSample) {
    static_assert(kSample / kThreads == 2 && kSample / 8 <= kThreads, "two sample logits a thread");
    const int run = tid >> 2, part = tid & 3;  // 128 runs x 4 threads; a thread takes 2 logits
    const int p0 = ((int)(((int64_t)run * L) / (kSample / 8)) & ~7) + 2 * part;
    const float2 v = __ldg(reinterpret_cast<const float2*>(lg + p0));
    sv[0] = v.x;
    sv[1] = v.y;
  } else {
#pragma unroll
    for (int j = 0; j < kSample / kThreads; j++)
      sv[j] = __ldg(lg + (int)(((int64_t)(j * kThreads + tid) * L) / kSample));
  }
  float x[kPer];
  const int t0 = c0 + tid * kPer;
  if (((reinterpret_cast<uintptr_t>(lg + t0) & 15) == 0) && t0 + kPer <= L) {
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
    for (int q = 0; q < kPer; q++) x[q] = t0 + q < L ? __ldg(lg + t0 + q) : 0.0f;
  }
  if (tid < kSampleBins) sh.hist[tid] = 0;
  uint32_t smin = 0xFFFFFFFFu, smax = 0u;
#pragma unroll
  for (int j = 0; j < kSample / kThreads; j++) {
    smin = min(smin, order_key(sv[j]));
    smax = max(smax, order_key(sv[j]));
  }
  block_minmax(smin, smax, sh.uscratch);  // its barrier also orders the histogram clear
  const float lo = key_value(smin);
  const float sc = lin_scale(lo, key_value(smax)) * ((float)kSampleBins / (float)kBins);
  auto sbucket = [&](float v) -> int {
    const int b = lin_bucket(v, lo, sc);
    return b >= kSampleBins ? kSampleBins - 1 : b;
  };
#pragma unroll
  for (int j = 0; j < kSample / kThreads; j++) atomicAdd(&sh.hist[sbucket(sv[j])], 1);
  __syncthreads();
  // threshold bucket: keep the sample's expected share of k plus four standard deviations
  const float q = (float)k / (float)L;
  const float mean = q * (float)kSample;
  const int need = min(kSample, (int)ceilf(mean + 4.0f * sqrtf(mean * (1.0f - q)) + 8.0f));
  const int mine = tid < kSampleBins ? sh.hist[kSampleBins - 1 - tid] : 0;
  int tot;
  const int above = block_excl_scan(mine, sh.scratch, tot);
  if (tid < kSampleBins && above < need && need <= above + mine) sh.blo = kSampleBins - 1 - tid;
  __syncthreads();
  const int blo = sh.blo;

  // ---- order-preserving compaction of this chunk's candidates
  unsigned flags = 0;
  int nmine = 0;
#pragma unroll
  for (int qq = 0; qq < kPer; qq++) {
    const bool in = t0 + qq < L && sbucket(x[qq]) >= blo;
    flags |= (unsigned)in << qq;
    nmine += in;
  }
  int total;
  int w = block_excl_scan(nmine, sh.scratch, total);
  const int64_t base = row * cstride + c0;
#pragma unroll
  for (int qq = 0; qq < kPer; qq++) {
    if (flags & (1u << qq)) {
      cand_key[base + w] = order_key(x[qq]);
      cand_pos[base + w] = (uint16_t)(t0 + qq);  // positions < FP4IDX_MAX_CONTEXT = 65536
      w++;
    }
  }
  if (tid == 0) cnt[row * nch + c] = total;
  // publish (block barrier, then one thread's device-scope fence: the release pattern of a
  // grid barrier), then count arrivals: the row's last CTA to arrive selects
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const bool last = atomicAdd(arrivals + row, 1u) == (unsigned)(nrow - 1);
    if (last) __threadfence();
    sh.last = last;
  }
  __syncthreads();
  if (!sh.last) return;

  // ---- selection by the last CTA: concatenate the regions in chunk (= position) order
  uint32_t* ckey = dyn;
  uint16_t* cpos = reinterpret_cast<uint16_t*>(dyn + kCapB);
  if (tid < 32) {
    const int v = tid < nrow ? min(max(__ldcg(cnt + row * nch + tid), 0), kChunk) : 0;
    int xs = v;
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1) {
      const int n = __shfl_up_sync(kFull, xs, o2);
      if (tid >= o2) xs += n;
    }
    if (tid < nrow) sh.coff[tid] = xs - v;
    if (tid == 31) sh.coff[nrow] = xs;
  }
  if (tid == 0) sh.gcount = 0;
  for (int b = tid; b < kBins; b += kThreads) sh.hist[b] = 0;
  __syncthreads();
  const int m = sh.coff[nrow];
  if (m < k || m > kCapB) {
    select_whole_row(lg, L, k, o, sh);
    return;
  }
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  constexpr int kBatch = 8;  // loads a thread keeps in flight at once
#pragma unroll 1
  for (int i0 = 0; i0 < m; i0 += kBatch * kThreads) {
    uint32_t kk[kBatch];
    uint16_t pp[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; u++) {
      const int i = i0 + u * kThreads + tid;
      if (i < m) {
        int lo = 0, hi = nrow;  // chunk of element i: coff[lo] <= i < coff[lo + 1]
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (sh.coff[mid] <= i) lo = mid; else hi = mid;
        }
        const int64_t gi = row * cstride + (int64_t)lo * kChunk + (i - sh.coff[lo]);
        kk[u] = __ldcg(cand_key + gi);
        pp[u] = __ldcg(cand_pos + gi);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; u++) {
      const int i = i0 + u * kThreads + tid;
      if (i < m) {
        ckey[i] = kk[u];
        cpos[i] = pp[u];
        kmin = min(kmin, kk[u]);
        kmax = max(kmax, kk[u]);
      }
    }
  }
  block_minmax(kmin, kmax, sh.uscratch);  // also publishes ckey/cpos
  const float lo1 = key_value(kmin), sc1 = lin_scale(lo1, key_value(kmax));
  for (int i = tid; i < m; i += kThreads) atomicAdd(&sh.hist[lin_bucket(key_value(ckey[i]), lo1, sc1)], 1);
  __syncthreads();
  find_bin_from_top(sh.hist, k, sh.scratch, &sh.bin, &sh.rem);
  const int b1 = sh.bin, rem = sh.rem, nb = sh.hist[b1];
  __syncthreads();  // every thread has read nb before the radix path clears the histogram
  auto ck = [&](int i) -> uint32_t { return ckey[i]; };
  auto in_b1 = [&](int i) -> bool { return lin_bucket(key_value(ckey[i]), lo1, sc1) == b1; };
  if (nb <= kGather) {
    rank_bucket(m, ck, in_b1, nb, rem, sh);
  } else {
    radix_select(m, ck, in_b1, rem, sh.hist, sh.scratch, &sh.bin, &sh.rem, &sh.key, &sh.take);
  }
  const int got = emit_ordered(m, ck, [&](int i) { return (int)cpos[i]; }, sh.key, sh.take, o, k, sh.scratch);
  for (int i = got + tid; i < k; i += kThreads) o[i] = -1;  // only rows with non-finite logits
}

inline int num_chunks(int32_t max_context) { return (max(max_context, 1) + kChunk - 1) / kChunk; }
inline int64_t cand_stride(int32_t max_context) { return ((int64_t)max(max_context, 1) + 7) / 8 * 8; }
inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

// Workspace: [candidate keys u32][candidate positions u16][chunk counts i32][arrivals u32].
struct Layout {
  size_t pos, cnt, arr, total;
};
inline Layout layout(int64_t n_rows, int32_t max_context) {
  const size_t cells = (size_t)n_rows * (size_t)cand_stride(max_context);
  Layout l;
  l.pos = align256(cells * sizeof(uint32_t));
  l.cnt = l.pos + align256(cells * sizeof(uint16_t));
  l.arr = l.cnt + align256((size_t)n_rows * (size_t)num_chunks(max_context) * sizeof(int32_t));
  l.total = l.arr + align256((size_t)n_rows * sizeof(uint32_t));
  return l;
}

__global__ void topk_clear_kernel(unsigned int* arrivals, int32_t n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) arrivals[i] = 0u;
}

std::atomic<bool> g_attr_done[64];

}  // namespace

size_t topk_workspace_bytes(int64_t n_rows, int32_t max_context) { return layout(n_rows, max_context).total; }

uint32_t* topk_arrival_counters(void* workspace, int64_t n_rows, int32_t max_context) {
  return reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(workspace) + layout(n_rows, max_context).arr);
}

cudaError_t launch_topk(const float* logits, int64_t stride, const int32_t* context_lens, int32_t n_rows,
                        int32_t max_context, int32_t k, void* workspace, int32_t* out, int32_t* status,
                        cudaStream_t stream, bool counters_zeroed) {
  if (n_rows == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !g_attr_done[dev].load()) {
    e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmem);
    if (e != cudaSuccess) return e;
    // both kernels keep the SM's largest shared-memory split: no reconfiguration between them
    e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk_clear_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) g_attr_done[dev].store(true);
  }
  const Layout l = layout(n_rows, max_context);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  if (!counters_zeroed)
    topk_clear_kernel<<<(n_rows + 255) / 256, 256, 0, stream>>>(reinterpret_cast<unsigned int*>(ws + l.arr), n_rows);
  const int nch = num_chunks(max_context);
  topk_kernel<<<dim3((unsigned)n_rows, (unsigned)nch), kThreads, kDynSmem, stream>>>(
      logits, stride, context_lens, max_context, k, reinterpret_cast<uint32_t*>(ws),
      reinterpret_cast<uint16_t*>(ws + l.pos), cand_stride(max_context), reinterpret_cast<int32_t*>(ws + l.cnt), nch,
      reinterpret_cast<unsigned int*>(ws + l.arr), out, status);
  return cudaGetLastError();
}

}  // namespace fp4idx
