// Per-row top-k of the logits, emitted as ascending compressed-token indices.
//
// [AMD] DeepSeek-V4.1-Flash on MI350X (gfx950) -- Changes: "sorted top-k selection";
// Historical results: the decode top-k is ordered by position, not by KV slot.
// [AMD] Enable FP4 indexer for Deepseek V4 -- Attention runtime: padded rows keep
// context length 0 (their selection is empty: all -1).
//
// One thread-block cluster per query row (1, 2, 4 or 8 CTAs: wide clusters when there are
// few rows, so a decode batch still fills the GPU).  CTA `rank` owns a contiguous segment
// of the row and caches it in shared memory as order-preserving 32-bit keys; the cluster
// combines its statistics in the shared memory of rank 0 (distributed shared memory).
// Selection = the k largest logits, ties at the k-th value to the lower positions:
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
//      keys equal to it: each thread owns a contiguous run of positions and block and
//      cluster scans give the output offsets, so the selection comes out sorted.
#include <cooperative_groups.h>

#include "fp4idx_internal.cuh"

namespace cg = cooperative_groups;

namespace fp4idx {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kThreads;
constexpr int kGather = 1024;
constexpr int kMaxCluster = 8;
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

// Cluster-wide state; the copy in rank 0's shared memory is the one the cluster uses.
struct ClusterState {
  uint32_t kmin, kmax, kmin2, kmax2;
  int bin, rem;
  int nbk;     // elements in the bucket just selected
  int gcount;  // gathered candidates
  uint32_t key;
  int take;
  int gt[kMaxCluster], eq[kMaxCluster];
};

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(const float* __restrict__ logits, int64_t stride,
                                                        const int32_t* __restrict__ context_lens, int32_t max_context,
                                                        int32_t k, int32_t* __restrict__ out, int32_t seg_cap,
                                                        int32_t* status) {
  extern __shared__ __align__(16) uint32_t keys[];
  __shared__ int hist[kBins];
  __shared__ uint32_t gkey[kGather];
  __shared__ int gidx[kGather];
  __shared__ int scratch[kWarps];
  __shared__ uint32_t uscratch[kWarps];
  __shared__ ClusterState cst;

  cg::cluster_group cluster = cg::this_cluster();
  const int cs = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t row = blockIdx.x / cs;
  const int tid = threadIdx.x;
  ClusterState* c0 = cluster.map_shared_rank(&cst, 0);
  int* hist0 = cluster.map_shared_rank(hist, 0);
  uint32_t* gkey0 = cluster.map_shared_rank(gkey, 0);
  int* gidx0 = cluster.map_shared_rank(gidx, 0);

  int32_t L = __ldg(context_lens + row);
  if (L < 0 || L > max_context) {
    if (tid == 0 && rank == 0) record_error(status, FP4IDX_ERR_BAD_LENGTH);
    L = L < 0 ? 0 : max_context;
  }
  int32_t* o = out + row * k;
  if (L <= k) {  // the same for every CTA of the cluster; no distributed memory touched
    for (int i = rank * kThreads + tid; i < k; i += cs * kThreads) o[i] = i < L ? i : -1;
    return;
  }
  int chunk = (L + cs - 1) / cs;
  chunk = (chunk + 3) & ~3;
  const int seg0 = min(L, rank * chunk), n = min(L, seg0 + chunk) - seg0;
  const bool cached = chunk <= seg_cap;
  const float* lg = logits + row * stride + seg0;
  if (rank == 0 && tid == 0) {
    cst.kmin = 0xFFFFFFFFu;
    cst.kmax = 0u;
    cst.kmin2 = 0xFFFFFFFFu;
    cst.kmax2 = 0u;
    cst.gcount = 0;
  }
  for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;

  // load the segment (four 16-byte loads in flight per thread), keys and local min/max
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  auto take = [&](int s, float x) {
    const uint32_t u = order_key(x);
    kmin = min(kmin, u);
    kmax = max(kmax, u);
    if (cached) keys[s] = u;
  };
  int s_done = 0;
  if ((reinterpret_cast<uintptr_t>(lg) & 15) == 0) {
    const float4* lg4 = reinterpret_cast<const float4*>(lg);
    const int n4 = n >> 2;
    for (int v0 = 0; v0 < n4; v0 += 4 * kThreads) {
      float4 x[4];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int v = v0 + u * kThreads + tid;
        x[u] = v < n4 ? __ldg(lg4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int v = v0 + u * kThreads + tid;
        if (v < n4) {
          take(4 * v, x[u].x);
          take(4 * v + 1, x[u].y);
          take(4 * v + 2, x[u].z);
          take(4 * v + 3, x[u].w);
        }
      }
    }
    s_done = n4 << 2;
  }
  for (int b0 = s_done; b0 < n; b0 += 4 * kThreads) {
    float x[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int s = b0 + u * kThreads + tid;
      x[u] = s < n ? __ldg(lg + s) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int s = b0 + u * kThreads + tid;
      if (s < n) take(s, x[u]);
    }
  }
  kmin = block_reduce<false>(kmin, uscratch);
  kmax = block_reduce<true>(kmax, uscratch);
  cluster.sync();  // rank 0's state initialised, every histogram zeroed
  if (tid == 0) {
    atomicMin(&c0->kmin, kmin);
    atomicMax(&c0->kmax, kmax);
  }
  cluster.sync();
  auto key_at = [&](int s) -> uint32_t { return cached ? keys[s] : order_key(__ldg(lg + s)); };

  // 1. bucket histogram over [min, max], merged into rank 0
  const float lo1 = key_value(c0->kmin), sc1 = lin_scale(lo1, key_value(c0->kmax));
  for (int s = tid; s < n; s += kThreads) atomicAdd(&hist[lin_bucket(key_value(key_at(s)), lo1, sc1)], 1);
  __syncthreads();
  if (rank != 0)
    for (int b = tid; b < kBins; b += kThreads) {
      const int c = hist[b];
      if (c) atomicAdd(hist0 + b, c);
    }
  cluster.sync();
  if (rank == 0) {
    find_bin_from_top(hist, k, scratch, &cst.bin, &cst.rem);
    if (tid == 0) cst.nbk = hist[cst.bin];
  }
  cluster.sync();
  const int b1 = c0->bin;
  int rem = c0->rem;
  int nb = c0->nbk;

  // optional refinement of a crowded bucket over its own value range
  float lo2 = 0.0f, sc2 = 0.0f;
  int b2 = -1;
  if (nb > kGather) {
    uint32_t bmin = 0xFFFFFFFFu, bmax = 0u;
    for (int s = tid; s < n; s += kThreads) {
      const uint32_t u = key_at(s);
      if (lin_bucket(key_value(u), lo1, sc1) == b1) {
        bmin = min(bmin, u);
        bmax = max(bmax, u);
      }
    }
    bmin = block_reduce<false>(bmin, uscratch);
    bmax = block_reduce<true>(bmax, uscratch);
    if (tid == 0) {
      atomicMin(&c0->kmin2, bmin);
      atomicMax(&c0->kmax2, bmax);
    }
    for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
    cluster.sync();
    lo2 = key_value(c0->kmin2);
    sc2 = lin_scale(lo2, key_value(c0->kmax2));
    for (int s = tid; s < n; s += kThreads) {
      const float x = key_value(key_at(s));
      if (lin_bucket(x, lo1, sc1) == b1) atomicAdd(&hist[lin_bucket(x, lo2, sc2)], 1);
    }
    __syncthreads();
    if (rank != 0)
      for (int b = tid; b < kBins; b += kThreads) {
        const int c = hist[b];
        if (c) atomicAdd(hist0 + b, c);
      }
    cluster.sync();
    if (rank == 0) {
      find_bin_from_top(hist, rem, scratch, &cst.bin, &cst.rem);
      if (tid == 0) cst.nbk = hist[cst.bin];
    }
    cluster.sync();
    b2 = c0->bin;
    rem = c0->rem;
    nb = c0->nbk;
  }
  auto in_bucket = [&](uint32_t u) -> bool {
    const float x = key_value(u);
    return lin_bucket(x, lo1, sc1) == b1 && (b2 < 0 || lin_bucket(x, lo2, sc2) == b2);
  };

  // 2. resolve the bucket: threshold key tau and how many keys equal to tau to keep
  if (nb <= kGather) {
    for (int s = tid; s < n; s += kThreads) {
      const uint32_t u = key_at(s);
      if (in_bucket(u)) {
        const int slot = atomicAdd(&c0->gcount, 1);
        gkey0[slot] = u;
        gidx0[slot] = seg0 + s;
      }
    }
    cluster.sync();
    if (rank == 0) {
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
          cst.key = ki;
          cst.take = rem - gt;
        }
      }
    }
    cluster.sync();
  } else {
    // crowded bucket (many equal values): exact radix select over its keys (11 + 11 + 10 bits)
    uint32_t prefix = 0, pmask = 0;
    int r = rem;
#pragma unroll 1
    for (int pass = 0; pass < 3; pass++) {
      const int dshift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
      for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
      cluster.sync();
      for (int s_base = 0; s_base < n; s_base += kThreads) {
        const int s = s_base + tid;
        bool in = false;
        uint32_t digit = 0;
        if (s < n) {
          const uint32_t u = key_at(s);
          in = in_bucket(u) && (u & pmask) == prefix;
          digit = (u >> dshift) & dmask;
        }
        const unsigned active = __ballot_sync(kFull, in);
        if (in) {
          const unsigned peers = __match_any_sync(active, digit);
          if ((__ffs(peers) - 1) == (tid & 31)) atomicAdd(&hist[digit], __popc(peers));
        }
      }
      __syncthreads();
      if (rank != 0)
        for (int b = tid; b < kBins; b += kThreads) {
          const int c = hist[b];
          if (c) atomicAdd(hist0 + b, c);
        }
      cluster.sync();
      if (rank == 0) find_bin_from_top(hist, r, scratch, &cst.bin, &cst.rem);
      cluster.sync();
      prefix |= (uint32_t)c0->bin << dshift;
      pmask |= dmask << dshift;
      r = c0->rem;
    }
    if (rank == 0 && tid == 0) {
      cst.key = prefix;
      cst.take = r;
    }
    cluster.sync();
  }
  const uint32_t tau = c0->key;
  const int take_total = c0->take;

  // 3. ordered output: per-thread contiguous runs inside this CTA's segment
  const int tchunk = ((n + kThreads - 1) / kThreads) | 1;  // odd stride: conflict-free reads
  const int s0 = min(n, tid * tchunk), s1 = min(n, s0 + tchunk);
  int gt = 0, eq = 0;
  for (int s = s0; s < s1; s++) {
    const uint32_t u = key_at(s);
    gt += u > tau;
    eq += u == tau;
  }
  int tot_gt, tot_eq;
  (void)block_excl_scan(gt, scratch, tot_gt);
  const int eq_local = block_excl_scan(eq, scratch, tot_eq);
  if (tid == 0) {
    c0->gt[rank] = tot_gt;
    c0->eq[rank] = tot_eq;
  }
  cluster.sync();
  int eq_before_cta = 0, sel_before_cta = 0;
  for (int c = 0; c < rank; c++) {
    const int e = c0->eq[c];
    sel_before_cta += c0->gt[c] + max(0, min(e, take_total - eq_before_cta));
    eq_before_cta += e;
  }
  const int take_eq = max(0, min(eq, take_total - eq_before_cta - eq_local));
  int tot_sel;
  const int pos = sel_before_cta + block_excl_scan(gt + take_eq, scratch, tot_sel);
  int w = pos, te = 0;
  for (int s = s0; s < s1 && w < k; s++) {
    const uint32_t u = key_at(s);
    if (u > tau || (u == tau && te++ < take_eq)) o[w++] = seg0 + s;
  }
  if (rank == cs - 1)  // only for rows with non-finite logits can the selection fall short of k
    for (int i = sel_before_cta + tot_sel + tid; i < k; i += kThreads) o[i] = -1;
  cluster.sync();  // rank 0's shared memory is read until here
}

}  // namespace

int32_t topk_smem_cap() { return 49152; }

int topk_cluster_size(int32_t n_rows) {
  return n_rows <= 19 ? 8 : (n_rows <= 76 ? 4 : (n_rows <= 152 ? 2 : 1));
}

cudaError_t launch_topk(const float* logits, int64_t stride, const int32_t* context_lens, int32_t n_rows,
                        int32_t max_context, int32_t k, int32_t* out, int32_t* status, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(topk_smem_cap() * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int cs = topk_cluster_size(n_rows);
  const int chunk = (((max_context + cs - 1) / cs) + 3) & ~3;
  const int32_t seg_cap = min(chunk, topk_smem_cap());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_rows * cs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)(seg_cap > 0 ? seg_cap : 1) * sizeof(uint32_t);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel, logits, stride, context_lens, max_context, k, out, seg_cap, status);
}

}  // namespace fp4idx
