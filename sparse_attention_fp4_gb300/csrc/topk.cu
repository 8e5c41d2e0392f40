// Per-row top-k of the logits, emitted as ascending compressed-token indices.
//
// [AMD] DeepSeek-V4.1-Flash on MI350X (gfx950) -- Changes: "sorted top-k selection";
// Historical results: the decode top-k is ordered by position, not by KV slot.
// [AMD] Enable FP4 indexer for Deepseek V4 -- Attention runtime: padded rows keep
// context length 0 (their selection is empty: all -1).
//
// Selection = the k largest logits of a row, ties at the k-th value to the lower
// positions, emitted in ascending position order.  One CTA of 1,024 threads per row, no
// communication between CTAs (every hand-off between CTAs -- a global candidate list, a
// fence and an arrival counter -- cost microseconds of latency on this path), and an
// exact plan with no sampling:
//   1. the row is read once with coalesced 16-byte loads and turned into order-preserving
//      uint32 keys.  They stay in shared memory (the first kRes of them; the rest of a
//      longer row goes to the row's region of the caller's workspace), while a 4,096-bin
//      histogram counts their top 12 bits (sign, exponent, three mantissa bits);
//   2. a scan of the histogram from the top finds the bin B that holds the k-th largest
//      key and how many of B's keys the selection still needs;
//   3. two radix passes over the keys, each counting only the keys still in the running
//      (10 + 10 low bits), resolve the k-th key tau and how many keys equal to tau are
//      taken;
//   4. one ordered pass emits every key above tau and the lowest-positioned keys equal to
//      it: per thread a bit mask over a contiguous run of positions, one block scan of the
//      mask counts, then the set bits are written out.
#include "fp4idx_internal.cuh"

#include <atomic>

namespace fp4idx {
namespace {

#ifndef FP4IDX_TOPK_THREADS
#define FP4IDX_TOPK_THREADS 1024
#endif
constexpr int kThreads = FP4IDX_TOPK_THREADS;
constexpr int kWarps = kThreads / 32;
constexpr int kRes = 32768;    // keys a CTA keeps in shared memory
constexpr int kHistBits = 12;  // top bits of the key counted by the first histogram
constexpr int kHist = 1 << kHistBits;
constexpr int kLowBits = 32 - kHistBits;  // bits the radix passes resolve inside bin B
constexpr int kDigitBits = kLowBits / 2;
constexpr int kDigits = 1 << kDigitBits;
constexpr int kU = 8192 / kThreads;   // 16-byte loads in flight per thread (128 KB per CTA)
constexpr int kEmitGroups = 8 * kThreads;  // groups of four positions per emit block
constexpr int kRunMax = ((kEmitGroups + kThreads - 1) / kThreads) | 1;  // groups a thread owns in a block
static_assert(4 * kRunMax <= 64, "a run fits one 64-bit mask");
static_assert(kWarps <= 32 && kHist % (4 * kThreads) == 0 && kDigits % kThreads == 0, "layout");
static_assert(kLowBits == 2 * kDigitBits, "two digit passes");
static_assert(kHist >= FP4IDX_MAX_TOPK, "the histogram doubles as the output stage");
static_assert(4 * kEmitGroups <= 65535, "16-bit block counts in the emit scan");
constexpr unsigned kFull = 0xFFFFFFFFu;

// Dynamic shared memory: hist[kHist] (int; reused as the stage of the k outputs), then
// keys[res].
constexpr size_t kFixedSmem = kHist * sizeof(int);
static_assert(kFixedSmem % 16 == 0, "keys start 16-byte aligned");

// Order-preserving key; -0 maps to +0 so that equal values are equal keys.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = f == 0.0f ? 0u : __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct Shared {
  uint32_t scratch[kWarps];
  int bin, rem;
};

// Exclusive block scan of a uint32 (sums wrap modulo 2^32); `total` gets the block sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* scratch, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  uint32_t w = lane < kWarps ? scratch[lane] : 0u;  // every warp scans the warp sums itself
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(kFull, w, o);
    if (lane >= o) w += n;
  }
  const uint32_t before = __shfl_sync(kFull, w, warp) - scratch[warp] + x - v;
  total = __shfl_sync(kFull, w, kWarps - 1);
  __syncthreads();  // scratch may be reused
  return before;
}

// Over kPerLane * 32 * kWarps bins counted from the top (warp 0, lane 0 own the highest
// bins): the bin that holds the rank-th largest element (1 <= rank <= the total) into
// sh.bin, and rank minus the elements in the bins above it into sh.rem.  Two barriers;
// the last one makes the result visible to the whole CTA.
template <int kPerLane>
__device__ __forceinline__ void find_bin_from_top(const int* counts, int rank, Shared& sh) {
  static_assert(kPerLane == 1 || kPerLane == 2 || kPerLane % 4 == 0, "bins a lane");
  constexpr int kPerWarp = kPerLane * 32;
  constexpr int kBins = kPerWarp * kWarps;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lo = kBins - warp * kPerWarp - (lane + 1) * kPerLane;  // this lane's lowest bin
  int c[kPerLane];
  if constexpr (kPerLane % 4 == 0) {
#pragma unroll
    for (int j = 0; j < kPerLane; j += 4) {
      const int4 v = *reinterpret_cast<const int4*>(counts + lo + j);
      c[j] = v.x;
      c[j + 1] = v.y;
      c[j + 2] = v.z;
      c[j + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kPerLane; j++) c[j] = counts[lo + j];
  }
  int s = 0;
#pragma unroll
  for (int j = 0; j < kPerLane; j++) s += c[j];
  int x = s;  // inclusive scan from the top lane down
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) sh.scratch[warp] = (uint32_t)x;
  __syncthreads();
  const int ws = lane < kWarps ? (int)sh.scratch[lane] : 0;
  int wx = ws;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(kFull, wx, o);
    if (lane >= o) wx += n;
  }
  const unsigned hit = __ballot_sync(kFull, wx - ws < rank && rank <= wx);
  const int W = __ffs(hit) - 1;  // the warp whose bins hold the rank-th element
  if (warp == W) {
    const int above = __shfl_sync(kFull, wx - ws, W) + x - s;
    if (above < rank && rank <= above + s) {
      int acc = above;
#pragma unroll
      for (int j = kPerLane - 1; j >= 0; j--) {
        if (acc < rank && rank <= acc + c[j]) {
          sh.bin = lo + j;
          sh.rem = rank - acc;
        }
        acc += c[j];
      }
    }
  }
  __syncthreads();
}

// This thread's group v of four logits (positions 4v .. 4v+3); past L reads nothing.
__device__ __forceinline__ float4 load_group(const float* lg, bool vec, int v, int L) {
  const int i = 4 * v;
  if (vec && i + 4 <= L) return __ldg(reinterpret_cast<const float4*>(lg) + v);
  float4 r;
  r.x = i < L ? __ldg(lg + i) : 0.0f;
  r.y = i + 1 < L ? __ldg(lg + i + 1) : 0.0f;
  r.z = i + 2 < L ? __ldg(lg + i + 2) : 0.0f;
  r.w = i + 3 < L ? __ldg(lg + i + 3) : 0.0f;
  return r;
}

// Dynamic shared memory of the top-k kernel (declared here so that helpers address it as
// shared memory).
extern __shared__ __align__(16) uint32_t topk_dyn[];

// The row's keys: positions below res in shared memory (after the histogram), the rest in
// the row's spill region of the workspace (res is a multiple of 4, so a group of four is
// in one place).
struct RowKeys {
  uint32_t* spill;
  int res;
  __device__ __forceinline__ uint4 get(int v) const {
    const int i = 4 * v;
    if (i < res) return reinterpret_cast<const uint4*>(topk_dyn + kHist)[v];
    return __ldcg(reinterpret_cast<const uint4*>(spill + (i - res)));
  }
  __device__ __forceinline__ void put(int v, uint4 q) const {
    const int i = 4 * v;
    if (i < res) reinterpret_cast<uint4*>(topk_dyn + kHist)[v] = q;
    else *reinterpret_cast<uint4*>(spill + (i - res)) = q;
  }
};

// Nibble of the four keys of a group that satisfy pred (bit e = key e); keys at positions
// 4v + e >= L (only in the row's last group) are left out.
template <class Pred>
__device__ __forceinline__ uint32_t group_mask(const uint4& q, int v, int L, Pred pred) {
  uint32_t m = (uint32_t)pred(q.x) | ((uint32_t)pred(q.y) << 1) | ((uint32_t)pred(q.z) << 2) |
               ((uint32_t)pred(q.w) << 3);
  const int lim = L - 4 * v;  // >= 1 for every group of the row
  if (lim < 4) m &= (1u << lim) - 1u;
  return m;
}

__device__ __forceinline__ uint32_t lane_of(const uint4& q, int e) {
  return e == 0 ? q.x : (e == 1 ? q.y : (e == 2 ? q.z : q.w));
}

// One radix pass: per digit (key >> shift) & (kDigits - 1), the number of the row's keys
// whose bits from match_shift up equal `match`.  Ends with the digit picked for `rank`.
__device__ __forceinline__ void digit_pass(const RowKeys& keys, int L, int ng, uint32_t match, int match_shift,
                                           int shift, int rank, int* hist, Shared& sh) {
  const int tid = threadIdx.x;
  for (int b = tid; b < kDigits; b += kThreads) hist[b] = 0;
  __syncthreads();
  for (int v0 = 0; v0 < ng; v0 += kU * kThreads) {
#pragma unroll
    for (int j = 0; j < kU; j++) {
      const int v = v0 + j * kThreads + tid;
      if (v < ng) {
        const uint4 q = keys.get(v);
        const uint32_t m = group_mask(q, v, L, [&](uint32_t u) { return (u >> match_shift) == match; });
        if (m) {  // members are a few percent of the row
#pragma unroll
          for (int e = 0; e < 4; e++)
            if ((m >> e) & 1u) atomicAdd(&hist[(lane_of(q, e) >> shift) & (kDigits - 1)], 1);
        }
      }
    }
  }
  __syncthreads();
  find_bin_from_top<kDigits / (32 * kWarps)>(hist, rank, sh);
}

// Writes o[0..k): every position i < L whose key is above tau and the first take_total
// (by position) whose key equals tau, ascending, then -1.  Positions go in blocks of
// kEmitGroups groups of four; in a block each thread owns a contiguous run of groups (an
// odd number of them, so that the 16-byte shared-memory reads of a quarter warp hit
// distinct banks) and marks its keys above tau and equal to tau in two bit masks.  One
// block scan of the packed mask counts gives the output offsets.  The positions are
// staged in `stage` (k ints) and copied out coalesced.
__device__ void emit_ordered(const RowKeys& keys, int L, int ng, uint32_t tau, int take_total, int32_t* o, int k,
                             Shared& sh, int32_t* stage) {
  const int tid = threadIdx.x;
  int g_done = 0, e_done = 0;  // keys above / equal to tau in earlier blocks
  for (int b0 = 0; b0 < ng; b0 += kEmitGroups) {
    const int nbg = min(kEmitGroups, ng - b0);
    const int run = ((nbg + kThreads - 1) / kThreads) | 1;  // at most kRunMax
    const int g0 = b0 + min(nbg, tid * run);
    const int mine = min(run, b0 + nbg - g0);
    uint64_t gtm = 0, eqm = 0;
#pragma unroll
    for (int j = 0; j < kRunMax; j++) {
      if (j < mine) {
        const int g = g0 + j;
        const uint4 q = keys.get(g);
        gtm |= (uint64_t)group_mask(q, g, L, [&](uint32_t u) { return u > tau; }) << (4 * j);
        eqm |= (uint64_t)group_mask(q, g, L, [&](uint32_t u) { return u == tau; }) << (4 * j);
      }
    }
    const int gt = __popcll(gtm), eq = __popcll(eqm);
    uint32_t tot;  // gt in the low 16 bits, eq in the high 16 (a block has at most 32,768 keys)
    const uint32_t pre = block_excl_scan((uint32_t)gt | ((uint32_t)eq << 16), sh.scratch, tot);
    const int G = g_done + (int)(pre & 0xFFFFu), E = e_done + (int)(pre >> 16);
    // the keys equal to tau are taken greedily in position order: keep this run's first
    // take_eq of them
    const int take_eq = max(0, min(eq, take_total - E));
    for (int drop = eq - take_eq; drop > 0; drop--) eqm &= ~(1ull << (63 - __clzll(eqm)));
    uint64_t sel = gtm | eqm;
    int w = G + min(E, take_total);
    while (sel) {
      const int b = __ffsll(sel) - 1;
      sel &= sel - 1;
      if (w < k) stage[w] = 4 * g0 + b;
      w++;
    }
    g_done += (int)(tot & 0xFFFFu);
    e_done += (int)(tot >> 16);
  }
  __syncthreads();
  const int got = min(g_done + min(e_done, take_total), k);  // equal to k whenever L > k
  for (int i = tid; i < k; i += kThreads) o[i] = i < got ? stage[i] : -1;
}

// One CTA per row.  keys[0..res) of the row stay in shared memory (res a multiple of 4);
// spill + row * sstride holds the keys of positions res and up (sstride a multiple of 4).
__global__ void __launch_bounds__(kThreads, 1)
    topk_row_kernel(const float* __restrict__ logits, int64_t stride, const int32_t* __restrict__ context_lens,
                    int32_t max_context, int32_t k, int32_t res, uint32_t* spill, int64_t sstride,
                    int32_t* __restrict__ out, int32_t* status) {
  __shared__ Shared sh;
  int* const hist = reinterpret_cast<int*>(topk_dyn);
  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x;
  // launched as a programmatic dependent of the kernel before it on the stream (the
  // logits): wait until that grid has completed and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
  const bool vec = (reinterpret_cast<uintptr_t>(lg) & 15) == 0;
  const int ng = (L + 3) >> 2;
  const RowKeys keys{spill + row * sstride, res};

  // ---- 1. keys and the top-bits histogram; the first loads are issued before the
  // histogram is cleared
  float4 r[kU];
#pragma unroll
  for (int u = 0; u < kU; u++) {
    const int v = u * kThreads + tid;
    if (v < ng) r[u] = load_group(lg, vec, v, L);
  }
  for (int b = tid; b < kHist; b += kThreads) hist[b] = 0;
  __syncthreads();
  for (int v0 = 0; v0 < ng; v0 += kU * kThreads) {
#pragma unroll
    for (int u = 0; u < kU; u++) {
      const int v = v0 + u * kThreads + tid;
      if (v < ng) {
        const uint4 q = make_uint4(order_key(r[u].x), order_key(r[u].y), order_key(r[u].z), order_key(r[u].w));
        keys.put(v, q);
        const int i = 4 * v;
        atomicAdd(&hist[q.x >> kLowBits], 1);
        if (i + 1 < L) atomicAdd(&hist[q.y >> kLowBits], 1);
        if (i + 2 < L) atomicAdd(&hist[q.z >> kLowBits], 1);
        if (i + 3 < L) atomicAdd(&hist[q.w >> kLowBits], 1);
      }
    }
    const int vn = v0 + kU * kThreads;
    if (vn < ng) {
#pragma unroll
      for (int u = 0; u < kU; u++) {
        const int v = vn + u * kThreads + tid;
        if (v < ng) r[u] = load_group(lg, vec, v, L);
      }
    }
  }
  __syncthreads();

  // ---- 2. the bin holding the k-th largest key
  find_bin_from_top<kHist / (32 * kWarps)>(hist, k, sh);
  const uint32_t B = (uint32_t)sh.bin;
  const int rem = sh.rem;

  // ---- 3. two radix passes inside bin B
  digit_pass(keys, L, ng, B, kLowBits, kDigitBits, rem, hist, sh);
  const uint32_t d1 = (uint32_t)sh.bin;
  const int rem1 = sh.rem;
  const uint32_t hi22 = (B << kDigitBits) | d1;
  digit_pass(keys, L, ng, hi22, kDigitBits, 0, rem1, hist, sh);
  const uint32_t tau = (hi22 << kDigitBits) | (uint32_t)sh.bin;
  const int take = sh.rem;

  // ---- 4. ordered emit (the histogram's space becomes the output stage)
  emit_ordered(keys, L, ng, tau, take, o, k, sh, hist);
}

inline int64_t spill_stride(int32_t max_context) {
  return max((int64_t)0, ((int64_t)max(max_context, 1) + 3) / 4 * 4 - kRes);
}
inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

std::atomic<bool> g_attr_done[64];

}  // namespace

// Workspace: per row, the keys of positions past the kRes a CTA keeps in shared memory
// (none when max_context <= kRes; the size is still at least 256 bytes).  Nothing in it
// needs to be initialised.
size_t topk_workspace_bytes(int64_t n_rows, int32_t max_context) {
  return align256(max((size_t)1, (size_t)n_rows * (size_t)spill_stride(max_context) * sizeof(uint32_t)));
}

cudaError_t launch_topk(const float* logits, int64_t stride, const int32_t* context_lens, int32_t n_rows,
                        int32_t max_context, int32_t k, void* workspace, int32_t* out, int32_t* status,
                        cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !g_attr_done[dev].load()) {
    e = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kFixedSmem + kRes * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) g_attr_done[dev].store(true);
  }
  const int32_t res = (int32_t)min((int64_t)kRes, ((int64_t)max(max_context, 1) + 3) / 4 * 4);
  const size_t smem = kFixedSmem + (size_t)res * sizeof(uint32_t);
  // A programmatic dependent launch: the CTAs may become resident while the previous
  // kernel on the stream is still running (as its CTAs exit), and wait in the kernel for
  // its completion.  Without a trigger in the previous kernel this is an ordinary
  // stream-ordered launch.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_rows);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_row_kernel, logits, stride, context_lens, max_context, k, res,
                            reinterpret_cast<uint32_t*>(workspace), spill_stride(max_context), out, status);
}

}  // namespace fp4idx
