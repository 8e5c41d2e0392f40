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
//      taken.  The second pass is skipped when the first one's boundary sub-bin is taken
//      whole (then the selection is every key from that sub-bin up, with no ties), or
//      holds at most kListMax keys (then those keys are ranked directly in the emit);
//   4. one ordered pass emits every key above tau and the lowest-positioned keys equal to
//      it: per thread a bit mask over a contiguous run of positions, one block scan of the
//      mask counts, then the set bits are written out (straight to the output when there
//      are no ties, else through a shared-memory stage).
#include "launchers.cuh"

#include <cooperative_groups.h>

#include <atomic>

namespace cg = cooperative_groups;

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
constexpr int kListMax = 64;  // boundary sub-bin keys of a row ranked directly (all CTAs of a row)


// Order-preserving key; -0 maps to +0 so that equal values are equal keys.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = f == 0.0f ? 0u : __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct Shared {
  uint32_t scratch[kWarps];
  int bin, rem;
  uint32_t tot;  // a cluster CTA's packed emit totals, read by its peers
  int nlist;     // entries in this CTA's list of boundary sub-bin keys, read by its peers
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

// The row's keys.  A CTA holds the keys of its slice of the row: groups v >= v0 with
// 4 * (v - v0) < res in shared memory at topk_dyn + koff, the rest in the row's spill
// region of the workspace (res is a multiple of 4, so a group of four is in one place;
// distinct positions take distinct spill entries whichever CTA writes them).
struct RowKeys {
  uint32_t* spill;
  int res, v0, koff;
  __device__ __forceinline__ uint4 get(int v) const {
    const int i = 4 * (v - v0);
    if (i < res) return *reinterpret_cast<const uint4*>(topk_dyn + koff + i);
    return __ldcg(reinterpret_cast<const uint4*>(spill + (4 * v - res)));
  }
  __device__ __forceinline__ void put(int v, uint4 q) const {
    const int i = 4 * (v - v0);
    if (i < res) *reinterpret_cast<uint4*>(topk_dyn + koff + i) = q;
    else *reinterpret_cast<uint4*>(spill + (4 * v - res)) = q;
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

// One radix pass over this CTA's groups [vs, ve): per digit (key >> shift) &
// (kDigits - 1), the number of keys whose bits from match_shift up equal `match`, into
// hist[0 .. kDigits).  Ends with a barrier.
__device__ __forceinline__ void digit_count(const RowKeys& keys, int L, int vs, int ve, uint32_t match,
                                            int match_shift, int shift, int* hist) {
  const int tid = threadIdx.x;
  for (int b = tid; b < kDigits; b += kThreads) hist[b] = 0;
  __syncthreads();
  for (int v0 = vs; v0 < ve; v0 += kU * kThreads) {
#pragma unroll
    for (int j = 0; j < kU; j++) {
      const int v = v0 + j * kThreads + tid;
      if (v < ve) {
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

// The emit of a row split over a cluster of kC CTAs: this CTA's groups [vs, ve) (at most
// one emit block) in masks as in emit_ordered, one block scan for the offsets inside the
// slice, then the totals of the lower-ranked CTAs (read from their shared memory) for the
// slice's place in the output.  The caller's last cluster barrier keeps every CTA's
// totals readable until its peers have read them.
template <int kC>
__device__ void emit_cluster(const RowKeys& keys, int L, int vs, int ve, uint32_t tau, int take_total, int32_t* o,
                             int k, Shared& sh, int32_t* stage) {
  cg::cluster_group cl = cg::this_cluster();
  const int tid = threadIdx.x;
  const int nbg = ve - vs;  // <= kEmitGroups
  const int run = ((nbg + kThreads - 1) / kThreads) | 1;
  const int g0 = vs + min(nbg, tid * run);
  const int mine = min(run, ve - g0);
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
  uint32_t tot;
  const uint32_t pre = block_excl_scan((uint32_t)gt | ((uint32_t)eq << 16), sh.scratch, tot);
  if (tid == 0) sh.tot = tot;
  cl.sync();
  const int rank = (int)cl.block_rank();
  int Gb = 0, Eb = 0;  // keys above / equal to tau in the lower-ranked CTAs' slices
  for (int q = 0; q < rank; q++) {
    const uint32_t t = *cl.map_shared_rank(&sh.tot, q);
    Gb += (int)(t & 0xFFFFu);
    Eb += (int)(t >> 16);
  }
  const int G = Gb + (int)(pre & 0xFFFFu), E = Eb + (int)(pre >> 16);
  const int take_eq = max(0, min(eq, take_total - E));
  for (int drop = eq - take_eq; drop > 0; drop--) eqm &= ~(1ull << (63 - __clzll(eqm)));
  uint64_t sel = gtm | eqm;
  const int out0 = Gb + min(Eb, take_total);  // this slice's first output
  const int out1 = Gb + (int)(tot & 0xFFFFu) + min(Eb + (int)(tot >> 16), take_total);
  int w = G + min(E, take_total);
  while (sel) {
    const int b = __ffsll(sel) - 1;
    sel &= sel - 1;
    if (w < k) stage[w - out0] = 4 * g0 + b;
    w++;
  }
  __syncthreads();
  for (int i = out0 + tid; i < min(out1, k); i += kThreads) o[i] = stage[i - out0];
  if (rank == kC - 1)  // past the selection (only rows with fewer than k keys in total)
    for (int i = out1 + tid; i < k; i += kThreads) o[i] = -1;
}

// The emit when the boundary sub-bin (keys whose top 22 bits equal hi22) holds at most
// kListMax keys in the row: every key above the sub-bin is taken, and of the sub-bin's keys
// the rem1 largest, equal keys by position.  The sub-bin's keys are collected as (key,
// position) pairs, the CTAs of a pair read each other's, and each key is taken when fewer
// than rem1 of the row's sub-bin keys come before it; this replaces a second radix pass.
// Exactly k keys are taken, so a pair fills the output from both ends as in emit_above.
// `list` holds 2 * kListMax pairs (this CTA's, then the row's) and must not overlap the
// first kDigits counts.  One emit block a CTA.
template <int kC>
__device__ void emit_ranked(const RowKeys& keys, int L, int vs, int ve, uint32_t hi22, int rem1, int32_t* o, int k,
                            Shared& sh, uint32_t* list) {
  static_assert(kC == 1 || kC == 2, "one CTA or a pair per row");
  const int tid = threadIdx.x;
  const int rank = kC > 1 ? (int)(blockIdx.x % kC) : 0;
  const int nbg = ve - vs;  // <= kEmitGroups
  const int run = ((nbg + kThreads - 1) / kThreads) | 1;
  const int g0 = vs + min(nbg, tid * run);
  const int mine = min(run, ve - g0);
  uint64_t sel = 0, mem = 0;
#pragma unroll
  for (int j = 0; j < kRunMax; j++) {
    if (j < mine) {
      const int g = g0 + j;
      const uint4 q = keys.get(g);
      sel |= (uint64_t)group_mask(q, g, L, [&](uint32_t u) { return (u >> kDigitBits) > hi22; }) << (4 * j);
      const uint32_t m = group_mask(q, g, L, [&](uint32_t u) { return (u >> kDigitBits) == hi22; });
      if (m) {  // a few keys in the whole row
        mem |= (uint64_t)m << (4 * j);
        for (int e = 0; e < 4; e++)
          if ((m >> e) & 1u) {
            const int i = atomicAdd(&sh.nlist, 1);
            if (i < kListMax) {
              list[2 * i] = lane_of(q, e);
              list[2 * i + 1] = (uint32_t)(4 * g + e);
            }
          }
      }
    }
  }
  uint32_t* all = list + 2 * kListMax;
  int n_all;
  if constexpr (kC > 1) {
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();  // every CTA's list is complete
    const int n_own = min(sh.nlist, kListMax);
    const int n_peer = min(*cl.map_shared_rank(&sh.nlist, rank ^ 1), kListMax);
    const uint32_t* plist = cl.map_shared_rank(list, rank ^ 1);
    // the row's list in position order of the slices: the lower CTA's pairs first
    const int off_own = rank == 0 ? 0 : n_peer, off_peer = rank == 0 ? n_own : 0;
    if (tid < 2 * n_own) all[2 * off_own + tid] = list[tid];
    if (tid < 2 * n_peer) all[2 * off_peer + tid] = plist[tid];
    n_all = n_own + n_peer;
    __syncthreads();
    // this CTA's reads of its peer's shared memory are done; wait only before leaving
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  } else {
    __syncthreads();
    n_all = min(sh.nlist, kListMax);
    all = list;
  }
  for (uint64_t mm = mem; mm;) {
    const int b = __ffsll(mm) - 1;
    mm &= mm - 1;
    const uint32_t key = lane_of(keys.get(g0 + (b >> 2)), b & 3);
    const uint32_t pos = (uint32_t)(4 * g0 + b);
    int before = 0;
    for (int i = 0; i < n_all; i++) {
      const uint32_t kk = all[2 * i], pp = all[2 * i + 1];
      before += (kk > key || (kk == key && pp < pos)) ? 1 : 0;
    }
    if (before < rem1) sel |= 1ull << b;
  }
  uint32_t tot;
  const uint32_t pre = block_excl_scan((uint32_t)__popcll(sel), sh.scratch, tot);
  int w = (rank == 1 ? k - (int)tot : 0) + (int)pre;
  while (sel) {
    const int b = __ffsll(sel) - 1;
    sel &= sel - 1;
    if (w >= 0 && w < k) o[w] = 4 * g0 + b;
    w++;
  }
  if constexpr (kC > 1) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The emit when the selection is exactly the keys above tau (no ties to resolve): this
// CTA's keys above tau, in position order, written straight to the output.  In a pair
// (kC = 2, one emit block a CTA) the lower CTA fills the output from its start and the
// upper one from its end: a row longer than k has exactly k keys above tau, so the two
// exchange no counts.  One CTA (kC = 1) walks its emit blocks in order.
template <int kC>
__device__ void emit_above(const RowKeys& keys, int L, int vs, int ve, uint32_t tau, int32_t* o, int k,
                           Shared& sh) {
  static_assert(kC == 1 || kC == 2, "one CTA or a pair per row");
  const int tid = threadIdx.x;
  const int rank = kC > 1 ? (int)(blockIdx.x % kC) : 0;
  int done = 0;  // keys above tau in this slice's earlier emit blocks
  for (int b0 = vs; b0 < ve; b0 += kEmitGroups) {
    const int nbg = min(kEmitGroups, ve - b0);
    const int run = ((nbg + kThreads - 1) / kThreads) | 1;  // at most kRunMax
    const int g0 = b0 + min(nbg, tid * run);
    const int mine = min(run, b0 + nbg - g0);
    uint64_t gtm = 0;
#pragma unroll
    for (int j = 0; j < kRunMax; j++) {
      if (j < mine) {
        const int g = g0 + j;
        gtm |= (uint64_t)group_mask(keys.get(g), g, L, [&](uint32_t u) { return u > tau; }) << (4 * j);
      }
    }
    uint32_t tot;
    const uint32_t pre = block_excl_scan((uint32_t)__popcll(gtm), sh.scratch, tot);
    int w = (rank == 1 ? k - (int)tot : done) + (int)pre;
    while (gtm) {
      const int b = __ffsll(gtm) - 1;
      gtm &= gtm - 1;
      if (w >= 0 && w < k) o[w] = 4 * g0 + b;
      w++;
    }
    done += (int)tot;
  }
}

// Sum of the kC CTAs' copies of counts[0 .. n) (n a multiple of 4) into merged[0 .. n).
template <int kC, int n>
__device__ __forceinline__ void merge_counts(int* counts, int* merged) {
  cg::cluster_group cl = cg::this_cluster();
  for (int i = 4 * (int)threadIdx.x; i < n; i += 4 * kThreads) {
    int4 acc = make_int4(0, 0, 0, 0);
#pragma unroll
    for (int q = 0; q < kC; q++) {
      const int4 v = *reinterpret_cast<const int4*>(cl.map_shared_rank(counts + i, q));
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    *reinterpret_cast<int4*>(merged + i) = acc;
  }
  __syncthreads();
}

// kC CTAs (a cluster) per row; each owns a contiguous slice of the row's groups.  Shared
// memory: hist[kHist] (also the output stage), for kC > 1 merged[kHist] and
// dhist[kDigits], then the slice's keys[res] (res a multiple of 4).  spill + row * sstride
// holds keys past res (sstride a multiple of 4).
template <int kC>
__global__ void __launch_bounds__(kThreads, 1)
    topk_row_kernel(const float* __restrict__ logits, int64_t stride, const int32_t* __restrict__ context_lens,
                    int32_t max_context, int32_t k, int32_t res, uint32_t* spill, int64_t sstride,
                    int32_t* __restrict__ out, int32_t* status) {
  __shared__ Shared sh;
  int* const hist = reinterpret_cast<int*>(topk_dyn);
  int* const merged = kC > 1 ? hist + kHist : hist;
  int* const dhist = kC > 1 ? hist + 2 * kHist : hist;
  const int64_t row = blockIdx.x / kC;
  const int rank = (int)(blockIdx.x % kC);
  const int tid = threadIdx.x;
  if (tid == 0) sh.nlist = 0;  // many barriers pass before its first use
  int32_t L = __ldg(context_lens + row);
  if (L < 0 || L > max_context) {
    if (tid == 0 && rank == 0) record_error(status, FP4IDX_ERR_BAD_LENGTH);
    L = L < 0 ? 0 : max_context;
  }
  int32_t* o = out + row * k;
  if (L <= k) {  // the same for every CTA of the row: none of them reaches a cluster barrier
    for (int i = rank * kThreads + tid; i < k; i += kC * kThreads) o[i] = i < L ? i : -1;
    return;
  }
  const float* lg = logits + row * stride;
  const bool vec = (reinterpret_cast<uintptr_t>(lg) & 15) == 0;
  const int ng = (L + 3) >> 2;
  const int per = (ng + kC - 1) / kC;
  const int vs = min(ng, rank * per), ve = min(ng, vs + per);
  const RowKeys keys{spill + row * sstride, res, vs, kC > 1 ? 2 * kHist + kDigits : kHist};

  // ---- 1. keys of the slice and their top-bits histogram; the first loads are issued
  // before the histogram is cleared
  float4 r[kU];
#pragma unroll
  for (int u = 0; u < kU; u++) {
    const int v = vs + u * kThreads + tid;
    if (v < ve) r[u] = load_group(lg, vec, v, L);
  }
  for (int b = tid; b < kHist; b += kThreads) hist[b] = 0;
  __syncthreads();
  for (int v0 = vs; v0 < ve; v0 += kU * kThreads) {
#pragma unroll
    for (int u = 0; u < kU; u++) {
      const int v = v0 + u * kThreads + tid;
      if (v < ve) {
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
    if (vn < ve) {
#pragma unroll
      for (int u = 0; u < kU; u++) {
        const int v = vn + u * kThreads + tid;
        if (v < ve) r[u] = load_group(lg, vec, v, L);
      }
    }
  }
  if constexpr (kC > 1) {
    cg::this_cluster().sync();
    merge_counts<kC, kHist>(hist, merged);  // peers read this CTA's hist until the next cluster barrier
  } else {
    __syncthreads();
  }

  // ---- 2. the bin holding the k-th largest key
  find_bin_from_top<kHist / (32 * kWarps)>(merged, k, sh);
  const uint32_t B = (uint32_t)sh.bin;
  const int rem = sh.rem;

  // ---- 3. two radix passes inside bin B
  digit_count(keys, L, vs, ve, B, kLowBits, kDigitBits, dhist);
  if constexpr (kC > 1) {
    cg::this_cluster().sync();  // also: every peer is done with this CTA's hist
    merge_counts<kC, kDigits>(dhist, merged);
  }
  find_bin_from_top<kDigits / (32 * kWarps)>(merged, rem, sh);
  const uint32_t d1 = (uint32_t)sh.bin;
  const int rem1 = sh.rem;
  const uint32_t hi22 = (B << kDigitBits) | d1;
  const int nd1 = merged[d1];  // keys of the row in the boundary sub-bin
  if (nd1 == rem1 && hi22 != 0u) {
    // Every key of the boundary sub-bin is taken (usually it holds a single key): the
    // selection is every key whose top 22 bits are at least hi22, i.e. every key above
    // the sub-bin's lowest value minus one, with no ties to resolve.  The same counts give
    // every CTA of a pair the same decision.  The pair's last reads of each other's shared
    // memory (the merge above) are done: arrive now, wait only before leaving.
    if constexpr (kC > 1) asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    emit_above<kC>(keys, L, vs, ve, (hi22 << kDigitBits) - 1u, o, k, sh);
    if constexpr (kC > 1) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    return;
  }
  if (nd1 <= kListMax && (kC > 1 || ng <= kEmitGroups)) {
    // a few keys in the boundary sub-bin: rank them directly instead of a second pass (the
    // list sits past the first kDigits counts, which hold the sub-bin counts when kC = 1)
    emit_ranked<kC>(keys, L, vs, ve, hi22, rem1, o, k, sh, reinterpret_cast<uint32_t*>(hist) + kDigits);
    return;
  }
  digit_count(keys, L, vs, ve, hi22, kDigitBits, 0, hist);
  if constexpr (kC > 1) {
    cg::this_cluster().sync();
    merge_counts<kC, kDigits>(hist, merged);
  }
  find_bin_from_top<kDigits / (32 * kWarps)>(merged, rem1, sh);
  const uint32_t tau = (hi22 << kDigitBits) | (uint32_t)sh.bin;
  const int take = sh.rem;

  // ---- 4. ordered emit (the histogram's space becomes the output stage)
  if constexpr (kC > 1) {
    emit_cluster<kC>(keys, L, vs, ve, tau, take, o, k, sh, hist);
    cg::this_cluster().sync();  // no CTA leaves while a peer may still read its shared memory
  } else {
    emit_ordered(keys, L, ng, tau, take, o, k, sh, hist);
  }
}

inline int64_t spill_stride(int32_t max_context) {
  return max((int64_t)0, ((int64_t)max(max_context, 1) + 3) / 4 * 4 - kRes);
}
inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

std::atomic<bool> g_attr_done[2][64];
std::atomic<int> g_sms[64];

// Shared memory of a kC-CTA launch with `res` keys a CTA.
template <int kC>
constexpr size_t smem_bytes(int32_t res) {
  return (kC > 1 ? 2 * kHist + kDigits : kHist) * sizeof(int) + (size_t)res * sizeof(uint32_t);
}

template <int kC>
cudaError_t launch_rows(int dev, const float* logits, int64_t stride, const int32_t* context_lens, int32_t n_rows,
                        int32_t max_context, int32_t k, void* workspace, int32_t* out, int32_t* status,
                        cudaStream_t stream) {
  if (dev < 0 || dev >= 64 || !g_attr_done[kC - 1][dev].load()) {
    const cudaError_t e = cudaFuncSetAttribute(topk_row_kernel<kC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem_bytes<kC>(kRes));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) g_attr_done[kC - 1][dev].store(true);
  }
  // keys a CTA holds: its slice of the longest row, rounded to groups of four
  const int64_t groups = ((int64_t)max(max_context, 1) + 3) / 4;
  const int32_t res = (int32_t)min((int64_t)kRes, 4 * ((groups + kC - 1) / kC));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_rows * kC);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes<kC>(res);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kC > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, topk_row_kernel<kC>, logits, stride, context_lens, max_context, k, res,
                            reinterpret_cast<uint32_t*>(workspace), spill_stride(max_context), out, status);
}

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
  int sms = dev >= 0 && dev < 64 ? g_sms[dev].load() : 0;
  if (sms <= 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) g_sms[dev].store(sms);
  }
  // Few rows leave most SMs idle: then each row goes to a pair of CTAs (a cluster), which
  // halves the passes over its keys.
  if (2 * (int64_t)n_rows <= sms)
    return launch_rows<2>(dev, logits, stride, context_lens, n_rows, max_context, k, workspace, out, status, stream);
  return launch_rows<1>(dev, logits, stride, context_lens, n_rows, max_context, k, workspace, out, status, stream);
}

}  // namespace fp4idx
