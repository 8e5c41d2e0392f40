// The schedule build (schedule.cuh's format) as the body of one block of NT threads, shared
// by the schedule kernel and the step-preparation kernel.
//
// dsv4.1-amd: KV cache layouts, FP4 indexer, compressor and router kernels -- Summary:
// the in-tree decode schedule writes its work list in dispatches whose registers do not
// grow with the row count (the single-kernel schedule it replaced spilled past ~1K rows
// and broke graph capture at 1,536 rows).  [AMD] Enable FP4 indexer for Deepseek V4 --
// Attention runtime: decode schedules are built during graph capture and reused by all
// C4 layers of a forward.
//
// One block walks the rows in chunks of NT with carried block scans (registers fixed, any
// row count), entirely on the device: capturable, no host synchronisation, a pure
// function of its inputs.
#pragma once

#include "fp4idx_internal.cuh"
#include "schedule.cuh"

namespace fp4idx {

// Inclusive block scan (sum or max) of a 64-bit value; every thread gets its prefix and
// the block total.  `scratch` holds kWarps entries.
template <int NT, bool kMax>
__device__ __forceinline__ int64_t sched_block_scan(int64_t v, int64_t* scratch, int64_t& total) {
  constexpr int kWarps = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int64_t n = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v = kMax ? (n > v ? n : v) : v + n;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int64_t w = lane < kWarps ? scratch[lane] : (kMax ? INT64_MIN : 0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int64_t n = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w = kMax ? (n > w ? n : w) : w + n;
    }
    if (lane < kWarps) scratch[lane] = w;
  }
  __syncthreads();
  if (warp > 0) {
    int64_t p = scratch[warp - 1];
    v = kMax ? (p > v ? p : v) : v + p;
  }
  total = scratch[kWarps - 1];
  __syncthreads();
  return v;
}

template <int NT>
__device__ __forceinline__ void build_schedule_block(const int32_t* __restrict__ context_lens,
                                                     const int32_t* __restrict__ row_seq, int32_t n_rows,
                                                     int32_t num_ctas, void* ws) {
  constexpr int kThreads = NT;
  constexpr int kWarps = NT / 32;
  __shared__ int64_t scratch[kWarps];
  // Shared copies for the common case of at most kThreads rows (one chunk): the group
  // starts, the cost prefix and the rows' context lengths, so that phases B and C wait on
  // no global reads.  Larger inputs read the global arrays past the first chunk.
  __shared__ int32_t row0_s[kThreads + 1];
  __shared__ int64_t prefix_s[kThreads + 1];
  __shared__ int32_t len_s[kThreads];
  SchedView s = sched_view(ws, n_rows);
  const int tid = threadIdx.x;
  // the first chunk's context lengths: in flight while phase A scans
  const int32_t len0 = tid < n_rows ? context_lens[tid] : 0;

  // Phase A: group starts.  run_start(t) = last t' <= t where row_seq changes; a group
  // starts where (t - run_start) is a multiple of kGroupMax.
  int64_t carry_run = 0, carry_groups = 0;
  for (int32_t base = 0; base < n_rows; base += kThreads) {
    const int32_t t = base + tid;
    const bool valid = t < n_rows;
    int32_t rs = valid ? row_seq[t] : 0;
    const bool seg = valid && (t == 0 || rs != row_seq[t - 1]);
    int64_t run_tot, tot;
    const int64_t run = sched_block_scan<NT, true>(seg ? (int64_t)t : carry_run, scratch, run_tot);
    const bool gstart = valid && ((t - run) % kGroupMax == 0);
    const int64_t cnt = sched_block_scan<NT, false>(gstart ? 1 : 0, scratch, tot);
    if (gstart) {
      const int64_t gi = carry_groups + cnt - 1;
      s.row0[gi] = t;
      if (gi <= kThreads) row0_s[gi] = t;
    }
    carry_groups += tot;
    carry_run = run_tot;
  }
  const int32_t n_groups = (int32_t)carry_groups;
  if (tid == 0) {
    s.row0[n_groups] = n_rows;
    if (n_groups <= kThreads) row0_s[n_groups] = n_rows;
  }
  len_s[tid] = len0;
  for (int32_t t = tid; t < n_rows; t += kThreads) s.sel_cnt[t] = 0u;
  __syncthreads();

  // Phase B: per-group longest (clamped) context and cost prefix.
  int64_t carry_cost = 0;
  if (tid == 0) s.prefix[0] = prefix_s[0] = 0;
  for (int32_t base = 0; base < n_groups; base += kThreads) {
    const int32_t g = base + tid;
    int64_t cost = 0;
    if (g < n_groups) {
      int32_t r0, r1;
      if (g < kThreads) {
        r0 = row0_s[g];
        r1 = row0_s[g + 1];
      } else {
        r0 = s.row0[g];
        r1 = s.row0[g + 1];
      }
      int32_t mx = 0;
      for (int32_t r = r0; r < r1; r++) {
        int32_t L = r < kThreads ? len_s[r] : context_lens[r];
        L = L < 0 ? 0 : (L > FP4IDX_MAX_CONTEXT ? FP4IDX_MAX_CONTEXT : L);
        mx = L > mx ? L : mx;
      }
      s.maxlen[g] = mx;
      s.seq[g] = row_seq[r0];
      cost = group_cost(mx, r1 - r0);
    }
    int64_t tot;
    int64_t inc = sched_block_scan<NT, false>(cost, scratch, tot);
    if (g < n_groups) {
      s.prefix[g + 1] = carry_cost + inc;
      if (g < kThreads) prefix_s[g + 1] = carry_cost + inc;
    }
    carry_cost += tot;
  }
  __syncthreads();
  // Phase C: each logits CTA's cost range and first work item, so that the kernel starts
  // its page-table reads without walking the schedule.
  // (up to kThreads groups from the shared copies, more from the global arrays)
  const bool small_cost = carry_cost * (int64_t)num_ctas < ((int64_t)1 << 31);
  auto write_start = [&](int32_t c, auto row0_at, auto maxlen_at, auto seq_at, auto prefix_at, const int64_t* pre) {
    CtaStart cs;
    if (small_cost) {  // 32-bit division when every product fits
      cs.lo = (int64_t)((uint32_t)carry_cost * (uint32_t)c / (uint32_t)num_ctas);
      cs.hi = (int64_t)((uint32_t)carry_cost * (uint32_t)(c + 1) / (uint32_t)num_ctas);
    } else {
      cs.lo = carry_cost * c / num_ctas;
      cs.hi = carry_cost * (c + 1) / num_ctas;
    }
    cs.n_groups = n_groups;
    int32_t g = first_group_after(pre, n_groups, cs.lo);
    Item it;
    if (next_item(row0_at, maxlen_at, seq_at, prefix_at, n_groups, cs.lo, cs.hi, g, it)) {
      cs.g = it.g;
      cs.t0 = it.t0;
      cs.t1 = it.t1;
      cs.r0 = it.r0;
      cs.rows = it.rows;
      cs.seq = it.seq;
      cs.maxlen = it.maxlen;
    } else {
      cs.g = n_groups;
      cs.t0 = cs.t1 = cs.r0 = cs.rows = cs.seq = cs.maxlen = 0;
    }
    s.cta[c] = cs;
  };
  if (n_groups <= kThreads) {
    // a group's longest clamped context, recomputed from its rows' lengths as in phase B
    auto maxlen_at = [&](int32_t i) {
      int32_t mx = 0;
      for (int32_t r = row0_s[i]; r < row0_s[i + 1]; r++) {
        int32_t L = r < kThreads ? len_s[r] : context_lens[r];
        L = L < 0 ? 0 : (L > FP4IDX_MAX_CONTEXT ? FP4IDX_MAX_CONTEXT : L);
        mx = L > mx ? L : mx;
      }
      return mx;
    };
    for (int32_t c = tid; c < num_ctas; c += kThreads)
      write_start(c, [&](int32_t i) { return row0_s[i]; }, maxlen_at, [&](int32_t i) { return row_seq[row0_s[i]]; },
                  [&](int32_t i) { return prefix_s[i]; }, prefix_s);
  } else {
    for (int32_t c = tid; c < num_ctas; c += kThreads)
      write_start(c, [&](int32_t i) { return s.row0[i]; }, [&](int32_t i) { return s.maxlen[i]; },
                  [&](int32_t i) { return s.seq[i]; }, [&](int32_t i) { return s.prefix[i]; }, s.prefix);
  }
  if (tid == 0) {
    s.hdr->magic = kSchedMagic;
    s.hdr->n_rows = n_rows;
    s.hdr->num_ctas = num_ctas;
    s.hdr->n_groups = n_groups;
    s.hdr->total_cost = carry_cost;
    s.hdr->group_max = kGroupMax;
    s.hdr->reserved = 0;
  }
}


}  // namespace fp4idx
