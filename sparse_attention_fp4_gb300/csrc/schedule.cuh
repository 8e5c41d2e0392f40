// Schedule format shared by the schedule builder and the logits kernel.
//
// Query rows are cut into groups: maximal runs of consecutive rows with the same
// row_seq, split every kGroupMax rows.  A group's rows share every K tile (all draft
// rows of a sequence, or a block of prefill rows), so one tile load serves them all.
// Group g covers tiles [0, ntiles) of 128 tokens, ntiles = ceil(max context / 128), and
// costs ntiles * (kTileCost + rows) units: one unit per row for the epilogue plus a
// fixed charge for streaming the tile.  The logits grid splits the total cost into
// num_ctas equal ranges; CTA c takes every tile whose cost interval starts in its range.
// The split decides only which CTA computes a logit, never its value.
#pragma once

#include <stdint.h>

namespace fp4idx {

constexpr int kGroupMax = 6;  // six draft rows of a sequence share one group
constexpr int kTileTokens = 128;
constexpr int kTileCost = 2;
constexpr int32_t kSchedMagic = 0x46344944;  // "F4ID"

struct SchedHeader {
  int32_t magic;
  int32_t n_rows;
  int32_t num_ctas;
  int32_t n_groups;
  int64_t total_cost;
  int32_t group_max;
  int32_t reserved;
};

struct SchedView {
  SchedHeader* hdr;
  int32_t* row0;     // [n_rows + 1] first row of each group (entry n_groups = n_rows)
  int32_t* maxlen;   // [n_rows] largest clamped context length in the group
  int32_t* seq;      // [n_rows] the group's sequence (row_seq of its rows), so that a work
                     // item's first page-table read need not wait on a row_seq load
  int64_t* prefix;   // [n_rows + 1] exclusive prefix of group costs
  int32_t* cta_g0;   // [num_ctas] first group whose cost interval ends after the CTA's range start
};

__host__ __device__ inline size_t sched_align16(size_t x) { return (x + 15) & ~(size_t)15; }

__host__ __device__ inline size_t sched_bytes(int64_t n_rows, int64_t num_ctas) {
  size_t b = sched_align16(sizeof(SchedHeader));
  b += sched_align16(sizeof(int32_t) * (size_t)(n_rows + 1));
  b += sched_align16(sizeof(int32_t) * (size_t)(n_rows + 1));
  b += sched_align16(sizeof(int32_t) * (size_t)(n_rows + 1));
  b += sched_align16(sizeof(int64_t) * (size_t)(n_rows + 1));
  b += sched_align16(sizeof(int32_t) * (size_t)num_ctas);
  return b;
}

__host__ __device__ inline SchedView sched_view(void* base, int64_t n_rows) {
  uint8_t* p = reinterpret_cast<uint8_t*>(base);
  SchedView v;
  v.hdr = reinterpret_cast<SchedHeader*>(p);
  p += sched_align16(sizeof(SchedHeader));
  v.row0 = reinterpret_cast<int32_t*>(p);
  p += sched_align16(sizeof(int32_t) * (size_t)(n_rows + 1));
  v.maxlen = reinterpret_cast<int32_t*>(p);
  p += sched_align16(sizeof(int32_t) * (size_t)(n_rows + 1));
  v.seq = reinterpret_cast<int32_t*>(p);
  p += sched_align16(sizeof(int32_t) * (size_t)(n_rows + 1));
  v.prefix = reinterpret_cast<int64_t*>(p);
  p += sched_align16(sizeof(int64_t) * (size_t)(n_rows + 1));
  v.cta_g0 = reinterpret_cast<int32_t*>(p);
  return v;
}

__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// First group whose cost interval [prefix[g], prefix[g+1]) ends after `lo`.
__host__ __device__ inline int32_t first_group_after(const int64_t* prefix, int32_t n_groups, int64_t lo) {
  int32_t a = 0, b = n_groups;
  while (a < b) {
    const int32_t m = (a + b) >> 1;
    if (prefix[m + 1] <= lo) a = m + 1;
    else b = m;
  }
  return a;
}

// Iterates the (group, tile range) items of one CTA in a fixed order.
struct ItemIter {
  const int32_t* row0;
  const int32_t* maxlen;
  const int64_t* prefix;
  int32_t n_groups;
  int64_t lo, hi;
  int32_t g;

  __device__ void init(const SchedView& s, int cta, int num_ctas) {
    row0 = s.row0;
    maxlen = s.maxlen;
    prefix = s.prefix;
    n_groups = s.hdr->n_groups;
    const int64_t W = s.hdr->total_cost;
    lo = W * cta / num_ctas;
    hi = W * (cta + 1) / num_ctas;
    g = s.cta_g0[cta];  // precomputed by the schedule kernel
  }

  // Next non-empty item; false when this CTA's range is exhausted.
  __device__ bool next(int32_t& grp, int32_t& t0, int32_t& t1) {
    while (g < n_groups && prefix[g] < hi) {
      const int32_t gg = g++;
      const int32_t rows = row0[gg + 1] - row0[gg];
      const int64_t u = kTileCost + rows;
      const int64_t ntiles = ceil_div64(maxlen[gg], kTileTokens);
      const int64_t base = prefix[gg];
      int64_t i0 = lo > base ? ceil_div64(lo - base, u) : 0;
      int64_t i1 = hi > base ? ceil_div64(hi - base, u) : 0;
      if (i1 > ntiles) i1 = ntiles;
      if (i0 < i1) {
        grp = gg;
        t0 = (int32_t)i0;
        t1 = (int32_t)i1;
        return true;
      }
    }
    return false;
  }
};

}  // namespace fp4idx
