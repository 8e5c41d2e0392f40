// Schedule format shared by the schedule builder and the logits kernel.
//
// Query rows are cut into groups: maximal runs of consecutive rows with the same
// row_seq, split every kGroupMax rows.  A group's rows share every K tile (all draft
// rows of a sequence, or a block of prefill rows), so one tile load serves them all.
// Group g covers tiles [0, ntiles) of 128 tokens, ntiles = ceil(max context / 128), and
// costs kItemStartCost + ntiles * (kTileCost + rows) units (nothing when ntiles = 0): one
// unit per row and tile for the epilogue, a fixed charge per tile for streaming it, and a
// charge at the group's start for the CTA that switches to it mid-stream (its queries,
// head weights and lengths, about two pipeline stages of time).  The logits grid splits
// the total cost into num_ctas equal ranges; CTA c takes every tile whose cost interval
// starts in its range.  The split decides only which CTA computes a logit, never its value.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace fp4idx {

constexpr int kGroupMax = 6;  // six draft rows of a sequence share one group
constexpr int kTileTokens = 128;
constexpr int kTileCost = 2;
constexpr int kItemStartCost = 10;
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

// The first work item of one logits CTA, resolved by the schedule builder, so that the
// kernel's first page-table read waits on one load of this record and nothing else.
struct alignas(16) CtaStart {
  int64_t lo, hi;       // the CTA's cost range [lo, hi)
  int32_t g;            // group of the first item; n_groups when the range holds no item
  int32_t t0, t1;       // its tile range
  int32_t r0, rows;     // the group's first row and row count
  int32_t seq, maxlen;  // the group's sequence and longest clamped context
  int32_t n_groups;
};
static_assert(sizeof(CtaStart) == 48, "CtaStart layout");

struct SchedView {
  SchedHeader* hdr;
  int32_t* row0;     // [n_rows + 1] first row of each group (entry n_groups = n_rows)
  int32_t* maxlen;   // [n_rows] largest clamped context length in the group
  int32_t* seq;      // [n_rows] the group's sequence (row_seq of its rows), so that a work
                     // item's first page-table read need not wait on a row_seq load
  int64_t* prefix;   // [n_rows + 1] exclusive prefix of group costs
  uint32_t* sel_cnt; // [n_rows] per row, in a fused logits + selection call: the (tile,
                     // TMEM lane quarter) pieces of the row's logits written so far; zeroed
                     // by the build, put back to zero by the CTA that selects the row
  CtaStart* cta;     // [num_ctas] each logits CTA's cost range and first item
};

__host__ __device__ inline size_t sched_align16(size_t x) { return (x + 15) & ~(size_t)15; }

__host__ __device__ inline size_t sched_bytes(int64_t n_rows, int64_t num_ctas) {
  size_t b = sched_align16(sizeof(SchedHeader));
  b += sched_align16(sizeof(int32_t) * (size_t)(n_rows + 1));
  b += sched_align16(sizeof(int32_t) * (size_t)(n_rows + 1));
  b += sched_align16(sizeof(int32_t) * (size_t)(n_rows + 1));
  b += sched_align16(sizeof(int64_t) * (size_t)(n_rows + 1));
  b += sched_align16(sizeof(uint32_t) * (size_t)(n_rows + 1));
  b += sizeof(CtaStart) * (size_t)num_ctas;
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
  v.sel_cnt = reinterpret_cast<uint32_t*>(p);
  p += sched_align16(sizeof(uint32_t) * (size_t)(n_rows + 1));
  v.cta = reinterpret_cast<CtaStart*>(p);
  return v;
}

__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Cost of a group of `rows` rows whose longest clamped context is maxlen.
__host__ __device__ inline int64_t group_cost(int32_t maxlen, int32_t rows) {
  const int64_t ntiles = ceil_div64(maxlen, kTileTokens);
  return ntiles > 0 ? kItemStartCost + ntiles * (int64_t)(kTileCost + rows) : 0;
}

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

// One work item: tiles [t0, t1) of group g.
struct Item {
  int32_t g, t0, t1;
  int32_t r0, rows;     // the group's rows
  int32_t seq, maxlen;  // its sequence and longest clamped context
};

// Tile range [i0, i1) of a group whose cost interval starts at `base`, costs u per tile
// and has ntiles tiles, cut to the cost range [lo, hi).  The differences are clamped to
// the group's cost first, so the divisions are 32-bit.
__host__ __device__ __forceinline__ void item_tiles(int64_t lo, int64_t hi, int64_t base, int32_t u, int32_t ntiles,
                                           int32_t& i0, int32_t& i1) {
  const int64_t span = (int64_t)ntiles * u;
  const int32_t dl = (int32_t)(lo > base ? (lo - base < span ? lo - base : span) : 0);
  const int32_t dh = (int32_t)(hi > base ? (hi - base < span ? hi - base : span) : 0);
  i0 = (dl + u - 1) / u;
  i1 = (dh + u - 1) / u;
}

// First non-empty item of the cost range [lo, hi) at or after group g (advanced past
// it); false when there is none.  Accessors give a group's first row (row0(n_groups) =
// the row count), longest clamped context, sequence and cost-prefix entry.
template <class Row0, class MaxLen, class Seq, class Prefix>
__host__ __device__ __forceinline__ bool next_item(Row0 row0, MaxLen maxlen, Seq seq, Prefix prefix, int32_t n_groups,
                                          int64_t lo, int64_t hi, int32_t& g, Item& it) {
  while (g < n_groups && prefix(g) < hi) {
    const int32_t gg = g++;
    const int32_t r0 = row0(gg), rows = row0(gg + 1) - r0;
    const int32_t mx = maxlen(gg);
    const int32_t ntiles = (mx + kTileTokens - 1) / kTileTokens;
    int32_t i0, i1;
    item_tiles(lo, hi, prefix(gg) + kItemStartCost, kTileCost + rows, ntiles, i0, i1);
    if (i0 < i1) {
      it.g = gg;
      it.t0 = i0;
      it.t1 = i1;
      it.r0 = r0;
      it.rows = rows;
      it.seq = seq(gg);
      it.maxlen = mx;
      return true;
    }
  }
  return false;
}

// Iterates the items of one CTA in a fixed order: the first from the CTA's start record,
// the rest from the group arrays.
struct ItemIter {
  const int32_t* row0;
  const int32_t* maxlen;
  const int32_t* seq;
  const int64_t* prefix;
  int32_t n_groups;
  int64_t lo, hi;
  int32_t g;
  Item first;
  bool first_pending;

  __device__ void init(const SchedView& s, const CtaStart& c) {
    row0 = s.row0;
    maxlen = s.maxlen;
    seq = s.seq;
    prefix = s.prefix;
    n_groups = c.n_groups;
    lo = c.lo;
    hi = c.hi;
    first_pending = c.g < c.n_groups;
    g = first_pending ? c.g + 1 : c.n_groups;
    first.g = c.g;
    first.t0 = c.t0;
    first.t1 = c.t1;
    first.r0 = c.r0;
    first.rows = c.rows;
    first.seq = c.seq;
    first.maxlen = c.maxlen;
  }

  // Next non-empty item; false when this CTA's range is exhausted.
  __device__ bool next(Item& it) {
    if (first_pending) {
      first_pending = false;
      it = first;
      return true;
    }
    const int32_t* r = row0;
    const int32_t* m = maxlen;
    const int32_t* q = seq;
    const int64_t* x = prefix;
    return next_item([r](int32_t i) { return r[i]; }, [m](int32_t i) { return m[i]; },
                     [q](int32_t i) { return q[i]; }, [x](int32_t i) { return x[i]; }, n_groups, lo, hi, g, it);
  }
};

}  // namespace fp4idx
