// Paged-MQA logits over the split FP4 index-K cache, on the block-scaled tensor cores.
//
// [AMD] Enable FP4 indexer for Deepseek V4 -- Modifications: decode and prefill "FP4
// paged-MQA logits" read the 64-byte payload / 4-byte UE8M0 scale tensors through a
// guarded page table; the logits are
//   logits[t,s] = sum_h w[t,h] * ReLU(q_fp4[t,h] . k_fp4[s]),   s < context_lens[t].
//
// GB300 design (one persistent CTA per SM, 16 warps):
//   A tile is 128 tokens = two cache pages, the A operand of an M = 128 MMA laid out as
//   [block c][page][64 tokens][16 B] (canonical no-swizzle K-major).  A pipeline stage
//   holds two tiles (four pages).
//   warps 6-7 producers, taking alternate stages (issuing a gather4 occupies a warp
//           for about 120 cycles, so one warp alone cannot keep up with the SM's
//           share of HBM bandwidth): per stage, four TMA tile::gather4 loads of the
//           payload (each fetches the 1 KB rows (page, c) of two pages for two blocks,
//           landing directly in the interleaved operand layout) and one gather4 of the
//           four 256 B scale pages; warp 6 also loads each work item's query rows (one
//           bulk copy for the payloads, one for the scales).  Page ids are read 32 at
//           a time.
//   warps 0-3 scale writers, one per TMEM lane group: per tile, lane m of group m/32
//           gathers token m's four block-scale bytes from the [page][c][token] scale
//           pages and writes them with tcgen05.st to lane m, column m/32 of the tile's
//           four scale columns, where the block-scaled MMA reads row m's scales; per
//           work item, the query rows' head scales go to every lane group (heads l and
//           32 + l in lane l).  Four warps on four schedulers keep this transposition,
//           which every stage needs, off the critical path.
//   warps 4-5 MMA issuers (lane 0 of each), taking alternate stages: a lone issuing
//           thread runs its per-stage path of dependent instructions at a few cycles
//           each, which made it the pipeline's bottleneck.  Per (stage, query row), two
//           kind::mxf4 MMAs (K = 64 each) per
//           tile into a 64-column TMEM slot of its own (6 slots): D[128 tokens x 64 heads].
//           Slots per tile let the epilogue release each tile as soon as it has read
//           it and keep the MMAs up to three stages ahead of it.
//   warps 8-15 epilogue, two per TMEM lane group (half h reads tile h): thread =
//           TMEM lane = token; ReLU, head-weighted sum, mask at the row's context
//           length, coalesced fp32 store.
// Work items come from the length-balanced schedule (schedule.cuh).  Every wait is
// bounded: on expiry the CTA records FP4IDX_ERR_TIMEOUT, lets in-flight copies land,
// frees its tensor memory and returns.
//
// Fused top-k selection ([AMD] DeepSeek-V4.1-Flash on MI350X -- Changes: "sorted top-k
// selection"), when the launch has a CTA for every query row (decode batches): the
// epilogue warps publish, per item, how many (tile, lane quarter) pieces of each row they
// wrote (a release add on the row's counter in the schedule).  After its own work CTA c
// waits for row c's counter to reach all of the row's pieces, then selects the row from
// the logits in L2 (select.cuh), so the selection needs no second launch.  The launch is
// cooperative, so those waits cannot outlast a CTA that never ran.
#include <cooperative_groups.h>
#include <cuda.h>

#include <atomic>

#include "fp4idx_internal.cuh"
#include "launchers.cuh"
#include "pipeline.cuh"
#include "ptx.cuh"
#include "schedule.cuh"
#include "select.cuh"

namespace fp4idx {
namespace {

namespace cg = cooperative_groups;

constexpr int kStages = 8;          // pipeline stages, two tiles each
constexpr int kTilesPerStage = 2;
constexpr int kAccSlots = 3;        // TMEM accumulator slots, one (stage, query row) each: 128 columns
constexpr int kEpiWarps = 8;
constexpr int kProducers = 2;
constexpr int kScaleWarps = 4;
constexpr int kMmaWarps = 2;
constexpr int kWarps = kScaleWarps + kMmaWarps + kProducers + kEpiWarps;
constexpr int kThreads = kWarps * 32;
constexpr int kWarpMma = kScaleWarps, kWarpProducer = kWarpMma + kMmaWarps, kWarpEpi0 = kWarpProducer + kProducers;
static_assert(kStages % kProducers == 0 && kStages % kMmaWarps == 0 && kEpiWarps == 8,
              "stage ownership; four consecutive warps per epilogue half");
constexpr unsigned kFull = 0xFFFFFFFFu;
using pipe::Ctl;
using pipe::poll;
using pipe::prefetch_l2;
using pipe::wait_counts;
using pipe::wait_lane0;
using pipe::wait_warp;

// tensor memory columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColAcc = 0;                                     // kAccSlots x 128 fp32
constexpr uint32_t kColSfa = kAccSlots * 128;                       // kStages x 2 tiles x 4
constexpr uint32_t kColSfb = kColSfa + kStages * kTilesPerStage * 4;  // 2 x kGroupMax x 4
static_assert(kColSfb + 2 * kGroupMax * 4 <= kTmemCols, "tensor memory budget");
// Every epilogue warp consumes every slot use in order (half h reads tile h), so no
// parity wait is ever more than one phase ahead of its barrier.

// shared memory layout (bytes from the 1 KB-aligned dynamic base)
constexpr uint32_t kTileBytes = 8192;   // [c][2 pages][64][16]
constexpr uint32_t kKPayBytes = kTilesPerStage * kTileBytes;
constexpr uint32_t kKScBytes = 4 * 256;  // [4 pages][c][64]
constexpr uint32_t kQPayBytes = kGroupMax * 4096;
constexpr uint32_t kQScBytes = kGroupMax * 256;
constexpr uint32_t OFF_KPAY = 0;
constexpr uint32_t OFF_KSC = OFF_KPAY + kStages * kKPayBytes;
constexpr uint32_t OFF_QPAY = OFF_KSC + kStages * kKScBytes;
constexpr uint32_t OFF_QSC = OFF_QPAY + 2 * kQPayBytes;
constexpr uint32_t OFF_WEPI = OFF_QSC + 2 * kQScBytes;  // per epilogue warp: the item's head weights, [kGroupMax][64] fp32
constexpr uint32_t OFF_LEN = OFF_WEPI + kEpiWarps * kGroupMax * 256;  // per epilogue warp: [kGroupMax] int32
constexpr uint32_t OFF_BAR = OFF_LEN + kEpiWarps * kGroupMax * 4;
constexpr int kNumBars = 2 * kStages + 6 + kAccSlots;
// Monotonic arrival counters: per stage buffer, scale-writer warps that finished it
// (kScaleWarps per use); per accumulator slot, epilogue warps that released it
// (kEpiWarps per use).  The MMA issuer reads both with plain acquire loads issued
// together, which costs it one shared-memory round trip where two mbarrier probes
// (about 200 cycles each) would cost four times as much; counts that only grow
// cannot alias the way a phase-parity wait can.
constexpr uint32_t OFF_CNT = OFF_BAR + kNumBars * 8;
constexpr uint32_t OFF_MISC = OFF_CNT + (kStages + kAccSlots) * 4;
constexpr uint32_t kSmemBytes = OFF_MISC + 16;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(OFF_BAR % 8 == 0 && OFF_QPAY % 1024 == 0 && OFF_KSC % 128 == 0 && OFF_WEPI % 16 == 0, "alignment");

// The fused selection runs after every role has finished and reuses the dynamic shared
// memory from its start (the stage ring and query buffers): Sel::smem_words<1>(kSelRes)
// words, below the barriers.
constexpr int kSelRes = 32768;  // sort keys a CTA keeps in shared memory
using Sel = sel::Select<kThreads>;
static_assert(Sel::smem_words<1>(kSelRes) * 4 <= (int)OFF_BAR, "selection shared memory");

// barrier slots
__device__ __forceinline__ uint32_t bar_kfull(uint32_t b, int s) { return b + OFF_BAR + 8u * s; }
__device__ __forceinline__ uint32_t bar_kempty(uint32_t b, int s) { return b + OFF_BAR + 8u * (kStages + s); }
__device__ __forceinline__ uint32_t bar_qfull(uint32_t b, int q) { return b + OFF_BAR + 8u * (2 * kStages + q); }
__device__ __forceinline__ uint32_t bar_qempty(uint32_t b, int q) { return b + OFF_BAR + 8u * (2 * kStages + 2 + q); }
__device__ __forceinline__ uint32_t bar_qsf(uint32_t b, int q) { return b + OFF_BAR + 8u * (2 * kStages + 4 + q); }
__device__ __forceinline__ uint32_t bar_accfull(uint32_t b, int s) { return b + OFF_BAR + 8u * (2 * kStages + 6 + s); }
__device__ __forceinline__ uint32_t cnt_sf(uint32_t b, int s) { return b + OFF_CNT + 4u * s; }
__device__ __forceinline__ uint32_t cnt_slot(uint32_t b, int s) { return b + OFF_CNT + 4u * (kStages + s); }

struct LogitsParams {
  const uint8_t* q_payload;
  const uint8_t* q_scale;
  const float* w;
  int64_t num_pages;
  const int32_t* page_table;
  int64_t num_seqs;
  int32_t max_pages;
  const int32_t* row_seq;
  const int32_t* context_lens;
  int32_t max_context;
  int32_t n_rows;
  const void* schedule;
  float* out;
  int64_t out_stride;
  int32_t* status;
  // fused selection (k > 0): topk[n_rows][k]; per row, the spill of its sort keys past
  // kSelRes (the group counters live in the schedule)
  int32_t k;
  int32_t* topk;
  uint32_t* spill;
  int64_t spill_stride;
  uint64_t wait_limit_ns;  // how long one pipeline wait may last
  int32_t idle_producers;  // test switch: the producers issue nothing (every wait then runs out)
};

__device__ __forceinline__ uint32_t pack4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return a | (b << 8) | (c << 16) | (d << 24);
}

// TMA tile::gather4: rows r0..r3 (each one box of the 2D map) -> 4 consecutive rows in smem.
__device__ __forceinline__ void gather4(uint32_t dst, const CUtensorMap* map, int32_t r0, int32_t r1, int32_t r2,
                                        int32_t r3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(map), "r"(0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}

// Lane l's share of the 32 page ids starting at logical page 2 * tile0 of the item's
// sequence: the physical page, or -2 where the page lies past the item's longest context
// or the sequence is out of range.
__device__ __forceinline__ int32_t page_ids(const LogitsParams& p, const Item& it, int32_t tile0, int lane) {
  const bool seq_ok = it.seq >= 0 && (int64_t)it.seq < p.num_seqs;
  const int64_t span = min((int64_t)min(it.maxlen, p.max_context), (int64_t)p.max_pages * kPage);
  const int64_t npages = (span + kPage - 1) / kPage;
  const int64_t lp = 2 * (int64_t)tile0 + lane;
  if (!seq_ok || lp < 0 || lp >= npages) return -2;
  return __ldg(p.page_table + (int64_t)it.seq * p.max_pages + lp);
}

// Stage bookkeeping shared by all roles: tile pairs [i, i+1] of an item, in order.
__device__ __forceinline__ int stage_tiles(int32_t i, int32_t t1) { return min(kTilesPerStage, t1 - i); }

// A row's context length as every role reads it: clamped to [0, max_context], recording
// BAD_LENGTH once (by the caller's choice of `report`).
__device__ __forceinline__ int32_t clamped_len(const LogitsParams& p, int32_t row, bool report) {
  int32_t L = p.context_lens[row];
  if (L < 0 || L > p.max_context) {
    if (report) record_error(p.status, FP4IDX_ERR_BAD_LENGTH);
    L = L < 0 ? 0 : p.max_context;
  }
  return L;
}

// Fused selection (k > 0): the kSelC consecutive CTAs of group c select row c -- one CTA,
// or a pair in a thread-block cluster (the pair splits the row's positions and merges its
// counts through distributed shared memory).  The launch is cooperative, so every CTA is
// resident and may wait for the others.  A row with at most k tokens takes them all.
// Otherwise each CTA of the group waits, bounded, until the row's counter in the schedule
// shows every (tile, TMEM lane quarter) piece of its logits written -- each epilogue warp
// adds its pieces with a release after writing them.  The CTAs of a pair then tell each
// other whether they may go on (a CTA that timed out, or aborted its own pipeline, may
// not), so that neither enters the pair's cluster barriers alone; if both may, they select
// the row from the logits in L2 (select.cuh) and the counter goes back to zero.  Every
// thread of every CTA calls it once its roles have finished, aborted or not.
template <int kSelC>
__device__ __forceinline__ void select_own_row(const LogitsParams& p, const SchedView& sv, uint32_t* dyn,
                                              sel::Shared& sh, int32_t* go, bool aborted) {
  const int32_t row = blockIdx.x / kSelC;
  const int rank = (int)(blockIdx.x % kSelC);
  int32_t L = 0;
  bool need = false;
  if (row < p.n_rows) {
    L = clamped_len(p, row, threadIdx.x == 0 && rank == 0);
    if (L <= p.k) {
      int32_t* o = p.topk + (int64_t)row * p.k;
      if (rank == 0)
        for (int i = threadIdx.x; i < p.k; i += kThreads) o[i] = i < L ? i : -1;
    } else {
      need = !aborted;
    }
  }
  if (threadIdx.x == 0) {
    int ok = 0;
    if (need) {
      const uint32_t target = 4u * (uint32_t)((L + kTileTokens - 1) / kTileTokens);
      const uint64_t t0 = ptx::globaltimer();
      for (;;) {
        const uint32_t v = ptx::gmem_ld_acquire(sv.sel_cnt + row);
        if (v == target) {
          ok = 1;
          break;
        }
        if (v > target) {  // more pieces than the row has: the counters were not zero
          record_error(p.status, FP4IDX_ERR_SCHEDULE);
          break;
        }
        if (ptx::globaltimer() - t0 > p.wait_limit_ns) {
          record_error(p.status, FP4IDX_ERR_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    *go = ok;
  }
  int32_t* o = p.topk + (int64_t)row * p.k;
  const float* lg = p.out + (int64_t)row * p.out_stride;
  uint32_t* spill = p.spill + (int64_t)row * p.spill_stride;
  if constexpr (kSelC == 1) {
    __syncthreads();
    if (!*go) return;
    if (threadIdx.x == 0) sv.sel_cnt[row] = 0u;  // no other CTA touches it again in this call
    const int res = (int)min((int64_t)kSelRes, ((int64_t)L + 3) / 4 * 4);
    Sel::row<1, true>(lg, L, p.k, o, spill, res, dyn, sh, 0, p.status);
  } else {
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();  // both CTAs' flags are written
    const bool both = *go != 0 && *cl.map_shared_rank(go, rank ^ 1) != 0;
    cl.sync();  // both have read them
    if (!both) return;
    if (threadIdx.x == 0 && rank == 0) sv.sel_cnt[row] = 0u;  // both CTAs have seen it complete
    const int64_t per = (((int64_t)L + 3) / 4 + 1) / 2;  // groups of four a CTA
    const int res = (int)min((int64_t)kSelRes, 4 * per);
    Sel::row<2, true>(lg, L, p.k, o, spill, res, dyn, sh, rank, p.status);
  }
}

// kSelC: the CTAs that select each row in the fused call (1 or 2); 0 for a launch without
// the selection, which compiles out the epilogue's piece counting and the selecting tail.
template <int kSelC>
__global__ void __launch_bounds__(kThreads, 1) logits_mxf4_kernel(const __grid_constant__ CUtensorMap pay_map,
                                                                 const __grid_constant__ CUtensorMap sc_map,
                                                                 const LogitsParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sb = ptx::smem_addr(smem);

  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + OFF_MISC + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; s++) {
      ptx::mbar_init(bar_kfull(sb, s), 1);
      ptx::mbar_init(bar_kempty(sb, s), 1);
    }
    for (int i = 0; i < kStages + kAccSlots; i++) reinterpret_cast<uint32_t*>(smem + OFF_CNT)[i] = 0u;
    for (int q = 0; q < 2; q++) {
      ptx::mbar_init(bar_qfull(sb, q), 1);
      ptx::mbar_init(bar_qempty(sb, q), kMmaWarps);  // each issuer commits once per item
      ptx::mbar_init(bar_qsf(sb, q), kScaleWarps);
    }
    for (int s = 0; s < kAccSlots; s++) ptx::mbar_init(bar_accfull(sb, s), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kWarpProducer && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&pay_map) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&sc_map) : "memory");
  }
  if (warp == kWarpMma) ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{abort_flag, p.status, p.wait_limit_ns};

  // Everything above runs while a preceding kernel launched as this launch's programmatic
  // primary (the step preparation: schedule, queries, new cache rows) may still be working;
  // nothing below may read before its results are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // The schedule must describe exactly these rows and this grid (the same header in every
  // CTA, so every CTA takes the same branch).  The CTA's start record (inside the
  // workspace the host checked against this grid) loads with the header.
  const SchedView sv = sched_view(const_cast<void*>(p.schedule), p.n_rows);
  const SchedHeader hdr = *sv.hdr;
  const CtaStart cs = sv.cta[blockIdx.x];
  const bool valid = hdr.magic == kSchedMagic && hdr.n_rows == p.n_rows && hdr.num_ctas == (int32_t)gridDim.x &&
                     hdr.group_max == kGroupMax;
  if (!valid && threadIdx.x == 0) record_error(p.status, FP4IDX_ERR_SCHEDULE);
  ItemIter items;
  items.init(sv, cs);
  const bool is_producer = warp >= kWarpProducer && warp < kWarpEpi0;
  Item it;
  bool have = false;
  int32_t pid_cur = -2, pid_next = -2;
  if (valid && is_producer && !p.idle_producers) {
    have = items.next(it);
    if (have) {
      pid_cur = page_ids(p, it, it.t0, lane);
      pid_next = page_ids(p, it, it.t0 + 16, lane);
    }
  }

  if (!valid) {
    // no work: straight to the end
  } else if (is_producer) {
    // ------------------------------------------------------------ producers
    const int pw = warp - kWarpProducer;  // issues the stages with kctr % kProducers == pw
    uint32_t kctr = 0, ictr = 0;
    bool ok = true;
    while (ok && have) {
      const int32_t r0 = it.r0, rows = it.rows;
      const bool seq_ok = it.seq >= 0 && (int64_t)it.seq < p.num_seqs;
      const int qb = ictr & 1;
      if (pw == 0) {
        ok = wait_lane0(bar_qempty(sb, qb), ((ictr >> 1) & 1) ^ 1, ctl);
        if (!ok) break;
        if (lane == 0) {
          const uint32_t qbar = bar_qfull(sb, qb);
          ptx::mbar_arrive_expect_tx(qbar, (uint32_t)rows * (4096u + 256u));
          ptx::bulk_g2s(sb + OFF_QPAY + qb * kQPayBytes, p.q_payload + (int64_t)r0 * 4096, rows * 4096u, qbar);
          ptx::bulk_g2s(sb + OFF_QSC + qb * kQScBytes, p.q_scale + (int64_t)r0 * 256, rows * 256u, qbar);
          if (!seq_ok) record_error(p.status, FP4IDX_ERR_BAD_PAGE);
        }
      }
      // The next item is looked up, and its first page ids requested, once this warp has
      // filled its share of the ring (or at the end of a shorter item), so that a CTA
      // whose range spans two groups does not stall on that chain at the switch.  Warp 0
      // also warms the next item's query rows, head weights and lengths in L2.
      Item nx;
      bool have_nx = false, looked = false;
      int32_t nx_cur = -2, nx_next = -2;
      auto look_ahead = [&]() {
        looked = true;
        have_nx = items.next(nx);
        if (!have_nx) return;
        nx_cur = page_ids(p, nx, nx.t0, lane);
        nx_next = page_ids(p, nx, nx.t0 + 16, lane);
        if (pw == 0) {
          for (int j = lane; j < nx.rows * 32; j += 32) prefetch_l2(p.q_payload + (int64_t)nx.r0 * 4096 + j * 128);
          if (lane < 2 * nx.rows) {
            prefetch_l2(p.q_scale + (int64_t)nx.r0 * 256 + lane * 128);
            prefetch_l2(reinterpret_cast<const uint8_t*>(p.w + (int64_t)nx.r0 * 64) + lane * 128);
          }
          if (lane == 0) prefetch_l2(p.context_lens + nx.r0);
        }
      };
      int own = 0;
      int32_t chunk = it.t0;
      for (int32_t i = it.t0; i < it.t1; i += kTilesPerStage, kctr++) {
        if (i - chunk >= 16) {
          chunk += 16;
          pid_cur = pid_next;
          pid_next = page_ids(p, it, chunk + 16, lane);
        }
        if ((int)(kctr % kProducers) != pw) continue;
        const int s = kctr % kStages;
        ok = wait_lane0(bar_kempty(sb, s), ((kctr / kStages) & 1) ^ 1, ctl);
        if (!ok) break;
        const int tiles = stage_tiles(i, it.t1);
        // pages of this stage in lanes 0..3 (tile a: pages 2a, 2a+1)
        int32_t pg = __shfl_sync(kFull, pid_cur, (2 * (i - chunk) + (lane & 3)) & 31);
        const bool needed = (lane & 3) < 2 * tiles && pg != -2;
        const bool valid = pg >= 0 && (int64_t)pg < p.num_pages;
        if (lane < 4 && needed && !valid) record_error(p.status, FP4IDX_ERR_BAD_PAGE);
        if (!valid) pg = 0;
        const int32_t q0 = __shfl_sync(kFull, pg, 0), q1 = __shfl_sync(kFull, pg, 1);
        const int32_t q2 = __shfl_sync(kFull, pg, 2), q3 = __shfl_sync(kFull, pg, 3);
        const uint32_t kbar = bar_kfull(sb, s);
        if (lane == 0) ptx::mbar_arrive_expect_tx(kbar, (uint32_t)tiles * kTileBytes + kKScBytes);
        __syncwarp();
        // lanes 0-3: tile lane/2, blocks (2h, 2h+1) with h = lane%2, each row (page, block)
        // 1 KB; lane 4: the four scale pages
        if (lane < 4) {
          const int a = lane >> 1, h = lane & 1;
          const int32_t pa = a ? q2 : q0, pb = a ? q3 : q1;
          if (a < tiles)
            gather4(sb + OFF_KPAY + s * kKPayBytes + a * kTileBytes + h * 4096, &pay_map, 4 * pa + 2 * h,
                    4 * pb + 2 * h, 4 * pa + 2 * h + 1, 4 * pb + 2 * h + 1, kbar);
        } else if (lane == 4) {
          gather4(sb + OFF_KSC + s * kKScBytes, &sc_map, q0, q1, q2, q3, kbar);
        }
        __syncwarp();
        if (!looked && ++own == kStages / kProducers) look_ahead();
      }
      ictr++;  // also after a failed stage wait: this item's query copies were issued
      if (!ok) break;
      if (!looked) look_ahead();
      it = nx;
      have = have_nx;
      pid_cur = nx_cur;
      pid_next = nx_next;
    }
    // Tail: every copy a warp issued must land, and (when not aborting) every stage must
    // be released by the MMAs that read it, before the CTA may exit.  kctr stops at the
    // stage a failed wait was for, which this warp did not issue.
    for (uint32_t u = (kctr > (uint32_t)kStages ? kctr - kStages : 0); u < kctr; u++) {
      if ((int)(u % kProducers) != pw) continue;
      wait_lane0(bar_kfull(sb, u % kStages), (u / kStages) & 1, ctl, false);
      if (!*abort_flag) wait_lane0(bar_kempty(sb, u % kStages), (u / kStages) & 1, ctl);
    }
    if (pw == 0) {
      for (uint32_t u = (ictr > 2u ? ictr - 2 : 0); u < ictr; u++) {
        wait_lane0(bar_qfull(sb, u & 1), (u >> 1) & 1, ctl, false);
        if (!*abort_flag) wait_lane0(bar_qempty(sb, u & 1), (u >> 1) & 1, ctl);
      }
    }
  } else if (warp >= kWarpMma && warp < kWarpMma + kMmaWarps) {
    // ------------------------------------------------------------ MMA issuers (lane 0)
    const int mw = warp - kWarpMma;  // issues the stages with kctr % kMmaWarps == mw
    if (lane == 0) {
      uint32_t kctr = 0, ictr = 0, ucnt = 0;
      bool ok = true;
      constexpr uint32_t kIdesc0 = ptx::idesc_mxf4(64, 0, 0);
      constexpr uint32_t kIdesc1 = ptx::idesc_mxf4(64, 2, 2);
      Item it;
      while (ok && items.next(it)) {
        const int32_t rows = it.rows;
        const int qb = ictr & 1;
        bool q_ready = false;
        for (int32_t i = it.t0; i < it.t1 && ok; i += kTilesPerStage, kctr++, ucnt += rows) {
          if ((int)(kctr % kMmaWarps) != mw) continue;
          if (!q_ready) {
            // query rows landed and their scales are in tensor memory
            ok = poll(bar_qsf(sb, qb), (ictr >> 1) & 1, ctl, true);
            if (!ok) break;
            ptx::tc_fence_after();
            q_ready = true;
          }
          const int s = kctr % kStages;
          const int tiles = stage_tiles(i, it.t1);
          // the stage's tiles landed with their scales in tensor memory (every scale
          // writer done with this use of the buffer), and each row's accumulator slot
          // is free (every epilogue warp released its previous use)
          const uint32_t need_sf = (uint32_t)kScaleWarps * (kctr / kStages + 1);
          for (int r = 0; r < rows; r++) {
            const uint32_t u = ucnt + r;
            const int slot = u % kAccSlots;
            ok = wait_counts(cnt_sf(sb, s), need_sf, cnt_slot(sb, slot), (uint32_t)kEpiWarps * (u / kAccSlots), ctl);
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t b0 = sb + OFF_QPAY + qb * kQPayBytes + r * 4096;
            const uint32_t sfbt = tmem + kColSfb + (qb * kGroupMax + r) * 4;
            for (int a = 0; a < tiles; a++) {
              const uint32_t a0 = sb + OFF_KPAY + s * kKPayBytes + a * kTileBytes;
              const uint32_t d = tmem + kColAcc + slot * 128 + a * 64;
              const uint32_t sfa = tmem + kColSfa + (s * kTilesPerStage + a) * 4;
              ptx::mma_mxf4(d, ptx::smem_desc(a0, 2048, 128), ptx::smem_desc(b0, 1024, 128), kIdesc0, sfa, sfbt, 0);
              ptx::mma_mxf4(d, ptx::smem_desc(a0 + 4096, 2048, 128), ptx::smem_desc(b0 + 2048, 1024, 128), kIdesc1,
                            sfa, sfbt, 1);
            }
            ptx::mma_commit(bar_accfull(sb, slot));
          }
          if (!ok) break;
          ptx::mma_commit(bar_kempty(sb, s));
        }
        if (!ok) break;
        // this issuer is done with the item's queries: once its MMAs have read them, or, when
        // it issued none for this item, once the item's rows are in place.  An arrival made
        // before that would count toward the buffer's previous use, which the other issuer
        // may still be reading, and let the producer overwrite it.
        if (q_ready) {
          ptx::mma_commit(bar_qempty(sb, qb));
        } else {
          ok = poll(bar_qsf(sb, qb), (ictr >> 1) & 1, ctl, true);
          if (!ok) break;
          ptx::mbar_arrive(bar_qempty(sb, qb));
        }
        ictr++;
      }
    }
  } else if (warp < kScaleWarps) {
    // ------------------------------------------------------------ scale writers
    const int qd = warp;  // TMEM lane group: tile rows 32*qd .. 32*qd + 31
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    uint32_t kctr = 0, ictr = 0;
    bool ok = true;
    Item it;
    while (ok && items.next(it)) {
      const int32_t rows = it.rows;
      const int qb = ictr & 1;
      ok = wait_warp(bar_qfull(sb, qb), (ictr >> 1) & 1, ctl);
      if (!ok) break;
      for (int r = 0; r < rows; r++) {
        // query row r: B operand of 64 heads, the same in every lane group; lane l holds
        // heads l and 32 + l in the row's first two scale columns
        const uint8_t* src = smem + OFF_QSC + qb * kQScBytes + r * 256 + lane;  // [c][64 heads]
        const uint32_t w0 = pack4(src[0], src[64], src[128], src[192]);
        const uint32_t w1 = pack4(src[32], src[96], src[160], src[224]);
        ptx::tmem_st4(tmem + lane_base + kColSfb + (qb * kGroupMax + r) * 4, w0, w1, 0u, 0u);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_qsf(sb, qb));
      for (int32_t i = it.t0; i < it.t1; i += kTilesPerStage) {
        const int s = kctr % kStages;
        const int tiles = stage_tiles(i, it.t1);
        ok = wait_warp(bar_kfull(sb, s), (kctr / kStages) & 1, ctl);
        if (!ok) break;
        for (int a = 0; a < tiles; a++) {
          // tile a: token m = 32*qd + lane is token 32*(qd & 1) + lane of page 2a + qd/2
          const uint8_t* src = smem + OFF_KSC + s * kKScBytes + (2 * a + (qd >> 1)) * 256 + (qd & 1) * 32 + lane;
          const uint32_t wv = pack4(src[0], src[64], src[128], src[192]);
          ptx::tmem_st4(tmem + lane_base + kColSfa + (s * kTilesPerStage + a) * 4, qd == 0 ? wv : 0u,
                        qd == 1 ? wv : 0u, qd == 2 ? wv : 0u, qd == 3 ? wv : 0u);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::smem_add_release(cnt_sf(sb, s), 1u);
        kctr++;
      }
      ictr++;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - kWarpEpi0;  // 0..7: private copy of the group's lengths
    const int half = ew >> 2;         // reads tile `half` of every slot use
    const int quad = warp & 3;        // TMEM lanes this warp may read
    const int m = quad * 32 + lane;   // token row of a tile
    int32_t* lsm = reinterpret_cast<int32_t*>(smem + OFF_LEN) + ew * kGroupMax;
    float* wsm = reinterpret_cast<float*>(smem + OFF_WEPI) + ew * kGroupMax * 64;  // this warp's copy
    uint32_t ucnt = 0;
    bool ok = true;
    Item it;
    while (ok && items.next(it)) {
      const int32_t r0 = it.r0, rows = it.rows;
      __syncwarp();
      if (lane < rows) {
        int32_t L = __ldg(p.context_lens + r0 + lane);
        if (L < 0 || L > p.max_context) {
          if (ew == 0) record_error(p.status, FP4IDX_ERR_BAD_LENGTH);
          L = L < 0 ? 0 : p.max_context;
        }
        lsm[lane] = L;
      }
      // the group's head weights, copied once per item into this warp's own shared memory
      // (read back as broadcast shared loads, off the global-load scoreboard)
      for (int j = lane; j < rows * 16; j += 32)
        reinterpret_cast<float4*>(wsm)[j] = __ldg(reinterpret_cast<const float4*>(p.w + (int64_t)r0 * 64) + j);
      __syncwarp();
      // fused selection: lane r counts the (tile, lane quarter) pieces of row r0 + r this
      // warp writes in the item
      uint32_t pieces = 0;
      for (int32_t i = it.t0; i < it.t1 && ok; i += kTilesPerStage) {
        const int tiles = stage_tiles(i, it.t1);
        for (int r = 0; r < rows && ok; r++) {
          const float* wr = wsm + r * 64;  // same address in every lane: shared-memory broadcast
          const int32_t L = lsm[r];
          float* orow = p.out + (int64_t)(r0 + r) * p.out_stride;
          {
            const int a = half;
            const int slot = ucnt % kAccSlots;
            ok = wait_warp(bar_accfull(sb, slot), (ucnt / kAccSlots) & 1, ctl);
            ucnt++;
            if (!ok) break;
            ptx::tc_fence_after();
            float d[64];
            if (a < tiles) ptx::tmem_ld64_sync(tmem + ((uint32_t)(quad * 32) << 16) + kColAcc + slot * 128 + a * 64, d);
            // released as soon as read (also by a warp with no tile here: every epilogue
            // warp arrives once per use)
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::smem_add_release(cnt_slot(sb, slot), 1u);
            if (a >= tiles) continue;
            const int32_t tok = (i + a) * kTileTokens + m;
            // a row the launch selects (more than k tokens) and a tile holding some of them
            const bool counted = kSelC > 0 && p.k > 0 && L > p.k && (i + a) * kTileTokens < L;
            if (counted && lane == r) pieces++;
            if (tok < L) {
              // sum_h w_h * ReLU(d_h): scalar ReLU, packed pair FMAs, eight partial sums
              // (head h goes to partial h mod 8) so that the dependent chains are short
              float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f, a4 = 0.f, a5 = 0.f, a6 = 0.f, a7 = 0.f;
#pragma unroll
              for (int h = 0; h < 64; h += 8) {
                const float4 wv = *reinterpret_cast<const float4*>(wr + h);
                const float4 wu = *reinterpret_cast<const float4*>(wr + h + 4);
                ptx::ffma2(a0, a1, wv.x, wv.y, fmaxf(d[h + 0], 0.f), fmaxf(d[h + 1], 0.f));
                ptx::ffma2(a2, a3, wv.z, wv.w, fmaxf(d[h + 2], 0.f), fmaxf(d[h + 3], 0.f));
                ptx::ffma2(a4, a5, wu.x, wu.y, fmaxf(d[h + 4], 0.f), fmaxf(d[h + 5], 0.f));
                ptx::ffma2(a6, a7, wu.z, wu.w, fmaxf(d[h + 6], 0.f), fmaxf(d[h + 7], 0.f));
              }
              orow[tok] = ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
            }
          }
        }
      }
      // this warp's pieces of the item's rows are written: publish them (release at GPU
      // scope, after the warp's logits stores)
      __syncwarp();
      if constexpr (kSelC > 0) {
        if (ok && pieces > 0) ptx::gmem_red_release_add(sv.sel_cnt + r0 + lane, pieces);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kWarpMma) ptx::tmem_dealloc(tmem, kTmemCols);
  if constexpr (kSelC > 0) {
    if (p.k > 0 && valid) {
      __shared__ sel::Shared sel_sh;
      __shared__ int32_t sel_go;
      select_own_row<kSelC>(p, sv, reinterpret_cast<uint32_t*>(smem), sel_sh, &sel_go, *abort_flag != 0);
    }
  }
}

inline int64_t select_spill_stride(int32_t max_context) {
  return max((int64_t)0, ((int64_t)max(max_context, 1) + 3) / 4 * 4 - kSelRes);
}

}  // namespace

namespace {

// Whether num_ctas CTAs of the logits kernel in clusters of two can all be resident at
// once on the current device (asked once per device and grid).
bool pairs_fit(int32_t num_ctas) {
  static std::atomic<int> known[64];  // 0 unknown, else 1 + answer, for the last grid asked
  static std::atomic<int> known_grid[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return false;
  }
  if (known_grid[dev].load() == num_ctas && known[dev].load() != 0) return known[dev].load() == 2;
  bool fit = false;
  if (num_ctas % 2 == 0 &&
      set_smem_attr_once(reinterpret_cast<const void*>(logits_mxf4_kernel<2>), kSmemBytes) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num_ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    fit = cudaOccupancyMaxActiveClusters(&clusters, logits_mxf4_kernel<2>, &cfg) == cudaSuccess &&
          2 * clusters >= num_ctas;
  }
  cudaGetLastError();
  known_grid[dev].store(num_ctas);
  known[dev].store(fit ? 2 : 1);
  return fit;
}

}  // namespace

size_t logits_select_spill_bytes(int64_t n_rows, int32_t max_context) {
  return (((size_t)n_rows * (size_t)select_spill_stride(max_context) * sizeof(uint32_t) + 255) & ~(size_t)255) + 256;
}

cudaError_t launch_logits_mxf4(const uint8_t* q_payload, const uint8_t* q_scale, const float* w, int32_t n_rows,
                               const uint8_t* payload, const uint8_t* scale, int64_t num_pages,
                               const int32_t* page_table, int64_t num_seqs, int32_t max_pages,
                               const int32_t* row_seq, const int32_t* context_lens, int32_t max_context,
                               const void* schedule, int32_t num_ctas, float* out, int64_t out_stride,
                               int32_t k, int32_t* topk, void* spill, int32_t* status, cudaStream_t stream) {
  if (num_pages < 1) return cudaErrorInvalidValue;
  CUtensorMap pay_map, sc_map;
  if (!encode_rows(&pay_map, payload, num_pages * 4, 1024) || !encode_rows(&sc_map, scale, num_pages, 256))
    return cudaErrorInvalidValue;
  LogitsParams prm;
  prm.q_payload = q_payload;
  prm.q_scale = q_scale;
  prm.w = w;
  prm.num_pages = num_pages;
  prm.page_table = page_table;
  prm.num_seqs = num_seqs;
  prm.max_pages = max_pages;
  prm.row_seq = row_seq;
  prm.context_lens = context_lens;
  prm.max_context = max_context;
  prm.n_rows = n_rows;
  prm.schedule = schedule;
  prm.out = out;
  prm.out_stride = out_stride;
  prm.status = status;
  prm.k = topk ? k : 0;
  prm.topk = topk;
  prm.spill = reinterpret_cast<uint32_t*>(spill);
  prm.spill_stride = select_spill_stride(max_context);
  prm.wait_limit_ns = pipeline_wait_limit_ns();
  prm.idle_producers = pipeline_idle_producers() ? 1 : 0;
  if (prm.k > 0 && n_rows > num_ctas) return cudaErrorInvalidValue;  // the selection needs a CTA per row
  // A pair of CTAs per row when the grid holds two for every row and the pairs (clusters
  // of two) can all be resident at once; else one CTA per row.
  // (no selection: the instantiation without the epilogue's piece counting and the tail)
  const int sel_c = prm.k == 0 ? 0 : 2 * (int64_t)n_rows <= num_ctas && pairs_fit(num_ctas) ? 2 : 1;
  const void* fn = sel_c == 2   ? reinterpret_cast<const void*>(logits_mxf4_kernel<2>)
                   : sel_c == 1 ? reinterpret_cast<const void*>(logits_mxf4_kernel<1>)
                                : reinterpret_cast<const void*>(logits_mxf4_kernel<0>);
  cudaError_t e = set_smem_attr_once(fn, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  // With the fused selection, CTAs wait for rows that other CTAs write: the launch must
  // be cooperative, which guarantees that every CTA is resident at once.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = prm.k > 0 ? sel_c : 0;
  if (prm.k == 0) {
    // a programmatic dependent launch: its set-up may overlap the end of the kernel before
    // it on the stream (the kernel waits for that kernel's results before reading them)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
  }
  if (sel_c == 2) return cudaLaunchKernelEx(&cfg, logits_mxf4_kernel<2>, pay_map, sc_map, prm);
  if (sel_c == 1) return cudaLaunchKernelEx(&cfg, logits_mxf4_kernel<1>, pay_map, sc_map, prm);
  return cudaLaunchKernelEx(&cfg, logits_mxf4_kernel<0>, pay_map, sc_map, prm);
}

}  // namespace fp4idx
