// Paged-MQA logits over the 132 B/token FP8 indexer cache, on the tensor cores
// (tcgen05 kind::f8f6f4): the FP8 side of the FP4/FP8 comparison.
//
// [AMD] Enable FP4 indexer for Deepseek V4 -- Device memory and sizing: the FP4 entry of
// 68 B a token replaces a fused FP8 entry of 132 B (128 e4m3 values and one fp32 scale).
// The logits are those of the FP4 path,
//   logits[t,s] = sum_h w[t,h] * ReLU(q[t,h] . k[s]),   s < context_lens[t],
// with q = e4m3(q8) * q8_scale[t,h] and k = e4m3(k8) * k_scale[s].  Both scales are
// positive, so they leave the contraction:
//   logits[t,s] = k_scale[s] * sum_h (w[t,h] q8_scale[t,h]) * ReLU(q8[t,h] . k8[s]).
//
// The pipeline is that of the FP4 kernel (logits_mxf4.cu): one persistent CTA per SM,
// 16 warps, the same length-balanced schedule and 128-token tiles, bounded waits.  What
// differs:
//   - A page of the fused layout is 66 rows of 128 B: 64 token rows, then the 256 B of
//     token scales.  A 3-D tensor map {128 B, 66 rows, pages} with a box {16 B, 64, 1}
//     lands the 16-byte chunk c of a page's 64 token rows as 1 KB, so a tile (two pages)
//     arrives in the canonical no-swizzle K-major operand layout [chunk][page][64][16 B]
//     (16 KB, 8 chunks).  A stage holds two tiles: each lane of a producer warp issues
//     one of its 32 loads.
//   - No block scales, hence no scale writers: warps 0-3 are the producers, one stage
//     buffer each.  Warps 4-5 issue the MMAs; warps 6-7 have no role.
//   - Per (tile, query row), four MMAs of M = 128, N = 64, K = 32 (e4m3 x e4m3 -> f32).
//   - The epilogue folds q8_scale into its copy of the head weights and multiplies each
//     token's sum by the token's scale, read from the page's scale rows (which the
//     producer warms in L2 when it loads the page).
//   - Query rows are 8 KB, so one query buffer of a full group sits beside four stages.
#include <cuda.h>

#include "fp4idx_internal.cuh"
#include "launchers.cuh"
#include "pipeline.cuh"
#include "ptx.cuh"
#include "schedule.cuh"

namespace fp4idx {
namespace {

constexpr int kStages = 4;  // pipeline stages, two tiles each
constexpr int kTilesPerStage = 2;
constexpr int kAccSlots = 3;  // TMEM accumulator slots, one (stage, query row) each: 128 columns
constexpr int kProducers = 4;
constexpr int kMmaWarps = 2;
constexpr int kIdleWarps = 2;
constexpr int kEpiWarps = 8;
constexpr int kWarps = kProducers + kMmaWarps + kIdleWarps + kEpiWarps;
constexpr int kThreads = kWarps * 32;
constexpr int kWarpMma = kProducers, kWarpEpi0 = kProducers + kMmaWarps + kIdleWarps;
// A producer (an issuer) owns every use of the stage buffers it fills (reads), so that no
// parity wait on a stage barrier can be more than one phase ahead of it.
static_assert(kStages % kProducers == 0 && kStages % kMmaWarps == 0, "stage ownership");
static_assert(kEpiWarps == 8 && kWarpEpi0 % 4 == 0, "four consecutive warps per epilogue half, quad = warp % 4");
constexpr unsigned kFull = 0xFFFFFFFFu;
using pipe::Ctl;
using pipe::poll;
using pipe::prefetch_l2;
using pipe::wait_lane0;
using pipe::wait_warp;

constexpr uint32_t kPageBytes = 8448;   // 64 x 128 B e4m3, then 64 x 4 B fp32 scales
constexpr uint32_t kScaleOff = 8192;
constexpr uint32_t kTmemCols = 512;     // kAccSlots x 128 fp32 columns, rounded up to a power of two
static_assert(kAccSlots * 128 <= kTmemCols, "tensor memory budget");

// shared memory layout (bytes from the 1 KB-aligned dynamic base)
constexpr uint32_t kTileBytes = 16384;  // [8 chunks][2 pages][64 tokens][16 B]
constexpr uint32_t kStageBytes = kTilesPerStage * kTileBytes;
constexpr uint32_t kQRowBytes = 8192;   // [8 chunks][64 heads][16 B]
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_Q = OFF_K + kStages * kStageBytes;
constexpr uint32_t OFF_WEPI = OFF_Q + kGroupMax * kQRowBytes;  // per epilogue warp: [kGroupMax][64] fp32
constexpr uint32_t OFF_LEN = OFF_WEPI + kEpiWarps * kGroupMax * 256;  // per epilogue warp: [kGroupMax] int32
constexpr uint32_t OFF_BAR = OFF_LEN + kEpiWarps * kGroupMax * 4;
constexpr int kNumBars = 2 * kStages + 2 + kAccSlots;
// per accumulator slot: epilogue warps that released it (kEpiWarps per use); only grows
constexpr uint32_t OFF_CNT = OFF_BAR + kNumBars * 8;
constexpr uint32_t OFF_MISC = OFF_CNT + kAccSlots * 4;
constexpr uint32_t kSmemBytes = OFF_MISC + 16;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(OFF_Q % 1024 == 0 && OFF_WEPI % 16 == 0 && OFF_BAR % 8 == 0, "alignment");

__device__ __forceinline__ uint32_t bar_kfull(uint32_t b, int s) { return b + OFF_BAR + 8u * s; }
__device__ __forceinline__ uint32_t bar_kempty(uint32_t b, int s) { return b + OFF_BAR + 8u * (kStages + s); }
__device__ __forceinline__ uint32_t bar_qfull(uint32_t b) { return b + OFF_BAR + 8u * (2 * kStages); }
__device__ __forceinline__ uint32_t bar_qempty(uint32_t b) { return b + OFF_BAR + 8u * (2 * kStages + 1); }
__device__ __forceinline__ uint32_t bar_accfull(uint32_t b, int s) { return b + OFF_BAR + 8u * (2 * kStages + 2 + s); }
__device__ __forceinline__ uint32_t cnt_slot(uint32_t b, int s) { return b + OFF_CNT + 4u * s; }

struct LogitsFp8Params {
  const uint8_t* q8;
  const float* q8_scale;
  const float* w;
  const uint8_t* pages;
  int64_t num_pages;
  const int32_t* page_table;
  int64_t num_seqs;
  int32_t max_pages;
  const int32_t* context_lens;
  int32_t max_context;
  int32_t n_rows;
  const void* schedule;
  float* out;
  int64_t out_stride;
  int32_t* status;
  uint64_t wait_limit_ns;  // how long one pipeline wait may last
  int32_t idle_producers;  // test switch: the producers issue nothing (every wait then runs out)
};

// Bounded wait, by one thread, until the shared-memory counter at `a` has reached `need`.
__device__ __forceinline__ bool wait_count(uint32_t a, uint32_t need, const Ctl& c) {
  return pipe::wait_counts(a, need, a, need, c);
}

// TMA tiled load of one box of a 3-D tensor map; x is the innermost coordinate (bytes
// here, a multiple of 16).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Instruction descriptor, kind::f8f6f4: D f32 (bits 4-5 = 1), A and B e4m3 (format 0 in
// bits 7-9 and 10-12), both K-major, no negation, N >> 3 in bits 17-22, M >> 4 in bits
// 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3(int n, int m) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D[tmem] (+)= A[smem] x B[smem]^T, e4m3 x e4m3 -> f32, one CTA, issued by one thread.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Lane l's share of the 32 page ids starting at logical page 2 * tile0 of the item's
// sequence: the physical page, or -2 past the item's longest context or for a sequence
// out of range.
__device__ __forceinline__ int32_t page_ids(const LogitsFp8Params& p, const Item& it, int32_t tile0, int lane) {
  const bool seq_ok = it.seq >= 0 && (int64_t)it.seq < p.num_seqs;
  const int64_t span = min((int64_t)min(it.maxlen, p.max_context), (int64_t)p.max_pages * kPage);
  const int64_t npages = (span + kPage - 1) / kPage;
  const int64_t lp = 2 * (int64_t)tile0 + lane;
  if (!seq_ok || lp < 0 || lp >= npages) return -2;
  return __ldg(p.page_table + (int64_t)it.seq * p.max_pages + lp);
}

__device__ __forceinline__ int stage_tiles(int32_t i, int32_t t1) { return min(kTilesPerStage, t1 - i); }

__global__ void __launch_bounds__(kThreads, 1) logits_fp8_kernel(const __grid_constant__ CUtensorMap k_map,
                                                                const LogitsFp8Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sb = ptx::smem_addr(smem);

  const SchedView sv = sched_view(const_cast<void*>(p.schedule), p.n_rows);
  const SchedHeader hdr = *sv.hdr;
  const CtaStart cs = sv.cta[blockIdx.x];
  if (hdr.magic != kSchedMagic || hdr.n_rows != p.n_rows || hdr.num_ctas != (int32_t)gridDim.x ||
      hdr.group_max != kGroupMax) {
    if (threadIdx.x == 0) record_error(p.status, FP4IDX_ERR_SCHEDULE);
    return;
  }
  ItemIter items;
  items.init(sv, cs);

  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + OFF_MISC + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; s++) {
      ptx::mbar_init(bar_kfull(sb, s), 1);
      ptx::mbar_init(bar_kempty(sb, s), 1);
    }
    ptx::mbar_init(bar_qfull(sb), 1);
    ptx::mbar_init(bar_qempty(sb), kMmaWarps);  // each issuer releases once per item
    for (int s = 0; s < kAccSlots; s++) {
      ptx::mbar_init(bar_accfull(sb, s), 1);
      reinterpret_cast<uint32_t*>(smem + OFF_CNT)[s] = 0u;
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(&k_map) : "memory");
  if (warp == kWarpMma) ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{abort_flag, p.status, p.wait_limit_ns};

  if (warp < kProducers) {
    // ------------------------------------------------------------ producers
    const int pw = warp;  // issues the stages with kctr % kProducers == pw
    uint32_t kctr = 0, ictr = 0;
    bool ok = true;
    Item it;
    bool have = !p.idle_producers && items.next(it);
    int32_t pid_cur = -2, pid_next = -2;
    if (have) {
      pid_cur = page_ids(p, it, it.t0, lane);
      pid_next = page_ids(p, it, it.t0 + 16, lane);
    }
    while (ok && have) {
      const int32_t r0 = it.r0, rows = it.rows;
      if (pw == 0) {
        // the item's query rows, once every issuer has released the previous item's
        ok = wait_lane0(bar_qempty(sb), (ictr & 1) ^ 1, ctl);
        if (!ok) break;
        if (lane == 0) {
          const uint32_t qbar = bar_qfull(sb);
          ptx::mbar_arrive_expect_tx(qbar, (uint32_t)rows * kQRowBytes);
          ptx::bulk_g2s(sb + OFF_Q, p.q8 + (int64_t)r0 * kQRowBytes, (uint32_t)rows * kQRowBytes, qbar);
          if (!(it.seq >= 0 && (int64_t)it.seq < p.num_seqs)) record_error(p.status, FP4IDX_ERR_BAD_PAGE);
        }
      }
      // The next item and its first page ids are looked up once this warp has issued its
      // first stage of this item (or at its end), so that the switch does not wait on them.
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
          for (int j = lane; j < nx.rows * 64; j += 32) prefetch_l2(p.q8 + (int64_t)nx.r0 * kQRowBytes + j * 128);
          if (lane < 2 * nx.rows) {
            prefetch_l2(reinterpret_cast<const uint8_t*>(p.w + (int64_t)nx.r0 * 64) + lane * 128);
            prefetch_l2(reinterpret_cast<const uint8_t*>(p.q8_scale + (int64_t)nx.r0 * 64) + lane * 128);
          }
          if (lane == 0) prefetch_l2(p.context_lens + nx.r0);
        }
      };
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
        // lane -> (page j of the stage = tile j/2, page j%2 of that tile; chunk c)
        const int j = (lane >> 3) & 3, c = lane & 7;
        int32_t pg = __shfl_sync(kFull, pid_cur, (2 * (i - chunk) + j) & 31);
        const bool needed = j < 2 * tiles && pg != -2;
        const bool valid = pg >= 0 && (int64_t)pg < p.num_pages;
        if (c == 0 && needed && !valid) record_error(p.status, FP4IDX_ERR_BAD_PAGE);
        if (!valid) pg = 0;
        const uint32_t kbar = bar_kfull(sb, s);
        if (lane == 0) ptx::mbar_arrive_expect_tx(kbar, (uint32_t)tiles * kTileBytes);
        __syncwarp();
        const int a = j >> 1, b = j & 1;
        if (a < tiles) {
          tma_load_3d(sb + OFF_K + s * kStageBytes + a * kTileBytes + c * 2048 + b * 1024, &k_map, 16 * c, 0, pg,
                      kbar);
          if (valid && c < 2) prefetch_l2(p.pages + (int64_t)pg * kPageBytes + kScaleOff + c * 128);
        }
        __syncwarp();
        if (!looked) look_ahead();
      }
      ictr++;  // also after a failed stage wait: this item's query copy was issued
      if (!ok) break;
      if (!looked) look_ahead();
      it = nx;
      have = have_nx;
      pid_cur = nx_cur;
      pid_next = nx_next;
    }
    // Tail: every copy a warp issued must land, and (when not aborting) every stage must
    // be released by the MMAs that read it, before the CTA may exit.
    for (uint32_t u = (kctr > (uint32_t)kStages ? kctr - kStages : 0); u < kctr; u++) {
      if ((int)(u % kProducers) != pw) continue;
      wait_lane0(bar_kfull(sb, u % kStages), (u / kStages) & 1, ctl, false);
      if (!*abort_flag) wait_lane0(bar_kempty(sb, u % kStages), (u / kStages) & 1, ctl);
    }
    if (pw == 0 && ictr > 0) {
      wait_lane0(bar_qfull(sb), (ictr - 1) & 1, ctl, false);
      if (!*abort_flag) wait_lane0(bar_qempty(sb), (ictr - 1) & 1, ctl);
    }
  } else if (warp >= kWarpMma && warp < kWarpMma + kMmaWarps) {
    // ------------------------------------------------------------ MMA issuers (lane 0)
    const int mw = warp - kWarpMma;
    if (lane == 0) {
      uint32_t kctr = 0, ictr = 0, ucnt = 0;
      bool ok = true;
      constexpr uint32_t kIdesc = idesc_e4m3(64, 128);
      Item it;
      while (ok && items.next(it)) {
        const int32_t rows = it.rows;
        // The item's query rows are in place.  Waited for even by an issuer with no stage
        // in this item, so that its release below counts toward this item's use of the
        // buffer and not toward the previous one.
        ok = poll(bar_qfull(sb), ictr & 1, ctl, true);
        if (!ok) break;
        ptx::tc_fence_after();
        bool issued = false;
        for (int32_t i = it.t0; i < it.t1 && ok; i += kTilesPerStage, kctr++, ucnt += rows) {
          if ((int)(kctr % kMmaWarps) != mw) continue;
          const int s = kctr % kStages;
          const int tiles = stage_tiles(i, it.t1);
          ok = poll(bar_kfull(sb, s), (kctr / kStages) & 1, ctl, true);
          if (!ok) break;
          ptx::tc_fence_after();
          for (int r = 0; r < rows; r++) {
            const uint32_t u = ucnt + r;
            const int slot = u % kAccSlots;
            ok = wait_count(cnt_slot(sb, slot), (uint32_t)kEpiWarps * (u / kAccSlots), ctl);
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t b0 = sb + OFF_Q + r * kQRowBytes;
            for (int a = 0; a < tiles; a++) {
              const uint32_t a0 = sb + OFF_K + s * kStageBytes + a * kTileBytes;
              const uint32_t d = tmem + slot * 128 + a * 64;
#pragma unroll
              for (int kk = 0; kk < 4; kk++)  // K = 32 e4m3 = chunks 2kk, 2kk + 1
                mma_e4m3(d, ptx::smem_desc(a0 + kk * 4096, 2048, 128), ptx::smem_desc(b0 + kk * 2048, 1024, 128),
                         kIdesc, kk);
            }
            ptx::mma_commit(bar_accfull(sb, slot));
          }
          if (!ok) break;
          ptx::mma_commit(bar_kempty(sb, s));
          issued = true;
        }
        if (!ok) break;
        if (issued)
          ptx::mma_commit(bar_qempty(sb));  // once its MMAs have read the rows
        else
          ptx::mbar_arrive(bar_qempty(sb));
        ictr++;
      }
    }
  } else if (warp >= kWarpEpi0) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - kWarpEpi0;
    const int half = ew >> 2;       // reads tile `half` of every slot use
    const int quad = warp & 3;      // TMEM lanes this warp may read
    const int m = quad * 32 + lane;  // token row of a tile
    const float kNaN = __int_as_float(0x7fc00000);
    int32_t* lsm = reinterpret_cast<int32_t*>(smem + OFF_LEN) + ew * kGroupMax;
    float* wsm = reinterpret_cast<float*>(smem + OFF_WEPI) + ew * kGroupMax * 64;
    uint32_t ucnt = 0;
    bool ok = true;
    Item it;
    while (ok && items.next(it)) {
      const int32_t r0 = it.r0, rows = it.rows;
      const bool seq_ok = it.seq >= 0 && (int64_t)it.seq < p.num_seqs;
      const int32_t span = min(it.maxlen, p.max_context);
      __syncwarp();
      if (lane < rows) {
        int32_t L = __ldg(p.context_lens + r0 + lane);
        if (L < 0 || L > p.max_context) {
          if (ew == 0) record_error(p.status, FP4IDX_ERR_BAD_LENGTH);
          L = L < 0 ? 0 : p.max_context;
        }
        lsm[lane] = L;
      }
      // head weights times the query's head scales, this warp's own copy
      for (int j = lane; j < rows * 16; j += 32) {
        const float4 wv = __ldg(reinterpret_cast<const float4*>(p.w + (int64_t)r0 * 64) + j);
        const float4 sv = __ldg(reinterpret_cast<const float4*>(p.q8_scale + (int64_t)r0 * 64) + j);
        reinterpret_cast<float4*>(wsm)[j] = make_float4(wv.x * sv.x, wv.y * sv.y, wv.z * sv.z, wv.w * sv.w);
      }
      __syncwarp();
      for (int32_t i = it.t0; i < it.t1 && ok; i += kTilesPerStage) {
        const int tiles = stage_tiles(i, it.t1);
        const int a = half;
        const int32_t tok = (i + a) * kTileTokens + m;
        // the token's scale (NaN where its page is missing or out of range)
        float sk = kNaN;
        if (a < tiles && tok < span && seq_ok) {
          const int64_t lp = tok >> 6;
          if (lp < p.max_pages) {
            const int32_t pg = __ldg(p.page_table + (int64_t)it.seq * p.max_pages + lp);
            if (pg >= 0 && (int64_t)pg < p.num_pages)
              sk = __ldg(reinterpret_cast<const float*>(p.pages + (int64_t)pg * kPageBytes + kScaleOff) + (m & 63));
          }
        }
        for (int r = 0; r < rows && ok; r++) {
          const float* wr = wsm + r * 64;
          const int32_t L = lsm[r];
          float* orow = p.out + (int64_t)(r0 + r) * p.out_stride;
          const int slot = ucnt % kAccSlots;
          ok = wait_warp(bar_accfull(sb, slot), (ucnt / kAccSlots) & 1, ctl);
          ucnt++;
          if (!ok) break;
          ptx::tc_fence_after();
          float d[64];
          if (a < tiles) ptx::tmem_ld64_sync(tmem + ((uint32_t)(quad * 32) << 16) + slot * 128 + a * 64, d);
          // released as soon as read, by every epilogue warp (also one with no tile here)
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::smem_add_release(cnt_slot(sb, slot), 1u);
          if (a >= tiles || tok >= L) continue;
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
          orow[tok] = sk * (((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7)));
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kWarpMma) ptx::tmem_dealloc(tmem, kTmemCols);
}

// The fused pages as a 3-D uint8 tensor {128 B, 66 rows, num_pages}; box = 16 B of 64 rows
// of one page.
bool encode_pages(CUtensorMap* map, const uint8_t* pages, int64_t num_pages) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, kPageBytes / 128, (cuuint64_t)num_pages};
  cuuint64_t strides[2] = {128, kPageBytes};
  cuuint32_t box[3] = {16, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(pages), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_logits_fp8(const uint8_t* q8, const float* q8_scale, const float* w, int32_t n_rows,
                              const uint8_t* pages, int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                              int32_t max_pages, const int32_t* context_lens, int32_t max_context,
                              const void* schedule, int32_t num_ctas, float* out, int64_t out_stride,
                              int32_t* status, cudaStream_t stream) {
  const cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(logits_fp8_kernel), kSmemBytes);
  if (e != cudaSuccess) return e;
  if (num_pages < 1 || num_pages > (int64_t)INT32_MAX) return cudaErrorInvalidValue;
  CUtensorMap k_map;
  if (!encode_pages(&k_map, pages, num_pages)) return cudaErrorInvalidValue;
  LogitsFp8Params prm;
  prm.q8 = q8;
  prm.q8_scale = q8_scale;
  prm.w = w;
  prm.pages = pages;
  prm.num_pages = num_pages;
  prm.page_table = page_table;
  prm.num_seqs = num_seqs;
  prm.max_pages = max_pages;
  prm.context_lens = context_lens;
  prm.max_context = max_context;
  prm.n_rows = n_rows;
  prm.schedule = schedule;
  prm.out = out;
  prm.out_stride = out_stride;
  prm.status = status;
  prm.wait_limit_ns = pipeline_wait_limit_ns();
  prm.idle_producers = pipeline_idle_producers() ? 1 : 0;
  logits_fp8_kernel<<<num_ctas, kThreads, kSmemBytes, stream>>>(k_map, prm);
  return cudaGetLastError();
}

}  // namespace fp4idx
