// Per-row top-k of the logits, emitted as ascending compressed-token indices: the
// standalone launch of the selection in select.cuh.
//
// [AMD] DeepSeek-V4.1-Flash on MI350X (gfx950) -- Changes: "sorted top-k selection";
// Historical results: the decode top-k is ordered by position, not by KV slot.
// [AMD] Enable FP4 indexer for Deepseek V4 -- Attention runtime: padded rows keep
// context length 0 (their selection is empty: all -1).
//
// One CTA of 1,024 threads per row; when the rows are few (two CTAs per row still fit
// on the GPU), a pair of CTAs per row in a thread-block cluster, each owning half of
// the row's positions; when they are many (more than the SMs), one CTA of 512 threads
// per row, two of them an SM, so that two rows' latency-bound phases overlap.  The two CTAs of a pair exchange only histogram counts, emit
// totals and a short list of boundary keys, through distributed shared memory.  No
// other hand-off between CTAs: a global candidate list, a fence and an arrival counter
// each cost microseconds of latency on this path.
#include "launchers.cuh"
#include "select.cuh"

#include <atomic>

namespace fp4idx {
namespace {

constexpr int kRes = 32768;  // keys a CTA keeps in shared memory

// Dynamic shared memory of the top-k kernel: Select<NT>::smem_words<kC>(res) words.
extern __shared__ __align__(16) uint32_t topk_dyn[];

// kC CTAs (a cluster) of NT threads per row; each owns a contiguous slice of the row's
// groups.  spill + row * sstride holds keys past res (sstride a multiple of 4).
template <int kC, int NT, int kMinBlocks>
__global__ void __launch_bounds__(NT, kMinBlocks)
    topk_row_kernel(const float* __restrict__ logits, int64_t stride, const int32_t* __restrict__ context_lens,
                    int32_t max_context, int32_t k, int32_t res, uint32_t* spill, int64_t sstride,
                    int32_t* __restrict__ out, int32_t* status) {
  using Sel = sel::Select<NT>;
  constexpr int kThreads = NT;
  __shared__ sel::Shared sh;
  const int64_t row = blockIdx.x / kC;
  const int rank = (int)(blockIdx.x % kC);
  const int tid = threadIdx.x;
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
  Sel::template row<kC, false>(logits + row * stride, L, k, o, spill + row * sstride, res, topk_dyn, sh, rank,
                               status);
}

inline int64_t spill_stride(int32_t max_context) {
  return max((int64_t)0, ((int64_t)max(max_context, 1) + 3) / 4 * 4 - kRes);
}
inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

std::atomic<int> g_sms[64];

// Shared memory of a kC-CTA launch of NT threads with `res` keys a CTA.
template <int kC, int NT>
constexpr size_t smem_bytes(int32_t res) {
  return (size_t)sel::Select<NT>::template smem_words<kC>(res) * sizeof(uint32_t);
}

template <int kC, int NT, int kMinBlocks>
cudaError_t launch_rows(const float* logits, int64_t stride, const int32_t* context_lens, int32_t n_rows,
                        int32_t max_context, int32_t k, void* workspace, int32_t* out, int32_t* status,
                        cudaStream_t stream) {
  const void* fn = reinterpret_cast<const void*>(topk_row_kernel<kC, NT, kMinBlocks>);
  const cudaError_t e = set_smem_attr_once(fn, smem_bytes<kC, NT>(kRes));
  if (e != cudaSuccess) return e;
  // keys a CTA holds: its slice of the longest row, rounded to groups of four
  const int64_t groups = ((int64_t)max(max_context, 1) + 3) / 4;
  const int32_t res = (int32_t)min((int64_t)kRes, 4 * ((groups + kC - 1) / kC));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_rows * kC);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem_bytes<kC, NT>(res);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kC > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, topk_row_kernel<kC, NT, kMinBlocks>, logits, stride, context_lens, max_context, k,
                            res, reinterpret_cast<uint32_t*>(workspace), spill_stride(max_context), out, status);
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
  // Few long rows leave most SMs idle: then each row goes to a pair of CTAs (a cluster),
  // which halves the passes over its keys.  For short rows the pair's cluster launch and
  // exchanges cost more than they save (one row of 4,096: 10.2 us a launch alone against
  // 12.3 us as a pair).  Many rows queue on the SMs: then two CTAs of 512 threads an SM
  // overlap two rows' barrier- and latency-bound phases.
  constexpr int32_t kPairMinContext = 8192;
  if (2 * (int64_t)n_rows <= sms && max_context > kPairMinContext)
    return launch_rows<2, 1024, 1>(logits, stride, context_lens, n_rows, max_context, k, workspace, out, status,
                                   stream);
  if ((int64_t)n_rows > sms)
    return launch_rows<1, 512, 2>(logits, stride, context_lens, n_rows, max_context, k, workspace, out, status,
                                  stream);
  return launch_rows<1, 1024, 1>(logits, stride, context_lens, n_rows, max_context, k, workspace, out, status,
                                 stream);
}

}  // namespace fp4idx
