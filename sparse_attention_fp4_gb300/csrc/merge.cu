// Merge of per-shard top-k selections into a row's top-k (the exchange step of a
// context-parallel indexer).
//
// [AMD] DeepSeek-V4.1-Flash on MI350X (gfx950) -- the context-parallel runs shard one
// long sequence's compressed tokens over GPUs; each shard scores its token range and
// keeps its own top-k, and the row's selection is the top-k of the gathered (value,
// index) candidates.  Every token of the row's top-k is in its shard's top-k (anything
// that ranks above it inside the shard also ranks above it in the row), ties included
// when both use the lower-position rule, so the merge is exact.
//
// Candidates of a row arrive as n_shards lists of k (value, global index) pairs, each
// list ascending in index with -1 padding at its end, the shards in ascending position
// order.  The merge compacts the valid pairs of a row in shard order -- which is then
// global position order -- selects the k largest values of the compacted row with the
// top-k kernel (ties to the lower slot, i.e. the lower position), and maps the selected
// slots back to global indices, ascending.
#include "launchers.cuh"

namespace fp4idx {
namespace {

constexpr int kMergeThreads = 256;

// values[t][i] = logits[t][idx[t][i]] for idx >= 0 (idx < context_lens[t] < stride),
// -inf for padding.
__global__ void __launch_bounds__(kMergeThreads) gather_values_kernel(const float* __restrict__ logits, int64_t stride,
                                                                      const int32_t* __restrict__ idx, int32_t k,
                                                                      float* __restrict__ values) {
  const int64_t t = blockIdx.y;
  for (int i = blockIdx.x * kMergeThreads + threadIdx.x; i < k; i += gridDim.x * kMergeThreads) {
    const int32_t s = __ldg(idx + t * k + i);
    values[t * k + i] = s >= 0 && (int64_t)s < stride ? __ldg(logits + t * stride + s) : -INFINITY;
  }
}

// One CTA per row: the valid count of each shard's list (its entries up to the first -1),
// their prefix, and the row's valid pairs packed in shard order into cv/ci; count[t] =
// the row's total.
__global__ void __launch_bounds__(kMergeThreads) compact_kernel(const float* __restrict__ cand_values,
                                                                const int32_t* __restrict__ cand_idx,
                                                                int32_t n_shards, int32_t k, float* __restrict__ cv,
                                                                int32_t* __restrict__ ci, int32_t* __restrict__ count) {
  extern __shared__ int32_t valid[];  // [n_shards + 1]: valid counts, then exclusive prefix
  const int64_t t = blockIdx.x;
  const int64_t row = t * (int64_t)n_shards * k;
  for (int s = threadIdx.x; s < n_shards; s += kMergeThreads) {
    // entries >= 0 form a prefix of the list: binary search for its length
    const int32_t* l = cand_idx + row + (int64_t)s * k;
    int a = 0, b = k;
    while (a < b) {
      const int m = (a + b) >> 1;
      if (__ldg(l + m) >= 0) a = m + 1;
      else b = m;
    }
    valid[s] = a;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int s = 0; s < n_shards; s++) {
      const int v = valid[s];
      valid[s] = run;
      run += v;
    }
    valid[n_shards] = run;
    count[t] = run;
  }
  __syncthreads();
  const int64_t out = t * (int64_t)n_shards * k;
  for (int s = 0; s < n_shards; s++) {
    const int off = valid[s], n = valid[s + 1] - off;
    for (int i = threadIdx.x; i < n; i += kMergeThreads) {
      cv[out + off + i] = __ldg(cand_values + row + (int64_t)s * k + i);
      ci[out + off + i] = __ldg(cand_idx + row + (int64_t)s * k + i);
    }
  }
}

// topk_idx[t][i] = ci[t][slot[t][i]] for slot >= 0, else -1.
__global__ void __launch_bounds__(kMergeThreads) map_slots_kernel(const int32_t* __restrict__ slot,
                                                                  const int32_t* __restrict__ ci, int64_t ci_stride,
                                                                  int32_t k, int32_t* __restrict__ topk_idx) {
  const int64_t t = blockIdx.y;
  for (int i = blockIdx.x * kMergeThreads + threadIdx.x; i < k; i += gridDim.x * kMergeThreads) {
    const int32_t s = __ldg(slot + t * k + i);
    topk_idx[t * k + i] = s >= 0 ? __ldg(ci + t * ci_stride + s) : -1;
  }
}

inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

size_t merge_workspace_bytes(int64_t n_rows, int32_t n_shards, int32_t k) {
  const size_t nc = (size_t)n_rows * (size_t)n_shards * (size_t)k;
  return align256(nc * sizeof(float)) + align256(nc * sizeof(int32_t)) + align256((size_t)n_rows * sizeof(int32_t)) +
         align256((size_t)n_rows * (size_t)k * sizeof(int32_t)) +
         topk_workspace_bytes(n_rows, (int32_t)((int64_t)n_shards * k));
}

cudaError_t launch_gather_values(const float* logits, int64_t stride, const int32_t* idx, int32_t n_rows, int32_t k,
                                 float* values, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  const dim3 grid((unsigned)((k + kMergeThreads - 1) / kMergeThreads), (unsigned)n_rows);
  gather_values_kernel<<<grid, kMergeThreads, 0, stream>>>(logits, stride, idx, k, values);
  return cudaGetLastError();
}

cudaError_t launch_topk_merge(const float* cand_values, const int32_t* cand_idx, int32_t n_rows, int32_t n_shards,
                              int32_t k, void* workspace, int32_t* topk_idx, int32_t* status, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  const int64_t width = (int64_t)n_shards * k;
  const size_t nc = (size_t)n_rows * (size_t)width;
  uint8_t* w = reinterpret_cast<uint8_t*>(workspace);
  float* cv = reinterpret_cast<float*>(w);
  w += align256(nc * sizeof(float));
  int32_t* ci = reinterpret_cast<int32_t*>(w);
  w += align256(nc * sizeof(int32_t));
  int32_t* count = reinterpret_cast<int32_t*>(w);
  w += align256((size_t)n_rows * sizeof(int32_t));
  int32_t* slot = reinterpret_cast<int32_t*>(w);
  w += align256((size_t)n_rows * (size_t)k * sizeof(int32_t));
  compact_kernel<<<(unsigned)n_rows, kMergeThreads, (size_t)(n_shards + 1) * sizeof(int32_t), stream>>>(
      cand_values, cand_idx, n_shards, k, cv, ci, count);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_topk(cv, width, count, n_rows, (int32_t)width, k, w, slot, status, stream);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((k + kMergeThreads - 1) / kMergeThreads), (unsigned)n_rows);
  map_slots_kernel<<<grid, kMergeThreads, 0, stream>>>(slot, ci, width, k, topk_idx);
  return cudaGetLastError();
}

}  // namespace fp4idx
