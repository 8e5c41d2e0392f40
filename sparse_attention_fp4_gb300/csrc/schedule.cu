// Length-balanced split of the logits work over the grid: the schedule kernel, one block
// of 1,024 threads running the build of schedule_build.cuh.
#include "launchers.cuh"
#include "schedule_build.cuh"

#include <atomic>

namespace fp4idx {
namespace {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads) build_schedule_kernel(const int32_t* __restrict__ context_lens,
                                                                  const int32_t* __restrict__ row_seq,
                                                                  int32_t n_rows, int32_t num_ctas, void* ws) {
  build_schedule_block<kThreads>(context_lens, row_seq, n_rows, num_ctas, ws);
}

}  // namespace

cudaError_t launch_build_schedule(const int32_t* context_lens, const int32_t* row_seq, int32_t n_rows,
                                  int32_t num_ctas, void* ws, cudaStream_t stream) {
  // no shared-memory needs of its own; the largest carveout keeps the SMs configured for
  // the logits kernel that follows
  static std::atomic<bool> carve_done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !carve_done[dev].load()) {
    e = cudaFuncSetAttribute(build_schedule_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) carve_done[dev].store(true);
  }
  build_schedule_kernel<<<1, kThreads, 0, stream>>>(context_lens, row_seq, n_rows, num_ctas, ws);
  return cudaGetLastError();
}

}  // namespace fp4idx
