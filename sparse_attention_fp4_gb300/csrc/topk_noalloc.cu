// fp4idx_topk_noalloc: the top-k selection of fp4idx_topk with its scratch in
// a fixed array of this library's own device memory instead of a caller's workspace.
//
// It exists for callers that may not allocate device memory at the point where they
// select.  One kind is a serving runtime that hands its whole memory budget to its own
// pool at start-up: a cudaMalloc from a library would then fail or squeeze the pool,
// and it also synchronises the device, stalling every stream in flight.  Another is a
// plug-in host that gives a library only a stream and the tensors of the call, with no
// way to pass it extra memory.  Such callers get a bounded scratch that lives as long as
// the library's device code is loaded on the device and is never resized.
//
// The array: FP4IDX_TOPK_NOALLOC_MAX_BYTES bytes per device, 256-byte aligned.  A call
// fits when fp4idx_topk_workspace_bytes(n_rows, max_context) is at most that; a larger
// one is refused with FP4IDX_ERR_SCRATCH_LIMIT and nothing is enqueued.
//
// Setup: the first valid call on each device, with that device current, looks up the
// array's device address once (cudaGetSymbolAddress) and keeps it for later calls on the
// same device.  Under CUDA's lazy module loading (the default), that lookup is also what
// loads this file's device code on the device and so commits the array's memory there:
// it can fail for lack of memory, and it may synchronise.  So make that first call at
// start-up, before a memory pool reserves the device's memory and before any stream
// capture begins; a call with n_rows = 0 does the set-up and nothing else.  The address
// is kept for the life of the process: after cudaDeviceReset (or anything else that
// destroys the device's primary context) it is stale, and this entry point must not be
// used on that device again in the same process.
//
// Zero state: nothing in the array needs to start at zero.  A row's sort keys go there
// only for positions past what shared memory holds, and each call reads back only the
// keys it wrote itself.  So no call clears the array.
//
// Every call on a device uses the same array.  Calls whose kernels may overlap (on
// streams with no ordering between them, or from host threads at once) race on it and
// corrupt each other's keys; order such calls on one stream.
#include <mutex>

#include "launchers.cuh"

static __device__ __align__(256) unsigned char g_topk_noalloc_scratch[FP4IDX_TOPK_NOALLOC_MAX_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device (looked up once per device).
int current_device_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FP4IDX_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return FP4IDX_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_topk_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();  // do not leave the error for the next launch check to find
      return FP4IDX_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FP4IDX_OK;
}

inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" int fp4idx_topk_noalloc(const float* logits, int64_t logits_stride, const int32_t* context_lens,
                                   int64_t n_rows, int32_t max_context, int32_t k, int32_t* topk_idx,
                                   int32_t* status_dev, void* stream) {
  // every argument check comes before the first CUDA call, so a bad call is reported as
  // such and never triggers the set-up
  if (n_rows < 0 || n_rows > INT32_MAX - 1 || max_context < 0 || k < 1 || k > FP4IDX_MAX_TOPK)
    return FP4IDX_ERR_INVALID_ARG;
  if (max_context > FP4IDX_MAX_CONTEXT) return FP4IDX_ERR_UNSUPPORTED;
  if (fp4idx::topk_workspace_bytes(n_rows, max_context) > (size_t)FP4IDX_TOPK_NOALLOC_MAX_BYTES)
    return FP4IDX_ERR_SCRATCH_LIMIT;
  if (n_rows > 0) {
    if (!logits || !context_lens || !topk_idx || !aligned4(logits) || !aligned4(context_lens) ||
        !aligned4(topk_idx) || logits_stride < max_context)
      return FP4IDX_ERR_INVALID_ARG;
    if (status_dev && !aligned4(status_dev)) return FP4IDX_ERR_INVALID_ARG;
  }
  // an n_rows = 0 call does the set-up and nothing else
  void* scratch = nullptr;
  const int rc = current_device_scratch(&scratch);
  if (rc != FP4IDX_OK) return rc;
  if (n_rows == 0) return FP4IDX_OK;
  const cudaError_t e = fp4idx::launch_topk(logits, logits_stride, context_lens, (int32_t)n_rows, max_context, k,
                                            scratch, topk_idx, status_dev, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP4IDX_OK : FP4IDX_ERR_CUDA;
}
