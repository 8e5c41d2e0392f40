// Host helpers shared by the launchers: the tensor-map encoder, per-device kernel
// attributes, and the pipeline-wait settings (including the test switch that makes a
// wait run out on purpose).
#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <set>
#include <utility>

#include "launchers.cuh"

namespace fp4idx {

EncodeTiledFn encode_tiled_fn() {
  // looked up once through the runtime (no libcuda link); thread-safe initialisation
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

bool encode_rows(CUtensorMap* map, const void* base, int64_t rows, uint32_t row_bytes) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 8), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {row_bytes / 8, 1};
  cuuint32_t es[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t set_smem_attr_once(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done.insert({kernel, dev});
  return e;
}

cudaError_t resident_ctas(const void* kernel, int threads, size_t smem, int* out) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> known;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto it = known.find({kernel, dev});
  if (it != known.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  int per_sm = 0, sms = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  *out = std::max(1, per_sm) * sms;
  known[{kernel, dev}] = *out;
  return cudaSuccess;
}

namespace {
std::atomic<int64_t> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int32_t> g_idle_producers{0};
}  // namespace

uint64_t pipeline_wait_limit_ns() { return (uint64_t)g_wait_limit_ns.load(); }
bool pipeline_idle_producers() { return g_idle_producers.load() != 0; }

}  // namespace fp4idx

extern "C" int fp4idx_test_pipeline_waits(int32_t idle_producers, int64_t wait_limit_ns) {
  if (wait_limit_ns < 0) return FP4IDX_ERR_INVALID_ARG;
  fp4idx::g_wait_limit_ns.store(wait_limit_ns == 0 ? fp4idx::kDefaultWaitLimitNs : wait_limit_ns);
  fp4idx::g_idle_producers.store(idle_producers ? 1 : 0);
  return FP4IDX_OK;
}
