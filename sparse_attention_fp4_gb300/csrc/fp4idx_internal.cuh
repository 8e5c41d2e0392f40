// Constants and device helpers shared by the kernels of libfp4idx.so (the host launchers
// are declared in launchers.cuh).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp4idx.h"

namespace fp4idx {

constexpr int kHeadDim = 128;
constexpr int kHeads = 64;
constexpr int kPage = 64;
constexpr int kRope = 64;

// First data-dependent error wins; never traps.
__device__ __forceinline__ void record_error(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

}  // namespace fp4idx
