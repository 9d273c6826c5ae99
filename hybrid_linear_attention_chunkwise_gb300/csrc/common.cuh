// common.cuh -- small device helpers shared by the libhypic kernels.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "internal.h"

namespace hypic {

__device__ __forceinline__ float load_in(const void *p, int64_t i, int in_dtype) {
  if (in_dtype == HYPIC_IN_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
  return static_cast<const float *>(p)[i];
}

__device__ __forceinline__ void report(uint32_t *status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ bool finite_f(float x) { return isfinite(x); }

}  // namespace hypic
