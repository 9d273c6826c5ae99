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

// The next plan item for this CTA (called by the one thread that fetches the
// CTA's items; `taken` counts its fetches): the shared ticket for an LPT
// plan, the static round-robin sequence blockIdx.x + k * gridDim.x otherwise.
__device__ __forceinline__ int take_item(PlanHeader *plan, int &taken) {
  if (plan->mode == PLAN_ROUND_ROBIN) return (int)blockIdx.x + (int)gridDim.x * taken++;
  return atomicAdd(&plan->ticket, 1);
}

}  // namespace hypic
