// build_noalloc.cu -- hypic_segment_build_noalloc: the segment build for
// callers that cannot allocate device memory.  The work plan (header with the
// dynamic ticket, then one item per (segment, value head)) lives in a fixed
// file-scope device array instead of a caller workspace; the host side uses
// fixed static buffers, so the call allocates nothing on the device or the
// heap.  The checks and the plan are the ones hypic_segment_build runs
// (check_build_*, fill_build_plan), so both entry points accept the same
// calls and plan them identically.
//
// The array is shared by every call in the process: calls that overlap on
// the GPU (different streams without ordering between them) race on it.
// Calls on one stream, or ordered by events, are safe, since the plan copy
// that opens each call is stream-ordered after the previous call's kernel.
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"

using namespace hypic;

namespace {

constexpr size_t kScratchBytes = (size_t)HYPIC_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The plan at the stated maximum number of pairs fills the array exactly.
static_assert(sizeof(PlanHeader) + (size_t)HYPIC_NOALLOC_MAX_PAIRS * sizeof(BuildItem) <= kScratchBytes,
              "pair limit does not fit the fixed scratch");
static_assert(sizeof(PlanHeader) + ((size_t)HYPIC_NOALLOC_MAX_PAIRS + 1) * sizeof(BuildItem) > kScratchBytes,
              "pair limit leaves a whole item of the fixed scratch unused");

// The fixed device scratch (one copy per device, from this module's load).
static __device__ __align__(256) unsigned char g_plan_scratch[kScratchBytes];

// Host staging of the plan and of the slot check; guarded by g_mu.
alignas(256) static unsigned char h_plan[kScratchBytes];
static int32_t h_slots[HYPIC_NOALLOC_MAX_PAIRS];
static void *g_dev_scratch[kMaxDevices];
static std::mutex g_mu;

// Device address of the scratch on the current device, looked up once per
// device with that device current.
int scratch_ptr(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HYPIC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return HYPIC_ERR_UNSUPPORTED;
  if (!g_dev_scratch[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || !p) return HYPIC_ERR_CUDA;
    g_dev_scratch[dev] = p;
  }
  *out = g_dev_scratch[dev];
  return HYPIC_OK;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

}  // namespace

extern "C" {

int hypic_segment_build_noalloc(const hypic_build_desc *d, hypic_stream_t stream) {
  int st = check_build_shapes(d);
  if (st) return st;
  // the size limit is checked before any CUDA call
  if ((int64_t)d->n_seg * d->h_v > HYPIC_NOALLOC_MAX_PAIRS) return HYPIC_ERR_WORKSPACE;
  if (d->n_seg == 0) return HYPIC_OK;
  if ((st = check_build_pointers(d))) return st;
  BuildParams p = build_params(d);
  const int path = build_path(p, d->n_tokens);
  if ((d->flags & HYPIC_FLAG_REQUIRE_TENSOR_CORES) && d->n_tokens > 0 && path == HYPIC_PATH_F32_TOKEN)
    return HYPIC_ERR_UNSUPPORTED;

  std::lock_guard<std::mutex> lock(g_mu);
  if ((st = check_build_slots(d, h_slots))) return st;
  void *scratch = nullptr;
  if ((st = scratch_ptr(&scratch))) return st;
  p.plan = reinterpret_cast<PlanHeader *>(scratch);
  p.items = reinterpret_cast<const BuildItem *>(p.plan + 1);
  // one item per (segment, value head); the ticket starts at zero
  const int64_t n_items = fill_build_plan(d, h_plan);
  if (n_items == 0) return HYPIC_OK;
  const size_t bytes = build_plan_size(n_items);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // pageable source: the call returns once the bytes are staged, so the
  // static buffer may be rewritten by the next call
  if (cudaMemcpyAsync(scratch, h_plan, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return HYPIC_ERR_CUDA;
  if (launch_build(p, d->n_tokens, (int)n_items, sm_count(), s) != cudaSuccess) return HYPIC_ERR_CUDA;
  return HYPIC_OK;
}

}  // extern "C"
