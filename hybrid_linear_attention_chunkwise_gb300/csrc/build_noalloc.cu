// build_noalloc.cu -- hypic_segment_build_noalloc: the segment build for
// callers that cannot allocate device memory.  The work plan (header with the
// dynamic ticket, then the LPT-ordered items) lives in a fixed file-scope
// device array instead of a caller workspace; the host side uses fixed
// static buffers, so the call allocates nothing on the device or the heap.
//
// The array is shared by every call in the process: calls that overlap on
// the GPU (different streams without ordering between them) race on it.
// Calls on one stream, or ordered by events, are safe, since the plan copy
// that opens each call is stream-ordered after the previous call's kernel.
#include <algorithm>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"

using namespace hypic;

namespace {

constexpr size_t kScratchBytes = (size_t)HYPIC_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Plan header + up to two items per (segment, head) pair fit the array at
// the stated maximum number of pairs.
static_assert(sizeof(PlanHeader) + 2 * (size_t)HYPIC_NOALLOC_MAX_PAIRS * sizeof(BuildItem) <= kScratchBytes,
              "pair limit does not fit the fixed scratch");

// The fixed device scratch (one copy per device, from this module's load).
static __device__ __align__(256) unsigned char g_plan_scratch[kScratchBytes];

// Host staging of the plan and of the slot check; guarded by g_mu.
alignas(256) static unsigned char h_plan[kScratchBytes];
static int32_t h_slots[HYPIC_NOALLOC_MAX_PAIRS];
static void *g_dev_scratch[kMaxDevices];
static std::mutex g_mu;

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shapes(const hypic_build_desc *d) {
  if (d->h_k < 1 || d->h_v < 1 || d->d_k < 1 || d->d_v < 1 || d->seam_w < 0) return HYPIC_ERR_INVALID_ARG;
  if (d->h_v % d->h_k != 0) return HYPIC_ERR_INVALID_ARG;
  if (d->variant < HYPIC_GDN || d->variant > HYPIC_DIAG_GATE) return HYPIC_ERR_INVALID_ARG;
  if (d->in_dtype != HYPIC_IN_BF16 && d->in_dtype != HYPIC_IN_F32) return HYPIC_ERR_INVALID_ARG;
  if (d->d_k > 128 || d->d_v > 128) return HYPIC_ERR_UNSUPPORTED;
  if (d->n_tokens < 0 || d->n_seg < 0 || d->n_slots < 0) return HYPIC_ERR_INVALID_ARG;
  if (!d->seg_offsets) return HYPIC_ERR_INVALID_ARG;
  if (d->seg_offsets[0] != 0 || d->seg_offsets[d->n_seg] != d->n_tokens) return HYPIC_ERR_INVALID_ARG;
  for (int i = 0; i < d->n_seg; i++)
    if (d->seg_offsets[i + 1] < d->seg_offsets[i]) return HYPIC_ERR_INVALID_ARG;
  return HYPIC_OK;
}

int check_pointers(const hypic_build_desc *d) {
  const int esz = d->in_dtype == HYPIC_IN_BF16 ? 2 : 4;
  if (d->n_tokens > 0) {
    if (!d->k || !d->v || !aligned(d->k, esz) || !aligned(d->v, esz)) return HYPIC_ERR_INVALID_ARG;
  }
  const bool needs_g = d->variant == HYPIC_GDN || d->variant == HYPIC_CHANNEL_DELTA ||
                       d->variant == HYPIC_DIAG_GATE || d->variant == HYPIC_SCALAR_DECAY;
  if (needs_g && (!d->g || !aligned(d->g, 4))) return HYPIC_ERR_INVALID_ARG;
  if (is_delta(d->variant) && d->n_tokens > 0 && (!d->beta || !aligned(d->beta, 4))) return HYPIC_ERR_INVALID_ARG;
  if (!d->T_pool || !d->S_pool || !aligned(d->T_pool, 4) || !aligned(d->S_pool, 4)) return HYPIC_ERR_INVALID_ARG;
  return HYPIC_OK;
}

// Slots in range and distinct (two items writing one slot would race); sorts
// a copy in the static buffer.
int check_slots(const hypic_build_desc *d) {
  for (int i = 0; i < d->n_seg; i++) h_slots[i] = d->slot_of_seg ? d->slot_of_seg[i] : i;
  std::sort(h_slots, h_slots + d->n_seg);
  for (int i = 0; i < d->n_seg; i++) {
    if (h_slots[i] < 0 || h_slots[i] >= d->n_slots) return HYPIC_ERR_INVALID_ARG;
    if (i && h_slots[i] == h_slots[i - 1]) return HYPIC_ERR_INVALID_ARG;
  }
  return HYPIC_OK;
}

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
  if (!d) return HYPIC_ERR_INVALID_ARG;
  int st = check_shapes(d);
  if (st) return st;
  // the size limit is checked before any CUDA call
  if ((int64_t)d->n_seg * d->h_v > HYPIC_NOALLOC_MAX_PAIRS) return HYPIC_ERR_WORKSPACE;
  if (d->n_seg == 0) return HYPIC_OK;
  if ((st = check_pointers(d))) return st;

  std::lock_guard<std::mutex> lock(g_mu);
  if ((st = check_slots(d))) return st;
  void *scratch = nullptr;
  if ((st = scratch_ptr(&scratch))) return st;

  BuildParams p{};
  p.h_k = d->h_k;
  p.h_v = d->h_v;
  p.d_k = d->d_k;
  p.d_v = d->d_v;
  p.variant = d->variant;
  p.in_dtype = d->in_dtype;
  p.flags = d->flags;
  p.n_slots = d->n_slots;
  p.k = d->k;
  p.v = d->v;
  p.g = d->g;
  p.beta = d->beta;
  p.T_pool = d->T_pool;
  p.S_pool = d->S_pool;
  p.plan = reinterpret_cast<PlanHeader *>(scratch);
  p.items = reinterpret_cast<const BuildItem *>(p.plan + 1);
  p.status = d->status;
  const int parts = 1;  // one item per (segment, value head) on every kernel
  const int64_t n_items = (int64_t)d->n_seg * d->h_v * parts;

  // Plan in the static host buffer: the ticket starts at zero, items go
  // longest body first (ties: lower segment, head, part first), the order the
  // LPT rule hands them out in.
  const size_t bytes = sizeof(PlanHeader) + (size_t)n_items * sizeof(BuildItem);
  PlanHeader *hdr = reinterpret_cast<PlanHeader *>(h_plan);
  std::memset(hdr, 0, sizeof(PlanHeader));
  hdr->ticket = 0;
  hdr->n_items = (int32_t)n_items;
  BuildItem *items = reinterpret_cast<BuildItem *>(hdr + 1);
  int64_t r = 0;
  for (int i = 0; i < d->n_seg; i++) {
    const int64_t start = std::min(d->seg_offsets[i] + d->seam_w, d->seg_offsets[i + 1]);
    const int32_t slot = d->slot_of_seg ? d->slot_of_seg[i] : i;
    for (int h = 0; h < d->h_v; h++)
      for (int part = 0; part < parts; part++) {
        BuildItem b;
        b.seg = i;
        b.head = h;
        b.slot = slot;
        b.part = part;
        b.start = start;
        b.end = d->seg_offsets[i + 1];
        items[r++] = b;
      }
  }
  std::sort(items, items + n_items, [](const BuildItem &a, const BuildItem &b) {
    const int64_t ca = a.end - a.start, cb = b.end - b.start;
    if (ca != cb) return ca > cb;
    if (a.seg != b.seg) return a.seg < b.seg;
    if (a.head != b.head) return a.head < b.head;
    return a.part < b.part;
  });

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // pageable source: the call returns once the bytes are staged, so the
  // static buffer may be rewritten by the next call
  if (cudaMemcpyAsync(scratch, h_plan, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return HYPIC_ERR_CUDA;
  if (launch_build(p, d->n_tokens, (int)n_items, sm_count(), s) != cudaSuccess) return HYPIC_ERR_CUDA;
  return HYPIC_OK;
}

}  // extern "C"
