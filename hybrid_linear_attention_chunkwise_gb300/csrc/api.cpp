// api.cpp -- host side of libhypic: descriptor validation, the LPT work plan,
// workspace sizing and kernel launches behind the C ABI of hypic.h.
#include <algorithm>
#include <mutex>
#include <cstdlib>
#include <cstring>
#include <numeric>
#include <queue>
#include <vector>

#include <cuda_runtime.h>

#include "internal.h"

using namespace hypic;

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int in_size(int dt) { return dt == HYPIC_IN_BF16 ? 2 : 4; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

int check_common_shapes(int h_k, int h_v, int d_k, int d_v, int seam_w, int variant, int in_dtype) {
  if (h_k < 1 || h_v < 1 || d_k < 1 || d_v < 1 || seam_w < 0) return HYPIC_ERR_INVALID_ARG;
  if (h_v % h_k != 0) return HYPIC_ERR_INVALID_ARG;
  if (variant < HYPIC_GDN || variant > HYPIC_DIAG_GATE) return HYPIC_ERR_INVALID_ARG;
  if (in_dtype != HYPIC_IN_BF16 && in_dtype != HYPIC_IN_F32) return HYPIC_ERR_INVALID_ARG;
  if (d_k > 128 || d_v > 128) return HYPIC_ERR_UNSUPPORTED;
  return HYPIC_OK;
}

int64_t n_build_items(const hypic_build_desc *d) { return (int64_t)d->n_seg * d->h_v; }


}  // namespace

namespace hypic {
uint32_t wait_limit() {
  // default: ~2^24 polls of try_wait (seconds); the debug override lets a
  // test make a wait run out on purpose
  static const uint32_t lim = [] {
    const char *e = std::getenv("HYPIC_DEBUG_WAIT_LIMIT");
    if (e && *e) {
      long v = std::strtol(e, nullptr, 10);
      if (v >= 1) return (uint32_t)v;
    }
    return (uint32_t)(1u << 24);
  }();
  return lim;
}

bool debug_stall() {
  static const bool on = [] {
    const char *e = std::getenv("HYPIC_DEBUG_STALL");
    return e && e[0] == '1';
  }();
  return on;
}
}  // namespace hypic

namespace hypic {

// The build kernel for the call: bf16 inputs with 128-wide heads run
// chunkwise on the tensor cores (scalar-gate delta rules, the per-channel
// gated delta rule, and the fast path of the transitions without an erase:
// scalar decay, ungated, diagonal gate); every other case runs the fp32 token
// recurrence.
int build_path(const BuildParams &p, int64_t n_tokens) {
  // no tokens at all: every pair is (I, 0) (or the empty gate product), which
  // the token kernel writes without reading an input; the tensor-core
  // kernels cannot describe an empty token tensor
  if (n_tokens == 0) return HYPIC_PATH_F32_TOKEN;
  if (build_tc_supported(p)) return HYPIC_PATH_TC_CHUNKWISE;
  if (build_channel_supported(p)) return HYPIC_PATH_TC_CHANNEL;
  if (build_fast_supported(p)) return HYPIC_PATH_TC_FAST;
  return HYPIC_PATH_F32_TOKEN;
}

cudaError_t launch_build(const BuildParams &p, int64_t n_tokens, int n_items, int n_sm, cudaStream_t s) {
  switch (build_path(p, n_tokens)) {
    case HYPIC_PATH_TC_CHUNKWISE: return launch_build_tc(p, n_tokens, n_items, n_sm, wait_limit(), s);
    case HYPIC_PATH_TC_CHANNEL: return launch_build_channel(p, n_tokens, n_items, n_sm, wait_limit(), s);
    case HYPIC_PATH_TC_FAST: return launch_build_fast(p, n_tokens, n_items, n_sm, wait_limit(), s);
    default: return launch_build_token(p, n_items, n_sm, s);
  }
}

// ---- build descriptors: the checks and the plan every build entry point
// shares (no heap use, so that the allocation-free entry point runs them too)
int check_build_shapes(const hypic_build_desc *d) {
  if (!d) return HYPIC_ERR_INVALID_ARG;
  int st = check_common_shapes(d->h_k, d->h_v, d->d_k, d->d_v, d->seam_w, d->variant, d->in_dtype);
  if (st) return st;
  if (d->n_tokens < 0 || d->n_seg < 0 || d->n_slots < 0) return HYPIC_ERR_INVALID_ARG;
  if (!d->seg_offsets) return HYPIC_ERR_INVALID_ARG;
  if (d->seg_offsets[0] != 0 || d->seg_offsets[d->n_seg] != d->n_tokens) return HYPIC_ERR_INVALID_ARG;
  for (int i = 0; i < d->n_seg; i++)
    if (d->seg_offsets[i + 1] < d->seg_offsets[i]) return HYPIC_ERR_INVALID_ARG;
  if (d->flags & ~(HYPIC_FLAG_CHECK_FINITE | HYPIC_FLAG_ROUND_ROBIN | HYPIC_FLAG_REQUIRE_TENSOR_CORES))
    return HYPIC_ERR_INVALID_ARG;
  if (n_build_items(d) > INT32_MAX / 2) return HYPIC_ERR_UNSUPPORTED;
  return HYPIC_OK;
}

int check_build_pointers(const hypic_build_desc *d) {
  const int esz = in_size(d->in_dtype);
  if (d->n_tokens > 0) {
    if (!d->k || !d->v || !aligned(d->k, esz) || !aligned(d->v, esz)) return HYPIC_ERR_INVALID_ARG;
  }
  const bool delta = is_delta(d->variant);
  const bool needs_g = d->variant == HYPIC_GDN || d->variant == HYPIC_CHANNEL_DELTA ||
                       d->variant == HYPIC_DIAG_GATE || d->variant == HYPIC_SCALAR_DECAY;
  // per-token log-gates are read only when there are tokens; the per-head
  // decay always
  const bool reads_g = needs_g && (d->n_tokens > 0 || d->variant == HYPIC_SCALAR_DECAY);
  if (reads_g && (!d->g || !aligned(d->g, 4))) return HYPIC_ERR_INVALID_ARG;
  if (delta && d->n_tokens > 0 && (!d->beta || !aligned(d->beta, 4))) return HYPIC_ERR_INVALID_ARG;
  if (!d->T_pool || !d->S_pool || !aligned(d->T_pool, 4) || !aligned(d->S_pool, 4)) return HYPIC_ERR_INVALID_ARG;
  return HYPIC_OK;
}

int check_build_slots(const hypic_build_desc *d, int32_t *sorted) {
  for (int i = 0; i < d->n_seg; i++) sorted[i] = d->slot_of_seg ? d->slot_of_seg[i] : i;
  std::sort(sorted, sorted + d->n_seg);
  for (int i = 0; i < d->n_seg; i++) {
    if (sorted[i] == HYPIC_SLOT_SKIP) continue;  // segment not built
    if (sorted[i] < 0 || sorted[i] >= d->n_slots) return HYPIC_ERR_INVALID_ARG;
    if (i && sorted[i] == sorted[i - 1]) return HYPIC_ERR_INVALID_ARG;  // two items writing one slot would race
  }
  return HYPIC_OK;
}

size_t build_plan_size(int64_t n_items) { return sizeof(PlanHeader) + (size_t)n_items * sizeof(BuildItem); }

int64_t fill_build_plan(const hypic_build_desc *d, void *plan) {
  PlanHeader *hdr = static_cast<PlanHeader *>(plan);
  std::memset(hdr, 0, sizeof(PlanHeader));
  const bool rr = (d->flags & HYPIC_FLAG_ROUND_ROBIN) != 0;
  hdr->mode = rr ? PLAN_ROUND_ROBIN : PLAN_LPT;
  BuildItem *items = reinterpret_cast<BuildItem *>(hdr + 1);
  int64_t r = 0;
  for (int i = 0; i < d->n_seg; i++) {
    BuildItem b;
    b.seg = i;
    b.slot = d->slot_of_seg ? d->slot_of_seg[i] : i;
    if (b.slot == HYPIC_SLOT_SKIP) continue;
    b.part = 0;
    b.start = std::min(d->seg_offsets[i] + d->seam_w, d->seg_offsets[i + 1]);
    b.end = d->seg_offsets[i + 1];
    for (int h = 0; h < d->h_v; h++) {
      b.head = h;
      items[r++] = b;
    }
  }
  const int64_t n_items = r;
  hdr->n_items = (int32_t)n_items;
  if (rr) return n_items;  // index order: segment-major, head-minor
  // LPT: longest body first; ties in index order (a total order, so the
  // in-place sort is deterministic)
  std::sort(items, items + n_items, [](const BuildItem &a, const BuildItem &b) {
    const int64_t ca = a.end - a.start, cb = b.end - b.start;
    if (ca != cb) return ca > cb;
    if (a.seg != b.seg) return a.seg < b.seg;
    return a.head < b.head;
  });
  return n_items;
}

BuildParams build_params(const hypic_build_desc *d) {
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
  p.status = d->status;
  return p;
}

}  // namespace hypic

extern "C" {

int hypic_version(void) { return 100; }

const char *hypic_status_string(int s) {
  switch (s) {
    case HYPIC_OK: return "ok";
    case HYPIC_ERR_INVALID_ARG: return "invalid argument";
    case HYPIC_ERR_UNSUPPORTED: return "unsupported configuration";
    case HYPIC_ERR_WORKSPACE: return "workspace missing or too small";
    case HYPIC_ERR_CUDA: return "CUDA error";
    case HYPIC_ERR_TIMEOUT: return "device wait timed out";
    case HYPIC_ERR_NONFINITE: return "non-finite output";
    case HYPIC_ERR_BAD_SLOT: return "pool slot index out of range";
    default: return "unknown status";
  }
}

int hypic_status_from_word(uint32_t w) {
  if (w & HYPIC_STATUS_TIMEOUT) return HYPIC_ERR_TIMEOUT;
  if (w & HYPIC_STATUS_BAD_SLOT) return HYPIC_ERR_BAD_SLOT;
  if (w & HYPIC_STATUS_NONFINITE) return HYPIC_ERR_NONFINITE;
  return HYPIC_OK;
}

int hypic_plan_lpt(const int64_t *costs, int32_t n_items, int32_t n_workers, int32_t *order_out,
                   int32_t *worker_out, int64_t *makespan_out) {
  if (n_items < 0 || n_workers < 1 || (n_items > 0 && (!costs || !order_out))) return HYPIC_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_items; i++)
    if (costs[i] < 0) return HYPIC_ERR_INVALID_ARG;
  std::vector<int32_t> order(n_items);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return costs[a] > costs[b]; });
  // least-loaded worker first; ties to the lower worker index
  using W = std::pair<int64_t, int32_t>;
  std::priority_queue<W, std::vector<W>, std::greater<W>> heap;
  for (int32_t w = 0; w < n_workers; w++) heap.push({0, w});
  int64_t makespan = 0;
  for (int32_t r = 0; r < n_items; r++) {
    const int32_t it = order[r];
    W top = heap.top();
    heap.pop();
    top.first += costs[it];
    makespan = std::max(makespan, top.first);
    if (worker_out) worker_out[it] = top.second;
    heap.push(top);
    order_out[r] = it;
  }
  if (makespan_out) *makespan_out = makespan;
  return HYPIC_OK;
}

size_t hypic_build_workspace_bytes(const hypic_build_desc *d) {
  if (!d || d->n_seg < 0 || d->h_v < 1) return 0;
  return round_up(build_plan_size(n_build_items(d)), kAlign);  // one item per (segment, value head)
}

}  // extern "C"

namespace {
// the argument checks of a build (everything but the workspace); fills the
// slot of every segment
int check_build(const hypic_build_desc *d, std::vector<int32_t> &slots) {
  int st = check_build_shapes(d);
  if (st || d->n_seg == 0) return st;
  if ((st = check_build_pointers(d))) return st;
  std::vector<int32_t> sorted(d->n_seg);
  if ((st = check_build_slots(d, sorted.data()))) return st;
  slots.assign(d->n_seg, 0);
  for (int i = 0; i < d->n_seg; i++) slots[i] = d->slot_of_seg ? d->slot_of_seg[i] : i;
  return HYPIC_OK;
}

// HYPIC_FLAG_REQUIRE_TENSOR_CORES: refuse a call that would run an fp32
// CUDA-core kernel (a call with no tokens has nothing to compute and passes)
bool refused_fallback(uint32_t flags, int path, int64_t n_tokens) {
  return (flags & HYPIC_FLAG_REQUIRE_TENSOR_CORES) && n_tokens > 0 &&
         (path == HYPIC_PATH_F32_TOKEN || path == HYPIC_PATH_F32_COMPOSE);
}

// The tensor-core forward's workspace after the plan: per chunk record
// (64-token chunk of a built segment's body) and value head, the chunk's
// start state (64 KiB) and Delta (32 KiB), then one output item each.
// `chunk_base` (optional) receives every segment's first record index.
struct FwdLayout {
  int64_t n_rec = 0;  // chunk records (per value head)
  size_t plan = 0, rec_S = 0, rec_D = 0, items = 0, total = 0;
};
FwdLayout forward_layout(const hypic_build_desc *d, std::vector<int32_t> *chunk_base) {
  FwdLayout f;
  if (chunk_base) chunk_base->assign(d->n_seg, 0);
  for (int i = 0; i < d->n_seg; i++) {
    if (chunk_base) (*chunk_base)[i] = (int32_t)f.n_rec;
    if (d->slot_of_seg && d->slot_of_seg[i] == HYPIC_SLOT_SKIP) continue;
    const int64_t body = d->seg_offsets[i + 1] - std::min(d->seg_offsets[i] + d->seam_w, d->seg_offsets[i + 1]);
    f.n_rec += (body + 63) / 64;
  }
  const size_t n = (size_t)f.n_rec * d->h_v;
  f.plan = round_up(build_plan_size(n_build_items(d)), kAlign);
  f.rec_S = f.plan;
  f.rec_D = f.rec_S + round_up(n * 128 * 128 * 4, kAlign);
  f.items = f.rec_D + round_up(n * 64 * 128 * 4, kAlign);
  f.total = f.items + round_up(n * forward_item_bytes(), kAlign);
  return f;
}

// the build (q == NULL) or the prefill forward (q, o_out): validation, LPT
// plan, launch
int build_impl(const hypic_build_desc *d, const void *q, float *o_out, hypic_stream_t stream) {
  std::vector<int32_t> slots;
  int st = check_build(d, slots);
  if (st || d->n_seg == 0) return st;
  BuildParams p = build_params(d);
  if (refused_fallback(d->flags, build_path(p, d->n_tokens), d->n_tokens)) return HYPIC_ERR_UNSUPPORTED;
  p.q = q;
  p.o_out = o_out;
  // the forward's outputs: tensor cores from the recording build's chunk
  // records where they apply, else the fp32 token recurrence (CUDA cores)
  const bool tc_fwd = o_out && d->n_tokens > 0 && forward_tc_supported(p);
  if (o_out && !tc_fwd && refused_fallback(d->flags, HYPIC_PATH_F32_TOKEN, d->n_tokens)) return HYPIC_ERR_UNSUPPORTED;
  p.plan = reinterpret_cast<PlanHeader *>(d->workspace);
  p.items = reinterpret_cast<const BuildItem *>(p.plan + 1);

  // one item per (segment, value head) on every kernel (see launch_build);
  // skipped segments have none
  const size_t need_plan = round_up(build_plan_size(n_build_items(d)), kAlign);
  std::vector<int32_t> chunk_base;
  const FwdLayout fl = tc_fwd ? forward_layout(d, &chunk_base) : FwdLayout{};
  const size_t need = tc_fwd ? fl.total : need_plan;
  if (!d->workspace || d->workspace_bytes < need || !aligned(d->workspace, kAlign)) return HYPIC_ERR_WORKSPACE;
  std::vector<unsigned char> host(need_plan, 0);
  const int64_t n_items = fill_build_plan(d, host.data());
  if (n_items == 0) return HYPIC_OK;
  if (tc_fwd) {
    // every item's first chunk record (BuildItem.part)
    BuildItem *it = reinterpret_cast<BuildItem *>(reinterpret_cast<PlanHeader *>(host.data()) + 1);
    for (int64_t r = 0; r < n_items; r++) it[r].part = chunk_base[it[r].seg];
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // pageable source: the call returns once the bytes are staged, so `host`
  // may be released when it goes out of scope
  if (cudaMemcpyAsync(d->workspace, host.data(), need_plan, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return HYPIC_ERR_CUDA;
  BuildParams pb = p;
  pb.q = nullptr;
  pb.o_out = nullptr;
  if (tc_fwd) {
    char *ws = static_cast<char *>(d->workspace);
    pb.rec_S = reinterpret_cast<float *>(ws + fl.rec_S);
    pb.rec_D = reinterpret_cast<float *>(ws + fl.rec_D);
  }
  if (launch_build(pb, d->n_tokens, (int)n_items, sm_count(), s) != cudaSuccess) return HYPIC_ERR_CUDA;
  if (tc_fwd) {
    // the outputs: one item per (chunk record, value head)
    const int64_t n_out = fl.n_rec * d->h_v;
    if (n_out > INT32_MAX) return HYPIC_ERR_UNSUPPORTED;
    std::vector<unsigned char> fitems((size_t)n_out * forward_item_bytes());
    int64_t r = 0;
    for (int i = 0; i < d->n_seg; i++) {
      if (d->slot_of_seg && d->slot_of_seg[i] == HYPIC_SLOT_SKIP) continue;
      const int64_t start = std::min(d->seg_offsets[i] + d->seam_w, d->seg_offsets[i + 1]);
      const int64_t end = d->seg_offsets[i + 1];
      for (int64_t t0 = start, c = 0; t0 < end; t0 += 64, c++)
        for (int h = 0; h < d->h_v; h++)
          forward_fill_item(fitems.data(), r++, chunk_base[i] + (int32_t)c, h, (int32_t)std::min<int64_t>(64, end - t0),
                            t0);
    }
    char *ws = static_cast<char *>(d->workspace);
    if (cudaMemcpyAsync(ws + fl.items, fitems.data(), fitems.size(), cudaMemcpyHostToDevice, s) != cudaSuccess)
      return HYPIC_ERR_CUDA;
    BuildParams pf = p;
    pf.rec_S = pb.rec_S;
    pf.rec_D = pb.rec_D;
    if (launch_forward_tc(pf, ws + fl.items, (int)n_out, d->n_tokens, wait_limit(), s) != cudaSuccess)
      return HYPIC_ERR_CUDA;
  } else if (o_out) {
    // the forward: the pairs above, then the outputs by the fp32 token
    // recurrence over the S columns alone, from a fresh ticket over the same
    // plan
    if (cudaMemsetAsync(d->workspace, 0, sizeof(int32_t), s) != cudaSuccess) return HYPIC_ERR_CUDA;
    if (launch_forward_out(p, (int)n_items, sm_count(), s) != cudaSuccess) return HYPIC_ERR_CUDA;
  }
  return HYPIC_OK;
}
}  // namespace


namespace {
int check_compose(const hypic_compose_desc *d) {
  if (!d) return HYPIC_ERR_INVALID_ARG;
  int st = check_common_shapes(d->h_k, d->h_v, d->d_k, d->d_v, d->seam_w, d->variant, d->in_dtype);
  if (st) return st;
  if (d->n_layers < 0 || d->n_seg < 0 || d->n_slots < 0) return HYPIC_ERR_INVALID_ARG;
  if (d->seg_stride != 0 && d->seg_stride < d->n_seg) return HYPIC_ERR_INVALID_ARG;
  if (d->flags & ~(HYPIC_FLAG_CHECK_FINITE | HYPIC_FLAG_REQUIRE_TENSOR_CORES | HYPIC_FLAG_TRANSITION_ONLY))
    return HYPIC_ERR_INVALID_ARG;
  const bool trans = (d->flags & HYPIC_FLAG_TRANSITION_ONLY) != 0;
  if (trans && d->d_v != d->d_k) return HYPIC_ERR_INVALID_ARG;  // the state is a transition
  if (d->n_layers == 0) return HYPIC_OK;
  if (!d->S_out || !aligned(d->S_out, 4)) return HYPIC_ERR_INVALID_ARG;
  if (d->S_init && !aligned(d->S_init, 4)) return HYPIC_ERR_INVALID_ARG;
  if (d->n_seg > 0) {
    if (!d->slot || !aligned(d->slot, 4) || !d->T_pool || (!d->S_pool && !trans)) return HYPIC_ERR_INVALID_ARG;
    if (!aligned(d->T_pool, 4) || !aligned(d->S_pool, 4)) return HYPIC_ERR_INVALID_ARG;
  }
  const bool delta = is_delta(d->variant);
  const int esz = in_size(d->in_dtype);
  if (d->seam_w > 0 && d->n_seg > 0) {
    if (!d->seam_k || !d->seam_v || !d->seam_q || (!d->seam_out && !trans)) return HYPIC_ERR_INVALID_ARG;
    if (!aligned(d->seam_k, esz) || !aligned(d->seam_v, esz) || !aligned(d->seam_q, esz)) return HYPIC_ERR_INVALID_ARG;
    if (!aligned(d->seam_out, 4)) return HYPIC_ERR_INVALID_ARG;
    if (delta && !d->seam_beta) return HYPIC_ERR_INVALID_ARG;
    if ((d->variant == HYPIC_GDN || is_vector_gate(d->variant)) && !d->seam_g) return HYPIC_ERR_INVALID_ARG;
  }
  if (d->variant == HYPIC_SCALAR_DECAY && !d->seam_g) return HYPIC_ERR_INVALID_ARG;
  return HYPIC_OK;
}

ComposeParams compose_params(const hypic_compose_desc *d) {
  ComposeParams p{};
  p.n_layers = d->n_layers;
  p.n_seg = d->n_seg;
  p.h_k = d->h_k;
  p.h_v = d->h_v;
  p.d_k = d->d_k;
  p.d_v = d->d_v;
  p.seam_w = d->seam_w;
  p.seg_stride = d->seg_stride ? d->seg_stride : d->n_seg;
  p.variant = d->variant;
  p.in_dtype = d->in_dtype;
  p.flags = d->flags;
  p.slot = d->slot;
  p.n_slots = d->n_slots;
  p.T_pool = d->T_pool;
  p.S_pool = d->S_pool;
  p.seam_k = d->seam_k;
  p.seam_v = d->seam_v;
  p.seam_q = d->seam_q;
  p.seam_g = d->seam_g;
  p.seam_beta = d->seam_beta;
  p.S_init = d->S_init;
  p.S_out = d->S_out;
  p.seam_out = d->seam_out;
  p.status = d->status;
  return p;
}

int check_merge(const hypic_merge_desc *d) {
  if (!d) return HYPIC_ERR_INVALID_ARG;
  if (d->n_merge < 0 || d->h_v < 1 || d->d_k < 1 || d->d_v < 1) return HYPIC_ERR_INVALID_ARG;
  if (d->variant < HYPIC_GDN || d->variant > HYPIC_DIAG_GATE) return HYPIC_ERR_INVALID_ARG;
  if (d->d_k > 128 || d->d_v > 128) return HYPIC_ERR_UNSUPPORTED;
  if (d->n_slots_a < 0 || d->n_slots_b < 0 || d->n_slots_out < 0) return HYPIC_ERR_INVALID_ARG;
  if ((int64_t)d->n_merge * d->h_v > INT32_MAX) return HYPIC_ERR_UNSUPPORTED;
  if (d->n_merge == 0) return HYPIC_OK;
  if (!d->later || !d->earlier || !d->out || !aligned(d->later, 4) || !aligned(d->earlier, 4) || !aligned(d->out, 4))
    return HYPIC_ERR_INVALID_ARG;
  const float *pools[6] = {d->T_a, d->S_a, d->T_b, d->S_b, d->T_out, d->S_out};
  for (const float *q : pools)
    if (!q || !aligned(q, 4)) return HYPIC_ERR_INVALID_ARG;
  return HYPIC_OK;
}

// One compose launch: tensor cores where they apply, else the fp32 kernel.
// Transition-only with no S_init starts from the identity, written into
// S_out first (the kernels allow S_out to alias S_init).
int compose_launch(ComposeParams p, hypic_stream_t stream) {
  const int path = compose_tc_supported(p) ? HYPIC_PATH_TC_COMPOSE : HYPIC_PATH_F32_COMPOSE;
  if (refused_fallback(p.flags, path, p.n_seg)) return HYPIC_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((p.flags & HYPIC_FLAG_TRANSITION_ONLY) && !p.S_init) {
    if (launch_fill_identity(p.S_out, (int64_t)p.n_layers * p.h_v, p.d_k, s) != cudaSuccess) return HYPIC_ERR_CUDA;
    p.S_init = p.S_out;
  }
  const cudaError_t e = path == HYPIC_PATH_TC_COMPOSE ? launch_compose_tc(p, wait_limit(), s) : launch_compose_simt(p, s);
  return e == cudaSuccess ? HYPIC_OK : HYPIC_ERR_CUDA;
}

// S_start[0] = S_init (or 0); S_start[s] = T_span[s-1] S_start[s-1] +
// S_span[s-1], one single-pair compose per step (no seam tokens).  `slots`
// is device scratch of n_layers int32.
int span_scan_impl(int L, int n_spans, int H, int dk, int dv, const float *T_span, const float *S_span,
                   const float *S_init, float *S_start, int32_t *slots, uint32_t *status, hypic_stream_t stream) {
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const size_t T_per = (size_t)L * H * dk * dk, S_per = (size_t)L * H * dk * dv;
  if (S_init) {
    if (cudaMemcpyAsync(S_start, S_init, S_per * 4, cudaMemcpyDeviceToDevice, cs) != cudaSuccess) return HYPIC_ERR_CUDA;
  } else if (cudaMemsetAsync(S_start, 0, S_per * 4, cs) != cudaSuccess) {
    return HYPIC_ERR_CUDA;
  }
  if (n_spans < 2) return HYPIC_OK;
  std::vector<int32_t> idx(L);
  std::iota(idx.begin(), idx.end(), 0);
  // pageable source: the copy is staged before the call returns
  if (cudaMemcpyAsync(slots, idx.data(), (size_t)L * 4, cudaMemcpyHostToDevice, cs) != cudaSuccess)
    return HYPIC_ERR_CUDA;
  for (int s = 1; s < n_spans; s++) {
    ComposeParams p{};
    p.n_layers = L;
    p.n_seg = 1;
    p.seg_stride = 1;
    p.h_k = H;
    p.h_v = H;
    p.d_k = dk;
    p.d_v = dv;
    p.seam_w = 0;
    p.variant = HYPIC_DELTANET;  // a dense transition, no seam token
    p.in_dtype = HYPIC_IN_BF16;
    p.slot = slots;
    p.n_slots = L;
    p.T_pool = T_span + (s - 1) * T_per;
    p.S_pool = S_span + (s - 1) * S_per;
    p.S_init = S_start + (s - 1) * S_per;
    p.S_out = S_start + s * S_per;
    p.status = status;
    const int st = compose_launch(p, stream);
    if (st) return st;
  }
  return HYPIC_OK;
}

MergeParams merge_params(const hypic_merge_desc *d) {
  MergeParams p{};
  p.n_merge = d->n_merge;
  p.h_v = d->h_v;
  p.d_k = d->d_k;
  p.d_v = d->d_v;
  p.variant = d->variant;
  p.later = d->later;
  p.earlier = d->earlier;
  p.out = d->out;
  p.n_slots_a = d->n_slots_a;
  p.n_slots_b = d->n_slots_b;
  p.n_slots_out = d->n_slots_out;
  p.T_a = d->T_a;
  p.S_a = d->S_a;
  p.T_b = d->T_b;
  p.S_b = d->S_b;
  p.T_out = d->T_out;
  p.S_out = d->S_out;
  p.status = d->status;
  return p;
}
}  // namespace

// ---- the host-buffer calls: copy streams and events per (device, caller
// stream), created on first use and kept for the life of the process, so
// that host-buffer calls on different streams overlap their copies.  Past
// kPipesPerDevice caller streams, the first pipe is shared (still correct,
// without the overlap).  An event may be recorded again while earlier waits
// on it are pending: a wait takes the record that precedes it.
namespace {
constexpr int kMaxHostChunks = 64;
constexpr int kMaxDevices = 64;
constexpr int kPipesPerDevice = 8;
struct HostPipe {
  bool ready = false;
  bool used = false;
  cudaStream_t owner = nullptr;  // the caller stream this pipe serves
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, fin = nullptr;
  cudaEvent_t in_done[kMaxHostChunks] = {}, built[kMaxHostChunks] = {};
};
std::mutex g_host_mu;
HostPipe g_pipes[kMaxDevices][kPipesPerDevice];

int host_pipe(HostPipe *&hp, cudaStream_t owner) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HYPIC_ERR_CUDA;
  hp = &g_pipes[dev][0];
  for (int i = 0; i < kPipesPerDevice; i++) {
    HostPipe &c = g_pipes[dev][i];
    if (c.used && c.owner == owner) {
      hp = &c;
      break;
    }
    if (!c.used) {
      c.used = true;
      c.owner = owner;
      hp = &c;
      break;
    }
  }
  if (hp->ready) return HYPIC_OK;
  auto ev = [](cudaEvent_t *e) { return *e || cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
  if (!hp->in && cudaStreamCreateWithFlags(&hp->in, cudaStreamNonBlocking) != cudaSuccess) return HYPIC_ERR_CUDA;
  if (!hp->out && cudaStreamCreateWithFlags(&hp->out, cudaStreamNonBlocking) != cudaSuccess) return HYPIC_ERR_CUDA;
  if (!ev(&hp->start) || !ev(&hp->fin)) return HYPIC_ERR_CUDA;
  for (int i = 0; i < kMaxHostChunks; i++)
    if (!ev(&hp->in_done[i]) || !ev(&hp->built[i])) return HYPIC_ERR_CUDA;
  hp->ready = true;
  return HYPIC_OK;
}

int64_t T_slot_floats(const hypic_build_desc &b) {
  if (is_dense_T(b.variant)) return (int64_t)b.h_v * b.d_k * b.d_k;
  if (b.variant == HYPIC_DIAG_GATE) return (int64_t)b.h_v * b.d_k;
  return b.h_v;
}
}  // namespace

extern "C" {

int hypic_segment_build(const hypic_build_desc *d, hypic_stream_t stream) {
  return build_impl(d, nullptr, nullptr, stream);
}

int hypic_segment_build_host(const hypic_host_build_desc *d, hypic_stream_t stream) {
  if (!d) return HYPIC_ERR_INVALID_ARG;
  const hypic_build_desc &b = d->build;
  std::vector<int32_t> slots;
  int st = check_build(&b, slots);
  if (st) return st;
  if (d->n_chunks < 1 || !d->host_T || !d->host_S) return HYPIC_ERR_INVALID_ARG;
  if (b.n_tokens > 0 && (!d->host_k || !d->host_v)) return HYPIC_ERR_INVALID_ARG;
  if ((b.g == nullptr) != (d->host_g == nullptr) || (b.beta == nullptr) != (d->host_beta == nullptr))
    return HYPIC_ERR_INVALID_ARG;
  if (b.n_seg == 0) return HYPIC_OK;
  if (!b.workspace || b.workspace_bytes < hypic_build_workspace_bytes(&b) || !aligned(b.workspace, kAlign))
    return HYPIC_ERR_WORKSPACE;

  const int n_seg = b.n_seg;
  const int n_ch = std::min(std::min(d->n_chunks, n_seg), kMaxHostChunks);
  // group boundaries: about equal token counts, at least one segment each
  std::vector<int> bnd(n_ch + 1);
  bnd[0] = 0;
  bnd[n_ch] = n_seg;
  for (int c = 1; c < n_ch; c++) {
    const int64_t target = (int64_t)((double)b.n_tokens * c / n_ch);
    int j = (int)(std::lower_bound(b.seg_offsets, b.seg_offsets + n_seg + 1, target) - b.seg_offsets);
    j = std::max(j, bnd[c - 1] + 1);
    j = std::min(j, n_seg - (n_ch - c));
    bnd[c] = j;
  }
  const size_t es = (size_t)in_size(b.in_dtype);
  const bool vec = is_vector_gate(b.variant);
  const bool tok_g = b.variant == HYPIC_GDN || vec;  // g per token (else per head, or none)
  const size_t k_tok = (size_t)b.h_k * b.d_k * es, v_tok = (size_t)b.h_v * b.d_v * es;
  const size_t g_tok = (size_t)b.h_v * (vec ? b.d_k : 1) * 4, beta_tok = (size_t)b.h_v * 4;
  const size_t T_slot = (size_t)T_slot_floats(b) * 4, S_slot = (size_t)b.h_v * b.d_k * b.d_v * 4;

  std::lock_guard<std::mutex> lock(g_host_mu);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  HostPipe *hp = nullptr;
  if ((st = host_pipe(hp, s))) return st;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  auto h2d = [&](const void *dst, const void *src, size_t n) {
    return n == 0 || ok(cudaMemcpyAsync(const_cast<void *>(dst), src, n, cudaMemcpyHostToDevice, hp->in));
  };
  if (!ok(cudaEventRecord(hp->start, s)) || !ok(cudaStreamWaitEvent(hp->in, hp->start, 0)) ||
      !ok(cudaStreamWaitEvent(hp->out, hp->start, 0)))
    return HYPIC_ERR_CUDA;
  const bool has_beta = is_delta(b.variant) && b.beta;
  if (b.variant == HYPIC_SCALAR_DECAY && !h2d(b.g, d->host_g, (size_t)b.h_v * 4)) return HYPIC_ERR_CUDA;  // per head
  std::vector<int64_t> off;
  for (int c = 0; c < n_ch; c++) {
    const int a = bnd[c], e = bnd[c + 1];
    const int64_t t0 = b.seg_offsets[a], nt = b.seg_offsets[e] - t0;
    auto at = [](const void *base, size_t bytes) { return static_cast<const char *>(base) + bytes; };
    if (nt > 0) {
      if (!h2d(at(b.k, t0 * k_tok), at(d->host_k, t0 * k_tok), nt * k_tok) ||
          !h2d(at(b.v, t0 * v_tok), at(d->host_v, t0 * v_tok), nt * v_tok))
        return HYPIC_ERR_CUDA;
      if (tok_g && !h2d(at(b.g, t0 * g_tok), at(d->host_g, t0 * g_tok), nt * g_tok)) return HYPIC_ERR_CUDA;
      if (has_beta && !h2d(at(b.beta, t0 * beta_tok), at(d->host_beta, t0 * beta_tok), nt * beta_tok))
        return HYPIC_ERR_CUDA;
    }
    if (!ok(cudaEventRecord(hp->in_done[c], hp->in)) || !ok(cudaStreamWaitEvent(s, hp->in_done[c], 0)))
      return HYPIC_ERR_CUDA;
    // the group's build: the same descriptor over its segments, rebased
    off.assign(e - a + 1, 0);
    for (int i = a; i <= e; i++) off[i - a] = b.seg_offsets[i] - t0;
    hypic_build_desc cb = b;
    cb.n_tokens = (int32_t)nt;
    cb.n_seg = e - a;
    cb.seg_offsets = off.data();
    cb.slot_of_seg = slots.data() + a;
    cb.k = at(b.k, t0 * k_tok);
    cb.v = at(b.v, t0 * v_tok);
    if (tok_g) cb.g = reinterpret_cast<const float *>(at(b.g, t0 * g_tok));
    if (has_beta) cb.beta = reinterpret_cast<const float *>(at(b.beta, t0 * beta_tok));
    if ((st = build_impl(&cb, nullptr, nullptr, stream))) return st;
    if (!ok(cudaEventRecord(hp->built[c], s)) || !ok(cudaStreamWaitEvent(hp->out, hp->built[c], 0)))
      return HYPIC_ERR_CUDA;
    // its slots out, runs of consecutive slots as one copy
    for (int i = a; i < e;) {
      if (slots[i] == HYPIC_SLOT_SKIP) {
        i++;
        continue;
      }
      int j = i + 1;
      while (j < e && slots[j] == slots[j - 1] + 1) j++;
      const size_t s0 = (size_t)slots[i], n = (size_t)(j - i);
      if (!ok(cudaMemcpyAsync(reinterpret_cast<char *>(d->host_T) + s0 * T_slot, at(b.T_pool, s0 * T_slot),
                              n * T_slot, cudaMemcpyDeviceToHost, hp->out)) ||
          !ok(cudaMemcpyAsync(reinterpret_cast<char *>(d->host_S) + s0 * S_slot, at(b.S_pool, s0 * S_slot),
                              n * S_slot, cudaMemcpyDeviceToHost, hp->out)))
        return HYPIC_ERR_CUDA;
      i = j;
    }
  }
  if (!ok(cudaEventRecord(hp->fin, hp->out)) || !ok(cudaStreamWaitEvent(s, hp->fin, 0))) return HYPIC_ERR_CUDA;
  return HYPIC_OK;
}


int hypic_compose_host(const hypic_host_compose_desc *d, hypic_stream_t stream) {
  if (!d) return HYPIC_ERR_INVALID_ARG;
  const hypic_compose_desc &c = d->compose;
  int st = check_compose(&c);
  if (st) return st;
  if (c.flags & HYPIC_FLAG_TRANSITION_ONLY) return HYPIC_ERR_INVALID_ARG;
  if (d->n_chunks < 1 || !d->host_S_out) return HYPIC_ERR_INVALID_ARG;
  const bool seam = c.seam_w > 0 && c.n_seg > 0;
  auto pair_ok = [](const void *dev, const void *host) { return (dev == nullptr) == (host == nullptr); };
  if (seam && (!d->host_seam_k || !d->host_seam_v || !d->host_seam_q || !d->host_seam_out)) return HYPIC_ERR_INVALID_ARG;
  if (!pair_ok(c.seam_g, d->host_seam_g) || !pair_ok(c.seam_beta, d->host_seam_beta)) return HYPIC_ERR_INVALID_ARG;
  if (d->host_S_init && !c.S_init) return HYPIC_ERR_INVALID_ARG;
  if (c.n_layers == 0) return HYPIC_OK;
  const ComposeParams base = compose_params(&c);
  const int L = c.n_layers;
  // groups of whole waves: a launch of fewer chains than the GPU holds at
  // once (two per SM on the tensor-core path) takes as long as a full wave,
  // so the layers are never split finer than the waves the chains need
  const int64_t slots = 2 * (int64_t)sm_count();
  const int waves = (int)std::max<int64_t>(1, ((int64_t)L * c.h_v + slots - 1) / slots);
  const int n_ch = std::min(std::min(std::min(d->n_chunks, L), waves), kMaxHostChunks);
  const size_t es = (size_t)in_size(c.in_dtype), w = (size_t)c.seam_w;
  const size_t seg_stride = (size_t)base.seg_stride;
  const bool vec = is_vector_gate(c.variant);
  // bytes per layer of each array
  const size_t k_l = seg_stride * w * c.h_k * c.d_k * es, v_l = seg_stride * w * c.h_v * c.d_v * es;
  const size_t g_l = c.variant == HYPIC_SCALAR_DECAY ? (size_t)c.h_v * 4 : seg_stride * w * c.h_v * (vec ? c.d_k : 1) * 4;
  const size_t b_l = seg_stride * w * c.h_v * 4, o_l = seg_stride * w * c.h_v * c.d_v * 4;
  const size_t s_l = (size_t)c.h_v * c.d_k * c.d_v * 4;

  std::lock_guard<std::mutex> lock(g_host_mu);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  HostPipe *hp = nullptr;
  if ((st = host_pipe(hp, s))) return st;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  auto at = [](const void *base_, size_t bytes) { return static_cast<const char *>(base_) + bytes; };
  auto h2d = [&](const void *dst, const void *src, size_t n) {
    return n == 0 || !dst || ok(cudaMemcpyAsync(const_cast<void *>(dst), src, n, cudaMemcpyHostToDevice, hp->in));
  };
  auto d2h = [&](void *dst, const void *src, size_t n) {
    return n == 0 || !dst || ok(cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, hp->out));
  };
  if (!ok(cudaEventRecord(hp->start, s)) || !ok(cudaStreamWaitEvent(hp->in, hp->start, 0)) ||
      !ok(cudaStreamWaitEvent(hp->out, hp->start, 0)))
    return HYPIC_ERR_CUDA;
  for (int g = 0; g < n_ch; g++) {
    const int l0 = (int)((int64_t)L * g / n_ch), l1 = (int)((int64_t)L * (g + 1) / n_ch), nl = l1 - l0;
    if (seam) {
      if (!h2d(at(c.seam_k, l0 * k_l), at(d->host_seam_k, l0 * k_l), nl * k_l) ||
          !h2d(at(c.seam_v, l0 * v_l), at(d->host_seam_v, l0 * v_l), nl * v_l) ||
          !h2d(at(c.seam_q, l0 * k_l), at(d->host_seam_q, l0 * k_l), nl * k_l) ||
          !h2d(c.seam_beta ? at(c.seam_beta, l0 * b_l) : nullptr, at(d->host_seam_beta, l0 * b_l), nl * b_l))
        return HYPIC_ERR_CUDA;
    }
    if ((seam || c.variant == HYPIC_SCALAR_DECAY) &&
        !h2d(c.seam_g ? at(c.seam_g, l0 * g_l) : nullptr, at(d->host_seam_g, l0 * g_l), nl * g_l))
      return HYPIC_ERR_CUDA;
    if (d->host_S_init && !h2d(at(c.S_init, l0 * s_l), at(d->host_S_init, l0 * s_l), nl * s_l)) return HYPIC_ERR_CUDA;
    if (!ok(cudaEventRecord(hp->in_done[g], hp->in)) || !ok(cudaStreamWaitEvent(s, hp->in_done[g], 0)))
      return HYPIC_ERR_CUDA;
    // the group's compose: the same call over its layers
    ComposeParams p = base;
    p.n_layers = nl;
    p.slot = c.slot ? c.slot + (size_t)l0 * seg_stride : nullptr;
    p.seam_k = c.seam_k ? at(c.seam_k, l0 * k_l) : nullptr;
    p.seam_v = c.seam_v ? at(c.seam_v, l0 * v_l) : nullptr;
    p.seam_q = c.seam_q ? at(c.seam_q, l0 * k_l) : nullptr;
    p.seam_g = c.seam_g ? reinterpret_cast<const float *>(at(c.seam_g, l0 * g_l)) : nullptr;
    p.seam_beta = c.seam_beta ? reinterpret_cast<const float *>(at(c.seam_beta, l0 * b_l)) : nullptr;
    p.S_init = c.S_init ? reinterpret_cast<const float *>(at(c.S_init, l0 * s_l)) : nullptr;
    p.S_out = c.S_out + (size_t)l0 * s_l / 4;
    p.seam_out = c.seam_out ? c.seam_out + (size_t)l0 * o_l / 4 : nullptr;
    if ((st = compose_launch(p, stream))) return st;
    if (!ok(cudaEventRecord(hp->built[g], s)) || !ok(cudaStreamWaitEvent(hp->out, hp->built[g], 0)))
      return HYPIC_ERR_CUDA;
    if (!d2h(reinterpret_cast<char *>(d->host_S_out) + l0 * s_l, p.S_out, nl * s_l) ||
        (seam && !d2h(reinterpret_cast<char *>(d->host_seam_out) + l0 * o_l, p.seam_out, nl * o_l)))
      return HYPIC_ERR_CUDA;
  }
  if (!ok(cudaEventRecord(hp->fin, hp->out)) || !ok(cudaStreamWaitEvent(s, hp->fin, 0))) return HYPIC_ERR_CUDA;
  return HYPIC_OK;
}

int hypic_segment_forward(const hypic_forward_desc *d, hypic_stream_t stream) {
  if (!d) return HYPIC_ERR_INVALID_ARG;
  const hypic_build_desc &b = d->build;
  if (b.n_tokens > 0 && b.n_seg > 0) {
    const size_t esz = b.in_dtype == HYPIC_IN_BF16 ? 2 : 4;
    if (!d->q || !aligned(d->q, esz) || !d->o_out || !aligned(d->o_out, 4)) return HYPIC_ERR_INVALID_ARG;
  }
  return build_impl(&b, d->q, d->o_out ? d->o_out : nullptr, stream);
}

size_t hypic_compose_workspace_bytes(const hypic_compose_desc *d) {
  (void)d;
  return 0;
}

int hypic_compose(const hypic_compose_desc *d, hypic_stream_t stream) {
  int st = check_compose(d);
  if (st || d->n_layers == 0) return st;
  return compose_launch(compose_params(d), stream);
}

size_t hypic_span_scan_workspace_bytes(const hypic_span_scan_desc *d) {
  if (!d) return 0;
  if (d->n_layers < 1 || d->n_spans < 1) return 0;
  return round_up((size_t)d->n_layers * 4, kAlign);
}

int hypic_span_scan(const hypic_span_scan_desc *d, hypic_stream_t stream) {
  if (!d) return HYPIC_ERR_INVALID_ARG;
  if (d->n_layers < 0 || d->n_spans < 0 || d->h_v < 1 || d->d_k < 1 || d->d_v < 1) return HYPIC_ERR_INVALID_ARG;
  if (d->d_k > 128 || d->d_v > 128) return HYPIC_ERR_UNSUPPORTED;
  if (d->n_layers == 0 || d->n_spans == 0) return HYPIC_OK;
  if (!d->S_start || !aligned(d->S_start, 4) || (d->S_init && !aligned(d->S_init, 4))) return HYPIC_ERR_INVALID_ARG;
  if (d->n_spans > 1 && (!d->T_span || !d->S_span || !aligned(d->T_span, 4) || !aligned(d->S_span, 4)))
    return HYPIC_ERR_INVALID_ARG;
  const size_t need = hypic_span_scan_workspace_bytes(d);
  if (!d->workspace || d->workspace_bytes < need || !aligned(d->workspace, kAlign)) return HYPIC_ERR_WORKSPACE;
  return span_scan_impl(d->n_layers, d->n_spans, d->h_v, d->d_k, d->d_v, d->T_span, d->S_span, d->S_init, d->S_start,
                        static_cast<int32_t *>(d->workspace), d->status, stream);
}

size_t hypic_compose_spans_workspace_bytes(const hypic_compose_desc *d, int32_t n_spans) {
  if (!d || d->n_layers < 1 || n_spans < 1 || d->h_v < 1 || d->d_k < 1 || d->d_v < 1) return 0;
  const size_t mat = (size_t)n_spans * d->n_layers * d->h_v;
  return round_up(mat * d->d_k * d->d_k * 4, kAlign) + 2 * round_up(mat * d->d_k * d->d_v * 4, kAlign) +
         round_up((size_t)d->n_layers * 4, kAlign);
}

int hypic_compose_spans(const hypic_compose_desc *d, int32_t n_spans, const int32_t *span_bounds,
                        hypic_stream_t stream) {
  int st = check_compose(d);
  if (st) return st;
  if (d->flags & HYPIC_FLAG_TRANSITION_ONLY) return HYPIC_ERR_INVALID_ARG;
  if (n_spans < 1 || !span_bounds || span_bounds[0] != 0 || span_bounds[n_spans] != d->n_seg)
    return HYPIC_ERR_INVALID_ARG;
  for (int s = 0; s < n_spans; s++)
    if (span_bounds[s + 1] < span_bounds[s]) return HYPIC_ERR_INVALID_ARG;
  if (d->n_layers == 0) return HYPIC_OK;
  const size_t need = hypic_compose_spans_workspace_bytes(d, n_spans);
  if (!d->workspace || d->workspace_bytes < need || !aligned(d->workspace, kAlign)) return HYPIC_ERR_WORKSPACE;
  const int L = d->n_layers, H = d->h_v, dk = d->d_k, dv = d->d_v;
  const size_t mat = (size_t)n_spans * L * H;
  char *ws = static_cast<char *>(d->workspace);
  float *T_span = reinterpret_cast<float *>(ws);
  ws += round_up(mat * dk * dk * 4, kAlign);
  float *S_span = reinterpret_cast<float *>(ws);
  ws += round_up(mat * dk * dv * 4, kAlign);
  float *S_start = reinterpret_cast<float *>(ws);
  ws += round_up(mat * dk * dv * 4, kAlign);
  int32_t *scan_slots = reinterpret_cast<int32_t *>(ws);
  const size_t T_per = (size_t)L * H * dk * dk, S_per = (size_t)L * H * dk * dv;  // one span, every layer
  const ComposeParams base = compose_params(d);
  const int esz = in_size(d->in_dtype);
  const bool vec = is_vector_gate(d->variant);
  const size_t w = (size_t)d->seam_w;
  // span s of every chain: the arrays advanced by a segments, n_seg = b - a,
  // the layer stride kept
  auto span_params = [&](int s) {
    ComposeParams p = base;
    const size_t a = (size_t)span_bounds[s];
    p.n_seg = span_bounds[s + 1] - span_bounds[s];
    p.slot = d->slot ? d->slot + a : nullptr;
    auto adv = [&](const void *x, size_t per_seg) {
      return x ? static_cast<const void *>(static_cast<const char *>(x) + a * per_seg) : nullptr;
    };
    p.seam_k = adv(d->seam_k, w * d->h_k * d->d_k * esz);
    p.seam_v = adv(d->seam_v, w * d->h_v * d->d_v * esz);
    p.seam_q = adv(d->seam_q, w * d->h_k * d->d_k * esz);
    if (d->variant != HYPIC_SCALAR_DECAY)  // per-token gates (a scalar decay is per layer)
      p.seam_g = static_cast<const float *>(adv(d->seam_g, w * d->h_v * (vec ? d->d_k : 1) * 4));
    p.seam_beta = static_cast<const float *>(adv(d->seam_beta, w * d->h_v * 4));
    p.seam_out = d->seam_out ? d->seam_out + a * w * d->h_v * d->d_v : nullptr;
    return p;
  };
  // 1. the pair of every span but the last (nothing follows it): S from
  // zero (its seam outputs are overwritten in step 3), T from the identity
  for (int s = 0; s + 1 < n_spans; s++) {
    ComposeParams p = span_params(s);
    p.S_init = nullptr;
    p.S_out = S_span + s * S_per;
    if ((st = compose_launch(p, stream))) return st;
    ComposeParams t = span_params(s);
    t.flags |= HYPIC_FLAG_TRANSITION_ONLY;
    t.d_v = dk;
    t.S_init = nullptr;  // the identity
    t.S_out = T_span + s * T_per;
    t.seam_out = nullptr;
    if ((st = compose_launch(t, stream))) return st;
  }
  // 2. the exclusive scan over the spans
  if ((st = span_scan_impl(L, n_spans, H, dk, dv, T_span, S_span, d->S_init, S_start, scan_slots, d->status, stream)))
    return st;
  // 3. every span from its start state, with its seam outputs; the last
  // span's final state is the chain's
  for (int s = 0; s < n_spans; s++) {
    ComposeParams p = span_params(s);
    p.S_init = S_start + s * S_per;
    p.S_out = s + 1 == n_spans ? d->S_out : S_span + s * S_per;  // earlier spans' final states: scratch
    if ((st = compose_launch(p, stream))) return st;
  }
  return HYPIC_OK;
}

int hypic_pair_merge(const hypic_merge_desc *d, hypic_stream_t stream) {
  int st = check_merge(d);
  if (st || d->n_merge == 0) return st;
  if (launch_merge(merge_params(d), wait_limit(), reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return HYPIC_ERR_CUDA;
  return HYPIC_OK;
}

// ---- which kernel a call runs (the same predicates as the dispatch above)
int hypic_build_path(const hypic_build_desc *d) {
  const int st = check_build_shapes(d);
  if (st) return -st;
  if (d->n_seg == 0) return HYPIC_PATH_NONE;
  return build_path(build_params(d), d->n_tokens);
}

int hypic_forward_path(const hypic_forward_desc *d) {
  if (!d) return -HYPIC_ERR_INVALID_ARG;
  const int st = check_build_shapes(&d->build);
  if (st) return -st;
  if (d->build.n_seg == 0) return HYPIC_PATH_NONE;
  BuildParams p = build_params(&d->build);
  p.q = d->q;
  p.o_out = d->o_out;
  return d->build.n_tokens > 0 && forward_tc_supported(p) ? HYPIC_PATH_TC_FORWARD : HYPIC_PATH_F32_TOKEN;
}

size_t hypic_forward_workspace_bytes(const hypic_forward_desc *d) {
  if (!d || check_build_shapes(&d->build) != HYPIC_OK) return 0;
  BuildParams p = build_params(&d->build);
  p.q = d->q;
  p.o_out = d->o_out;
  if (d->build.n_tokens > 0 && d->build.n_seg > 0 && forward_tc_supported(p))
    return forward_layout(&d->build, nullptr).total;
  return hypic_build_workspace_bytes(&d->build);
}

int hypic_compose_path(const hypic_compose_desc *d) {
  const int st = check_compose(d);
  if (st) return -st;
  if (d->n_layers == 0) return HYPIC_PATH_NONE;
  return compose_tc_supported(compose_params(d)) ? HYPIC_PATH_TC_COMPOSE : HYPIC_PATH_F32_COMPOSE;
}

int hypic_merge_path(const hypic_merge_desc *d) {
  const int st = check_merge(d);
  if (st) return -st;
  if (d->n_merge == 0) return HYPIC_PATH_NONE;
  return merge_tc_supported(merge_params(d)) ? HYPIC_PATH_TC_MERGE : HYPIC_PATH_F32_MERGE;
}

int hypic_pair_rerotate(const hypic_rerotate_desc *d, hypic_stream_t stream) {
  if (!d) return HYPIC_ERR_INVALID_ARG;
  if (d->n_items < 0 || d->h_v < 1 || d->d_k < 1 || d->d_v < 1) return HYPIC_ERR_INVALID_ARG;
  if (d->variant < HYPIC_GDN || d->variant > HYPIC_DIAG_GATE) return HYPIC_ERR_INVALID_ARG;
  if (d->layout != HYPIC_ROPE_INTERLEAVED && d->layout != HYPIC_ROPE_HALF) return HYPIC_ERR_INVALID_ARG;
  if (d->rot_dim < 2 || (d->rot_dim & 1) || d->rot_dim > d->d_k) return HYPIC_ERR_INVALID_ARG;
  if (d->layout == HYPIC_ROPE_HALF && (d->rot_dim % 8) != 0) return HYPIC_ERR_INVALID_ARG;
  if (!(d->base > 0.0)) return HYPIC_ERR_INVALID_ARG;
  if (d->n_slots_in < 0 || d->n_slots_out < 0) return HYPIC_ERR_INVALID_ARG;
  // per-channel and diagonal gates do not commute with the rotation
  if (d->variant == HYPIC_CHANNEL_DELTA || d->variant == HYPIC_DIAG_GATE) return HYPIC_ERR_UNSUPPORTED;
  if (d->d_k > 128 || d->d_v > 128 || (d->d_k % 4) != 0 || (d->d_v % 4) != 0) return HYPIC_ERR_UNSUPPORTED;
  if ((int64_t)d->n_items * ((d->h_v + 3) / 4) > INT32_MAX) return HYPIC_ERR_UNSUPPORTED;
  if (d->n_items == 0) return HYPIC_OK;
  if (!d->slot_in || !d->slot_out || !d->delta || !aligned(d->slot_in, 4) || !aligned(d->slot_out, 4) ||
      !aligned(d->delta, 8))
    return HYPIC_ERR_INVALID_ARG;
  const float *pools[4] = {d->T_in, d->S_in, d->T_out, d->S_out};
  for (const float *q : pools)
    if (!q || !aligned(q, 16)) return HYPIC_ERR_INVALID_ARG;
  RerotateParams p{};
  p.n_items = d->n_items;
  p.h_v = d->h_v;
  p.d_k = d->d_k;
  p.d_v = d->d_v;
  p.variant = d->variant;
  p.rot_dim = d->rot_dim;
  p.layout = d->layout;
  p.base = d->base;
  p.slot_in = d->slot_in;
  p.slot_out = d->slot_out;
  p.delta = d->delta;
  p.n_slots_in = d->n_slots_in;
  p.n_slots_out = d->n_slots_out;
  p.T_in = d->T_in;
  p.S_in = d->S_in;
  p.T_out = d->T_out;
  p.S_out = d->S_out;
  p.status = d->status;
  if (launch_rerotate(p, wait_limit(), reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return HYPIC_ERR_CUDA;
  return HYPIC_OK;
}

}  // extern "C"
