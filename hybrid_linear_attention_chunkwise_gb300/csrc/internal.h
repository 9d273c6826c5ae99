// internal.h -- types shared by the host library and the CUDA kernels of
// libhypic (not part of the public ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "hypic.h"

namespace hypic {

// One unit of build work: one (segment, value head) pair, or one half of it
// for kernels that split the augmented block [T | S] by columns.
struct BuildItem {
  int32_t seg;
  int32_t head;
  int32_t slot;
  int32_t part;   // kernel-specific sub-item (0 when unused)
  int64_t start;  // first body token (after the seam window)
  int64_t end;    // one past the last token
};

// Device-visible build plan header, followed by n_items BuildItem records.
// `ticket` is the dynamic work counter (zeroed by the host copy).  `mode`
// says how the persistent build kernels take items:
//   PLAN_LPT          items in LPT order (longest body first, ties by index),
//                     each CTA takes the next one from the shared ticket when
//                     it is free: greedy LPT list scheduling over the SMs;
//   PLAN_ROUND_ROBIN  items in index order (segment-major), CTA b takes items
//                     b, b + grid, b + 2 grid, ...: a static round-robin
//                     assignment, kept for measuring what LPT gains.
constexpr int32_t PLAN_LPT = 0;
constexpr int32_t PLAN_ROUND_ROBIN = 1;
struct PlanHeader {
  int32_t ticket;
  int32_t n_items;
  int32_t mode;
  int32_t pad[13];  // keeps the item array 64-byte aligned
};
static_assert(sizeof(PlanHeader) == 64, "plan header size");

struct BuildParams {
  int32_t h_k, h_v, d_k, d_v;
  int32_t variant, in_dtype;
  uint32_t flags;
  int64_t n_slots;
  const void *k, *v;
  const float *g, *beta;
  float *T_pool, *S_pool;
  const void *q;            // forward: [n_tokens, h_k, d_k] (NULL: pairs only)
  float *o_out;             // forward: [n_tokens, h_v, d_v] body-token outputs
  float *rec_S;             // recording build (tensor-core forward): per (chunk, head) the chunk's
  float *rec_D;             //   start state [128 d][128 j] and Delta = U - W S_0 [64 t][128 j];
                            //   the item's first chunk record is BuildItem.part (NULL: no records)
  PlanHeader *plan;         // device copy of the plan
  const BuildItem *items;   // = (BuildItem*)(plan + 1)
  uint32_t *status;
};

struct ComposeParams {
  int32_t n_layers, n_seg, h_k, h_v, d_k, d_v, seam_w;
  int32_t seg_stride;  // segments per layer in slot, seam_* and seam_out (>= n_seg)
  int32_t variant, in_dtype;
  uint32_t flags;
  const int32_t *slot;
  int64_t n_slots;
  const float *T_pool, *S_pool;
  const void *seam_k, *seam_v, *seam_q;
  const float *seam_g, *seam_beta;
  const float *S_init;
  float *S_out, *seam_out;
  uint32_t *status;
};

struct RerotateParams {
  int32_t n_items, h_v, d_k, d_v, variant, rot_dim, layout;
  double base;
  const int32_t *slot_in, *slot_out;
  const int64_t *delta;
  int64_t n_slots_in, n_slots_out;
  const float *T_in, *S_in;
  float *T_out, *S_out;
  uint32_t *status;
};

struct MergeParams {
  int32_t n_merge, h_v, d_k, d_v, variant;
  const int32_t *later, *earlier, *out;
  int64_t n_slots_a, n_slots_b, n_slots_out;
  const float *T_a, *S_a;  // later pairs
  const float *T_b, *S_b;  // earlier pairs
  float *T_out, *S_out;
  uint32_t *status;
};

__host__ __device__ inline bool is_delta(int v) { return v == HYPIC_GDN || v == HYPIC_DELTANET || v == HYPIC_CHANNEL_DELTA; }
__host__ __device__ inline bool is_dense_T(int v) { return is_delta(v); }
__host__ __device__ inline bool is_vector_gate(int v) { return v == HYPIC_CHANNEL_DELTA || v == HYPIC_DIAG_GATE; }

// ---- build descriptors (host, no heap use; shared by every build entry
// point so that they accept and plan exactly the same calls)
// Shapes, segment offsets and the size limits of the descriptor.
int check_build_shapes(const hypic_build_desc *d);
// Input, gate and pool pointers (only those the call reads or writes).
int check_build_pointers(const hypic_build_desc *d);
// Slots in range and distinct; `sorted` is caller scratch of n_seg entries.
int check_build_slots(const hypic_build_desc *d, int32_t *sorted);
// Bytes of a plan of n_items items (header + items, not rounded).
size_t build_plan_size(int64_t n_items);
// Writes the plan of every (segment, value head) item of d into `plan`
// (at most build_plan_size(n_seg * h_v) bytes; segments whose slot is
// HYPIC_SLOT_SKIP have no items) and returns the item count: LPT order and
// mode, or index order and PLAN_ROUND_ROBIN under HYPIC_FLAG_ROUND_ROBIN.
// In-place sort, no heap.
int64_t fill_build_plan(const hypic_build_desc *d, void *plan);
// Kernel parameters of a build descriptor; the plan pointer is left NULL.
BuildParams build_params(const hypic_build_desc *d);
// The kernel a build with these parameters runs (a hypic_path value).
int build_path(const BuildParams &p, int64_t n_tokens);

// Launchers (each returns a cudaError_t from the launch).
// The build kernel for the parameters (tensor-core paths where they apply,
// else the token recurrence), one item per (segment, value head).
cudaError_t launch_build(const BuildParams &p, int64_t n_tokens, int n_items, int n_sm, cudaStream_t s);
cudaError_t launch_build_token(const BuildParams &p, int n_items, int n_sm, cudaStream_t s);
cudaError_t launch_forward_out(const BuildParams &p, int n_items, int n_sm, cudaStream_t s);
// Tensor-core chunkwise build: GDN / DeltaNet, bf16 inputs, d_k = d_v = 128,
// 16-byte aligned k / v.  Items are (segment, head, half of [T | S]).
bool build_tc_supported(const BuildParams &p);
cudaError_t launch_build_tc(const BuildParams &p, int64_t n_tokens, int n_items, int n_sm, uint32_t wait_limit,
                            cudaStream_t s);
// Tensor-core per-token outputs of the prefill forward (GDN / DeltaNet, bf16,
// d = 128, 16-byte aligned q and o_out) from the recording build's chunk
// records: one item per (chunk record, value head); `items` holds
// forward_item_bytes() per item, written by forward_fill_item.
bool forward_tc_supported(const BuildParams &p);
cudaError_t launch_forward_tc(const BuildParams &p, const void *items, int n_items, int64_t n_tokens,
                              uint32_t wait_limit, cudaStream_t s);
size_t forward_item_bytes();
void forward_fill_item(void *items, int64_t idx, int32_t rec, int32_t head, int32_t nt, int64_t tok0);
// Tensor-core fast path (no erase: scalar decay, ungated, diagonal gate),
// bf16 inputs, d_k = d_v = 128, 16-byte aligned k / v.
bool build_fast_supported(const BuildParams &p);
cudaError_t launch_build_fast(const BuildParams &p, int64_t n_tokens, int n_items, int n_sm, uint32_t wait_limit,
                              cudaStream_t s);
// [n_tokens, heads, 128] elements of `esz` bytes as a 3-D TMA map with
// box_x-channel x 1-head x box_t-token boxes (false if the map cannot be
// encoded).  Out-of-range tokens read as zero.
bool make_tmap_3d(CUtensorMap *map, CUtensorMapDataType dt, uint32_t esz, const void *base, int64_t n_tokens,
                  int heads, uint32_t box_x, uint32_t box_t, CUtensorMapSwizzle swz);
// [n_tokens, heads, 128] bf16 with 64-channel x 1-head x `rows`-token boxes
// and 128-byte swizzle.
bool make_tmap_tokens(CUtensorMap *map, const void *base, int64_t n_tokens, int heads, int rows = 64);
// Tensor-core chunkwise build for the per-channel gated delta rule, bf16
// inputs, d_k = d_v = 128, 16-byte aligned k / v / g.
bool build_channel_supported(const BuildParams &p);
cudaError_t launch_build_channel(const BuildParams &p, int64_t n_tokens, int n_items, int n_sm, uint32_t wait_limit,
                                 cudaStream_t s);
// 2-D fp32 view [rows, 128] with 32-column x box_rows tiles and 128-byte
// swizzle (one K-slab of a K-major tf32 MMA operand per tile).
bool make_tmap_f32_rows(CUtensorMap *map, const float *base, uint64_t rows, uint32_t box_rows);
// Pair merge: tensor cores for dense d_k = d_v = 128 with 16-byte aligned
// pools, fp32 CUDA-core kernel otherwise.
bool merge_tc_supported(const MergeParams &p);
cudaError_t launch_merge(const MergeParams &p, uint32_t wait_limit, cudaStream_t s);
cudaError_t launch_rerotate(const RerotateParams &p, uint32_t wait_limit, cudaStream_t s);
cudaError_t launch_compose_simt(const ComposeParams &p, cudaStream_t s);
// out[m] = I (d x d) for m < n_mats
cudaError_t launch_fill_identity(float *out, int64_t n_mats, int d, cudaStream_t s);
cudaError_t launch_compose_tc(const ComposeParams &p, uint32_t wait_limit, cudaStream_t s);
// The tensor-core compose covers dense transitions, bf16 seam tokens,
// d_k = d_v = 128, h_v % 4 == 0 and 16-byte aligned tensors.
bool compose_tc_supported(const ComposeParams &p);

// Bounded-wait poll limit for the pipelined kernels (HYPIC_DEBUG_WAIT_LIMIT
// overrides it, for the timeout test).
uint32_t wait_limit();
// HYPIC_DEBUG_STALL=1: pipelined kernels first wait on a barrier that is never
// signalled, so the bounded wait runs out (the timeout test).
bool debug_stall();

}  // namespace hypic
