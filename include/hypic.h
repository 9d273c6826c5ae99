/*
 * hypic.h -- C ABI of the GB300 (sm_103a) library for the linear-attention
 * state algebra behind HYPIC's position-independent caching.
 *
 * Method (HYPIC news pages: nav.aitube.vip "首 token 延迟降 3.25 倍！...HYPIC..."
 * §2.1 linear layers and §2.2 seam window; xix.ai Spanish/Japanese pages,
 * paragraphs on linear layers and on full-attention seams):
 *   - for a segment C and a head, the segment-cumulative transition operator
 *     T_C is the product of every token transition matrix in the segment, and
 *     S(C|0) is the segment's final state from a zero initial state; the pair
 *     depends only on the segment's own tokens, so it is cached once;
 *   - at reuse the exact state under any prefix follows by left-multiplying
 *     with T_C and adding: S(C1·C2) = T(C2)·S(C1) + S(C2);
 *   - the first w tokens of each segment (the seam window, w = 8 by default)
 *     are not cached: at reuse the linear layer advances the running state
 *     through them token by token and emits each seam token's output.
 *
 * Per-token transitions (state S in R^{d_k x d_v}, S_t = T_t S_{t-1} + U_t,
 * output o_t = S_t^T q_t with the post-update state):
 *   HYPIC_GDN            T_t = a_t (I - b_t k_t k_t^T),          U_t = b_t k_t v_t^T
 *   HYPIC_DELTANET       T_t = I - b_t k_t k_t^T,                U_t = b_t k_t v_t^T
 *   HYPIC_CHANNEL_DELTA  T_t = (I - b_t k_t k_t^T) Diag(a_t),    U_t = b_t k_t v_t^T
 *   HYPIC_SCALAR_DECAY   T_t = gamma_h I (RetNet),               U_t = k_t v_t^T
 *   HYPIC_UNGATED        T_t = I,                                U_t = k_t v_t^T
 *   HYPIC_DIAG_GATE      T_t = Diag(a_t) (GLA-type),             U_t = k_t v_t^T
 * Gates are passed as fp32 log-gates g (a = exp(g), gamma = exp(g)).
 * Value head h reads key head floor(h * h_k / h_v) (grouped heads).
 *
 * Conventions for every entry point:
 *   - Pointers marked [dev] are caller-owned device memory, [host] are host
 *     memory read during the call only.  The library allocates no device
 *     memory.  Two entry points keep process-wide state and serialise their
 *     host calls with a lock: hypic_segment_build_host and
 *     hypic_compose_host (copy streams and events per device and caller
 *     stream, created on first use) and
 *     hypic_segment_build_noalloc (a fixed device array); see each.  Every
 *     other entry point keeps no global mutable state and is thread-safe.
 *   - Work is enqueued asynchronously on the caller's stream.  Host-side
 *     validation runs first: an invalid descriptor returns an error code and
 *     launches nothing.  A failed launch returns HYPIC_ERR_CUDA.
 *   - Conditions found on the device (bounded wait expired, slot index out of
 *     range, non-finite output under HYPIC_FLAG_CHECK_FINITE) set bits of the
 *     optional device status word; read it after synchronising the stream and
 *     decode it with hypic_status_from_word().  The library never traps.
 *   - Results are deterministic: no atomics in any reduction; the order in
 *     which work is scheduled never changes a result bit.
 *   - Row-major layouts throughout; all state, transition and pair tensors
 *     are fp32.
 */
#ifndef HYPIC_H_
#define HYPIC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *hypic_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  HYPIC_OK = 0,
  HYPIC_ERR_INVALID_ARG = 1, /* bad descriptor: null/misaligned pointer, bad size, offsets not monotone */
  HYPIC_ERR_UNSUPPORTED = 2, /* valid but not supported (head size > 128, variant/dtype combination) */
  HYPIC_ERR_WORKSPACE = 3,   /* workspace missing or smaller than the *_workspace_bytes query */
  HYPIC_ERR_CUDA = 4,        /* a CUDA call failed (launch, copy, attribute) */
  HYPIC_ERR_TIMEOUT = 5,     /* device: a bounded wait ran out (reported through the status word) */
  HYPIC_ERR_NONFINITE = 6,   /* device: non-finite output seen (HYPIC_FLAG_CHECK_FINITE) */
  HYPIC_ERR_BAD_SLOT = 7     /* device: a pool slot index was out of range; that chain was skipped */
} hypic_status;

typedef enum {
  HYPIC_GDN = 0,
  HYPIC_DELTANET = 1,
  HYPIC_CHANNEL_DELTA = 2,
  HYPIC_SCALAR_DECAY = 3,
  HYPIC_UNGATED = 4,
  HYPIC_DIAG_GATE = 5
} hypic_variant;

typedef enum {
  HYPIC_IN_BF16 = 0, /* k/v/q bf16: tensor-core paths, max relative error 5e-3 per head */
  HYPIC_IN_F32 = 1   /* k/v/q fp32: fp32 paths, max relative error 1e-5 per head */
} hypic_in_dtype;

/* flags */
#define HYPIC_FLAG_CHECK_FINITE 1u /* scan outputs for NaN/Inf and report through the status word */
/* Build only, for measurement: hand the (segment, value head) items to the
 * SMs round-robin in segment order (CTA b takes items b, b + grid, ...)
 * instead of longest-first through the dynamic ticket.  The results are the
 * same bit for bit; only the schedule, and so the makespan, changes (pages
 * §2.3 compare LPT with round-robin). */
#define HYPIC_FLAG_ROUND_ROBIN 2u
/* Build, forward and compose: refuse (HYPIC_ERR_UNSUPPORTED, nothing
 * launched) a call whose inputs would send it to an fp32 CUDA-core kernel
 * instead of a tensor-core one, e.g. a 128-wide bf16 build whose k or v is
 * not 16-byte aligned, or a compose with h_v not a multiple of 4.  A call
 * with no tokens (build) or no segments (compose) has nothing to compute and
 * is not refused.  The hypic_*_path queries below tell the path up front. */
#define HYPIC_FLAG_REQUIRE_TENSOR_CORES 4u

/* The kernel family a call runs, as returned by the hypic_*_path queries. */
typedef enum {
  HYPIC_PATH_NONE = 0,         /* nothing to launch (no segment, layer or merge) */
  HYPIC_PATH_TC_CHUNKWISE = 1, /* build: tensor-core chunkwise, GDN / DeltaNet */
  HYPIC_PATH_TC_CHANNEL = 2,   /* build: tensor-core chunkwise, per-channel gate */
  HYPIC_PATH_TC_FAST = 3,      /* build: tensor-core fast path (scalar decay, ungated, diagonal) */
  HYPIC_PATH_F32_TOKEN = 4,    /* build / forward outputs: fp32 token recurrence, CUDA cores */
  HYPIC_PATH_TC_COMPOSE = 5,   /* compose: tensor cores (dense T, bf16 seam, d = 128) */
  HYPIC_PATH_F32_COMPOSE = 6,  /* compose: fp32, CUDA cores */
  HYPIC_PATH_TC_MERGE = 7,     /* merge: tensor cores, split tf32 */
  HYPIC_PATH_F32_MERGE = 8,    /* merge: fp32, CUDA cores */
  HYPIC_PATH_TC_FORWARD = 9    /* forward outputs: tensor cores, from the build's chunk records */
} hypic_path;

/* Compose only: compose the transitions alone.  Every seam write U_t and
 * every cached S(C|0) counts as zero (S_pool is not read and may be NULL;
 * seam_v is read but its values do not matter; seam_out is not written and
 * may be NULL), so the chain's final state is  T_{C_n} T_n,w .. T_n,1 ...
 * T_{C_1} T_1,w .. T_1,1 S_init: from the identity, the transition of the
 * whole run of segments (the T of a span, pages §2.1 composition rule and
 * §2.3 segment parallelism).  d_v must equal d_k; S_init NULL stands for the
 * identity in this mode (not for zero). */
#define HYPIC_FLAG_TRANSITION_ONLY 8u

/* Slot value that leaves a segment out of a build (see hypic_segment_build). */
#define HYPIC_SLOT_SKIP (-1)

/* Device status word bits (OR-ed by kernels; cleared by the caller). */
#define HYPIC_STATUS_TIMEOUT   1u
#define HYPIC_STATUS_NONFINITE 2u
#define HYPIC_STATUS_BAD_SLOT  4u

/* Shape of the transition stored in a pool slot for each variant:
 *   dense  (GDN, DELTANET, CHANNEL_DELTA): T_pool [n_slots, h_v, d_k, d_k]
 *   scalar (SCALAR_DECAY, UNGATED):        T_pool [n_slots, h_v]
 *   diag   (DIAG_GATE):                    T_pool [n_slots, h_v, d_k]
 * and always S_pool [n_slots, h_v, d_k, d_v]. */

/*
 * hypic_segment_build -- cache the pair (T_C, S(C|0)) of every segment and
 * value head (pages: the pair is stored at a segment's first prefill, §2.1).
 *
 * Segment i spans tokens [seg_offsets[i], seg_offsets[i+1]); its first seam_w
 * tokens form the seam window and are left out of the pair (§2.2), so the
 * pair covers the body [seg_offsets[i] + seam_w, seg_offsets[i+1]).  A body
 * that is empty gives (I, 0).  The pair of segment i goes to pool slot
 * slot_of_seg[i] (or slot i when slot_of_seg is NULL); a segment whose slot
 * is HYPIC_SLOT_SKIP is not built (a worker that builds its own share of
 * the segments of one prompt, pages §2.3, passes the whole prompt and skips
 * the others' segments).
 *
 * Work is split into (segment, value head) items packed over the SMs
 * longest-first (LPT), the single-GPU analogue of the pages' greedy LPT
 * balancing of segments over workers (§2.3).
 */
typedef struct {
  int32_t n_tokens, n_seg;
  int32_t h_k, h_v, d_k, d_v; /* 1 <= d_k, d_v <= 128; h_v a multiple of h_k */
  int32_t seam_w;             /* >= 0 */
  int32_t variant;            /* hypic_variant */
  int32_t in_dtype;           /* hypic_in_dtype */
  uint32_t flags;
  const void *k;              /* [dev] [n_tokens, h_k, d_k] bf16 or fp32 */
  const void *v;              /* [dev] [n_tokens, h_v, d_v] bf16 or fp32 */
  const float *g;             /* [dev] log-gates: GDN [n_tokens,h_v]; CHANNEL_DELTA/DIAG_GATE
                                 [n_tokens,h_v,d_k]; SCALAR_DECAY [h_v]; NULL otherwise */
  const float *beta;          /* [dev] [n_tokens, h_v] for the delta variants, NULL otherwise */
  const int64_t *seg_offsets; /* [host] [n_seg+1], non-decreasing, from 0 to n_tokens */
  const int32_t *slot_of_seg; /* [host] [n_seg] distinct slots in [0, n_slots) or HYPIC_SLOT_SKIP, or NULL */
  int64_t n_slots;
  float *T_pool;              /* [dev] see the shape note above */
  float *S_pool;              /* [dev] [n_slots, h_v, d_k, d_v] */
  void *workspace;            /* [dev] >= hypic_build_workspace_bytes(), 256-byte aligned */
  size_t workspace_bytes;
  uint32_t *status;           /* [dev] optional status word (may be NULL) */
} hypic_build_desc;

/* Workspace the build needs for this descriptor (shapes only are read). */
size_t hypic_build_workspace_bytes(const hypic_build_desc *d);
/* Returns a hypic_status; work is enqueued on `stream`. */
int hypic_segment_build(const hypic_build_desc *d, hypic_stream_t stream);

/*
 * hypic_segment_forward -- the prefill forward of the cached segments: the
 * build above (the same pairs, into the same pools) and, for every body
 * token t (the seam window excluded) of every segment and value head h, the
 * output of the zero-initial body state (pages §2.1: a segment's first
 * prefill is position independent, its state starting from zero),
 *   o_out[t, h] = S_t^T q_t,   S_t = T_t S_{t-1} + U_t,   S = 0 before the body,
 * with the post-update state, as for the seam outputs of hypic_compose.
 * q is [n_tokens, h_k, d_k] in the build's in_dtype (grouped heads as for k);
 * o_out is [n_tokens, h_v, d_v] fp32, its seam-token rows are not written.
 * The pairs come from the build's own kernels.  For GDN and DeltaNet with
 * bf16 inputs, d_k = d_v = 128 and 16-byte aligned k, v, q and o_out, the
 * outputs run on the tensor cores: the build also records every 64-token
 * chunk's start state S_0 and its Delta = U - W S_0 in the workspace, and a
 * second kernel forms each chunk's outputs from them,
 *   o_t = G_t S_0^T q_t + sum_{i<=t} e^(lam_t - lam_i) (q_t . k_i) Delta_i,
 * independently for every (chunk, value head).  Every other case runs the
 * fp32 token recurrence over the state columns (CUDA cores).  The workspace
 * is hypic_forward_workspace_bytes() (about 96 KiB per chunk and value head
 * on the tensor-core path; the build's plan otherwise); validation as for
 * hypic_segment_build.
 */
typedef struct {
  hypic_build_desc build;
  const void *q;   /* [dev] [n_tokens, h_k, d_k] */
  float *o_out;    /* [dev] [n_tokens, h_v, d_v] */
} hypic_forward_desc;

size_t hypic_forward_workspace_bytes(const hypic_forward_desc *d);
int hypic_segment_forward(const hypic_forward_desc *d, hypic_stream_t stream);

/*
 * hypic_segment_build_host -- hypic_segment_build from inputs in host memory
 * to pairs in host memory, with the copies overlapped with the build.  The
 * pages have no counterpart: this is the deployment form of the same build
 * (pages §2.1: the pair is cached at a segment's first prefill), with the
 * same pool contents bit for bit.
 *
 * d->build is a full hypic_segment_build descriptor whose [dev] buffers
 * (k, v, g, beta, T_pool, S_pool, workspace) the call fills and reads as
 * staging: k, v, g, beta are overwritten with the host inputs, the pool
 * slots of the segments are written by the build.  The host_* arrays have the
 * same shapes as their device counterparts; host_T / host_S mirror the whole
 * pools, and only the slots of the segments are written.  host_g / host_beta
 * are NULL exactly when build.g / build.beta are.
 *
 * The segments are split into min(n_chunks, n_seg, 64) groups of
 * consecutive segments with about equal token counts.  Per group, the token
 * range of k, v, g, beta is copied in on a copy stream of the library, the
 * build of the group runs on `stream` once those copies are done, and the
 * group's pool slots are copied out on a second copy stream once its build
 * is done; so group c's build overlaps group c+1's inputs and group c-1's
 * outputs.  All of it is ordered after the work already on `stream`, and
 * `stream` waits for the last copy out: the host arrays are complete once
 * `stream` is synchronised.  Overlap needs page-locked host arrays; pageable
 * ones give the same results with the copies serialised.
 *
 * Returns a hypic_status.  Every argument is checked before anything is
 * enqueued; a CUDA error while enqueuing returns HYPIC_ERR_CUDA with the
 * outputs undefined.  Host calls are serialised by a lock.  The copy streams
 * and their events belong to the caller's stream (up to eight caller streams
 * per device; beyond that they are shared), so host-buffer calls on
 * different streams overlap their copies and kernels.
 */
typedef struct {
  hypic_build_desc build;
  const void *host_k;     /* [host] as build.k */
  const void *host_v;     /* [host] as build.v */
  const float *host_g;    /* [host] as build.g */
  const float *host_beta; /* [host] as build.beta */
  float *host_T;          /* [host] as build.T_pool */
  float *host_S;          /* [host] as build.S_pool */
  int32_t n_chunks;       /* >= 1 */
} hypic_host_build_desc;

int hypic_segment_build_host(const hypic_host_build_desc *d, hypic_stream_t stream);

/*
 * hypic_segment_build_noalloc -- hypic_segment_build for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is a
 * deployment variant of the same build, with the same results bit for bit.
 *
 * d->workspace and d->workspace_bytes are ignored.  The work plan (a 64-byte
 * header, then 32 bytes per (segment, value head) pair) goes to a fixed
 * device array of HYPIC_NOALLOC_SCRATCH_BYTES (1 MiB) inside the library; its
 * address is looked up once per device, by the first call on that device.
 * The call allocates no device or heap memory (no cudaMalloc / cudaFree).
 * It runs the same checks and the same plan as hypic_segment_build.
 *
 * Limit: n_seg * h_v <= HYPIC_NOALLOC_MAX_PAIRS (the plan then fills the
 * array exactly); a larger problem returns HYPIC_ERR_WORKSPACE before any
 * CUDA call and launches nothing.
 *
 * Every call in the process shares the one array.  Calls ordered on the GPU
 * (one stream, or ordered by events) are safe; calls that overlap on the GPU
 * race on the array and give undefined results.  Host calls are serialised
 * by a lock.  The dynamic work counter is reset to zero by the plan copy that
 * opens each call.
 */
#define HYPIC_NOALLOC_SCRATCH_BYTES 1048576
#define HYPIC_NOALLOC_MAX_PAIRS 32766
int hypic_segment_build_noalloc(const hypic_build_desc *d, hypic_stream_t stream);

/*
 * hypic_compose -- rebuild the running state of every (layer, value head)
 * from cached pairs in prompt order (pages §2.1 composition rule, §2.2 seam):
 *   S <- S_init (or 0)
 *   for segment i = 0 .. n_seg-1:
 *     for each seam token t of segment i:  S <- T_t S + U_t,  o_t = S^T q_t
 *     S <- T_{C_i} S + S(C_i|0)             (pair from pool slot slot[l, i])
 * Every segment has exactly seam_w seam tokens; a segment with fewer real
 * tokens passes identity tokens (k = v = q = 0, g = 0, beta = 0) in the rest,
 * whose outputs carry no meaning.
 */
typedef struct {
  int32_t n_layers, n_seg;
  int32_t h_k, h_v, d_k, d_v;
  int32_t seam_w;
  int32_t variant, in_dtype;
  uint32_t flags;
  const int32_t *slot;        /* [dev] [n_layers, n_seg] pool slot per (layer, segment) */
  int64_t n_slots;
  const float *T_pool;        /* [dev] as written by hypic_segment_build */
  const float *S_pool;        /* [dev] */
  const void *seam_k;         /* [dev] [n_layers, n_seg, seam_w, h_k, d_k] bf16 or fp32 */
  const void *seam_v;         /* [dev] [n_layers, n_seg, seam_w, h_v, d_v] */
  const void *seam_q;         /* [dev] [n_layers, n_seg, seam_w, h_k, d_k] */
  const float *seam_g;        /* [dev] GDN [L,n_seg,w,h_v]; CHANNEL/DIAG [L,n_seg,w,h_v,d_k];
                                 SCALAR_DECAY [n_layers, h_v]; NULL otherwise */
  const float *seam_beta;     /* [dev] [L, n_seg, w, h_v] for the delta variants, else NULL */
  const float *S_init;        /* [dev] [n_layers, h_v, d_k, d_v] or NULL (= 0) */
  float *S_out;               /* [dev] [n_layers, h_v, d_k, d_v]; may alias S_init */
  float *seam_out;            /* [dev] [n_layers, n_seg, seam_w, h_v, d_v] (NULL if seam_w = 0) */
  void *workspace;            /* [dev] >= hypic_compose_workspace_bytes() */
  size_t workspace_bytes;
  uint32_t *status;           /* [dev] optional */
  int32_t seg_stride;         /* segments per layer in slot, seam_* and seam_out (0: n_seg); with
                                 pointers advanced by a segments, n_seg = b - a composes the span
                                 [a, b) of longer per-layer arrays in place */
} hypic_compose_desc;

size_t hypic_compose_workspace_bytes(const hypic_compose_desc *d);
int hypic_compose(const hypic_compose_desc *d, hypic_stream_t stream);

/*
 * hypic_compose_host -- hypic_compose from seam tokens in host memory to
 * states and seam outputs in host memory, the cached pairs resident on the
 * device, with the copies overlapped with the compose.  The pages have no
 * counterpart: this is the deployment form of the same compose (pages §2.1
 * composition rule, §2.2 seam window), with the same results bit for bit.
 *
 * d->compose is a full hypic_compose descriptor whose [dev] seam arrays
 * (seam_k, seam_v, seam_q, seam_g, seam_beta), S_init, S_out and seam_out the
 * call uses as staging: the seam arrays (and S_init, when host_S_init is
 * given) are overwritten with the host inputs.  The host_* arrays have the
 * shapes of their device counterparts and are NULL exactly when those are;
 * host_S_out and host_seam_out (NULL when seam_w = 0) receive the results.
 *
 * The layers are split into min(n_chunks, n_layers, 64, W) groups of
 * consecutive layers, W the number of waves the n_layers x h_v chains take
 * on the device (two chains per SM), so that no group's launch runs a
 * partial wave for nothing.  Per group, the group's seam tokens (and initial
 * states) are copied in on a copy stream of the library, its compose runs
 * on `stream` once they are in, and its states and seam outputs are copied
 * out on a second copy stream once it is done; so group c's compose
 * overlaps group c+1's inputs and group c-1's outputs.  Everything is ordered
 * after the work already on `stream`, and `stream` waits for the last copy
 * out: the host arrays are complete once `stream` is synchronised.  Overlap
 * needs page-locked host arrays.  Returns a hypic_status; every argument is
 * checked first.  Host calls are serialised by a lock; the copy streams and
 * events belong to the caller's stream, as for hypic_segment_build_host (a
 * build and a compose from host buffers on two streams overlap).
 */
typedef struct {
  hypic_compose_desc compose;
  const void *host_seam_k, *host_seam_v, *host_seam_q; /* [host] as compose.seam_* */
  const float *host_seam_g, *host_seam_beta;           /* [host] */
  const float *host_S_init;                             /* [host] or NULL (then compose.S_init is read as is) */
  float *host_S_out;                                    /* [host] [n_layers, h_v, d_k, d_v] */
  float *host_seam_out;                                 /* [host] [n_layers, n_seg, seam_w, h_v, d_v] */
  int32_t n_chunks;                                     /* >= 1 */
} hypic_host_compose_desc;

int hypic_compose_host(const hypic_host_compose_desc *d, hypic_stream_t stream);

/*
 * hypic_span_scan -- the start state of every span of compose chains split
 * into n_spans consecutive spans of segments (pages §2.3 segment
 * parallelism, combined by the §2.1 composition rule): with the pair
 * (T_s, S_s) of span s of layer l (T_s from hypic_compose with
 * HYPIC_FLAG_TRANSITION_ONLY, S_s from hypic_compose from a zero state),
 *   S_start[0, l] = S_init[l] (or 0),
 *   S_start[s, l] = T_{s-1} S_start[s-1, l] + S_{s-1}      (s = 1 .. n_spans-1)
 * for every value head, an exclusive scan over the spans.  Span-major
 * layouts: T_span [n_spans, n_layers, h_v, d_k, d_k], S_span and S_start
 * [n_spans, n_layers, h_v, d_k, d_v], S_init [n_layers, h_v, d_k, d_v], all
 * fp32 device memory; S_start must not overlap the inputs.  Each step is one
 * hypic_compose launch of one pair per chain (tensor cores where
 * hypic_compose takes them), so n_spans - 1 launches.  The workspace holds
 * the slot indices (hypic_span_scan_workspace_bytes).  Returns a
 * hypic_status; device conditions go to the status word as for compose.
 */
typedef struct {
  int32_t n_layers, n_spans;
  int32_t h_v, d_k, d_v;
  const float *T_span;   /* [dev] */
  const float *S_span;   /* [dev] */
  const float *S_init;   /* [dev] or NULL (= 0) */
  float *S_start;        /* [dev] */
  void *workspace;       /* [dev] >= hypic_span_scan_workspace_bytes(), 256-byte aligned */
  size_t workspace_bytes;
  uint32_t *status;      /* [dev] optional */
} hypic_span_scan_desc;

size_t hypic_span_scan_workspace_bytes(const hypic_span_scan_desc *d);
int hypic_span_scan(const hypic_span_scan_desc *d, hypic_stream_t stream);

/*
 * hypic_compose_spans -- hypic_compose computed by segment parallelism on
 * one GPU (pages §2.3): the n_seg segments of every chain are split into
 * n_spans consecutive spans at span_bounds (host, [n_spans + 1], from 0 to
 * n_seg, non-decreasing); each span's pair comes from two composes of its
 * segments alone (its S from zero, its T with HYPIC_FLAG_TRANSITION_ONLY),
 * hypic_span_scan gives every span its start state, and each span is then
 * composed from that state, writing its seam outputs; the last span's final
 * state is S_out.  The results equal hypic_compose's within its accuracy.
 * On several GPUs each worker runs one span and only the span pairs are
 * exchanged (one (T, S) per layer, head and span); this entry point runs the
 * spans one after another and serves as the single-GPU form and reference.
 * `d` is an ordinary compose descriptor (d_v = d_k, no transition-only
 * flag); the workspace (hypic_compose_spans_workspace_bytes) holds the span
 * pairs, start states and slot indices, about
 * 3 * n_spans * n_layers * h_v * d_k * d_k * 4 bytes.
 */
size_t hypic_compose_spans_workspace_bytes(const hypic_compose_desc *d, int32_t n_spans);
int hypic_compose_spans(const hypic_compose_desc *d, int32_t n_spans, const int32_t *span_bounds,
                        hypic_stream_t stream);

/*
 * hypic_pair_merge -- merge cached pairs of adjacent spans (pages §2.1: the
 * composition rule applied to two segments, S(C1.C2) = T(C2) S(C1) + S(C2),
 * with the transition of the joined span T(C1.C2) = T(C2) T(C1)):
 *   for each merge m and value head h, with a = later[m], b = earlier[m],
 *   o = out[m] (pool slots):
 *     T_out[o, h] = T_a[a, h] T_b[b, h]
 *     S_out[o, h] = T_a[a, h] S_b[b, h] + S_a[a, h]
 * The later pairs come from pool (T_a, S_a), the earlier ones from pool
 * (T_b, S_b); the two may be the same pool.  The merge is associative, so
 * repeated merges build the pair of any run of consecutive spans (a tree of
 * merges composes a chain in log depth).
 * T layouts follow the variant as in hypic_segment_build: dense
 * [slots, h_v, d_k, d_k] for GDN / DELTANET / CHANNEL_DELTA (matrix
 * product), [slots, h_v] for SCALAR_DECAY / UNGATED (scalar product),
 * [slots, h_v, d_k] for DIAG_GATE (elementwise product; S rows scaled).
 * S pools are [slots, h_v, d_k, d_v].  All fp32.
 * A merge with a slot out of range of its pool (n_slots_a, n_slots_b,
 * n_slots_out) is skipped and reported (HYPIC_STATUS_BAD_SLOT).  Output
 * slots must be distinct, and no output slot of a call may alias an input
 * slot of the same call (results are undefined otherwise).
 * Dense d_k = d_v = 128 runs on the tensor cores with split tf32 operands
 * (about fp32 accuracy); other shapes and the scalar / diagonal forms run on
 * the CUDA cores in fp32.
 */
typedef struct {
  int32_t n_merge;
  int32_t h_v, d_k, d_v;
  int32_t variant;
  const int32_t *later;       /* [dev] [n_merge] slot of the later pair (T2, S2) in pool a */
  const int32_t *earlier;     /* [dev] [n_merge] slot of the earlier pair (T1, S1) in pool b */
  const int32_t *out;         /* [dev] [n_merge] output slot */
  int64_t n_slots_a, n_slots_b, n_slots_out;
  const float *T_a, *S_a;     /* [dev] pool of the later pairs */
  const float *T_b, *S_b;     /* [dev] pool of the earlier pairs */
  float *T_out, *S_out;       /* [dev] output pool */
  uint32_t *status;           /* [dev] optional */
} hypic_merge_desc;

int hypic_pair_merge(const hypic_merge_desc *d, hypic_stream_t stream);

/*
 * hypic_pair_rerotate -- state re-rotation of cached pairs for segments that
 * are reused at a shifted position (pages §2.1, last paragraph: for variants
 * with RoPE the cached state is re-rotated; the pages give no formula).
 * Reading used: rotary position embedding multiplies every key by block-
 * diagonal 2 x 2 rotations, pair i turning by (position x theta_i) with
 * theta_i = base^(-2i / rot_dim), i < rot_dim / 2.  A segment moved by delta
 * positions therefore has all its keys multiplied by R(delta); every token
 * transition of a scalar-gated variant becomes R T_t R^T and every write
 * R U_t, so for item m (i = slot_in[m], o = slot_out[m], R = R(delta[m])):
 *   T_out[o, h] = R T_in[i, h] R^T,   S_out[o, h] = R S_in[i, h]
 * for every value head h.  Channel pairs are (2i, 2i + 1) for
 * HYPIC_ROPE_INTERLEAVED and (i, i + rot_dim / 2) for HYPIC_ROPE_HALF;
 * channels >= rot_dim are not rotated.  rot_dim is even, 2 <= rot_dim <= d_k
 * (HYPIC_ROPE_HALF: a multiple of 8).
 * Variants: GDN and DELTANET (dense T [slots, h_v, d_k, d_k]); SCALAR_DECAY
 * and UNGATED (scalar T [slots, h_v], copied unchanged).  Per-channel and
 * diagonal gates do not commute with R, so the patch is not exact for them:
 * HYPIC_ERR_UNSUPPORTED.  S pools are [slots, h_v, d_k, d_v]; all fp32;
 * d_k and d_v are multiples of 4, at most 128.
 * The angles are formed in fp64 (exact for |delta| < 2^53), the rotation in
 * fp32.  slot_out[m] may equal slot_in[m] in the same pool (in place): each
 * (slot, head) block is read whole before it is written.  Items must not
 * share an output slot, nor read a slot that another item of the call
 * writes (results are undefined otherwise).  An item with a slot out of
 * range is skipped and reported (HYPIC_STATUS_BAD_SLOT).
 */
typedef enum { HYPIC_ROPE_INTERLEAVED = 0, HYPIC_ROPE_HALF = 1 } hypic_rope_layout;

typedef struct {
  int32_t n_items;
  int32_t h_v, d_k, d_v;
  int32_t variant;
  int32_t rot_dim;
  int32_t layout;             /* hypic_rope_layout */
  double base;                /* > 0 (10000 in the common RoPE setting) */
  const int32_t *slot_in;     /* [dev] [n_items] pair to re-rotate */
  const int32_t *slot_out;    /* [dev] [n_items] where the result goes */
  const int64_t *delta;       /* [dev] [n_items] position shift (new start - cached start) */
  int64_t n_slots_in, n_slots_out;
  const float *T_in, *S_in;   /* [dev] input pool */
  float *T_out, *S_out;       /* [dev] output pool (may be the input pool) */
  uint32_t *status;           /* [dev] optional */
} hypic_rerotate_desc;

int hypic_pair_rerotate(const hypic_rerotate_desc *d, hypic_stream_t stream);

/*
 * hypic_plan_lpt -- greedy longest-processing-time-first packing of items
 * over workers (pages §2.3: LPT balancing of segments over scatter workers).
 * Items are taken in order of decreasing cost (ties: lower index first) and
 * each goes to the currently least-loaded worker (ties: lower worker index).
 * Host-only.  order_out [n_items] receives the item order, worker_out
 * [n_items] (may be NULL) the worker of each item (indexed by item), and
 * *makespan_out (may be NULL) the largest worker load.
 */
int hypic_plan_lpt(const int64_t *costs, int32_t n_items, int32_t n_workers, int32_t *order_out,
                   int32_t *worker_out, int64_t *makespan_out);

/*
 * Path queries: the hypic_path the matching call would run for this
 * descriptor (the same predicates the dispatch uses: variant, dtype, head
 * sizes, h_v, pointer alignment), or minus a hypic_status when the shapes are
 * invalid.  Host-only; nothing is read from device memory and nothing is
 * launched.  hypic_forward_path reports the kernel of the per-token outputs
 * (its pairs come from the hypic_build_path kernel).
 */
int hypic_build_path(const hypic_build_desc *d);
int hypic_forward_path(const hypic_forward_desc *d);
int hypic_compose_path(const hypic_compose_desc *d);
int hypic_merge_path(const hypic_merge_desc *d);

/* Decode a device status word into the first hypic_status it reports. */
int hypic_status_from_word(uint32_t word);
const char *hypic_status_string(int status);
/* Library version: major * 10000 + minor * 100 + patch. */
int hypic_version(void);

#ifdef __cplusplus
}
#endif
#endif /* HYPIC_H_ */
