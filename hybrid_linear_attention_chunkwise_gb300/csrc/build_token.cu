// build_token.cu -- fp32 token-recurrence segment build (all six variants).
//
// The fp32-input path of hypic_segment_build: for each (segment, value head)
// item it applies the per-token transitions in order,
//     T <- T_t T,   S <- T_t S + U_t,
// which is the definition of the cached pair (T_C, S(C|0)) on the HYPIC news
// pages (nav.aitube.vip §2.1: T_C is the product of all token transition
// matrices of the segment; S(C|0) the final state from zero).
//
// Layout on chip: the augmented block X = [T | S] (d_k x (d_k + d_v)) is held
// one column per thread, in registers (DK fp32 values per thread), so the
// rank-1 erase  X <- a (X - b k (k^T X)) + [0 | b k v^T]  needs only a local
// dot product per column: no cross-thread reduction.  Token inputs are staged
// through shared memory in tiles of TB tokens (broadcast reads).  Variants
// without an erase (scalar decay, ungated, diagonal gate) carry no T columns:
// their T is a product of gates, formed from fp64 sums of the log-gates.
//
// Items are pulled from the LPT-ordered plan by an atomic ticket (dynamic
// list scheduling in LPT order); an item's result does not depend on which
// block computes it.
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "common.cuh"

namespace hypic {

namespace {

__device__ __forceinline__ void tc_named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

constexpr int TB = 16;  // tokens per shared-memory tile

// Ampere-style asynchronous copies into shared memory (16 bytes bypassing
// L1, or 4 bytes), completed per thread by a group wait
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

template <int DK>
struct TokSmem {
  float k[TB][DK];    // k (zero beyond d_k / past the end)
  float kd[TB][DK];   // vector gates: k * a (the erase acts after Diag(a)); else unused
  float a[TB][DK];    // vector gates: a = exp(g); else unused
  float lg[TB][DK];   // vector gates: g (for the log-sum of diagonal T)
  float v[TB][128];
  float gs[TB];       // scalar gate a_t (GDN) / 1
  float b[TB];        // beta_t (0 on padding tokens)
  int item;
};

template <int DK>
__global__ void __launch_bounds__(256) build_token_kernel(BuildParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TokSmem<DK> &sm = *reinterpret_cast<TokSmem<DK> *>(smem_raw);
  const int tid = threadIdx.x;
  const bool delta = is_delta(p.variant);
  const bool vec = is_vector_gate(p.variant);
  const int d_k = p.d_k, d_v = p.d_v;
  const int n_t_thr = delta ? DK : 0;              // threads [0, DK) own T columns
  const bool is_T = tid < n_t_thr;
  const int col = is_T ? tid : tid - n_t_thr;      // column within T or S
  const bool active = is_T ? (col < d_k) : (col < d_v);
  const int n_items = p.plan->n_items;

  for (;;) {
    if (tid == 0) sm.item = atomicAdd(&p.plan->ticket, 1);
    __syncthreads();
    const int idx = sm.item;
    __syncthreads();
    if (idx >= n_items) break;
    const BuildItem it = p.items[idx];
    const int h = it.head;
    const int kh = (int)(((int64_t)h * p.h_k) / p.h_v);

    float X[DK];
#pragma unroll
    for (int i = 0; i < DK; i++) X[i] = (is_T && i == col) ? 1.f : 0.f;
    double logsum = 0.0;  // non-delta variants: sum of log-gates of channel `tid`

    float gconst = 1.f;
    if (p.variant == HYPIC_SCALAR_DECAY) gconst = expf(p.g[h]);

    for (int64_t t0 = it.start; t0 < it.end; t0 += TB) {
      const int nt = (int)((it.end - t0) < TB ? (it.end - t0) : TB);
      for (int e = tid; e < TB * DK; e += blockDim.x) {
        const int t = e / DK, i = e % DK;
        float kv = 0.f, a = 1.f, lg = 0.f;
        if (t < nt && i < d_k) {
          kv = load_in(p.k, ((t0 + t) * p.h_k + kh) * (int64_t)d_k + i, p.in_dtype);
          if (vec) {
            lg = p.g[((t0 + t) * p.h_v + h) * (int64_t)d_k + i];
            a = expf(lg);
          }
        }
        sm.k[t][i] = kv;
        if (vec) {
          sm.a[t][i] = a;
          sm.kd[t][i] = kv * a;
          sm.lg[t][i] = lg;
        }
      }
      for (int e = tid; e < TB * 128; e += blockDim.x) {
        const int t = e / 128, j = e % 128;
        sm.v[t][j] = (t < nt && j < d_v) ? load_in(p.v, ((t0 + t) * p.h_v + h) * (int64_t)d_v + j, p.in_dtype) : 0.f;
      }
      for (int t = tid; t < TB; t += blockDim.x) {
        float gs = 1.f, b = 0.f;
        if (t < nt) {
          if (p.variant == HYPIC_GDN) gs = expf(p.g[(t0 + t) * p.h_v + h]);
          else if (p.variant == HYPIC_SCALAR_DECAY) gs = gconst;
          if (delta) b = p.beta[(t0 + t) * p.h_v + h];
        }
        sm.gs[t] = gs;
        sm.b[t] = b;
      }
      __syncthreads();
      if (!delta && vec && tid < d_k) {
        for (int t = 0; t < nt; t++) logsum += (double)sm.lg[t][tid];
      }
      if (active) {
        for (int t = 0; t < nt; t++) {
          const float b = sm.b[t], gs = sm.gs[t];
          const float vj = is_T ? 0.f : sm.v[t][col];
          if (delta) {
            const float *kd = vec ? sm.kd[t] : sm.k[t];
            float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
#pragma unroll
            for (int i = 0; i < DK; i += 4) {
              x0 = fmaf(kd[i + 0], X[i + 0], x0);
              x1 = fmaf(kd[i + 1], X[i + 1], x1);
              x2 = fmaf(kd[i + 2], X[i + 2], x2);
              x3 = fmaf(kd[i + 3], X[i + 3], x3);
            }
            const float x = (x0 + x1) + (x2 + x3);
            // X <- s (X - b k x) + b k v  with s = a_t (GDN), 1, or Diag(a) applied first
            const float c = vec ? (b * vj - b * x) : (gs * (-b * x) + b * vj);
            const float *kk = sm.k[t];
            if (vec) {
              const float *aa = sm.a[t];
#pragma unroll
              for (int i = 0; i < DK; i++) X[i] = fmaf(aa[i], X[i], kk[i] * c);
            } else {
#pragma unroll
              for (int i = 0; i < DK; i++) X[i] = fmaf(gs, X[i], kk[i] * c);
            }
          } else {
            const float *kk = sm.k[t];
            if (vec) {
              const float *aa = sm.a[t];
#pragma unroll
              for (int i = 0; i < DK; i++) X[i] = fmaf(aa[i], X[i], kk[i] * vj);
            } else {
#pragma unroll
              for (int i = 0; i < DK; i++) X[i] = fmaf(gs, X[i], kk[i] * vj);
            }
          }
        }
      }
      __syncthreads();
    }

    // epilogue: write the pair into the pool slot
    const int64_t sh = (int64_t)it.slot * p.h_v + h;
    bool bad = false;
    if (active) {
      if (is_T) {
        float *T = p.T_pool + sh * d_k * d_k;
#pragma unroll
        for (int i = 0; i < DK; i++)
          if (i < d_k) {
            T[(int64_t)i * d_k + col] = X[i];
            bad |= !finite_f(X[i]);
          }
      } else {
        float *S = p.S_pool + sh * d_k * d_v;
#pragma unroll
        for (int i = 0; i < DK; i++)
          if (i < d_k) {
            S[(int64_t)i * d_v + col] = X[i];
            bad |= !finite_f(X[i]);
          }
      }
    }
    if (!delta) {
      const int64_t L = it.end - it.start;
      if (p.variant == HYPIC_DIAG_GATE) {
        if (tid < d_k) {
          float tv = (float)exp(logsum);
          p.T_pool[sh * d_k + tid] = tv;
          bad |= !finite_f(tv);
        }
      } else if (tid == 0) {
        float tv = (p.variant == HYPIC_SCALAR_DECAY) ? (float)exp((double)L * (double)p.g[h]) : 1.f;
        p.T_pool[sh] = tv;
        bad |= !finite_f(tv);
      }
    }
    if ((p.flags & HYPIC_FLAG_CHECK_FINITE) && bad) report(p.status, HYPIC_STATUS_NONFINITE);
  }
}

template <int DK>
cudaError_t launch_dk(const BuildParams &p, int n_items, int n_sm, cudaStream_t s) {
  const bool delta = is_delta(p.variant);
  const int dvp = ((p.d_v + 31) / 32) * 32;
  int threads = (delta ? DK : 0) + dvp;
  const int dkp = ((p.d_k + 31) / 32) * 32;
  if (threads < dkp) threads = dkp;  // diagonal gates: one thread per channel for the log-sum
  threads = ((threads + 31) / 32) * 32;
  const size_t smem = sizeof(TokSmem<DK>);
  cudaError_t e = cudaFuncSetAttribute(build_token_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, build_token_kernel<DK>, threads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  int grid = n_sm * per_sm;
  if (grid > n_items) grid = n_items;
  if (grid < 1) return cudaSuccess;
  build_token_kernel<DK><<<grid, threads, smem, s>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// The outputs of the prefill forward (hypic_segment_forward): for every body
// token of every item, o_t = S_t^T q_t from the zero-initial body state, by
// the same token recurrence over the S columns only (the pairs come from the
// build kernels).  Each column is split over two threads, rows 0..DK/2-1 and
// DK/2..DK-1 (threads col and col + DVP, in warps w and w + DVP/32), so a
// column holds DK/2 registers per thread and twice as many warps fit an SM;
// the halves exchange their partial dot products through shared memory
// under a 64-thread barrier of their own (one per token), the lower half
// writing the output of a token after the next barrier.
// ---------------------------------------------------------------------------
template <int DK>
struct FwdSmem {
  TokSmem<DK> t;
  alignas(16) float q[TB][DK];  // rows read 16 bytes a time
  float xs[2][2][128];  // partial k^T S of the two halves, by token parity
  float os[2][128];     // partial q^T S of the upper half, by token parity
};
// every row read by 16-byte loads starts on a 16-byte boundary (and so does
// each half row: DK / 2 floats is a multiple of 4)
template <int DK>
constexpr bool fwd_rows_aligned() {
  return offsetof(FwdSmem<DK>, q) % 16 == 0 && offsetof(TokSmem<DK>, k) % 16 == 0 &&
         offsetof(TokSmem<DK>, kd) % 16 == 0 && offsetof(TokSmem<DK>, a) % 16 == 0 && (DK * 4) % 16 == 0 &&
         (DK / 2) % 4 == 0;
}
static_assert(fwd_rows_aligned<16>() && fwd_rows_aligned<32>() && fwd_rows_aligned<64>() && fwd_rows_aligned<128>(),
              "16-byte shared-memory rows");

// One stage of raw (input-dtype) token inputs for a tile, copied ahead by
// cp.async: k and q rows (DK elements apart), v rows (128 apart), the gate
// (a row of d_k floats per token for vector gates, else one float) and beta.
// Every part starts on a 16-byte boundary.
struct FwdRaw {
  int k, q, v, g, b, bytes;
};
__host__ __device__ inline FwdRaw fwd_raw_layout(int DK, int es, bool vec) {
  FwdRaw r;
  r.k = 0;
  r.q = TB * DK * es;
  r.v = 2 * TB * DK * es;
  r.g = r.v + TB * 128 * es;
  r.b = r.g + (vec ? TB * DK * 4 : TB * 4);
  r.bytes = r.b + TB * 4;
  return r;
}
template <int DK>
__host__ __device__ constexpr size_t fwd_raw_offset() {
  return (sizeof(FwdSmem<DK>) + 15) / 16 * 16;
}

template <int DK>
__global__ void __launch_bounds__(256) forward_out_kernel(BuildParams p, int dvp, int async_tiles) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  FwdSmem<DK> &fs = *reinterpret_cast<FwdSmem<DK> *>(smem_raw);
  TokSmem<DK> &sm = fs.t;
  constexpr int HALF = DK / 2;
  const int tid = threadIdx.x;
  const bool delta = is_delta(p.variant);
  const bool vec = is_vector_gate(p.variant);
  const int d_k = p.d_k, d_v = p.d_v;
  const int hf = tid / dvp, col = tid % dvp, r0 = hf * HALF;
  const bool active = col < d_v;
  const int bar = 1 + col / 32;  // the pair of warps holding this column
  const int n_items = p.plan->n_items;
  const int es = p.in_dtype == HYPIC_IN_BF16 ? 2 : 4;
  const FwdRaw lay = fwd_raw_layout(DK, es, vec);
  unsigned char *raw = smem_raw + fwd_raw_offset<DK>();  // two stages when async_tiles

  for (;;) {
    if (tid == 0) sm.item = atomicAdd(&p.plan->ticket, 1);
    __syncthreads();
    const int idx = sm.item;
    __syncthreads();
    if (idx >= n_items) break;
    const BuildItem it = p.items[idx];
    const int h = it.head;
    const int kh = (int)(((int64_t)h * p.h_k) / p.h_v);
    float X[HALF];
#pragma unroll
    for (int i = 0; i < HALF; i++) X[i] = 0.f;
    float gconst = 1.f;
    if (p.variant == HYPIC_SCALAR_DECAY) gconst = expf(p.g[h]);
    uint32_t u = 0;       // tokens so far: parity of the exchange buffers
    int64_t pend = -1;    // lower half: token whose output waits for the upper half's partial
    float opend = 0.f;
    // X <- Diag(a) X + k c (per-channel gate) or gs X + k c, 16 bytes a time
    auto update = [&](int t, float c) {
      const float *kk = sm.k[t] + r0;
      if (vec) {
        const float *aa = sm.a[t] + r0;
#pragma unroll
        for (int i = 0; i < HALF; i += 4) {
          const float4 kv = *reinterpret_cast<const float4 *>(kk + i);
          const float4 av = *reinterpret_cast<const float4 *>(aa + i);
          X[i + 0] = fmaf(av.x, X[i + 0], kv.x * c);
          X[i + 1] = fmaf(av.y, X[i + 1], kv.y * c);
          X[i + 2] = fmaf(av.z, X[i + 2], kv.z * c);
          X[i + 3] = fmaf(av.w, X[i + 3], kv.w * c);
        }
      } else {
        const float gs = sm.gs[t];
#pragma unroll
        for (int i = 0; i < HALF; i += 4) {
          const float4 kv = *reinterpret_cast<const float4 *>(kk + i);
          X[i + 0] = fmaf(gs, X[i + 0], kv.x * c);
          X[i + 1] = fmaf(gs, X[i + 1], kv.y * c);
          X[i + 2] = fmaf(gs, X[i + 2], kv.z * c);
          X[i + 3] = fmaf(gs, X[i + 3], kv.w * c);
        }
      }
    };
    auto flush = [&]() {
      if (hf == 0 && pend >= 0 && active)
        p.o_out[(pend * p.h_v + h) * (int64_t)d_v + col] = opend + fs.os[(u - 1) & 1][col];
      pend = -1;
    };

    // raw inputs of the tile at t0 (nt tokens) into stage st, by cp.async
    auto issue_tile = [&](int64_t t0, int nt, int st) {
      unsigned char *base = raw + st * lay.bytes;
      const int ck = d_k * es / 16, cv = d_v * es / 16;
      const char *kb = static_cast<const char *>(p.k), *qb = static_cast<const char *>(p.q);
      const char *vb = static_cast<const char *>(p.v);
      for (int e = tid; e < nt * ck; e += blockDim.x) {
        const int t = e / ck, c = e % ck;
        const int64_t src = ((t0 + t) * p.h_k + kh) * (int64_t)d_k * es + 16 * c;
        cp_async16(base + lay.k + t * DK * es + 16 * c, kb + src);
        cp_async16(base + lay.q + t * DK * es + 16 * c, qb + src);
      }
      for (int e = tid; e < nt * cv; e += blockDim.x) {
        const int t = e / cv, c = e % cv;
        cp_async16(base + lay.v + t * 128 * es + 16 * c, vb + ((t0 + t) * p.h_v + h) * (int64_t)d_v * es + 16 * c);
      }
      if (vec) {
        const int cg = d_k / 4;
        for (int e = tid; e < nt * cg; e += blockDim.x) {
          const int t = e / cg, c = e % cg;
          cp_async16(base + lay.g + (t * DK + 4 * c) * 4, p.g + ((t0 + t) * p.h_v + h) * (int64_t)d_k + 4 * c);
        }
      } else if (p.variant == HYPIC_GDN) {
        for (int t = tid; t < nt; t += blockDim.x) cp_async4(base + lay.g + 4 * t, p.g + (t0 + t) * p.h_v + h);
      }
      if (delta)
        for (int t = tid; t < nt; t += blockDim.x) cp_async4(base + lay.b + 4 * t, p.beta + (t0 + t) * p.h_v + h);
      cp_async_commit();
    };
    auto raw_in = [&](const unsigned char *b, int i) -> float {
      return es == 2 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(b)[i])
                     : reinterpret_cast<const float *>(b)[i];
    };
    const int64_t first_nt = (it.end - it.start) < TB ? (it.end - it.start) : TB;
    if (async_tiles && first_nt > 0) issue_tile(it.start, (int)first_nt, 0);

    int ti = 0;
    for (int64_t t0 = it.start; t0 < it.end; t0 += TB, ti++) {
      const int nt = (int)((it.end - t0) < TB ? (it.end - t0) : TB);
      if (async_tiles) {
        cp_async_wait_all();
        __syncthreads();  // this tile's raw inputs visible to all threads
        const unsigned char *base = raw + (ti & 1) * lay.bytes;
        for (int e = tid; e < TB * DK; e += blockDim.x) {
          const int t = e / DK, i = e % DK;
          float kv = 0.f, qv = 0.f, a = 1.f;
          if (t < nt && i < d_k) {
            kv = raw_in(base + lay.k, t * DK + i);
            qv = raw_in(base + lay.q, t * DK + i);
            if (vec) a = expf(reinterpret_cast<const float *>(base + lay.g)[t * DK + i]);
          }
          sm.k[t][i] = kv;
          fs.q[t][i] = qv;
          if (vec) {
            sm.a[t][i] = a;
            sm.kd[t][i] = kv * a;
          }
        }
        for (int e = tid; e < TB * 128; e += blockDim.x) {
          const int t = e / 128, j = e % 128;
          sm.v[t][j] = (t < nt && j < d_v) ? raw_in(base + lay.v, t * 128 + j) : 0.f;
        }
        for (int t = tid; t < TB; t += blockDim.x) {
          float gs = 1.f, b = 0.f;
          if (t < nt) {
            if (p.variant == HYPIC_GDN) gs = expf(reinterpret_cast<const float *>(base + lay.g)[t]);
            else if (p.variant == HYPIC_SCALAR_DECAY) gs = gconst;
            if (delta) b = reinterpret_cast<const float *>(base + lay.b)[t];
          }
          sm.gs[t] = gs;
          sm.b[t] = b;
        }
        // the next tile's copies run under this tile's recurrence; its stage
        // was last read by the conversion of the previous tile, which every
        // thread finished before the barrier above
        if (t0 + TB < it.end) {
          const int64_t rest = it.end - (t0 + TB);
          issue_tile(t0 + TB, (int)(rest < TB ? rest : TB), (ti + 1) & 1);
        }
      } else {
        for (int e = tid; e < TB * DK; e += blockDim.x) {
          const int t = e / DK, i = e % DK;
          float kv = 0.f, qv = 0.f, a = 1.f;
          if (t < nt && i < d_k) {
            kv = load_in(p.k, ((t0 + t) * p.h_k + kh) * (int64_t)d_k + i, p.in_dtype);
            qv = load_in(p.q, ((t0 + t) * p.h_k + kh) * (int64_t)d_k + i, p.in_dtype);
            if (vec) a = expf(p.g[((t0 + t) * p.h_v + h) * (int64_t)d_k + i]);
          }
          sm.k[t][i] = kv;
          fs.q[t][i] = qv;
          if (vec) {
            sm.a[t][i] = a;
            sm.kd[t][i] = kv * a;
          }
        }
        for (int e = tid; e < TB * 128; e += blockDim.x) {
          const int t = e / 128, j = e % 128;
          sm.v[t][j] = (t < nt && j < d_v) ? load_in(p.v, ((t0 + t) * p.h_v + h) * (int64_t)d_v + j, p.in_dtype) : 0.f;
        }
        for (int t = tid; t < TB; t += blockDim.x) {
          float gs = 1.f, b = 0.f;
          if (t < nt) {
            if (p.variant == HYPIC_GDN) gs = expf(p.g[(t0 + t) * p.h_v + h]);
            else if (p.variant == HYPIC_SCALAR_DECAY) gs = gconst;
            if (delta) b = p.beta[(t0 + t) * p.h_v + h];
          }
          sm.gs[t] = gs;
          sm.b[t] = b;
        }
      }
      __syncthreads();
      flush();  // the last token of the previous tile
      for (int t = 0; t < nt; t++) {
        const float b = sm.b[t], gs = sm.gs[t];
        const float vj = sm.v[t][col < 128 ? col : 0];
        if (delta) {
          const float *kd = (vec ? sm.kd[t] : sm.k[t]) + r0;
          float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
#pragma unroll
          for (int i = 0; i < HALF; i += 4) {
            const float4 w = *reinterpret_cast<const float4 *>(kd + i);  // 16-byte aligned rows
            x0 = fmaf(w.x, X[i + 0], x0);
            x1 = fmaf(w.y, X[i + 1], x1);
            x2 = fmaf(w.z, X[i + 2], x2);
            x3 = fmaf(w.w, X[i + 3], x3);
          }
          fs.xs[u & 1][hf][col] = (x0 + x1) + (x2 + x3);
          tc_named_bar(bar, 64);
          flush();
          // both halves sum in the same order: identical x
          const float x = fs.xs[u & 1][0][col] + fs.xs[u & 1][1][col];
          const float c = vec ? (b * vj - b * x) : (gs * (-b * x) + b * vj);
          update(t, c);
        } else {
          update(t, vj);
        }
        // the half output q^T S
        const float *qq = fs.q[t] + r0;
        float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
        for (int i = 0; i < HALF; i += 4) {
          const float4 w = *reinterpret_cast<const float4 *>(qq + i);
          o0 = fmaf(w.x, X[i + 0], o0);
          o1 = fmaf(w.y, X[i + 1], o1);
          o2 = fmaf(w.z, X[i + 2], o2);
          o3 = fmaf(w.w, X[i + 3], o3);
        }
        const float o = (o0 + o1) + (o2 + o3);
        if (hf) fs.os[u & 1][col] = o;
        opend = o;
        pend = t0 + t;
        u++;
        if (!delta) {
          // no erase barrier in these variants: the output exchange needs one
          tc_named_bar(bar, 64);
          flush();
        }
      }
      __syncthreads();  // the tile buffers are free
    }
    flush();
  }
}

}  // namespace

// the output pass of the prefill forward (pairs written elsewhere); the
// token inputs are copied a tile ahead by cp.async when every row they are
// read in starts on a 16-byte boundary, else staged by plain loads
cudaError_t launch_forward_out(const BuildParams &p, int n_items, int n_sm, cudaStream_t s) {
  const int dvp = ((p.d_v + 31) / 32) * 32;
  const int threads = 2 * dvp;
  const int es = p.in_dtype == HYPIC_IN_BF16 ? 2 : 4;
  const bool vec = is_vector_gate(p.variant);
  auto al16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
  const bool async_ok = (p.d_k * es) % 16 == 0 && (p.d_v * es) % 16 == 0 && al16(p.k) && al16(p.q) && al16(p.v) &&
                        (!vec || ((p.d_k % 4) == 0 && al16(p.g)));
  auto go = [&](auto kern, size_t base, int DK) -> cudaError_t {
    const size_t smem = base + (async_ok ? 2 * (size_t)fwd_raw_layout(DK, es, vec).bytes : 0);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    int grid = n_sm * per_sm;
    if (grid > n_items) grid = n_items;
    if (grid < 1) return cudaSuccess;
    kern<<<grid, threads, smem, s>>>(p, dvp, async_ok ? 1 : 0);
    return cudaGetLastError();
  };
  if (p.d_k <= 16) return go(forward_out_kernel<16>, fwd_raw_offset<16>(), 16);
  if (p.d_k <= 32) return go(forward_out_kernel<32>, fwd_raw_offset<32>(), 32);
  if (p.d_k <= 64) return go(forward_out_kernel<64>, fwd_raw_offset<64>(), 64);
  return go(forward_out_kernel<128>, fwd_raw_offset<128>(), 128);
}

cudaError_t launch_build_token(const BuildParams &p, int n_items, int n_sm, cudaStream_t s) {
  if (p.d_k <= 16) return launch_dk<16>(p, n_items, n_sm, s);
  if (p.d_k <= 32) return launch_dk<32>(p, n_items, n_sm, s);
  if (p.d_k <= 64) return launch_dk<64>(p, n_items, n_sm, s);
  return launch_dk<128>(p, n_items, n_sm, s);
}

}  // namespace hypic
