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
  int taken = 0;  // items fetched by this CTA (thread 0)

  for (;;) {
    if (tid == 0) sm.item = take_item(p.plan, taken);
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
// build kernels).
//
// A warp holds 16 state columns.  Lane 8*qr + pr keeps columns 2*pr and
// 2*pr + 1 of them over key rows [qr*DK/4, (qr+1)*DK/4), so the four
// quarters of a column pair sit in one warp: their partial dot products
// (k^T S for the erase, q^T S for the output) are summed by two xor
// shuffles, a butterfly that gives all four lanes the same bits, with no
// shared-memory exchange and no barrier per token.  Each 16-byte load of a
// k or q row feeds both columns.  In shared memory the rows are padded by
// 16 bytes per quarter, so the four quarters' broadcast loads fall in
// different banks.
// ---------------------------------------------------------------------------
template <int DK>
struct FwdSmem {
  static constexpr int QR = DK / 4;    // key rows per quarter
  static constexpr int RP = DK + 16;   // padded row: quarter q starts at q * (QR + 4)
  alignas(16) float k[TB][RP];
  alignas(16) float kd[TB][RP];  // vector gates: k * a (the erase acts after Diag(a)); else unused
  alignas(16) float a[TB][RP];   // vector gates: a = exp(g); else unused
  alignas(16) float q[TB][RP];
  float v[TB][128];
  float gs[TB];  // scalar gate a_t (GDN) / gamma (scalar decay) / 1
  float b[TB];   // beta_t (0 on padding tokens)
  int item;
};
template <int DK>
__host__ __device__ constexpr int fwd_pad(int i) {
  return i + 4 * (i / (DK / 4));
}
// every row, and every quarter of one, starts on a 16-byte boundary
template <int DK>
constexpr bool fwd_rows_aligned() {
  return offsetof(FwdSmem<DK>, k) % 16 == 0 && offsetof(FwdSmem<DK>, kd) % 16 == 0 &&
         offsetof(FwdSmem<DK>, a) % 16 == 0 && offsetof(FwdSmem<DK>, q) % 16 == 0 &&
         (FwdSmem<DK>::RP * 4) % 16 == 0 && (DK / 4) % 4 == 0;
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

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 8);
  return x + __shfl_xor_sync(0xffffffffu, x, 16);
}

template <int DK>
__global__ void __launch_bounds__(256) forward_out_kernel(BuildParams p, int async_tiles) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  FwdSmem<DK> &sm = *reinterpret_cast<FwdSmem<DK> *>(smem_raw);
  constexpr int QR = DK / 4;
  const int tid = threadIdx.x, lane = tid & 31;
  const bool delta = is_delta(p.variant);
  const bool vec = is_vector_gate(p.variant);
  const int d_k = p.d_k, d_v = p.d_v;
  const int qr = lane >> 3;
  const int c0 = (tid >> 5) * 16 + 2 * (lane & 7);  // the thread's first column
  const int ro = fwd_pad<DK>(qr * QR);              // its quarter in a padded row
  const int v0c = c0 < 128 ? c0 : 0, v1c = c0 + 1 < 128 ? c0 + 1 : 0;
  const int n_items = p.plan->n_items;
  const int es = p.in_dtype == HYPIC_IN_BF16 ? 2 : 4;
  const FwdRaw lay = fwd_raw_layout(DK, es, vec);
  unsigned char *raw = smem_raw + fwd_raw_offset<DK>();  // two stages when async_tiles
  int taken = 0;  // items fetched by this CTA (thread 0)

  for (;;) {
    if (tid == 0) sm.item = take_item(p.plan, taken);
    __syncthreads();
    const int idx = sm.item;
    __syncthreads();
    if (idx >= n_items) break;
    const BuildItem it = p.items[idx];
    const int h = it.head;
    const int kh = (int)(((int64_t)h * p.h_k) / p.h_v);
    // scalar gates: the state is A * X (A uniform over the block), so that
    // the gated update X <- g X + k c^T costs one FMA per element; vector
    // gates: the state is X
    float X0[QR], X1[QR];
#pragma unroll
    for (int i = 0; i < QR; i++) X0[i] = X1[i] = 0.f;
    float A = 1.f;
    float gconst = 1.f;
    if (p.variant == HYPIC_SCALAR_DECAY) gconst = expf(p.g[h]);

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
    // the fp32 tile from either source: k, q, a, k*a into padded rows
    auto put_row = [&](int t, int i, float kv, float qv, float a) {
      const int j = fwd_pad<DK>(i);
      sm.k[t][j] = kv;
      sm.q[t][j] = qv;
      if (vec) {
        sm.a[t][j] = a;
        sm.kd[t][j] = kv * a;
      }
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
          put_row(t, i, kv, qv, a);
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
          put_row(t, i, kv, qv, a);
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
      for (int t = 0; t < nt; t++) {
        const float b = sm.b[t], gs = sm.gs[t];
        const float v0 = sm.v[t][v0c], v1 = sm.v[t][v1c];
        float c0v = v0, c1v = v1;  // X <- G X + k c^T (the column coefficients)
        if (delta) {
          const float *kd = (vec ? sm.kd[t] : sm.k[t]) + ro;
          float xa = 0.f, xb = 0.f, ya = 0.f, yb = 0.f;
#pragma unroll
          for (int i = 0; i < QR; i += 4) {
            const float4 w = *reinterpret_cast<const float4 *>(kd + i);
            xa = fmaf(w.x, X0[i + 0], xa);
            xb = fmaf(w.y, X0[i + 1], xb);
            ya = fmaf(w.x, X1[i + 0], ya);
            yb = fmaf(w.y, X1[i + 1], yb);
            xa = fmaf(w.z, X0[i + 2], xa);
            xb = fmaf(w.w, X0[i + 3], xb);
            ya = fmaf(w.z, X1[i + 2], ya);
            yb = fmaf(w.w, X1[i + 3], yb);
          }
          float x0 = quad_sum(xa + xb), x1 = quad_sum(ya + yb);
          if (!vec) {
            x0 *= A;
            x1 *= A;
          }
          c0v = vec ? (b * v0 - b * x0) : (gs * (-b * x0) + b * v0);
          c1v = vec ? (b * v1 - b * x1) : (gs * (-b * x1) + b * v1);
        }
        const float *kk = sm.k[t] + ro;
        if (vec) {
          const float *aa = sm.a[t] + ro;
#pragma unroll
          for (int i = 0; i < QR; i += 4) {
            const float4 kv = *reinterpret_cast<const float4 *>(kk + i);
            const float4 av = *reinterpret_cast<const float4 *>(aa + i);
            X0[i + 0] = fmaf(av.x, X0[i + 0], kv.x * c0v);
            X0[i + 1] = fmaf(av.y, X0[i + 1], kv.y * c0v);
            X0[i + 2] = fmaf(av.z, X0[i + 2], kv.z * c0v);
            X0[i + 3] = fmaf(av.w, X0[i + 3], kv.w * c0v);
            X1[i + 0] = fmaf(av.x, X1[i + 0], kv.x * c1v);
            X1[i + 1] = fmaf(av.y, X1[i + 1], kv.y * c1v);
            X1[i + 2] = fmaf(av.z, X1[i + 2], kv.z * c1v);
            X1[i + 3] = fmaf(av.w, X1[i + 3], kv.w * c1v);
          }
        } else {
          // A g X + k c^T = A' (X + k (c / A')^T) with A' = A g; before A'
          // gets small enough for c / A' to overflow, it is folded into X
          float An = A * gs;
          if (An < 0x1p-64f) {
#pragma unroll
            for (int i = 0; i < QR; i++) {
              X0[i] *= An;
              X1[i] *= An;
            }
            An = 1.f;
          }
          const float inv = 1.f / An;
          const float d0 = c0v * inv, d1 = c1v * inv;
#pragma unroll
          for (int i = 0; i < QR; i += 4) {
            const float4 kv = *reinterpret_cast<const float4 *>(kk + i);
            X0[i + 0] = fmaf(kv.x, d0, X0[i + 0]);
            X0[i + 1] = fmaf(kv.y, d0, X0[i + 1]);
            X0[i + 2] = fmaf(kv.z, d0, X0[i + 2]);
            X0[i + 3] = fmaf(kv.w, d0, X0[i + 3]);
            X1[i + 0] = fmaf(kv.x, d1, X1[i + 0]);
            X1[i + 1] = fmaf(kv.y, d1, X1[i + 1]);
            X1[i + 2] = fmaf(kv.z, d1, X1[i + 2]);
            X1[i + 3] = fmaf(kv.w, d1, X1[i + 3]);
          }
          A = An;
        }
        // the output q^T S of both columns
        const float *qq = sm.q[t] + ro;
        float oa = 0.f, ob = 0.f, pa = 0.f, pb = 0.f;
#pragma unroll
        for (int i = 0; i < QR; i += 4) {
          const float4 w = *reinterpret_cast<const float4 *>(qq + i);
          oa = fmaf(w.x, X0[i + 0], oa);
          ob = fmaf(w.y, X0[i + 1], ob);
          pa = fmaf(w.x, X1[i + 0], pa);
          pb = fmaf(w.y, X1[i + 1], pb);
          oa = fmaf(w.z, X0[i + 2], oa);
          ob = fmaf(w.w, X0[i + 3], ob);
          pa = fmaf(w.z, X1[i + 2], pa);
          pb = fmaf(w.w, X1[i + 3], pb);
        }
        const float sc = vec ? 1.f : A;
        const float o0 = sc * quad_sum(oa + ob), o1 = sc * quad_sum(pa + pb);
        if (qr == 0) {
          float *dst = p.o_out + ((t0 + t) * p.h_v + h) * (int64_t)d_v;
          if (c0 < d_v) dst[c0] = o0;
          if (c0 + 1 < d_v) dst[c0 + 1] = o1;
        }
      }
      __syncthreads();  // the tile buffers are free
    }
  }
}

}  // namespace

// the output pass of the prefill forward (pairs written elsewhere); the
// token inputs are copied a tile ahead by cp.async when every row they are
// read in starts on a 16-byte boundary, else staged by plain loads
cudaError_t launch_forward_out(const BuildParams &p, int n_items, int n_sm, cudaStream_t s) {
  const int threads = 32 * ((p.d_v + 15) / 16);  // a warp per 16 state columns
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
    kern<<<grid, threads, smem, s>>>(p, async_ok ? 1 : 0);
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
