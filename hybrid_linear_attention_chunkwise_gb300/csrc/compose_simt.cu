// compose_simt.cu -- fp32 compose of cached pairs in prompt order (all
// variants), the fp32-input path of hypic_compose.
//
// One block per (layer, value head) chain.  Thread n holds column n of the
// running state S (d_k fp32 values in registers).  For each segment, in
// prompt order (HYPIC news pages, nav.aitube.vip §2.1 composition rule and
// §2.2 seam window):
//   seam: for each of the w seam tokens, S <- T_t S + U_t (a local dot
//         product k^T S[:, n] and a rank-1 update per column), then
//         o_t[n] = q_t . S[:, n];
//   pair: S <- T_C S + S(C|0).  Dense T_C is staged in shared memory and each
//         thread forms its column of T_C S with broadcast reads of T_C; scalar
//         and diagonal T_C scale S in place.
// Every product is an fp32 FMA chain (no tensor cores): this path exists for
// fp32 inputs, where the 1e-5 bar leaves no room for tf32/bf16 operands.
#include <algorithm>

#include <cuda_runtime.h>

#include "common.cuh"

namespace hypic {

namespace {

constexpr int SB = 8;  // seam tokens per shared-memory tile

template <int DK>
struct ComposeSmem {
  float T[DK][DK];     // dense T_C of the current segment
  float S[DK][128];    // new rows of T_C S while they are being formed
  float k[SB][DK], kd[SB][DK], a[SB][DK], q[SB][DK];
  float v[SB][128];
  float gs[SB], b[SB];
};

template <int DK>
__global__ void __launch_bounds__(128) compose_simt_kernel(ComposeParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ComposeSmem<DK> &sm = *reinterpret_cast<ComposeSmem<DK> *>(smem_raw);
  const int chain = blockIdx.x;
  const int l = chain / p.h_v, h = chain % p.h_v;
  const int kh = (int)(((int64_t)h * p.h_k) / p.h_v);
  const int n = threadIdx.x;
  const int d_k = p.d_k, d_v = p.d_v, w = p.seam_w;
  const bool act = n < d_v;
  const bool delta = is_delta(p.variant), vec = is_vector_gate(p.variant);
  const int64_t state = (int64_t)chain * d_k * d_v;
  const bool trans = (p.flags & HYPIC_FLAG_TRANSITION_ONLY) != 0;  // U_t and S(C|0) count as zero

  float S[DK];
#pragma unroll
  for (int i = 0; i < DK; i++) S[i] = (act && i < d_k && p.S_init) ? p.S_init[state + (int64_t)i * d_v + n] : 0.f;

  bool bad = false;
  for (int seg = 0; seg < p.n_seg; seg++) {
    const int64_t tok0 = ((int64_t)l * p.seg_stride + seg) * w;
    // ---- seam tokens ----
    for (int s0 = 0; s0 < w; s0 += SB) {
      const int nt = min(SB, w - s0);
      __syncthreads();
      for (int e = n; e < SB * DK; e += blockDim.x) {
        const int t = e / DK, i = e % DK;
        float kv = 0.f, qv = 0.f, a = 1.f;
        if (t < nt && i < d_k) {
          const int64_t tk = tok0 + s0 + t;
          kv = load_in(p.seam_k, (tk * p.h_k + kh) * (int64_t)d_k + i, p.in_dtype);
          qv = load_in(p.seam_q, (tk * p.h_k + kh) * (int64_t)d_k + i, p.in_dtype);
          if (vec) a = expf(p.seam_g[(tk * p.h_v + h) * (int64_t)d_k + i]);
        }
        sm.k[t][i] = kv;
        sm.q[t][i] = qv;
        sm.a[t][i] = a;
        sm.kd[t][i] = kv * a;
      }
      for (int e = n; e < SB * 128; e += blockDim.x) {
        const int t = e / 128, j = e % 128;
        // transition-only: v is not read (d_v is then d_k, not the v rows' width)
        sm.v[t][j] = (t < nt && j < d_v && !trans)
                         ? load_in(p.seam_v, ((tok0 + s0 + t) * p.h_v + h) * (int64_t)d_v + j, p.in_dtype)
                         : 0.f;
      }
      for (int t = n; t < SB; t += blockDim.x) {
        float gs = 1.f, b = 0.f;
        if (t < nt) {
          const int64_t tk = tok0 + s0 + t;
          if (p.variant == HYPIC_GDN) gs = expf(p.seam_g[tk * p.h_v + h]);
          else if (p.variant == HYPIC_SCALAR_DECAY) gs = expf(p.seam_g[(int64_t)l * p.h_v + h]);
          if (delta) b = p.seam_beta[tk * p.h_v + h];
        }
        sm.gs[t] = gs;
        sm.b[t] = b;
      }
      __syncthreads();
      for (int t = 0; t < nt; t++) {
        const float vj = act && !trans ? sm.v[t][n] : 0.f;  // transition-only: no write
        const float gs = sm.gs[t], b = sm.b[t];
        if (delta) {
          const float *kd = vec ? sm.kd[t] : sm.k[t];
          float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
#pragma unroll
          for (int i = 0; i < DK; i += 4) {
            x0 = fmaf(kd[i], S[i], x0);
            x1 = fmaf(kd[i + 1], S[i + 1], x1);
            x2 = fmaf(kd[i + 2], S[i + 2], x2);
            x3 = fmaf(kd[i + 3], S[i + 3], x3);
          }
          const float x = (x0 + x1) + (x2 + x3);
          const float c = vec ? (b * vj - b * x) : (gs * (-b * x) + b * vj);
          if (vec) {
#pragma unroll
            for (int i = 0; i < DK; i++) S[i] = fmaf(sm.a[t][i], S[i], sm.k[t][i] * c);
          } else {
#pragma unroll
            for (int i = 0; i < DK; i++) S[i] = fmaf(gs, S[i], sm.k[t][i] * c);
          }
        } else if (vec) {
#pragma unroll
          for (int i = 0; i < DK; i++) S[i] = fmaf(sm.a[t][i], S[i], sm.k[t][i] * vj);
        } else {
#pragma unroll
          for (int i = 0; i < DK; i++) S[i] = fmaf(gs, S[i], sm.k[t][i] * vj);
        }
        float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
        for (int i = 0; i < DK; i += 4) {
          o0 = fmaf(sm.q[t][i], S[i], o0);
          o1 = fmaf(sm.q[t][i + 1], S[i + 1], o1);
          o2 = fmaf(sm.q[t][i + 2], S[i + 2], o2);
          o3 = fmaf(sm.q[t][i + 3], S[i + 3], o3);
        }
        if (act && !trans) {
          const float o = (o0 + o1) + (o2 + o3);
          p.seam_out[((tok0 + s0 + t) * p.h_v + h) * (int64_t)d_v + n] = o;
          bad |= !finite_f(o);
        }
      }
    }
    // ---- cached pair ----
    const int slot = p.slot[(int64_t)l * p.seg_stride + seg];
    if (slot < 0 || slot >= p.n_slots) {
      if (n == 0) report(p.status, HYPIC_STATUS_BAD_SLOT);
      continue;  // uniform across the block: the chain skips this pair
    }
    const int64_t sh = (int64_t)slot * p.h_v + h;
    const float *Sc = trans ? nullptr : p.S_pool + sh * d_k * d_v;
    if (delta) {
      __syncthreads();
      const float *Tc = p.T_pool + sh * d_k * d_k;
      for (int e = n; e < DK * DK; e += blockDim.x) {
        const int r = e / DK, c = e % DK;
        sm.T[r][c] = (r < d_k && c < d_k) ? Tc[(int64_t)r * d_k + c] : 0.f;
      }
      __syncthreads();
      // column n of T_C S from the old column in registers, RB rows at a
      // time; new rows wait in shared memory until every row is formed
      constexpr int RB = DK < 32 ? DK : 32;
      for (int rb = 0; rb < DK; rb += RB) {
        float acc[RB];
#pragma unroll
        for (int r = 0; r < RB; r++) acc[r] = 0.f;
#pragma unroll
        for (int c = 0; c < DK; c += 4) {
#pragma unroll
          for (int r = 0; r < RB; r++) {
            const float4 t4 = *reinterpret_cast<const float4 *>(&sm.T[rb + r][c]);
            acc[r] = fmaf(t4.x, S[c], acc[r]);
            acc[r] = fmaf(t4.y, S[c + 1], acc[r]);
            acc[r] = fmaf(t4.z, S[c + 2], acc[r]);
            acc[r] = fmaf(t4.w, S[c + 3], acc[r]);
          }
        }
#pragma unroll
        for (int r = 0; r < RB; r++) sm.S[rb + r][n] = acc[r];
      }
#pragma unroll
      for (int r = 0; r < DK; r++) {
        const float sc = (act && r < d_k && !trans) ? Sc[(int64_t)r * d_v + n] : 0.f;
        S[r] = sm.S[r][n] + sc;
      }
    } else if (vec) {
      const float *Tc = p.T_pool + sh * d_k;
#pragma unroll
      for (int i = 0; i < DK; i++)
        if (i < d_k && act) S[i] = fmaf(Tc[i], S[i], trans ? 0.f : Sc[(int64_t)i * d_v + n]);
    } else {
      const float tc = p.T_pool[sh];
#pragma unroll
      for (int i = 0; i < DK; i++)
        if (i < d_k && act) S[i] = fmaf(tc, S[i], trans ? 0.f : Sc[(int64_t)i * d_v + n]);
    }
  }
  if (act) {
#pragma unroll
    for (int i = 0; i < DK; i++)
      if (i < d_k) {
        p.S_out[state + (int64_t)i * d_v + n] = S[i];
        bad |= !finite_f(S[i]);
      }
  }
  if ((p.flags & HYPIC_FLAG_CHECK_FINITE) && bad) report(p.status, HYPIC_STATUS_NONFINITE);
}

template <int DK>
cudaError_t launch_dk(const ComposeParams &p, cudaStream_t s) {
  const size_t smem = sizeof(ComposeSmem<DK>);
  cudaError_t e = cudaFuncSetAttribute(compose_simt_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = p.n_layers * p.h_v;
  if (grid < 1) return cudaSuccess;
  compose_simt_kernel<DK><<<grid, 128, smem, s>>>(p);
  return cudaGetLastError();
}

__global__ void fill_identity_kernel(float *out, int64_t n_mats, int d) {
  const int64_t total = n_mats * d * d;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = (e / d) % d, c = e % d;
    out[e] = r == c ? 1.f : 0.f;
  }
}

}  // namespace

cudaError_t launch_fill_identity(float *out, int64_t n_mats, int d, cudaStream_t s) {
  if (n_mats < 1) return cudaSuccess;
  const int64_t total = n_mats * d * d;
  const int grid = (int)std::min<int64_t>((total + 255) / 256, 4096);
  fill_identity_kernel<<<grid, 256, 0, s>>>(out, n_mats, d);
  return cudaGetLastError();
}

cudaError_t launch_compose_simt(const ComposeParams &p, cudaStream_t s) {
  if (p.d_k <= 16) return launch_dk<16>(p, s);
  if (p.d_k <= 32) return launch_dk<32>(p, s);
  if (p.d_k <= 64) return launch_dk<64>(p, s);
  return launch_dk<128>(p, s);
}

}  // namespace hypic
