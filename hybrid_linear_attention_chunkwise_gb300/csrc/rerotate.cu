// rerotate.cu -- state re-rotation of cached pairs for segments reused at a
// shifted position (HYPIC news pages, nav.aitube.vip §2.1, last paragraph:
// variants with RoPE re-rotate the cached state).  With keys multiplied by
// the block-diagonal rotation R = R(delta), a scalar-gated pair becomes
// (R T_C R^T, R S(C|0)).
//
// R acts on a key-channel vector x as (R x)[a] = C[a] x[a] + G[a] x[P[a]]:
// P[a] is the channel paired with a, C[a] = cos(phi), G[a] = -sin(phi) for
// the first channel of a pair and +sin(phi) for the second, phi = delta *
// theta_i; an unrotated channel has C = 1, G = 0, P[a] = a.  Hence
//   (R S)[a][j]     = C[a] S[a][j] + G[a] S[P[a]][j]
//   (R T R^T)[a][b] = sum over p in {a, P[a]}, q in {b, P[b]} of
//                     R[a][p] T[p][q] R[b][q].
// Every output element depends only on the 2 x 2 (or 2 x 1) block of its
// channel pairs, so each (slot, head) block is staged whole in shared memory
// and then written: the operation may run in place.
//
// One CTA per (item, group of HPC value heads): the angle table is formed
// once per CTA in fp64 (pow and sincos of the library; the shift is exact up
// to 2^53) and rounded to fp32; the data is moved with 16-byte loads and
// stores.  This is a bandwidth-bound kernel: each pool byte is read once and
// written once.
#include <cuda_runtime.h>

#include "common.cuh"

namespace hypic {

namespace {

constexpr int NT = 256;  // threads per CTA
constexpr int HPC = 4;   // value heads per CTA

struct RerotSmem {
  float buf[128 * 128];  // one (slot, head) block of T or S
  float C[128], G[128];
  int P[128];
};

// stage rows x cols (cols a multiple of 4) of src into buf, 16 bytes a time
__device__ __forceinline__ void stage(float *buf, const float *src, int n4) {
  const float4 *s4 = reinterpret_cast<const float4 *>(src);
  float4 *b4 = reinterpret_cast<float4 *>(buf);
  for (int i = threadIdx.x; i < n4; i += NT) b4[i] = s4[i];
}

__global__ void __launch_bounds__(NT) rerotate_kernel(const RerotateParams p) {
  extern __shared__ unsigned char smem_raw[];
  RerotSmem &sm = *reinterpret_cast<RerotSmem *>(smem_raw);
  const int hgroups = (p.h_v + HPC - 1) / HPC;
  const int m = blockIdx.x / hgroups;
  const int h0 = (blockIdx.x % hgroups) * HPC;
  const int si = p.slot_in[m], so = p.slot_out[m];
  if (si < 0 || si >= p.n_slots_in || so < 0 || so >= p.n_slots_out) {
    if (threadIdx.x == 0) report(p.status, HYPIC_STATUS_BAD_SLOT);
    return;
  }
  const int dk = p.d_k, dv = p.d_v;
  // the channel table of R(delta)
  if (threadIdx.x < dk) {
    const int a = threadIdx.x;
    const int h = p.rot_dim / 2;
    float c = 1.f, g = 0.f;
    int partner = a;
    if (a < p.rot_dim) {
      int i, first;
      if (p.layout == HYPIC_ROPE_INTERLEAVED) {
        i = a >> 1;
        first = !(a & 1);
        partner = a ^ 1;
      } else {
        i = a < h ? a : a - h;
        first = a < h;
        partner = a < h ? a + h : a - h;
      }
      const double phi = (double)p.delta[m] * pow(p.base, -2.0 * i / p.rot_dim);
      double sn, cs;
      sincos(phi, &sn, &cs);
      c = (float)cs;
      g = first ? (float)-sn : (float)sn;
    }
    sm.C[a] = c;
    sm.G[a] = g;
    sm.P[a] = partner;
  }
  const bool dense = p.variant == HYPIC_GDN || p.variant == HYPIC_DELTANET;
  for (int hh = 0; hh < HPC; hh++) {
    const int h = h0 + hh;
    if (h >= p.h_v) break;
    if (dense) {
      __syncthreads();  // table written / previous block consumed
      stage(sm.buf, p.T_in + ((int64_t)si * p.h_v + h) * dk * dk, dk * dk / 4);
      __syncthreads();
      const int q4 = dk / 4;
      for (int idx = threadIdx.x; idx < dk * q4; idx += NT) {
        const int a = idx / q4, b0 = 4 * (idx % q4);
        const float ca = sm.C[a], ga = sm.G[a];
        const float *ra = sm.buf + a * dk, *rp = sm.buf + sm.P[a] * dk;
        float o[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
          const int b = b0 + j, pb = sm.P[b];
          const float cb = sm.C[b], gb = sm.G[b];
          // R[a][a] T[a][.] R[b][.] + R[a][P a] T[P a][.] R[b][.]
          const float top = fmaf(cb, ra[b], gb * ra[pb]);
          const float bot = fmaf(cb, rp[b], gb * rp[pb]);
          o[j] = fmaf(ca, top, ga * bot);
        }
        *reinterpret_cast<float4 *>(p.T_out + ((int64_t)so * p.h_v + h) * dk * dk + a * dk + b0) =
            make_float4(o[0], o[1], o[2], o[3]);
      }
    } else if (threadIdx.x == 0) {
      p.T_out[(int64_t)so * p.h_v + h] = p.T_in[(int64_t)si * p.h_v + h];  // gamma^L I commutes with R
    }
    __syncthreads();
    stage(sm.buf, p.S_in + ((int64_t)si * p.h_v + h) * dk * dv, dk * dv / 4);
    __syncthreads();
    const int v4 = dv / 4;
    for (int idx = threadIdx.x; idx < dk * v4; idx += NT) {
      const int a = idx / v4, j0 = 4 * (idx % v4);
      const float ca = sm.C[a], ga = sm.G[a];
      const float4 x = *reinterpret_cast<const float4 *>(sm.buf + a * dv + j0);
      const float4 y = *reinterpret_cast<const float4 *>(sm.buf + sm.P[a] * dv + j0);
      *reinterpret_cast<float4 *>(p.S_out + ((int64_t)so * p.h_v + h) * dk * dv + a * dv + j0) =
          make_float4(fmaf(ca, x.x, ga * y.x), fmaf(ca, x.y, ga * y.y), fmaf(ca, x.z, ga * y.z),
                      fmaf(ca, x.w, ga * y.w));
    }
  }
}

}  // namespace

cudaError_t launch_rerotate(const RerotateParams &p, cudaStream_t s) {
  const int64_t grid = (int64_t)p.n_items * ((p.h_v + HPC - 1) / HPC);
  if (grid < 1) return cudaSuccess;
  const int smem = (int)sizeof(RerotSmem);
  cudaError_t e = cudaFuncSetAttribute(rerotate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  rerotate_kernel<<<(unsigned)grid, NT, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace hypic
