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
// One CTA per (item, group of HPC value heads), one CTA per SM: the angle
// table is formed once per CTA in fp64 (pow and sincos of the library; the
// shift is exact up to 2^53) and rounded to fp32, while the first blocks are
// already in flight.  The CTA's blocks (T then S of each head) stream through
// a ring of NBUF shared-memory buffers by 1-D bulk copies, two blocks ahead
// of the one being rotated; results leave by 16-byte stores.  This is a
// bandwidth-bound kernel: each pool byte is read once and written once.
// Every wait is bounded (HYPIC_STATUS_TIMEOUT; copies in flight are drained
// before the CTA exits).
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc.cuh"

namespace hypic {

namespace {

constexpr int NT = 256;    // threads per CTA
constexpr int HPC = 8;     // value heads per CTA
constexpr int NBUF = 3;    // block buffers (two blocks in flight ahead)
constexpr uint32_t DRAIN_LIMIT = 1u << 22;

struct __align__(128) RerotSmem {
  float buf[NBUF][128 * 128];  // (slot, head) blocks of T or S
  float C[128], G[128];
  int P[128];
  int PQ[32], SW[32];  // per channel quad: the quad holding its partners, and
                       // whether partners sit swapped within it (interleaved)
  uint64_t full[NBUF];
};

__global__ void __launch_bounds__(NT, 1) rerotate_kernel(const RerotateParams p, uint32_t lim) {
  extern __shared__ unsigned char smem_raw[];
  RerotSmem &sm = *reinterpret_cast<RerotSmem *>(smem_raw + ((128u - (tc::smem_u32(smem_raw) & 127u)) & 127u));
  const int tid = threadIdx.x;
  const int hgroups = (p.h_v + HPC - 1) / HPC;
  const int m = blockIdx.x / hgroups;
  const int h0 = (blockIdx.x % hgroups) * HPC;
  const int si = p.slot_in[m], so = p.slot_out[m];
  if (si < 0 || si >= p.n_slots_in || so < 0 || so >= p.n_slots_out) {
    if (tid == 0) report(p.status, HYPIC_STATUS_BAD_SLOT);
    return;
  }
  const int dk = p.d_k, dv = p.d_v;
  const bool dense = p.variant == HYPIC_GDN || p.variant == HYPIC_DELTANET;
  const int per_head = dense ? 2 : 1;  // blocks per head: T and S, or S
  const int nj = min(HPC, p.h_v - h0) * per_head;
  auto is_T = [&](int j) { return dense && (j % per_head) == 0; };
  auto head = [&](int j) { return h0 + j / per_head; };
  // block j of this CTA into buffer j % NBUF (thread 0)
  auto issue = [&](int j) {
    if (j >= nj) return;
    const int h = head(j);
    const float *src = is_T(j) ? p.T_in + ((int64_t)si * p.h_v + h) * dk * dk
                               : p.S_in + ((int64_t)si * p.h_v + h) * dk * dv;
    const uint32_t bytes = (uint32_t)(is_T(j) ? dk * dk : dk * dv) * 4u;
    tc::mbar_expect_tx(&sm.full[j % NBUF], bytes);
    tc::bulk_load(sm.buf[j % NBUF], src, bytes, &sm.full[j % NBUF]);
  };
  if (tid == 0) {
    for (int b = 0; b < NBUF; b++) tc::mbar_init(&sm.full[b], 1);
    tc::fence_mbar_init();
    for (int j = 0; j < NBUF - 1; j++) issue(j);
  }
  // the channel table of R(delta), while the first blocks land
  if (tid < dk) {
    const int a = tid;
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
  __syncthreads();  // channel table visible
  // Quad q's partners, channel by channel, are the quad P[4q] / 4: for the
  // interleaved pairing that is q itself with neighbours swapped (a channel
  // of the quad left unrotated has G = 0, so its swapped partner adds a
  // zero); for the half pairing (rot_dim a multiple of 8) a quad lies wholly
  // in one half or wholly unrotated, so its partners form one aligned quad.
  if (tid < dk / 4) {
    const int pa = sm.P[4 * tid];
    sm.PQ[tid] = pa / 4;
    sm.SW[tid] = pa == 4 * tid + 1;
  }
  if (!dense && tid < min(HPC, p.h_v - h0))  // gamma^L I commutes with R
    p.T_out[(int64_t)so * p.h_v + h0 + tid] = p.T_in[(int64_t)si * p.h_v + h0 + tid];
  __syncthreads();  // table and barrier init visible

  bool ok = true;
  int first_fail = nj;  // thread 0: the first block whose wait ran out
  for (int j = 0; j < nj; j++) {
    // buffer (j + NBUF - 1) % NBUF was last read in iteration j - 1; after a
    // wait has run out no further copy is issued
    if (tid == 0 && ok) issue(j + NBUF - 1);
    ok = ok && tc::mbar_wait(&sm.full[j % NBUF], (j / NBUF) & 1, lim);
    if (!ok && tid == 0 && first_fail == nj) {
      first_fail = j;
      report(p.status, HYPIC_STATUS_TIMEOUT);
    }
    const float *blk = sm.buf[j % NBUF];
    const int h = head(j);
    if (ok && is_T(j)) {
      // four outputs (a, b0 .. b0 + 3) per step from 16-byte loads: the
      // quad of b0 and its partner quad (swapped in place when the pairs
      // are interleaved), in rows a and P[a]
      const int q4 = dk / 4;
      float *dst = p.T_out + ((int64_t)so * p.h_v + h) * dk * dk;
      auto rot4 = [&](int a, int bq, const float4 cb, const float4 gb, int pq, bool sw) {
        const float ca = sm.C[a], ga = sm.G[a];
        const float *ra = blk + a * dk, *rp = blk + sm.P[a] * dk;
        const float4 xa = *reinterpret_cast<const float4 *>(ra + 4 * bq);
        const float4 xp = *reinterpret_cast<const float4 *>(rp + 4 * bq);
        float4 ya = *reinterpret_cast<const float4 *>(ra + 4 * pq);
        float4 yp = *reinterpret_cast<const float4 *>(rp + 4 * pq);
        if (sw) {
          ya = make_float4(ya.y, ya.x, ya.w, ya.z);
          yp = make_float4(yp.y, yp.x, yp.w, yp.z);
        }
        // R[a][a] T[a][.] R[b][.] + R[a][P a] T[P a][.] R[b][.]
        auto one = [&](float cbj, float gbj, float xaj, float yaj, float xpj, float ypj) {
          return fmaf(ca, fmaf(cbj, xaj, gbj * yaj), ga * fmaf(cbj, xpj, gbj * ypj));
        };
        *reinterpret_cast<float4 *>(dst + a * dk + 4 * bq) =
            make_float4(one(cb.x, gb.x, xa.x, ya.x, xp.x, yp.x), one(cb.y, gb.y, xa.y, ya.y, xp.y, yp.y),
                        one(cb.z, gb.z, xa.z, ya.z, xp.z, yp.z), one(cb.w, gb.w, xa.w, ya.w, xp.w, yp.w));
      };
      auto quad = [&](int bq, float4 &cb, float4 &gb, int &pq, bool &sw) {
        cb = *reinterpret_cast<const float4 *>(sm.C + 4 * bq);
        gb = *reinterpret_cast<const float4 *>(sm.G + 4 * bq);
        pq = sm.PQ[bq];
        sw = sm.SW[bq] != 0;
      };
      if (NT % q4 == 0) {  // each thread keeps one column quad
        const int bq = tid % q4;
        float4 cb, gb;
        int pq;
        bool sw;
        quad(bq, cb, gb, pq, sw);
        for (int a = tid / q4; a < dk; a += NT / q4) rot4(a, bq, cb, gb, pq, sw);
      } else {
        for (int idx = tid; idx < dk * q4; idx += NT) {
          float4 cb, gb;
          int pq;
          bool sw;
          quad(idx % q4, cb, gb, pq, sw);
          rot4(idx / q4, idx % q4, cb, gb, pq, sw);
        }
      }
    } else if (ok) {
      const int v4 = dv / 4;
      float *dst = p.S_out + ((int64_t)so * p.h_v + h) * dk * dv;
      for (int idx = tid; idx < dk * v4; idx += NT) {
        const int a = idx / v4, j0 = 4 * (idx % v4);
        const float ca = sm.C[a], ga = sm.G[a];
        const float4 x = *reinterpret_cast<const float4 *>(blk + a * dv + j0);
        const float4 y = *reinterpret_cast<const float4 *>(blk + sm.P[a] * dv + j0);
        *reinterpret_cast<float4 *>(dst + a * dv + j0) =
            make_float4(fmaf(ca, x.x, ga * y.x), fmaf(ca, x.y, ga * y.y), fmaf(ca, x.z, ga * y.z),
                        fmaf(ca, x.w, ga * y.w));
      }
    }
    __syncthreads();  // this buffer is free for block j + NBUF
  }
  // drain: copies issued but not yet seen complete (only after a timeout:
  // blocks first_fail .. first_fail + NBUF - 1) land before the CTA exits
  if (tid == 0)
    for (int j = first_fail; j < nj && j < first_fail + NBUF; j++)
      tc::mbar_wait(&sm.full[j % NBUF], (j / NBUF) & 1, DRAIN_LIMIT);
}

}  // namespace

cudaError_t launch_rerotate(const RerotateParams &p, uint32_t wait_limit, cudaStream_t s) {
  const int64_t grid = (int64_t)p.n_items * ((p.h_v + HPC - 1) / HPC);
  if (grid < 1) return cudaSuccess;
  const int smem = (int)sizeof(RerotSmem) + 128;
  cudaError_t e = cudaFuncSetAttribute(rerotate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  rerotate_kernel<<<(unsigned)grid, NT, smem, s>>>(p, wait_limit);
  return cudaGetLastError();
}

}  // namespace hypic
