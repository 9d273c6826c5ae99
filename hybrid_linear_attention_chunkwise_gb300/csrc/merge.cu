// merge.cu -- batched pair merge (T2, S2) o (T1, S1) = (T2 T1, T2 S1 + S2).
//
// The composition rule of the HYPIC news pages (nav.aitube.vip §2.1:
// S(C1.C2) = T(C2) S(C1) + S(C2)) applied to two cached pairs, with the
// transition of the joined span being the product T(C2) T(C1).  Items are
// (merge, value head).
//
// Dense transitions with d_k = d_v = 128 run on the tensor cores, one CTA
// per item, in transposed form so that the outputs are written column by
// column with coalesced stores:
//     D_T = T1^T T2^T = (T2 T1)^T,    D_S = S1^T T2^T = (T2 S1)^T,
// A operand from TMEM (thread pair n holds column n of T1, then of S1), B
// operand the TMA-loaded K-slabs of T2 (K-major, 128-byte swizzle), fp32
// accumulators in TMEM.  Operands are split for about fp32 accuracy:
// A = hi + lo with hi = RN_tf32(x), lo = RN_tf32(x - hi); the tensor core
// reads the raw fp32 T2 slabs truncated to tf32 (B_hi), and the threads write
// B_lo = x - trunc_tf32(x) beside them; each product is
// A_hi B_hi + A_hi B_lo + A_lo B_hi (kind::tf32).
// Other shapes and the scalar / diagonal transitions run a plain fp32 kernel
// on the CUDA cores.  All waits are bounded.
#include <cstddef>

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace hypic {

namespace {

constexpr int NT = 256;
constexpr int SLAB = 16384;  // one K-slab [128 rows x 32 k] fp32
constexpr uint32_t DRAIN_LIMIT = 1u << 22;

// TMEM columns (512: one CTA per SM)
constexpr uint32_t TM_AH = 0;    // A hi  (lane n, column k)
constexpr uint32_t TM_AL = 128;  // A lo
constexpr uint32_t TM_DT = 256;  // (T2 T1)^T
constexpr uint32_t TM_DS = 384;  // (T2 S1)^T

struct __align__(1024) MergeSmem {
  unsigned char bh[4][SLAB];  // T2 K-slabs as loaded (read truncated: B hi)
  unsigned char bl[4][SLAB];  // T2 - trunc_tf32(T2), same layout (B lo)
  uint64_t full, mma_t, mma_s;
  uint32_t tmem_base;
  int skip;
};

struct MergeArgs {
  MergeParams p;
  uint32_t wait_limit;
};

__device__ __forceinline__ uint32_t trunc_tf32(float x) { return __float_as_uint(x) & 0xFFFFE000u; }

__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

// rows 64 hf .. 64 hf + 63 of column n of a [128 x 128] matrix (row pitch
// 128), held in x -> A hi / lo in TMEM (this thread's lane, columns k)
__device__ __forceinline__ void stage_a(const float (&x)[64], uint32_t ah, uint32_t al) {
#pragma unroll
  for (int b = 0; b < 4; b++) {
    uint32_t h[16], l[16];
#pragma unroll
    for (int j = 0; j < 16; j++) {
      h[j] = tc::to_tf32(x[16 * b + j]);
      l[j] = tc::to_tf32(x[16 * b + j] - __uint_as_float(h[j]));
    }
    tc::tmem_st16(ah + 16 * b, h);
    tc::tmem_st16(al + 16 * b, l);
  }
  tc::tmem_wait_st();
}
__device__ __forceinline__ void load_col(const float *M, int n, int hf, float (&x)[64]) {
#pragma unroll
  for (int j = 0; j < 64; j++) x[j] = M[(int64_t)(64 * hf + j) * 128 + n];
}

// D (+)= A B with A from TMEM (columns a0.., 128 k) and B the four K-slabs
__device__ __forceinline__ void issue_product(uint32_t d, uint32_t a, const unsigned char (*b)[SLAB], uint32_t id,
                                              bool accumulate) {
  for (int sl = 0; sl < 4; sl++) {
    const uint32_t base = tc::smem_u32(b[sl]);
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
      const uint64_t bd = tc::smem_desc(base + 32 * kk, 16, 1024, tc::SW_128B);
      tc::mma_ts_tf32(d, a + 32 * sl + 8 * kk, bd, id, (accumulate || sl | kk) ? 1u : 0u);
    }
  }
}

__global__ void __launch_bounds__(NT, 1)
    merge_tc_kernel(const __grid_constant__ MergeArgs args, const __grid_constant__ CUtensorMap tmap_T) {
  extern __shared__ unsigned char smem_raw[];
  MergeSmem &sm = *reinterpret_cast<MergeSmem *>(smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  const MergeParams &p = args.p;
  const uint32_t LIM = args.wait_limit;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int n = tid & 127, hf = tid >> 7;  // column n, rows / k 64 hf .. 64 hf + 63
  const int m = blockIdx.x / p.h_v, h = blockIdx.x % p.h_v;

  if (tid == 0) {
    tc::mbar_init(&sm.full, 1);
    tc::mbar_init(&sm.mma_t, 1);
    tc::mbar_init(&sm.mma_s, 1);
    const int a = p.later[m], b = p.earlier[m], o = p.out[m];
    const bool bad = a < 0 || a >= p.n_slots_a || b < 0 || b >= p.n_slots_b || o < 0 || o >= p.n_slots_out;
    sm.skip = bad ? 1 : 0;
    if (bad) report(p.status, HYPIC_STATUS_BAD_SLOT);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&sm.tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = sm.tmem_base;
  const bool skip = sm.skip != 0;
  if (!skip) {
    const int a = p.later[m], b = p.earlier[m], o = p.out[m];
    const int64_t pa = ((int64_t)a * p.h_v + h) * 128 * 128, pb = ((int64_t)b * p.h_v + h) * 128 * 128;
    const int64_t po = ((int64_t)o * p.h_v + h) * 128 * 128;
    if (tid == 0) {
      // S2 (read in the epilogue) into L2 now, and T2 by TMA
      prefetch_l2(p.S_a + pa, 65536u);
      tc::prefetch_tmap(&tmap_T);
      tc::mbar_expect_tx(&sm.full, 4u * SLAB);
      for (int sl = 0; sl < 4; sl++)
        tc::tma_load_2d(sm.bh[sl], &tmap_T, 32 * sl, (int32_t)(((int64_t)a * p.h_v + h) * 128), &sm.full);
    }
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t ah = tm + lane_base + TM_AH + 64 * hf, al = tm + lane_base + TM_AL + 64 * hf;
    const uint32_t id = tc::idesc(tc::FMT_TF32, 128, 128);
    // ---- A = T1^T (hi, lo); S1's column loads in flight meanwhile; B lo
    // from the landed slabs
    float s1[64];
    {
      float x[64];
      load_col(p.T_b + pb, n, hf, x);
      load_col(p.S_b + pb, n, hf, s1);
      stage_a(x, ah, al);
    }
    bool ok = tc::mbar_wait(&sm.full, 0, LIM);
    if (!ok) report(p.status, HYPIC_STATUS_TIMEOUT);
    {
      const uint4 *src = reinterpret_cast<const uint4 *>(&sm.bh[0][0]);
      uint4 *dst = reinterpret_cast<uint4 *>(&sm.bl[0][0]);
#pragma unroll 4
      for (int e = tid; e < 4 * SLAB / 16; e += NT) {
        const uint4 x = src[e];
        uint4 y;
        y.x = __float_as_uint(__uint_as_float(x.x) - __uint_as_float(trunc_tf32(__uint_as_float(x.x))));
        y.y = __float_as_uint(__uint_as_float(x.y) - __uint_as_float(trunc_tf32(__uint_as_float(x.y))));
        y.z = __float_as_uint(__uint_as_float(x.z) - __uint_as_float(trunc_tf32(__uint_as_float(x.z))));
        y.w = __float_as_uint(__uint_as_float(x.w) - __uint_as_float(trunc_tf32(__uint_as_float(x.w))));
        dst[e] = y;
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
      tc::tc_fence_after();
      issue_product(tm + TM_DT, tm + TM_AH, sm.bh, id, false);
      issue_product(tm + TM_DT, tm + TM_AH, sm.bl, id, true);
      issue_product(tm + TM_DT, tm + TM_AL, sm.bh, id, true);
      tc::mma_commit(&sm.mma_t);
    }
    // ---- A = S1^T once the T product has read A
    if (ok && !tc::mbar_wait(&sm.mma_t, 0, DRAIN_LIMIT)) {
      ok = false;
      report(p.status, HYPIC_STATUS_TIMEOUT);
    }
    tc::tc_fence_after();
    stage_a(s1, ah, al);
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
      tc::tc_fence_after();
      issue_product(tm + TM_DS, tm + TM_AH, sm.bh, id, false);
      issue_product(tm + TM_DS, tm + TM_AH, sm.bl, id, true);
      issue_product(tm + TM_DS, tm + TM_AL, sm.bh, id, true);
      tc::mma_commit(&sm.mma_s);
    }
    // ---- T_out column n, rows 64 hf .. (lane n of D_T, columns = rows r)
    const uint32_t dt = tm + lane_base + TM_DT + 64 * hf, ds = tm + lane_base + TM_DS + 64 * hf;
    float *To = p.T_out + po + n, *So = p.S_out + po + n;
    const float *S2 = p.S_a + pa + n;
#pragma unroll 1
    for (int b4 = 0; b4 < 4; b4++) {
      uint32_t r[16];
      tc::tmem_ld16(dt + 16 * b4, r);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; j++) To[(int64_t)(64 * hf + 16 * b4 + j) * 128] = __uint_as_float(r[j]);
    }
    float s2[64];
#pragma unroll
    for (int j = 0; j < 64; j++) s2[j] = S2[(int64_t)(64 * hf + j) * 128];
    if (ok && !tc::mbar_wait(&sm.mma_s, 0, DRAIN_LIMIT)) report(p.status, HYPIC_STATUS_TIMEOUT);
    tc::tc_fence_after();
#pragma unroll
    for (int b4 = 0; b4 < 4; b4++) {
      uint32_t r[16];
      tc::tmem_ld16(ds + 16 * b4, r);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; j++)
        So[(int64_t)(64 * hf + 16 * b4 + j) * 128] = __uint_as_float(r[j]) + s2[16 * b4 + j];
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tm, 512);
  }
}

// ------------------------------------------------------------------ fp32
// One CTA per item.  Dense: thread c owns output column c of [T | S] (c <
// d_k + d_v) and forms it as T2 x with x = column c of [T1 | S1], T2 read
// from shared memory; scalar / diagonal: elementwise.
constexpr int DMAX = 128;
__global__ void __launch_bounds__(256) merge_simt_kernel(const MergeParams p) {
  __shared__ float t2[DMAX * DMAX / 2];  // dense T2 in two row halves (32 KiB)
  const int m = blockIdx.x / p.h_v, h = blockIdx.x % p.h_v;
  const int a = p.later[m], b = p.earlier[m], o = p.out[m];
  if (a < 0 || a >= p.n_slots_a || b < 0 || b >= p.n_slots_b || o < 0 || o >= p.n_slots_out) {
    if (threadIdx.x == 0) report(p.status, HYPIC_STATUS_BAD_SLOT);
    return;
  }
  const int dk = p.d_k, dv = p.d_v;
  const int64_t sa = ((int64_t)a * p.h_v + h) * dk * dv, sb = ((int64_t)b * p.h_v + h) * dk * dv;
  const int64_t so = ((int64_t)o * p.h_v + h) * dk * dv;
  if (is_dense_T(p.variant)) {
    const int64_t ta = ((int64_t)a * p.h_v + h) * dk * dk, tb = ((int64_t)b * p.h_v + h) * dk * dk;
    const int64_t to = ((int64_t)o * p.h_v + h) * dk * dk;
    const int c = threadIdx.x;
    const bool active = c < dk + dv;
    float x[DMAX];
#pragma unroll 1
    for (int k = 0; k < dk; k++)
      x[k] = active ? (c < dk ? p.T_b[tb + (int64_t)k * dk + c] : p.S_b[sb + (int64_t)k * dv + (c - dk)]) : 0.f;
    for (int half = 0; half < 2; half++) {
      const int r0 = half * ((dk + 1) / 2), r1 = half ? dk : (dk + 1) / 2;
      __syncthreads();
      for (int e = threadIdx.x; e < (r1 - r0) * dk; e += blockDim.x) t2[e] = p.T_a[ta + (int64_t)r0 * dk + e];
      __syncthreads();
      if (active) {
        for (int r = r0; r < r1; r++) {
          const float *row = t2 + (r - r0) * dk;
          float acc = 0.f;
          for (int k = 0; k < dk; k++) acc = fmaf(row[k], x[k], acc);
          if (c < dk) p.T_out[to + (int64_t)r * dk + c] = acc;
          else p.S_out[so + (int64_t)r * dv + (c - dk)] = acc + p.S_a[sa + (int64_t)r * dv + (c - dk)];
        }
      }
    }
  } else if (is_vector_gate(p.variant)) {  // diagonal
    const int64_t ta = ((int64_t)a * p.h_v + h) * dk, tb = ((int64_t)b * p.h_v + h) * dk;
    const int64_t to = ((int64_t)o * p.h_v + h) * dk;
    for (int r = threadIdx.x; r < dk; r += blockDim.x) p.T_out[to + r] = p.T_a[ta + r] * p.T_b[tb + r];
    for (int e = threadIdx.x; e < dk * dv; e += blockDim.x)
      p.S_out[so + e] = fmaf(p.T_a[ta + e / dv], p.S_b[sb + e], p.S_a[sa + e]);
  } else {  // scalar
    const int64_t ta = (int64_t)a * p.h_v + h, tb = (int64_t)b * p.h_v + h, to = (int64_t)o * p.h_v + h;
    const float t = p.T_a[ta];
    if (threadIdx.x == 0) p.T_out[to] = t * p.T_b[tb];
    for (int e = threadIdx.x; e < dk * dv; e += blockDim.x) p.S_out[so + e] = fmaf(t, p.S_b[sb + e], p.S_a[sa + e]);
  }
}

}  // namespace

bool merge_tc_supported(const MergeParams &p) {
  auto a16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  return is_dense_T(p.variant) && p.d_k == 128 && p.d_v == 128 && a16(p.T_a) && a16(p.S_a) && a16(p.T_b) &&
         a16(p.S_b);
}

cudaError_t launch_merge(const MergeParams &p, uint32_t wait_limit, cudaStream_t s) {
  const int grid = p.n_merge * p.h_v;
  if (grid < 1) return cudaSuccess;
  if (merge_tc_supported(p)) {
    CUtensorMap tmap;
    if (!make_tmap_f32_rows(&tmap, p.T_a, (uint64_t)p.n_slots_a * p.h_v * 128, 128)) return cudaErrorInvalidValue;
    const size_t smem = sizeof(MergeSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(merge_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    MergeArgs a;
    a.p = p;
    a.wait_limit = wait_limit;
    merge_tc_kernel<<<grid, NT, smem, s>>>(a, tmap);
  } else {
    merge_simt_kernel<<<grid, 256, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace hypic
