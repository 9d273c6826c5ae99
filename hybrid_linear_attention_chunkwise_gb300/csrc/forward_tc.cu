// forward_tc.cu -- the per-token outputs of the prefill forward on the
// tensor cores, for the scalar-gate delta rules (GDN, DeltaNet) with bf16
// inputs and d_k = d_v = 128.
//
// A segment's first prefill runs its body from a zero state (HYPIC news
// pages, nav.aitube.vip §2.1: the segment's state is position independent),
// and every body token t emits o_t = S_t^T q_t with the post-update state.
// The recording build (build_tc.cu) leaves, for every 64-token chunk of every
// (segment, value head), the chunk's start state S_0 and
// Delta = U - W S_0, the chunk's WY-form state increments.  Inside the
// chunk, with lam_t = sum_{j<=t} g_j from the chunk start and G_t = e^lam_t,
//     S_t = G_t S_0 + sum_{i<=t} (G_t / G_i) k_i Delta_i^T,
// so the outputs of the chunk are
//     o_t = G_t (S_0^T q_t) + sum_{i<=t} e^(lam_t - lam_i) (q_t . k_i) Delta_i,
// two small contractions per chunk that need nothing from any other chunk:
// every (chunk, value head) is an independent item.
//
// One CTA of 256 threads per item, two CTAs per SM (80 KB of shared memory,
// 256 TMEM columns each):
//   TMA:      Q and K tiles [64 t x 128] bf16 (rows 0-63 and 64-127 of one
//             K-major tile, so one MMA with M = 128 gives Q K^T)
//   threads:  S_0^T (column j of S_0 per TMEM lane) as bf16 hi + lo, packed
//             two per column, into TMEM (the A operand of term 1); Delta^T
//             hi + lo into shared memory (the A operand of term 2)
//   MMA:      Q K^T (kind::f16), then term 1 O1^T = S_0^T Q^T (A from TMEM,
//             B = the Q tile, exact bf16)
//   threads:  B2[t, i] = e^(lam_t - lam_i) (q_t . k_i) for i <= t < n_t, hi + lo
//   MMA:      term 2 O2^T = Delta^T B2^T (three products of the split pairs)
//   epilogue: o_t[j] = G_t O1^T[j, t] + O2^T[j, t], coalesced rows of o_out.
// Splitting S_0, Delta and B2 into bf16 hi + lo (about 2^-17 each) keeps the
// outputs at fp32-like accuracy; Q and K are exact bf16 inputs.  All waits
// are bounded.
#include <cstddef>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc.cuh"

namespace hypic {

namespace {

constexpr int NT = 256;
constexpr int C = 64;
constexpr uint32_t DRAIN_LIMIT = 1u << 22;

// TMEM columns (256 allocated: two CTAs per SM)
constexpr uint32_t TM_S = 0;     // S_0^T hi (0-63) and lo (64-127), bf16 pairs: A of term 1
constexpr uint32_t TM_O1 = 128;  // O1^T [128 j x 64 t]
constexpr uint32_t TM_O2 = 192;  // Q K^T (lanes 0-63), then O2^T [128 j x 64 t]

struct __align__(1024) FwdTcSmem {
  unsigned char qk[2][16384];   // [Q; K] K-major, 128 rows x 64 channels per slab
  unsigned char dth[16384];     // Delta^T hi [128 j x 64 i] bf16, K-major
  unsigned char dtl[16384];     //   lo
  unsigned char b2h[8192];      // B2 hi [64 t x 64 i] bf16, K-major
  unsigned char b2l[8192];      //   lo
  float lam[C];
  float E[C], R[C];             // e^{lam_t} and e^{-lam_t} (R only when the chunk's decay span is <= 80)
  uint64_t full, qk_done, o1_done, o2_done;
  uint32_t tmem_base;
  int ok;                       // the tiles landed in time (set by thread 0)
  int fact;                     // e^{lam_t - lam_i} = E_t R_i is in range
};

struct FwdItem {
  int32_t rec;   // chunk record index (start state / Delta of this chunk)
  int32_t head;  // value head
  int32_t nt;    // tokens in the chunk (<= 64)
  int32_t pad;
  int64_t tok0;  // first token of the chunk
};
static_assert(sizeof(FwdItem) == 24, "forward item size");

struct FwdTcArgs {
  BuildParams p;
  const FwdItem *items;
  uint32_t wait_limit;
};

__device__ __forceinline__ uint32_t sw16(int r, int k, int R) {
  const uint32_t byte = (uint32_t)(k & 63) * 2u;
  return (uint32_t)((k >> 6) * R * 128 + r * 128) + ((((byte >> 4) ^ (uint32_t)(r & 7)) << 4) | (byte & 15u));
}
__device__ __forceinline__ uint64_t kdesc16(uint32_t base, int k, int R) {
  return tc::smem_desc(base + (uint32_t)((k >> 6) * R * 128 + (k & 63) * 2), 16, 1024, tc::SW_128B);
}
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  const float r0 = x0 - __uint_as_float(hi << 16), r1 = x1 - __uint_as_float(hi & 0xFFFF0000u);
  const __nv_bfloat162 l = __floats2bfloat162_rn(r0, r1);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}

__global__ void __launch_bounds__(NT, 2)
    forward_tc_kernel(const __grid_constant__ FwdTcArgs args, const __grid_constant__ CUtensorMap tmap_q,
                      const __grid_constant__ CUtensorMap tmap_k) {
  extern __shared__ unsigned char smem_raw[];
  FwdTcSmem &sm = *reinterpret_cast<FwdTcSmem *>(smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  const BuildParams &p = args.p;
  const uint32_t LIM = args.wait_limit;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = tid & 127, hf = tid >> 7;  // value column j (TMEM lane), half hf of the work along K / t
  const FwdItem it = args.items[blockIdx.x];
  const int kh = (int)(((int64_t)it.head * p.h_k) / p.h_v);

  if (tid == 0) {
    tc::mbar_init(&sm.full, 1);
    tc::mbar_init(&sm.qk_done, 1);
    tc::mbar_init(&sm.o1_done, 1);
    tc::mbar_init(&sm.o2_done, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&sm.tmem_base, 256);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = sm.tmem_base;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  bool ok = true;

  // ---- Q and K tiles by TMA (rows of other segments or past the tensor are
  // masked below)
  if (tid == 0) {
    tc::prefetch_tmap(&tmap_q);
    tc::prefetch_tmap(&tmap_k);
    tc::mbar_expect_tx(&sm.full, 32768u);
    for (int s = 0; s < 2; s++) {
      tc::tma_load_3d(sm.qk[s], &tmap_q, 64 * s, kh, (int32_t)it.tok0, &sm.full);
      tc::tma_load_3d(sm.qk[s] + 8192, &tmap_k, 64 * s, kh, (int32_t)it.tok0, &sm.full);
    }
  }
  // ---- chunk-local cumulative log-gates
  if (warp == 0) {
    float x0 = 0.f, x1 = 0.f;
    if (p.variant == HYPIC_GDN) {
      if (lane < it.nt) x0 = p.g[(it.tok0 + lane) * p.h_v + it.head];
      if (lane + 32 < it.nt) x1 = p.g[(it.tok0 + lane + 32) * p.h_v + it.head];
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y0 = __shfl_up_sync(0xffffffffu, x0, o);
      const float y1 = __shfl_up_sync(0xffffffffu, x1, o);
      if (lane >= o) {
        x0 += y0;
        x1 += y1;
      }
    }
    x1 += __shfl_sync(0xffffffffu, x0, 31);
    sm.lam[lane] = x0;
    sm.lam[lane + 32] = x1;
    // factors of e^{lam_t - lam_i} = E_t R_i (i <= t): in fp32 range when the
    // chunk's log-gates sum above -80; else B2 forms each factor directly
    float mn = fminf(x0, x1), mx = fmaxf(x0, x1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    sm.E[lane] = __expf(x0);
    sm.E[lane + 32] = __expf(x1);
    sm.R[lane] = __expf(-x0);
    sm.R[lane + 32] = __expf(-x1);
    if (lane == 0) sm.fact = mn >= -80.f && mx <= 80.f;
  }
  // ---- S_0^T (hi, lo) into TMEM: thread (j, hf) packs rows d = 64 hf ..
  // 64 hf + 63 of column j of S_0; Delta^T (hi, lo) into shared memory:
  // thread (j, hf) converts tokens 32 hf .. 32 hf + 31 of column j
  const int64_t rc = (int64_t)it.rec * p.h_v + it.head;
  {
    const float *S0 = p.rec_S + rc * 128 * 128 + j;
    float xs[64];  // every row of this thread's half in flight at once
#pragma unroll
    for (int e = 0; e < 64; e++) xs[e] = S0[(int64_t)(64 * hf + e) * 128];
#pragma unroll
    for (int b = 0; b < 2; b++) {  // 32 rows at a time
      const float *x = xs + 32 * b;
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int e = 0; e < 16; e++) split_bf16x2(x[2 * e], x[2 * e + 1], hi[e], lo[e]);
      // column c of the packed operand holds rows 2c, 2c + 1
      tc::tmem_st16(tm + lane_base + TM_S + 32 * hf + 16 * b, hi);
      tc::tmem_st16(tm + lane_base + TM_S + 64 + 32 * hf + 16 * b, lo);
    }
    const float *D = p.rec_D + rc * 64 * 128 + j;
    float x[32];
#pragma unroll
    for (int e = 0; e < 32; e++) x[e] = D[(int64_t)(32 * hf + e) * 128];
#pragma unroll
    for (int q8 = 0; q8 < 4; q8++) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int e = 0; e < 4; e++) split_bf16x2(x[8 * q8 + 2 * e], x[8 * q8 + 2 * e + 1], hw[e], lw[e]);
      const uint32_t off = sw16(j, 32 * hf + 8 * q8, 128);
      *reinterpret_cast<uint4 *>(sm.dth + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4 *>(sm.dtl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }
  tc::tmem_wait_st();
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();

  // ---- Q K^T, then term 1 (issued by one thread)
  const uint32_t qkb = tc::smem_u32(sm.qk[0]);
  const uint32_t id64 = tc::idesc(tc::FMT_BF16, 128, 64);
  if (tid == 0) {
    ok = tc::mbar_wait(&sm.full, 0, LIM);
    tc::tc_fence_after();
    if (ok) {
      // rows 0-63 of D: Q K^T (A = [Q; K], B = K rows 64-127 of the tile)
#pragma unroll
      for (int ks = 0; ks < 8; ks++)
        tc::mma_ss_f16(tm + TM_O2, kdesc16(qkb, 16 * ks, 128), kdesc16(qkb + 8192, 16 * ks, 128), id64, ks > 0);
    }
    tc::mma_commit(&sm.qk_done);
    if (ok) {
      // O1^T = S_0^T Q^T: A = S_0^T from TMEM (8 packed columns per K-step of
      // 16), hi then lo; B = the Q rows
#pragma unroll
      for (int ks = 0; ks < 8; ks++)
        tc::mma_ts_f16(tm + TM_O1, tm + TM_S + 8 * ks, kdesc16(qkb, 16 * ks, 128), id64, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 8; ks++)
        tc::mma_ts_f16(tm + TM_O1, tm + TM_S + 64 + 8 * ks, kdesc16(qkb, 16 * ks, 128), id64, 1u);
    }
    tc::mma_commit(&sm.o1_done);
    if (!ok) report(p.status, HYPIC_STATUS_TIMEOUT);
    sm.ok = ok ? 1 : 0;  // published by the barrier after B2
  }
  // ---- B2 = e^(lam_t - lam_i) (q_t . k_i), i <= t < n_t: rows t = 0..63
  // live in TMEM lanes 0..63, which warps 0, 1, 4 and 5 can read; warps 0
  // and 1 form columns 0..31, warps 4 and 5 columns 32..63
  if ((warp & 3) < 2) {
    const int t = j;              // lane of the warp's quadrant
    const int c0 = 32 * hf;       // this warp's columns
    const bool got = tc::mbar_wait(&sm.qk_done, 0, DRAIN_LIMIT);
    tc::tc_fence_after();
    const bool fact = sm.fact != 0;
    const float lt = sm.lam[t], Et = sm.E[t];
    uint32_t r[32];
    tc::tmem_ld32(tm + lane_base + TM_O2 + c0, r);
    tc::tmem_wait_ld();
#pragma unroll
    for (int q8 = 0; q8 < 4; q8++) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int i0 = c0 + 8 * q8 + 2 * e;
        const float w0 = fact ? Et * sm.R[i0] : __expf(lt - sm.lam[i0]);
        const float w1 = fact ? Et * sm.R[i0 + 1] : __expf(lt - sm.lam[i0 + 1]);
        const float y0 = (got && i0 <= t && t < it.nt) ? w0 * __uint_as_float(r[8 * q8 + 2 * e]) : 0.f;
        const float y1 = (got && i0 + 1 <= t && t < it.nt) ? w1 * __uint_as_float(r[8 * q8 + 2 * e + 1]) : 0.f;
        split_bf16x2(y0, y1, hw[e], lw[e]);
      }
      const uint32_t off = sw16(t, c0 + 8 * q8, 64);
      *reinterpret_cast<uint4 *>(sm.b2h + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4 *>(sm.b2l + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  // ---- term 2 into the columns Q K^T was read from
  ok = sm.ok != 0;
  if (tid == 0) {
    tc::tc_fence_after();
    if (ok) {
      const uint32_t ah = tc::smem_u32(sm.dth), al = tc::smem_u32(sm.dtl);
      const uint32_t bh = tc::smem_u32(sm.b2h), bl = tc::smem_u32(sm.b2l);
#pragma unroll
      for (int ks = 0; ks < 4; ks++) {
        tc::mma_ss_f16(tm + TM_O2, kdesc16(ah, 16 * ks, 128), kdesc16(bh, 16 * ks, 64), id64, ks > 0);
        tc::mma_ss_f16(tm + TM_O2, kdesc16(ah, 16 * ks, 128), kdesc16(bl, 16 * ks, 64), id64, 1u);
        tc::mma_ss_f16(tm + TM_O2, kdesc16(al, 16 * ks, 128), kdesc16(bh, 16 * ks, 64), id64, 1u);
      }
    }
    tc::mma_commit(&sm.o2_done);
  }
  // ---- epilogue: thread (j, hf) writes tokens 32 hf .. 32 hf + 31 of column j
  const bool g1 = tc::mbar_wait(&sm.o1_done, 0, DRAIN_LIMIT);
  const bool g2 = tc::mbar_wait(&sm.o2_done, 0, DRAIN_LIMIT);
  tc::tc_fence_after();
  {
    uint32_t a[32], b[32];
    tc::tmem_ld32(tm + lane_base + TM_O1 + 32 * hf, a);
    tc::tmem_ld32(tm + lane_base + TM_O2 + 32 * hf, b);
    tc::tmem_wait_ld();
    bool bad = false;
    if (ok && g1 && g2) {
      float *o = p.o_out + ((it.tok0 + 32 * hf) * p.h_v + it.head) * 128 + j;
#pragma unroll
      for (int e = 0; e < 32; e++) {
        const int t = 32 * hf + e;
        if (t < it.nt) {
          const float v = fmaf(sm.E[t], __uint_as_float(a[e]), __uint_as_float(b[e]));
          o[(int64_t)e * p.h_v * 128] = v;
          bad |= !finite_f(v);
        }
      }
    } else if (tid == 0 && ok) {
      report(p.status, HYPIC_STATUS_TIMEOUT);
    }
    if ((p.flags & HYPIC_FLAG_CHECK_FINITE) && bad) report(p.status, HYPIC_STATUS_NONFINITE);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tm, 256);
  }
}

}  // namespace

bool forward_tc_supported(const BuildParams &p) {
  auto a16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  return build_tc_supported(p) && p.q && a16(p.q) && p.o_out && a16(p.o_out);
}

cudaError_t launch_forward_tc(const BuildParams &p, const void *items, int n_items, int64_t n_tokens,
                              uint32_t wait_limit, cudaStream_t s) {
  if (n_items < 1) return cudaSuccess;
  CUtensorMap tq, tk;
  if (!make_tmap_tokens(&tq, p.q, n_tokens, p.h_k) || !make_tmap_tokens(&tk, p.k, n_tokens, p.h_k))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(FwdTcSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(forward_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  FwdTcArgs a;
  a.p = p;
  a.items = static_cast<const FwdItem *>(items);
  a.wait_limit = wait_limit;
  forward_tc_kernel<<<n_items, NT, smem, s>>>(a, tq, tk);
  return cudaGetLastError();
}

size_t forward_item_bytes() { return sizeof(FwdItem); }

void forward_fill_item(void *items, int64_t idx, int32_t rec, int32_t head, int32_t nt, int64_t tok0) {
  FwdItem &f = static_cast<FwdItem *>(items)[idx];
  f.rec = rec;
  f.head = head;
  f.nt = nt;
  f.pad = 0;
  f.tok0 = tok0;
}

}  // namespace hypic
