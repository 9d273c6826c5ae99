// build_tc.cu -- tensor-core chunkwise segment build for the scalar-gate
// delta rules (GDN, DeltaNet) with bf16 inputs and d_k = d_v = 128.
//
// Caches the pair (T_C, S(C|0)) of every (segment, value head): T_C is the
// product of the body's token transitions and S(C|0) its final state from
// zero (HYPIC news pages, nav.aitube.vip §2.1).  The body is consumed in
// chunks of C = 64 tokens with the WY / UT form of the delta rule.  Inside a
// chunk, with lam_t = sum_{j<=t} g_j, G_t = exp(lam_t) and the strictly lower
// M_ti = b_t exp(lam_t - lam_i) k_t.k_i:
//     A = (I + M)^-1,   W = A diag(b G) K,   U = A diag(b) V,
// and on the augmented block X = [T | S] the chunk acts as
//     Y = W X - [0 | U],   X <- G_C X - K^T (diag(exp(lam_C - lam)) Y),
// which is the token recurrence exactly (checked in fp64 against the token
// oracle).
//
// Layout.  The kernel works on X^T, whose rows are the 256 columns of
// [T | S].  The T half and the S half are independent chains that share W,
// so each CTA owns one half of one (segment, head): a 128 x 128 block of
// X^T, kept in TMEM as the fp32 accumulator (lane j = column j of the half,
// TMEM column d) next to a tf32-rounded copy, the A operand of chain 1.
// The TMA-loaded bf16 K and V tiles [64 tokens x 128] serve directly as MMA
// operands -- K-major for the Gram, MN-major (transposed view) elsewhere --
// so no operand is ever transposed by the threads.  Per chunk:
//   Gram     K K^T                                   kind::f16, exact inputs
//   UT       A = (I + M)^-1                          SIMT, 16 x 16 blocks
//   W        W^T  = K^T (A diag(bG))^T               kind::f16, factor split hi + lo
//   U        -U^T = V^T (-A diag(b))^T   (S half)    kind::f16, factor split hi + lo
//   chain 1  Y^T (+)= X^T W^T                        kind::tf32, A from TMEM
//   chain 2  X^T += Ytilde^T K                       kind::f16, Ytilde split hi + lo
// with Ytilde = -Y diag(exp(lam_C - lam)) and X scaled by G_C in TMEM before
// chain 2.  Split operands make those products exact to ~2^-17 (K and V are
// exact bf16); chain 1 uses tf32 operands rounded to nearest by the threads
// (the tensor core itself truncates fp32 operands).  fp32 accumulation
// throughout.  This keeps long products (8192 tokens) inside 5e-3 per head.
//
// Items are (segment, value head, half) in LPT order, pulled by an atomic
// ticket.  Inputs come in by TMA (3-D maps over [token, head, channel],
// 128-byte swizzle), two chunks ahead; the per-token gates by plain loads one
// chunk ahead.  All waits are bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc.cuh"

namespace hypic {

namespace {

constexpr int C = 64;      // tokens per chunk
constexpr int NT = 256;    // threads per CTA (warps w and w+4 share TMEM lanes)
constexpr uint32_t DRAIN_LIMIT = 1u << 22;

// TMEM columns (512 allocated, one CTA per SM)
constexpr uint32_t TM_X = 0;     // X^T half, fp32 accumulator           [128 x 128]
constexpr uint32_t TM_XR = 128;  // tf32-rounded copy (A of chain 1)     [128 x 128]
constexpr uint32_t TM_Y = 256;   // Y^T half                             [128 x 64]
constexpr uint32_t TM_W = 320;   // W^T                                  [128 x 64]
constexpr uint32_t TM_G = 384;   // K K^T (lanes 0..63)                  [128 x 64]

// Byte offsets in K-major, 128-byte-swizzled tiles of R rows (the layout the
// shared-memory descriptors describe and TMA writes): 4-byte elements sit 32
// to a 128-byte row segment, 2-byte elements 64.
__device__ __forceinline__ uint32_t sw32(int r, int k, int R) {
  const uint32_t byte = (uint32_t)(k & 31) * 4u;
  return (uint32_t)((k >> 5) * R * 128 + r * 128) + ((((byte >> 4) ^ (uint32_t)(r & 7)) << 4) | (byte & 15u));
}
__device__ __forceinline__ uint32_t sw16(int r, int k, int R) {
  const uint32_t byte = (uint32_t)(k & 63) * 2u;
  return (uint32_t)((k >> 6) * R * 128 + r * 128) + ((((byte >> 4) ^ (uint32_t)(r & 7)) << 4) | (byte & 15u));
}
// K-major operand: descriptor of the K-step starting at column k
__device__ __forceinline__ uint64_t kdesc32(uint32_t base, int k, int R) {
  return tc::smem_desc(base + (uint32_t)((k >> 5) * R * 128 + (k & 31) * 4), 16, 1024, tc::SW_128B);
}
__device__ __forceinline__ uint64_t kdesc16(uint32_t base, int k, int R) {
  return tc::smem_desc(base + (uint32_t)((k >> 6) * R * 128 + (k & 63) * 2), 16, 1024, tc::SW_128B);
}
// MN-major view of a [64 token x 128 channel] TMA tile (channel contiguous):
// the K-step starting at token t; the two 64-channel slabs are MN atoms 8 KiB
// apart, consecutive groups of 8 tokens 1 KiB apart
__device__ __forceinline__ uint64_t mndesc16(uint32_t base, int t) {
  return tc::smem_desc(base + (uint32_t)(t * 128), 8192, 1024, tc::SW_128B);
}

struct __align__(1024) BuildTcSmem {
  struct In {                   // one chunk of inputs (TMA tiles, two slabs each)
    unsigned char k[16384];     // K [64 t x 128 d] bf16
    unsigned char v[16384];     // V [64 t x 128 j] bf16 (S half); also pads the Gram's rows 64..127
  } in[2];
  unsigned char wt[32768];      // W  [64 t x 128 d] tf32, K-major: B of chain 1
  unsigned char yh[16384];      // Ytilde hi [128 j x 64 t] bf16: A of chain 2
  unsigned char yl[16384];      // Ytilde lo
  unsigned char bwh[8192];      // A diag(bG) hi [64 t x 64 t'] bf16: B of the W MMA
  unsigned char bwl[8192];      //   lo
  unsigned char buh[8192];      // -A diag(b) hi: B of the U MMA
  unsigned char bul[8192];      //   lo
  float nm[64][65];             // M
  float am[64][65];             // A = (I + M)^-1
  float pm[3][16][17];          // block products of the inverse
  float lam[64], bg[64], bt[64], dec[64];
  float gC;
  uint64_t full[2];
  uint64_t bar_g, bar_w, bar_y, bar_x;
  uint64_t never;
  uint32_t tmem_base;
  int item;
  int abort;
};

struct BuildTcArgs {
  BuildParams p;
  uint32_t wait_limit;
  int debug_stall;
};

__device__ __forceinline__ bool aborted(BuildTcSmem &sm) { return *(volatile int *)&sm.abort != 0; }
__device__ __forceinline__ void fail(BuildTcSmem &sm, const BuildParams &p) {
  *(volatile int *)&sm.abort = 1;
  report(p.status, HYPIC_STATUS_TIMEOUT);
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}
__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 a, __nv_bfloat16 b) {
  return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// TMEM address of this thread's lane at column `col` (warps w and w+4 share
// the lane quadrant w % 4)
__device__ __forceinline__ uint32_t trow(uint32_t base, int col) {
  return base + ((uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16) + (uint32_t)col;
}

__device__ __forceinline__ void wait_mma(BuildTcSmem &sm, const BuildParams &p, uint64_t *bar, uint32_t &phase) {
  if (!tc::mbar_wait(bar, phase & 1, DRAIN_LIMIT)) fail(sm, p);
  phase++;
  tc::tc_fence_after();
}
// ---------------------------------------------------------------- UT inverse
// A = (I + N)^-1 for the strictly lower 64 x 64 N in sm.nm, into sm.am:
// diagonal 16 x 16 blocks by forward substitution (one thread per column),
// then the off-diagonal blocks level by level,
//     A_ij = -A_ii * sum_{k=j}^{i-1} N_ik A_kj      (i > j).
// Called by all threads; ends with a barrier.
__device__ void ut_inverse(BuildTcSmem &sm) {
  const int n = threadIdx.x;
  for (int e = n; e < 64 * 64; e += NT) sm.am[e >> 6][e & 63] = 0.f;
  __syncthreads();
  if (n < 64) {
    const int b = 16 * (n >> 4), l = n & 15;
    float a[16];
#pragma unroll
    for (int r = 0; r < 16; r++) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int i = 0; i < r; i++) {
        if (i & 1) s1 = fmaf(sm.nm[b + r][b + i], a[i], s1);
        else s0 = fmaf(sm.nm[b + r][b + i], a[i], s0);
      }
      a[r] = (r < l) ? 0.f : (r == l ? 1.f : -(s0 + s1));
    }
#pragma unroll
    for (int r = 0; r < 16; r++) sm.am[b + r][b + l] = a[r];
  }
  __syncthreads();
  for (int d = 1; d < 4; d++) {
    const int nb = 4 - d;  // blocks (i, i - d), i = d .. 3
    for (int e = n; e < nb * 256; e += NT) {
      const int q = e >> 8, r = (e >> 4) & 15, c = e & 15;
      const int i = d + q, j = i - d;
      float s0 = 0.f, s1 = 0.f;
      for (int k = j; k < i; k++) {
#pragma unroll
        for (int m = 0; m < 16; m += 2) {
          s0 = fmaf(sm.nm[16 * i + r][16 * k + m], sm.am[16 * k + m][16 * j + c], s0);
          s1 = fmaf(sm.nm[16 * i + r][16 * k + m + 1], sm.am[16 * k + m + 1][16 * j + c], s1);
        }
      }
      sm.pm[q][r][c] = s0 + s1;
    }
    __syncthreads();
    for (int e = n; e < nb * 256; e += NT) {
      const int q = e >> 8, r = (e >> 4) & 15, c = e & 15;
      const int i = d + q, j = i - d;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int m = 0; m < 16; m += 2) {
        s0 = fmaf(sm.am[16 * i + r][16 * i + m], sm.pm[q][m][c], s0);
        s1 = fmaf(sm.am[16 * i + r][16 * i + m + 1], sm.pm[q][m + 1][c], s1);
      }
      sm.am[16 * i + r][16 * j + c] = -(s0 + s1);
    }
    __syncthreads();
  }
}

// Split factor tiles A diag(bG) and -A diag(b) (K-major bf16 [64 t x 64 t'],
// hi and lo): thread n writes 16 consecutive t' of row n / 4.
__device__ __forceinline__ void write_factors(BuildTcSmem &sm, bool s_half) {
  const int n = threadIdx.x, t = n >> 2, q0 = 16 * (n & 3);
#pragma unroll
  for (int h8 = 0; h8 < 2; h8++) {
    const int c0 = q0 + 8 * h8;
    uint32_t wh[4], wl[4], uh[4], ul[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      __nv_bfloat16 h0, l0, h1, l1;
      const float a0 = sm.am[t][c0 + 2 * j], a1 = sm.am[t][c0 + 2 * j + 1];
      split_bf16(a0 * sm.bg[c0 + 2 * j], h0, l0);
      split_bf16(a1 * sm.bg[c0 + 2 * j + 1], h1, l1);
      wh[j] = pack2(h0, h1);
      wl[j] = pack2(l0, l1);
      split_bf16(-a0 * sm.bt[c0 + 2 * j], h0, l0);
      split_bf16(-a1 * sm.bt[c0 + 2 * j + 1], h1, l1);
      uh[j] = pack2(h0, h1);
      ul[j] = pack2(l0, l1);
    }
    const uint32_t off = sw16(t, c0, 64);
    *reinterpret_cast<uint4 *>(sm.bwh + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
    *reinterpret_cast<uint4 *>(sm.bwl + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    if (s_half) {
      *reinterpret_cast<uint4 *>(sm.buh + off) = make_uint4(uh[0], uh[1], uh[2], uh[3]);
      *reinterpret_cast<uint4 *>(sm.bul + off) = make_uint4(ul[0], ul[1], ul[2], ul[3]);
    }
  }
}

// K (and, for the S half, V) of chunk `ch` of item `it` into input buffer b
__device__ __forceinline__ void issue_chunk(BuildTcSmem &sm, const BuildItem &it, int ch, int b, bool s_half,
                                            int kh, const CUtensorMap *tk, const CUtensorMap *tv) {
  const int32_t t0 = (int32_t)(it.start + (int64_t)C * ch);
  tc::mbar_expect_tx(&sm.full[b], s_half ? 32768u : 16384u);
  for (int s = 0; s < 2; s++) tc::tma_load_3d(sm.in[b].k + s * 8192, tk, 64 * s, kh, t0, &sm.full[b]);
  if (s_half)
    for (int s = 0; s < 2; s++) tc::tma_load_3d(sm.in[b].v + s * 8192, tv, 64 * s, it.head, t0, &sm.full[b]);
}
__global__ void __launch_bounds__(NT, 1)
    build_tc_kernel(const __grid_constant__ BuildTcArgs args, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte alignment by pointer arithmetic on the shared array, so the
  // compiler keeps every access in the shared address space
  BuildTcSmem &sm = *reinterpret_cast<BuildTcSmem *>(smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  const BuildParams &p = args.p;
  const uint32_t LIM = args.wait_limit;
  const int n = threadIdx.x, warp = n >> 5, lane = n & 31;
  const int lj = 32 * (warp & 3) + lane;  // TMEM lane of this thread
  const int hsel = warp >> 2;             // which half of the TMEM columns it handles
  const bool gdn = p.variant == HYPIC_GDN;

  if (n == 0) {
    tc::mbar_init(&sm.full[0], 1);
    tc::mbar_init(&sm.full[1], 1);
    tc::mbar_init(&sm.bar_g, 1);
    tc::mbar_init(&sm.bar_w, 1);
    tc::mbar_init(&sm.bar_y, 1);
    tc::mbar_init(&sm.bar_x, 1);
    tc::mbar_init(&sm.never, 1);
    sm.abort = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmap_k);
    tc::prefetch_tmap(&tmap_v);
  }
  if (warp == 0) {
    tc::tmem_alloc(&sm.tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = sm.tmem_base;
  if (args.debug_stall && !tc::mbar_wait(&sm.never, 0, LIM)) fail(sm, p);

  const uint32_t id_gram = tc::idesc(tc::FMT_BF16, 128, 64);
  const uint32_t id_wu = tc::idesc(tc::FMT_BF16, 128, 64, false, false, /*a_mn=*/true, false);
  const uint32_t id_c1 = tc::idesc(tc::FMT_TF32, 128, 64);
  const uint32_t id_c2 = tc::idesc(tc::FMT_BF16, 128, 128, false, false, false, /*b_mn=*/true);
  uint32_t ph_full[2] = {0, 0}, ph_g = 0, ph_w = 0, ph_y = 0, ph_x = 0;
  const int n_items = p.plan->n_items;

  for (;;) {
    if (n == 0) sm.item = aborted(sm) ? n_items : atomicAdd(&p.plan->ticket, 1);
    __syncthreads();
    const int idx = sm.item;
    __syncthreads();
    if (idx >= n_items) break;
    const BuildItem it = p.items[idx];
    const bool s_half = it.part == 1;
    const int h = it.head;
    const int kh = (int)(((int64_t)h * p.h_k) / p.h_v);
    const int64_t L = it.end - it.start;
    const int n_ch = (int)((L + C - 1) / C);

    // X^T half := T half: identity, S half: zero (accumulator and rounded copy)
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 32) {
      const int col = 64 * hsel + c0;
      uint32_t r[32];
#pragma unroll
      for (int j = 0; j < 32; j++) r[j] = (!s_half && col + j == lj) ? 0x3f800000u : 0u;
      tc::tmem_st32(trow(tm + TM_X, col), r);
      tc::tmem_st32(trow(tm + TM_XR, col), r);
    }
    tc::tmem_wait_st();
    if (n == 0)
      for (int ch = 0; ch < 2 && ch < n_ch; ch++) issue_chunk(sm, it, ch, ch & 1, s_half, kh, &tmap_k, &tmap_v);
    float g_cur = 0.f, b_cur = 0.f;
    if (n < C && n < L) {
      if (gdn) g_cur = p.g[(it.start + n) * p.h_v + h];
      b_cur = p.beta[(it.start + n) * p.h_v + h];
    }

    for (int ch = 0; ch < n_ch; ch++) {
      const int b = ch & 1;
      const int64_t t0 = it.start + (int64_t)C * ch;
      const int nt = (it.end - t0) < C ? (int)(it.end - t0) : C;
      float g_nxt = 0.f, b_nxt = 0.f;  // gates of the next chunk, one chunk ahead
      if (n < C && t0 + C + n < it.end) {
        if (gdn) g_nxt = p.g[(t0 + C + n) * p.h_v + h];
        b_nxt = p.beta[(t0 + C + n) * p.h_v + h];
      }
      // ---- A: inputs landed (once aborted: wait with the drain limit, the copy lands)
      if (!tc::mbar_wait(&sm.full[b], ph_full[b] & 1, aborted(sm) ? DRAIN_LIMIT : LIM)) fail(sm, p);
      ph_full[b]++;
      unsigned char *kin = sm.in[b].k, *vin = sm.in[b].v;
      if (nt < C) {  // ragged tail: identity tokens (k = v = 0; their gates and beta are 0)
        for (int e = n; e < (C - nt) * 16; e += NT) {
          const int r = nt + (e >> 4), q = e & 15;  // 16 x 16 B per row: 8 per slab
          const uint4 z = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4 *>(kin + (q >> 3) * 8192 + r * 128 + (q & 7) * 16) = z;
          if (s_half) *reinterpret_cast<uint4 *>(vin + (q >> 3) * 8192 + r * 128 + (q & 7) * 16) = z;
        }
      }
      if (n < C) {
        sm.bt[n] = b_cur;
        sm.lam[n] = g_cur;
      }
      __syncthreads();
      if (warp == 0) {  // lam_t = sum_{j<=t} g_j (two tokens per lane)
        float x0 = sm.lam[lane], x1 = sm.lam[lane + 32];
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
        const float lc = __shfl_sync(0xffffffffu, x1, 31);
        sm.lam[lane] = x0;
        sm.lam[lane + 32] = x1;
        sm.bg[lane] = sm.bt[lane] * __expf(x0);
        sm.bg[lane + 32] = sm.bt[lane + 32] * __expf(x1);
        sm.dec[lane] = __expf(lc - x0);
        sm.dec[lane + 32] = __expf(lc - x1);
        if (lane == 0) sm.gC = __expf(lc);
      }
      tc::fence_proxy_async_smem();  // zeroed tail rows are MMA operands
      tc::tc_fence_before();
      __syncthreads();

      // ---- B: Gram K K^T (K-major view of the K tile; rows 64..127 of the
      // padded M read the adjacent tiles and are ignored)
      if (n == 0) {
        tc::tc_fence_after();
        const uint32_t kb = tc::smem_u32(kin);
#pragma unroll
        for (int ks = 0; ks < 8; ks++)
          tc::mma_ss_f16(tm + TM_G, kdesc16(kb, 16 * ks, 64), kdesc16(kb, 16 * ks, 64), id_gram, ks > 0);
        tc::mma_commit(&sm.bar_g);
      }
      wait_mma(sm, p, &sm.bar_g, ph_g);
      // ---- C: M_ti = b_t exp(lam_t - lam_i) k_t.k_i (i < t): warps 0, 1, 4, 5
      if ((warp & 3) < 2) {
        const int t = lj, c0 = 32 * hsel;
        uint32_t r[32];
        tc::tmem_ld32(trow(tm + TM_G, c0), r);
        tc::tmem_wait_ld();
        const float lt = sm.lam[t], btt = sm.bt[t];
#pragma unroll
        for (int j = 0; j < 32; j++) {
          const int i = c0 + j;
          sm.nm[t][i] = (i < t) ? btt * __expf(lt - sm.lam[i]) * __uint_as_float(r[j]) : 0.f;
        }
      }
      __syncthreads();
      ut_inverse(sm);
      write_factors(sm, s_half);
      tc::fence_proxy_async_smem();
      __syncthreads();

      // ---- D: W^T = K^T (A diag(bG))^T;  S half: Y^T := V^T (-A diag(b))^T = -U^T
      if (n == 0) {
        tc::tc_fence_after();
        const uint32_t kb = tc::smem_u32(kin), vb = tc::smem_u32(vin);
        const uint32_t wh = tc::smem_u32(sm.bwh), wl = tc::smem_u32(sm.bwl);
        const uint32_t uh = tc::smem_u32(sm.buh), ul = tc::smem_u32(sm.bul);
#pragma unroll
        for (int ks = 0; ks < 4; ks++) {
          tc::mma_ss_f16(tm + TM_W, mndesc16(kb, 16 * ks), kdesc16(wh, 16 * ks, 64), id_wu, ks > 0);
          tc::mma_ss_f16(tm + TM_W, mndesc16(kb, 16 * ks), kdesc16(wl, 16 * ks, 64), id_wu, 1u);
          if (s_half) {
            tc::mma_ss_f16(tm + TM_Y, mndesc16(vb, 16 * ks), kdesc16(uh, 16 * ks, 64), id_wu, ks > 0);
            tc::mma_ss_f16(tm + TM_Y, mndesc16(vb, 16 * ks), kdesc16(ul, 16 * ks, 64), id_wu, 1u);
          }
        }
        tc::mma_commit(&sm.bar_w);
      }
      wait_mma(sm, p, &sm.bar_w, ph_w);

      // ---- E: W (tf32, rounded) as the K-major B tile [64 t x 128 d] of
      // chain 1 (each warp writes whole 128-byte row segments); X scaled by G_C
      {
        const int c0 = 32 * hsel;  // tokens c0 .. c0 + 31 of column d = lj
        uint32_t r[32];
        tc::tmem_ld32(trow(tm + TM_W, c0), r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; j++) *reinterpret_cast<uint32_t *>(sm.wt + sw32(c0 + j, lj, 64)) = tc::to_tf32(__uint_as_float(r[j]));
        const float gC = sm.gC;
#pragma unroll
        for (int cc = 0; cc < 64; cc += 32) {
          const int col = 64 * hsel + cc;
          tc::tmem_ld32(trow(tm + TM_X, col), r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; j++) r[j] = __float_as_uint(gC * __uint_as_float(r[j]));
          tc::tmem_st32(trow(tm + TM_X, col), r);
        }
        tc::tmem_wait_st();
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      __syncthreads();

      // ---- F: chain 1, Y^T (+)= X^T W^T  (the S half accumulates onto -U^T)
      if (n == 0) {
        tc::tc_fence_after();
        const uint32_t wb = tc::smem_u32(sm.wt);
#pragma unroll
        for (int ks = 0; ks < 16; ks++)
          tc::mma_ts_tf32(tm + TM_Y, tm + TM_XR + 8 * ks, kdesc32(wb, 8 * ks, 64), id_c1, (s_half || ks > 0) ? 1u : 0u);
        tc::mma_commit(&sm.bar_y);
      }
      wait_mma(sm, p, &sm.bar_y, ph_y);

      // ---- G: Ytilde = -Y diag(exp(lam_C - lam_t)), split hi + lo, as the
      // K-major A tiles [128 j x 64 t] of chain 2
      {
        const int c0 = 32 * hsel;
        uint32_t r[32];
        tc::tmem_ld32(trow(tm + TM_Y, c0), r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int q8 = 0; q8 < 4; q8++) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int j = 0; j < 4; j++) {
            const int t = c0 + 8 * q8 + 2 * j;
            __nv_bfloat16 h0, l0, h1, l1;
            split_bf16(-sm.dec[t] * __uint_as_float(r[8 * q8 + 2 * j]), h0, l0);
            split_bf16(-sm.dec[t + 1] * __uint_as_float(r[8 * q8 + 2 * j + 1]), h1, l1);
            hw[j] = pack2(h0, h1);
            lw[j] = pack2(l0, l1);
          }
          const uint32_t off = sw16(lj, c0 + 8 * q8, 128);
          *reinterpret_cast<uint4 *>(sm.yh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4 *>(sm.yl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      __syncthreads();

      // ---- H: chain 2, X^T += Ytilde^T K  (B = K tile, MN-major view)
      if (n == 0) {
        tc::tc_fence_after();
        const uint32_t kb = tc::smem_u32(kin), yhb = tc::smem_u32(sm.yh), ylb = tc::smem_u32(sm.yl);
#pragma unroll
        for (int ks = 0; ks < 4; ks++) {
          tc::mma_ss_f16(tm + TM_X, kdesc16(yhb, 16 * ks, 128), mndesc16(kb, 16 * ks), id_c2, 1u);
          tc::mma_ss_f16(tm + TM_X, kdesc16(ylb, 16 * ks, 128), mndesc16(kb, 16 * ks), id_c2, 1u);
        }
        tc::mma_commit(&sm.bar_x);
      }
      wait_mma(sm, p, &sm.bar_x, ph_x);

      // ---- I: rounded copy of X for the next chunk; this input buffer is
      // now consumed by every MMA: refill it with chunk ch + 2
#pragma unroll
      for (int cc = 0; cc < 64; cc += 32) {
        const int col = 64 * hsel + cc;
        uint32_t r[32];
        tc::tmem_ld32(trow(tm + TM_X, col), r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; j++) r[j] = tc::to_tf32(__uint_as_float(r[j]));
        tc::tmem_st32(trow(tm + TM_XR, col), r);
      }
      tc::tmem_wait_st();
      if (n == 0 && ch + 2 < n_ch && !aborted(sm)) issue_chunk(sm, it, ch + 2, b, s_half, kh, &tmap_k, &tmap_v);
      tc::tc_fence_before();
      __syncthreads();
      g_cur = g_nxt;
      b_cur = b_nxt;
    }

    // ---- epilogue: lane lj holds column lj of its half of [T | S]
    {
      const int64_t sh = (int64_t)it.slot * p.h_v + h;
      float *out = (s_half ? p.S_pool : p.T_pool) + sh * 128 * 128 + lj;
      bool bad = false;
#pragma unroll
      for (int cc = 0; cc < 64; cc += 32) {
        const int col = 64 * hsel + cc;
        uint32_t r[32];
        tc::tmem_ld32(trow(tm + TM_X, col), r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; j++) {
          const float x = __uint_as_float(r[j]);
          out[(int64_t)(col + j) * 128] = x;
          bad |= !finite_f(x);
        }
      }
      if ((p.flags & HYPIC_FLAG_CHECK_FINITE) && bad) report(p.status, HYPIC_STATUS_NONFINITE);
    }
    tc::tc_fence_before();
    __syncthreads();
  }
  // every copy issued for an item is consumed inside it: nothing in flight
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tm, 512);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// [n_tokens, heads, 128] bf16 as a 3-D map with 64-channel x 1-head x
// 64-token boxes and 128-byte swizzle
bool make_tmap_tokens(CUtensorMap *map, const void *base, int64_t n_tokens, int heads) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)n_tokens};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool build_tc_supported(const BuildParams &p) {
  auto a16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  return (p.variant == HYPIC_GDN || p.variant == HYPIC_DELTANET) && p.in_dtype == HYPIC_IN_BF16 && p.d_k == 128 &&
         p.d_v == 128 && a16(p.k) && a16(p.v);
}

cudaError_t launch_build_tc(const BuildParams &p, int64_t n_tokens, int n_items, int n_sm, uint32_t wait_limit,
                            cudaStream_t s) {
  CUtensorMap tk, tv;
  if (!make_tmap_tokens(&tk, p.k, n_tokens, p.h_k) || !make_tmap_tokens(&tv, p.v, n_tokens, p.h_v))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(BuildTcSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(build_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = n_sm < n_items ? n_sm : n_items;
  if (grid < 1) return cudaSuccess;
  BuildTcArgs a;
  a.p = p;
  a.wait_limit = wait_limit;
  a.debug_stall = debug_stall() ? 1 : 0;
  build_tc_kernel<<<grid, NT, smem, s>>>(a, tk, tv);
  return cudaGetLastError();
}

}  // namespace hypic
