// build_channel.cu -- tensor-core chunkwise segment build for the delta rule
// with a per-channel gate, T_t = (I - b_t k_t k_t^T) Diag(a_t), bf16 inputs,
// d_k = d_v = 128.
//
// Caches the pair (T_C, S(C|0)) of every (segment, value head) (HYPIC news
// pages, nav.aitube.vip §2.1: T_C the product of the body's token
// transitions, S(C|0) its final state from zero).  The body is consumed in
// chunks of C = 32 tokens.  With lam_t = sum_{j<=t} g_j (a d_k vector of
// log-gates), the strictly lower
//     M_ti = b_t sum_c k_t[c] k_i[c] exp(lam_t[c] - lam_i[c])     (i < t),
// A = (I + M)^-1 and F = A diag(b), the chunk acts on X = [T | S] as
//     W = F (K * exp(lam)),  U = F V,  Y = W X - [0 | U],
//     X <- Diag(exp(lam_C)) X - Khat^T Y,   Khat_i = k_i * exp(lam_C - lam_i),
// which is the token recurrence exactly (checked in fp64 against the token
// oracle).  Every exponential above is <= 1 for log-gates <= 0 except in M,
// whose terms pair a large and a small factor; M is formed in two 16-token
// sub-blocks of rows, each with its own reference point ref (lam just before
// the sub-block), as Q R^T with Q_t = k_t exp(lam_t - ref) and
// R_i = k_i exp(ref - lam_i), so that no factor leaves [e^-80, e^80] unless
// the gates move the log-decay by more than 80 inside a sub-block.  Such a
// chunk forms M term by term instead.
//
// Layout and pipeline follow the scalar-gate build: the kernel works on X^T
// (rows = the 256 columns of [T | S]) with both 128 x 128 halves in TMEM as
// fp32 accumulators, and two warp groups run one chunk apart:
//   P (warps 4-7) prepares chunk c+1 from its inputs alone
//       lam     per-channel prefix sums of the log-gate tile (TMA, fp32)
//       tiles   K * exp(lam) and Khat, split hi + lo in bf16
//       Gram    Q R^T on the legacy warp MMA (m16n8k16 bf16, operands split
//               hi + lo, one k-quarter per warp, partials summed in order)
//       UT      A = (I + M)^-1 (SIMT, 16 x 16 blocks)
//       W, U    W^T = (K exp(lam))^T F^T,  -U^T = -V^T F^T   kind::f16, split
//               (-U^T straight into the chain-1 accumulator);
//   X (warps 0-3) advances both halves through chunk c, S half first
//       W        staged from TMEM as chain 1's B operand (tf32, rounded)
//       chain 1  Y^T = X^T W^T (- U^T)                kind::tf32, A from TMEM
//       Ytilde   = -Y, split hi + lo
//       chain 2  X^T = X^T Diag(exp(lam_C)) + Ytilde^T Khat   kind::f16
// handing off through mbarriers.  fp32 accumulation throughout.
//
// Items are (segment, value head) in LPT order, pulled by an atomic ticket.
// K, V and the log-gates come in by TMA through two buffers; chunk c + 1 is
// copied in while chunk c is prepared.  All waits are bounded.
#include <cstddef>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc.cuh"

namespace hypic {

namespace {

constexpr int C = 32;      // tokens per chunk
constexpr int SB = 16;     // tokens per Gram sub-block
constexpr int NT = 256;    // threads: X group = warps 0-3, P group = warps 4-7
constexpr int NG = 128;    // threads per group
constexpr int BAR_X = 1, BAR_P = 2;
constexpr uint32_t DRAIN_LIMIT = 1u << 22;
constexpr float RANGE_MAX = 80.f;  // largest |exponent| of a Gram factor

// TMEM columns (512 allocated, one CTA per SM)
constexpr uint32_t TM_XT = 0;    // T half of X^T
constexpr uint32_t TM_XS = 128;  // S half of X^T
constexpr uint32_t TM_XR = 256;  // tf32-rounded copy of the half being chained: A of chain 1
constexpr uint32_t TM_Y = 384;   // chain 1 output [128 j x 32 t]; -U^T written there by P
constexpr uint32_t TM_W = 416;   // W^T [128 d x 32 t] (P group)

// K-major, 128-byte-swizzled tiles of R rows (4-byte elements 32 to a
// 128-byte row segment, 2-byte elements 64)
__device__ __forceinline__ uint32_t sw32(int r, int k, int R) {
  const uint32_t byte = (uint32_t)(k & 31) * 4u;
  return (uint32_t)((k >> 5) * R * 128 + r * 128) + ((((byte >> 4) ^ (uint32_t)(r & 7)) << 4) | (byte & 15u));
}
__device__ __forceinline__ uint32_t sw16(int r, int k, int R) {
  const uint32_t byte = (uint32_t)(k & 63) * 2u;
  return (uint32_t)((k >> 6) * R * 128 + r * 128) + ((((byte >> 4) ^ (uint32_t)(r & 7)) << 4) | (byte & 15u));
}
__device__ __forceinline__ uint64_t kdesc32(uint32_t base, int k, int R) {
  return tc::smem_desc(base + (uint32_t)((k >> 5) * R * 128 + (k & 31) * 4), 16, 1024, tc::SW_128B);
}
__device__ __forceinline__ uint64_t kdesc16(uint32_t base, int k, int R) {
  return tc::smem_desc(base + (uint32_t)((k >> 6) * R * 128 + (k & 63) * 2), 16, 1024, tc::SW_128B);
}
// MN-major view of a [32 token x 128 channel] tile in the TMA layout
// (channel contiguous, two 64-channel slabs 4 KiB apart): the K-step that
// starts at token t
__device__ __forceinline__ uint64_t mndesc(uint32_t base, int t) {
  return tc::smem_desc(base + (uint32_t)(t * 128), 4096, 1024, tc::SW_128B);
}
// byte offset of channels c8 .. c8 + 7 (c8 % 8 == 0) of token t in a
// [32 x 128] bf16 tile in the TMA layout
__device__ __forceinline__ uint32_t tile16(int t, int c8) {
  return (uint32_t)((c8 >> 6) * 4096 + t * 128) + ((((uint32_t)(c8 & 63) >> 3) ^ (uint32_t)(t & 7)) << 4);
}
// the log-gate / lam table [32 t x 128 c] fp32: lam is stored with the
// channel index XORed by 8 (t % 8), so that the warp-MMA fragment reads
// (8 rows x 4 column pairs) touch distinct banks
__device__ __forceinline__ int lsw(int t, int c) { return c ^ ((t & 7) << 3); }

struct __align__(1024) BuildChSmem {
  unsigned char kin[2][8192];   // K tiles [32 t x 128] bf16 (TMA layout)
  unsigned char vin[2][8192];   // V tiles
  float gin[2][C][128];         // log-gate tiles (TMA, plain rows); lam in place (swizzled columns)
  unsigned char wt[16384];      // W [32 t x 128 d] tf32, K-major: B of chain 1
  unsigned char khh[2][8192];   // Khat hi of chunk c in [c % 2] (TMA layout): B of chain 2
  unsigned char khl[2][8192];   //   lo
  unsigned char kgh[8192];      // K * exp(lam) hi (TMA layout): A of the W MMA
  unsigned char kgl[8192];      //   lo
  unsigned char yh[16384];      // Ytilde hi [128 j x 64 t] bf16 K-major (t < 32 used): A of chain 2
  unsigned char yl[16384];      //   lo
  unsigned char fh[4096];       // F = A diag(b) hi [32 t x 64 t'] bf16 K-major (t' < 32 used)
  unsigned char fl[4096];       //   lo
  float4 part[4][6][32];        // Gram partials: [warp = k quarter][tile][lane]
  float nm[C][C + 4];           // M (rows 16-byte aligned)
  float am[C][C + 2];           // A = (I + M)^-1 (rows 8-byte aligned)
  float pm[16][18];             // block product of the inverse
  float gcv[2][128];            // exp(lam_C) of chunk c in [c % 2] (read by X)
  float bt[C];
  int fb[4];                    // per-warp flags: a Gram factor out of range
  uint64_t full[2];
  uint64_t bar_wu;              // P's MMA completion
  uint64_t bar_y1, bar_y2;      // X's chain 1 completions (S half, T half)
  uint64_t bar_x1;              // X's chain 2 completion, S half
  uint64_t bar_x2[2];           // X's chain 2 completion, T half, of chunks g with g % 2 = [i]
                                // (phase g / 2)
  uint64_t wt_ready, ys_done;   // P -> X: W / U MMAs issued; X -> P: chain-1 output consumed
  uint64_t wg_free;             // X -> P: W read out of TM_W (the next W MMA may overwrite it)
  uint64_t never;
  uint32_t tmem_base;
  int item;
  int abort;
};

static_assert(offsetof(BuildChSmem, am) % 8 == 0 && offsetof(BuildChSmem, nm) % 16 == 0 &&
                  offsetof(BuildChSmem, part) % 16 == 0 && offsetof(BuildChSmem, gcv) % 16 == 0,
              "vector accesses");
static_assert(sizeof(BuildChSmem) + 1024 <= 232448, "shared memory");

struct BuildChArgs {
  BuildParams p;
  uint32_t wait_limit;
  int debug_stall;
};

__device__ __forceinline__ bool aborted(BuildChSmem &sm) { return *(volatile int *)&sm.abort != 0; }
__device__ __forceinline__ void fail(BuildChSmem &sm, const BuildParams &p) {
  *(volatile int *)&sm.abort = 1;
  report(p.status, HYPIC_STATUS_TIMEOUT);
}
__device__ __forceinline__ void wait_phase(BuildChSmem &sm, const BuildParams &p, uint64_t *bar, uint32_t ph,
                                           uint32_t lim) {
  if (!tc::mbar_wait(bar, ph & 1, aborted(sm) ? DRAIN_LIMIT : lim)) fail(sm, p);
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi), for a pair, packed (x0
// in the low half)
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  const float r0 = x0 - __uint_as_float(hi << 16), r1 = x1 - __uint_as_float(hi & 0xFFFF0000u);
  const __nv_bfloat162 l = __floats2bfloat162_rn(r0, r1);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// TMEM address of this thread's lane (warp w covers lanes 32 (w % 4) ..)
__device__ __forceinline__ uint32_t trow(uint32_t base, int col) {
  return base + ((uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16) + (uint32_t)col;
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- P group
// lam = per-channel prefix sums of the chunk's log-gates (zero past nt),
// written back in place with swizzled columns; exp(lam_C) for X; the range
// flag of the Gram factors.  Thread q owns channel q.
__device__ __forceinline__ void lam_pass(BuildChSmem &sm, int bk, int b2, int nt, int q) {
  float(*G)[128] = sm.gin[bk];
  float l[C];
  float acc = 0.f;
#pragma unroll
  for (int t = 0; t < C; t++) {
    acc += (t < nt) ? G[t][q] : 0.f;
    l[t] = acc;
  }
  // exponents of the Gram factors: sub-block 0 (ref 0) uses +-lam_t, t < 16;
  // sub-block 1 (ref lam_15) uses +-(lam_i - lam_15), i < 32
  float r = 0.f;
#pragma unroll
  for (int t = 0; t < C; t++) {
    if (t < SB) r = fmaxf(r, fabsf(l[t]));
    r = fmaxf(r, fabsf(l[t] - l[SB - 1]));
  }
  const unsigned bad = __ballot_sync(0xffffffffu, !(r <= RANGE_MAX));  // NaN counts as out of range
  if ((q & 31) == 0) sm.fb[q >> 5] = bad != 0u;
  sm.gcv[b2][q] = __expf(l[C - 1]);
  tc::named_bar(BAR_P, NG);  // every column has been read
#pragma unroll
  for (int t = 0; t < C; t++) G[t][lsw(t, q)] = l[t];
}

// K * exp(lam) (A of the W MMA) and Khat = K * exp(lam_C - lam) (B of chain
// 2), split hi + lo, in the TMA tile layout: thread q forms 8 channels of 4
// tokens.
__device__ __forceinline__ void tiles_pass(BuildChSmem &sm, int bk, int b2, int q) {
  const float(*L)[128] = sm.gin[bk];
  const unsigned char *kin = sm.kin[bk];
#pragma unroll 1
  for (int m = 0; m < 4; m++) {
    const int u = q + NG * m, t = u >> 4, c8 = (u & 15) << 3;
    const uint32_t off = tile16(t, c8);
    const uint4 kw = *reinterpret_cast<const uint4 *>(kin + off);
    const float4 l0 = *reinterpret_cast<const float4 *>(&L[t][lsw(t, c8)]);
    const float4 l1 = *reinterpret_cast<const float4 *>(&L[t][lsw(t, c8) + 4]);
    const float4 e0 = *reinterpret_cast<const float4 *>(&L[C - 1][lsw(C - 1, c8)]);
    const float4 e1 = *reinterpret_cast<const float4 *>(&L[C - 1][lsw(C - 1, c8) + 4]);
    const uint32_t kk[4] = {kw.x, kw.y, kw.z, kw.w};
    const float lt[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
    const float lc[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
    uint32_t gh[4], gl[4], hh[4], hl[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const float k0 = bf_lo(kk[j]), k1 = bf_hi(kk[j]);
      split_bf16x2(k0 * __expf(lt[2 * j]), k1 * __expf(lt[2 * j + 1]), gh[j], gl[j]);
      split_bf16x2(k0 * __expf(lc[2 * j] - lt[2 * j]), k1 * __expf(lc[2 * j + 1] - lt[2 * j + 1]), hh[j], hl[j]);
    }
    *reinterpret_cast<uint4 *>(sm.kgh + off) = make_uint4(gh[0], gh[1], gh[2], gh[3]);
    *reinterpret_cast<uint4 *>(sm.kgl + off) = make_uint4(gl[0], gl[1], gl[2], gl[3]);
    *reinterpret_cast<uint4 *>(sm.khh[b2] + off) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
    *reinterpret_cast<uint4 *>(sm.khl[b2] + off) = make_uint4(hl[0], hl[1], hl[2], hl[3]);
  }
}

// (k0 exp(e0), k1 exp(e1)) for the packed bf16 pair kw = (k0, k1), split
// hi + lo
__device__ __forceinline__ void factor_pair(uint32_t kw, float e0, float e1, uint32_t &hi, uint32_t &lo) {
  split_bf16x2(bf_lo(kw) * __expf(e0), bf_hi(kw) * __expf(e1), hi, lo);
}

// Gram partials on the legacy warp MMA: warp wp takes channels 32 wp ..
// 32 wp + 31.  Tiles (m16n8): 0, 1 = sub-block 0 (rows t 0..15) x columns
// i 0..7, 8..15; 2..5 = sub-block 1 (rows 16..31) x columns 0..31 in
// eighths.  Lane (g = lane / 4, u = lane % 4) ends with rows g, g + 8 and
// columns 2u, 2u + 1 of each tile.  The rows a lane's fragments touch are
// g + 8 rr (rr = 0..3), all with t % 8 = g, so each is loaded once and every
// factor it feeds is formed from it:
//     rows of sub-block 0:  Q0 = k exp(lam),  R0 = k exp(-lam),  R1 = k exp(lam_15 - lam)
//     rows of sub-block 1:  Q1 = k exp(lam - lam_15),  R1
// (ref 0 for sub-block 0, lam_15 for sub-block 1).
__device__ __forceinline__ void gram_pass(BuildChSmem &sm, int bk, int wp, int lane) {
  const float *L = &sm.gin[bk][0][0];
  const unsigned char *kin = sm.kin[bk];
  const int g = lane >> 2, u = lane & 3;
  float acc[6][4];
#pragma unroll
  for (int i = 0; i < 6; i++) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll 1
  for (int kk = 0; kk < 2; kk++) {
    const int c0 = 32 * wp + 16 * kk, c8 = (c0 & 63) >> 3;
    // byte offsets (within a row) of the k pairs at channels c0 + 2u and
    // c0 + 8 + 2u, and the lam columns of those pairs, for rows with t % 8 = g
    const uint32_t ko[2] = {(uint32_t)((c0 >> 6) * 4096 + ((c8 ^ g) << 4) + 4 * u),
                            (uint32_t)((c0 >> 6) * 4096 + (((c8 + 1) ^ g) << 4) + 4 * u)};
    const int lc[2] = {(c0 + 2 * u) ^ (g << 3), (c0 + 8 + 2 * u) ^ (g << 3)};
    uint32_t a0h[4], a0l[4], a1h[4], a1l[4], b0h[2][2], b0l[2][2], b1h[4][2], b1l[4][2];
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const float2 x = *reinterpret_cast<const float2 *>(&L[(SB - 1) * 128 + lsw(SB - 1, c0 + 8 * h + 2 * u)]);
#pragma unroll
      for (int rr = 0; rr < 4; rr++) {
        const int row = g + 8 * rr;
        const uint32_t kw = *reinterpret_cast<const uint32_t *>(kin + row * 128 + ko[h]);
        const float2 l = *reinterpret_cast<const float2 *>(&L[row * 128 + lc[h]]);
        if (rr < 2) {
          factor_pair(kw, l.x, l.y, a0h[2 * h + rr], a0l[2 * h + rr]);
          factor_pair(kw, -l.x, -l.y, b0h[rr][h], b0l[rr][h]);
        } else {
          factor_pair(kw, l.x - x.x, l.y - x.y, a1h[2 * h + rr - 2], a1l[2 * h + rr - 2]);
        }
        factor_pair(kw, x.x - l.x, x.y - l.y, b1h[rr][h], b1l[rr][h]);
      }
    }
#pragma unroll
    for (int n = 0; n < 2; n++) {
      float(&d)[4] = acc[n];
      mma_bf16_16816(d, a0h[0], a0h[1], a0h[2], a0h[3], b0h[n][0], b0h[n][1]);
      mma_bf16_16816(d, a0h[0], a0h[1], a0h[2], a0h[3], b0l[n][0], b0l[n][1]);
      mma_bf16_16816(d, a0l[0], a0l[1], a0l[2], a0l[3], b0h[n][0], b0h[n][1]);
    }
#pragma unroll
    for (int n = 0; n < 4; n++) {
      float(&d)[4] = acc[2 + n];
      mma_bf16_16816(d, a1h[0], a1h[1], a1h[2], a1h[3], b1h[n][0], b1h[n][1]);
      mma_bf16_16816(d, a1h[0], a1h[1], a1h[2], a1h[3], b1l[n][0], b1l[n][1]);
      mma_bf16_16816(d, a1l[0], a1l[1], a1l[2], a1l[3], b1h[n][0], b1h[n][1]);
    }
  }
#pragma unroll
  for (int i = 0; i < 6; i++) sm.part[wp][i][lane] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
}

// M = diag(b) (sum of the four partials, in warp order), strictly lower
__device__ __forceinline__ void gram_reduce(BuildChSmem &sm, int q) {
  for (int e = q; e < 6 * 32; e += NG) {
    const int tile = e >> 5, ln = e & 31, g = ln >> 2, u = ln & 3;
    float4 s = sm.part[0][tile][ln];
#pragma unroll
    for (int w = 1; w < 4; w++) {
      const float4 x = sm.part[w][tile][ln];
      s.x += x.x;
      s.y += x.y;
      s.z += x.z;
      s.w += x.w;
    }
    const int b = tile < 2 ? 0 : 1, n = tile < 2 ? tile : tile - 2;
    const int t0 = SB * b + g, t1 = t0 + 8, i0 = 8 * n + 2 * u;
    const float b0 = sm.bt[t0], b1 = sm.bt[t1];
    sm.nm[t0][i0] = i0 < t0 ? b0 * s.x : 0.f;
    sm.nm[t0][i0 + 1] = i0 + 1 < t0 ? b0 * s.y : 0.f;
    sm.nm[t1][i0] = i0 < t1 ? b1 * s.z : 0.f;
    sm.nm[t1][i0 + 1] = i0 + 1 < t1 ? b1 * s.w : 0.f;
  }
}

// M term by term (a chunk whose log-decay moves by more than the factor
// range inside a sub-block)
__device__ void gram_direct(BuildChSmem &sm, int bk, int q) {
  const float(*L)[128] = sm.gin[bk];
  const unsigned char *kin = sm.kin[bk];
  for (int e = q; e < C * C; e += NG) {
    const int t = e >> 5, i = e & 31;
    float s = 0.f;
    if (i < t) {
      for (int c = 0; c < 128; c++) {
        const float kt = __bfloat162float(
            *reinterpret_cast<const __nv_bfloat16 *>(kin + tile16(t, c & ~7) + (c & 7) * 2));
        const float ki = __bfloat162float(
            *reinterpret_cast<const __nv_bfloat16 *>(kin + tile16(i, c & ~7) + (c & 7) * 2));
        s = fmaf(kt * ki, __expf(L[t][lsw(t, c)] - L[i][lsw(i, c)]), s);
      }
    }
    sm.nm[t][i] = (i < t) ? sm.bt[t] * s : 0.f;
  }
}

// A = (I + N)^-1 for the strictly lower 32 x 32 N in sm.nm, into sm.am:
// the two diagonal 16 x 16 blocks by forward substitution (one thread per
// column), then A_10 = -A_11 (N_10 A_00).  Ends with a group barrier.
__device__ void ut_inverse(BuildChSmem &sm, int q) {
  if (q < 32) {
    const int b = SB * (q >> 4), l = q & 15;
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
  } else if (q < 64) {  // the upper block is zero
    const int r = q - 32;
    if (r < 16) {
#pragma unroll
      for (int c = 0; c < 16; c += 2) *reinterpret_cast<float2 *>(&sm.am[r][SB + c]) = make_float2(0.f, 0.f);
    }
  }
  tc::named_bar(BAR_P, NG);
  const int r = 2 * (q >> 3), c = 2 * (q & 7);
  if (q < 64) {  // pm = N_10 A_00
    float s00 = 0.f, s01 = 0.f, s10 = 0.f, s11 = 0.f;
#pragma unroll
    for (int m = 0; m < 16; m++) {
      const float n0 = sm.nm[SB + r][m], n1 = sm.nm[SB + r + 1][m];
      const float2 a = *reinterpret_cast<const float2 *>(&sm.am[m][c]);
      s00 = fmaf(n0, a.x, s00);
      s01 = fmaf(n0, a.y, s01);
      s10 = fmaf(n1, a.x, s10);
      s11 = fmaf(n1, a.y, s11);
    }
    *reinterpret_cast<float2 *>(&sm.pm[r][c]) = make_float2(s00, s01);
    *reinterpret_cast<float2 *>(&sm.pm[r + 1][c]) = make_float2(s10, s11);
  }
  tc::named_bar(BAR_P, NG);
  if (q < 64) {  // A_10 = -A_11 pm
    float s00 = 0.f, s01 = 0.f, s10 = 0.f, s11 = 0.f;
#pragma unroll
    for (int m = 0; m < 16; m++) {
      const float a0 = sm.am[SB + r][SB + m], a1 = sm.am[SB + r + 1][SB + m];
      const float2 pv = *reinterpret_cast<const float2 *>(&sm.pm[m][c]);
      s00 = fmaf(a0, pv.x, s00);
      s01 = fmaf(a0, pv.y, s01);
      s10 = fmaf(a1, pv.x, s10);
      s11 = fmaf(a1, pv.y, s11);
    }
    *reinterpret_cast<float2 *>(&sm.am[SB + r][c]) = make_float2(-s00, -s01);
    *reinterpret_cast<float2 *>(&sm.am[SB + r + 1][c]) = make_float2(-s10, -s11);
  }
  tc::named_bar(BAR_P, NG);
}

// F = A diag(b), split hi + lo, as the K-major B tiles [32 t x 32 t'] of the
// W and U MMAs: thread q writes 8 consecutive t' of row q / 4.
__device__ __forceinline__ void write_factors(BuildChSmem &sm, int q) {
  const int t = q >> 2, c0 = 8 * (q & 3);
  uint32_t h[4], l[4];
#pragma unroll
  for (int j = 0; j < 4; j++) {
    const float2 a = *reinterpret_cast<const float2 *>(&sm.am[t][c0 + 2 * j]);
    split_bf16x2(a.x * sm.bt[c0 + 2 * j], a.y * sm.bt[c0 + 2 * j + 1], h[j], l[j]);
  }
  const uint32_t off = sw16(t, c0, C);
  *reinterpret_cast<uint4 *>(sm.fh + off) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4 *>(sm.fl + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

// K, V and the log-gates of chunk `ch` of item `it`, into input buffer ch % 2
__device__ __forceinline__ void issue_chunk(BuildChSmem &sm, const BuildItem &it, int ch, int kh,
                                            const CUtensorMap *tk, const CUtensorMap *tv, const CUtensorMap *tg) {
  const int32_t t0 = (int32_t)(it.start + (int64_t)C * ch);
  const int b = ch & 1;
  tc::mbar_expect_tx(&sm.full[b], 4 * 4096u + (uint32_t)sizeof(sm.gin[0]));
  for (int s = 0; s < 2; s++) tc::tma_load_3d(sm.kin[b] + s * 4096, tk, 64 * s, kh, t0, &sm.full[b]);
  for (int s = 0; s < 2; s++) tc::tma_load_3d(sm.vin[b] + s * 4096, tv, 64 * s, it.head, t0, &sm.full[b]);
  tc::tma_load_3d(&sm.gin[b][0][0], tg, 0, it.head, t0, &sm.full[b]);
}

struct ItemCtx {
  BuildItem it;
  int kh;
  int n_ch;
  uint32_t gch0;  // index of the item's first chunk in this CTA's chunk sequence
};

struct MmaIds {
  uint32_t wu, wu_neg, c1, c2;
};

// Prepares chunk ch (q = thread index in the group).  Once-per-chunk
// barriers are waited on with the phase of the chunk they belong to (global
// chunk index g).
__device__ void prep_chunk(BuildChSmem &sm, const BuildParams &p, const ItemCtx &x, int ch, int q, uint32_t tm,
                           const MmaIds &id, uint32_t LIM, uint32_t (&ph_full)[2], float &b_cur,
                           const CUtensorMap *tk, const CUtensorMap *tv, const CUtensorMap *tg) {
  const BuildItem &it = x.it;
  const uint32_t g = x.gch0 + (uint32_t)ch;
  const int bk = ch & 1, b2 = (int)(g & 1);
  const int64_t t0 = it.start + (int64_t)C * ch;
  const int nt = (it.end - t0) < C ? (int)(it.end - t0) : C;
  const int wp = q >> 5, lane = q & 31;
  float b_nxt = 0.f;  // beta of the next chunk, one chunk ahead
  if (q < C && t0 + C + q < it.end) b_nxt = p.beta[(t0 + C + q) * p.h_v + it.head];
  // ---- inputs landed; ragged tail -> identity tokens (k = v = 0, g = 0)
  if (!tc::mbar_wait(&sm.full[bk], ph_full[bk] & 1, aborted(sm) ? DRAIN_LIMIT : LIM)) fail(sm, p);
  ph_full[bk]++;
  if (nt < C) {
    for (int e = q; e < (C - nt) * 16; e += NG) {
      const int r = nt + (e >> 4), s = (e >> 3) & 1, c16 = e & 7;
      const uint4 zz = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(sm.kin[bk] + s * 4096 + r * 128 + c16 * 16) = zz;
      *reinterpret_cast<uint4 *>(sm.vin[bk] + s * 4096 + r * 128 + c16 * 16) = zz;
    }
  }
  if (q < C) sm.bt[q] = b_cur;
  // the Khat buffer and exp(lam_C) slot of this chunk held chunk g - 2: its
  // chain 2 (the last reader) must be complete.  That barrier's next phase is
  // chunk g's, which needs this chunk's wt_ready: the phase waited on is its
  // latest.  (An item's first two chunks follow the item barrier.)
  if (ch >= 2) wait_phase(sm, p, &sm.bar_x2[(g - 2) & 1], (g - 2) >> 1, LIM);
  lam_pass(sm, bk, b2, nt, q);
  tc::named_bar(BAR_P, NG);
  const bool direct = (sm.fb[0] | sm.fb[1] | sm.fb[2] | sm.fb[3]) != 0;  // uniform over the group
  tiles_pass(sm, bk, b2, q);
  if (q == 0 && ch >= 1 && ch + 1 < x.n_ch) {
    // chunk ch + 1 goes to input buffer (ch + 1) % 2, which held chunk ch - 1:
    // its U MMA (the last reader of its V tile) is complete once bar_wu of
    // chunk g - 1 is (the phase waited on is the latest: the next one needs
    // this chunk's W / U MMAs, issued below)
    wait_phase(sm, p, &sm.bar_wu, g - 1, LIM);
    if (!aborted(sm)) issue_chunk(sm, it, ch + 1, x.kh, tk, tv, tg);
  }
  if (!direct) {
    gram_pass(sm, bk, wp, lane);
    tc::named_bar(BAR_P, NG);
    gram_reduce(sm, q);
  } else {
    gram_direct(sm, bk, q);
  }
  tc::named_bar(BAR_P, NG);
  ut_inverse(sm, q);
  write_factors(sm, q);
  tc::fence_proxy_async_smem();  // zeroed rows, tiles and factors are MMA operands
  tc::tc_fence_before();
  tc::named_bar(BAR_P, NG);
  // ---- W^T = (K exp(lam))^T F^T, and -U^T = -V^T F^T straight into the
  // chain-1 accumulator once X has consumed the previous chunk's chain-1 output
  if (g > 0) {
    wait_phase(sm, p, &sm.ys_done, g - 1, LIM);
    wait_phase(sm, p, &sm.wg_free, g - 1, LIM);  // X has read the previous W out of TM_W
  }
  if (q == 0 || q == 32) {
    // two issuers (lane 0 of the first two warps), one accumulator each: W
    // into TM_W, -U into TM_Y; X waits for both commits and both arrivals
    tc::tc_fence_after();
    const uint32_t fh = tc::smem_u32(sm.fh), fl = tc::smem_u32(sm.fl);
    if (q == 0) {
      const uint32_t gh = tc::smem_u32(sm.kgh), gl = tc::smem_u32(sm.kgl);
#pragma unroll
      for (int ks = 0; ks < 2; ks++) {
        tc::mma_ss_f16(tm + TM_W, mndesc(gh, 16 * ks), kdesc16(fh, 16 * ks, C), id.wu, ks > 0);
        tc::mma_ss_f16(tm + TM_W, mndesc(gh, 16 * ks), kdesc16(fl, 16 * ks, C), id.wu, 1u);
        tc::mma_ss_f16(tm + TM_W, mndesc(gl, 16 * ks), kdesc16(fh, 16 * ks, C), id.wu, 1u);
      }
    } else {
      const uint32_t vb = tc::smem_u32(sm.vin[bk]);
#pragma unroll
      for (int ks = 0; ks < 2; ks++) {
        tc::mma_ss_f16(tm + TM_Y, mndesc(vb, 16 * ks), kdesc16(fh, 16 * ks, C), id.wu_neg, ks > 0);
        tc::mma_ss_f16(tm + TM_Y, mndesc(vb, 16 * ks), kdesc16(fl, 16 * ks, C), id.wu_neg, 1u);
      }
    }
    tc::mma_commit(&sm.bar_wu);
    tc::mbar_arrive(&sm.wt_ready);  // hand chunk g to X
  }
  b_cur = b_nxt;
}

// ---------------------------------------------------------------- X group
// XR <- RN(X_h) (chain 1 reads the start-of-chunk state), X_h <- X_h
// Diag(exp(lam_C)) (TMEM column d = row d of X), in one pass over the half.
__device__ __forceinline__ void stage_half(uint32_t tm, uint32_t tx, const float *gC) {
#pragma unroll 1
  for (int c0 = 0; c0 < 128; c0 += 64) {
    uint32_t r[64];
    tc::tmem_ld32(trow(tm + tx, c0), *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
    tc::tmem_ld32(trow(tm + tx, c0 + 32), *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
    tc::tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < 2; h++) {
      uint32_t xr[32];
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const float4 s4 = *reinterpret_cast<const float4 *>(&gC[c0 + 32 * h + j]);
        const float sc[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const float v = __uint_as_float(r[32 * h + j + e]);
          xr[j + e] = tc::to_tf32_fast(v);  // X itself keeps any NaN (it is the accumulator)
          r[32 * h + j + e] = __float_as_uint(sc[e] * v);
        }
      }
      tc::tmem_st32(trow(tm + TM_XR, c0 + 32 * h), xr);
    }
    tc::tmem_st32(trow(tm + tx, c0), *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
    tc::tmem_st32(trow(tm + tx, c0 + 32), *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
  }
  tc::tmem_wait_st();
}

// chain 1 into TM_Y: Y^T (+)= XR^T W^T (issued by lane 0 of the group)
__device__ __forceinline__ void issue_chain1(BuildChSmem &sm, uint32_t tm, const MmaIds &id, bool onto_u,
                                             uint64_t *bar) {
  tc::tc_fence_after();
  const uint32_t wb = tc::smem_u32(sm.wt);
#pragma unroll
  for (int ks = 0; ks < 16; ks++)
    tc::mma_ts_tf32(tm + TM_Y, tm + TM_XR + 8 * ks, kdesc32(wb, 8 * ks, C), id.c1, (onto_u || ks > 0) ? 1u : 0u);
  tc::mma_commit(bar);
}

// chain 2 into the half tx: X^T += Ytilde^T Khat (B = the chunk's Khat tiles,
// MN-major)
__device__ __forceinline__ void issue_chain2(BuildChSmem &sm, uint32_t tm, uint32_t tx, int b2, const MmaIds &id,
                                             uint64_t *bar) {
  tc::tc_fence_after();
  const uint32_t kh = tc::smem_u32(sm.khh[b2]), kl = tc::smem_u32(sm.khl[b2]);
  const uint32_t yhb = tc::smem_u32(sm.yh), ylb = tc::smem_u32(sm.yl);
#pragma unroll
  for (int ks = 0; ks < 2; ks++) {
    tc::mma_ss_f16(tm + tx, kdesc16(yhb, 16 * ks, 128), mndesc(kh, 16 * ks), id.c2, 1u);
    tc::mma_ss_f16(tm + tx, kdesc16(ylb, 16 * ks, 128), mndesc(kh, 16 * ks), id.c2, 1u);
    tc::mma_ss_f16(tm + tx, kdesc16(yhb, 16 * ks, 128), mndesc(kl, 16 * ks), id.c2, 1u);
  }
  tc::mma_commit(bar);
}

// Ytilde = -Y, split hi + lo, as the K-major A tiles [128 j x 32 t] of chain
// 2 (the S half's Y already holds -U)
__device__ __forceinline__ void split_y(BuildChSmem &sm, uint32_t tm, int n) {
  uint32_t r[32];
  tc::tmem_ld32(trow(tm + TM_Y, 0), r);
  tc::tmem_wait_ld();
#pragma unroll
  for (int q8 = 0; q8 < 4; q8++) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int jj = 8 * q8 + 2 * j;
      split_bf16x2(-__uint_as_float(r[jj]), -__uint_as_float(r[jj + 1]), hw[j], lw[j]);
    }
    const uint32_t off = sw16(n, 8 * q8, 128);
    *reinterpret_cast<uint4 *>(sm.yh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4 *>(sm.yl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
}

// Advances both halves of the state through chunk ch (n = thread = TMEM
// lane), the S half first: its chain 1 accumulates onto the -U^T that P put
// in TM_Y.
__device__ void chain_chunk(BuildChSmem &sm, const BuildParams &p, const ItemCtx &x, int ch, int n, uint32_t tm,
                            const MmaIds &id, uint32_t LIM) {
  const uint32_t g = x.gch0 + (uint32_t)ch;
  const int b2 = (int)(g & 1);
  wait_phase(sm, p, &sm.wt_ready, g, LIM);
  // ---- W (tf32, rounded) as chain 1's B tile once P's W / U MMAs are
  // complete (lane n holds row n of W^T; the previous chunk's chain 1 that
  // read the tile was waited on before its Ytilde)
  wait_phase(sm, p, &sm.bar_wu, g, DRAIN_LIMIT);
  tc::tc_fence_after();
  {
    uint32_t r[32];
    tc::tmem_ld32(trow(tm + TM_W, 0), r);
    tc::tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; j++)
      // a NaN in W comes from an input that reaches X through K, U or the
      // gates as well
      *reinterpret_cast<uint32_t *>(sm.wt + sw32(j, n, C)) = tc::to_tf32_fast(__uint_as_float(r[j]));
  }
  tc::fence_proxy_async_smem();
  const float *gC = sm.gcv[b2];
  // ---- S half (its chain 2 of the previous chunk was waited on before the
  // T half's Ytilde)
  stage_half(tm, TM_XS, gC);
  tc::tc_fence_before();
  tc::named_bar(BAR_X, NG);
  if (n == 0) {
    tc::mbar_arrive(&sm.wg_free);  // TM_W is free for the next chunk's W
    issue_chain1(sm, tm, id, true, &sm.bar_y1);
  }
  wait_phase(sm, p, &sm.bar_y1, g, DRAIN_LIMIT);
  tc::tc_fence_after();
  split_y(sm, tm, n);
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  tc::named_bar(BAR_X, NG);
  if (n == 0) issue_chain2(sm, tm, TM_XS, b2, id, &sm.bar_x1);
  // ---- T half: XR is free (chain 1 of S is complete); the T half's chain 2
  // of the previous chunk must be
  if (ch > 0) wait_phase(sm, p, &sm.bar_x2[(g - 1) & 1], (g - 1) >> 1, DRAIN_LIMIT);
  tc::tc_fence_after();
  stage_half(tm, TM_XT, gC);
  tc::tc_fence_before();
  tc::named_bar(BAR_X, NG);
  if (n == 0) issue_chain1(sm, tm, id, false, &sm.bar_y2);
  wait_phase(sm, p, &sm.bar_y2, g, DRAIN_LIMIT);
  // the Ytilde tiles are free once the S half's chain 2 has read them
  wait_phase(sm, p, &sm.bar_x1, g, DRAIN_LIMIT);
  tc::tc_fence_after();
  split_y(sm, tm, n);
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  tc::named_bar(BAR_X, NG);
  if (n == 0) {
    tc::mbar_arrive(&sm.ys_done);  // TM_Y is free for the next chunk's -U
    issue_chain2(sm, tm, TM_XT, b2, id, &sm.bar_x2[g & 1]);
  }
}

__global__ void __launch_bounds__(NT, 1)
    build_channel_kernel(const __grid_constant__ BuildChArgs args, const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_g) {
  extern __shared__ unsigned char smem_raw[];
  BuildChSmem &sm =
      *reinterpret_cast<BuildChSmem *>(smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  const BuildParams &p = args.p;
  const uint32_t LIM = args.wait_limit;
  const int n = threadIdx.x, warp = n >> 5;
  const bool is_p = warp >= 4;
  const int q = n - NG;

  if (n == 0) {
    for (int b = 0; b < 2; b++) tc::mbar_init(&sm.full[b], 1);
    tc::mbar_init(&sm.bar_wu, 2);
    tc::mbar_init(&sm.bar_y1, 1);
    tc::mbar_init(&sm.bar_y2, 1);
    tc::mbar_init(&sm.bar_x1, 1);
    tc::mbar_init(&sm.bar_x2[0], 1);
    tc::mbar_init(&sm.bar_x2[1], 1);
    tc::mbar_init(&sm.wt_ready, 2);
    tc::mbar_init(&sm.ys_done, 1);
    tc::mbar_init(&sm.wg_free, 1);
    tc::mbar_init(&sm.never, 1);
    sm.abort = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmap_k);
    tc::prefetch_tmap(&tmap_v);
    tc::prefetch_tmap(&tmap_g);
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

  MmaIds id;
  id.wu = tc::idesc(tc::FMT_BF16, 128, C, false, false, /*a_mn=*/true, false);
  id.wu_neg = tc::idesc(tc::FMT_BF16, 128, C, /*neg_a=*/true, false, /*a_mn=*/true, false);
  id.c1 = tc::idesc(tc::FMT_TF32, 128, C);
  id.c2 = tc::idesc(tc::FMT_BF16, 128, 128, false, false, false, /*b_mn=*/true);
  uint32_t ph_full[2] = {0, 0};
  uint32_t gch = 0;  // chunks processed by this CTA so far
  const int n_items = p.plan->n_items;
  int taken = 0;  // items fetched by this CTA (thread n == 0)

  for (;;) {
    if (n == 0) sm.item = aborted(sm) ? n_items : take_item(p.plan, taken);
    __syncthreads();
    const int idx = sm.item;
    __syncthreads();
    if (idx >= n_items) break;
    ItemCtx x;
    x.it = p.items[idx];
    x.kh = (int)(((int64_t)x.it.head * p.h_k) / p.h_v);
    x.n_ch = (int)((x.it.end - x.it.start + C - 1) / C);
    x.gch0 = gch;

    if (is_p) {
      if (q == 0)  // chunks 0 and 1; chunk c + 2 is issued at the end of prep(c)
        for (int ch = 0; ch < 2 && ch < x.n_ch; ch++) issue_chunk(sm, x.it, ch, x.kh, &tmap_k, &tmap_v, &tmap_g);
      float b_cur = 0.f;
      if (q < C && x.it.start + q < x.it.end) b_cur = p.beta[(x.it.start + q) * p.h_v + x.it.head];
      for (int ch = 0; ch < x.n_ch; ch++)
        prep_chunk(sm, p, x, ch, q, tm, id, LIM, ph_full, b_cur, &tmap_k, &tmap_v, &tmap_g);
    } else {
      // X^T := [I | 0]
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t r[32], z[32];
#pragma unroll
        for (int j = 0; j < 32; j++) {
          r[j] = (c0 + j == n) ? 0x3f800000u : 0u;
          z[j] = 0u;
        }
        tc::tmem_st32(trow(tm + TM_XT, c0), r);
        tc::tmem_st32(trow(tm + TM_XS, c0), z);
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
      tc::named_bar(BAR_X, NG);
      for (int ch = 0; ch < x.n_ch; ch++) chain_chunk(sm, p, x, ch, n, tm, id, LIM);
      if (x.n_ch > 0) {
        const uint32_t gl = gch + (uint32_t)x.n_ch - 1;
        wait_phase(sm, p, &sm.bar_x2[gl & 1], gl >> 1, DRAIN_LIMIT);
        tc::tc_fence_after();
      }
      // epilogue: lane n holds column n of T and of S
      const int64_t sh = ((int64_t)x.it.slot * p.h_v + x.it.head) * 128 * 128 + n;
      bool bad = false;
#pragma unroll 1
      for (int h = 0; h < 2; h++) {
        float *out = (h ? p.S_pool : p.T_pool) + sh;
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t r[32];
          tc::tmem_ld32(trow(tm + (h ? TM_XS : TM_XT), c0), r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; j++) {
            const float v = __uint_as_float(r[j]);
            out[(int64_t)(c0 + j) * 128] = v;
            bad |= !finite_f(v);
          }
        }
      }
      if ((p.flags & HYPIC_FLAG_CHECK_FINITE) && bad) report(p.status, HYPIC_STATUS_NONFINITE);
    }
    gch += (uint32_t)x.n_ch;
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

}  // namespace

bool build_channel_supported(const BuildParams &p) {
  auto a16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  return p.variant == HYPIC_CHANNEL_DELTA && p.in_dtype == HYPIC_IN_BF16 && p.d_k == 128 && p.d_v == 128 &&
         a16(p.k) && a16(p.v) && a16(p.g);
}

cudaError_t launch_build_channel(const BuildParams &p, int64_t n_tokens, int n_items, int n_sm, uint32_t wait_limit,
                                 cudaStream_t s) {
  CUtensorMap tk, tv, tg;
  if (!make_tmap_tokens(&tk, p.k, n_tokens, p.h_k, C) || !make_tmap_tokens(&tv, p.v, n_tokens, p.h_v, C) ||
      !make_tmap_3d(&tg, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.g, n_tokens, p.h_v, 128, C,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(BuildChSmem) + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(build_channel_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = n_sm < n_items ? n_sm : n_items;
  if (grid < 1) return cudaSuccess;
  BuildChArgs a;
  a.p = p;
  a.wait_limit = wait_limit;
  a.debug_stall = debug_stall() ? 1 : 0;
  build_channel_kernel<<<grid, NT, smem, s>>>(a, tk, tv, tg);
  return cudaGetLastError();
}

}  // namespace hypic
