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
// [T | S].  The T half and the S half are independent chains that share the
// chunk's preparation (W, and U for S), so one CTA owns one (segment, head):
// both 128 x 128 halves of X^T stay in TMEM as fp32 accumulators (lane j =
// column j of the half, TMEM column d), and one tf32-rounded copy, the A
// operand of chain 1, is restaged for each half in turn.
// The TMA-loaded bf16 K and V tiles [64 tokens x 128] are MMA operands as
// they land -- K-major for the Gram, MN-major (transposed view) elsewhere --
// so no operand is ever transposed by the threads.
//
// Two warp groups run one chunk apart:
//   P (warps 4-7) prepares chunk c+1 from its inputs alone
//       Gram   K K^T                              kind::f16, exact inputs
//       UT     A = (I + M)^-1                     recursive doubling: 16 x 16
//                                                 diagonal blocks SIMT, the rest
//                                                 on the legacy warp MMA
//       W, U   W^T = K^T (A diag(bG))^T,  U^T = V^T (A diag(b))^T
//                                                 kind::f16, factors split hi + lo
//       (U goes straight to the chain-1 accumulator as -U^T);
//   X (warps 0-3) advances both halves through chunk c, S half first
//       W        staged from TMEM as chain 1's B operand (tf32, rounded)
//       chain 1  Y^T = X^T W^T (- U^T)            kind::tf32, A from TMEM
//       Ytilde   = -Y diag(exp(lam_C - lam)), split hi + lo
//       chain 2  X^T = G_C X^T + Ytilde^T K       kind::f16 (B = K tile, MN-major)
// handing off through mbarriers.  Split operands make W, U and chain 2 exact
// to ~2^-17 (K and V are exact bf16); chain 1 uses tf32 operands rounded to
// nearest by the threads (the tensor core itself truncates fp32 operands).
// fp32 accumulation throughout.  This keeps long products (8192 tokens)
// inside 5e-3 per head.
//
// Items are (segment, value head) in LPT order, pulled by an atomic
// ticket.  Inputs come in by TMA (3-D maps over [token, head, channel],
// 128-byte swizzle) through three K and two V buffers; chunk c + 1 is
// copied in while chunk c is prepared.  X stages W itself once P's W / U
// MMAs are complete, so P hands a chunk over as soon as they are issued.
// All waits are bounded.
#include <cstddef>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc.cuh"

namespace hypic {

namespace {

constexpr int C = 64;      // tokens per chunk
constexpr int NT = 256;    // threads: X group = warps 0-3, P group = warps 4-7
constexpr int NG = 128;    // threads per group
constexpr int NBUF = 3;    // input buffers
constexpr int BAR_X = 1, BAR_P = 2;  // named barriers of the two groups
constexpr uint32_t DRAIN_LIMIT = 1u << 22;

// TMEM columns (512 allocated, one CTA per SM)
constexpr uint32_t TM_XT = 0;    // T half of X^T, fp32 accumulator  (X group)
constexpr uint32_t TM_XS = 128;  // S half of X^T, fp32 accumulator  (X group)
constexpr uint32_t TM_XR = 256;  // tf32-rounded copy of the half being chained: A of chain 1
constexpr uint32_t TM_Y = 384;   // chain 1 output; -U^T written there by P before the S half's chain 1
constexpr uint32_t TM_WG = 448;  // K K^T (lanes 0..63), then W^T   (P group)

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

// An item as the X group needs it (slot / head of the output, chunk count,
// index of its first chunk in the CTA's chunk sequence); valid = 0 ends the
// sequence.
struct XItem {
  int32_t slot, head, n_ch, valid;
  uint32_t gch0;
  int32_t cbase;  // recording build: index of the item's first chunk record
};
// The copy issuer of the P group (its thread 0; kept in shared memory):
// chunks are loaded in the CTA's chunk order, one ahead of the chunk being
// prepared, from the current item and the next one (fetched one item ahead).
struct Issuer {
  BuildItem it[2];  // [0] the current item, [1] the next
  int kh[2], nch[2];
  bool ok[2];
  int w, ch;        // cursor: chunk ch of it[w]
  uint32_t g;       // the CTA's index of the chunk at the cursor
  int taken;        // items fetched by this CTA so far
};
struct PItem {
  BuildItem it;
  int32_t kh, n_ch, valid;
  uint32_t gch0;
};

struct __align__(1024) BuildTcSmem {
  // inputs as TMA tiles [64 t x 128] bf16 in two 64-channel slabs: K of
  // chunk c in kin[c % 3] (read by P's Gram and W and by X's chains 2 one
  // chunk later), V in vin[c % 2] (read only by P's U MMA).  V follows K so
  // the Gram's padded rows 64..127 read valid (ignored) bytes.
  unsigned char kin[NBUF][16384];
  unsigned char vin[2][16384];
  unsigned char wt[32768];      // W  [64 t x 128 d] tf32, K-major: B of chain 1
  unsigned char yh[16384];      // Ytilde hi [128 j x 64 t] bf16: A of chain 2
  unsigned char yl[16384];      // Ytilde lo
  unsigned char bwh[8192];      // A diag(bG) hi [64 t x 64 t'] bf16: B of the W MMA
  unsigned char bwl[8192];      //   lo
  unsigned char buh[8192];      // A diag(b) hi: B of the U MMA
  unsigned char bul[8192];      //   lo
  float nm[64][68];             // M (rows 16-byte aligned for vector stores)
  float am[64][68];             // A = (I + M)^-1 (pitch 68: conflict-free fragment columns)
  float lam[64], bg[64], bt[64];
  float ea[64], eb[64];         // b_t exp(lam_t - lam_0), exp(lam_0 - lam_i): M_ti = ea_t eb_i k_t.k_i
  float dec[3][64];             // exp(lam_C - lam_t) of chunk c in [c % 3] (read by X; pair loads)
  float gc[3];                  // G_C of chunk c in [c % 3] (read by X)
  int fact;                     // the factored form is in range for this chunk
  uint64_t full[NBUF];
  uint64_t bar_g, bar_wu;       // P's MMA completions
  uint64_t bar_y1, bar_y2;      // X's chain 1 completions (S half, T half; P waits on the T half's)
  uint64_t bar_x1;              // X's chain 2 completion, S half
  uint64_t bar_x2[2];           // X's chain 2 completion, T half, of chunks g with g % 2 = [i]
                                // (phase g / 2): P can wait for chunk g - 2 while chunk g - 1
                                // may already be complete
  uint64_t wt_ready, ys_done;   // P -> X: W / U MMAs issued; X -> P: chain-1 output consumed
  uint64_t wg_free;             // X -> P: W read out of TM_WG (the next Gram may overwrite it)
  uint64_t never;
  uint64_t item_full[2], item_free[2];  // P -> X item hand-off (two slots)
  XItem xslot[2];
  PItem pitem;                  // the P group's current item (broadcast by its thread 0)
  Issuer iss;
  uint32_t tmem_base;
  int abort;
};

static_assert(offsetof(BuildTcSmem, dec) % 8 == 0 && offsetof(BuildTcSmem, am) % 8 == 0, "pair loads");

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
// bounded wait on phase `ph` of an mbarrier that completes once per chunk
__device__ __forceinline__ void wait_phase(BuildTcSmem &sm, const BuildParams &p, uint64_t *bar, uint32_t ph,
                                           uint32_t lim) {
  if (!tc::mbar_wait(bar, ph & 1, aborted(sm) ? DRAIN_LIMIT : lim)) fail(sm, p);
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi), for a pair, packed (x0
// in the low half): one paired conversion for the high parts, one for the
// exact residuals
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  const float r0 = x0 - __uint_as_float(hi << 16), r1 = x1 - __uint_as_float(hi & 0xFFFF0000u);
  const __nv_bfloat162 l = __floats2bfloat162_rn(r0, r1);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}
// TMEM address of this thread's lane (warp w covers lanes 32 (w % 4) ..)
__device__ __forceinline__ uint32_t trow(uint32_t base, int col) {
  return base + ((uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16) + (uint32_t)col;
}
// ---------------------------------------------------------------- UT inverse
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Accumulator of one 16 x 16 block product on the warp MMA (two n-tiles),
// kept as three independent partial sums (hi*hi, hi*lo, lo*hi) so that the
// three products of a split operand pair do not wait on one another.
struct Acc3 {
  float d[3][2][4];
};
__device__ __forceinline__ void acc_zero(Acc3 &c) {
#pragma unroll
  for (int s = 0; s < 3; s++)
#pragma unroll
    for (int n = 0; n < 2; n++) c.d[s][n][0] = c.d[s][n][1] = c.d[s][n][2] = c.d[s][n][3] = 0.f;
}
// c += Z Y^T for the A operand Z (fragments split hi + lo in ah / al) and
// Y a 16 x 16 block in shared memory (pitch yp): element (k, n) of the B
// operand is Y[n][k]
__device__ __forceinline__ void acc_mma(Acc3 &c, const uint32_t (&ah)[4], const uint32_t (&al)[4], const float *Y,
                                        int yp, int g, int u) {
#pragma unroll
  for (int nt = 0; nt < 2; nt++) {
    const float *Yr = Y + (8 * nt + g) * yp;
    const float2 y0 = *reinterpret_cast<const float2 *>(&Yr[2 * u]);
    const float2 y1 = *reinterpret_cast<const float2 *>(&Yr[2 * u + 8]);
    uint32_t bh0, bl0, bh1, bl1;
    split_bf16x2(y0.x, y0.y, bh0, bl0);
    split_bf16x2(y1.x, y1.y, bh1, bl1);
    mma16816(c.d[0][nt], ah, bh0, bh1);
    mma16816(c.d[1][nt], ah, bl0, bl1);
    mma16816(c.d[2][nt], al, bh0, bh1);
  }
}
// A operand X^T for a 16 x 16 block X in shared memory (pitch xp): element
// (m, k) = X[k][m], split hi + lo
__device__ __forceinline__ void frag_t(const float *X, int xp, int g, int u, uint32_t (&ah)[4], uint32_t (&al)[4]) {
  split_bf16x2(X[(2 * u) * xp + g], X[(2 * u + 1) * xp + g], ah[0], al[0]);
  split_bf16x2(X[(2 * u) * xp + g + 8], X[(2 * u + 1) * xp + g + 8], ah[1], al[1]);
  split_bf16x2(X[(2 * u + 8) * xp + g], X[(2 * u + 9) * xp + g], ah[2], al[2]);
  split_bf16x2(X[(2 * u + 8) * xp + g + 8], X[(2 * u + 9) * xp + g + 8], ah[3], al[3]);
}
// A operand from an accumulator (its C fragments are A fragments), split
__device__ __forceinline__ void frag_acc(const Acc3 &c, uint32_t (&ah)[4], uint32_t (&al)[4]) {
  float v[2][4];
#pragma unroll
  for (int n = 0; n < 2; n++)
#pragma unroll
    for (int e = 0; e < 4; e++) v[n][e] = c.d[0][n][e] + (c.d[1][n][e] + c.d[2][n][e]);
  split_bf16x2(v[0][0], v[0][1], ah[0], al[0]);
  split_bf16x2(v[0][2], v[0][3], ah[1], al[1]);
  split_bf16x2(v[1][0], v[1][1], ah[2], al[2]);
  split_bf16x2(v[1][2], v[1][3], ah[3], al[3]);
}
// c = (A_ij)^T accumulated with the opposite sign: write A_ij = -c^T
__device__ __forceinline__ void store_neg_t(const Acc3 &c, float *Ao, int g, int u) {
#pragma unroll
  for (int nt = 0; nt < 2; nt++) {
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; e++) v[e] = c.d[0][nt][e] + (c.d[1][nt][e] + c.d[2][nt][e]);
    Ao[(8 * nt + 2 * u) * 68 + g] = -v[0];
    Ao[(8 * nt + 2 * u + 1) * 68 + g] = -v[1];
    Ao[(8 * nt + 2 * u) * 68 + g + 8] = -v[2];
    Ao[(8 * nt + 2 * u + 1) * 68 + g + 8] = -v[3];
  }
}
// c = X^T: write X (the same sums frag_acc would split)
__device__ __forceinline__ void store_t(const Acc3 &c, float *Ao, int g, int u) {
#pragma unroll
  for (int nt = 0; nt < 2; nt++) {
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; e++) v[e] = c.d[0][nt][e] + (c.d[1][nt][e] + c.d[2][nt][e]);
    Ao[(8 * nt + 2 * u) * 68 + g] = v[0];
    Ao[(8 * nt + 2 * u + 1) * 68 + g] = v[1];
    Ao[(8 * nt + 2 * u) * 68 + g + 8] = v[2];
    Ao[(8 * nt + 2 * u + 1) * 68 + g + 8] = v[3];
  }
}
__device__ __forceinline__ const float *nblk(const BuildTcSmem &sm, int i, int j) { return &sm.nm[16 * i][16 * j]; }
__device__ __forceinline__ float *ablk(BuildTcSmem &sm, int i, int j) { return &sm.am[16 * i][16 * j]; }

// A = (I + N)^-1 for the strictly lower 64 x 64 N in sm.nm, into the lower
// blocks of sm.am (blocks above the block diagonal are left unwritten), by
// recursive doubling over 16 x 16 blocks (i > j:  A_ij = -sum A_ia N_ak A_kj
// over j <= k < a <= i, from (I + N) A = I):
//   1. the diagonal blocks by forward substitution (one thread per column);
//   2. the lower-left block of each 32 x 32 half, A_10 and A_32:
//        A_ij = -A_ii (N_ij A_jj);
//   3. the lower-left 32 x 32 quarter in two steps of one warp per block
//      (a or i in {2, 3}, j in {0, 1}):
//        P_aj = sum_{k=j}^{1} N_ak A_kj   (into the unused block (j, a) of nm),
//        A_ij = -sum_{a=2}^{i} A_ia P_aj.
//      Each warp's chain is two block products per step instead of six
//      when every warp formed the P blocks it needs itself.
// Stages 2 and 3 run on the legacy warp MMA in transposed form (in stage 2
// each product's accumulator is the next one's A operand), operands split
// hi + lo.  Called by the 128 threads of the P group; ends with a group
// barrier.
__device__ void ut_inverse(BuildTcSmem &sm, int q) {
  if (q < 64) {
    const int b = 16 * (q >> 4), l = q & 15;
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
  tc::named_bar(BAR_P, NG);
  const int wp = q >> 5, lane = q & 31, g = lane >> 2, u = lane & 3;
  uint32_t ah[4], al[4];
  if (wp < 2) {  // A_10 (warp 0), A_32 (warp 1)
    const int i = 2 * wp + 1, j = 2 * wp;
    Acc3 pc, ac;
    acc_zero(pc);
    frag_t(ablk(sm, j, j), 68, g, u, ah, al);
    acc_mma(pc, ah, al, nblk(sm, i, j), 68, g, u);  // (N_ij A_jj)^T
    frag_acc(pc, ah, al);
    acc_zero(ac);
    acc_mma(ac, ah, al, ablk(sm, i, i), 68, g, u);  // (A_ii N_ij A_jj)^T
    store_neg_t(ac, ablk(sm, i, j), g, u);
  }
  tc::named_bar(BAR_P, NG);
  {  // P_aj = sum_{k=j}^{1} N_ak A_kj into the unused block (j, a) of nm
    const int a = 2 + (wp & 1), j = wp >> 1;
    Acc3 pc;
    acc_zero(pc);
    for (int k = j; k < 2; k++) {
      frag_t(ablk(sm, k, j), 68, g, u, ah, al);
      acc_mma(pc, ah, al, nblk(sm, a, k), 68, g, u);
    }
    store_t(pc, &sm.nm[16 * j][16 * a], g, u);
  }
  tc::named_bar(BAR_P, NG);
  {
    const int i = 2 + (wp & 1), j = wp >> 1;
    Acc3 ac;
    acc_zero(ac);
    for (int a = 2; a <= i; a++) {
      frag_t(&sm.nm[16 * j][16 * a], 68, g, u, ah, al);
      acc_mma(ac, ah, al, ablk(sm, i, a), 68, g, u);  // += (A_ia P_aj)^T
    }
    store_neg_t(ac, ablk(sm, i, j), g, u);
  }
  tc::named_bar(BAR_P, NG);
}

// Split factor tiles A diag(bG) and A diag(b) (K-major bf16 [64 t x 64 t'],
// hi and lo): thread q writes 32 consecutive t' of row q / 2.
__device__ __forceinline__ void write_factors(BuildTcSmem &sm, int q) {
  const int t = q >> 1, q0 = 32 * (q & 1);
#pragma unroll 1
  for (int h8 = 0; h8 < 4; h8++) {
    const int c0 = q0 + 8 * h8;
    uint32_t wh[4], wl[4], uh[4], ul[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      // blocks above the block diagonal of am are not written: mask t' > t
      const float2 a2 = *reinterpret_cast<const float2 *>(&sm.am[t][c0 + 2 * j]);
      const float ax = (c0 + 2 * j <= t) ? a2.x : 0.f, ay = (c0 + 2 * j + 1 <= t) ? a2.y : 0.f;
      split_bf16x2(ax * sm.bg[c0 + 2 * j], ay * sm.bg[c0 + 2 * j + 1], wh[j], wl[j]);
      split_bf16x2(ax * sm.bt[c0 + 2 * j], ay * sm.bt[c0 + 2 * j + 1], uh[j], ul[j]);
    }
    const uint32_t off = sw16(t, c0, 64);
    *reinterpret_cast<uint4 *>(sm.bwh + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
    *reinterpret_cast<uint4 *>(sm.bwl + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    *reinterpret_cast<uint4 *>(sm.buh + off) = make_uint4(uh[0], uh[1], uh[2], uh[3]);
    *reinterpret_cast<uint4 *>(sm.bul + off) = make_uint4(ul[0], ul[1], ul[2], ul[3]);
  }
}

// K and V of chunk `ch` of item `it`, the CTA's chunk g (buffers g % 3 and
// g % 2)
__device__ __forceinline__ void issue_chunk(BuildTcSmem &sm, const BuildItem &it, int ch, uint32_t g, int kh,
                                            const CUtensorMap *tk, const CUtensorMap *tv) {
  const int32_t t0 = (int32_t)(it.start + (int64_t)C * ch);
  const int bk = (int)(g % NBUF), bv = (int)(g & 1);
  tc::mbar_expect_tx(&sm.full[bk], 32768u);
  for (int s = 0; s < 2; s++) tc::tma_load_3d(sm.kin[bk] + s * 8192, tk, 64 * s, kh, t0, &sm.full[bk]);
  for (int s = 0; s < 2; s++) tc::tma_load_3d(sm.vin[bv] + s * 8192, tv, 64 * s, it.head, t0, &sm.full[bk]);
}
struct ItemCtx {
  BuildItem it;
  int kh;
  int n_ch;
  uint32_t gch0;  // index of the item's first chunk in this CTA's chunk sequence
};

// the next chunk to issue exists (moves the cursor into the next item when
// the current one is exhausted)
__device__ __forceinline__ bool iss_pending(Issuer &s) {
  if (s.w == 0 && s.ch >= s.nch[0] && s.ok[1]) {
    s.w = 1;
    s.ch = 0;
  }
  return s.ok[s.w] && s.ch < s.nch[s.w];
}
__device__ __forceinline__ void iss_issue(BuildTcSmem &sm, Issuer &s, const CUtensorMap *tk, const CUtensorMap *tv) {
  issue_chunk(sm, s.it[s.w], s.ch, s.g, s.kh[s.w], tk, tv);
  s.ch++;
  s.g++;
}
__device__ __forceinline__ void fetch_item(BuildTcSmem &sm, const BuildParams &p, int n_items, BuildItem &it, int &kh,
                                           int &nch, bool &ok) {
  const int idx = aborted(sm) ? n_items : take_item(p.plan, sm.iss.taken);
  ok = idx < n_items;
  nch = 0;
  kh = 0;
  if (ok) {
    it = p.items[idx];
    kh = (int)(((int64_t)it.head * p.h_k) / p.h_v);
    nch = (int)((it.end - it.start + C - 1) / C);
  }
}

struct MmaIds {
  uint32_t gram, wu, wu_neg, c1, c2;
};

// ---------------------------------------------------------------- P group
// Prepares chunk ch: everything that depends on the inputs alone.  q is the
// thread's index in the group (0..127).  Once-per-chunk barriers are waited
// on with the phase of the chunk they belong to (global chunk index).
__device__ void prep_chunk(BuildTcSmem &sm, const BuildParams &p, const ItemCtx &x, int ch, int q,
                           uint32_t tm, const MmaIds &id, uint32_t LIM, uint32_t (&ph_full)[NBUF], float &g_cur,
                           float &b_cur, const CUtensorMap *tk, const CUtensorMap *tv) {
  const BuildItem &it = x.it;
  const bool gdn = p.variant == HYPIC_GDN;
  const uint32_t g = x.gch0 + (uint32_t)ch;  // global chunk index
  const int bk = (int)(g % NBUF), bv = (int)(g & 1), b3 = (int)(g % 3);
  const int64_t t0 = it.start + (int64_t)C * ch;
  const int nt = (it.end - t0) < C ? (int)(it.end - t0) : C;
  const int wp = q >> 5, lane = q & 31;
  // gates of the next chunk, one chunk ahead
  float g_nxt = 0.f, b_nxt = 0.f;
  if (q < C && t0 + C + q < it.end) {
    if (gdn) g_nxt = p.g[(t0 + C + q) * p.h_v + it.head];
    b_nxt = p.beta[(t0 + C + q) * p.h_v + it.head];
  }
  // ---- inputs landed; ragged tail -> identity tokens (k = v = 0)
  if (!tc::mbar_wait(&sm.full[bk], ph_full[bk] & 1, aborted(sm) ? DRAIN_LIMIT : LIM)) fail(sm, p);
  ph_full[bk]++;
  unsigned char *kin = sm.kin[bk], *vin = sm.vin[bv];
  if (nt < C) {
    for (int e = q; e < (C - nt) * 16; e += NG) {
      const int r = nt + (e >> 4), s = (e >> 3) & 1, c16 = e & 7;
      const uint4 z = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(kin + s * 8192 + r * 128 + c16 * 16) = z;
      *reinterpret_cast<uint4 *>(vin + s * 8192 + r * 128 + c16 * 16) = z;
    }
  }
  if (q < C) {
    sm.bt[q] = b_cur;
    sm.lam[q] = g_cur;
  }
  tc::fence_proxy_async_smem();  // zeroed tail rows are MMA operands
  tc::tc_fence_before();
  tc::named_bar(BAR_P, NG);
  if (q == 0) {
    // ---- Gram K K^T (K-major view; padded rows 64..127 are ignored) once X
    // has read the previous chunk's W out of TM_WG.  That also means the U
    // MMA of chunk g - 1 is complete (X waits for it first), so V buffer
    // (g + 1) % 2 is free: the CTA's chunk g + 1 is copied in now, into K
    // buffer (g + 1) % 3 once X's chain 2 of chunk g - 2 (its last reader) is
    // complete.  That barrier's next phase is chunk g's, which needs wt_ready
    // of chunk g, arrived below: the phase waited on is its latest.  The
    // gate scan below runs on another warp meanwhile.
    if (g > 0) wait_phase(sm, p, &sm.wg_free, g - 1, LIM);
    if (iss_pending(sm.iss) && sm.iss.g == g + 1 && !aborted(sm)) {
      if (g >= 2) wait_phase(sm, p, &sm.bar_x2[(g - 2) & 1], (g - 2) >> 1, LIM);
      iss_issue(sm, sm.iss, tk, tv);
    }
    tc::tc_fence_after();
    const uint32_t kb = tc::smem_u32(kin);
#pragma unroll
    for (int ks = 0; ks < 8; ks++)
      tc::mma_ss_f16(tm + TM_WG, kdesc16(kb, 16 * ks, 64), kdesc16(kb, 16 * ks, 64), id.gram, ks > 0);
    tc::mma_commit(&sm.bar_g);
  } else if (wp == 1) {  // lam_t = sum_{j<=t} g_j (two tokens per lane)
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
    sm.dec[b3][lane] = __expf(lc - x0);
    sm.dec[b3][lane + 32] = __expf(lc - x1);
    // factors of exp(lam_t - lam_i) = exp(lam_t - lam_0) exp(lam_0 - lam_i);
    // in fp32 range when the chunk's log-gates sum above -80
    const float l0 = __shfl_sync(0xffffffffu, x0, 0);
    sm.ea[lane] = sm.bt[lane] * __expf(x0 - l0);
    sm.ea[lane + 32] = sm.bt[lane + 32] * __expf(x1 - l0);
    sm.eb[lane] = __expf(l0 - x0);
    sm.eb[lane + 32] = __expf(l0 - x1);
    if (lane == 0) {
      sm.gc[b3] = __expf(lc);
      sm.fact = (l0 - lc) <= 80.f;
    }
  }
  tc::named_bar(BAR_P, NG);  // the scan's results
  wait_phase(sm, p, &sm.bar_g, g, DRAIN_LIMIT);
  tc::tc_fence_after();
  // ---- M_ti = b_t exp(lam_t - lam_i) k_t.k_i (i < t): warps holding lanes 0..63
  if (wp < 2) {
    const int t = q;
    const bool fact = sm.fact != 0;  // uniform over the chunk
    const float lt = sm.lam[t], btt = sm.bt[t], eat = sm.ea[t];
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 32) {
      uint32_t r[32];
      float li[32];
      tc::tmem_ld32(trow(tm + TM_WG, c0), r);
#pragma unroll
      for (int j = 0; j < 32; j += 4) {  // into registers before any store
        const float4 l4 = *reinterpret_cast<const float4 *>(fact ? &sm.eb[c0 + j] : &sm.lam[c0 + j]);
        li[j] = l4.x;
        li[j + 1] = l4.y;
        li[j + 2] = l4.z;
        li[j + 3] = l4.w;
      }
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; j++)
        li[j] = (c0 + j < t) ? (fact ? eat * li[j] : btt * __expf(lt - li[j])) * __uint_as_float(r[j]) : 0.f;
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4 *>(&sm.nm[t][c0 + j]) = make_float4(li[j], li[j + 1], li[j + 2], li[j + 3]);
    }
  }
  tc::named_bar(BAR_P, NG);
  ut_inverse(sm, q);
  write_factors(sm, q);
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  tc::named_bar(BAR_P, NG);
  // ---- W^T = K^T (A diag(bG))^T, and -U^T = -V^T (A diag(b))^T straight
  // into the chain-1 accumulator once X has consumed the previous chunk's
  // chain-1 output
  if (g > 0) wait_phase(sm, p, &sm.ys_done, g - 1, LIM);
  if (q == 0 || q == 32) {
    // two issuers (lane 0 of the first two warps), one accumulator each: W
    // into TM_WG, -U into TM_Y; X waits for both commits and both arrivals
    tc::tc_fence_after();
    if (q == 0) {
      const uint32_t kb = tc::smem_u32(kin);
      const uint32_t wh = tc::smem_u32(sm.bwh), wl = tc::smem_u32(sm.bwl);
#pragma unroll
      for (int ks = 0; ks < 4; ks++) {
        tc::mma_ss_f16(tm + TM_WG, mndesc16(kb, 16 * ks), kdesc16(wh, 16 * ks, 64), id.wu, ks > 0);
        tc::mma_ss_f16(tm + TM_WG, mndesc16(kb, 16 * ks), kdesc16(wl, 16 * ks, 64), id.wu, 1u);
      }
    } else {
      const uint32_t vb = tc::smem_u32(vin);
      const uint32_t uh = tc::smem_u32(sm.buh), ul = tc::smem_u32(sm.bul);
#pragma unroll
      for (int ks = 0; ks < 4; ks++) {
        tc::mma_ss_f16(tm + TM_Y, mndesc16(vb, 16 * ks), kdesc16(uh, 16 * ks, 64), id.wu_neg, ks > 0);
        tc::mma_ss_f16(tm + TM_Y, mndesc16(vb, 16 * ks), kdesc16(ul, 16 * ks, 64), id.wu_neg, 1u);
      }
    }
    tc::mma_commit(&sm.bar_wu);
    tc::mbar_arrive(&sm.wt_ready);  // hand chunk g to X
  }
  g_cur = g_nxt;
  b_cur = b_nxt;
}

// ---------------------------------------------------------------- X group
// XR <- RN(X_h) (chain 1 reads the start-of-chunk state), X_h <- G_C X_h
// (the accumulator chain 2 adds onto), in one pass over the half.
// Recording build: `rec` (non-NULL for the S half) receives the
// start-of-chunk state, column n of S (this thread's lane) at rec[d * 128]
// (a warp's stores fill whole 128-byte lines).
template <bool REC>
__device__ __forceinline__ void stage_half(uint32_t tm, uint32_t tx, float gC, float *rec) {
#pragma unroll 1
  for (int c0 = 0; c0 < 128; c0 += 64) {
    uint32_t r[64];
    tc::tmem_ld32(trow(tm + tx, c0), *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
    tc::tmem_ld32(trow(tm + tx, c0 + 32), *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
    tc::tmem_wait_ld();
    if (REC && rec) {
#pragma unroll
      for (int e = 0; e < 64; e++) rec[(int64_t)(c0 + e) * 128] = __uint_as_float(r[e]);
    }
#pragma unroll
    for (int h = 0; h < 2; h++) {
      uint32_t xr[32];
#pragma unroll
      for (int j = 0; j < 32; j++) {
        const float v = __uint_as_float(r[32 * h + j]);
        xr[j] = tc::to_tf32_fast(v);  // X itself keeps any NaN (it is the accumulator)
        r[32 * h + j] = __float_as_uint(gC * v);
      }
      tc::tmem_st32(trow(tm + TM_XR, c0 + 32 * h), xr);
    }
    tc::tmem_st32(trow(tm + tx, c0), *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
    tc::tmem_st32(trow(tm + tx, c0 + 32), *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
  }
  tc::tmem_wait_st();
}

// chain 1 into TM_Y: Y^T (+)= XR^T W^T (issued by lane 0 of the group)
__device__ __forceinline__ void issue_chain1(BuildTcSmem &sm, uint32_t tm, const MmaIds &id, bool onto_u,
                                             uint64_t *bar) {
  tc::tc_fence_after();
  const uint32_t wb = tc::smem_u32(sm.wt);
#pragma unroll
  for (int ks = 0; ks < 16; ks++)
    tc::mma_ts_tf32(tm + TM_Y, tm + TM_XR + 8 * ks, kdesc32(wb, 8 * ks, 64), id.c1, (onto_u || ks > 0) ? 1u : 0u);
  tc::mma_commit(bar);
}

// chain 2 into the half tx: X^T += Ytilde^T K (B = the chunk's K tile, MN-major)
__device__ __forceinline__ void issue_chain2(BuildTcSmem &sm, uint32_t tm, uint32_t tx, int bk, const MmaIds &id,
                                             uint64_t *bar) {
  tc::tc_fence_after();
  const uint32_t kb = tc::smem_u32(sm.kin[bk]), yhb = tc::smem_u32(sm.yh), ylb = tc::smem_u32(sm.yl);
#pragma unroll
  for (int ks = 0; ks < 4; ks++) {
    tc::mma_ss_f16(tm + tx, kdesc16(yhb, 16 * ks, 128), mndesc16(kb, 16 * ks), id.c2, 1u);
    tc::mma_ss_f16(tm + tx, kdesc16(ylb, 16 * ks, 128), mndesc16(kb, 16 * ks), id.c2, 1u);
  }
  tc::mma_commit(bar);
}

// Ytilde = -Y diag(exp(lam_C - lam_t)), split hi + lo, as the K-major A
// tiles [128 j x 64 t] of chain 2 (the S half's Y already holds -U)
// Recording build: `rec` (non-NULL for the S half) receives
// Delta = U - W S_0 = -Y of the chunk, column n, at rec[t * 128].
template <bool REC>
__device__ __forceinline__ void split_y(BuildTcSmem &sm, uint32_t tm, int n, int b3, float *rec) {
#pragma unroll 1
  for (int c0 = 0; c0 < 64; c0 += 32) {
    uint32_t r[32];
    tc::tmem_ld32(trow(tm + TM_Y, c0), r);
    tc::tmem_wait_ld();
    if (REC && rec) {
#pragma unroll
      for (int j = 0; j < 32; j++) rec[(int64_t)(c0 + j) * 128] = -__uint_as_float(r[j]);
    }
#pragma unroll
    for (int q8 = 0; q8 < 4; q8++) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const int jj = 8 * q8 + 2 * j, t = c0 + jj;
        const float2 dd = *reinterpret_cast<const float2 *>(&sm.dec[b3][t]);
        split_bf16x2(-dd.x * __uint_as_float(r[jj]), -dd.y * __uint_as_float(r[jj + 1]), hw[j], lw[j]);
      }
      const uint32_t off = sw16(n, c0 + 8 * q8, 128);
      *reinterpret_cast<uint4 *>(sm.yh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4 *>(sm.yl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }
}

// Advances both halves of the state through chunk ch (n = thread = TMEM
// lane), the S half first: its chain 1 accumulates onto the -U^T that P put
// in TM_Y.
template <bool REC>
__device__ void chain_chunk(BuildTcSmem &sm, const BuildParams &p, const ItemCtx &x, int ch, int n, uint32_t tm,
                            const MmaIds &id, uint32_t LIM) {
  const uint32_t g = x.gch0 + (uint32_t)ch;
  const int bk = (int)(g % NBUF), b3 = (int)(g % 3);
  // recording build: this chunk's records (S half only)
  float *rec_s = nullptr, *rec_d = nullptr;
  if (REC) {
    const int64_t rc = (int64_t)(x.it.part + ch) * p.h_v + x.it.head;
    rec_s = p.rec_S + rc * 128 * 128 + n;  // S_0 [128 d][128 j], column n
    rec_d = p.rec_D + rc * 64 * 128 + n;   // Delta [64 t][128 j], column n
  }
  wait_phase(sm, p, &sm.wt_ready, g, LIM);
  // ---- W (tf32, rounded) as chain 1's B tile, once P's W / U MMAs are
  // complete (lane n holds row n of W^T; the previous chunk's chain 1 that
  // read the tile was waited on before its Ytilde)
  wait_phase(sm, p, &sm.bar_wu, g, DRAIN_LIMIT);
  tc::tc_fence_after();
#pragma unroll 1
  for (int c0 = 0; c0 < 64; c0 += 32) {
    uint32_t r[32];
    tc::tmem_ld32(trow(tm + TM_WG, c0), r);
    tc::tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; j++)
      // a NaN in W comes from an input that reaches X through K, U or the
      // gates as well
      *reinterpret_cast<uint32_t *>(sm.wt + sw32(c0 + j, n, 64)) = tc::to_tf32_fast(__uint_as_float(r[j]));
  }
  tc::fence_proxy_async_smem();
  const float gC = sm.gc[b3];
  // ---- S half (its chain 2 of the previous chunk was waited on before the
  // T half's Ytilde)
  stage_half<REC>(tm, TM_XS, gC, rec_s);
  tc::tc_fence_before();
  tc::named_bar(BAR_X, NG);
  if (n == 0) {
    tc::mbar_arrive(&sm.wg_free);  // TM_WG is free for the next chunk's Gram
    issue_chain1(sm, tm, id, true, &sm.bar_y1);
  }
  wait_phase(sm, p, &sm.bar_y1, g, DRAIN_LIMIT);
  tc::tc_fence_after();
  split_y<REC>(sm, tm, n, b3, rec_d);
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  tc::named_bar(BAR_X, NG);
  if (n == 0) issue_chain2(sm, tm, TM_XS, bk, id, &sm.bar_x1);
  // ---- T half: XR is free (chain 1 of S is complete); the T half's chain 2
  // of the previous chunk must be
  if (ch > 0) wait_phase(sm, p, &sm.bar_x2[(g - 1) & 1], (g - 1) >> 1, DRAIN_LIMIT);
  tc::tc_fence_after();
  stage_half<REC>(tm, TM_XT, gC, nullptr);
  tc::tc_fence_before();
  tc::named_bar(BAR_X, NG);
  if (n == 0) issue_chain1(sm, tm, id, false, &sm.bar_y2);
  wait_phase(sm, p, &sm.bar_y2, g, DRAIN_LIMIT);
  // the Ytilde tiles are free once the S half's chain 2 has read them
  wait_phase(sm, p, &sm.bar_x1, g, DRAIN_LIMIT);
  tc::tc_fence_after();
  split_y<REC>(sm, tm, n, b3, nullptr);
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  tc::named_bar(BAR_X, NG);
  if (n == 0) {
    tc::mbar_arrive(&sm.ys_done);  // TM_Y is free for the next chunk's -U
    issue_chain2(sm, tm, TM_XT, bk, id, &sm.bar_x2[g & 1]);
  }
}

template <bool REC>
__global__ void __launch_bounds__(NT, 1)
    build_tc_kernel(const __grid_constant__ BuildTcArgs args, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte alignment by pointer arithmetic on the shared array, so the
  // compiler keeps every access in the shared address space
  BuildTcSmem &sm = *reinterpret_cast<BuildTcSmem *>(smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  const BuildParams &p = args.p;
  const uint32_t LIM = args.wait_limit;
  const int n = threadIdx.x, warp = n >> 5;
  const bool is_p = warp >= 4;
  const int q = n - NG;  // index inside the P group

  if (n == 0) {
    for (int b = 0; b < NBUF; b++) tc::mbar_init(&sm.full[b], 1);
    tc::mbar_init(&sm.bar_g, 1);
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
    for (int b = 0; b < 2; b++) {
      tc::mbar_init(&sm.item_full[b], 1);
      tc::mbar_init(&sm.item_free[b], 1);
    }
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

  MmaIds id;
  id.gram = tc::idesc(tc::FMT_BF16, 128, 64);
  id.wu = tc::idesc(tc::FMT_BF16, 128, 64, false, false, /*a_mn=*/true, false);
  id.wu_neg = tc::idesc(tc::FMT_BF16, 128, 64, /*neg_a=*/true, false, /*a_mn=*/true, false);
  id.c1 = tc::idesc(tc::FMT_TF32, 128, 64);
  id.c2 = tc::idesc(tc::FMT_BF16, 128, 128, false, false, false, /*b_mn=*/true);
  uint32_t ph_full[NBUF] = {0, 0, 0};
  const int n_items = p.plan->n_items;

  Issuer &iss = sm.iss;
  if (is_p) {
    if (q == 0) {
      iss.w = 0;
      iss.ch = 0;
      iss.g = 0;
      iss.taken = 0;
      fetch_item(sm, p, n_items, iss.it[0], iss.kh[0], iss.nch[0], iss.ok[0]);
      iss.ok[1] = false;
      iss.nch[1] = 0;
      if (iss.ok[0]) fetch_item(sm, p, n_items, iss.it[1], iss.kh[1], iss.nch[1], iss.ok[1]);
    }
  }
  uint32_t gch = 0;  // chunks prepared by this CTA so far (P group)
  for (int k = 0;; k++) {
    if (is_p) {
      if (q == 0) {
        // item k to slot k % 2 once X has taken item k - 2 from it
        if (k >= 2) wait_phase(sm, p, &sm.item_free[k & 1], (uint32_t)(k - 2) >> 1, LIM);
        XItem xi;
        xi.slot = iss.it[0].slot;
        xi.head = iss.it[0].head;
        xi.n_ch = iss.nch[0];
        xi.valid = iss.ok[0] ? 1 : 0;
        xi.gch0 = gch;
        xi.cbase = iss.it[0].part;
        sm.xslot[k & 1] = xi;
        tc::mbar_arrive(&sm.item_full[k & 1]);
        sm.pitem.it = iss.it[0];
        sm.pitem.kh = iss.kh[0];
        sm.pitem.n_ch = iss.nch[0];
        sm.pitem.valid = iss.ok[0] ? 1 : 0;
        sm.pitem.gch0 = gch;
        // the item's first chunk, if not yet issued (only at the start, or
        // after items with an empty body).  Its buffers last held chunks
        // gch - 3 (K) and gch - 2 (V); once X has read W of chunk gch - 1,
        // X has waited for chain 2 of chunk gch - 3 and for the W / U MMAs
        // of chunk gch - 1.  The second chunk is issued by prep(gch).
        if (iss_pending(iss) && iss.g <= gch) {
          if (gch > 0) wait_phase(sm, p, &sm.wg_free, gch - 1, LIM);
          while (iss_pending(iss) && iss.g <= gch) iss_issue(sm, iss, &tmap_k, &tmap_v);
        }
      }
      tc::named_bar(BAR_P, NG);
      ItemCtx x;
      x.it = sm.pitem.it;
      x.kh = sm.pitem.kh;
      x.n_ch = sm.pitem.n_ch;
      x.gch0 = sm.pitem.gch0;
      const bool valid = sm.pitem.valid != 0;
      tc::named_bar(BAR_P, NG);
      if (!valid) break;
      float g_cur = 0.f, b_cur = 0.f;
      if (q < C && x.it.start + q < x.it.end) {
        if (p.variant == HYPIC_GDN) g_cur = p.g[(x.it.start + q) * p.h_v + x.it.head];
        b_cur = p.beta[(x.it.start + q) * p.h_v + x.it.head];
      }
      for (int ch = 0; ch < x.n_ch; ch++)
        prep_chunk(sm, p, x, ch, q, tm, id, LIM, ph_full, g_cur, b_cur, &tmap_k, &tmap_v);
      gch += (uint32_t)x.n_ch;
      if (q == 0) {  // the next item becomes current; fetch the one after it
        if (iss.w == 1) {
          iss.w = 0;
        } else {
          iss.ch = 0;
        }
        iss.it[0] = iss.it[1];
        iss.kh[0] = iss.kh[1];
        iss.nch[0] = iss.nch[1];
        iss.ok[0] = iss.ok[1];
        iss.ok[1] = false;
        iss.nch[1] = 0;
        if (iss.ok[0]) fetch_item(sm, p, n_items, iss.it[1], iss.kh[1], iss.nch[1], iss.ok[1]);
      }
    } else {
      const bool got = tc::mbar_wait(&sm.item_full[k & 1], ((uint32_t)k >> 1) & 1, aborted(sm) ? DRAIN_LIMIT : LIM);
      if (!got) fail(sm, p);
      const XItem xi = sm.xslot[k & 1];
      tc::named_bar(BAR_X, NG);
      if (n == 0) tc::mbar_arrive(&sm.item_free[k & 1]);
      if (!got || !xi.valid) break;
      ItemCtx x;
      x.it.slot = xi.slot;
      x.it.part = xi.cbase;
      x.it.head = xi.head;
      x.n_ch = xi.n_ch;
      x.gch0 = xi.gch0;
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
      for (int ch = 0; ch < x.n_ch; ch++) chain_chunk<REC>(sm, p, x, ch, n, tm, id, LIM);
      if (x.n_ch > 0) {
        const uint32_t gl = x.gch0 + (uint32_t)x.n_ch - 1;
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
      tc::tc_fence_before();
    }
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


}  // namespace

bool make_tmap_3d(CUtensorMap *map, CUtensorMapDataType dt, uint32_t esz, const void *base, int64_t n_tokens,
                  int heads, uint32_t box_x, uint32_t box_t, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)n_tokens};
  cuuint64_t strides[2] = {128 * (cuuint64_t)esz, (cuuint64_t)heads * 128 * esz};
  cuuint32_t box[3] = {box_x, 1, box_t};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, dt, 3, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_tokens(CUtensorMap *map, const void *base, int64_t n_tokens, int heads, int rows) {
  return make_tmap_3d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, n_tokens, heads, 64, (uint32_t)rows,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

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
  // the recording build (the prefill forward's first pass) also writes every
  // chunk's start state and Delta
  auto kern = p.rec_S ? build_tc_kernel<true> : build_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = n_sm < n_items ? n_sm : n_items;
  if (grid < 1) return cudaSuccess;
  BuildTcArgs a;
  a.p = p;
  a.wait_limit = wait_limit;
  a.debug_stall = debug_stall() ? 1 : 0;
  kern<<<grid, NT, smem, s>>>(a, tk, tv);
  return cudaGetLastError();
}

}  // namespace hypic
