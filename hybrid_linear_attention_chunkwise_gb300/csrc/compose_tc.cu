// compose_tc.cu -- tensor-core compose of cached pairs for the dense-transition
// variants (GDN, DeltaNet, per-channel delta) with bf16 seam tokens and
// d_k = d_v = 128: the bandwidth-bound left-multiply-add S <- T_C S + S(C|0)
// of the HYPIC news pages (nav.aitube.vip §2.1), with the seam-window advance
// and per-token outputs of §2.2, in one kernel (compose_seam_mma_kernel,
// below): one CTA of 256 threads per (layer, value head) chain, two CTAs per
// SM, the seam tokens in groups of eight on the tensor cores, the last group
// of a segment fused with the pair's T_C S product.
//
// Data movement:
//   T_C   four 16 KiB K-slabs per pair (TMA 2-D tiles, 128-byte swizzle = the
//         K-major MMA operand layout) through a ring of shared-memory slots;
//   S(C|0) bulk-copied into the slots T_C has just freed;
//   seam  k/q/v rows by bulk copies, gates and betas by plain loads, one or
//         two groups ahead.
// Each pool byte crosses HBM once: 128 KiB per (segment, head) pair.
//
// Every wait is bounded: one that runs out sets HYPIC_STATUS_TIMEOUT; the CTA
// then skips its remaining work (control flow stays uniform across threads),
// waits for the copies it issued and releases its TMEM.
#include <cstddef>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc.cuh"

namespace hypic {

namespace {

constexpr int NSLOT = 5;   // T_C K-slab ring (16 KiB each)
constexpr int SLAB = 16384;
constexpr int MAX_HV = 128;
constexpr uint32_t DRAIN_LIMIT = 1u << 22;

struct TcArgs {
  ComposeParams p;
  uint32_t wait_limit;
  int debug_stall;  // wait first on a barrier nothing signals (timeout test)
};

template <class SM>
__device__ __forceinline__ bool aborted(SM &sm) { return *(volatile int *)&sm.abort != 0; }

template <class SM>
__device__ __forceinline__ void fail(SM &sm, const ComposeParams &p) {
  *(volatile int *)&sm.abort = 1;
  report(p.status, HYPIC_STATUS_TIMEOUT);
}

__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

// eight bf16 values (one 16-byte shared-memory load) to fp32
__device__ __forceinline__ void unpack8(const __nv_bfloat16 *src, float (&out)[8]) {
  const uint4 u = *reinterpret_cast<const uint4 *>(src);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; j++) {
    out[2 * j] = __uint_as_float(w[j] << 16);
    out[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

struct Chain {
  int l, h, kh, n_seg, w, groups;
};

__device__ __forceinline__ int pair_slot(const ComposeParams &p, const Chain &c, int seg) {
  const int s = p.slot[(int64_t)c.l * p.seg_stride + seg];
  return (s < 0 || s >= p.n_slots) ? -1 : s;
}

// T_C K-slab r (pair r/4, columns 32*(r%4) .. +32) into ring slot r % NSLOT
template <class SM>
__device__ __forceinline__ void issue_slab(SM &sm, const ComposeParams &p, const Chain &c, const CUtensorMap *tmap,
                                           uint32_t r, int ring = NSLOT) {
  if (r >= 4u * (uint32_t)c.n_seg) return;
  const int seg = (int)(r / 4), j = (int)(r % 4);
  int slot = pair_slot(p, c, seg);
  if (slot < 0) slot = 0;  // keep the ring in step; the pair is skipped at use
  const int si = r % ring;
  tc::mbar_expect_tx(&sm.full[si], SLAB);
  tc::tma_load_2d(sm.slot[si], tmap, 32 * j, (int32_t)(((int64_t)slot * p.h_v + c.h) * 128), &sm.full[si]);
}

// T_C of segment seg's pair (64 KiB) into L2.  Warming S(C|0) as well, or
// warming further ahead, measured slower on the warm-prompt workload: the
// extra L2 footprint of 300 chains evicts lines before they are used.
__device__ __forceinline__ void prefetch_T(const ComposeParams &p, const Chain &c, int seg) {
  if (seg >= c.n_seg) return;
  const int slot = pair_slot(p, c, seg);
  if (slot < 0) return;
  prefetch_l2(p.T_pool + ((int64_t)slot * p.h_v + c.h) * 128 * 128, 128 * 128 * 4);
}

// ---------------------------------------------------------------------------
// The seam tokens on the tensor cores (GDN and DeltaNet; the per-channel gate
// through prep_group_channel above, with the changes described there).
//
// For a group of nt <= 8 seam tokens entered with state S0, cumulative
// log-gates lam_t = g_0 + ... + g_t (DeltaNet: 0) and c_t = b_t (v_t - xh_t),
// the token updates S_t = a_t S_{t-1} + k_t c_t^T (the GDN rule
// a (I - b k k^T) S + b k v^T written per column) unroll to
//   S_t  = e^{lam_t} S0 + sum_{i<=t} e^{lam_t - lam_i} k_i c_i^T
//   xh_t = a_t k_t^T S_{t-1} = e^{lam_t} k_t^T S0 + sum_{i<t} e^{lam_t-lam_i} (k_t.k_i) c_i
//   o_t  = q_t^T S_t         = e^{lam_t} q_t^T S0 + sum_{i<=t} e^{lam_t-lam_i} (q_t.k_i) c_i
// so one MMA gives k_t^T S0 and q_t^T S0 for the 8 tokens and all 128
// columns (D = S0^T [K;Q]^T: M = 128, N = 16, A = S0 in TMEM), and per column
// c = M (v - e^{lam} . k^T S0) with the 8 x 8 lower-triangular
// M = (I + diag(b) Gk)^{-1} diag(b), Gk the decayed key Gram.  For the last
// group of a segment the state never has to be formed: with S0 the state
// entering it,
//   T_C S_n + S(C|0) = e^{lam_last} (T_C S0 + sum_i (T_C k_i) e^{-lam_i} c_i^T) + S(C|0)
// so the same MMA round also gives T_C k_i (A = the T_C K-slabs), the T_C S0
// product starts at once from the same TMEM operand, and the rank-8 seam term
// is accumulated onto it by one more MMA (K = 8) from two 128 x 8 tiles.
// Earlier groups of a long seam window, a group whose decay underflows and a
// skipped pair update the exact state (kept in S_out) instead.  Everything
// that depends on the seam tokens only (the [K;Q] operand tile, the decayed
// Grams, M) is prepared by warps 5..7 while warps 0..3 run the previous
// group's recurrence; warp 4 issues the T_C S0 product and the seam copies.
//
// Issue and data movement.  One tcgen05.mma takes tens of cycles to issue,
// so the 32 small products of a fused group (S0^T [K;Q]^T and T_C [K;Q]^T,
// K = 128 in steps of 8) are issued by lane 0 of warps 4..7, one K-slab each,
// into separate partial accumulators that the readers sum.  Once the T_C S0
// product is complete, the pair's S(C|0) (64 KiB, contiguous in the pool)
// is bulk-copied into the four slots its T_C K-slabs have just freed and the
// epilogue reads it from shared memory; the slots take the next pair's
// K-slabs at the top of the next segment.  Only T_C is warmed in L2, one
// segment ahead.
// ---------------------------------------------------------------------------
constexpr int GW = 8;             // seam tokens per group
constexpr int NT2 = 256;          // threads per CTA: two per state column (rows 0..63, 64..127)
constexpr int ISSUER_WARP = 4;    // lane 0 issues the MMAs; the warp issues the seam copies
constexpr int PREP_WARP0 = 5;     // warps 5..7 prepare the next seam group
constexpr int NPREP = 96;
constexpr int BAR_PREP = 1;       // named barrier of the preparing warps
constexpr int BAR_CORR = 2;       // warps 0..4: the seam term tile is written
constexpr float AL_MIN = 1e-30f;  // smallest e^{lam_last} of a fused group

struct SeamRaw {
  __nv_bfloat16 k[GW][128];
  __nv_bfloat16 q[GW][128];
  __nv_bfloat16 v[GW][128];
};

// constants of one seam group (double-buffered by group parity)
struct GroupConst {
  float gk[GW][GW];  // e^{lam_t - lam_i} (k_t.k_i), i < t
  float gq[GW][GW];  // e^{lam_t - lam_i} (q_t.k_i), i <= t
  float mm[GW][GW];  // (I + diag(beta) gk)^{-1} diag(beta)
  float ea[GW];      // e^{lam_t}
  float eb[GW];      // e^{lam_last - lam_i}
  float beta[GW];
  float glog[GW];
  float alast;       // e^{lam_last}
  float pad[3];
};

struct __align__(1024) SeamMmaSmem {
  unsigned char slot[NSLOT][SLAB];  // T_C K-slab ring (swizzled TMA tiles)
  float bt[4][16][32];              // [K;Q] operand: tf32, K-major, 128-byte swizzle, 4 K-slabs
  float tk[128][GW];                // (T_C k_i)[r]: tf32, K-major, 32-byte swizzle
  float cp[128][GW];                // e^{-lam_i} c_i[n]: tf32, K-major, 32-byte swizzle
  SeamRaw raw[2];                   // seam k / q / v rows of a group (bulk copies)
  GroupConst gc[2];
  uint64_t full[NSLOT];
  uint64_t raw_full[2];
  uint64_t mma_done;
  uint64_t t_done;     // the T_C S0 product of a pair is complete (its slabs are free)
  uint64_t sc_full;    // the pair's S(C|0) has landed in its four slots
  uint64_t seam_done;  // fused group: the seam products are in D (four issuing threads)
  uint64_t tk_done;    // fused group: T_C [K;Q]^T is in D (four issuing threads)
  uint64_t d_read;     // fused group: every thread has read its seam columns of D
  uint64_t never;
  uint32_t tmem_base;
  int abort;
  int stop;
};
static_assert(offsetof(SeamMmaSmem, bt) % 1024 == 0, "B tile must sit on a swizzle atom");
static_assert(offsetof(SeamMmaSmem, tk) % 1024 == 0 && offsetof(SeamMmaSmem, cp) % 1024 == 0,
              "32-byte swizzled tiles must sit on a swizzle atom");

// a 32-byte row (8 tf32) of a K-major tile with 32-byte swizzle: the two
// 16-byte halves trade places in rows whose index has bit 2 set
__device__ __forceinline__ void store_row_sw32(float (*tile)[GW], int row, const float (&v)[GW]) {
  const int sw = (row >> 2) & 1;
  float4 *dst = reinterpret_cast<float4 *>(&tile[row][0]);
  dst[sw] = make_float4(__uint_as_float(tc::to_tf32(v[0])), __uint_as_float(tc::to_tf32(v[1])),
                        __uint_as_float(tc::to_tf32(v[2])), __uint_as_float(tc::to_tf32(v[3])));
  dst[sw ^ 1] = make_float4(__uint_as_float(tc::to_tf32(v[4])), __uint_as_float(tc::to_tf32(v[5])),
                            __uint_as_float(tc::to_tf32(v[6])), __uint_as_float(tc::to_tf32(v[7])));
}

struct SeamGroup {
  int64_t tok0;  // first seam token of the group in [L, n_seg, w] order
  int nt;        // real tokens in the group
};

__device__ __forceinline__ SeamGroup seam_group(const ComposeParams &p, const Chain &c, int gq) {
  const int seg = gq / c.groups, gi = gq % c.groups;
  SeamGroup g;
  g.tok0 = ((int64_t)c.l * p.seg_stride + seg) * c.w + gi * GW;
  g.nt = min(GW, c.w - gi * GW);
  return g;
}

// register select of lam[u] for a run-time u (keeps lam[] in registers)
__device__ __forceinline__ float pick(const float (&lam)[GW], int u) {
  float r = 0.f;
#pragma unroll
  for (int j = 0; j < GW; j++) r = (j == u) ? lam[j] : r;
  return r;
}

// Gram of the group on the legacy warp MMA (one warp, 8 x m16n8k16 bf16,
// exact products, fp32 sums): D[m][i] = A[m] . k_i with A = [k_0..k_7;
// q_0..q_7]; lane (g = lane/4, u = lane%4) receives D[g][2u], D[g][2u+1],
// D[g+8][2u], D[g+8][2u+1].
__device__ __forceinline__ void gram_mma(const SeamRaw &r, float (&dd)[4]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, u = lane & 3;
  dd[0] = dd[1] = dd[2] = dd[3] = 0.f;
  const uint32_t *kg = reinterpret_cast<const uint32_t *>(r.k[g]);
  const uint32_t *qg = reinterpret_cast<const uint32_t *>(r.q[g]);
#pragma unroll
  for (int kc = 0; kc < 8; kc++) {
    const int w0 = 8 * kc + u, w1 = 8 * kc + 4 + u;  // 32-bit words: channels 16kc+2u.., 16kc+8+2u..
    const uint32_t a0 = kg[w0], a1 = qg[w0], a2 = kg[w1], a3 = qg[w1];
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(dd[0]), "+f"(dd[1]), "+f"(dd[2]), "+f"(dd[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(a0), "r"(a2));
  }
}

// M = (I + diag(beta) Gk)^{-1} diag(beta), column j, by forward substitution
// (Gk strictly lower triangular: the decayed key Gram of the group)
__device__ __forceinline__ void solve_m(GroupConst &G, int j) {
  float m[GW];
#pragma unroll
  for (int t = 0; t < GW; t++) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < t; i++) s = fmaf(G.gk[t][i], (i >= j) ? m[i] : 0.f, s);
    m[t] = t < j ? 0.f : (t == j ? G.beta[t] : -G.beta[t] * s);
    G.mm[t][j] = m[t];
  }
}

// State-independent preparation of group gq by the NPREP threads of warps
// PREP_WARP0.. (its raw buffer has landed).  Threads ptid < GW pass beta and
// the log-gate of the group's token ptid (loaded one group ahead; zero past
// nt).  The raw buffer stays in use until the group's recurrence has read its
// v rows; the results become visible to the other warps at their next
// CTA-wide barrier.
__device__ __forceinline__ void prep_group(SeamMmaSmem &sm, const ComposeParams &p, const Chain &c, int gq,
                                           float b_n, float g_n) {
  const int ptid = threadIdx.x - 32 * PREP_WARP0;
  const SeamGroup sg = seam_group(p, c, gq);
  const int nt = sg.nt;
  const SeamRaw &r = sm.raw[gq & 1];
  GroupConst &G = sm.gc[gq & 1];
  if (ptid < GW) {
    G.beta[ptid] = b_n;
    G.glog[ptid] = g_n;
  }
  tc::named_bar(BAR_PREP, NPREP);
  float lam[GW];
  float acc = 0.f;
#pragma unroll
  for (int t = 0; t < GW; t++) {
    acc += G.glog[t];  // zero past nt
    lam[t] = acc;
  }
  const float lam_last = pick(lam, nt - 1);

  // [K;Q] operand tile: task -> row task/16 (k_0..k_7, q_0..q_7), 8 channels
  for (int task = ptid; task < 256; task += NPREP) {
    const int row = task >> 4, kb = (task & 15) * 8;
    float f[8];
    if ((row & 7) < nt) {
      unpack8((row < 8 ? r.k[row] : r.q[row - 8]) + kb, f);
    } else {
#pragma unroll
      for (int j = 0; j < 8; j++) f[j] = 0.f;
    }
    // bf16 values are exact in tf32; 128-byte swizzle: 16-byte chunk ^ (row % 8)
    unsigned char *slab = reinterpret_cast<unsigned char *>(&sm.bt[kb >> 5][0][0]);
#pragma unroll
    for (int q4 = 0; q4 < 2; q4++) {
      const int chunk = ((kb & 31) >> 2) + q4;
      float4 *dst = reinterpret_cast<float4 *>(slab + row * 128 + ((chunk ^ (row & 7)) << 4));
      *dst = make_float4(f[4 * q4], f[4 * q4 + 1], f[4 * q4 + 2], f[4 * q4 + 3]);
    }
  }
  // decayed Grams; rows and columns past nt (stale raw rows) are masked out
  if (ptid < 32) {
    float dd[4];
    gram_mma(r, dd);
    const int t = ptid >> 2;
#pragma unroll
    for (int j = 0; j < 2; j++) {
      const int i = 2 * (ptid & 3) + j;
      const bool in = t < nt && i < nt;
      const float e = __expf(pick(lam, t) - pick(lam, i));
      G.gk[t][i] = (in && i < t) ? dd[j] * e : 0.f;
      G.gq[t][i] = (in && i <= t) ? dd[2 + j] * e : 0.f;
    }
  } else if (ptid < 32 + GW) {
    const int t = ptid - 32;
    const float li = pick(lam, t);
    G.ea[t] = t < nt ? __expf(li) : 0.f;
    G.eb[t] = t < nt ? __expf(lam_last - li) : 0.f;
  } else if (ptid == 32 + GW) {
    G.alast = __expf(lam_last);
  }
  tc::named_bar(BAR_PREP, NPREP);
  if (ptid < GW) solve_m(G, ptid);
  tc::fence_proxy_async_smem();  // the operand tile is read by the tensor cores
}

// Per-channel gate tiles in the fifth slot (the ring of this variant has
// four): the T_C k-hat operand (16 rows, K-major, 128-byte swizzle; rows
// 8..15 zero), k-hat [128][GW] and E_last [128] fp32 for the register path,
// and reduction scratch.
struct ChTiles {
  float *ktile;   // 8 KiB
  float *khat;    // [128][GW]
  float *elast;   // [128]
  float *red;     // [3 warps][64] Gram partials, then [3] minima
};
__device__ __forceinline__ ChTiles ch_tiles(SeamMmaSmem &sm) {
  float *base = reinterpret_cast<float *>(sm.slot[NSLOT - 1]);
  return ChTiles{base, base + 2048, base + 2048 + 128 * GW, base + 2048 + 128 * GW + 128};
}

// Per-channel gate: the group constants of gq, by the NPREP preparing
// threads (beta of token ptid passed in by threads ptid < GW).  With lam_t
// the per-channel cumulative log-gate over the group and E_t = e^{lam_t},
// the per-token update S_t = Diag(a_t) S_{t-1} + k_t c_t^T (c_t = b_t (v_t -
// x_t), x_t = (a_t . k_t)^T S_{t-1}) unrolls to
//   x_t = (E_t . k_t)^T S0 + sum_{i<t} [sum_ch k_t k_i e^{lam_t - lam_i}] c_i
//   o_t = (E_t . q_t)^T S0 + sum_{i<=t} [sum_ch q_t k_i e^{lam_t - lam_i}] c_i
//   S_n = E_last . S0 + sum_i (e^{lam_last - lam_i} . k_i) c_i^T  (rows scaled)
// A group is fused with the pair when e^{lam_last} >= e^{-80} on every
// channel (and the seam window is one group): TMEM A then holds RN(E_last .
// S0) (the epilogue before scales it), so the operand rows are
// e^{lam_t - lam_last} . k_t and . q_t (<= e^{80}), and
//   T_C S_n = T_C (E_last . S0) + sum_i (T_C k-hat_i) c_i^T,
// k-hat_i = e^{lam_last - lam_i} . k_i, one more operand tile.  Otherwise the
// rows are E_t . k_t and E_t . q_t and the register path updates the exact
// state with k-hat and E_last.  The Grams take a per-channel weight: for a
// fused group the two operand tiles already carry it (one warp multiplies
// them, gram_tiles_tf32), otherwise it is formed per (t, i) pair and summed
// over the channels on the CUDA cores.  The gates gl are loaded by the caller
// (load_gates_channel).  Flags for the kernel: alast = 1 (fused) or 0, ea =
// 1, eb = 1.
// per-channel log-gates of group gq for the channels of preparing thread
// ptid (ptid and ptid + NPREP), zero past the group and past the prompt;
// issued ahead of prep_group_channel so that their latency overlaps other work
__device__ __forceinline__ void load_gates_channel(const ComposeParams &p, const Chain &c, int gq, int total_groups,
                                                   float (&gl)[2][GW]) {
  const int ptid = threadIdx.x - 32 * PREP_WARP0;
  const bool any = gq < total_groups;
  const SeamGroup sg = seam_group(p, c, any ? gq : 0);
#pragma unroll
  for (int u = 0; u < 2; u++) {
    const int ch = ptid + NPREP * u;
#pragma unroll
    for (int t = 0; t < GW; t++)
      gl[u][t] = any && ch < 128 && t < sg.nt ? p.seam_g[((sg.tok0 + t) * p.h_v + c.h) * 128 + ch] : 0.f;
  }
}

// Decayed Grams of a fused group from its two operand tiles, on the legacy
// warp MMA (one warp, 16 x m16n8k8 tf32): row t of the [K;Q] tile holds
// e^{lam_t - lam_last} . k_t (rows 8..15: . q_t) and row i of the T_C k-hat
// tile e^{lam_last - lam_i} . k_i, so their channel sums are the decayed
// products of the unrolled recurrence, at the tf32 precision of the other
// operands of the group.  Lane (g = lane/4, u = lane%4) receives D[g][2u],
// D[g][2u+1], D[g+8][2u], D[g+8][2u+1].
__device__ __forceinline__ void gram_tiles_tf32(const float *bt, const float *kt, float (&dd)[4]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, u = lane & 3;
  const uint32_t *A = reinterpret_cast<const uint32_t *>(bt);
  const uint32_t *B = reinterpret_cast<const uint32_t *>(kt);
  dd[0] = dd[1] = dd[2] = dd[3] = 0.f;
#pragma unroll
  for (int s = 0; s < 16; s++) {
    // channels 8s + u and 8s + u + 4: slab s/4, 16-byte chunks 2(s%4) and
    // 2(s%4) + 1 (swizzled by the row), word u
    const int slab = (s >> 2) * 512, c0 = 2 * (s & 3);
    const int w0 = ((c0 ^ g) << 2) + u, w1 = (((c0 + 1) ^ g) << 2) + u;
    const uint32_t a0 = A[slab + g * 32 + w0], a1 = A[slab + (g + 8) * 32 + w0];
    const uint32_t a2 = A[slab + g * 32 + w1], a3 = A[slab + (g + 8) * 32 + w1];
    const uint32_t b0 = B[slab + g * 32 + w0], b1 = B[slab + g * 32 + w1];
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(dd[0]), "+f"(dd[1]), "+f"(dd[2]), "+f"(dd[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ void prep_group_channel(SeamMmaSmem &sm, const ComposeParams &p, const Chain &c, int gq,
                                                   float b_n, const float (&gl)[2][GW]) {
  const int ptid = threadIdx.x - 32 * PREP_WARP0;
  const SeamGroup sg = seam_group(p, c, gq);
  const int nt = sg.nt;
  const SeamRaw &r = sm.raw[gq & 1];
  GroupConst &G = sm.gc[gq & 1];
  const ChTiles T = ch_tiles(sm);
  const int wp = ptid >> 5, lane = ptid & 31;
  if (ptid < GW) {
    G.beta[ptid] = b_n;
    G.ea[ptid] = ptid < nt ? 1.f : 0.f;  // the decay is inside the operand rows
    G.eb[ptid] = ptid < nt ? 1.f : 0.f;
  }
  // pass 1: this thread's channels (ptid and, for ptid < 32, ptid + 96)
  float lam[2][GW], kt[2][GW], qt[2][GW];
  float mn = 0.f;
#pragma unroll
  for (int u = 0; u < 2; u++) {
    const int ch = ptid + NPREP * u;
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t < GW; t++) {
      const bool in = ch < 128 && t < nt;
      acc += gl[u][t];  // zero past nt
      lam[u][t] = acc;
      kt[u][t] = in ? __bfloat162float(r.k[t][ch]) : 0.f;
      qt[u][t] = in ? __bfloat162float(r.q[t][ch]) : 0.f;
    }
    if (ch < 128) mn = fminf(mn, pick(lam[u], nt - 1));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  if (lane == 0) T.red[192 + wp] = mn;
  tc::named_bar(BAR_PREP, NPREP);
  // fused: a one-group seam window, a valid pair (a skipped pair runs the
  // register path), and no channel decaying below e^{-80} over the group
  const bool fuse = c.groups == 1 && pair_slot(p, c, gq / c.groups) >= 0 &&
                    fminf(fminf(T.red[192], T.red[193]), T.red[194]) >= -80.f;
  if (ptid == 0) G.alast = fuse ? 1.f : 0.f;
  if (fuse) {
    // pass 2, fused: every channel decays by at least e^{-80} over the
    // group, so the decay factors split as e^{lam_t - lam_i} = E_t R_i with
    // E_t = e^{lam_t} <= 1 and R_i = e^{-lam_i} <= e^80: 16 exponentials
    // per channel, and the two operand tiles carry every decay the Grams need
#pragma unroll
    for (int u = 0; u < 2; u++) {
      const int ch = ptid + NPREP * u;
      if (ch >= 128) break;
      const float ll = pick(lam[u], nt - 1);
      unsigned char *slab = reinterpret_cast<unsigned char *>(&sm.bt[ch >> 5][0][0]);
      unsigned char *kslab = reinterpret_cast<unsigned char *>(T.ktile) + 2048 * (ch >> 5);
      const int chunk = (ch & 31) >> 2, within = (ch & 3) * 4;
      const float El = __expf(ll), Rl = __expf(-ll);
#pragma unroll
      for (int t = 0; t < GW; t++) {
        const float e = __expf(lam[u][t]) * Rl;  // operand rows e^{lam_t - lam_last}
        *reinterpret_cast<uint32_t *>(slab + t * 128 + ((chunk ^ t) << 4) + within) = tc::to_tf32(e * kt[u][t]);
        *reinterpret_cast<uint32_t *>(slab + (GW + t) * 128 + ((chunk ^ t) << 4) + within) =
            tc::to_tf32(e * qt[u][t]);
        const float kh = (El * __expf(-lam[u][t])) * kt[u][t];  // k-hat_t
        *reinterpret_cast<uint32_t *>(kslab + t * 128 + ((chunk ^ t) << 4) + within) = tc::to_tf32(kh);
      }
      T.elast[ch] = El;
    }
    tc::named_bar(BAR_PREP, NPREP);  // both tiles are complete
    if (wp == 0) {
      float dd[4];
      gram_tiles_tf32(&sm.bt[0][0][0], T.ktile, dd);
      const int t = lane >> 2;
#pragma unroll
      for (int j = 0; j < 2; j++) {
        const int i = 2 * (lane & 3) + j;
        const bool in = t < nt && i < nt;
        G.gk[t][i] = (in && i < t) ? dd[j] : 0.f;
        G.gq[t][i] = (in && i <= t) ? dd[2 + j] : 0.f;
      }
      __syncwarp();
      if (lane < GW) solve_m(G, lane);
    }
  } else {
    // pass 2, a channel decays below e^{-80} over the group: every factor
    // formed directly (bounded by 1), k-hat kept for the register path, and
    // the Grams summed over the channels on the CUDA cores (2 channels per
    // thread, then a warp tree and the three warps, in a fixed order)
#pragma unroll
    for (int u = 0; u < 2; u++) {
      const int ch = ptid + NPREP * u;
      if (ch >= 128) break;
      const float ll = pick(lam[u], nt - 1);
      unsigned char *slab = reinterpret_cast<unsigned char *>(&sm.bt[ch >> 5][0][0]);
      unsigned char *kslab = reinterpret_cast<unsigned char *>(T.ktile) + 2048 * (ch >> 5);
      const int chunk = (ch & 31) >> 2, within = (ch & 3) * 4;
#pragma unroll
      for (int t = 0; t < GW; t++) {
        const float e = __expf(lam[u][t]);
        *reinterpret_cast<uint32_t *>(slab + t * 128 + ((chunk ^ t) << 4) + within) = tc::to_tf32(e * kt[u][t]);
        *reinterpret_cast<uint32_t *>(slab + (GW + t) * 128 + ((chunk ^ t) << 4) + within) =
            tc::to_tf32(e * qt[u][t]);
        const float kh = __expf(ll - lam[u][t]) * kt[u][t];
        *reinterpret_cast<uint32_t *>(kslab + t * 128 + ((chunk ^ t) << 4) + within) = tc::to_tf32(kh);
        T.khat[ch * GW + t] = kh;
      }
      T.elast[ch] = __expf(ll);
    }
    // the 64 Gram partials (gk: t(t-1)/2 + i, i < t; gq: 28 + t(t+1)/2 + i,
    // i <= t) in four rounds of 16, each summed over the warp by a
    // reduce-scatter: at the level with lane offset o a lane keeps the half
    // of its values selected by (lane & o) and adds its partner's copy of
    // that half; after the levels 16, 8, 4, 2 and a last exchange with lane
    // offset 1, lane l holds the warp sum of partial (l / 2) % 16 of the round
#pragma unroll
    for (int rd = 0; rd < 4; rd++) {
      float part[16];
#pragma unroll
      for (int j = 0; j < 16; j++) part[j] = 0.f;
#pragma unroll
      for (int u = 0; u < 2; u++) {
        if (ptid + NPREP * u >= 128) break;
#pragma unroll
        for (int t = 0; t < GW; t++) {
#pragma unroll
          for (int i = 0; i <= t; i++) {
            const int jk = t * (t - 1) / 2 + i - 16 * rd, jq = 28 + t * (t + 1) / 2 + i - 16 * rd;
            const bool ink = i < t && jk >= 0 && jk < 16, inq = jq >= 0 && jq < 16;
            if (!ink && !inq) continue;
            const float w = __expf(lam[u][t] - lam[u][i]);
            if (ink) part[jk] = fmaf(kt[u][t] * kt[u][i], w, part[jk]);
            if (inq) part[jq] = fmaf(qt[u][t] * kt[u][i], w, part[jq]);
          }
        }
      }
#pragma unroll
      for (int o = 16, n = 8; o > 1; o >>= 1, n >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < n; j++) {
          const float keep = up ? part[n + j] : part[j];
          const float send = up ? part[j] : part[n + j];
          part[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      part[0] += __shfl_xor_sync(0xffffffffu, part[0], 1);
      if ((lane & 1) == 0) T.red[wp * 64 + 16 * rd + ((lane >> 1) & 15)] = part[0];
    }
    tc::named_bar(BAR_PREP, NPREP);
    if (ptid < 64) {
      const float v = (T.red[ptid] + T.red[64 + ptid]) + T.red[128 + ptid];
      if (ptid < 28) {
        const int j = ptid;
        int t = 1;
        while (t * (t + 1) / 2 <= j) t++;  // t(t-1)/2 <= j < t(t+1)/2
        G.gk[t][j - t * (t - 1) / 2] = v;
      } else {
        const int j = ptid - 28;
        int t = 0;
        while ((t + 1) * (t + 2) / 2 <= j) t++;  // t(t+1)/2 <= j < (t+1)(t+2)/2
        G.gq[t][j - t * (t + 1) / 2] = v;
      }
    }
    tc::named_bar(BAR_PREP, NPREP);
    if (ptid < GW) solve_m(G, ptid);
  }
  tc::fence_proxy_async_smem();  // the operand tiles are read by the tensor cores
}

// bulk copies of group gq's k / q / v rows, one per lane of the calling warp
// (all 32 lanes call); its beta and scalar gate rows (all heads, contiguous)
// and, for the per-channel gate, this head's gate rows are warmed in L2 for
// the plain loads of the preparing warps
template <int VAR>
__device__ __forceinline__ void issue_raw_warp(SeamMmaSmem &sm, const ComposeParams &p, const Chain &c, int gq) {
  constexpr bool GDN = VAR == HYPIC_GDN;
  const int lane = threadIdx.x & 31;
  const SeamGroup sg = seam_group(p, c, gq);
  const int b = gq & 1;
  SeamRaw &r = sm.raw[b];
  if (lane == 0) tc::mbar_expect_tx(&sm.raw_full[b], (uint32_t)sg.nt * 3 * 256);
  __syncwarp();
  if (lane < 3 * sg.nt) {
    const int t = lane / 3, kind = lane % 3;
    const int64_t tok = sg.tok0 + t;
    const __nv_bfloat16 *src =
        kind == 0 ? static_cast<const __nv_bfloat16 *>(p.seam_k) + (tok * p.h_k + c.kh) * 128
        : kind == 1 ? static_cast<const __nv_bfloat16 *>(p.seam_q) + (tok * p.h_k + c.kh) * 128
                    : static_cast<const __nv_bfloat16 *>(p.seam_v) + (tok * p.h_v + c.h) * 128;
    __nv_bfloat16 *dst = kind == 0 ? r.k[t] : kind == 1 ? r.q[t] : r.v[t];
    tc::bulk_load(dst, src, 256, &sm.raw_full[b]);
  } else if (lane == 31) {
    const uint32_t gbytes = (uint32_t)(sg.nt * p.h_v * 4);
    prefetch_l2(p.seam_beta + sg.tok0 * p.h_v, gbytes);
    if (GDN) prefetch_l2(p.seam_g + sg.tok0 * p.h_v, gbytes);
  }
  // lanes 24 .. 24 + nt - 1 (never copy lanes: 3 nt <= 24): one token's
  // 512-byte gate row each
  if (VAR == HYPIC_CHANNEL_DELTA && lane >= 24 && lane - 24 < sg.nt)
    prefetch_l2(p.seam_g + ((sg.tok0 + (lane - 24)) * p.h_v + c.h) * 128, 512);
}

// VAR: HYPIC_GDN, HYPIC_DELTANET or HYPIC_CHANNEL_DELTA
template <int VAR>
__global__ void __launch_bounds__(NT2, 2)
    compose_seam_mma_kernel(const __grid_constant__ TcArgs args, const __grid_constant__ CUtensorMap tmap_T) {
  constexpr bool GDN = VAR == HYPIC_GDN;
  constexpr bool CH = VAR == HYPIC_CHANNEL_DELTA;
  // the per-channel gate streams T_C through four slots; the fifth holds its
  // group tiles (the T_C k-hat operand, k-hat and E_last for the register
  // path, reduction scratch)
  constexpr int RING = CH ? 4 : NSLOT;
  extern __shared__ unsigned char smem_raw[];
  SeamMmaSmem &sm = *reinterpret_cast<SeamMmaSmem *>(smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  const ComposeParams &p = args.p;
  const uint32_t LIM = args.wait_limit;
  const bool trans = (p.flags & HYPIC_FLAG_TRANSITION_ONLY) != 0;  // U_t and S(C|0) count as zero
  const int tid = threadIdx.x;
  const int n = tid & 127;   // column of S
  const int hf = tid >> 7;   // rows 64*hf .. 64*hf+63 of that column
  const int warp = tid / 32;
  const bool preper = warp >= PREP_WARP0;
  Chain c;
  c.l = blockIdx.x / p.h_v;
  c.h = blockIdx.x % p.h_v;
  c.kh = (int)(((int64_t)c.h * p.h_k) / p.h_v);
  c.n_seg = p.n_seg;
  c.w = p.seam_w;
  c.groups = (c.w + GW - 1) / GW;
  const int total_groups = c.n_seg * c.groups;
  const uint32_t total_slabs = 4u * (uint32_t)c.n_seg;
  const bool has_seam = c.groups > 0 && c.n_seg > 0;  // no segment: no seam group to wait for

  if (tid == 0) {
    for (int i = 0; i < NSLOT; i++) tc::mbar_init(&sm.full[i], 1);
    tc::mbar_init(&sm.raw_full[0], 1);
    tc::mbar_init(&sm.raw_full[1], 1);
    tc::mbar_init(&sm.mma_done, 1);
    tc::mbar_init(&sm.t_done, 1);
    tc::mbar_init(&sm.sc_full, 1);
    tc::mbar_init(&sm.seam_done, 4);
    tc::mbar_init(&sm.tk_done, 4);
    tc::mbar_init(&sm.d_read, NT2);
    tc::mbar_init(&sm.never, 1);
    sm.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&sm.tmem_base, 256);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  // warps w and w + 4 share the TMEM lane quadrant w % 4 (lanes = columns)
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t tD = sm.tmem_base, tA = sm.tmem_base + 128;
  const uint32_t tDh = tD + lane_base + 64 * hf, tAh = tA + lane_base + 64 * hf;  // this thread's rows
  const bool issuer = tid == 32 * ISSUER_WARP;
  const bool slab_issuer = warp >= ISSUER_WARP && (tid & 31) == 0;  // lane 0 of warps 4..7

  uint32_t issued = 0;  // T_C slabs issued (thread 0)
  int raw_issued = min(2, total_groups);  // seam groups issued (uniform)
  if (tid == 0) {
    tc::prefetch_tmap(&tmap_T);
    for (; issued < (uint32_t)RING && issued < total_slabs; issued++) issue_slab(sm, p, c, &tmap_T, issued, RING);
    for (int s = 0; s < 2; s++) prefetch_T(p, c, s);
  }
  if (warp == ISSUER_WARP) {
    for (int g = 0; g < raw_issued; g++) issue_raw_warp<VAR>(sm, p, c, g);
  }

  if (args.debug_stall && !tc::mbar_wait(&sm.never, 0, LIM)) fail(sm, p);

  // The exact fp32 state lives in global memory (S_init, then S_out: this
  // thread's 64 rows of column n) only where a register-path group or the
  // end needs it; the MMAs read RN(S) from TMEM A.
  const int64_t state = (int64_t)blockIdx.x * 128 * 128 + (int64_t)(64 * hf) * 128 + n;
  const float *exact = p.S_init ? p.S_init + state : nullptr;  // NULL: zero
  float *const out = p.S_out + state;
  bool bad = false;
  const uint32_t id_T = tc::idesc(tc::FMT_TF32, 128, 128);
  const uint32_t id_s = tc::idesc(tc::FMT_TF32, 128, 16);
  uint32_t mcount = 0;  // commits to mma_done so far (uniform)
  uint32_t nfused = 0;  // fused groups so far (uniform): phase of seam_done / tk_done / d_read
  uint32_t npair = 0;   // pairs applied so far (uniform): phase of t_done / sc_full
  bool refill_pending = false;  // thread 0: the last pair's slots await the next slabs
  const int ptid = tid - 32 * PREP_WARP0;
  float pb = 0.f, pg = 0.f;  // preparing threads ptid < GW: beta / log-gate of token ptid of the next group
  float gl[2][GW];           // per-channel gate: the preparing thread's gates of group gl_for
  int gl_for = -1;

  auto load_bg = [&](int gq) {
    pb = 0.f;
    pg = 0.f;
    if (ptid >= 0 && ptid < GW && gq < total_groups) {
      const SeamGroup sg = seam_group(p, c, gq);
      if (ptid < sg.nt) {
        pb = p.seam_beta[(sg.tok0 + ptid) * p.h_v + c.h];
        if (GDN) pg = p.seam_g[(sg.tok0 + ptid) * p.h_v + c.h];
      }
    }
  };
  // preparing warps: raw group gq has landed, prepare it and start the loads
  // of the next group's beta / gates
  auto prepare = [&](int gq) {
    const bool ok = !aborted(sm) && tc::mbar_wait(&sm.raw_full[gq & 1], (gq >> 1) & 1, LIM);
    if (!ok) fail(sm, p);
    if (CH) {
      if (gl_for != gq) load_gates_channel(p, c, gq, total_groups, gl);
      prep_group_channel(sm, p, c, gq, pb, gl);
    } else
      prep_group(sm, p, c, gq, pb, pg);
    load_bg(gq + 1);
  };
  // after a barrier that follows group gq's recurrence: its raw buffer is
  // free, refill it with group gq + 2 (uniform call; the issuer warp copies)
  auto release_raw = [&](int gq) {
    if (gq + 2 < total_groups) {
      if (warp == ISSUER_WARP && !aborted(sm)) issue_raw_warp<VAR>(sm, p, c, gq + 2);
      raw_issued = gq + 3;
    }
  };
  auto wait_mma = [&]() {
    if (!tc::mbar_wait(&sm.mma_done, mcount & 1, DRAIN_LIMIT)) fail(sm, p);
    mcount++;
    tc::tc_fence_after();
  };
  // S^T [K;Q]^T (issuer) as four independent partial products, one per
  // K-slab a of 32 channels, in D cols 32a .. 32a + 15 (short dependent
  // accumulation chains; read_seam sums them)
  auto issue_seam_mma = [&]() {
    const uint32_t base = tc::smem_u32(&sm.bt[0][0][0]);
#pragma unroll
    for (int k4 = 0; k4 < 4; k4++) {
#pragma unroll
      for (int a = 0; a < 4; a++) {
        const uint64_t bd = tc::smem_desc(base + 2048 * a + 32 * k4, 16, 1024, tc::SW_128B);
        tc::mma_ts_tf32(tD + 32 * a, tA + 32 * a + 8 * k4, bd, id_s, k4 != 0);
      }
    }
  };
  // k_t^T S0 (d[0..7]) and q_t^T S0 (d[8..15]) for column n (warp-collective)
  auto read_seam = [&](uint32_t (&d)[16]) {
    uint32_t e[16];
    tc::tmem_ld16(tD + lane_base, d);
#pragma unroll
    for (int a = 1; a < 4; a++) {
      tc::tmem_ld16(tD + lane_base + 32 * a, e);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; j++) d[j] = __float_as_uint(__uint_as_float(d[j]) + __uint_as_float(e[j]));
    }
  };
  // D = S^T T_C^T from TMEM A and the four K-slabs at ring position q (issuer)
  auto issue_T_mma = [&](uint32_t q) {
    for (int sl = 0; sl < 4; sl++) {
      const uint32_t base = tc::smem_u32(sm.slot[(q + sl) % RING]);
#pragma unroll
      for (int kk = 0; kk < 4; kk++) {
        const uint64_t bd = tc::smem_desc(base + 32 * kk, 16, 1024, tc::SW_128B);
        tc::mma_ts_tf32(tD, tA + 32 * sl + 8 * kk, bd, id_T, (sl | kk) != 0);
      }
    }
  };
  // issuer, once the T_C S0 product of the pair at ring position q (slot
  // `slot` of the pool) is issued: when it completes, the pair's S(C|0)
  // (64 KiB, contiguous) replaces T_C in the four slots, 16 KiB (32 rows)
  // per slot
  auto load_sc = [&](uint32_t q, int slot, uint32_t ph) {
    tc::mma_commit(&sm.t_done);
    if (!tc::mbar_wait(&sm.t_done, ph, DRAIN_LIMIT)) fail(sm, p);
    tc::mbar_expect_tx(&sm.sc_full, 4 * SLAB);
    // transition-only: S(C|0) counts as zero; the copy (kept so the pipeline
    // is unchanged) reads the pair's T_C instead of S_pool, which may be NULL
    const float *src = (trans ? p.T_pool : p.S_pool) + ((int64_t)slot * p.h_v + c.h) * 128 * 128;
    for (int j = 0; j < 4; j++) tc::bulk_load(sm.slot[(q + j) % RING], src + j * 32 * 128, SLAB, &sm.sc_full);
  };
  // the four K-slabs at ring position q have landed (one thread)
  auto wait_slabs = [&](uint32_t q) {
    for (int sl = 0; sl < 4; sl++) {
      const uint32_t r = q + sl;
      if (!tc::mbar_wait(&sm.full[r % RING], (r / RING) & 1, LIM)) {
        fail(sm, p);
        return false;
      }
    }
    return true;
  };
  // c_t of every token of group gq for column n (c = M u, u = v - e^{lam} x0),
  // and (first half only) the outputs o_t
  auto seam_recurrence = [&](const uint32_t (&d)[16], int gq, float (&cc)[GW]) {
    const SeamGroup sg = seam_group(p, c, gq);
    const SeamRaw &raw = sm.raw[gq & 1];
    const GroupConst &G = sm.gc[gq & 1];
    float u[GW];
#pragma unroll
    for (int t = 0; t < GW; t++)
      u[t] = t < sg.nt ? (trans ? 0.f : __bfloat162float(raw.v[t][n])) - G.ea[t] * __uint_as_float(d[t]) : 0.f;
#pragma unroll
    for (int t = 0; t < GW; t++) {
      float x = 0.f;
#pragma unroll
      for (int i = 0; i <= t; i++) x = fmaf(G.mm[t][i], u[i], x);
      cc[t] = x;
    }
    if (hf == 0) {
#pragma unroll
      for (int t = 0; t < GW; t++) {
        if (t < sg.nt) {
          float o = G.ea[t] * __uint_as_float(d[8 + t]);
#pragma unroll
          for (int i = 0; i <= t; i++) o = fmaf(G.gq[t][i], cc[i], o);
          if (!trans) p.seam_out[((sg.tok0 + t) * p.h_v + c.h) * 128 + n] = o;
          bad |= !finite_f(o);
        }
      }
    }
  };

  if (CH) {
    // rows 8..15 of the T_C k-hat operand stay zero
    float *kt = ch_tiles(sm).ktile;
    for (int e = tid; e < 4 * 256; e += NT2) kt[(e >> 8) * 512 + 256 + (e & 255)] = 0.f;
  }
  if (preper) {
    load_bg(0);
    if (has_seam) prepare(0);
  }
  // RN(S_init) -> TMEM A (per-channel gate, first group fused: RN(E_last .
  // S_init))
  bool scale0 = false;
  if (CH) {
    __syncthreads();  // the first group's constants and tiles
    scale0 = has_seam && c.n_seg > 0 && pair_slot(p, c, 0) >= 0 && sm.gc[0].alast >= AL_MIN;
  }
#pragma unroll
  for (int b = 0; b < 4; b++) {
    uint32_t r[16];
#pragma unroll
    for (int j = 0; j < 16; j++) {
      const float x = exact ? exact[(int64_t)(16 * b + j) * 128] : 0.f;
      r[j] = tc::to_tf32(CH && scale0 ? x * ch_tiles(sm).elast[64 * hf + 16 * b + j] : x);
    }
    tc::tmem_st16(tAh + 16 * b, r);
  }
  tc::tmem_wait_st();
  tc::tc_fence_before();
  int slot_next = c.n_seg > 0 ? pair_slot(p, c, 0) : 0;

  // invariant at the top of a segment: TMEM A holds RN(S), the first seam
  // group is prepared, and the exact S is at `exact` (NULL: zero) whenever
  // this segment runs a register-path group
  for (int seg = 0; seg < c.n_seg; seg++) {
    // uniform stop decision (sm.stop is read by all before thread 0 passes
    // the next barrier)
    if (tid == 0) sm.stop = *(volatile int *)&sm.abort;
    __syncthreads();
    if (*(volatile int *)&sm.stop != 0) break;

    if (tid == 0 && refill_pending) {
      // the last pair's slots (T_C, then S(C|0)) are free: refill them, and
      // warm L2 with the next segment's T_C (S(C|0) streams from HBM by its
      // bulk copies)
      refill_pending = false;
      if (!aborted(sm)) {
        for (int sl = 0; sl < 4 && issued < total_slabs; sl++, issued++) issue_slab(sm, p, c, &tmap_T, issued, RING);
        prefetch_T(p, c, seg + 1);
      }
    }
    const int slot = slot_next;  // uniform
    const bool last = seg + 1 == c.n_seg;
    slot_next = last ? 0 : pair_slot(p, c, seg + 1);
    const bool pair_ok = slot >= 0;
    if (!pair_ok && tid == 0) report(p.status, HYPIC_STATUS_BAD_SLOT);
    const uint32_t q = 4u * (uint32_t)seg;

    // ---- seam groups on the exact state: all but a fused last group.
    // S <- e^{lam_last} S + sum_i e^{lam_last - lam_i} k_i c_i^T (k_i from
    // the operand tile); exact S to S_out, RN(S) to TMEM A.
    bool fused = false;
    for (int gi = 0; gi < c.groups; gi++) {
      const int gq = seg * c.groups + gi;
      if (gi > 0) {
        if (preper) prepare(gq);
        __syncthreads();
      }
      if (gi == c.groups - 1 && pair_ok && sm.gc[gq & 1].alast >= AL_MIN) {
        fused = true;
        break;
      }
      if (issuer) {
        tc::tc_fence_after();
        if (!aborted(sm)) issue_seam_mma();
        tc::mma_commit(&sm.mma_done);
      }
      wait_mma();
      uint32_t d[16];
      read_seam(d);
      tc::tmem_wait_ld();
      if (!aborted(sm)) {
        float cc[GW];
        seam_recurrence(d, gq, cc);
        const GroupConst &G = sm.gc[gq & 1];
        if (CH) {
          // row r: S <- E_last[r] S + sum_i k-hat_i[r] c_i (k-hat and E_last
          // from the tk / cp tiles)
          const float *kh = ch_tiles(sm).khat + 64 * hf * GW;
          const float *el = ch_tiles(sm).elast + 64 * hf;
#pragma unroll 1
          for (int r0 = 0; r0 < 64; r0 += 16) {
            float ex[16];  // 16 independent loads in flight
#pragma unroll
            for (int j = 0; j < 16; j++) ex[j] = exact ? exact[(int64_t)(r0 + j) * 128] : 0.f;
#pragma unroll
            for (int j = 0; j < 16; j++) {
              const int rr = r0 + j;
              const float4 k0 = *reinterpret_cast<const float4 *>(kh + rr * GW);
              const float4 k1 = *reinterpret_cast<const float4 *>(kh + rr * GW + 4);
              float x = el[rr] * ex[j];
              x = fmaf(k0.x, cc[0], x);
              x = fmaf(k0.y, cc[1], x);
              x = fmaf(k0.z, cc[2], x);
              x = fmaf(k0.w, cc[3], x);
              x = fmaf(k1.x, cc[4], x);
              x = fmaf(k1.y, cc[5], x);
              x = fmaf(k1.z, cc[6], x);
              x = fmaf(k1.w, cc[7], x);
              out[(int64_t)rr * 128] = x;
              bad |= !finite_f(x);
              ex[j] = x;
            }
            uint32_t rn[16];
#pragma unroll
            for (int j = 0; j < 16; j++) rn[j] = tc::to_tf32(ex[j]);
            tc::tmem_st16(tAh + r0, rn);
          }
        } else {
#pragma unroll
          for (int i = 0; i < GW; i++) cc[i] *= G.eb[i];
          const float al = G.alast;
          const float *bt = &sm.bt[0][0][0] + 1024 * hf;  // K-slabs 2*hf, 2*hf+1 hold this thread's rows
#pragma unroll 1
          for (int r0 = 0; r0 < 64; r0 += 16) {
            float ex[16];  // 16 independent loads in flight
#pragma unroll
            for (int j = 0; j < 16; j++) ex[j] = exact ? exact[(int64_t)(r0 + j) * 128] : 0.f;
#pragma unroll
            for (int j = 0; j < 16; j++) {
              const int rr = r0 + j;
              float x = al * ex[j];
              const float *row = bt + (rr >> 5) * 512 + (rr & 3);
              const int chunk = (rr & 31) >> 2;
#pragma unroll
              for (int i = 0; i < GW; i++) x = fmaf(row[i * 32 + ((chunk ^ i) << 2)], cc[i], x);
              out[(int64_t)rr * 128] = x;
              bad |= !finite_f(x);
              ex[j] = x;
            }
            uint32_t rn[16];
#pragma unroll
            for (int j = 0; j < 16; j++) rn[j] = tc::to_tf32(ex[j]);
            tc::tmem_st16(tAh + r0, rn);
          }
        }
        exact = out;  // RN(S) went to TMEM A row block by row block above
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
      __syncthreads();
      release_raw(gq);
    }
    const int gq_next = (seg + 1) * c.groups;  // the group that opens the next segment

    if (!pair_ok) {
      // a bad slot skips the pair; its slabs (loaded from slot 0) still pass
      // through the ring
      if (tid == 0 && !aborted(sm) && wait_slabs(q)) {
        for (int sl = 0; sl < 4 && issued < total_slabs; sl++, issued++) issue_slab(sm, p, c, &tmap_T, issued, RING);
        prefetch_T(p, c, seg + 2);
      }
      if (preper && !last && has_seam) prepare(gq_next);
      if (CH && !last && has_seam) {
        // the epilogue that scales TMEM A is skipped: if the next group is
        // fused, A <- RN(E_last . S) from the exact state the register path
        // left in S_out
        __syncthreads();
        if (sm.gc[gq_next & 1].alast >= AL_MIN && !aborted(sm)) {
          const float *el = ch_tiles(sm).elast + 64 * hf;
#pragma unroll
          for (int b = 0; b < 4; b++) {
            uint32_t r[16];
#pragma unroll
            for (int j = 0; j < 16; j++) r[j] = tc::to_tf32(out[(int64_t)(16 * b + j) * 128] * el[16 * b + j]);
            tc::tmem_st16(tAh + 16 * b, r);
          }
          tc::tmem_wait_st();
        }
      }
      tc::tc_fence_before();
      continue;
    }

    float al = 1.f;
    if (fused) {
      // ---- last seam group, fused with the pair.  With S0 the state entering
      // it (RN in TMEM A), D = T_C S0 + sum_i (T_C k_i) e^{-lam_i} c_i^T and
      // the segment ends at e^{lam_last} D + S(C|0).
      const int gq = seg * c.groups + c.groups - 1;
      al = sm.gc[gq & 1].alast;
      const uint32_t fph = nfused & 1;
      nfused++;
      if (CH && preper && !last) {
        // the gates of the group that opens the next segment, in flight
        // while these warps issue and read the products below
        load_gates_channel(p, c, gq_next, total_groups, gl);
        gl_for = gq_next;
      }
      if (slab_issuer) {
        // lane 0 of warps 4..7, one K-slab a each (the issue of one MMA takes
        // tens of cycles, so four threads issue the 32 small products in a
        // quarter of the time): the seam partial product a, then, once T_C's
        // K-slab a has landed, (T_C [K;Q]^T)'s partial product a
        const int a = warp - ISSUER_WARP;
        tc::tc_fence_after();
        if (!aborted(sm)) {
          const uint32_t bbase = tc::smem_u32(&sm.bt[0][0][0]);
#pragma unroll
          for (int k4 = 0; k4 < 4; k4++) {
            const uint64_t bd = tc::smem_desc(bbase + 2048 * a + 32 * k4, 16, 1024, tc::SW_128B);
            tc::mma_ts_tf32(tD + 32 * a, tA + 32 * a + 8 * k4, bd, id_s, k4 != 0);
          }
        }
        tc::mma_commit(&sm.seam_done);
        const uint32_t r = q + a;
        if (!aborted(sm)) {
          if (!tc::mbar_wait(&sm.full[r % RING], (r / RING) & 1, LIM)) {
            fail(sm, p);
          } else {
            // D cols 32 a + 16 .. 32 a + 31: lane r holds partial (T_C k_i)[r]
            const uint32_t abase = tc::smem_u32(sm.slot[r % RING]);
            const uint32_t bbase = (CH ? tc::smem_u32(ch_tiles(sm).ktile) : tc::smem_u32(&sm.bt[0][0][0])) + 2048 * a;
#pragma unroll
            for (int kk = 0; kk < 4; kk++) {
              const uint64_t ad = tc::smem_desc(abase + 32 * kk, 16, 1024, tc::SW_128B);
              const uint64_t bd = tc::smem_desc(bbase + 32 * kk, 16, 1024, tc::SW_128B);
              tc::mma_ss_tf32(tD + 32 * a + 16, ad, bd, id_s, kk != 0);
            }
          }
        }
        tc::mma_commit(&sm.tk_done);
      }
      __syncwarp();
      // warps 0..3 read the seam products as soon as they are in; warps 4..7
      // the T_C k_i, into the seam term's B tile; the product may overwrite D
      // once every thread has arrived at d_read
      uint32_t d[16];
      if (hf == 0) {
        if (!tc::mbar_wait(&sm.seam_done, fph, DRAIN_LIMIT)) fail(sm, p);
        tc::tc_fence_after();
        read_seam(d);
        tc::tmem_wait_ld();
      } else {
        if (!tc::mbar_wait(&sm.tk_done, fph, DRAIN_LIMIT)) fail(sm, p);
        tc::tc_fence_after();
        uint32_t e[8], f[8];
        tc::tmem_ld8(tD + lane_base + 16, e);
#pragma unroll
        for (int a = 1; a < 4; a++) {
          tc::tmem_ld8(tD + lane_base + 32 * a + 16, f);
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 8; j++) e[j] = __float_as_uint(__uint_as_float(e[j]) + __uint_as_float(f[j]));
        }
        tc::tmem_wait_ld();
        float tkr[GW];
#pragma unroll
        for (int i = 0; i < GW; i++) tkr[i] = __uint_as_float(e[i]);
        store_row_sw32(sm.tk, n, tkr);
        tc::fence_proxy_async_smem();
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&sm.d_read);
      if (hf == 0) {
        // warps 0..3, while the product runs: the group's recurrence and
        // outputs, and the seam term tile
        float cc[GW];
        if (!aborted(sm)) {
          seam_recurrence(d, gq, cc);
          const GroupConst &G = sm.gc[gq & 1];
          const float inv_al = 1.f / al;  // one division, not one per token
#pragma unroll
          for (int i = 0; i < GW; i++) cc[i] *= G.eb[i] * inv_al;  // e^{-lam_i} c_i
        } else {
#pragma unroll
          for (int i = 0; i < GW; i++) cc[i] = 0.f;
        }
        store_row_sw32(sm.cp, n, cc);
        tc::fence_proxy_async_smem();
        tc::named_bar(BAR_CORR, 160);
      } else if (warp == ISSUER_WARP) {
        if (issuer) {
          if (!tc::mbar_wait(&sm.d_read, fph, DRAIN_LIMIT)) fail(sm, p);
          tc::tc_fence_after();
          if (!aborted(sm) && wait_slabs(q)) issue_T_mma(q);
          load_sc(q, slot, npair & 1);
        }
        tc::named_bar(BAR_CORR, 160);
        if (issuer) {
          if (!aborted(sm)) {
            const uint64_t ad = tc::smem_desc(tc::smem_u32(&sm.cp[0][0]), 16, 256, tc::SW_32B);
            const uint64_t bd = tc::smem_desc(tc::smem_u32(&sm.tk[0][0]), 16, 256, tc::SW_32B);
            tc::mma_ss_tf32(tD, ad, bd, id_T, 1);
          }
          tc::mma_commit(&sm.mma_done);
        }
        __syncwarp();
      } else if (!last) {
        // warps 5..7: the group that opens the next segment
        prepare(gq_next);
      }
      release_raw(gq);
    } else {
      if (issuer) {
        tc::tc_fence_after();
        if (!aborted(sm) && wait_slabs(q)) issue_T_mma(q);
        tc::mma_commit(&sm.mma_done);
        load_sc(q, slot, npair & 1);
      }
      if (preper && has_seam && !last) prepare(gq_next);
    }

    // ---- S <- al D + S(C|0) for this thread's 64 rows, S(C|0) from the
    // pair's slots (rows 32 j .. 32 j + 31 in slot q + j); RN(S) back to
    // TMEM A, the exact S to S_out where needed
    // the next segment's first group is prepared (and visible) past here
    if (has_seam) __syncthreads();
    // the exact state is needed after this segment if it is the last one or
    // if the next one runs a register-path group
    const bool keep = last || slot_next < 0 || c.groups > 1 || (has_seam && sm.gc[gq_next & 1].alast < AL_MIN);
    const bool scale_next = CH && !keep && has_seam;  // the next segment's group is fused
    const float *el_next = CH ? ch_tiles(sm).elast + 64 * hf : nullptr;
    wait_mma();
    // (the copies are issued on every applied pair, aborted or not, and always land)
    if (!tc::mbar_wait(&sm.sc_full, npair & 1, DRAIN_LIMIT)) fail(sm, p);
    npair++;
    if (tid == 0) refill_pending = true;  // at the top of the next segment, after every read of the slots
    const bool use = !aborted(sm);
    if (use) {
      const float *sc0 = reinterpret_cast<const float *>(sm.slot[(q + 2 * hf) % RING]) + n;
      const float *sc1 = reinterpret_cast<const float *>(sm.slot[(q + 2 * hf + 1) % RING]) + n;
      // nf turns NaN once any x is not finite (x * 0 is NaN exactly then):
      // the fast rounding may lose a NaN, so a warp that holds one (rare)
      // forms its rows again with the guarded rounding; reported on every
      // segment, where the non-finite value appears
      float nfa[8];  // eight short chains (none on the critical path)
#pragma unroll
      for (int i = 0; i < 8; i++) nfa[i] = 0.f;
#pragma unroll
      for (int b = 0; b < 4; b++) {
        uint32_t r[16];
        tc::tmem_ld16(tDh + 16 * b, r);
        float sc[16];
#pragma unroll
        for (int j = 0; j < 16; j++) sc[j] = (b < 2 ? sc0 : sc1)[(16 * (b & 1) + j) * 128];
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; j++) {
          const float x = fmaf(al, __uint_as_float(r[j]), trans ? 0.f : sc[j]);
          if (keep) out[(int64_t)(16 * b + j) * 128] = x;
          nfa[j & 7] = fmaf(x, 0.f, nfa[j & 7]);
          // per-channel gate, next group fused: TMEM A holds RN(E_last . S)
          r[j] = tc::to_tf32_fast(CH && scale_next ? x * el_next[16 * b + j] : x);
        }
        tc::tmem_st16(tAh + 16 * b, r);
      }
      const float nf = ((nfa[0] + nfa[1]) + (nfa[2] + nfa[3])) + ((nfa[4] + nfa[5]) + (nfa[6] + nfa[7]));
      if (__any_sync(0xffffffffu, nf != nf)) {  // warp-uniform: the TMEM accesses are .sync.aligned
        bad |= nf != nf;
        tc::tmem_wait_st();
#pragma unroll 1
        for (int b = 0; b < 4; b++) {
          uint32_t r[16];
          tc::tmem_ld16(tDh + 16 * b, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; j++) {
            const float sc = (b < 2 ? sc0 : sc1)[(16 * (b & 1) + j) * 128];
            const float x = fmaf(al, __uint_as_float(r[j]), trans ? 0.f : sc);
            r[j] = tc::to_tf32(CH && scale_next ? x * el_next[16 * b + j] : x);
          }
          tc::tmem_st16(tAh + 16 * b, r);
        }
      }
      if (keep) exact = out;
    }
    tc::tmem_wait_st();
    tc::tc_fence_before();  // TMEM reads and writes done before the next MMA
  }

  // no segment at all: the state passes through
  if (c.n_seg == 0) {
#pragma unroll 8
    for (int i = 0; i < 64; i++) out[(int64_t)i * 128] = exact ? exact[(int64_t)i * 128] : 0.f;
  }
  if ((p.flags & HYPIC_FLAG_CHECK_FINITE) && bad) report(p.status, HYPIC_STATUS_NONFINITE);
  // drain: every copy issued lands before the CTA releases its smem
  if (tid == 0) {
    const uint32_t first = issued > (uint32_t)RING ? issued - RING : 0;
    for (uint32_t r = first; r < issued; r++) tc::mbar_wait(&sm.full[r % RING], (r / RING) & 1, DRAIN_LIMIT);
    for (int r = raw_issued > 2 ? raw_issued - 2 : 0; r < raw_issued; r++)
      tc::mbar_wait(&sm.raw_full[r & 1], (r >> 1) & 1, DRAIN_LIMIT);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(sm.tmem_base, 256);
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

// 2-D fp32 view [rows, 128] with 32-column x box_rows tiles and 128-byte
// swizzle (one K-slab of a K-major tf32 MMA operand per tile).
bool make_tmap_f32_rows(CUtensorMap *map, const float *base, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {128, rows};
  cuuint64_t strides[1] = {128 * sizeof(float)};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool compose_tc_supported(const ComposeParams &p) {
  const bool dense = p.variant == HYPIC_GDN || p.variant == HYPIC_DELTANET || p.variant == HYPIC_CHANNEL_DELTA;
  auto a16 = [](const void *x) { return x == nullptr || (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  return dense && p.in_dtype == HYPIC_IN_BF16 && p.d_k == 128 && p.d_v == 128 && p.h_v <= MAX_HV &&
         (p.h_v % 4) == 0 && a16(p.T_pool) && a16(p.S_pool) && a16(p.seam_k) && a16(p.seam_q) && a16(p.seam_v) &&
         a16(p.seam_g) && a16(p.seam_beta);
}

cudaError_t launch_compose_tc(const ComposeParams &p, uint32_t wait_limit, cudaStream_t s) {
  CUtensorMap tmap;
  if (!make_tmap_f32_rows(&tmap, p.T_pool, (uint64_t)p.n_slots * p.h_v * 128, 128)) return cudaErrorInvalidValue;
  // seam tokens on the tensor cores for every dense variant
  const size_t smem = sizeof(SeamMmaSmem) + 1024;
  auto kern = p.variant == HYPIC_GDN        ? compose_seam_mma_kernel<HYPIC_GDN>
              : p.variant == HYPIC_DELTANET ? compose_seam_mma_kernel<HYPIC_DELTANET>
                                            : compose_seam_mma_kernel<HYPIC_CHANNEL_DELTA>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = p.n_layers * p.h_v;
  if (grid < 1) return cudaSuccess;
  TcArgs a;
  a.p = p;
  a.wait_limit = wait_limit;
  a.debug_stall = debug_stall() ? 1 : 0;
  kern<<<grid, NT2, smem, s>>>(a, tmap);
  return cudaGetLastError();
}

}  // namespace hypic
