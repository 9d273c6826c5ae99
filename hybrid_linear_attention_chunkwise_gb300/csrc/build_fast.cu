// build_fast.cu -- tensor-core fast path of the segment build for the
// transitions without an erase: RetNet-style scalar decay (gamma_h I), the
// ungated rule (I) and the GLA-type diagonal gate (Diag(a_t)), bf16 inputs,
// d_k = d_v = 128.
//
// The cached pair (HYPIC news pages, nav.aitube.vip §2.1: T_C the product of
// the segment's token transitions, S(C|0) its final state from zero) needs
// no dense T here: T_C is gamma^L, 1 or Diag(prod_t a_t), and
//     S(C|0) = sum_t (w_t . k_t) v_t^T,   w_t = prod_{j > t} a_j
// (gamma^(L-1-t) for the scalar decay, 1 when ungated) -- one GEMM over the
// body's tokens.  The body is walked backwards in chunks of 64 tokens, so
// each per-channel weight is a running suffix product of the gates (no
// overflow: every weight is <= 1; the scalar decay's weight is formed in
// closed form, once per token), and D = S^T accumulates in TMEM:
//     D[j][c] += sum_t V[t][j] (w_t[c] k_t[c])     (kind::f16, A = the V
// tile, B = the weighted K tile, both MN-major views of [token x channel]
// tiles; the weighted keys are split hi + lo in bf16, ~2^-17; ungated
// bodies use the TMA K tile as it lands).  Thread j then owns column j of
// S(C|0) and writes it with coalesced stores.
//
// Items are (segment, value head) in LPT order, pulled by an atomic ticket;
// two CTAs per SM.  All waits are bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc.cuh"

namespace hypic {

namespace {

constexpr int C = 64;    // tokens per chunk
constexpr int NT = 128;  // threads: thread c owns channel c (weights) and column c of S (epilogue)
constexpr uint32_t DRAIN_LIMIT = 1u << 22;

struct __align__(1024) FastSmem {
  unsigned char kin[2][16384];  // TMA tiles [64 t x 128 c] bf16, two 64-channel slabs
  unsigned char vin[2][16384];
  unsigned char kh[16384];      // weighted keys, hi part (same layout as the K tile)
  unsigned char kl[16384];      //   lo part
  uint64_t full[2];
  uint64_t mma_done;
  uint64_t never;
  uint32_t tmem_base;
  int item;
  int abort;
};

struct FastArgs {
  BuildParams p;
  uint32_t wait_limit;
  int debug_stall;
};

// byte offset of element (t, c) in a [64 x 128] bf16 TMA tile (128-byte
// swizzle, two 64-channel slabs of 8 KiB)
__device__ __forceinline__ uint32_t tile_off(int t, int c) {
  const uint32_t byte = (uint32_t)(c & 63) * 2u;
  return (uint32_t)((c >> 6) * 8192 + t * 128) + ((((byte >> 4) ^ (uint32_t)(t & 7)) << 4) | (byte & 15u));
}
// MN-major operand view of such a tile, K-step of 16 tokens starting at t
__device__ __forceinline__ uint64_t mn_desc(uint32_t base, int t) {
  return tc::smem_desc(base + (uint32_t)(t * 128), 8192, 1024, tc::SW_128B);
}

__device__ __forceinline__ bool aborted(FastSmem &sm) { return *(volatile int *)&sm.abort != 0; }
__device__ __forceinline__ void fail(FastSmem &sm, const BuildParams &p) {
  *(volatile int *)&sm.abort = 1;
  report(p.status, HYPIC_STATUS_TIMEOUT);
}

__global__ void __launch_bounds__(NT, 2)
    build_fast_kernel(const __grid_constant__ FastArgs args, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ unsigned char smem_raw[];
  FastSmem &sm = *reinterpret_cast<FastSmem *>(smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  const BuildParams &p = args.p;
  const uint32_t LIM = args.wait_limit;
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool diag = p.variant == HYPIC_DIAG_GATE;
  const bool scalar = p.variant == HYPIC_SCALAR_DECAY;
  const bool weighted = diag || scalar;

  if (tid == 0) {
    tc::mbar_init(&sm.full[0], 1);
    tc::mbar_init(&sm.full[1], 1);
    tc::mbar_init(&sm.mma_done, 1);
    tc::mbar_init(&sm.never, 1);
    sm.abort = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmap_k);
    tc::prefetch_tmap(&tmap_v);
  }
  if (warp == 0) {
    tc::tmem_alloc(&sm.tmem_base, 128);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tD = sm.tmem_base;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  if (args.debug_stall && !tc::mbar_wait(&sm.never, 0, LIM)) fail(sm, p);

  // D = S^T: A = V (M = 128 value channels), B = weighted K (N = 128 key
  // channels), K-steps of 16 tokens, both operands MN-major
  const uint32_t id = tc::idesc(tc::FMT_BF16, 128, 128, false, false, /*a_mn=*/true, /*b_mn=*/true);
  uint32_t ph_full[2] = {0, 0};
  uint32_t mcount = 0;  // commits to mma_done so far (uniform)
  const int n_items = p.plan->n_items;
  int taken = 0;  // items fetched by this CTA (thread 0)

  for (;;) {
    if (tid == 0) sm.item = aborted(sm) ? n_items : take_item(p.plan, taken);
    __syncthreads();
    const int idx = sm.item;
    __syncthreads();
    if (idx >= n_items) break;
    const BuildItem it = p.items[idx];
    const int h = it.head;
    const int kh = (int)(((int64_t)h * p.h_k) / p.h_v);
    const int n_ch = (int)((it.end - it.start + C - 1) / C);
    const float g_scalar = scalar ? p.g[h] : 0.f;

    // chunk r of the walk is chunk n_ch - 1 - r of the body, buffer r % 2
    auto issue = [&](int r) {
      const int ch = n_ch - 1 - r;
      const int32_t t0 = (int32_t)(it.start + (int64_t)C * ch);
      const int b = r & 1;
      tc::mbar_expect_tx(&sm.full[b], 32768u);
      for (int s = 0; s < 2; s++) tc::tma_load_3d(sm.kin[b] + s * 8192, &tmap_k, 64 * s, kh, t0, &sm.full[b]);
      for (int s = 0; s < 2; s++) tc::tma_load_3d(sm.vin[b] + s * 8192, &tmap_v, 64 * s, h, t0, &sm.full[b]);
    };
    if (tid == 0 && !aborted(sm))
      for (int r = 0; r < 2 && r < n_ch; r++) issue(r);

    float s_log = 0.f;  // per-channel gate: log of the weight of the token just before the chunk walked so far (channel tid)
    for (int r = 0; r < n_ch; r++) {
      const int ch = n_ch - 1 - r;
      const int64_t t0 = it.start + (int64_t)C * ch;
      const int nt = (it.end - t0) < C ? (int)(it.end - t0) : C;
      const int b = r & 1;
      // gates of this chunk for channel tid (per-channel gate) into registers
      float gl[C];
      if (diag) {
#pragma unroll
        for (int t = 0; t < C; t++) gl[t] = t < nt ? p.g[((t0 + t) * p.h_v + h) * 128 + tid] : 0.f;
      }
      if (!tc::mbar_wait(&sm.full[b], ph_full[b] & 1, aborted(sm) ? DRAIN_LIMIT : LIM)) fail(sm, p);
      ph_full[b]++;
      if (r > 0) {
        // the previous chunk's MMAs are done: its buffers and the weighted
        // key tiles are free; the buffer refills with chunk r + 1
        if (!tc::mbar_wait(&sm.mma_done, mcount & 1, DRAIN_LIMIT)) fail(sm, p);
        mcount++;
        tc::tc_fence_after();
        if (tid == 0 && r + 1 < n_ch && !aborted(sm)) issue(r + 1);
      }
      if (scalar) {
        // w_t = gamma^(end - 1 - t) in closed form (one exponential per
        // token, shared by its channels): thread tid forms 8 vectors of 8
        // channels, tokens t = v / 16, with 16-byte loads and stores
#pragma unroll 2
        for (int m = 0; m < 8; m++) {
          const int v = tid + NT * m, t = v >> 4, c8 = (v & 15) << 3;
          const uint32_t off = tile_off(t, c8);
          const float w = t < nt ? __expf((float)(it.end - 1 - (t0 + t)) * g_scalar) : 0.f;
          const uint4 kw = *reinterpret_cast<const uint4 *>(sm.kin[b] + off);
          const uint32_t kk[4] = {kw.x, kw.y, kw.z, kw.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int j = 0; j < 4; j++) {
            const float k0 = __uint_as_float(kk[j] << 16) * w, k1 = __uint_as_float(kk[j] & 0xFFFF0000u) * w;
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(k0, k1);
            hi[j] = *reinterpret_cast<const uint32_t *>(&h2);
            const __nv_bfloat162 l2 = __floats2bfloat162_rn(k0 - __uint_as_float(hi[j] << 16),
                                                            k1 - __uint_as_float(hi[j] & 0xFFFF0000u));
            lo[j] = *reinterpret_cast<const uint32_t *>(&l2);
          }
          *reinterpret_cast<uint4 *>(sm.kh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4 *>(sm.kl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      } else if (diag) {
        // w_t = exp(sum of the gates after t) per channel, walking the chunk
        // backwards in blocks of 16 tokens: the block's keys are loaded
        // before any of its weighted keys is stored (the loads do not wait
        // behind the stores)
        const unsigned char *kt = sm.kin[b];
#pragma unroll
        for (int t1 = C; t1 > 0; t1 -= 16) {
          float kv[16];
#pragma unroll
          for (int j = 0; j < 16; j++)
            kv[j] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(kt + tile_off(t1 - 1 - j, tid)));
#pragma unroll
          for (int j = 0; j < 16; j++) {
            const int t = t1 - 1 - j;
            float k = 0.f;
            if (t < nt) {
              k = kv[j] * __expf(s_log);
              s_log += gl[t];
            }
            const __nv_bfloat16 hi = __float2bfloat16_rn(k);
            const __nv_bfloat16 lo = __float2bfloat16_rn(k - __bfloat162float(hi));
            *reinterpret_cast<__nv_bfloat16 *>(sm.kh + tile_off(t, tid)) = hi;
            *reinterpret_cast<__nv_bfloat16 *>(sm.kl + tile_off(t, tid)) = lo;
          }
        }
      } else if (nt < C) {
        // ragged chunk, ungated: zero the key rows past the body
        for (int e = tid; e < (C - nt) * 16; e += NT) {
          const int row = nt + (e >> 4), sl = (e >> 3) & 1, c16 = e & 7;
          *reinterpret_cast<uint4 *>(sm.kin[b] + sl * 8192 + row * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc::tc_fence_after();
        if (!aborted(sm)) {
          const uint32_t vb = tc::smem_u32(sm.vin[b]);
          const uint32_t k0 = tc::smem_u32(weighted ? sm.kh : sm.kin[b]), k1 = tc::smem_u32(sm.kl);
#pragma unroll
          for (int ks = 0; ks < 4; ks++) {
            tc::mma_ss_f16(tD, mn_desc(vb, 16 * ks), mn_desc(k0, 16 * ks), id, (r > 0 || ks > 0) ? 1u : 0u);
            if (weighted) tc::mma_ss_f16(tD, mn_desc(vb, 16 * ks), mn_desc(k1, 16 * ks), id, 1u);
          }
        }
        tc::mma_commit(&sm.mma_done);
      }
    }

    // ---- epilogue: thread j holds column j of S(C|0); T_C
    const int64_t sh = (int64_t)it.slot * p.h_v + h;
    bool bad = false;
    if (n_ch > 0) {
      if (!tc::mbar_wait(&sm.mma_done, mcount & 1, DRAIN_LIMIT)) fail(sm, p);
      mcount++;
      tc::tc_fence_after();
    }
    float *S = p.S_pool + sh * 128 * 128 + tid;
#pragma unroll
    for (int c0 = 0; c0 < 128; c0 += 32) {
      uint32_t v[32];
      if (n_ch > 0) {
        tc::tmem_ld32(tD + lane_base + (uint32_t)c0, v);
        tc::tmem_wait_ld();
      } else {
#pragma unroll
        for (int j = 0; j < 32; j++) v[j] = 0u;
      }
#pragma unroll
      for (int j = 0; j < 32; j++) {
        const float x = __uint_as_float(v[j]);
        S[(int64_t)(c0 + j) * 128] = x;
        bad |= !finite_f(x);
      }
    }
    if (diag) {
      const float tv = __expf(s_log);  // prod of the body's gates, channel tid
      p.T_pool[sh * 128 + tid] = tv;
      bad |= !finite_f(tv);
    } else if (tid == 0) {
      const float tv = scalar ? (float)exp((double)(it.end - it.start) * (double)g_scalar) : 1.f;
      p.T_pool[sh] = tv;
      bad |= !finite_f(tv);
    }
    if ((p.flags & HYPIC_FLAG_CHECK_FINITE) && bad) report(p.status, HYPIC_STATUS_NONFINITE);
    tc::tc_fence_before();
    __syncthreads();  // the TMEM reads are done before the next item's MMAs
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tD, 128);
  }
}

}  // namespace

bool build_fast_supported(const BuildParams &p) {
  auto a16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  return (p.variant == HYPIC_SCALAR_DECAY || p.variant == HYPIC_UNGATED || p.variant == HYPIC_DIAG_GATE) &&
         p.in_dtype == HYPIC_IN_BF16 && p.d_k == 128 && p.d_v == 128 && a16(p.k) && a16(p.v);
}

cudaError_t launch_build_fast(const BuildParams &p, int64_t n_tokens, int n_items, int n_sm, uint32_t wait_limit,
                              cudaStream_t s) {
  CUtensorMap tk, tv;
  if (!make_tmap_tokens(&tk, p.k, n_tokens, p.h_k) || !make_tmap_tokens(&tv, p.v, n_tokens, p.h_v))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(FastSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(build_fast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int grid = 2 * n_sm;
  if (grid > n_items) grid = n_items;
  if (grid < 1) return cudaSuccess;
  FastArgs a;
  a.p = p;
  a.wait_limit = wait_limit;
  a.debug_stall = debug_stall() ? 1 : 0;
  build_fast_kernel<<<grid, NT, smem, s>>>(a, tk, tv);
  return cudaGetLastError();
}

}  // namespace hypic
