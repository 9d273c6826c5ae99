/*
 * hypic_oracle.c -- plain fp64 CPU oracle for the HYPIC linear-attention
 * state algebra.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * bench's CPU-baseline leg call it; the product path never does.  It shares no
 * code, header, table or constant with the CUDA library.
 *
 * Sources (the three news pages retelling the HYPIC paper):
 *  - "首 token 延迟降 3.25 倍！小红书联合北大、上交提出 HYPIC ..." (nav.aitube.vip),
 *    §2.1 (linear layers: the segment-cumulative transition operator T_C is
 *    the product of every token transition matrix in the segment; the true
 *    final state obeys S(C1·C2) = T(C2)·S(C1) + S(C2); the pair
 *    (T_C, S(C|0)) depends only on the segment's own tokens) and §2.2 (seam
 *    window: the first w tokens of a reused segment are not cached; at reuse
 *    the linear layer advances the running state through them one token at a
 *    time and forwards each seam token's output upward).
 *  - the same content on the xix.ai Spanish and Japanese pages, paragraph on
 *    linear layers and paragraph on full-attention seams.
 *
 * The per-token transitions are the standard forms of the family the pages
 * name (RetNet, GLA, DeltaNet, GDN, KDA), state S in R^{d_k x d_v}:
 *     S_t = T_t S_{t-1} + U_t,          o_t = S_t^T q_t  (post-update state)
 *   gdn      T_t = a_t (I - b_t k k^T)          U_t = b_t k v^T
 *   deltanet T_t = I - b_t k k^T                U_t = b_t k v^T
 *   channel  T_t = (I - b_t k k^T) Diag(a_t)    U_t = b_t k v^T
 *   scalar   T_t = gamma_h I                    U_t = k v^T
 *   ungated  T_t = I                            U_t = k v^T
 *   diag     T_t = Diag(a_t)                    U_t = k v^T
 * with a = exp(g) from fp32 log-gates.  Value head h reads key head
 * floor(h * h_k / h_v).
 *
 * Every routine is token-by-token in fp64 with no blocking or reordering
 * beyond applying T_t to a matrix X through the exact identity
 * (I - b k k^T) X = X - b k (k^T X).  OpenMP runs independent
 * (segment, head) / (layer, head) items in parallel; each item is a plain
 * sequential loop, so results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_GDN = 0, OR_DELTANET = 1, OR_CHANNEL = 2, OR_SCALAR = 3, OR_UNGATED = 4, OR_DIAG = 5 };

static int has_beta(int var) { return var == OR_GDN || var == OR_DELTANET || var == OR_CHANNEL; }

/* Per-token gate of value head h at token t: scalar variants use gs, the
 * per-channel ones the vector gv (length dk).  Returns 0 = no gate, 1 =
 * scalar, 2 = vector. */
static int token_gate(int var, const double *g, int64_t t, int h, int hv, int dk,
                      double *gs, const double **gv) {
  switch (var) {
  case OR_GDN: *gs = exp(g[t * hv + h]); return 1;
  case OR_SCALAR: *gs = exp(g[h]); return 1;
  case OR_CHANNEL:
  case OR_DIAG: *gv = g + (t * hv + h) * (int64_t)dk; return 2;
  default: return 0;
  }
}

/* X (dk x m, row-major, leading dim ld) <- T_t X, for the token described by
 * (kind, gs, gv, b, kv).  tmp holds m doubles.  The vector gate a = exp(gv)
 * is applied before the rank-1 erase, following T_t = (I - b k k^T) Diag(a). */
static void apply_T(int var, int kind, double gs, const double *gv, double b, const double *kv,
                    double *X, int dk, int m, int ld, double *tmp) {
  if (kind == 2) {
    for (int i = 0; i < dk; i++) {
      double a = exp(gv[i]);
      for (int j = 0; j < m; j++) X[i * ld + j] *= a;
    }
  }
  if (has_beta(var)) {
    for (int j = 0; j < m; j++) tmp[j] = 0.0;
    for (int i = 0; i < dk; i++)
      for (int j = 0; j < m; j++) tmp[j] += kv[i] * X[i * ld + j];
    for (int i = 0; i < dk; i++)
      for (int j = 0; j < m; j++) X[i * ld + j] -= b * kv[i] * tmp[j];
  }
  if (kind == 1) {
    for (int i = 0; i < dk; i++)
      for (int j = 0; j < m; j++) X[i * ld + j] *= gs;
  }
}

/* S (dk x dv, ld) += U_t = c k v^T with c = b (delta variants) or 1. */
static void add_U(int var, double b, const double *kv, const double *vv, double *S, int dk, int dv, int ld) {
  double c = has_beta(var) ? b : 1.0;
  for (int i = 0; i < dk; i++)
    for (int j = 0; j < dv; j++) S[i * ld + j] += c * kv[i] * vv[j];
}

/* One token step on the augmented block X = [T | S] (dk x (dk+dv)):
 * T <- T_t T, S <- T_t S + U_t.  For a state-only step pass with_T = 0 and
 * X = S (dk x dv). */
static void token_step(int var, const double *k, const double *v, const double *g, const double *beta,
                       int64_t t, int h, int hk, int hv, int dk, int dv, double *X, int with_T, double *tmp) {
  int kh = (int)(((int64_t)h * hk) / hv);
  const double *kv = k + (t * hk + kh) * (int64_t)dk;
  const double *vv = v + (t * hv + h) * (int64_t)dv;
  double gs = 1.0, b = 0.0;
  const double *gv = NULL;
  int kind = token_gate(var, g, t, h, hv, dk, &gs, &gv);
  if (has_beta(var)) b = beta[t * hv + h];
  int m = with_T ? dk + dv : dv;
  apply_T(var, kind, gs, gv, b, kv, X, dk, m, m, tmp);
  add_U(var, b, kv, vv, X + (with_T ? dk : 0), dk, dv, m);
}

/*
 * oracle_build: for every segment i and value head h, the pair
 *   T_C = T_{e-1} ... T_{s+w}   (product of the body's token transitions)
 *   S(C|0) = state after the body starting from S = 0,
 * body = tokens [seg_offsets[i] + seam_w, seg_offsets[i+1]) (the seam is not
 * cached; a body that is empty gives (I, 0)).
 * Inputs: k [N,hk,dk], v [N,hv,dv], g per variant (gdn [N,hv]; channel/diag
 * [N,hv,dk]; scalar [hv]; else NULL), beta [N,hv] or NULL.
 * Outputs: T_out [n_seg,hv,dk,dk], S_out [n_seg,hv,dk,dv].  Returns 0.
 */
int oracle_build(int var, int n_seg, const int64_t *seg_offsets, int seam_w, int hk, int hv, int dk, int dv,
                 const double *k, const double *v, const double *g, const double *beta,
                 double *T_out, double *S_out, int n_threads) {
  int64_t n_items = (int64_t)n_seg * hv;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#endif
#pragma omp parallel
  {
    int m = dk + dv;
    double *X = (double *)malloc(sizeof(double) * dk * m);
    double *tmp = (double *)malloc(sizeof(double) * m);
#pragma omp for schedule(dynamic, 1)
    for (int64_t it = 0; it < n_items; it++) {
      int i = (int)(it / hv), h = (int)(it % hv);
      memset(X, 0, sizeof(double) * dk * m);
      for (int r = 0; r < dk; r++) X[r * m + r] = 1.0;
      int64_t s = seg_offsets[i] + seam_w, e = seg_offsets[i + 1];
      for (int64_t t = s; t < e; t++) token_step(var, k, v, g, beta, t, h, hk, hv, dk, dv, X, 1, tmp);
      double *To = T_out + it * (int64_t)dk * dk, *So = S_out + it * (int64_t)dk * dv;
      for (int r = 0; r < dk; r++) {
        memcpy(To + (int64_t)r * dk, X + (int64_t)r * m, sizeof(double) * dk);
        memcpy(So + (int64_t)r * dv, X + (int64_t)r * m + dk, sizeof(double) * dv);
      }
    }
    free(X);
    free(tmp);
  }
  return 0;
}

/*
 * oracle_compose: for every layer l and value head h, S <- S_init (or 0); then
 * for each segment i in prompt order:
 *   (1) for each of the w seam tokens: S <- T_t S + U_t, o_t = S^T q_t;
 *   (2) S <- T_C S + S(C|0)  (left-multiply, then add: the composition rule).
 * Pairs arrive in prompt order: T_pairs [L,n_seg,hv,dk,dk], S_pairs
 * [L,n_seg,hv,dk,dv].  Seam token arrays are [L,n_seg,w,heads,...]; the
 * scalar-decay gate is per head [hv] (shared by all layers in this routine).
 * Outputs: S_out [L,hv,dk,dv], seam_out [L,n_seg,w,hv,dv].
 */
int oracle_compose(int var, int n_layers, int n_seg, int w, int hk, int hv, int dk, int dv,
                   const double *T_pairs, const double *S_pairs,
                   const double *sk, const double *sv, const double *sq, const double *sg, const double *sb,
                   const double *S_init, double *S_out, double *seam_out, int n_threads) {
  int64_t n_items = (int64_t)n_layers * hv;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#endif
#pragma omp parallel
  {
    double *S = (double *)malloc(sizeof(double) * dk * dv);
    double *S2 = (double *)malloc(sizeof(double) * dk * dv);
    double *tmp = (double *)malloc(sizeof(double) * dv);
#pragma omp for schedule(dynamic, 1)
    for (int64_t it = 0; it < n_items; it++) {
      int l = (int)(it / hv), h = (int)(it % hv);
      if (S_init) memcpy(S, S_init + it * (int64_t)dk * dv, sizeof(double) * dk * dv);
      else memset(S, 0, sizeof(double) * dk * dv);
      for (int i = 0; i < n_seg; i++) {
        int64_t base = ((int64_t)l * n_seg + i) * w; /* token index into [L*n_seg*w] */
        for (int t = 0; t < w; t++) {
          int64_t tt = base + t;
          /* the seam arrays are token arrays of N = L*n_seg*w tokens */
          token_step(var, sk, sv, sg, sb, tt, h, hk, hv, dk, dv, S, 0, tmp);
          int kh = (int)(((int64_t)h * hk) / hv);
          const double *qv = sq + (tt * hk + kh) * (int64_t)dk;
          double *o = seam_out + (tt * hv + h) * (int64_t)dv;
          for (int j = 0; j < dv; j++) o[j] = 0.0;
          for (int r = 0; r < dk; r++)
            for (int j = 0; j < dv; j++) o[j] += S[r * dv + j] * qv[r];
        }
        const double *Tc = T_pairs + (((int64_t)l * n_seg + i) * hv + h) * (int64_t)dk * dk;
        const double *Sc = S_pairs + (((int64_t)l * n_seg + i) * hv + h) * (int64_t)dk * dv;
        for (int r = 0; r < dk; r++)
          for (int j = 0; j < dv; j++) {
            double acc = 0.0;
            for (int c = 0; c < dk; c++) acc += Tc[r * dk + c] * S[c * dv + j];
            S2[r * dv + j] = acc + Sc[r * dv + j];
          }
        memcpy(S, S2, sizeof(double) * dk * dv);
      }
      memcpy(S_out + it * (int64_t)dk * dv, S, sizeof(double) * dk * dv);
    }
    free(S);
    free(S2);
    free(tmp);
  }
  return 0;
}

/*
 * oracle_full: the plain recurrence over every token of one layer's prompt,
 * from S_init (or 0), with outputs o_t = S_t^T q_t at the listed positions.
 * This is the full recompute that the cached pairs must reproduce.
 * Outputs: S_final [hv,dk,dv], outs [n_out,hv,dv].
 */
int oracle_full(int var, int64_t n_tokens, int hk, int hv, int dk, int dv,
                const double *k, const double *v, const double *q, const double *g, const double *beta,
                const double *S_init, const int64_t *out_pos, int64_t n_out,
                double *S_final, double *outs, int n_threads) {
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#endif
#pragma omp parallel
  {
    double *S = (double *)malloc(sizeof(double) * dk * dv);
    double *tmp = (double *)malloc(sizeof(double) * dv);
#pragma omp for schedule(dynamic, 1)
    for (int h = 0; h < hv; h++) {
      if (S_init) memcpy(S, S_init + (int64_t)h * dk * dv, sizeof(double) * dk * dv);
      else memset(S, 0, sizeof(double) * dk * dv);
      int64_t p = 0;
      int kh = (int)(((int64_t)h * hk) / hv);
      for (int64_t t = 0; t < n_tokens; t++) {
        token_step(var, k, v, g, beta, t, h, hk, hv, dk, dv, S, 0, tmp);
        while (p < n_out && out_pos[p] == t) {
          const double *qv = q + (t * hk + kh) * (int64_t)dk;
          double *o = outs + (p * hv + h) * (int64_t)dv;
          for (int j = 0; j < dv; j++) o[j] = 0.0;
          for (int r = 0; r < dk; r++)
            for (int j = 0; j < dv; j++) o[j] += S[r * dv + j] * qv[r];
          p++;
        }
      }
      memcpy(S_final + (int64_t)h * dk * dv, S, sizeof(double) * dk * dv);
    }
    free(S);
    free(tmp);
  }
  return 0;
}

/* Pair merge (T2,S2) o (T1,S1) = (T2 T1, T2 S1 + S2): the composition rule
 * applied to two adjacent spans, second span on the left. */
int oracle_merge(int n, int dk, int dv, const double *T2, const double *S2, const double *T1, const double *S1,
                 double *T_out, double *S_out) {
  for (int64_t it = 0; it < n; it++) {
    const double *a = T2 + it * dk * dk, *s2 = S2 + it * dk * dv, *b = T1 + it * dk * dk, *s1 = S1 + it * dk * dv;
    double *to = T_out + it * dk * dk, *so = S_out + it * dk * dv;
    for (int r = 0; r < dk; r++) {
      for (int c = 0; c < dk; c++) {
        double acc = 0.0;
        for (int x = 0; x < dk; x++) acc += a[r * dk + x] * b[x * dk + c];
        to[r * dk + c] = acc;
      }
      for (int c = 0; c < dv; c++) {
        double acc = 0.0;
        for (int x = 0; x < dk; x++) acc += a[r * dk + x] * s1[x * dv + c];
        so[r * dv + c] = acc + s2[r * dv + c];
      }
    }
  }
  return 0;
}
