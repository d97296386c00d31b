/*
 * gdn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, FP64 CPU oracle for the gated delta rule ("GDN") and its
 * boundary-state algebra.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library; the product path never does.  It
 * shares no code, header or constant with the CUDA library.
 *
 * What it follows (page titles as cited throughout this file):
 *   [AG]  "Attention Gym -- Linear Attention", section "Gated Delta Rule":
 *         per token, with a natural-log scalar gate g and write gate beta,
 *             decayed  = exp(g) * S
 *             residual = beta * (v - decayed @ k)
 *             S        = decayed + outer(residual, k)
 *             out      = scale * S @ q
 *         The query reads the UPDATED state.  State axis order [N, H, V, K].
 *   [AG-CP] same page, section "Context Parallelism": every token step is
 *         affine in the V-major state, so a token range maps an entry state to
 *         S_out = S_in @ A + B; the cuDNN paragraph there builds B by running
 *         the state pass from a zero entry state and A by running it from an
 *         identity entry state with the value term disabled.  Entry states of
 *         consecutive ranges come from a prefix (exclusive) scan of the maps.
 *   [SF]  "StateFlow: Sequence Pipeline Parallelism ...", section 3.1,
 *         Eq. 4-7: the output state of a chunk is the input state of the next
 *         (forward), and the input-state gradient of chunk i+1 is the
 *         output-state gradient of chunk i (backward).
 *
 * The backward is plain reverse-mode differentiation of the per-token rule
 * above (the pages state its structure, [SF] Eq. 6-7, not its formulas).
 *
 * Layouts (row-major, contiguous):
 *   q, k  [B, T, H, K]      v, out [B, T, H, V]      g, beta [B, T, H]
 *   state [N, H, V, K]      cu_seqlens int32 [N+1] (then B == 1) or NULL
 * With cu_seqlens == NULL, N == B and sequence n is batch row n.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Index helpers                                                        */
/* ------------------------------------------------------------------ */

/* Token rows [bos, eos) of sequence n, as flattened (b*T + t) rows. */
static int seq_rows(int n, int B, int T, const int32_t *cu, int64_t *bos,
                    int64_t *eos) {
  if (cu) {
    if (B != 1) return -1;
    *bos = cu[n];
    *eos = cu[n + 1];
  } else {
    *bos = (int64_t)n * T;
    *eos = (int64_t)(n + 1) * T;
  }
  if (*bos < 0 || *eos < *bos || *eos > (int64_t)B * T) return -1;
  return 0;
}

/* ------------------------------------------------------------------ */
/* One token of the recurrence, [AG] "Gated Delta Rule".               */
/* S is [V,K].  Optionally records the decayed state and the residual   */
/* (the backward needs both).                                           */
/* ------------------------------------------------------------------ */
static void token_step(int K, int V, double *S, const double *kv, const double *vv,
                       double g, double beta, double *decayed_out,
                       double *residual_out) {
  const double a = exp(g);
  for (int i = 0; i < V * K; ++i) S[i] *= a;            /* decayed = exp(g) S */
  if (decayed_out) memcpy(decayed_out, S, sizeof(double) * (size_t)V * K);
  for (int r = 0; r < V; ++r) {
    double dot = 0.0;                                    /* (decayed @ k)_r   */
    for (int c = 0; c < K; ++c) dot += S[(size_t)r * K + c] * kv[c];
    const double res = beta * ((vv ? vv[r] : 0.0) - dot);
    if (residual_out) residual_out[r] = res;
    for (int c = 0; c < K; ++c) S[(size_t)r * K + c] += res * kv[c];
  }
}

/* out = scale * S @ q  (S [V,K], q [K]) */
static void read_out(int K, int V, const double *S, const double *qv, double scale,
                     double *o) {
  for (int r = 0; r < V; ++r) {
    double acc = 0.0;
    for (int c = 0; c < K; ++c) acc += S[(size_t)r * K + c] * qv[c];
    o[r] = scale * acc;
  }
}

/* ------------------------------------------------------------------ */
/* Forward                                                              */
/* ------------------------------------------------------------------ */
/* Returns 0, or -1 on malformed arguments.  out rows outside every
 * sequence are left untouched.  Sfinal may be NULL. */
int oracle_gdn_fwd(int B, int T, int H, int K, int V, int N, const int32_t *cu,
                   const double *q, const double *k, const double *v,
                   const double *g, const double *beta, const double *S0,
                   double scale, double *out, double *Sfinal) {
  if (B < 0 || T < 0 || H <= 0 || K <= 0 || V <= 0 || N < 0) return -1;
  if (!cu && N != B) return -1;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int nh = 0; nh < N * H; ++nh) {
    const int n = nh / H, h = nh % H;
    int64_t bos, eos;
    if (seq_rows(n, B, T, cu, &bos, &eos)) { bad = 1; continue; }
    double *S = (double *)malloc(sizeof(double) * (size_t)V * K);
    if (S0)
      memcpy(S, S0 + ((size_t)n * H + h) * V * K, sizeof(double) * (size_t)V * K);
    else
      memset(S, 0, sizeof(double) * (size_t)V * K);
    for (int64_t row = bos; row < eos; ++row) {
      const size_t tk = ((size_t)row * H + h);
      token_step(K, V, S, k + tk * K, v + tk * V, g[tk], beta[tk], NULL, NULL);
      read_out(K, V, S, q + tk * K, scale, out + tk * V);
    }
    if (Sfinal)
      memcpy(Sfinal + ((size_t)n * H + h) * V * K, S, sizeof(double) * (size_t)V * K);
    free(S);
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* Backward: reverse-mode of the per-token rule.                        */
/* For token t (a = exp(g), S_prev -> decayed D = a S_prev,             */
/* p = D k, r = beta (v - p), S = D + r k^T, o = scale S q):            */
/*   dS  += scale do q^T            dq = scale S^T do                   */
/*   dr   = dS k                    dk = dS^T r - beta D^T dr           */
/*   dbeta = dr . (v - p)           dv = beta dr                        */
/*   dD   = dS - beta dr k^T        dg = <dD, D>_F                      */
/*   dS_prev = a dD                                                     */
/* States are checkpointed every `blk` tokens and recomputed inside.   */
/* ------------------------------------------------------------------ */
int oracle_gdn_bwd(int B, int T, int H, int K, int V, int N, const int32_t *cu,
                   const double *q, const double *k, const double *v,
                   const double *g, const double *beta, const double *S0,
                   double scale, const double *dout, const double *dSfinal,
                   double *dq, double *dk, double *dv, double *dg, double *dbeta,
                   double *dS0) {
  if (B < 0 || T < 0 || H <= 0 || K <= 0 || V <= 0 || N < 0) return -1;
  if (!cu && N != B) return -1;
  const int blk = 64;
  const size_t SZ = (size_t)V * K;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int nh = 0; nh < N * H; ++nh) {
    const int n = nh / H, h = nh % H;
    int64_t bos, eos;
    if (seq_rows(n, B, T, cu, &bos, &eos)) { bad = 1; continue; }
    const int64_t L = eos - bos;
    const int64_t nblk = (L + blk - 1) / blk;
    double *ckpt = (double *)malloc(sizeof(double) * SZ * (size_t)(nblk > 0 ? nblk : 1));
    double *Dec = (double *)malloc(sizeof(double) * SZ * blk);    /* decayed state  */
    double *Res = (double *)malloc(sizeof(double) * (size_t)V * blk);
    double *S = (double *)malloc(sizeof(double) * SZ);
    double *dS = (double *)malloc(sizeof(double) * SZ);
    double *dr = (double *)malloc(sizeof(double) * (size_t)V);

    /* forward replay, checkpoint at block starts */
    if (S0) memcpy(S, S0 + (size_t)nh * SZ, sizeof(double) * SZ);
    else memset(S, 0, sizeof(double) * SZ);
    for (int64_t i = 0; i < L; ++i) {
      if (i % blk == 0) memcpy(ckpt + (size_t)(i / blk) * SZ, S, sizeof(double) * SZ);
      const size_t tk = (size_t)(bos + i) * H + h;
      token_step(K, V, S, k + tk * K, v + tk * V, g[tk], beta[tk], NULL, NULL);
    }
    /* reverse */
    if (dSfinal) memcpy(dS, dSfinal + (size_t)nh * SZ, sizeof(double) * SZ);
    else memset(dS, 0, sizeof(double) * SZ);
    for (int64_t b0 = nblk - 1; b0 >= 0; --b0) {
      const int64_t t0 = b0 * blk;
      const int64_t t1 = (t0 + blk < L) ? t0 + blk : L;
      memcpy(S, ckpt + (size_t)b0 * SZ, sizeof(double) * SZ);
      for (int64_t i = t0; i < t1; ++i) {
        const size_t tk = (size_t)(bos + i) * H + h;
        token_step(K, V, S, k + tk * K, v + tk * V, g[tk], beta[tk],
                   Dec + (size_t)(i - t0) * SZ, Res + (size_t)(i - t0) * V);
      }
      /* S now holds the state after token t1-1; walk back */
      for (int64_t i = t1 - 1; i >= t0; --i) {
        const size_t tk = (size_t)(bos + i) * H + h;
        const double *qt = q + tk * K, *kt = k + tk * K, *vt = v + tk * V;
        const double *dot_ = dout + tk * V;
        const double *D = Dec + (size_t)(i - t0) * SZ;
        const double *r = Res + (size_t)(i - t0) * V;
        const double bt = beta[tk], a = exp(g[tk]);
        /* S_t = D + r k^T (recompute from D to avoid storing it) */
        /* dq = scale S_t^T do */
        for (int c = 0; c < K; ++c) {
          double acc = 0.0;
          for (int rr = 0; rr < V; ++rr)
            acc += (D[(size_t)rr * K + c] + r[rr] * kt[c]) * dot_[rr];
          dq[tk * K + c] = scale * acc;
        }
        /* dS += scale do q^T */
        for (int rr = 0; rr < V; ++rr)
          for (int c = 0; c < K; ++c) dS[(size_t)rr * K + c] += scale * dot_[rr] * qt[c];
        /* dr = dS k */
        for (int rr = 0; rr < V; ++rr) {
          double acc = 0.0;
          for (int c = 0; c < K; ++c) acc += dS[(size_t)rr * K + c] * kt[c];
          dr[rr] = acc;
        }
        /* dk = dS^T r - beta D^T dr */
        for (int c = 0; c < K; ++c) {
          double acc = 0.0;
          for (int rr = 0; rr < V; ++rr)
            acc += dS[(size_t)rr * K + c] * r[rr] - bt * D[(size_t)rr * K + c] * dr[rr];
          dk[tk * K + c] = acc;
        }
        /* dbeta = dr . (v - D k); dv = beta dr */
        double db = 0.0;
        for (int rr = 0; rr < V; ++rr) {
          double p = 0.0;
          for (int c = 0; c < K; ++c) p += D[(size_t)rr * K + c] * kt[c];
          db += dr[rr] * (vt[rr] - p);
          dv[tk * V + rr] = bt * dr[rr];
        }
        dbeta[tk] = db;
        /* dD = dS - beta dr k^T ; dg = <dD, D> ; dS_prev = a dD */
        double dgt = 0.0;
        for (int rr = 0; rr < V; ++rr)
          for (int c = 0; c < K; ++c) {
            const double dd = dS[(size_t)rr * K + c] - bt * dr[rr] * kt[c];
            dgt += dd * D[(size_t)rr * K + c];
            dS[(size_t)rr * K + c] = a * dd;
          }
        dg[tk] = dgt;
      }
    }
    if (dS0) memcpy(dS0 + (size_t)nh * SZ, dS, sizeof(double) * SZ);
    free(ckpt); free(Dec); free(Res); free(S); free(dS); free(dr);
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* Segment summary by probing, [AG-CP]:                                 */
/*   E = state after the range from a zero entry state (value term on) */
/*   P = state after the range from the identity (K x K) entry state    */
/*       with the value term disabled.                                  */
/* Then for any entry state S_in: S_out = S_in P + E.                   */
/* bounds: [R,2] flattened token rows (b*T + t), a range may not cross  */
/* a batch row.  Outputs P [R,H,K,K], E [R,H,V,K].                       */
/* ------------------------------------------------------------------ */
int oracle_gdn_summary(int B, int T, int H, int K, int V, const double *k,
                       const double *v, const double *g, const double *beta,
                       const int32_t *bounds, int R, double *P, double *E) {
  if (B < 0 || T <= 0 || H <= 0 || K <= 0 || V <= 0 || R < 0) return -1;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int rh = 0; rh < R * H; ++rh) {
    const int r = rh / H, h = rh % H;
    const int64_t s0 = bounds[2 * r], s1 = bounds[2 * r + 1];
    if (s0 < 0 || s1 < s0 || s1 > (int64_t)B * T ||
        (s1 > s0 && s0 / T != (s1 - 1) / T)) { bad = 1; continue; }
    double *Se = E + (size_t)rh * V * K;
    double *Sp = P + (size_t)rh * K * K;
    memset(Se, 0, sizeof(double) * (size_t)V * K);
    memset(Sp, 0, sizeof(double) * (size_t)K * K);
    for (int i = 0; i < K; ++i) Sp[(size_t)i * K + i] = 1.0;
    for (int64_t row = s0; row < s1; ++row) {
      const size_t tk = (size_t)row * H + h;
      token_step(K, V, Se, k + tk * K, v + tk * V, g[tk], beta[tk], NULL, NULL);
      token_step(K, K, Sp, k + tk * K, NULL, g[tk], beta[tk], NULL, NULL);
    }
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* Exclusive scan of segment maps, [AG-CP] prefix scan over summaries: */
/*   entry_0 = S0,  entry_{j+1} = entry_j P_j + E_j.                    */
/* final = entry_R (the state after the last segment).                 */
/* P [R,H,K,K], E [R,H,V,K], S0 [H,V,K] or NULL (= 0),                  */
/* entry [R,H,V,K], final [H,V,K] or NULL.                              */
/* ------------------------------------------------------------------ */
int oracle_state_scan(int R, int H, int K, int V, const double *P, const double *E,
                      const double *S0, double *entry, double *final_state) {
  if (R < 0 || H <= 0 || K <= 0 || V <= 0) return -1;
  const size_t SZ = (size_t)V * K;
#pragma omp parallel for schedule(static)
  for (int h = 0; h < H; ++h) {
    double *cur = (double *)malloc(sizeof(double) * SZ);
    double *nxt = (double *)malloc(sizeof(double) * SZ);
    if (S0) memcpy(cur, S0 + (size_t)h * SZ, sizeof(double) * SZ);
    else memset(cur, 0, sizeof(double) * SZ);
    for (int j = 0; j < R; ++j) {
      memcpy(entry + ((size_t)j * H + h) * SZ, cur, sizeof(double) * SZ);
      const double *Pj = P + ((size_t)j * H + h) * K * K;
      const double *Ej = E + ((size_t)j * H + h) * SZ;
      for (int rr = 0; rr < V; ++rr)
        for (int c = 0; c < K; ++c) {
          double acc = Ej[(size_t)rr * K + c];
          for (int m = 0; m < K; ++m) acc += cur[(size_t)rr * K + m] * Pj[(size_t)m * K + c];
          nxt[(size_t)rr * K + c] = acc;
        }
      double *tmp = cur; cur = nxt; nxt = tmp;
    }
    if (final_state) memcpy(final_state + (size_t)h * SZ, cur, sizeof(double) * SZ);
    free(cur); free(nxt);
  }
  return 0;
}

/* Threads the OpenMP runtime will use (for the CPU-baseline report). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
