/*
 * gdn_oracle.c -- plain fp64 CPU reference of the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (per batch b and value head j, key head kh = j / (Hv/Hk)):
 *
 *   the per-token gated delta rule, written on the transposed state
 *   h = S^T (d_k x d_v):
 *       a_t  = exp(g_t)
 *       h_t  = a_t (I - beta_t k_t k_t^T) h_{t-1} + beta_t k_t v_t^T
 *       o_t  = h_t^T q_t
 *   This is the rule S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T)
 *   + beta_t v_t k_t^T, o_t = S_t q_t ("Shard the GatedDeltaNet sequence
 *   under ici_context_parallelism", description: the inter-chunk step is the
 *   chunked form of this rule; the per-token statement itself is the
 *   problem statement of the chunked Gated DeltaNet forward), transposed.
 *
 *   and its exact per-token adjoint (reverse-mode derivative of the loop
 *   above), walking t downwards.  With dH the gradient reaching h_t
 *   (the future's contribution plus q_t do_t^T), p = h_{t-1}^T k_t,
 *   u = dH^T k_t and e = v_t - a_t p:
 *       dq_t   = h_t do_t
 *       dv_t   = beta_t u
 *       dbeta_t= u . e
 *       dk_t   = beta_t dH e - a_t beta_t h_{t-1} u
 *       dg_t   = a_t ( <dH, h_{t-1}> - beta_t p . u )
 *       dh_{t-1} = a_t (dH - beta_t k_t u^T)
 *
 * Inputs q, k, v, dO arrive as bf16 bit patterns (uint16) and are widened
 * exactly; g, beta, h0, dhT arrive as fp32.  All arithmetic is fp64.
 * Layouts: q,k [B,T,Hk,dk]; v,dO [B,T,Hv,dv]; g,beta [B,T,Hv];
 * h0,dhT [B,Hv,dk,dv].
 *
 * Parallelism is over independent work only: heads, and in the forward also
 * blocks of state columns (each column of h follows its own recurrence given
 * k, a and beta, so splitting columns changes no arithmetic).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double widen_bf16(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Forward.  Selected heads (sel_b[i], sel_j[i]), i < n_sel.
 * o:  [n_sel, T, dv] fp64, may be NULL.   hT: [n_sel, dk, dv] fp64, may be NULL.
 * col_block: columns of h per parallel task (dv % col_block == 0).
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int orc_fwd(int B, int T, int Hk, int Hv, int dk, int dv,
            const uint16_t* q, const uint16_t* k, const uint16_t* v,
            const float* g, const float* beta, const float* h0,
            int n_sel, const int* sel_b, const int* sel_j,
            double* o, double* hT, int col_block) {
  if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || Hv % Hk || dk <= 0 || dv <= 0) return -1;
  if (col_block <= 0 || dv % col_block) return -1;
  const int group = Hv / Hk;
  const int nblk = dv / col_block;
  const long ntask = (long)n_sel * nblk;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (long task = 0; task < ntask; ++task) {
    const int si = (int)(task / nblk), blk = (int)(task % nblk);
    const int b = sel_b[si], j = sel_j[si], kh = j / group;
    const int c0 = blk * col_block, nc = col_block;
    double* h = (double*)malloc(sizeof(double) * (size_t)dk * nc);
    double* kt = (double*)malloc(sizeof(double) * (size_t)dk);
    double* qt = (double*)malloc(sizeof(double) * (size_t)dk);
    double* p = (double*)malloc(sizeof(double) * (size_t)nc);
    if (!h || !kt || !qt || !p) {
      bad |= 1;
      free(h); free(kt); free(qt); free(p);
      continue;
    }
    for (int i = 0; i < dk; ++i)
      for (int c = 0; c < nc; ++c)
        h[(size_t)i * nc + c] =
            h0 ? (double)h0[(((size_t)b * Hv + j) * dk + i) * dv + c0 + c] : 0.0;
    for (int t = 0; t < T; ++t) {
      const size_t tok = (size_t)b * T + t;
      const double a = exp((double)g[tok * Hv + j]);
      const double bt = (double)beta[tok * Hv + j];
      for (int i = 0; i < dk; ++i) {
        kt[i] = widen_bf16(k[(tok * Hk + kh) * dk + i]);
        qt[i] = widen_bf16(q[(tok * Hk + kh) * dk + i]);
      }
      /* p = h^T k */
      for (int c = 0; c < nc; ++c) p[c] = 0.0;
      for (int i = 0; i < dk; ++i)
        for (int c = 0; c < nc; ++c) p[c] += h[(size_t)i * nc + c] * kt[i];
      /* h = a (h - beta k p^T) + beta k v^T */
      for (int i = 0; i < dk; ++i)
        for (int c = 0; c < nc; ++c) {
          const double vc = widen_bf16(v[(tok * Hv + j) * dv + c0 + c]);
          double* hic = &h[(size_t)i * nc + c];
          *hic = a * (*hic - bt * kt[i] * p[c]) + bt * kt[i] * vc;
        }
      /* o_t = h^T q */
      if (o) {
        for (int c = 0; c < nc; ++c) {
          double s = 0.0;
          for (int i = 0; i < dk; ++i) s += h[(size_t)i * nc + c] * qt[i];
          o[((size_t)si * T + t) * dv + c0 + c] = s;
        }
      }
    }
    if (hT)
      for (int i = 0; i < dk; ++i)
        for (int c = 0; c < nc; ++c)
          hT[((size_t)si * dk + i) * dv + c0 + c] = h[(size_t)i * nc + c];
    free(h); free(kt); free(qt); free(p);
  }
  return bad ? -1 : 0;
}

/*
 * Backward (exact adjoint of orc_fwd) for selected heads.
 * dO: [B,T,Hv,dv] bf16 bits; dhT: [B,Hv,dk,dv] fp32 or NULL (zero).
 * Outputs, per selected head (fp64):
 *   dq, dk_out: [n_sel, T, dk]  (this value head's contribution; the caller
 *               sums the heads that share a key head)
 *   dv_out:     [n_sel, T, dv]
 *   dg, dbeta:  [n_sel, T]
 *   dh0:        [n_sel, dk, dv]
 * ckpt: tokens between stored forward states (states inside a block are
 * recomputed from the block's stored start state).
 */
int orc_bwd(int B, int T, int Hk, int Hv, int dk, int dv,
            const uint16_t* q, const uint16_t* k, const uint16_t* v,
            const float* g, const float* beta, const float* h0,
            const uint16_t* dO, const float* dhT,
            int n_sel, const int* sel_b, const int* sel_j,
            double* dq, double* dk_out, double* dv_out, double* dg,
            double* dbeta, double* dh0, int ckpt) {
  if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || Hv % Hk || dk <= 0 || dv <= 0) return -1;
  if (ckpt <= 0) return -1;
  const int group = Hv / Hk;
  const size_t hs = (size_t)dk * dv;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int si = 0; si < n_sel; ++si) {
    const int b = sel_b[si], j = sel_j[si], kh = j / group;
    const int nck = (T + ckpt - 1) / ckpt;
    /* ck[c] = state before token c*ckpt;  blk[i] = state after token t0+i */
    double* ck = (double*)malloc(sizeof(double) * hs * (size_t)(nck > 0 ? nck : 1));
    double* blk = (double*)malloc(sizeof(double) * hs * (size_t)(ckpt + 1));
    double* dH = (double*)malloc(sizeof(double) * hs);
    double* kt = (double*)malloc(sizeof(double) * (size_t)dk);
    double* qt = (double*)malloc(sizeof(double) * (size_t)dk);
    double* vt = (double*)malloc(sizeof(double) * (size_t)dv);
    double* dot = (double*)malloc(sizeof(double) * (size_t)dv);
    double* p = (double*)malloc(sizeof(double) * (size_t)dv);
    double* u = (double*)malloc(sizeof(double) * (size_t)dv);
    double* e = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!ck || !blk || !dH || !kt || !qt || !vt || !dot || !p || !u || !e) {
      bad |= 1;
      free(ck); free(blk); free(dH); free(kt); free(qt); free(vt); free(dot);
      free(p); free(u); free(e);
      continue;
    }
#define LOADTOK(t_)                                                        \
  do {                                                                     \
    const size_t tok_ = (size_t)b * T + (t_);                              \
    for (int i = 0; i < dk; ++i) {                                         \
      kt[i] = widen_bf16(k[(tok_ * Hk + kh) * dk + i]);                    \
      qt[i] = widen_bf16(q[(tok_ * Hk + kh) * dk + i]);                    \
    }                                                                      \
    for (int c = 0; c < dv; ++c) vt[c] = widen_bf16(v[(tok_ * Hv + j) * dv + c]); \
  } while (0)
    /* one forward step: hout = a (hin - beta k (hin^T k)^T) + beta k v^T */
#define STEP(hin, hout, a_, bt_)                                           \
  do {                                                                     \
    for (int c = 0; c < dv; ++c) p[c] = 0.0;                               \
    for (int i = 0; i < dk; ++i)                                           \
      for (int c = 0; c < dv; ++c) p[c] += (hin)[(size_t)i * dv + c] * kt[i]; \
    for (int i = 0; i < dk; ++i)                                           \
      for (int c = 0; c < dv; ++c)                                         \
        (hout)[(size_t)i * dv + c] =                                       \
            (a_) * ((hin)[(size_t)i * dv + c] - (bt_) * kt[i] * p[c]) +    \
            (bt_) * kt[i] * vt[c];                                         \
  } while (0)

    /* forward sweep: store checkpoints */
    double* cur = blk; /* scratch state */
    for (size_t x = 0; x < hs; ++x)
      cur[x] = h0 ? (double)h0[((size_t)b * Hv + j) * hs + x] : 0.0;
    for (int t = 0; t < T; ++t) {
      if (t % ckpt == 0) memcpy(&ck[(size_t)(t / ckpt) * hs], cur, sizeof(double) * hs);
      const size_t tok = (size_t)b * T + t;
      const double a = exp((double)g[tok * Hv + j]);
      const double bt = (double)beta[tok * Hv + j];
      LOADTOK(t);
      double* nxt = blk + hs; /* ping-pong inside blk[0], blk[1] */
      STEP(cur, nxt, a, bt);
      memcpy(cur, nxt, sizeof(double) * hs);
    }
    /* dH starts as dhT */
    for (size_t x = 0; x < hs; ++x)
      dH[x] = dhT ? (double)dhT[((size_t)b * Hv + j) * hs + x] : 0.0;
    for (int cb = nck - 1; cb >= 0; --cb) {
      const int t0 = cb * ckpt;
      const int t1 = (t0 + ckpt < T) ? t0 + ckpt : T;
      /* blk[0] = state before t0; blk[i+1] = state after token t0+i */
      memcpy(blk, &ck[(size_t)cb * hs], sizeof(double) * hs);
      for (int t = t0; t < t1; ++t) {
        const size_t tok = (size_t)b * T + t;
        const double a = exp((double)g[tok * Hv + j]);
        const double bt = (double)beta[tok * Hv + j];
        LOADTOK(t);
        STEP(&blk[(size_t)(t - t0) * hs], &blk[(size_t)(t - t0 + 1) * hs], a, bt);
      }
      for (int t = t1 - 1; t >= t0; --t) {
        const size_t tok = (size_t)b * T + t;
        const double a = exp((double)g[tok * Hv + j]);
        const double bt = (double)beta[tok * Hv + j];
        LOADTOK(t);
        for (int c = 0; c < dv; ++c) dot[c] = widen_bf16(dO[(tok * Hv + j) * dv + c]);
        const double* hprev = &blk[(size_t)(t - t0) * hs];
        const double* hcur = &blk[(size_t)(t - t0 + 1) * hs];
        /* dH += q do^T */
        for (int i = 0; i < dk; ++i)
          for (int c = 0; c < dv; ++c) dH[(size_t)i * dv + c] += qt[i] * dot[c];
        /* dq_t = h_t do_t */
        for (int i = 0; i < dk; ++i) {
          double s = 0.0;
          for (int c = 0; c < dv; ++c) s += hcur[(size_t)i * dv + c] * dot[c];
          dq[((size_t)si * T + t) * dk + i] = s;
        }
        /* p = h_{t-1}^T k ; u = dH^T k ; e = v - a p */
        for (int c = 0; c < dv; ++c) { p[c] = 0.0; u[c] = 0.0; }
        for (int i = 0; i < dk; ++i)
          for (int c = 0; c < dv; ++c) {
            p[c] += hprev[(size_t)i * dv + c] * kt[i];
            u[c] += dH[(size_t)i * dv + c] * kt[i];
          }
        double db = 0.0, pu = 0.0;
        for (int c = 0; c < dv; ++c) {
          e[c] = vt[c] - a * p[c];
          db += u[c] * e[c];
          pu += p[c] * u[c];
          dv_out[((size_t)si * T + t) * dv + c] = bt * u[c];
        }
        dbeta[(size_t)si * T + t] = db;
        double hh = 0.0;
        for (size_t x = 0; x < hs; ++x) hh += dH[x] * hprev[x];
        dg[(size_t)si * T + t] = a * (hh - bt * pu);
        /* dk_t = beta dH e - a beta h_{t-1} u */
        for (int i = 0; i < dk; ++i) {
          double s1 = 0.0, s2 = 0.0;
          for (int c = 0; c < dv; ++c) {
            s1 += dH[(size_t)i * dv + c] * e[c];
            s2 += hprev[(size_t)i * dv + c] * u[c];
          }
          dk_out[((size_t)si * T + t) * dk + i] = bt * s1 - a * bt * s2;
        }
        /* dh_{t-1} = a (dH - beta k u^T) */
        for (int i = 0; i < dk; ++i)
          for (int c = 0; c < dv; ++c)
            dH[(size_t)i * dv + c] = a * (dH[(size_t)i * dv + c] - bt * kt[i] * u[c]);
      }
    }
    memcpy(&dh0[(size_t)si * hs], dH, sizeof(double) * hs);
#undef LOADTOK
#undef STEP
    free(ck); free(blk); free(dH); free(kt); free(qt); free(vt); free(dot);
    free(p); free(u); free(e);
  }
  return bad ? -1 : 0;
}
