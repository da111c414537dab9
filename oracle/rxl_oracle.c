/*
 * Float64 CPU oracle for Transformer-XL relative-position memory attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file's library. It shares no code,
 * header, table or constant with the CUDA library, and the CUDA library never
 * calls it.
 *
 * It is the plain definition written out, with explicit loops over the query
 * row i and the key position j and a direct lookup of R at the distance i-j:
 *
 *  - key positions: memory -m..-1, current 0..L-1; query positions 0..L-1
 *    (Transformer-XL page, "Causal Mask With Memory");
 *  - allow(i,j) = 1 if j<0, 1 if 0<=j<=i, else 0 (same section, eq. allow);
 *  - per-row document reset: a batch row that entered a new document must
 *    not see the previous document's memory (same section, the note after the
 *    mask picture; "Batched Streams": the reset is per row). Read here as a
 *    mask: batch row b sees only its newest mvis[b] memory rows, i.e. memory
 *    key j is visible iff j >= -mvis[b] (mvis NULL: every row sees all m);
 *  - A_ij = q_i.k_j + q_i.r_{i-j} + u.k_j + v.r_{i-j}
 *         = (q_i+u).k_j + (q_i+v).r_{i-j}
 *    (Transformer-XL page, "Relative Positional Encoding", four-term score;
 *    the same regrouping is printed on the iopencloud page, section 2.2);
 *  - Attn = softmax((A + M_causal)/sqrt(d_h)) V (Transformer-XL page,
 *    "Dimension Walkthrough"); the scale multiplies all four terms;
 *  - R has one row per distance, row d = distance d, d in [0, m+L-1]
 *    ("Dimension Walkthrough": R is (M+L) x d_h);
 *  - stop-gradient: the backward gives dK/dV for memory rows (W_K/W_V still
 *    learn from them) but nothing flows into the cached states (Transformer-XL
 *    page, "Why Stop Gradient"; wq-win page, "stop-gradient到底切断哪里").
 *
 * Positions are carried as absolute integers p = pos0 + index so that the
 * translation-invariance property ("Relative Positional Encoding": shifting
 * every position by c leaves i-j unchanged) can be checked on the oracle.
 *
 * Layouts (all float64, contiguous, row-major, d_h innermost):
 *   q   [B,H,L,dh]          k, v [B,H,m+L,dh] in LOGICAL order: row t<m is
 *   u,vb [H,dh]             memory row t (oldest first), row m+i is current i
 *   r   [H,m+L,dh]          o [B,H,L,dh], lse [B,H,L] (natural log)
 *   dq  [B,H,L,dh]          dk, dv [B,H,m+L,dh], dr [H,m+L,dh], du, dvb [H,dh]
 *
 * Parallelism: independent (b,h) units on POSIX threads. Per-head sums over
 * the batch (dR, du, dv) are taken from per-unit partials in the fixed order
 * b = 0..B-1, so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int B, H, L, m, dh;
  double scale;
  long long pos0;
  const double *q, *k, *v, *r, *u, *vb, *dout;
  double *o, *lse;                 /* forward outputs */
  double *logits;                  /* optional [B,H,L,m+L] */
  double *dq, *dk, *dv;            /* backward outputs per unit */
  double *dr_part, *du_part, *dvb_part; /* per-unit partials */
  const int *sel;                  /* row subset: (b,h,i) triples */
  const int *mvis;                 /* per batch row: newest memory rows visible (or NULL) */
  int nsel;
  int next;                        /* work counter */
  int nunits;
  pthread_mutex_t lock;
} problem;

/* allow(i,j) with absolute positions: the segment starts at pos0, memory keys
 * sit before it and are always visible, current keys up to the query. */
static int allow(long long pi, long long pj, long long pos0) {
  if (pj < pos0) return 1;
  return pj <= pi;
}

/* allow(i,j) for batch row b, with the row's document reset: of the memory
 * keys only the newest mvis[b] are visible. */
static int allow_b(const problem *P, int b, int i, int j) {
  if (P->mvis && j < 0 && j < -P->mvis[b]) return 0;
  return allow(P->pos0 + i, P->pos0 + j, P->pos0);
}

/* scaled score s*A_ij of query row i against key position j (j in [-m, L)). */
static double scaled_score(const problem *P, int b, int h, int i, int j) {
  const int dh = P->dh, mL = P->m + P->L;
  const double *qi = P->q + (((size_t)b * P->H + h) * P->L + i) * dh;
  const double *kj = P->k + (((size_t)b * P->H + h) * mL + (P->m + j)) * dh;
  const long long pi = P->pos0 + i, pj = P->pos0 + j;
  const long long d = pi - pj; /* relative distance */
  const double *rd = P->r + ((size_t)h * mL + (size_t)d) * dh;
  const double *u = P->u + (size_t)h * dh, *vb = P->vb + (size_t)h * dh;
  double content = 0.0, position = 0.0;
  for (int c = 0; c < dh; ++c) content += (qi[c] + u[c]) * kj[c];
  for (int c = 0; c < dh; ++c) position += (qi[c] + vb[c]) * rd[c];
  return P->scale * (content + position);
}

/* Softmax statistics of row i: fills z[j+m] (scaled scores, -inf if masked),
 * returns the max and the sum of exp(z - max). */
static void row_stats(const problem *P, int b, int h, int i, double *z, double *mx_out,
                      double *l_out) {
  double mx = -INFINITY;
  for (int j = -P->m; j < P->L; ++j) {
    if (allow_b(P, b, i, j)) {
      z[j + P->m] = scaled_score(P, b, h, i, j);
      if (z[j + P->m] > mx) mx = z[j + P->m];
    } else {
      z[j + P->m] = -INFINITY;
    }
  }
  double l = 0.0;
  for (int j = -P->m; j < P->L; ++j)
    if (z[j + P->m] != -INFINITY) l += exp(z[j + P->m] - mx);
  *mx_out = mx;
  *l_out = l;
}

static void fwd_row(const problem *P, int b, int h, int i, double *z, double *o_row,
                    double *lse_out) {
  const int dh = P->dh, mL = P->m + P->L;
  double mx, l;
  row_stats(P, b, h, i, z, &mx, &l);
  for (int c = 0; c < dh; ++c) o_row[c] = 0.0;
  for (int j = -P->m; j < P->L; ++j) {
    if (z[j + P->m] == -INFINITY) continue;
    const double p = exp(z[j + P->m] - mx) / l;
    const double *vj = P->v + (((size_t)b * P->H + h) * mL + (P->m + j)) * dh;
    for (int c = 0; c < dh; ++c) o_row[c] += p * vj[c];
  }
  *lse_out = mx + log(l);
}

static int take(problem *P) {
  pthread_mutex_lock(&P->lock);
  int u = P->next < P->nunits ? P->next++ : -1;
  pthread_mutex_unlock(&P->lock);
  return u;
}

static void *fwd_worker(void *arg) {
  problem *P = (problem *)arg;
  double *z = (double *)malloc(sizeof(double) * (size_t)(P->m + P->L));
  for (int unit; (unit = take(P)) >= 0;) {
    const int b = unit / P->H, h = unit % P->H;
    for (int i = 0; i < P->L; ++i) {
      const size_t row = ((size_t)b * P->H + h) * P->L + i;
      fwd_row(P, b, h, i, z, P->o + row * P->dh, P->lse + row);
    }
  }
  free(z);
  return NULL;
}

static void *rows_worker(void *arg) {
  problem *P = (problem *)arg;
  double *z = (double *)malloc(sizeof(double) * (size_t)(P->m + P->L));
  for (int s; (s = take(P)) >= 0;) {
    const int b = P->sel[3 * s], h = P->sel[3 * s + 1], i = P->sel[3 * s + 2];
    fwd_row(P, b, h, i, z, P->o + (size_t)s * P->dh, P->lse + s);
  }
  free(z);
  return NULL;
}

static void *logits_worker(void *arg) {
  problem *P = (problem *)arg;
  const int mL = P->m + P->L;
  for (int unit; (unit = take(P)) >= 0;) {
    const int b = unit / P->H, h = unit % P->H;
    for (int i = 0; i < P->L; ++i)
      for (int j = -P->m; j < P->L; ++j) {
        double *dst = P->logits + ((((size_t)b * P->H + h) * P->L + i) * mL + (P->m + j));
        *dst = allow_b(P, b, i, j) ? scaled_score(P, b, h, i, j) : -INFINITY;
      }
  }
  return NULL;
}

/* Backward of one (b,h) unit, following the chain rule of the score:
 *   D_i = sum_j P_ij (dO_i . V_j),  dS_ij = P_ij (dO_i . V_j - D_i),
 *   dA_ij = scale * dS_ij,
 *   dq_i += dA_ij (k_j + r_{i-j}),  dk_j += dA_ij (q_i + u),
 *   dv_j += P_ij dO_i,  dr_{i-j} += dA_ij (q_i + v),
 *   du += dA_ij k_j,  dvb += dA_ij r_{i-j}. */
static void *bwd_worker(void *arg) {
  problem *P = (problem *)arg;
  const int dh = P->dh, mL = P->m + P->L;
  double *z = (double *)malloc(sizeof(double) * (size_t)mL);
  for (int unit; (unit = take(P)) >= 0;) {
    const int b = unit / P->H, h = unit % P->H;
    const size_t bh = (size_t)b * P->H + h;
    double *dr = P->dr_part + (size_t)unit * mL * dh;
    double *du = P->du_part + (size_t)unit * dh;
    double *dvb = P->dvb_part + (size_t)unit * dh;
    const double *u = P->u + (size_t)h * dh, *vb = P->vb + (size_t)h * dh;
    for (int i = 0; i < P->L; ++i) {
      const double *qi = P->q + (bh * P->L + i) * dh;
      const double *doi = P->dout + (bh * P->L + i) * dh;
      double *dqi = P->dq + (bh * P->L + i) * dh;
      double mx, l;
      row_stats(P, b, h, i, z, &mx, &l);
      double Di = 0.0;
      for (int j = -P->m; j < P->L; ++j) {
        if (z[j + P->m] == -INFINITY) continue;
        const double p = exp(z[j + P->m] - mx) / l;
        const double *vj = P->v + (bh * mL + (P->m + j)) * dh;
        double dp = 0.0;
        for (int c = 0; c < dh; ++c) dp += doi[c] * vj[c];
        Di += p * dp;
      }
      for (int j = -P->m; j < P->L; ++j) {
        if (z[j + P->m] == -INFINITY) continue;
        const double p = exp(z[j + P->m] - mx) / l;
        const double *kj = P->k + (bh * mL + (P->m + j)) * dh;
        const double *vj = P->v + (bh * mL + (P->m + j)) * dh;
        const long long d = (P->pos0 + i) - (P->pos0 + j);
        const double *rd = P->r + ((size_t)h * mL + (size_t)d) * dh;
        double dp = 0.0;
        for (int c = 0; c < dh; ++c) dp += doi[c] * vj[c];
        const double dA = P->scale * p * (dp - Di);
        double *dkj = P->dk + (bh * mL + (P->m + j)) * dh;
        double *dvj = P->dv + (bh * mL + (P->m + j)) * dh;
        double *drd = dr + (size_t)d * dh;
        for (int c = 0; c < dh; ++c) {
          dqi[c] += dA * (kj[c] + rd[c]);
          dkj[c] += dA * (qi[c] + u[c]);
          dvj[c] += p * doi[c];
          drd[c] += dA * (qi[c] + vb[c]);
          du[c] += dA * kj[c];
          dvb[c] += dA * rd[c];
        }
      }
    }
  }
  free(z);
  return NULL;
}

static void run(problem *P, void *(*fn)(void *), int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > P->nunits) nthreads = P->nunits > 0 ? P->nunits : 1;
  pthread_mutex_init(&P->lock, NULL);
  P->next = 0;
  pthread_t *t = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  for (int n = 1; n < nthreads; ++n) pthread_create(&t[n], NULL, fn, P);
  fn(P);
  for (int n = 1; n < nthreads; ++n) pthread_join(t[n], NULL);
  free(t);
  pthread_mutex_destroy(&P->lock);
}

static void setup(problem *P, int B, int H, int L, int m, int dh, double scale,
                  long long pos0, const double *q, const double *k, const double *v,
                  const double *r, const double *u, const double *vb) {
  memset(P, 0, sizeof(*P));
  P->B = B; P->H = H; P->L = L; P->m = m; P->dh = dh; P->scale = scale; P->pos0 = pos0;
  P->q = q; P->k = k; P->v = v; P->r = r; P->u = u; P->vb = vb;
  P->nunits = B * H;
}

/* Forward over all (b,h,i): O and LSE. */
void oracle_fwd(int B, int H, int L, int m, int dh, double scale, long long pos0,
                const double *q, const double *k, const double *v, const double *r,
                const double *u, const double *vb, double *o, double *lse, int nthreads) {
  problem P;
  setup(&P, B, H, L, m, dh, scale, pos0, q, k, v, r, u, vb);
  P.o = o; P.lse = lse;
  run(&P, fwd_worker, nthreads);
}

/* Forward of selected rows only: sel holds nsel (b,h,i) triples; o is
 * [nsel,dh], lse [nsel]. */
void oracle_fwd_rows(int B, int H, int L, int m, int dh, double scale, long long pos0,
                     const double *q, const double *k, const double *v, const double *r,
                     const double *u, const double *vb, int nsel, const int *sel, double *o,
                     double *lse, int nthreads) {
  problem P;
  setup(&P, B, H, L, m, dh, scale, pos0, q, k, v, r, u, vb);
  P.o = o; P.lse = lse; P.sel = sel; P.nsel = nsel; P.nunits = nsel;
  run(&P, rows_worker, nthreads);
}

/* Scaled logits s*A_ij, -inf where masked: [B,H,L,m+L]. */
void oracle_logits(int B, int H, int L, int m, int dh, double scale, long long pos0,
                   const double *q, const double *k, const double *r, const double *u,
                   const double *vb, double *logits, int nthreads) {
  problem P;
  setup(&P, B, H, L, m, dh, scale, pos0, q, k, NULL, r, u, vb);
  P.logits = logits;
  run(&P, logits_worker, nthreads);
}

/* Backward: all outputs are overwritten. dk/dv cover memory rows too (the
 * K/V gradient of cached rows); nothing is returned for the cached states. */
static int bwd_impl(int B, int H, int L, int m, int dh, double scale, long long pos0,
                    const double *q, const double *k, const double *v, const double *r,
                    const double *u, const double *vb, const int *mvis, const double *dout,
                    double *dq, double *dk, double *dv, double *dr, double *du, double *dvb,
                    int nthreads) {
  problem P;
  setup(&P, B, H, L, m, dh, scale, pos0, q, k, v, r, u, vb);
  P.mvis = mvis;
  const int mL = m + L;
  const size_t units = (size_t)B * H;
  P.dout = dout; P.dq = dq; P.dk = dk; P.dv = dv;
  memset(dq, 0, sizeof(double) * units * L * dh);
  memset(dk, 0, sizeof(double) * units * mL * dh);
  memset(dv, 0, sizeof(double) * units * mL * dh);
  P.dr_part = (double *)calloc(units * mL * dh, sizeof(double));
  P.du_part = (double *)calloc(units * dh, sizeof(double));
  P.dvb_part = (double *)calloc(units * dh, sizeof(double));
  if (!P.dr_part || !P.du_part || !P.dvb_part) {
    free(P.dr_part); free(P.du_part); free(P.dvb_part);
    return -1;
  }
  run(&P, bwd_worker, nthreads);
  /* per-head sums over the batch in the fixed order b = 0..B-1 */
  memset(dr, 0, sizeof(double) * (size_t)H * mL * dh);
  memset(du, 0, sizeof(double) * (size_t)H * dh);
  memset(dvb, 0, sizeof(double) * (size_t)H * dh);
  for (int h = 0; h < H; ++h)
    for (int b = 0; b < B; ++b) {
      const size_t unit = (size_t)b * H + h;
      for (size_t e = 0; e < (size_t)mL * dh; ++e)
        dr[(size_t)h * mL * dh + e] += P.dr_part[unit * mL * dh + e];
      for (int c = 0; c < dh; ++c) {
        du[(size_t)h * dh + c] += P.du_part[unit * dh + c];
        dvb[(size_t)h * dh + c] += P.dvb_part[unit * dh + c];
      }
    }
  free(P.dr_part); free(P.du_part); free(P.dvb_part);
  return 0;
}

int oracle_bwd(int B, int H, int L, int m, int dh, double scale, long long pos0,
               const double *q, const double *k, const double *v, const double *r,
               const double *u, const double *vb, const double *dout, double *dq, double *dk,
               double *dv, double *dr, double *du, double *dvb, int nthreads) {
  return bwd_impl(B, H, L, m, dh, scale, pos0, q, k, v, r, u, vb, NULL, dout, dq, dk, dv, dr, du,
                  dvb, nthreads);
}

/* The same with a per-batch-row document reset: mvis[b] in [0, m] is the
 * number of newest memory rows batch row b may attend to. */
void oracle_fwd_reset(int B, int H, int L, int m, int dh, double scale, long long pos0,
                      const double *q, const double *k, const double *v, const double *r,
                      const double *u, const double *vb, const int *mvis, double *o, double *lse,
                      int nthreads) {
  problem P;
  setup(&P, B, H, L, m, dh, scale, pos0, q, k, v, r, u, vb);
  P.mvis = mvis;
  P.o = o; P.lse = lse;
  run(&P, fwd_worker, nthreads);
}

int oracle_bwd_reset(int B, int H, int L, int m, int dh, double scale, long long pos0,
                     const double *q, const double *k, const double *v, const double *r,
                     const double *u, const double *vb, const int *mvis, const double *dout,
                     double *dq, double *dk, double *dv, double *dr, double *du, double *dvb,
                     int nthreads) {
  return bwd_impl(B, H, L, m, dh, scale, pos0, q, k, v, r, u, vb, mvis, dout, dq, dk, dv, dr, du,
                  dvb, nthreads);
}
