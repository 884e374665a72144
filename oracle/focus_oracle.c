/*
 * Focus centroid-gated sparse attention, forward and backward: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously correct statement of
 * what the CUDA path computes. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may build, load or call it. It shares no code, header, table or
 * helper with the CUDA library, and the CUDA library never calls it.
 *
 * Source: "Why Attend to Everything? Focus is the Key" (Yao, Chen et al.).
 *   [GS-CA]  gist.science technical summary, section 2 "Core Architecture":
 *            K learnable centroids C in R^{K x d_g}; each token's hidden state is
 *            projected into centroid space; local window w attends with exact
 *            softmax; distant tokens attend only within a shared group.
 *   [GS-TK]  same section, "Inference Efficiency (Top-k)": each token joins its
 *            top-k highest-scoring groups; distant tokens interact only if they
 *            share at least one group; cost O(n^2/K + n w).
 *   [GS-SH]  same summary, "Key Technical Innovation: Sinkhorn Normalization":
 *            Sinkhorn replaces softmax and enforces balanced group sizes
 *            (doubly-stochastic assignment).
 *   [JB-M]   jindou-blog deep read, method bullets: K centroids per layer,
 *            routing dimension 16, tokens scored against centroids by dot product;
 *            window part is full-precision softmax, long-range part is an exact
 *            softmax restricted to same-group pairs.
 *
 * Readings taken where the pages are silent (each one is listed in the design notes):
 *   - score s_ig = r_i . c_g (dot product, [JB-M]);
 *   - Sinkhorn is the log-domain SwAV-style iteration: column step gives each group
 *     mass N/K, row step gives each token mass 1; eps scales the scores; run over
 *     the whole sequence of one (batch, routing head); top-k ranks by the final
 *     column-normalised log-score kappa_ig = s_ig/eps + beta_g (the row potential
 *     cannot reorder a row);
 *   - top-k ties go to the lower group index;
 *   - window pairs are j <= i with i - j < w (diagonal included); long-range pairs
 *     are j <= i - w whose masks intersect; the attended set is the union, each key
 *     once, and one softmax runs over it;
 *   - logits are scale * q_i . k_j (scale = 1/sqrt(d) by default); LSE is the
 *     natural log of the sum of exp of those scaled logits.
 *
 * Numbers: Q/K/V arrive as bf16 bit patterns and are widened exactly to double;
 * r and C are fp32 and widened exactly. All arithmetic below is double, except the
 * optional fp32 score mode (score_fp32 = 1), which forms each score as the same
 * fixed-order fused multiply-add chain over t = 0..15 that a single-precision
 * implementation would use, so that argmax decisions can be compared in the
 * kernel's precision.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define DG 16

static double bf16_to_double(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ---------------------------------------------------------------- routing -- */

/* s_ig = sum_t r_it c_gt  ([JB-M]: dot-product score of token i against centroid g). */
static double score(const float* ri, const float* cg, int score_fp32) {
  if (score_fp32) {
    float s = 0.0f;
    for (int t = 0; t < DG; ++t) s = fmaf(ri[t], cg[t], s);
    return (double)s;
  }
  double s = 0.0;
  for (int t = 0; t < DG; ++t) s += (double)ri[t] * (double)cg[t];
  return s;
}

/* log sum_j exp(x_j) with the maximum shifted out. */
static double logsumexp(const double* x, int64_t n, int64_t stride) {
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) if (x[j * stride] > m) m = x[j * stride];
  if (m == -INFINITY) return -INFINITY;
  double s = 0.0;
  for (int64_t j = 0; j < n; ++j) s += exp(x[j * stride] - m);
  return m + log(s);
}

/*
 * Routing for every (b, routing head rho): scores, optional Sinkhorn, top-k.
 *   r      [B, N, R, 16] fp32      C [K, 16] fp32
 *   mask   [B, R, N] uint32 out: bit g set iff g is among the token's top_k groups
 *   margin [B, R, N] double out (nullable): kappa_(k) - kappa_(k+1), +inf if k == K
 *   kappa  [B, R, N, K] double out (nullable): the ranking keys
 *   beta   [B, R, K] double out (nullable): final column potentials (0 if T == 0)
 * Returns 0, or -1 on bad arguments.
 */
int oracle_route(int B, int N, int R, int K, int top_k, int T, double eps, int score_fp32,
                 const float* r, const float* C, uint32_t* mask, double* margin,
                 double* kappa_out, double* beta_out) {
  if (B < 1 || N < 1 || R < 1 || K < 1 || K > 32 || top_k < 1 || top_k > K || T < 0 ||
      !(eps > 0.0))
    return -1;
  double* L = (double*)malloc(sizeof(double) * (size_t)N * K);
  double* alpha = (double*)malloc(sizeof(double) * (size_t)N);
  double* col = (double*)malloc(sizeof(double) * (size_t)N);
  double beta[32];
  if (!L || !alpha || !col) { free(L); free(alpha); free(col); return -1; }

  for (int b = 0; b < B; ++b) {
    for (int rho = 0; rho < R; ++rho) {
      /* 1. scores ([JB-M]); divided by eps when Sinkhorn runs. */
      for (int64_t i = 0; i < N; ++i) {
        const float* ri = r + (((int64_t)b * N + i) * R + rho) * DG;
        for (int g = 0; g < K; ++g) {
          double s = score(ri, C + (int64_t)g * DG, score_fp32);
          L[i * K + g] = (T > 0) ? s / eps : s;
        }
      }
      /* 2. Sinkhorn ([GS-SH]), log domain: potentials alpha (rows), beta (columns). */
      for (int g = 0; g < K; ++g) beta[g] = 0.0;
      for (int64_t i = 0; i < N; ++i) alpha[i] = 0.0;
      for (int it = 0; it < T; ++it) {
        /* column step: sum_i P_ig = N / K */
        for (int g = 0; g < K; ++g) {
          for (int64_t i = 0; i < N; ++i) col[i] = L[i * K + g] + alpha[i];
          beta[g] = log((double)N / (double)K) - logsumexp(col, N, 1);
        }
        /* row step: sum_g P_ig = 1 */
        for (int64_t i = 0; i < N; ++i) {
          double row[32];
          for (int g = 0; g < K; ++g) row[g] = L[i * K + g] + beta[g];
          alpha[i] = -logsumexp(row, K, 1);
        }
      }
      if (beta_out)
        for (int g = 0; g < K; ++g) beta_out[((int64_t)b * R + rho) * K + g] = beta[g];
      /* 3. hard top-k membership ([GS-TK]); ties go to the lower group index. */
      for (int64_t i = 0; i < N; ++i) {
        double key[32];
        int taken[32] = {0};
        for (int g = 0; g < K; ++g) key[g] = L[i * K + g] + beta[g];
        uint32_t bits = 0;
        double kth = 0.0;
        for (int sel = 0; sel < top_k; ++sel) {
          int best = -1;
          for (int g = 0; g < K; ++g)
            if (!taken[g] && (best < 0 || key[g] > key[best])) best = g;
          taken[best] = 1;
          bits |= 1u << best;
          kth = key[best];
        }
        double next = -INFINITY;
        int any_left = 0;
        for (int g = 0; g < K; ++g)
          if (!taken[g]) { if (!any_left || key[g] > next) next = key[g]; any_left = 1; }
        int64_t o = ((int64_t)b * R + rho) * N + i;
        mask[o] = bits;
        if (margin) margin[o] = any_left ? kth - next : INFINITY;
        if (kappa_out)
          for (int g = 0; g < K; ++g) kappa_out[o * K + g] = key[g];
      }
    }
  }
  free(L); free(alpha); free(col);
  return 0;
}

/* ---------------------------------------------------------------- pairs ----- */

/* Is key j in query i's attended set?  ([GS-CA], [GS-TK], [JB-M]) */
static int allowed(int64_t i, int64_t j, int w, uint32_t mi, uint32_t mj) {
  if (j > i) return 0;                 /* causal */
  if (i - j < w) return 1;             /* local window, every pair */
  return (mi & mj) != 0;               /* distant: must share a group */
}

/* Number of allowed (i, j) pairs for every (b, routing head): out [B, R] int64.
 * Brute force over all pairs; meant for small N. */
int oracle_allowed_pairs(int B, int N, int R, int w, const uint32_t* mask, int64_t* out) {
  if (B < 1 || N < 1 || R < 1 || w < 1) return -1;
  for (int b = 0; b < B; ++b)
    for (int rho = 0; rho < R; ++rho) {
      const uint32_t* m = mask + ((int64_t)b * R + rho) * N;
      int64_t c = 0;
      for (int64_t i = 0; i < N; ++i)
        for (int64_t j = 0; j <= i; ++j) c += allowed(i, j, w, m[i], m[j]);
      out[(int64_t)b * R + rho] = c;
    }
  return 0;
}

/* ------------------------------------------------------------- attention ---- */

typedef struct {
  int B, N, H, H_kv, R, d, w;
  double scale;
  const uint16_t *q, *k, *v;
  const uint32_t* mask;
  const int64_t* rows; /* flattened (b * N + i) query rows, or NULL for all */
  int64_t n_rows;
  const int32_t* heads; /* query heads to compute, or NULL for all H */
  int n_heads;
  double *o, *lse;
  int64_t next;        /* work counter */
  pthread_mutex_t mu;
} attn_job;

/* One query row of one head: two-pass softmax over the union set A_i. */
static void attn_row(const attn_job* J, int64_t out_row, int64_t bi, int hs, double* s_buf,
                     int64_t* j_buf, double* qv) {
  const int h = J->heads ? J->heads[hs] : hs;
  const int b = (int)(bi / J->N);
  const int64_t i = bi % J->N;
  const int kvh = h / (J->H / J->H_kv);
  const int rho = kvh / (J->H_kv / J->R);
  const int d = J->d;
  const uint32_t* m = J->mask + ((int64_t)b * J->R + rho) * J->N;
  const uint16_t* qi = J->q + (((int64_t)b * J->N + i) * J->H + h) * d;
  for (int t = 0; t < d; ++t) qv[t] = bf16_to_double(qi[t]);

  /* logits over the attended set */
  int64_t n = 0;
  double mx = -INFINITY;
  for (int64_t j = 0; j <= i; ++j) {
    if (!allowed(i, j, J->w, m[i], m[j])) continue;
    const uint16_t* kj = J->k + (((int64_t)b * J->N + j) * J->H_kv + kvh) * d;
    double s = 0.0;
    for (int t = 0; t < d; ++t) s += qv[t] * bf16_to_double(kj[t]);
    s *= J->scale;
    s_buf[n] = s;
    j_buf[n] = j;
    if (s > mx) mx = s;
    ++n;
  }
  /* the diagonal is always in the window, so n >= 1 */
  double sum = 0.0;
  for (int64_t a = 0; a < n; ++a) sum += exp(s_buf[a] - mx);
  const double lse = mx + log(sum);
  double* o = J->o + (out_row * J->n_heads + hs) * d;
  for (int t = 0; t < d; ++t) o[t] = 0.0;
  for (int64_t a = 0; a < n; ++a) {
    const double p = exp(s_buf[a] - lse);
    const uint16_t* vj = J->v + (((int64_t)b * J->N + j_buf[a]) * J->H_kv + kvh) * d;
    for (int t = 0; t < d; ++t) o[t] += p * bf16_to_double(vj[t]);
  }
  J->lse[out_row * J->n_heads + hs] = lse;
}

static void* attn_worker(void* arg) {
  attn_job* J = (attn_job*)arg;
  double* s_buf = (double*)malloc(sizeof(double) * (size_t)J->N);
  int64_t* j_buf = (int64_t*)malloc(sizeof(int64_t) * (size_t)J->N);
  double* qv = (double*)malloc(sizeof(double) * (size_t)J->d);
  const int64_t total = J->n_rows * J->n_heads;
  const int64_t chunk = 4;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int64_t start = J->next;
    J->next += chunk;
    pthread_mutex_unlock(&J->mu);
    if (start >= total) break;
    int64_t end = start + chunk < total ? start + chunk : total;
    for (int64_t u = start; u < end; ++u) {
      int64_t out_row = u / J->n_heads;
      int hs = (int)(u % J->n_heads);
      int64_t bi = J->rows ? J->rows[out_row] : out_row;
      attn_row(J, out_row, bi, hs, s_buf, j_buf, qv);
    }
  }
  free(s_buf); free(j_buf); free(qv);
  return NULL;
}

/*
 * Attention forward over the union set, every head, for the requested query rows.
 *   q [B, N, H, d], k/v [B, N, H_kv, d]: bf16 bit patterns
 *   mask [B, R, N] uint32 (from oracle_route or from the kernel under test)
 *   rows (nullable) flattened query rows b*N + i, n_rows of them; NULL = all B*N rows
 *   heads (nullable) query heads to compute, n_heads of them; NULL = all H heads
 *   o   [n_rows, n_heads, d] double out;  lse [n_rows, n_heads] double out (natural log)
 * Head h reads KV head h / (H / H_kv) and routing head (h / (H / H_kv)) / (H_kv / R).
 */
int oracle_attn(int B, int N, int H, int H_kv, int R, int d, int w, double scale,
                const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint32_t* mask,
                const int64_t* rows, int64_t n_rows, const int32_t* heads, int n_heads,
                double* o, double* lse, int n_threads) {
  if (B < 1 || N < 1 || H < 1 || H_kv < 1 || R < 1 || d < 1 || w < 1 || H % H_kv ||
      H_kv % R || n_rows < 0)
    return -1;
  if (!rows) n_rows = (int64_t)B * N;
  for (int64_t a = 0; rows && a < n_rows; ++a)
    if (rows[a] < 0 || rows[a] >= (int64_t)B * N) return -1;
  if (!heads) n_heads = H;
  for (int a = 0; heads && a < n_heads; ++a)
    if (heads[a] < 0 || heads[a] >= H) return -1;
  attn_job J = {B, N, H, H_kv, R, d, w, scale, q, k, v, mask, rows, n_rows, heads, n_heads,
                o, lse, 0};
  pthread_mutex_init(&J.mu, NULL);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_t th[256];
  for (int t = 0; t < n_threads; ++t) pthread_create(&th[t], NULL, attn_worker, &J);
  for (int t = 0; t < n_threads; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&J.mu);
  return 0;
}

/* ------------------------------------------------------------ backward ------ */
/*
 * Gradients of the union-softmax attention with the hard (top-k) mask held fixed.
 * With s_ij = scale q_i.k_j over j in A_i, P_ij = exp(s_ij - LSE_i),
 * O_i = sum_j P_ij v_j and an upstream gradient dO:
 *   dP_ij = dO_i . v_j,  D_i = sum_j P_ij dP_ij,  dS_ij = P_ij (dP_ij - D_i),
 *   dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,  dv_j = sum_i P_ij dO_i
 * (the chain rule through softmax; the mask is piecewise constant in r and C, so
 * the routing inputs receive no gradient).  A KV head's gradients sum over the
 * query heads that read it.
 */
typedef struct {
  int B, N, H, H_kv, R, d, w;
  double scale;
  const uint16_t *q, *k, *v, *dout;
  const uint16_t* o_for_D; /* [B, N, H, d] bf16 or NULL: D_i = dO_i . o_i instead of sum P dP */
  const uint32_t* mask;
  const int64_t* row_slot; /* [B*N]: output slot of a query row, -1 if not wanted */
  const int64_t* key_slot; /* [B*N]: output slot of a key row, -1 if not wanted */
  int64_t n_keys;
  const int32_t* heads;
  int n_heads;
  double *dq, *dk, *dv;
  double *mq, *mk, *mv; /* nullable: magnitudes of the terms (error scales) */
  double d_rel;         /* weight of D's own error in mq, mk (see oracle_attn_bwd) */
  int64_t next, total;
  pthread_mutex_t mu;
} bwd_job;

static void* bwd_worker(void* arg) {
  bwd_job* J = (bwd_job*)arg;
  const int d = J->d;
  double* s_buf = (double*)malloc(sizeof(double) * (size_t)J->N);
  double* dp_buf = (double*)malloc(sizeof(double) * (size_t)J->N);
  double* sa_buf = (double*)malloc(sizeof(double) * (size_t)J->N); /* scale sum_t |q_t k_t| */
  double* pa_buf = (double*)malloc(sizeof(double) * (size_t)J->N); /* sum_t |dO_t v_t| */
  int64_t* j_buf = (int64_t*)malloc(sizeof(int64_t) * (size_t)J->N);
  double* qv = (double*)malloc(sizeof(double) * (size_t)d);
  double* gv = (double*)malloc(sizeof(double) * (size_t)d);
  const size_t acc_n = (size_t)J->n_keys * J->H_kv * d;
  double* dk_acc = (double*)calloc(acc_n ? acc_n : 1, sizeof(double));
  double* dv_acc = (double*)calloc(acc_n ? acc_n : 1, sizeof(double));
  const size_t macc_n = J->mk ? acc_n : 0;
  double* mk_acc = (double*)calloc(macc_n ? macc_n : 1, sizeof(double));
  double* mv_acc = (double*)calloc(macc_n ? macc_n : 1, sizeof(double));

  const int64_t chunk = 8;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    const int64_t start = J->next;
    J->next += chunk;
    pthread_mutex_unlock(&J->mu);
    if (start >= J->total) break;
    const int64_t end = start + chunk < J->total ? start + chunk : J->total;
    for (int64_t u = start; u < end; ++u) {
      /* u = (hs * B + b) * N + i */
      const int64_t i = u % J->N;
      const int b = (int)((u / J->N) % J->B);
      const int hs = (int)(u / ((int64_t)J->N * J->B));
      const int h = J->heads ? J->heads[hs] : hs;
      const int kvh = h / (J->H / J->H_kv);
      const int rho = kvh / (J->H_kv / J->R);
      const uint32_t* m = J->mask + ((int64_t)b * J->R + rho) * J->N;
      const int64_t bi = (int64_t)b * J->N + i;
      const uint16_t* qi = J->q + (bi * J->H + h) * d;
      const uint16_t* gi = J->dout + (bi * J->H + h) * d;
      for (int t = 0; t < d; ++t) {
        qv[t] = bf16_to_double(qi[t]);
        gv[t] = bf16_to_double(gi[t]);
      }
      /* forward quantities of the row: logits, LSE, dP, D */
      int64_t n = 0;
      double mx = -INFINITY;
      for (int64_t j = 0; j <= i; ++j) {
        if (!allowed(i, j, J->w, m[i], m[j])) continue;
        const int64_t bj = (int64_t)b * J->N + j;
        const uint16_t* kj = J->k + (bj * J->H_kv + kvh) * d;
        const uint16_t* vj = J->v + (bj * J->H_kv + kvh) * d;
        double s = 0.0, dp = 0.0, sa = 0.0, pa = 0.0;
        for (int t = 0; t < d; ++t) {
          const double kt = bf16_to_double(kj[t]), vt = bf16_to_double(vj[t]);
          s += qv[t] * kt;
          dp += gv[t] * vt;
          sa += fabs(qv[t] * kt);
          pa += fabs(gv[t] * vt);
        }
        s_buf[n] = s * J->scale;
        dp_buf[n] = dp;
        sa_buf[n] = sa * J->scale;
        pa_buf[n] = pa;
        j_buf[n] = j;
        if (s_buf[n] > mx) mx = s_buf[n];
        ++n;
      }
      double sum = 0.0;
      for (int64_t a = 0; a < n; ++a) sum += exp(s_buf[a] - mx);
      const double lse = mx + log(sum);
      double D = 0.0;
      if (J->o_for_D) {
        const uint16_t* oi = J->o_for_D + (bi * J->H + h) * d;
        for (int t = 0; t < d; ++t) D += gv[t] * bf16_to_double(oi[t]);
      } else {
        for (int64_t a = 0; a < n; ++a) D += exp(s_buf[a] - lse) * dp_buf[a];
      }
      /* e_i = sum_j P_ij sum_t |dO_it v_jt|: scale of D's error when each O_it carries
         an error relative to the magnitude of its terms, sum_j P_ij |v_jt| */
      double e = 0.0;
      for (int64_t a = 0; a < n; ++a) e += exp(s_buf[a] - lse) * pa_buf[a];
      /* scatter into the wanted outputs */
      const int64_t rs = J->row_slot[bi];
      double* dq = rs >= 0 ? J->dq + (rs * J->n_heads + hs) * d : NULL;
      double* mq = (rs >= 0 && J->mq) ? J->mq + (rs * J->n_heads + hs) * d : NULL;
      for (int64_t a = 0; a < n; ++a) {
        const double p = exp(s_buf[a] - lse);
        const double ds = p * (dp_buf[a] - D);
        /* first-order error scale of dS: its rounding, the logit's and dP's sums, D */
        const double ads = fabs(ds) * (1.0 + J->d_rel * sa_buf[a]) + J->d_rel * p * (pa_buf[a] + e);
        const int64_t bj = (int64_t)b * J->N + j_buf[a];
        if (dq) {
          const uint16_t* kj = J->k + (bj * J->H_kv + kvh) * d;
          for (int t = 0; t < d; ++t) dq[t] += J->scale * ds * bf16_to_double(kj[t]);
          if (mq)
            for (int t = 0; t < d; ++t) mq[t] += J->scale * ads * fabs(bf16_to_double(kj[t]));
        }
        const int64_t ks = J->key_slot[bj];
        if (ks >= 0) {
          double* dk = dk_acc + (ks * J->H_kv + kvh) * d;
          double* dv = dv_acc + (ks * J->H_kv + kvh) * d;
          for (int t = 0; t < d; ++t) {
            dk[t] += J->scale * ds * qv[t];
            dv[t] += p * gv[t];
          }
          if (macc_n) {
            double* mk = mk_acc + (ks * J->H_kv + kvh) * d;
            double* mv = mv_acc + (ks * J->H_kv + kvh) * d;
            for (int t = 0; t < d; ++t) {
              mk[t] += J->scale * ads * fabs(qv[t]);
              mv[t] += p * (1.0 + J->d_rel * sa_buf[a]) * fabs(gv[t]);
            }
          }
        }
      }
    }
  }
  pthread_mutex_lock(&J->mu);
  for (size_t x = 0; x < acc_n; ++x) {
    J->dk[x] += dk_acc[x];
    J->dv[x] += dv_acc[x];
  }
  for (size_t x = 0; x < macc_n; ++x) {
    J->mk[x] += mk_acc[x];
    J->mv[x] += mv_acc[x];
  }
  pthread_mutex_unlock(&J->mu);
  free(s_buf); free(dp_buf); free(sa_buf); free(pa_buf); free(j_buf); free(qv); free(gv); free(dk_acc); free(dv_acc);
  free(mk_acc); free(mv_acc);
  return NULL;
}

/*
 * Backward of oracle_attn for the requested outputs.
 *   q [B, N, H, d], k/v [B, N, H_kv, d], dout [B, N, H, d]: bf16 bit patterns
 *   mask [B, R, N] uint32
 *   rows (nullable) flattened query rows b*N+i for dq (NULL = all B*N rows)
 *   keys (nullable) flattened key rows b*N+j for dk, dv (NULL = all B*N rows)
 *   heads (nullable) query heads whose paths are differentiated (NULL = all H)
 *   dq [n_rows, n_heads, d] double out
 *   dk, dv [n_keys, H_kv, d] double out: sums over the selected query heads
 *   o_for_D (nullable) [B, N, H, d] bf16: when given, D_i = dO_i . o_i with this
 *           (rounded) forward output, the form an implementation that receives the
 *           forward output in bf16 uses; when NULL, D_i = sum_j P_ij dP_ij exactly
 *   mq [n_rows, n_heads, d], mk, mv [n_keys, H_kv, d] (nullable, all or none):
 *           first-order error scales: with a_ij = scale sum_t |q_it k_jt| (the logit's
 *           terms), b_ij = sum_t |dO_it v_jt| (dP's terms), e_i = sum_j P_ij b_ij (D's
 *           terms, with O's) and m_ij = |dS_ij| (1 + d_rel a_ij) + d_rel P_ij (b_ij + e_i),
 *           mq_i = scale sum_j m_ij |k_j|,  mk_j = scale sum_i m_ij |q_i|,
 *           mv_j = sum_i P_ij (1 + d_rel a_ij) |dO_i|: a relative error u on dS (or P)
 *           and u d_rel on the sums that form s, dP and D moves a gradient by at most
 *           about u times its scale
 * Every query row of the selected heads is visited (each one feeds the keys).
 * Returns 0, or -1 on bad arguments.
 */
int oracle_attn_bwd(int B, int N, int H, int H_kv, int R, int d, int w, double scale,
                    const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const uint32_t* mask, const uint16_t* dout, const uint16_t* o_for_D,
                    const int64_t* rows,
                    int64_t n_rows, const int64_t* keys, int64_t n_keys, const int32_t* heads,
                    int n_heads, double* dq, double* dk, double* dv, double* mq, double* mk,
                    double* mv, double d_rel, int n_threads) {
  if (B < 1 || N < 1 || H < 1 || H_kv < 1 || R < 1 || d < 1 || w < 1 || H % H_kv ||
      H_kv % R || n_rows < 0 || n_keys < 0)
    return -1;
  const int64_t BN = (int64_t)B * N;
  if (!rows) n_rows = BN;
  if (!keys) n_keys = BN;
  if (!heads) n_heads = H;
  for (int a = 0; heads && a < n_heads; ++a)
    if (heads[a] < 0 || heads[a] >= H) return -1;
  int64_t* row_slot = (int64_t*)malloc(sizeof(int64_t) * (size_t)BN);
  int64_t* key_slot = (int64_t*)malloc(sizeof(int64_t) * (size_t)BN);
  for (int64_t x = 0; x < BN; ++x) {
    row_slot[x] = rows ? -1 : x;
    key_slot[x] = keys ? -1 : x;
  }
  int bad = 0;
  for (int64_t a = 0; rows && a < n_rows; ++a) {
    if (rows[a] < 0 || rows[a] >= BN || row_slot[rows[a]] >= 0) bad = 1;
    else row_slot[rows[a]] = a;
  }
  for (int64_t a = 0; keys && a < n_keys; ++a) {
    if (keys[a] < 0 || keys[a] >= BN || key_slot[keys[a]] >= 0) bad = 1;
    else key_slot[keys[a]] = a;
  }
  if (bad) {
    free(row_slot); free(key_slot);
    return -1;
  }
  for (int64_t x = 0; x < n_rows * n_heads * d; ++x) dq[x] = 0.0;
  for (int64_t x = 0; x < n_keys * H_kv * d; ++x) dk[x] = dv[x] = 0.0;
  if (!mq || !mk || !mv) mq = mk = mv = NULL;
  for (int64_t x = 0; mq && x < n_rows * n_heads * d; ++x) mq[x] = 0.0;
  for (int64_t x = 0; mk && x < n_keys * H_kv * d; ++x) mk[x] = mv[x] = 0.0;
  bwd_job J = {B, N, H, H_kv, R, d, w, scale, q, k, v, dout, o_for_D, mask, row_slot, key_slot, n_keys,
               heads, n_heads, dq, dk, dv, mq, mk, mv, d_rel, 0, (int64_t)n_heads * BN};
  pthread_mutex_init(&J.mu, NULL);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_t th[256];
  for (int t = 0; t < n_threads; ++t) pthread_create(&th[t], NULL, bwd_worker, &J);
  for (int t = 0; t < n_threads; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&J.mu);
  free(row_slot); free(key_slot);
  return 0;
}
