/*
 * Reference oracle for causal kernelized linear attention — TEST INFRASTRUCTURE.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library.  It shares no code, header, table or helper with the
 * CUDA library; it is a plain, slow, fp64 transcription of the method so that a
 * reader can check it against the pages by eye.
 *
 * Sources (cited by page title and equation):
 *   [ET-II]  "Efficient Transformers II" (blog-8pb.pages.dev, .../efficient2/),
 *            §2.2 Linear Attention, eq (6)–(11).
 *   [ET-I]   "Efficient Transformers I" (blog-8pb.pages.dev, .../efficient1/),
 *            kernelized attention, eq (22)–(27).
 *   [LAR]    "Linear Attention Research 2026" (guijiagi.com), sections
 *            "Performer random features" and "Linear Transformer"; the
 *            selective (input-dependent) state update of its Mamba section.
 *
 * Conventions: row vectors; q_j, k_j, v_j in R^{1×d}; φ: R^d → R^{d'}; the
 * state μ is d'×d (row i = feature i, column c = value column c), ν is d'.
 * Tensors are dense row-major [B, H, n, d] (d innermost); μ is [B, H, d', d],
 * ν is [B, H, d'].  Everything is double precision.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - elu uses α = 1, so φ(x) = x + 1 for x > 0 and e^x otherwise [LAR].
 *   - a == 1 means the plain running sums of eq (7)–(8) (weight w = 1); any
 *     other a uses eq (10)–(11) with w = 1 − a [ET-II].
 *   - The causal readout uses μ_j, ν_j, i.e. token j itself is included
 *     ([ET-II] the causal form stated after eq (9)).
 *   - No ε is added to the normalizer.
 *   - Non-causal mode is eq (6)/(9) with μ_n, ν_n and no decay.
 *   - Per-token decay: [ET-II] eq (4), z_i = a·z_{i−1} + b·s_i, with a and b
 *     indexed by the token (the input-dependent step of [LAR]'s Mamba
 *     section) and s_i = k'_iᵀv_i (resp. k'_iᵀ): μ_i = a_i μ_{i−1} + b_i k'_iᵀv_i.
 *     When b is not given, b_i = 1 − a_i (eq (10)–(11) per token), with no
 *     special case at a_i = 1: such a token is skipped, it does not restart
 *     the plain running sum.
 *
 * parity pins: every function here is pinned by the CPU tests (quadratic form
 * of [ET-I] eq (25)–(26) by brute force and in exact rationals, the a = 0
 * closed form, eq (6) as dense products, positivity and convexity, the
 * Performer expectation, ω = 0 and single-entry ω closed forms).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_FM_ELU1 = 0, OR_FM_PERFORMER = 1 };

/* φ(x) = elu(x) + 1, α = 1  ([LAR] "Linear Transformer"). */
static double phi_elu1_scalar(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

/* Performer positive random features ([LAR] "Performer random features"):
 *   φ(x)_i = exp(x·ω_i − ½‖x‖²) / √m,
 * where ω is stored d×m row-major and ω_i is its i-th column. */
static void phi_performer_vec(const double* x, int64_t d, const double* omega,
                              int64_t m, double* out) {
  double sq = 0.0;
  for (int64_t c = 0; c < d; ++c) sq += x[c] * x[c];
  const double inv_sqrt_m = 1.0 / sqrt((double)m);
  for (int64_t i = 0; i < m; ++i) {
    double u = 0.0;
    for (int64_t c = 0; c < d; ++c) u += x[c] * omega[c * m + i];
    out[i] = exp(u - 0.5 * sq) * inv_sqrt_m;
  }
}

/* φ applied to one row x ∈ R^d, result in R^{d'}. */
static void phi_row(int fm, const double* x, int64_t d, const double* omega,
                    int64_t m, double* out) {
  if (fm == OR_FM_ELU1) {
    for (int64_t c = 0; c < d; ++c) out[c] = phi_elu1_scalar(x[c]);
  } else {
    phi_performer_vec(x, d, omega, m, out);
  }
}

/* Feature dimension d' of the map: d for elu+1, m for Performer. */
static int64_t feature_dim(int fm, int64_t d, int64_t m) {
  return fm == OR_FM_ELU1 ? d : m;
}

/* Public: φ on a batch of rows, x [rows, d] → out [rows, d']. */
int oracle_features(int64_t rows, int64_t d, int fm, int64_t m,
                    const double* x, const double* omega, double* out) {
  if (fm != OR_FM_ELU1 && fm != OR_FM_PERFORMER) return 1;
  if (fm == OR_FM_PERFORMER && (omega == NULL || m <= 0)) return 1;
  const int64_t dp = feature_dim(fm, d, m);
  for (int64_t r = 0; r < rows; ++r) phi_row(fm, x + r * d, d, omega, m, out + r * dp);
  return 0;
}

/*
 * One (b, h) head of the method.
 *
 * Causal ([ET-II] eq (7)–(11) and the causal readout after eq (9)): for each
 * token j in order
 *     k' = φ(k_j);  μ ← a·μ + w·k'^T v_j;  ν ← a·ν + w·k'^T;
 *     q' = φ(q_j);  o_j = (q'·μ) / (q'·ν).
 * Non-causal ([ET-II] eq (6) read as eq (9)): run the same sums over all n
 * tokens (a = 1), then o_j = (q'_j·μ_n) / (q'_j·ν_n) for every j.
 */
static void one_head(int64_t n, int64_t d, int64_t dp, int fm, int64_t m,
                     const double* q, const double* k, const double* v,
                     double a, const double* omega, int causal,
                     double* mu, double* nu, double* out,
                     double* kf, double* qf) {
  const double w = (a == 1.0) ? 1.0 : (1.0 - a);
  for (int64_t j = 0; j < n; ++j) {
    const double* kj = k + j * d;
    const double* vj = v + j * d;
    phi_row(fm, kj, d, omega, m, kf);
    for (int64_t i = 0; i < dp; ++i) {
      for (int64_t c = 0; c < d; ++c) {
        mu[i * d + c] = a * mu[i * d + c] + w * kf[i] * vj[c];
      }
      nu[i] = a * nu[i] + w * kf[i];
    }
    if (causal) {
      phi_row(fm, q + j * d, d, omega, m, qf);
      double den = 0.0;
      for (int64_t i = 0; i < dp; ++i) den += qf[i] * nu[i];
      for (int64_t c = 0; c < d; ++c) {
        double num = 0.0;
        for (int64_t i = 0; i < dp; ++i) num += qf[i] * mu[i * d + c];
        out[j * d + c] = num / den;
      }
    }
  }
  if (!causal) {
    for (int64_t j = 0; j < n; ++j) {
      phi_row(fm, q + j * d, d, omega, m, qf);
      double den = 0.0;
      for (int64_t i = 0; i < dp; ++i) den += qf[i] * nu[i];
      for (int64_t c = 0; c < d; ++c) {
        double num = 0.0;
        for (int64_t i = 0; i < dp; ++i) num += qf[i] * mu[i * d + c];
        out[j * d + c] = num / den;
      }
    }
  }
}

/*
 * Forward over B·H independent heads.
 *   q, k, v   [B,H,n,d]
 *   a         [H] per-head decay, or NULL for a = 1 (eq (7)–(8))
 *   omega     [d,m] for Performer, else NULL
 *   mu0, nu0  initial state [B,H,d',d], [B,H,d'], or NULL for zero
 *   out       [B,H,n,d]
 *   mu_out, nu_out  final state, or NULL
 * Returns 0 on success, 1 on invalid arguments (non-causal with a decay,
 * unknown feature map, missing ω, or a decay outside [0, 1]).
 * Heads run in parallel with OpenMP when the library is built with it.
 */
int oracle_forward(int64_t B, int64_t H, int64_t n, int64_t d, int fm, int64_t m,
                   const double* q, const double* k, const double* v,
                   const double* a, const double* omega, int causal,
                   const double* mu0, const double* nu0,
                   double* out, double* mu_out, double* nu_out) {
  if (fm != OR_FM_ELU1 && fm != OR_FM_PERFORMER) return 1;
  if (fm == OR_FM_PERFORMER && (omega == NULL || m <= 0)) return 1;
  if (!causal && a != NULL) return 1;
  if (a != NULL) {
    for (int64_t h = 0; h < H; ++h) {
      if (!(a[h] >= 0.0 && a[h] <= 1.0)) return 1;
    }
  }
  const int64_t dp = feature_dim(fm, d, m);
  int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < B * H; ++bh) {
    const int64_t h = bh % H;
    double* mu = (double*)malloc((size_t)(dp * d) * sizeof(double));
    double* nu = (double*)malloc((size_t)dp * sizeof(double));
    double* kf = (double*)malloc((size_t)dp * sizeof(double));
    double* qf = (double*)malloc((size_t)dp * sizeof(double));
    if (!mu || !nu || !kf || !qf) {
      failed = 1;
    } else {
      if (mu0) memcpy(mu, mu0 + bh * dp * d, (size_t)(dp * d) * sizeof(double));
      else memset(mu, 0, (size_t)(dp * d) * sizeof(double));
      if (nu0) memcpy(nu, nu0 + bh * dp, (size_t)dp * sizeof(double));
      else memset(nu, 0, (size_t)dp * sizeof(double));
      const double ah = a ? a[h] : 1.0;
      one_head(n, d, dp, fm, m, q + bh * n * d, k + bh * n * d, v + bh * n * d,
               ah, omega, causal, mu, nu, out + bh * n * d, kf, qf);
      if (mu_out) memcpy(mu_out + bh * dp * d, mu, (size_t)(dp * d) * sizeof(double));
      if (nu_out) memcpy(nu_out + bh * dp, nu, (size_t)dp * sizeof(double));
    }
    free(mu);
    free(nu);
    free(kf);
    free(qf);
  }
  return failed ? 2 : 0;
}

/*
 * One recurrent decode step ([ET-II] eq (10)–(11), then the causal readout):
 * the state (μ, ν) of every head is advanced in place by one token with the
 * elu+1 map and the head's decay, and o = q'μ / q'ν is written.
 *   mu [B,H,d,d], nu [B,H,d], q/k/v/out [B,H,d], a [H] or NULL.
 */
int oracle_decode_step(int64_t B, int64_t H, int64_t d, double* mu, double* nu,
                       const double* q, const double* k, const double* v,
                       const double* a, double* out) {
  return oracle_forward(B, H, 1, d, OR_FM_ELU1, 0, q, k, v, a, NULL, 1, mu, nu,
                        out, mu, nu);
}

/*
 * The same step with either feature map: fm = OR_FM_ELU1 (d' = d, omega
 * NULL) or OR_FM_PERFORMER (d' = m, omega [d, m], φ of [LAR] "Performer
 * random features").  mu [B,H,d',d], nu [B,H,d'] are advanced in place.
 */
int oracle_decode_step_fm(int64_t B, int64_t H, int64_t d, int fm, int64_t m, double* mu,
                          double* nu, const double* q, const double* k, const double* v,
                          const double* a, const double* omega, double* out) {
  return oracle_forward(B, H, 1, d, fm, m, q, k, v, a, omega, 1, mu, nu, out, mu, nu);
}

/*
 * One head with a per-token decay a_i and input weight b_i ([ET-II] eq (4)
 * with a, b indexed by the token; the readout after eq (9)):
 *     k' = φ(k_i);  μ ← a_i·μ + b_i·k'^T v_i;  ν ← a_i·ν + b_i·k'^T;
 *     q' = φ(q_i);  o_i = (q'·μ) / (q'·ν).
 * a, b point at this head's n values; b == NULL means b_i = 1 − a_i.
 */
static void one_head_token(int64_t n, int64_t d, int64_t dp, int fm, int64_t m,
                           const double* q, const double* k, const double* v,
                           const double* a, const double* b, const double* omega,
                           double* mu, double* nu, double* out, double* kf, double* qf) {
  for (int64_t j = 0; j < n; ++j) {
    const double aj = a[j];
    const double bj = b ? b[j] : 1.0 - aj;
    phi_row(fm, k + j * d, d, omega, m, kf);
    for (int64_t i = 0; i < dp; ++i) {
      for (int64_t c = 0; c < d; ++c) {
        mu[i * d + c] = aj * mu[i * d + c] + bj * kf[i] * v[j * d + c];
      }
      nu[i] = aj * nu[i] + bj * kf[i];
    }
    phi_row(fm, q + j * d, d, omega, m, qf);
    double den = 0.0;
    for (int64_t i = 0; i < dp; ++i) den += qf[i] * nu[i];
    for (int64_t c = 0; c < d; ++c) {
      double num = 0.0;
      for (int64_t i = 0; i < dp; ++i) num += qf[i] * mu[i * d + c];
      out[j * d + c] = num / den;
    }
  }
}

/*
 * Causal forward with a per-token decay over B·H independent heads.
 *   q, k, v   [B,H,n,d]
 *   a         [B,H,n] decays a_i ∈ [0, 1]
 *   b         [B,H,n] input weights b_i ≥ 0, or NULL for b_i = 1 − a_i
 *   omega     [d,m] for Performer, else NULL
 *   mu0, nu0  initial state [B,H,d',d], [B,H,d'], or NULL for zero
 *   out       [B,H,n,d];  mu_out, nu_out  final state, or NULL
 * Returns 0 on success, 1 on invalid arguments (unknown feature map, missing
 * ω, a missing a, a decay outside [0, 1] or a negative or non-finite weight).
 */
int oracle_forward_token_decay(int64_t B, int64_t H, int64_t n, int64_t d, int fm, int64_t m,
                               const double* q, const double* k, const double* v,
                               const double* a, const double* b, const double* omega,
                               const double* mu0, const double* nu0,
                               double* out, double* mu_out, double* nu_out) {
  if (fm != OR_FM_ELU1 && fm != OR_FM_PERFORMER) return 1;
  if (fm == OR_FM_PERFORMER && (omega == NULL || m <= 0)) return 1;
  if (a == NULL) return 1;
  for (int64_t i = 0; i < B * H * n; ++i) {
    if (!(a[i] >= 0.0 && a[i] <= 1.0)) return 1;
    if (b && !(b[i] >= 0.0 && isfinite(b[i]))) return 1;
  }
  const int64_t dp = feature_dim(fm, d, m);
  int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < B * H; ++bh) {
    double* mu = (double*)malloc((size_t)(dp * d) * sizeof(double));
    double* nu = (double*)malloc((size_t)dp * sizeof(double));
    double* kf = (double*)malloc((size_t)dp * sizeof(double));
    double* qf = (double*)malloc((size_t)dp * sizeof(double));
    if (!mu || !nu || !kf || !qf) {
      failed = 1;
    } else {
      if (mu0) memcpy(mu, mu0 + bh * dp * d, (size_t)(dp * d) * sizeof(double));
      else memset(mu, 0, (size_t)(dp * d) * sizeof(double));
      if (nu0) memcpy(nu, nu0 + bh * dp, (size_t)dp * sizeof(double));
      else memset(nu, 0, (size_t)dp * sizeof(double));
      one_head_token(n, d, dp, fm, m, q + bh * n * d, k + bh * n * d, v + bh * n * d,
                     a + bh * n, b ? b + bh * n : NULL, omega, mu, nu, out + bh * n * d,
                     kf, qf);
      if (mu_out) memcpy(mu_out + bh * dp * d, mu, (size_t)(dp * d) * sizeof(double));
      if (nu_out) memcpy(nu_out + bh * dp, nu, (size_t)dp * sizeof(double));
    }
    free(mu);
    free(nu);
    free(kf);
    free(qf);
  }
  return failed ? 2 : 0;
}

/* dφ for one row: given x ∈ R^d, φ(x) ∈ R^{d'} (already computed) and the
 * gradient gf ∈ R^{d'} with respect to φ(x), writes the gradient gx ∈ R^d
 * with respect to x:
 *   elu+1:      ∂φ_c/∂x_c = 1 for x_c > 0, e^{x_c} otherwise (d' = d);
 *   Performer:  ∂φ_i/∂x = φ_i·(ω_i − x), so gx = Σ_i gf_i φ_i (ω_i − x). */
static void phi_row_grad(int fm, const double* x, int64_t d, const double* omega, int64_t m,
                         const double* f, const double* gf, double* gx) {
  if (fm == OR_FM_ELU1) {
    for (int64_t c = 0; c < d; ++c) gx[c] = gf[c] * (x[c] > 0.0 ? 1.0 : exp(x[c]));
  } else {
    double tot = 0.0;
    for (int64_t i = 0; i < m; ++i) tot += gf[i] * f[i];
    for (int64_t c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int64_t i = 0; i < m; ++i) acc += gf[i] * f[i] * omega[c * m + i];
      gx[c] = acc - tot * x[c];
    }
  }
}

/*
 * Reverse-mode gradient of L = Σ_j g_j·o_j for one causal head of the
 * recurrence in one_head ([ET-II] eq (7)–(11) with the readout after eq (9)).
 * With ĝ_j = g_j / den_j and ρ_j = −(g_j·o_j) / den_j (o_j = num_j / den_j),
 * the adjoints of μ_j, ν_j obey M_j = q'_jᵀĝ_j + a·M_{j+1}, N_j = ρ_j q'_j +
 * a·N_{j+1}, and
 *   ∂q'_j = ĝ_j μ_jᵀ + ρ_j ν_j,   ∂k'_j = w (M_j v_jᵀ + N_j),   ∂v_j = w k'_j M_j,
 *   ∂a    = Σ_j ⟨M_j, μ_{j−1} + w'·k'_jᵀv_j⟩ + ⟨N_j, ν_{j−1} + w'·k'_j⟩,
 * w' = dw/da = −1 (0 when a = 1, where w = 1); then ∂q, ∂k by the chain
 * rule through φ.  The states μ_j, ν_j are recomputed block by block from
 * checkpoints taken every `blk` tokens in a first forward sweep.
 */
static int one_head_backward(int64_t n, int64_t d, int64_t dp, int fm, int64_t m,
                             const double* q, const double* k, const double* v, const double* g,
                             double a, const double* omega, double* dq, double* dk, double* dv,
                             double* da_out) {
  const int64_t blk = 64;
  const int64_t nblk = (n + blk - 1) / blk;
  const double w = (a == 1.0) ? 1.0 : (1.0 - a);
  const double wprime = (a == 1.0) ? 0.0 : -1.0;
  const size_t sd = (size_t)(dp * d);
  double* ck_mu = (double*)calloc((size_t)(nblk > 0 ? nblk : 1) * sd, sizeof(double));
  double* ck_nu = (double*)calloc((size_t)(nblk > 0 ? nblk : 1) * (size_t)dp, sizeof(double));
  double* mu = (double*)calloc((size_t)(blk + 1) * sd, sizeof(double));    /* μ_{j−1}, μ_j, … of a block */
  double* nu = (double*)calloc((size_t)(blk + 1) * (size_t)dp, sizeof(double));
  double* kf = (double*)malloc((size_t)(blk * dp) * sizeof(double));
  double* qf = (double*)malloc((size_t)(blk * dp) * sizeof(double));
  double* M = (double*)calloc(sd, sizeof(double));
  double* N = (double*)calloc((size_t)dp, sizeof(double));
  double* gq = (double*)malloc((size_t)dp * sizeof(double));
  double* gk = (double*)malloc((size_t)dp * sizeof(double));
  if (!ck_mu || !ck_nu || !mu || !nu || !kf || !qf || !M || !N || !gq || !gk) {
    free(ck_mu); free(ck_nu); free(mu); free(nu); free(kf); free(qf); free(M); free(N);
    free(gq); free(gk);
    return 2;
  }
  /* forward sweep: checkpoint the state entering every block */
  {
    double* cmu = mu;   /* running state */
    double* cnu = nu;
    for (int64_t j = 0; j < n; ++j) {
      if (j % blk == 0) {
        memcpy(ck_mu + (j / blk) * sd, cmu, sd * sizeof(double));
        memcpy(ck_nu + (j / blk) * dp, cnu, (size_t)dp * sizeof(double));
      }
      phi_row(fm, k + j * d, d, omega, m, kf);
      for (int64_t i = 0; i < dp; ++i) {
        for (int64_t c = 0; c < d; ++c) cmu[i * d + c] = a * cmu[i * d + c] + w * kf[i] * v[j * d + c];
        cnu[i] = a * cnu[i] + w * kf[i];
      }
    }
  }
  double da = 0.0;
  for (int64_t b = nblk - 1; b >= 0; --b) {
    const int64_t j0 = b * blk;
    const int64_t len = (n - j0 < blk) ? n - j0 : blk;
    /* recompute the block: mu[r] = μ_{j0+r−1} (r = 0 … len) */
    memcpy(mu, ck_mu + b * sd, sd * sizeof(double));
    memcpy(nu, ck_nu + b * dp, (size_t)dp * sizeof(double));
    for (int64_t r = 0; r < len; ++r) {
      const int64_t j = j0 + r;
      phi_row(fm, k + j * d, d, omega, m, kf + r * dp);
      phi_row(fm, q + j * d, d, omega, m, qf + r * dp);
      const double* pm = mu + r * sd;
      double* nm = mu + (r + 1) * sd;
      for (int64_t i = 0; i < dp; ++i) {
        for (int64_t c = 0; c < d; ++c)
          nm[i * d + c] = a * pm[i * d + c] + w * kf[r * dp + i] * v[j * d + c];
        nu[(r + 1) * dp + i] = a * nu[r * dp + i] + w * kf[r * dp + i];
      }
    }
    for (int64_t r = len - 1; r >= 0; --r) {
      const int64_t j = j0 + r;
      const double* muj = mu + (r + 1) * sd;     /* μ_j */
      const double* nuj = nu + (r + 1) * dp;
      const double* mup = mu + r * sd;           /* μ_{j−1} */
      const double* nup = nu + r * dp;
      const double* qj = qf + r * dp;
      const double* kj = kf + r * dp;
      const double* vj = v + j * d;
      const double* gj = g + j * d;
      /* readout of token j */
      double den = 0.0;
      for (int64_t i = 0; i < dp; ++i) den += qj[i] * nuj[i];
      double go = 0.0;
      for (int64_t c = 0; c < d; ++c) {
        double num = 0.0;
        for (int64_t i = 0; i < dp; ++i) num += qj[i] * muj[i * d + c];
        go += gj[c] * (num / den);
      }
      const double rho = -go / den;
      /* adjoints M_j = q'ᵀĝ + a·M_{j+1}, N_j = ρ q' + a·N_{j+1} */
      for (int64_t i = 0; i < dp; ++i) {
        for (int64_t c = 0; c < d; ++c) M[i * d + c] = a * M[i * d + c] + qj[i] * (gj[c] / den);
        N[i] = a * N[i] + rho * qj[i];
      }
      /* ∂q'_j = ĝ μ_jᵀ + ρ ν_j */
      for (int64_t i = 0; i < dp; ++i) {
        double acc = rho * nuj[i];
        for (int64_t c = 0; c < d; ++c) acc += (gj[c] / den) * muj[i * d + c];
        gq[i] = acc;
      }
      /* ∂k'_j = w (M v_j + N),  ∂v_j = w k'_j M */
      for (int64_t i = 0; i < dp; ++i) {
        double acc = N[i];
        for (int64_t c = 0; c < d; ++c) acc += M[i * d + c] * vj[c];
        gk[i] = w * acc;
      }
      for (int64_t c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int64_t i = 0; i < dp; ++i) acc += kj[i] * M[i * d + c];
        dv[j * d + c] = w * acc;
      }
      /* ∂a: μ_j = a μ_{j−1} + w(a) k'ᵀv */
      for (int64_t i = 0; i < dp; ++i) {
        for (int64_t c = 0; c < d; ++c)
          da += M[i * d + c] * (mup[i * d + c] + wprime * kj[i] * vj[c]);
        da += N[i] * (nup[i] + wprime * kj[i]);
      }
      phi_row_grad(fm, q + j * d, d, omega, m, qj, gq, dq + j * d);
      phi_row_grad(fm, k + j * d, d, omega, m, kj, gk, dk + j * d);
    }
  }
  *da_out = da;
  free(ck_mu); free(ck_nu); free(mu); free(nu); free(kf); free(qf); free(M); free(N);
  free(gq); free(gk);
  return 0;
}

/*
 * Backward of the causal forward over B·H heads: the gradients of
 * L = Σ g·o with respect to q, k, v [B,H,n,d] and to the per-head decay
 * a [H] (summed over the batch; da may be NULL, and is written only when a
 * is given).  g [B,H,n,d].  Returns 0, 1 on invalid arguments, 2 when out
 * of memory.
 */
int oracle_backward(int64_t B, int64_t H, int64_t n, int64_t d, int fm, int64_t m,
                    const double* q, const double* k, const double* v, const double* a,
                    const double* omega, const double* g, double* dq, double* dk, double* dv,
                    double* da) {
  if (fm != OR_FM_ELU1 && fm != OR_FM_PERFORMER) return 1;
  if (fm == OR_FM_PERFORMER && (omega == NULL || m <= 0)) return 1;
  if (a != NULL) {
    for (int64_t h = 0; h < H; ++h) {
      if (!(a[h] >= 0.0 && a[h] <= 1.0)) return 1;
    }
  }
  const int64_t dp = feature_dim(fm, d, m);
  double* da_bh = (double*)calloc((size_t)(B * H > 0 ? B * H : 1), sizeof(double));
  if (!da_bh) return 2;
  int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < B * H; ++bh) {
    const double ah = a ? a[bh % H] : 1.0;
    if (one_head_backward(n, d, dp, fm, m, q + bh * n * d, k + bh * n * d, v + bh * n * d,
                          g + bh * n * d, ah, omega, dq + bh * n * d, dk + bh * n * d,
                          dv + bh * n * d, da_bh + bh) != 0)
      failed = 1;
  }
  if (da && a) {
    for (int64_t h = 0; h < H; ++h) da[h] = 0.0;
    for (int64_t bh = 0; bh < B * H; ++bh) da[bh % H] += da_bh[bh];
  }
  free(da_bh);
  return failed ? 2 : 0;
}
