/*
 * lapl_oracle.c -- plain fp64 CPU oracle for Laplacian-kernel Nystrom attention.
 *
 * TEST INFRASTRUCTURE ONLY (see lapl_oracle.h).  Slow on purpose: plain loops in the order of
 * the method's steps, no blocking, fusion or reordering, so that each step can be checked
 * against its description by eye.  Build with -ffp-contract=off so that x86 and Arm hosts
 * round identically.
 *
 * Source of each step: "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel",
 * the explainer pages (English, German, Chinese, Korean and Japanese editions).  Where the
 * pages leave a detail open, the reading used is stated beside the code.
 */
#include "lapl_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- step 1: landmarks ---------------------------------------------------------------
 * English page, 2.C.1 (Nystrom Approximation): landmark keys are selected by average pooling.
 * Reading: 2-D average pooling over the grid_h x grid_w token grid with non-overlapping
 * windows of (grid_h/s) x (grid_w/s) tokens, s = sqrt(m); landmark j = jr*s + jc covers token
 * rows jr*ph .. jr*ph+ph-1 and columns jc*pw .. jc*pw+pw-1; token n = r*grid_w + c.
 * The window is summed in index order (rows, then columns) and divided by ph*pw.
 */
static void landmarks_avgpool(const double* K, int grid_w, int d, int s, int ph, int pw,
                              double* L) {
  for (int jr = 0; jr < s; ++jr) {
    for (int jc = 0; jc < s; ++jc) {
      const int j = jr * s + jc;
      for (int c = 0; c < d; ++c) {
        double sum = 0.0;
        for (int r = jr * ph; r < (jr + 1) * ph; ++r)
          for (int cc = jc * pw; cc < (jc + 1) * pw; ++cc)
            sum += K[(size_t)(r * grid_w + cc) * d + c];
        L[(size_t)j * d + c] = sum / (double)(ph * pw);
      }
    }
  }
}

/* ---- step 2: Laplacian kernel ---------------------------------------------------------
 * English page, 2.A; German page, 2 (Laplacian-Kernel als Ahnlichkeitsmass):
 * k(x,y) = exp(-||x - y||_1 / lambda), with the L1 (Manhattan) distance summed over the
 * d channels in ascending order.
 */
static double l1_distance(const double* x, const double* y, int d) {
  double sum = 0.0;
  for (int c = 0; c < d; ++c) sum += fabs(x[c] - y[c]);
  return sum;
}

/* The Gaussian kernel the pages compare against (English page, 1 "Theoretical Mismatch":
 * similarity decaying with the squared l2 distance): k(x,y) = exp(-||x - y||_2^2 / lambda),
 * the squared differences summed over the d channels in ascending order. */
static double sq_l2_distance(const double* x, const double* y, int d) {
  double sum = 0.0;
  for (int c = 0; c < d; ++c) sum += (x[c] - y[c]) * (x[c] - y[c]);
  return sum;
}

static double kernel_distance(const orc_config* cfg, const double* x, const double* y, int d) {
  return cfg->kernel == 1 ? sq_l2_distance(x, y, d) : l1_distance(x, y, d);
}

/* exp(-distance / lambda), for either distance. */
static double laplacian_of_distance(double dist, double lambda) { return exp(-dist / lambda); }

/* ---- step 3: Newton-Schulz inverse of W ---------------------------------------------
 * English page, 2.C.2; German page, 2 (Newton-Schulz Iteration fur Inversion); Korean page,
 * 2.3: the landmark kernel matrix is inverted with the multiply-only Newton-Schulz iteration
 * X <- X (2I - W X); a small eps*I keeps W strictly positive definite.
 * Reading: X0 = W^T / (|W|_1 |W|_inf) with |W|_1 the largest absolute column sum and
 * |W|_inf the largest absolute row sum, both of W after eps*I is added; exactly T steps,
 * no early exit; T = 0 returns X0.  Each step forms P = W X, then Z = 2I - P, then X Z.
 */
static double frob_residual(const double* W, const double* X, int m) {
  double acc = 0.0;
  for (int i = 0; i < m; ++i)
    for (int j = 0; j < m; ++j) {
      double wx = 0.0;
      for (int k = 0; k < m; ++k) wx += W[(size_t)i * m + k] * X[(size_t)k * m + j];
      const double r = (i == j ? 1.0 : 0.0) - wx;
      acc += r * r;
    }
  return sqrt(acc);
}

static int newton_schulz(const double* W, int m, int T, double* X, double* resid) {
  double n1 = 0.0, ninf = 0.0;
  for (int j = 0; j < m; ++j) { /* |W|_1: largest absolute column sum */
    double s = 0.0;
    for (int i = 0; i < m; ++i) s += fabs(W[(size_t)i * m + j]);
    if (s > n1) n1 = s;
  }
  for (int i = 0; i < m; ++i) { /* |W|_inf: largest absolute row sum */
    double s = 0.0;
    for (int j = 0; j < m; ++j) s += fabs(W[(size_t)i * m + j]);
    if (s > ninf) ninf = s;
  }
  const double scale = n1 * ninf;
  for (int i = 0; i < m; ++i)
    for (int j = 0; j < m; ++j) X[(size_t)i * m + j] = W[(size_t)j * m + i] / scale;
  if (resid) resid[0] = frob_residual(W, X, m);

  double* P = (double*)malloc(sizeof(double) * (size_t)m * m);
  double* Z = (double*)malloc(sizeof(double) * (size_t)m * m);
  double* Xn = (double*)malloc(sizeof(double) * (size_t)m * m);
  if (!P || !Z || !Xn) {
    free(P); free(Z); free(Xn);
    return ORC_ERR_NOMEM;
  }
  for (int t = 1; t <= T; ++t) {
    for (int i = 0; i < m; ++i) /* P = W X */
      for (int j = 0; j < m; ++j) {
        double s = 0.0;
        for (int k = 0; k < m; ++k) s += W[(size_t)i * m + k] * X[(size_t)k * m + j];
        P[(size_t)i * m + j] = s;
      }
    for (int i = 0; i < m; ++i) /* Z = 2I - P */
      for (int j = 0; j < m; ++j)
        Z[(size_t)i * m + j] = (i == j ? 2.0 : 0.0) - P[(size_t)i * m + j];
    for (int i = 0; i < m; ++i) /* X <- X Z */
      for (int j = 0; j < m; ++j) {
        double s = 0.0;
        for (int k = 0; k < m; ++k) s += X[(size_t)i * m + k] * Z[(size_t)k * m + j];
        Xn[(size_t)i * m + j] = s;
      }
    memcpy(X, Xn, sizeof(double) * (size_t)m * m);
    if (resid) resid[t] = frob_residual(W, X, m);
  }
  free(P); free(Z); free(Xn);
  return ORC_OK;
}

/* ---- step 3, alternative: conjugate-gradient solve of W M = B V (solver = 1) -----------
 * German page, 4 (Ablationsstudien), English page, 4 ("Solver Robustness") and Chinese page,
 * 4 (ablation): the pages compare the Newton-Schulz iteration with a conjugate-gradient (CG)
 * solver and report CG as less accurate and less stable on ill-conditioned matrices; they
 * give no details of the CG variant.
 * Reading: the classical (Hestenes-Stiefel) CG method for the symmetric positive definite W,
 * applied to W y = b for each column b of B V separately, from y0 = 0 (so r0 = p0 = b), with
 * the residual updated recursively; exactly T iterations, the same count T as the
 * Newton-Schulz steps.  Iteration t: q = W p; alpha = (r.r) / (p.q); y += alpha p;
 * r -= alpha q; beta = (r.r)_new / (r.r)_old; p = r + beta p.  A column stops early only
 * where no further step is defined: r.r == 0 (solved exactly) or p.q <= 0.  M gathers the
 * columns y.  resid[t] = sqrt(sum over columns of r.r after t iterations) / ||B V||_F
 * (0 when B V = 0).
 */
static int conjugate_gradient(const double* W, const double* BV, int m, int d, int T, double* M,
                              double* resid) {
  double* y = (double*)malloc(sizeof(double) * (size_t)m);
  double* r = (double*)malloc(sizeof(double) * (size_t)m);
  double* p = (double*)malloc(sizeof(double) * (size_t)m);
  double* q = (double*)malloc(sizeof(double) * (size_t)m);
  double* rr_hist = (double*)calloc((size_t)(T + 1), sizeof(double));
  if (!y || !r || !p || !q || !rr_hist) {
    free(y); free(r); free(p); free(q); free(rr_hist);
    return ORC_ERR_NOMEM;
  }
  for (int j = 0; j < d; ++j) {
    double rr = 0.0;
    for (int i = 0; i < m; ++i) {
      y[i] = 0.0;
      r[i] = BV[(size_t)i * d + j];
      p[i] = r[i];
      rr += r[i] * r[i];
    }
    rr_hist[0] += rr;
    int stopped = rr == 0.0;
    for (int t = 1; t <= T; ++t) {
      if (!stopped) {
        double pq = 0.0;
        for (int i = 0; i < m; ++i) {
          double acc = 0.0;
          for (int k = 0; k < m; ++k) acc += W[(size_t)i * m + k] * p[k];
          q[i] = acc;
          pq += p[i] * q[i];
        }
        if (!(pq > 0.0)) {
          stopped = 1;
        } else {
          const double alpha = rr / pq;
          double rr_new = 0.0;
          for (int i = 0; i < m; ++i) {
            y[i] += alpha * p[i];
            r[i] -= alpha * q[i];
            rr_new += r[i] * r[i];
          }
          const double beta = rr_new / rr;
          for (int i = 0; i < m; ++i) p[i] = r[i] + beta * p[i];
          rr = rr_new;
          if (rr == 0.0) stopped = 1;
        }
      }
      rr_hist[t] += rr;
    }
    for (int i = 0; i < m; ++i) M[(size_t)i * d + j] = y[i];
  }
  if (resid)
    for (int t = 0; t <= T; ++t)
      resid[t] = rr_hist[0] > 0.0 ? sqrt(rr_hist[t]) / sqrt(rr_hist[0]) : 0.0;
  free(y); free(r); free(p); free(q); free(rr_hist);
  return ORC_OK;
}

/* ---- step 4: whitening (injective feature map) ----------------------------------------
 * Korean page, 2.2: z_i = Sigma^{-1/2} (k(q_i, .) - mean) + bias, with Sigma replaced by a
 * diagonal estimator of the empirical variance (English page, 2.B; Japanese page, 2.2).
 * Reading: the similarity vector of query i is row i of A (over the m landmarks); mean and
 * variance are taken per landmark column over the N tokens of the (b,h) slice; the variance
 * divides by N; delta sits inside the square root; bias has shape [H,m] (zeros when absent).
 * Mean and variance are computed in two passes.
 */
static void whiten_columns(const double* A, int N, int m, double delta, const double* beta,
                           double* mu, double* var, double* Ahat) {
  for (int j = 0; j < m; ++j) {
    double s = 0.0;
    for (int i = 0; i < N; ++i) s += A[(size_t)i * m + j];
    const double mean = s / (double)N;
    double ss = 0.0;
    for (int i = 0; i < N; ++i) {
      const double dv = A[(size_t)i * m + j] - mean;
      ss += dv * dv;
    }
    const double variance = ss / (double)N;
    const double scale = 1.0 / sqrt(variance + delta);
    const double b = beta ? beta[j] : 0.0;
    for (int i = 0; i < N; ++i) Ahat[(size_t)i * m + j] = (A[(size_t)i * m + j] - mean) * scale + b;
    mu[j] = mean;
    var[j] = variance;
  }
}

/* ---- step 5: output chain --------------------------------------------------------------
 * Chinese page, 2.2: the N x N kernel matrix is approximated in low-rank form from the
 * landmark blocks without forming it explicitly.  Reading: O = A_hat (X (B V)), evaluated
 * right to left: BV = B V (m x d), M = X BV (m x d), O = A_hat M (N x d).
 */
static void matmul(const double* Aop, const double* Bop, int rows, int inner, int cols,
                   double* C) {
  for (int i = 0; i < rows; ++i)
    for (int j = 0; j < cols; ++j) {
      double s = 0.0;
      for (int k = 0; k < inner; ++k) s += Aop[(size_t)i * inner + k] * Bop[(size_t)k * cols + j];
      C[(size_t)i * cols + j] = s;
    }
}

static int isqrt_exact(int m) {
  for (int s = 1; s * s <= m; ++s)
    if (s * s == m) return s;
  return -1;
}

static int check_config(const orc_config* c) {
  if (!c) return ORC_ERR_ARG;
  if (c->batch < 0 || c->heads < 1 || c->grid_h < 1 || c->grid_w < 1 || c->head_dim < 1 ||
      c->num_landmarks < 1 || c->ns_steps < 0)
    return ORC_ERR_ARG;
  if (!(c->lambda > 0.0) || !(c->eps >= 0.0)) return ORC_ERR_ARG;
  if (c->whiten && !(c->delta > 0.0)) return ORC_ERR_ARG;
  if (c->kernel != 0 && c->kernel != 1) return ORC_ERR_ARG;
  if (c->solver != 0 && c->solver != 1) return ORC_ERR_ARG;
  const int s = isqrt_exact(c->num_landmarks);
  if (s < 0 || c->grid_h % s != 0 || c->grid_w % s != 0) return ORC_ERR_UNSUPPORTED;
  return ORC_OK;
}

/* One (b,h) slice.  Offsets into the intermediates are taken by the caller. */
static int forward_slice(const orc_config* cfg, int h, const double* Q, const double* K,
                         const double* V, const double* bias, double* O,
                         const orc_intermediates* im, long slice) {
  const int N = cfg->grid_h * cfg->grid_w, d = cfg->head_dim, m = cfg->num_landmarks;
  const int s = isqrt_exact(m), ph = cfg->grid_h / s, pw = cfg->grid_w / s;
  const int T = cfg->ns_steps;
  const size_t nm = (size_t)N * m, mm = (size_t)m * m, md = (size_t)m * d;

  double* L = (double*)malloc(sizeof(double) * md);
  double* Dql = (double*)malloc(sizeof(double) * nm);
  double* Dll = (double*)malloc(sizeof(double) * mm);
  double* Dlk = (double*)malloc(sizeof(double) * nm);
  double* A = (double*)malloc(sizeof(double) * nm);
  double* Bm = (double*)malloc(sizeof(double) * nm);
  double* W = (double*)malloc(sizeof(double) * mm);
  double* X = (double*)malloc(sizeof(double) * mm);
  double* mu = (double*)malloc(sizeof(double) * m);
  double* var = (double*)malloc(sizeof(double) * m);
  double* Ahat = (double*)malloc(sizeof(double) * nm);
  double* BV = (double*)malloc(sizeof(double) * md);
  double* M = (double*)malloc(sizeof(double) * md);
  double* resid = (double*)malloc(sizeof(double) * (size_t)(T + 1));
  int rc = ORC_OK;
  if (!L || !Dql || !Dll || !Dlk || !A || !Bm || !W || !X || !mu || !var || !Ahat || !BV || !M ||
      !resid) {
    rc = ORC_ERR_NOMEM;
    goto done;
  }

  /* 1. landmarks */
  landmarks_avgpool(K, cfg->grid_w, d, s, ph, pw, L);

  /* 2. kernel blocks: A = k(Q,L) [N,m], B = k(L,K) [m,N], W = k(L,L) + eps I [m,m] */
  for (int i = 0; i < N; ++i)
    for (int j = 0; j < m; ++j) {
      Dql[(size_t)i * m + j] = kernel_distance(cfg, Q + (size_t)i * d, L + (size_t)j * d, d);
      A[(size_t)i * m + j] = laplacian_of_distance(Dql[(size_t)i * m + j], cfg->lambda);
    }
  for (int j = 0; j < m; ++j)
    for (int n = 0; n < N; ++n) {
      Dlk[(size_t)j * N + n] = kernel_distance(cfg, L + (size_t)j * d, K + (size_t)n * d, d);
      Bm[(size_t)j * N + n] = laplacian_of_distance(Dlk[(size_t)j * N + n], cfg->lambda);
    }
  for (int j = 0; j < m; ++j)
    for (int k = 0; k < m; ++k) {
      Dll[(size_t)j * m + k] = kernel_distance(cfg, L + (size_t)j * d, L + (size_t)k * d, d);
      W[(size_t)j * m + k] = laplacian_of_distance(Dll[(size_t)j * m + k], cfg->lambda) +
                             (j == k ? cfg->eps : 0.0);
    }

  /* 3. Newton-Schulz (solver 0); with the CG solver (1) X is not formed and stays zero */
  if (cfg->solver == 0) {
    rc = newton_schulz(W, m, T, X, resid);
    if (rc != ORC_OK) goto done;
  } else {
    memset(X, 0, sizeof(double) * mm);
  }

  /* 4. whitening */
  if (cfg->whiten) {
    whiten_columns(A, N, m, cfg->delta, bias ? bias + (size_t)h * m : NULL, mu, var, Ahat);
  } else {
    memcpy(Ahat, A, sizeof(double) * nm);
    for (int j = 0; j < m; ++j) { /* statistics are still reported when whitening is off */
      double sacc = 0.0;
      for (int i = 0; i < N; ++i) sacc += A[(size_t)i * m + j];
      mu[j] = sacc / (double)N;
      double ss = 0.0;
      for (int i = 0; i < N; ++i) {
        const double dv = A[(size_t)i * m + j] - mu[j];
        ss += dv * dv;
      }
      var[j] = ss / (double)N;
    }
  }

  /* 5. output chain, right to left: M = X (B V), or the CG solution of W M = B V */
  matmul(Bm, V, m, N, d, BV);
  if (cfg->solver == 0) {
    matmul(X, BV, m, m, d, M);
  } else {
    rc = conjugate_gradient(W, BV, m, d, T, M, resid);
    if (rc != ORC_OK) goto done;
  }
  matmul(Ahat, M, N, m, d, O);

  if (im) {
#define COPY_OUT(field, src, count) \
  if (im->field) memcpy(im->field + (size_t)slice * (count), src, sizeof(double) * (count))
    COPY_OUT(landmarks, L, md);
    COPY_OUT(d_ql, Dql, nm);
    COPY_OUT(d_ll, Dll, mm);
    COPY_OUT(d_lk, Dlk, nm);
    COPY_OUT(a, A, nm);
    COPY_OUT(b, Bm, nm);
    COPY_OUT(w, W, mm);
    COPY_OUT(x, X, mm);
    COPY_OUT(mu, mu, (size_t)m);
    COPY_OUT(var, var, (size_t)m);
    COPY_OUT(a_hat, Ahat, nm);
    COPY_OUT(bv, BV, md);
    COPY_OUT(m_mat, M, md);
    COPY_OUT(ns_resid, resid, (size_t)(T + 1));
#undef COPY_OUT
  }

done:
  free(L); free(Dql); free(Dll); free(Dlk); free(A); free(Bm); free(W); free(X);
  free(mu); free(var); free(Ahat); free(BV); free(M); free(resid);
  return rc;
}

int orc_forward_slices(const orc_config* cfg, const double* q, const double* k, const double* v,
                       const double* bias, double* out, const orc_intermediates* im,
                       long slice_begin, long slice_count) {
  const int rc = check_config(cfg);
  if (rc != ORC_OK) return rc;
  const long slices = (long)cfg->batch * cfg->heads;
  if (slice_begin < 0 || slice_count < 0 || slice_begin + slice_count > slices) return ORC_ERR_ARG;
  if (slice_count == 0) return ORC_OK;
  if (!q || !k || !v || !out) return ORC_ERR_ARG;
  const size_t nd = (size_t)cfg->grid_h * cfg->grid_w * cfg->head_dim;
  for (long sl = slice_begin; sl < slice_begin + slice_count; ++sl) {
    const int h = (int)(sl % cfg->heads);
    const int r = forward_slice(cfg, h, q + (size_t)sl * nd, k + (size_t)sl * nd,
                                v + (size_t)sl * nd, bias, out + (size_t)sl * nd, im, sl);
    if (r != ORC_OK) return r;
  }
  return ORC_OK;
}

int orc_forward(const orc_config* cfg, const double* q, const double* k, const double* v,
                const double* bias, double* out, const orc_intermediates* im) {
  const int rc = check_config(cfg);
  if (rc != ORC_OK) return rc;
  return orc_forward_slices(cfg, q, k, v, bias, out, im, 0, (long)cfg->batch * cfg->heads);
}

/* =========================================================================================
 * Backward: reverse-mode derivative of the forward above for a scalar loss whose gradient
 * with respect to O is G (dO).  The pages claim CUDA kernels for the forward and the backward
 * pass (English page, 2 "CUDA Acceleration"; German page, 2) and describe no gradient; every
 * step below is the chain rule applied to the forward step named beside it, in the reverse
 * order of the forward.  The non-differentiable points take these readings:
 *   |x - y| at x == y: derivative 0 (the sign function with sgn(0) = 0; for D_LL's diagonal,
 *     D_jj == 0 identically, so 0 is the derivative);
 *   the max in |W|_1 and |W|_inf: the derivative of the first maximal column (row) sum.
 * Only the Newton-Schulz solver is differentiated (solver = 1 is rejected).
 * ======================================================================================= */

/* d D(x, y) / d x for the kernel's distance: sgn(x - y) (Laplacian) or 2 (x - y) (Gaussian). */
static double distance_slope(const orc_config* cfg, double x, double y) {
  if (cfg->kernel == 1) return 2.0 * (x - y);
  return x > y ? 1.0 : (x < y ? -1.0 : 0.0);
}

/* A pair whose sign decision a float32 computation may take the other way. */
static int near_tie(const orc_config* cfg, double x, double y, double tau) {
  return cfg->kernel == 0 && fabs(x - y) <= tau * (fabs(x) + fabs(y));
}

/* Newton-Schulz as in step 3, keeping every iterate X_0 .. X_T ([T+1][m][m]) and the first
 * maximal column (jc) and row (ir) of the norms of X0. */
static int newton_schulz_history(const double* W, int m, int T, double* Xs, double* scale,
                                 int* jc, int* ir) {
  double n1 = -1.0, ninf = -1.0;
  for (int j = 0; j < m; ++j) {
    double s = 0.0;
    for (int i = 0; i < m; ++i) s += fabs(W[(size_t)i * m + j]);
    if (s > n1) { n1 = s; *jc = j; }
  }
  for (int i = 0; i < m; ++i) {
    double s = 0.0;
    for (int j = 0; j < m; ++j) s += fabs(W[(size_t)i * m + j]);
    if (s > ninf) { ninf = s; *ir = i; }
  }
  *scale = n1 * ninf;
  const size_t mm = (size_t)m * m;
  for (int i = 0; i < m; ++i)
    for (int j = 0; j < m; ++j) Xs[(size_t)i * m + j] = W[(size_t)j * m + i] / *scale;
  double* P = (double*)malloc(sizeof(double) * mm);
  if (!P) return ORC_ERR_NOMEM;
  for (int t = 0; t < T; ++t) {
    const double* X = Xs + (size_t)t * mm;
    double* Xn = Xs + (size_t)(t + 1) * mm;
    matmul(W, X, m, m, m, P);                               /* P = W X */
    for (int i = 0; i < m; ++i) /* X_{t+1} = X (2I - P) */
      for (int j = 0; j < m; ++j) {
        double s = 0.0;
        for (int k = 0; k < m; ++k)
          s += X[(size_t)i * m + k] * ((k == j ? 2.0 : 0.0) - P[(size_t)k * m + j]);
        Xn[(size_t)i * m + j] = s;
      }
  }
  free(P);
  return ORC_OK;
}

/* C = A^T B for A [inner, rows], B [inner, cols]. */
static void matmul_tn(const double* Aop, const double* Bop, int rows, int inner, int cols,
                      double* C) {
  for (int i = 0; i < rows; ++i)
    for (int j = 0; j < cols; ++j) {
      double s = 0.0;
      for (int k = 0; k < inner; ++k) s += Aop[(size_t)k * rows + i] * Bop[(size_t)k * cols + j];
      C[(size_t)i * cols + j] = s;
    }
}

/* C = A B^T for A [rows, inner], B [cols, inner]. */
static void matmul_nt(const double* Aop, const double* Bop, int rows, int inner, int cols,
                      double* C) {
  for (int i = 0; i < rows; ++i)
    for (int j = 0; j < cols; ++j) {
      double s = 0.0;
      for (int k = 0; k < inner; ++k) s += Aop[(size_t)i * inner + k] * Bop[(size_t)j * inner + k];
      C[(size_t)i * cols + j] = s;
    }
}

static int backward_slice(const orc_config* cfg, int h, const double* Q, const double* K,
                          const double* V, const double* bias, const double* G, double* dQ,
                          double* dK, double* dV, double* dbias, double* amb_q, double* amb_k,
                          double tau) {
  const int N = cfg->grid_h * cfg->grid_w, d = cfg->head_dim, m = cfg->num_landmarks;
  const int s = isqrt_exact(m), ph = cfg->grid_h / s, pw = cfg->grid_w / s;
  const int T = cfg->ns_steps;
  const double lam = cfg->lambda;
  const size_t nm = (size_t)N * m, mm = (size_t)m * m, md = (size_t)m * d;
  double* L = (double*)malloc(sizeof(double) * md);
  double* A = (double*)malloc(sizeof(double) * nm);
  double* Bm = (double*)malloc(sizeof(double) * nm);
  double* W = (double*)malloc(sizeof(double) * mm);
  double* Xs = (double*)malloc(sizeof(double) * mm * (size_t)(T + 1));
  double* mu = (double*)malloc(sizeof(double) * m);
  double* var = (double*)malloc(sizeof(double) * m);
  double* Ahat = (double*)malloc(sizeof(double) * nm);
  double* Z = (double*)malloc(sizeof(double) * nm);
  double* BV = (double*)malloc(sizeof(double) * md);
  double* M = (double*)malloc(sizeof(double) * md);
  double* dAhat = (double*)malloc(sizeof(double) * nm);
  double* dM = (double*)malloc(sizeof(double) * md);
  double* gq = (double*)malloc(sizeof(double) * nm);      /* dLoss / dD_QL */
  double* dL = (double*)calloc(md, sizeof(double));
  double* ambL = (double*)calloc(md, sizeof(double));
  double* dBV = (double*)malloc(sizeof(double) * md);
  double* dX = (double*)malloc(sizeof(double) * mm);
  double* dXp = (double*)malloc(sizeof(double) * mm);
  double* dW = (double*)calloc(mm, sizeof(double));
  double* gk = (double*)malloc(sizeof(double) * nm);      /* dLoss / dD_LK, [m][N] */
  double* t1 = (double*)malloc(sizeof(double) * mm);
  double* t2 = (double*)malloc(sizeof(double) * mm);
  double scale = 1.0;
  int jc = 0, ir = 0, rc = ORC_OK;
  if (!L || !A || !Bm || !W || !Xs || !mu || !var || !Ahat || !Z || !BV || !M || !dAhat || !dM ||
      !gq || !dL || !ambL || !dBV || !dX || !dXp || !dW || !gk || !t1 || !t2) {
    rc = ORC_ERR_NOMEM;
    goto done;
  }

  /* forward, steps 1-5, keeping what the backward needs */
  landmarks_avgpool(K, cfg->grid_w, d, s, ph, pw, L);
  for (int i = 0; i < N; ++i)
    for (int j = 0; j < m; ++j)
      A[(size_t)i * m + j] =
          laplacian_of_distance(kernel_distance(cfg, Q + (size_t)i * d, L + (size_t)j * d, d), lam);
  for (int j = 0; j < m; ++j)
    for (int n = 0; n < N; ++n)
      Bm[(size_t)j * N + n] =
          laplacian_of_distance(kernel_distance(cfg, L + (size_t)j * d, K + (size_t)n * d, d), lam);
  for (int j = 0; j < m; ++j)
    for (int k = 0; k < m; ++k)
      W[(size_t)j * m + k] =
          laplacian_of_distance(kernel_distance(cfg, L + (size_t)j * d, L + (size_t)k * d, d), lam) +
          (j == k ? cfg->eps : 0.0);
  rc = newton_schulz_history(W, m, T, Xs, &scale, &jc, &ir);
  if (rc != ORC_OK) goto done;
  const double* X = Xs + (size_t)T * mm;
  if (cfg->whiten) {
    whiten_columns(A, N, m, cfg->delta, bias ? bias + (size_t)h * m : NULL, mu, var, Ahat);
    for (int i = 0; i < N; ++i)
      for (int j = 0; j < m; ++j)
        Z[(size_t)i * m + j] = (A[(size_t)i * m + j] - mu[j]) / sqrt(var[j] + cfg->delta);
  } else {
    memcpy(Ahat, A, sizeof(double) * nm);
  }
  matmul(Bm, V, m, N, d, BV);
  matmul(X, BV, m, m, d, M);

  /* step 5 back: O = A_hat M  ->  dA_hat = G M^T, dM = A_hat^T G */
  matmul_nt(G, M, N, d, m, dAhat);
  matmul_tn(Ahat, G, m, N, d, dM);

  /* step 4 back: A_hat = Z + bias, Z = (A - mu) r, r = 1/sqrt(var + delta), var over N:
   * dbias_j = sum_i dA_hat_ij;  dA_ij = r_j (dZ_ij - mean_i dZ_ij - Z_ij mean_i(dZ_ij Z_ij)) */
  if (cfg->whiten) {
    for (int j = 0; j < m; ++j) {
      double s1 = 0.0, s2 = 0.0;
      for (int i = 0; i < N; ++i) {
        s1 += dAhat[(size_t)i * m + j];
        s2 += dAhat[(size_t)i * m + j] * Z[(size_t)i * m + j];
      }
      if (dbias) dbias[j] += s1;
      const double r = 1.0 / sqrt(var[j] + cfg->delta);
      for (int i = 0; i < N; ++i) {
        const double da = r * (dAhat[(size_t)i * m + j] - s1 / (double)N -
                               Z[(size_t)i * m + j] * s2 / (double)N);
        gq[(size_t)i * m + j] = -A[(size_t)i * m + j] / lam * da;   /* step 2 back: d exp */
      }
    }
  } else {
    for (size_t e = 0; e < nm; ++e) gq[e] = -A[e] / lam * dAhat[e];
  }

  /* step 2 back, query block: D_QL[i][j] = sum_c D(Q_ic, L_jc) */
  for (int i = 0; i < N; ++i)
    for (int c = 0; c < d; ++c) {
      double acc = 0.0, amb = 0.0;
      const double qv = Q[(size_t)i * d + c];
      for (int j = 0; j < m; ++j) {
        const double lv = L[(size_t)j * d + c], g = gq[(size_t)i * m + j];
        const double sl = distance_slope(cfg, qv, lv);
        acc += g * sl;
        dL[(size_t)j * d + c] -= g * sl;
        if (near_tie(cfg, qv, lv, tau)) {
          amb += 2.0 * fabs(g);
          ambL[(size_t)j * d + c] += 2.0 * fabs(g);
        }
      }
      dQ[(size_t)i * d + c] = acc;
      if (amb_q) amb_q[(size_t)i * d + c] = amb;
    }

  /* step 5 back: M = X BV  ->  dBV = X^T dM, dX = dM BV^T */
  matmul_tn(X, dM, m, m, d, dBV);
  matmul_nt(dM, BV, m, d, m, dX);
  /* BV = B V  ->  dB = dBV V^T, dV = B^T dBV; step 2 back, key block: gk = -B/lambda dB */
  matmul_tn(Bm, dBV, N, m, d, dV);
  for (int j = 0; j < m; ++j)
    for (int n = 0; n < N; ++n) {
      double db = 0.0;
      for (int c = 0; c < d; ++c) db += dBV[(size_t)j * d + c] * V[(size_t)n * d + c];
      gk[(size_t)j * N + n] = -Bm[(size_t)j * N + n] / lam * db;
    }
  /* D_LK[j][n] = sum_c D(L_jc, K_nc) */
  for (int n = 0; n < N; ++n)
    for (int c = 0; c < d; ++c) {
      double acc = 0.0, amb = 0.0;
      const double kv = K[(size_t)n * d + c];
      for (int j = 0; j < m; ++j) {
        const double lv = L[(size_t)j * d + c], g = gk[(size_t)j * N + n];
        const double sl = distance_slope(cfg, lv, kv);
        dL[(size_t)j * d + c] += g * sl;
        acc -= g * sl;
        if (near_tie(cfg, lv, kv, tau)) {
          amb += 2.0 * fabs(g);
          ambL[(size_t)j * d + c] += 2.0 * fabs(g);
        }
      }
      dK[(size_t)n * d + c] = acc;
      if (amb_k) amb_k[(size_t)n * d + c] = amb;
    }

  /* step 3 back: X_{t+1} = X_t Y_t, Y_t = 2I - W X_t:
   *   dW += -X_t^T dX_{t+1} X_t^T;  dX_t = dX_{t+1} Y_t^T - W^T X_t^T dX_{t+1} */
  for (int t = T - 1; t >= 0; --t) {
    const double* Xt = Xs + (size_t)t * mm;
    matmul_tn(Xt, dX, m, m, m, t1);                  /* t1 = X_t^T dX_{t+1} */
    matmul_nt(t1, Xt, m, m, m, t2);                  /* t2 = t1 X_t^T */
    for (size_t e = 0; e < mm; ++e) dW[e] -= t2[e];
    matmul(W, Xt, m, m, m, t2);                      /* t2 = W X_t, Y_t = 2I - t2 */
    for (int i = 0; i < m; ++i)
      for (int j = 0; j < m; ++j) {
        double sy = 0.0, sw = 0.0;
        for (int k = 0; k < m; ++k) {
          sy += dX[(size_t)i * m + k] * ((j == k ? 2.0 : 0.0) - t2[(size_t)j * m + k]);
          sw += W[(size_t)k * m + i] * t1[(size_t)k * m + j];
        }
        dXp[(size_t)i * m + j] = sy - sw;
      }
    memcpy(dX, dXp, sizeof(double) * mm);
  }
  /* X_0 = W^T / (|W|_1 |W|_inf) */
  {
    double dsc = 0.0;
    for (int i = 0; i < m; ++i)
      for (int j = 0; j < m; ++j) {
        dW[(size_t)j * m + i] += dX[(size_t)i * m + j] / scale;
        dsc -= dX[(size_t)i * m + j] * W[(size_t)j * m + i] / (scale * scale);
      }
    double n1 = 0.0, ninf = 0.0;
    for (int i = 0; i < m; ++i) n1 += fabs(W[(size_t)i * m + jc]);
    for (int j = 0; j < m; ++j) ninf += fabs(W[(size_t)ir * m + j]);
    for (int i = 0; i < m; ++i) {
      const double w = W[(size_t)i * m + jc];
      dW[(size_t)i * m + jc] += dsc * ninf * (w > 0.0 ? 1.0 : (w < 0.0 ? -1.0 : 0.0));
    }
    for (int j = 0; j < m; ++j) {
      const double w = W[(size_t)ir * m + j];
      dW[(size_t)ir * m + j] += dsc * n1 * (w > 0.0 ? 1.0 : (w < 0.0 ? -1.0 : 0.0));
    }
  }
  /* step 2 back, landmark block: W = exp(-D_LL / lambda) + eps I; D_LL[j][k] = sum_c D(L_j, L_k):
   * dL_pc += sum_k (gw[p][k] + gw[k][p]) slope(L_pc, L_kc) */
  for (int p = 0; p < m; ++p)
    for (int k = 0; k < m; ++k) {
      if (k == p) continue;
      const double kpk = W[(size_t)p * m + k], kkp = W[(size_t)k * m + p];
      const double g = -kpk / lam * dW[(size_t)p * m + k] - kkp / lam * dW[(size_t)k * m + p];
      for (int c = 0; c < d; ++c) {
        const double lp = L[(size_t)p * d + c], lk = L[(size_t)k * d + c];
        dL[(size_t)p * d + c] += g * distance_slope(cfg, lp, lk);
        if (near_tie(cfg, lp, lk, tau)) ambL[(size_t)p * d + c] += 2.0 * fabs(g);
      }
    }

  /* step 1 back: L_j = mean of K over window j  ->  dK_n += dL_j(n) / (ph pw) */
  for (int r = 0; r < cfg->grid_h; ++r)
    for (int cc = 0; cc < cfg->grid_w; ++cc) {
      const int j = (r / ph) * s + cc / pw;
      const size_t n = (size_t)r * cfg->grid_w + cc;
      for (int c = 0; c < d; ++c) {
        dK[n * d + c] += dL[(size_t)j * d + c] / (double)(ph * pw);
        if (amb_k) amb_k[n * d + c] += ambL[(size_t)j * d + c] / (double)(ph * pw);
      }
    }

done:
  free(L); free(A); free(Bm); free(W); free(Xs); free(mu); free(var); free(Ahat); free(Z);
  free(BV); free(M); free(dAhat); free(dM); free(gq); free(dL); free(ambL); free(dBV); free(dX);
  free(dXp); free(dW); free(gk); free(t1); free(t2);
  return rc;
}

int orc_backward_slices(const orc_config* cfg, const double* q, const double* k, const double* v,
                        const double* bias, const double* dout, double* dq, double* dk,
                        double* dv, double* dbias, double* amb_dq, double* amb_dk, double tau,
                        long slice_begin, long slice_count) {
  const int rc = check_config(cfg);
  if (rc != ORC_OK) return rc;
  if (cfg->solver != 0) return ORC_ERR_UNSUPPORTED;
  const long slices = (long)cfg->batch * cfg->heads;
  if (slice_begin < 0 || slice_count < 0 || slice_begin + slice_count > slices) return ORC_ERR_ARG;
  if (slice_count == 0) return ORC_OK;
  if (!q || !k || !v || !dout || !dq || !dk || !dv) return ORC_ERR_ARG;
  const size_t nd = (size_t)cfg->grid_h * cfg->grid_w * cfg->head_dim;
  for (long sl = slice_begin; sl < slice_begin + slice_count; ++sl) {
    const int h = (int)(sl % cfg->heads);
    const size_t o = (size_t)sl * nd;
    const int r = backward_slice(cfg, h, q + o, k + o, v + o, bias, dout + o, dq + o, dk + o,
                                 dv + o, dbias ? dbias + (size_t)h * cfg->num_landmarks : NULL,
                                 amb_dq ? amb_dq + o : NULL, amb_dk ? amb_dk + o : NULL, tau);
    if (r != ORC_OK) return r;
  }
  return ORC_OK;
}
