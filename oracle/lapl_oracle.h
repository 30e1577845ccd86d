/*
 * lapl_oracle.h -- plain fp64 CPU oracle for Laplacian-kernel Nystrom attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the independent CPU reference that the CUDA library is
 * checked against.  Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no code, header, table or constant with the CUDA library: nothing under
 * laplacian_nystr_attention_gb300/ includes this file and nothing here includes theirs.
 *
 * What it computes (per batch b and head h, all in double precision), following
 * "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel" (explainer pages):
 *   1. landmarks L = 2-D average pooling of K over the token grid        (English page, 2.C.1)
 *   2. A = k(Q,L), B = k(L,K), W = k(L,L) + eps*I with
 *      k(x,y) = exp(-||x-y||_1 / lambda)                                  (English page, 2.A;
 *                                                                          small eps*I: 2.C.2)
 *   3. X = T Newton-Schulz steps X <- X(2I - W X) from X0 = W^T/(|W|_1 |W|_inf)
 *                                                                         (English page, 2.C.2)
 *   4. whitening of A column by column with a diagonal estimator:
 *      A_hat = (A - mean) / sqrt(var + delta) + bias                      (Korean page, 2.2)
 *   5. O = A_hat * (X * (B * V)): the N x N matrix is never formed        (Chinese page, 2.2)
 * With kernel = 1 the kernel of step 2 is the Gaussian one the pages compare against,
 * k(x,y) = exp(-||x-y||_2^2 / lambda): similarity decaying with the squared l2 distance
 * (English page, 1 "Theoretical Mismatch"); every other step is unchanged.
 * With solver = 1 steps 3 and 5 take the conjugate-gradient solver the pages compare the
 * Newton-Schulz iteration with (German page, 4; English page, 4 "Solver Robustness"):
 * M = T CG iterations on W M = B V, column by column from zero, replaces X (B V).
 */
#ifndef LAPL_ORACLE_H
#define LAPL_ORACLE_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int batch, heads;        /* B, H: independent (b,h) slices */
  int grid_h, grid_w;      /* token grid; N = grid_h * grid_w, token n = r * grid_w + c */
  int head_dim;            /* d */
  int num_landmarks;       /* m = s*s; grid_h % s == 0 and grid_w % s == 0 */
  double lambda;           /* kernel scale, > 0 */
  double eps;              /* diagonal perturbation of W, >= 0 */
  double delta;            /* whitening variance floor, > 0 when whiten != 0 */
  int ns_steps;            /* T >= 0 Newton-Schulz steps, no early exit */
  int whiten;              /* 1: whiten A; 0: A_hat = A (bias ignored) */
  int kernel;              /* 0: Laplacian, distance sum_c |x_c - y_c|;
                              1: Gaussian, distance sum_c (x_c - y_c)^2 */
  int solver;              /* 0: Newton-Schulz X, M = X (B V);
                              1: T conjugate-gradient iterations on W M = B V */
} orc_config;

/* Every pointer may be NULL.  Shapes are for the whole [B,H] batch, C order. */
typedef struct {
  double* landmarks; /* [B,H,m,d]   L                              */
  double* d_ql;      /* [B,H,N,m]   sum_c |Q_ic - L_jc| (squared terms when Gaussian) */
  double* d_ll;      /* [B,H,m,m]   sum_c |L_jc - L_kc|             */
  double* d_lk;      /* [B,H,m,N]   sum_c |L_jc - K_nc|             */
  double* a;         /* [B,H,N,m]   exp(-D_QL / lambda)             */
  double* b;         /* [B,H,m,N]   exp(-D_LK / lambda)             */
  double* w;         /* [B,H,m,m]   exp(-D_LL / lambda) + eps I     */
  double* x;         /* [B,H,m,m]   X_T (zeros with the CG solver)  */
  double* mu;        /* [B,H,m]     column means of A               */
  double* var;       /* [B,H,m]     column variances of A (divide by N) */
  double* a_hat;     /* [B,H,N,m]   whitened A                      */
  double* bv;        /* [B,H,m,d]   B V                             */
  double* m_mat;     /* [B,H,m,d]   X (B V), or the CG solution     */
  double* ns_resid;  /* [B,H,T+1]   Frobenius norm of I - W X_t, t = 0..T; with the CG
                                    solver the relative residual ||R_t||_F / ||B V||_F */
} orc_intermediates;

/* Status codes. */
enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_UNSUPPORTED = 2, ORC_ERR_NOMEM = 3 };

/*
 * Full forward over every (b,h) slice.
 * q, k, v, out: [B,H,N,d]; bias: [H,m] or NULL (zeros).
 */
int orc_forward(const orc_config* cfg, const double* q, const double* k, const double* v,
                const double* bias, double* out, const orc_intermediates* im);

/*
 * Same, restricted to the slices s = b*H + h with slice_begin <= s < slice_begin + slice_count.
 * Arrays are still the full [B,H,...] arrays; only those slices are read or written.
 */
/*
 * Backward of the forward for a loss with gradient dout = dLoss/dO ([B,H,N,d]), over the
 * slices s = b*H + h with slice_begin <= s < slice_begin + slice_count: dq, dk, dv
 * ([B,H,N,d]) are written for those slices; dbias ([H,m], or NULL) receives += each slice's
 * column sums of dLoss/dA_hat (zero when whiten = 0), so the caller zeroes it first.
 * amb_dq, amb_dk (nullable, [B,H,N,d]): for the Laplacian kernel, a bound on how far each
 * entry can move when a float32 computation takes a sign decision sgn(x - y) the other way:
 * the sum of 2 |gradient weight| over the pairs with |x - y| <= tau (|x| + |y|), landmark
 * pairs included and carried through the pooling (zero for the Gaussian kernel).
 * Newton-Schulz solver only (ORC_ERR_UNSUPPORTED for solver = 1).
 */
int orc_backward_slices(const orc_config* cfg, const double* q, const double* k, const double* v,
                        const double* bias, const double* dout, double* dq, double* dk,
                        double* dv, double* dbias, double* amb_dq, double* amb_dk, double tau,
                        long slice_begin, long slice_count);

int orc_forward_slices(const orc_config* cfg, const double* q, const double* k, const double* v,
                       const double* bias, double* out, const orc_intermediates* im,
                       long slice_begin, long slice_count);

#ifdef __cplusplus
}
#endif

#endif /* LAPL_ORACLE_H */
