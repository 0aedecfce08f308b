/*
 * fp64 oracle for FAVOR+ attention.  TEST INFRASTRUCTURE ONLY: only the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load this file's library. The CUDA path never calls it.
 *
 * Plain loops in double precision, OpenMP over heads, no BLAS, no blocking or reordering beyond
 * what the equations state. Each function names the passage it follows:
 *
 *  [P2-norm]  "Performer" paper note, *Normalization*: y_i = phi(q_i)^T (sum_j phi(k_j) v_j^T)
 *             / phi(q_i)^T (sum_j phi(k_j)).
 *  [P2-kern]  same page, *Kernel Attention View*: S = Phi(K)^T V computed once, Y~ = Phi(Q) S.
 *  [P2-favor] same page, *FAVOR+*: positive random features with E[phi(q)^T phi(k)] = exp(q^T k),
 *             m features.  The exact map is not printed there; this oracle uses
 *             phi_r(x) = exp(w_r^T x^ - |x^|^2/2 - stab) / sqrt(m), x^ = d^(-1/4) x, the standard
 *             positive map whose expectation over w ~ N(0, I) is exp(q^T k) (Gaussian moment
 *             generating function), which realises the 1/sqrt(d) of the page's softmax equation.
 *  [P4-steps] "Performer for vision", *How It Works*, Step 1 (features, numerator, denominator)
 *             and Step 2 (prefix sums in the causal setting, each token attends to itself and
 *             earlier tokens, then divide).
 *  [P4-relu]  same page, *What Is Performer?*, Key Feature 4: ReLU features; the form used is
 *             phi_r(x) = max(0, w_r^T x^) / sqrt(m) + eps, with no stabiliser.
 *
 * Stabilisers (the pages give none; any constant that is the same for all features of one query
 * row, or for all keys and features of one head, cancels between numerator and denominator):
 *   STAB_NONE 0: none;  STAB_ROW 1: per token, max over r of u_r;  STAB_HEAD 2: per head, max over
 *   tokens j and features r of u_r, where u_r(x) = w_r^T x^ - |x^|^2/2.
 * Attention stabiliser modes: ATT_CANONICAL 0 (queries STAB_ROW, keys STAB_HEAD), ATT_NONE 1,
 *   ATT_BOUND 2 (data-free bounds: keys max_r |w_r|^2/2, queries max_r |w_r||x^| - |x^|^2/2).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { KIND_EXP = 0, KIND_RELU = 1 };
enum { STAB_NONE = 0, STAB_ROW = 1, STAB_HEAD = 2 };
enum { ATT_CANONICAL = 0, ATT_NONE = 1, ATT_BOUND = 2 };

void oracle_set_threads(int t) {
#ifdef _OPENMP
    if (t > 0) omp_set_num_threads(t);
#else
    (void)t;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* w_r^T x^ for every r, with x^ = d^(-1/4) x; returns |x^|^2 / 2 through *half_norm2. */
static void project(const double* x, const double* omega, int d, int m, double* proj, double* half_norm2) {
    const double s = pow((double)d, -0.25);
    double nrm = 0.0;
    for (int c = 0; c < d; ++c) nrm += (s * x[c]) * (s * x[c]);
    *half_norm2 = 0.5 * nrm;
    for (int r = 0; r < m; ++r) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += omega[(int64_t)r * d + c] * (s * x[c]);
        proj[r] = acc;
    }
}

/* exponents u_r(x) = w_r^T x^ - |x^|^2/2  [P2-favor] */
static void exponents(const double* x, const double* omega, int d, int m, double* u) {
    double h;
    project(x, omega, d, m, u, &h);
    for (int r = 0; r < m; ++r) u[r] -= h;
}

static double max_of(const double* a, int m) {
    double v = -INFINITY;
    for (int r = 0; r < m; ++r) v = a[r] > v ? a[r] : v;
    return v;
}

/* phi(x) given a stabiliser value (exp family) [P2-favor] or the ReLU form [P4-relu]. */
static void feature_row(const double* x, const double* omega, int d, int m, int kind, double relu_eps,
                        double stab, double* phi) {
    const double inv_sqrt_m = 1.0 / sqrt((double)m);
    if (kind == KIND_RELU) {
        double h;
        project(x, omega, d, m, phi, &h);
        for (int r = 0; r < m; ++r) phi[r] = (phi[r] > 0.0 ? phi[r] : 0.0) * inv_sqrt_m + relu_eps;
    } else {
        exponents(x, omega, d, m, phi);
        for (int r = 0; r < m; ++r) phi[r] = exp(phi[r] - stab) * inv_sqrt_m;
    }
}

/* Largest exponent over all tokens and features of one head (STAB_HEAD). */
static double head_max_exponent(const double* X, const double* omega, int64_t n, int d, int m, double* tmp) {
    double mx = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        exponents(X + j * d, omega, d, m, tmp);
        double v = max_of(tmp, m);
        mx = v > mx ? v : mx;
    }
    return mx;
}

static double omega_half_norm2_max(const double* omega, int d, int m) {
    double mx = -INFINITY;
    for (int r = 0; r < m; ++r) {
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += omega[(int64_t)r * d + c] * omega[(int64_t)r * d + c];
        mx = 0.5 * s > mx ? 0.5 * s : mx;
    }
    return mx;
}

/* Stabiliser of one query row under attention mode `mode`. */
static double query_stab(const double* x, const double* omega, int d, int m, int mode, double* tmp) {
    if (mode == ATT_NONE) return 0.0;
    if (mode == ATT_BOUND) {
        const double s = pow((double)d, -0.25);
        double xn = 0.0, wmax = 0.0;
        for (int c = 0; c < d; ++c) xn += (s * x[c]) * (s * x[c]);
        for (int r = 0; r < m; ++r) {
            double w = 0.0;
            for (int c = 0; c < d; ++c) w += omega[(int64_t)r * d + c] * omega[(int64_t)r * d + c];
            wmax = w > wmax ? w : wmax;
        }
        return sqrt(wmax) * sqrt(xn) - 0.5 * xn;
    }
    exponents(x, omega, d, m, tmp);
    return max_of(tmp, m);
}

static double key_stab(const double* K, const double* omega, int64_t n, int d, int m, int mode, double* tmp) {
    if (mode == ATT_NONE) return 0.0;
    if (mode == ATT_BOUND) return omega_half_norm2_max(omega, d, m);
    return head_max_exponent(K, omega, n, d, m, tmp);
}

/*
 * Feature map of nh heads: X [nh, n, d] -> Phi [nh, n, m].  [P2-favor] / [P4-relu]
 * stab: STAB_NONE, STAB_ROW or STAB_HEAD (ignored for the ReLU family).
 */
void oracle_features(const double* X, const double* omega, double* Phi, int64_t nh, int64_t n, int d, int m,
                     int kind, double relu_eps, int stab) {
#pragma omp parallel for schedule(dynamic)
    for (int64_t hd = 0; hd < nh; ++hd) {
        const double* Xh = X + hd * n * d;
        double* Ph = Phi + hd * n * m;
        double* tmp = (double*)malloc(sizeof(double) * m);
        double head_stab = 0.0;
        if (kind == KIND_EXP && stab == STAB_HEAD) head_stab = head_max_exponent(Xh, omega, n, d, m, tmp);
        for (int64_t j = 0; j < n; ++j) {
            double st = 0.0;
            if (kind == KIND_EXP && stab == STAB_ROW) {
                exponents(Xh + j * d, omega, d, m, tmp);
                st = max_of(tmp, m);
            } else if (kind == KIND_EXP && stab == STAB_HEAD) {
                st = head_stab;
            }
            feature_row(Xh + j * d, omega, d, m, kind, relu_eps, st, Ph + j * m);
        }
        free(tmp);
    }
}

/*
 * Non-causal FAVOR+ attention of nh heads.  [P2-kern], [P2-norm], [P4-steps] Step 1.
 *   S = sum_j phi(k_j) v_j^T (m x d),  z = sum_j phi(k_j) (m),  y_i = phi(q_i)^T S / phi(q_i)^T z.
 */
void oracle_noncausal(const double* Q, const double* K, const double* V, const double* omega, double* Y,
                      int64_t nh, int64_t n, int d, int m, int kind, double relu_eps, int mode) {
#pragma omp parallel for schedule(dynamic)
    for (int64_t hd = 0; hd < nh; ++hd) {
        const double* Qh = Q + hd * n * d;
        const double* Kh = K + hd * n * d;
        const double* Vh = V + hd * n * d;
        double* Yh = Y + hd * n * d;
        double* S = (double*)calloc((size_t)m * d, sizeof(double));
        double* z = (double*)calloc((size_t)m, sizeof(double));
        double* phi = (double*)malloc(sizeof(double) * m);
        double* tmp = (double*)malloc(sizeof(double) * m);
        double ks = kind == KIND_EXP ? key_stab(Kh, omega, n, d, m, mode, tmp) : 0.0;
        for (int64_t j = 0; j < n; ++j) {
            feature_row(Kh + j * d, omega, d, m, kind, relu_eps, ks, phi);
            for (int r = 0; r < m; ++r) {
                z[r] += phi[r];
                for (int c = 0; c < d; ++c) S[(int64_t)r * d + c] += phi[r] * Vh[j * d + c];
            }
        }
        for (int64_t i = 0; i < n; ++i) {
            double qs = kind == KIND_EXP ? query_stab(Qh + i * d, omega, d, m, mode, tmp) : 0.0;
            feature_row(Qh + i * d, omega, d, m, kind, relu_eps, qs, phi);
            double den = 0.0;
            for (int r = 0; r < m; ++r) den += phi[r] * z[r];
            for (int c = 0; c < d; ++c) {
                double num = 0.0;
                for (int r = 0; r < m; ++r) num += phi[r] * S[(int64_t)r * d + c];
                Yh[i * d + c] = num / den;
            }
        }
        free(S); free(z); free(phi); free(tmp);
    }
}

/*
 * Causal FAVOR+ attention of nh heads as the plain per-token prefix-sum recurrence.
 * [P4-steps] Step 2, [P2-norm] with the sums running over j <= i:
 *   S_i = S_{i-1} + phi(k_i) v_i^T,  z_i = z_{i-1} + phi(k_i),  y_i = phi(q_i)^T S_i / phi(q_i)^T z_i.
 * The key stabiliser is one constant per head (over all of its keys), as in the non-causal form.
 */
void oracle_causal(const double* Q, const double* K, const double* V, const double* omega, double* Y,
                   int64_t nh, int64_t n, int d, int m, int kind, double relu_eps, int mode) {
#pragma omp parallel for schedule(dynamic)
    for (int64_t hd = 0; hd < nh; ++hd) {
        const double* Qh = Q + hd * n * d;
        const double* Kh = K + hd * n * d;
        const double* Vh = V + hd * n * d;
        double* Yh = Y + hd * n * d;
        double* S = (double*)calloc((size_t)m * d, sizeof(double));
        double* z = (double*)calloc((size_t)m, sizeof(double));
        double* phi = (double*)malloc(sizeof(double) * m);
        double* tmp = (double*)malloc(sizeof(double) * m);
        double ks = kind == KIND_EXP ? key_stab(Kh, omega, n, d, m, mode, tmp) : 0.0;
        for (int64_t i = 0; i < n; ++i) {
            feature_row(Kh + i * d, omega, d, m, kind, relu_eps, ks, phi);
            for (int r = 0; r < m; ++r) {
                z[r] += phi[r];
                for (int c = 0; c < d; ++c) S[(int64_t)r * d + c] += phi[r] * Vh[i * d + c];
            }
            double qs = kind == KIND_EXP ? query_stab(Qh + i * d, omega, d, m, mode, tmp) : 0.0;
            feature_row(Qh + i * d, omega, d, m, kind, relu_eps, qs, phi);
            double den = 0.0;
            for (int r = 0; r < m; ++r) den += phi[r] * z[r];
            for (int c = 0; c < d; ++c) {
                double num = 0.0;
                for (int r = 0; r < m; ++r) num += phi[r] * S[(int64_t)r * d + c];
                Yh[i * d + c] = num / den;
            }
        }
        free(S); free(z); free(phi); free(tmp);
    }
}
