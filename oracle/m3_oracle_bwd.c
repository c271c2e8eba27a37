/*
 * m3_oracle_bwd.c -- fp64 sequential gradient (adjoint) of the Mamba-3 scan.
 *
 * TEST INFRASTRUCTURE ONLY, like m3_oracle.c next to it: only tests/,
 * __graft_entry__.smoke() and the cpu_baseline / reference leg of bench.py may
 * load it.  It shares no code, header or constant with the CUDA library.
 *
 * Forward (m3_oracle.c, the complex frame; Mamba-3 summary page §3.1 eq.
 * (5)-(6), §3.2 Proposition 3.2.1, §3.3):
 *   alpha_t = exp(dt_t A), beta_t = (1 - lambda_t) dt_t alpha_t, gamma_t = lambda_t dt_t
 *   u_t  = sum_r B_t[r] x_t[r]^T
 *   z_t  = alpha_t h_{t-1} + beta_t u_{t-1}
 *   h_t  = R(theta_t) z_t + gamma_t u_t
 *   y_t[r] = C_t[r]^T h_t,         final = h_{T-1}
 * with h_{-1} = h0 and u_{-1} = sum_r prevB[r] prevx[r]^T.
 *
 * Given the loss L = <dy, y> + <dfinal, final> (dy, dfinal the upstream
 * gradients), this file computes dL/d(every input) by the reverse-mode rule
 * applied to the forward's statements in reverse order (the training-time
 * backward the pages ask for, Mamba-1 review page, "hardware-aware algorithm"
 * step 4; "Foundation Model Engineering" ch. 20.2 on training):
 *   g    = dL/dh_t  (accumulated: dfinal at t = T-1, plus the path through h_{t+1})
 *   g   += sum_r C_t[r] dy_t[r]^T                          (from y_t)
 *   dC_t[r] = h_t dy_t[r]                                   (N-vector: sum over p)
 *   dgamma_t = <g, u_t>,   du_t += gamma_t g
 *   dz   = R(theta_t)^T g = R(-theta_t) g
 *   dtheta_t[k] = sum_p ( -g[2k] w[2k+1] + g[2k+1] w[2k] ),  w = R(theta_t) z_t = h_t - gamma_t u_t
 *                 (d/dphi R(phi) = R(phi) J with J (a, b) = (-b, a))
 *   dalpha_t = <dz, h_{t-1}>,   dbeta_t = <dz, u_{t-1}>
 *   du_{t-1} += beta_t dz,      dL/dh_{t-1} = alpha_t dz
 *   dB_t[r] = du_t x_t[r],      dx_t[r] = du_t^T B_t[r]     (once du_t is complete)
 *   ddt_t    = dalpha alpha A + dbeta (1 - lambda) alpha (1 + dt A) + dgamma lambda
 *   dlambda_t = -dbeta dt alpha + dgamma dt
 *   dA      += dalpha alpha dt + dbeta (1 - lambda) dt^2 alpha
 * and at the end dh0 = dL/dh_{-1}, dprevB[r] = du_{-1} prevx[r],
 * dprevx[r] = du_{-1}^T prevB[r].
 *
 * The forward states h_t (t = -1 .. T-1) and inputs u_t are stored for the
 * whole sequence (plain, no recompute: this is the definition, not a schedule).
 *
 * Layouts (C-contiguous fp64) as in m3_oracle.c; the gradients have the shapes
 * of their inputs, except dA which is per (b, h): dA_bh [b, h] (the caller sums
 * over b).  lambda / theta / h0 / prevB,prevx / dfinal may be NULL (1, 0, 0,
 * none, 0); the gradient pointers of absent inputs may be NULL.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static void bwd_sequence(int64_t T, int64_t H, int64_t P, int64_t N, int64_t R, int64_t b, int64_t h,
                         const double* x, const double* dt, double A_h, const double* Bm, const double* Cm,
                         const double* lam, const double* theta, const double* h0, const double* prevB,
                         const double* prevx, const double* dy, const double* dfinal, double* dx, double* ddt,
                         double* dB, double* dC, double* dlam, double* dtheta, double* dA_bh, double* dh0,
                         double* dprevB, double* dprevx, double* hs /* (T+1) N P */, double* us /* (T+1) N P */,
                         double* g, double* dz, double* du /* (T+1) N P */) {
    const int64_t K = N / 2, NP = N * P;
    const int64_t unit = b * H + h;
    /* ---- forward, storing h_t at hs[(t+1) NP] and u_t at us[(t+1) NP] */
    if (h0) memcpy(hs, h0 + unit * NP, (size_t)NP * sizeof(double));
    else memset(hs, 0, (size_t)NP * sizeof(double));
    for (int64_t n = 0; n < N; ++n)
        for (int64_t p = 0; p < P; ++p) {
            double acc = 0.0;
            if (prevB)
                for (int64_t r = 0; r < R; ++r) acc += prevB[(unit * R + r) * N + n] * prevx[(unit * R + r) * P + p];
            us[n * P + p] = acc;
        }
    for (int64_t t = 0; t < T; ++t) {
        const int64_t bth = (b * T + t) * H + h;
        const double d = dt[bth], l = lam ? lam[bth] : 1.0;
        const double alpha = exp(d * A_h), beta = (1.0 - l) * d * alpha, gamma = l * d;
        const double* hp = hs + t * NP;
        const double* up = us + t * NP;
        double* hc = hs + (t + 1) * NP;
        double* uc = us + (t + 1) * NP;
        for (int64_t n = 0; n < N; ++n)
            for (int64_t p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int64_t r = 0; r < R; ++r) acc += Bm[(bth * R + r) * N + n] * x[(bth * R + r) * P + p];
                uc[n * P + p] = acc;
            }
        for (int64_t k = 0; k < K; ++k) {
            const double phi = theta ? theta[bth * K + k] : 0.0;
            const double c = cos(phi), s = sin(phi);
            for (int64_t p = 0; p < P; ++p) {
                const double z0 = alpha * hp[(2 * k) * P + p] + beta * up[(2 * k) * P + p];
                const double z1 = alpha * hp[(2 * k + 1) * P + p] + beta * up[(2 * k + 1) * P + p];
                hc[(2 * k) * P + p] = c * z0 - s * z1 + gamma * uc[(2 * k) * P + p];
                hc[(2 * k + 1) * P + p] = s * z0 + c * z1 + gamma * uc[(2 * k + 1) * P + p];
            }
        }
    }
    /* ---- reverse */
    if (dfinal) memcpy(g, dfinal + unit * NP, (size_t)NP * sizeof(double));
    else memset(g, 0, (size_t)NP * sizeof(double));
    memset(du, 0, (size_t)((T + 1) * NP) * sizeof(double));
    double dA_acc = 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
        const int64_t bth = (b * T + t) * H + h;
        const double d = dt[bth], l = lam ? lam[bth] : 1.0;
        const double alpha = exp(d * A_h), beta = (1.0 - l) * d * alpha, gamma = l * d;
        const double* hp = hs + t * NP;         /* h_{t-1} */
        const double* hc = hs + (t + 1) * NP;   /* h_t */
        const double* up = us + t * NP;         /* u_{t-1} */
        const double* uc = us + (t + 1) * NP;   /* u_t */
        double* dup = du + t * NP;              /* du_{t-1} */
        double* duc = du + (t + 1) * NP;        /* du_t */
        /* from y_t */
        for (int64_t n = 0; n < N; ++n)
            for (int64_t p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int64_t r = 0; r < R; ++r) acc += Cm[(bth * R + r) * N + n] * dy[(bth * R + r) * P + p];
                g[n * P + p] += acc;
            }
        for (int64_t r = 0; r < R; ++r)
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t p = 0; p < P; ++p) acc += hc[n * P + p] * dy[(bth * R + r) * P + p];
                dC[(bth * R + r) * N + n] = acc;
            }
        /* h_t = R(theta) z + gamma u_t */
        double dgamma = 0.0;
        for (int64_t e = 0; e < NP; ++e) {
            dgamma += g[e] * uc[e];
            duc[e] += gamma * g[e];
        }
        for (int64_t k = 0; k < K; ++k) {
            const double phi = theta ? theta[bth * K + k] : 0.0;
            const double c = cos(phi), s = sin(phi);
            double dth = 0.0;
            for (int64_t p = 0; p < P; ++p) {
                const double g0 = g[(2 * k) * P + p], g1 = g[(2 * k + 1) * P + p];
                dz[(2 * k) * P + p] = c * g0 + s * g1;          /* R(-phi) g */
                dz[(2 * k + 1) * P + p] = -s * g0 + c * g1;
                const double w0 = hc[(2 * k) * P + p] - gamma * uc[(2 * k) * P + p];
                const double w1 = hc[(2 * k + 1) * P + p] - gamma * uc[(2 * k + 1) * P + p];
                dth += -g0 * w1 + g1 * w0;
            }
            if (dtheta) dtheta[bth * K + k] = dth;
        }
        /* z = alpha h_{t-1} + beta u_{t-1} */
        double dalpha = 0.0, dbeta = 0.0;
        for (int64_t e = 0; e < NP; ++e) {
            dalpha += dz[e] * hp[e];
            dbeta += dz[e] * up[e];
            dup[e] += beta * dz[e];
            g[e] = alpha * dz[e];                 /* dL/dh_{t-1} */
        }
        /* u_t = sum_r B_t[r] x_t[r]^T: du_t is complete now */
        for (int64_t r = 0; r < R; ++r) {
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t p = 0; p < P; ++p) acc += duc[n * P + p] * x[(bth * R + r) * P + p];
                dB[(bth * R + r) * N + n] = acc;
            }
            for (int64_t p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) acc += duc[n * P + p] * Bm[(bth * R + r) * N + n];
                dx[(bth * R + r) * P + p] = acc;
            }
        }
        /* the scalars */
        ddt[bth] = dalpha * alpha * A_h + dbeta * (1.0 - l) * alpha * (1.0 + d * A_h) + dgamma * l;
        if (dlam) dlam[bth] = -dbeta * d * alpha + dgamma * d;
        dA_acc += dalpha * alpha * d + dbeta * (1.0 - l) * d * d * alpha;
    }
    dA_bh[unit] = dA_acc;
    if (dh0) memcpy(dh0 + unit * NP, g, (size_t)NP * sizeof(double));
    if (prevB && (dprevB || dprevx)) {
        const double* dum = du;   /* du_{-1} */
        for (int64_t r = 0; r < R; ++r) {
            if (dprevB)
                for (int64_t n = 0; n < N; ++n) {
                    double acc = 0.0;
                    for (int64_t p = 0; p < P; ++p) acc += dum[n * P + p] * prevx[(unit * R + r) * P + p];
                    dprevB[(unit * R + r) * N + n] = acc;
                }
            if (dprevx)
                for (int64_t p = 0; p < P; ++p) {
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n) acc += dum[n * P + p] * prevB[(unit * R + r) * N + n];
                    dprevx[(unit * R + r) * P + p] = acc;
                }
        }
    }
}

/* Gradient of the whole scan over all (b, h).  Returns 0, -1 on bad arguments,
 * -2 on allocation failure. */
int oracle_scan_bwd_f64(int64_t batch, int64_t T, int64_t H, int64_t P, int64_t N, int64_t R,
                        const double* x, const double* dt, const double* A, const double* Bm, const double* Cm,
                        const double* lam, const double* theta, const double* h0, const double* prevB,
                        const double* prevx, const double* dy, const double* dfinal, double* dx, double* ddt,
                        double* dB, double* dC, double* dlam, double* dtheta, double* dA_bh, double* dh0,
                        double* dprevB, double* dprevx, int nthreads) {
    if (batch < 0 || T < 0 || H <= 0 || P <= 0 || N <= 0 || (N % 2) != 0 || R <= 0) return -1;
    if (!dt || !A || !dA_bh || (T > 0 && (!x || !Bm || !Cm || !dy || !dx || !ddt || !dB || !dC))) return -1;
    if ((prevB == NULL) != (prevx == NULL)) return -1;
    const int64_t units = batch * H, NP = N * P;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t unit = 0; unit < units; ++unit) {
        const int64_t b = unit / H, h = unit % H;
        double* hs = (double*)malloc((size_t)((T + 1) * NP) * sizeof(double));
        double* us = (double*)malloc((size_t)((T + 1) * NP) * sizeof(double));
        double* du = (double*)malloc((size_t)((T + 1) * NP) * sizeof(double));
        double* g = (double*)malloc((size_t)NP * sizeof(double));
        double* dz = (double*)malloc((size_t)NP * sizeof(double));
        if (!hs || !us || !du || !g || !dz) {
            failed |= 1;
        } else {
            bwd_sequence(T, H, P, N, R, b, h, x, dt, A[h], Bm, Cm, lam, theta, h0, prevB, prevx, dy, dfinal, dx,
                         ddt, dB, dC, dlam, dtheta, dA_bh, dh0, dprevB, dprevx, hs, us, g, dz, du);
        }
        free(hs);
        free(us);
        free(du);
        free(g);
        free(dz);
    }
    return failed ? -2 : 0;
}
