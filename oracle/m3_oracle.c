/*
 * m3_oracle.c -- fp64 sequential oracle for the Mamba-3 selective SSM scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this library.  It shares
 * no code, header or constant with the CUDA library, and the CUDA library
 * never calls it.
 *
 * What it computes (primary form, the "complex frame"):
 *
 *   For every (batch b, head h) independently, starting from the state h'_{-1}
 *   (zero for a prefill) and the previous-token input u_{-1} (zero for a
 *   prefill), for t = 0 .. T-1:
 *
 *     alpha_t = exp(dt_t * A_h)                       Mamba-3 summary, §3.1.1,
 *     beta_t  = (1 - lambda_t) * dt_t * alpha_t       eq. (5)-(6) and the
 *     gamma_t = lambda_t * dt_t                       coefficient table
 *     u_t     = sum_r B_t[r] x_t[r]^T          (N x P; MIMO, §3.3: B X^T)
 *     h'_t    = R(theta_t) (alpha_t h'_{t-1} + beta_t u_{t-1}) + gamma_t u_t
 *     y_t[r]  = C_t[r]^T h'_t                  (P per rank column r)
 *
 *   R(theta_t) is block diagonal with one 2x2 rotation per state pair
 *   (2k, 2k+1), k < N/2 (Mamba-3 summary, §3.2.1, Proposition 3.2.1: a complex
 *   state of size N/2 is a real state of size N with 2x2 rotation blocks):
 *
 *     (a, b) -> (a cos phi - b sin phi,  a sin phi + b cos phi),  phi = theta_t[k]
 *
 *   i.e. multiplication of (a + i b) by exp(i phi).  This is the exponential-
 *   trapezoidal rule of eq. (5) applied to the complex system of §3.2
 *   (A -> A + i theta): the factor exp(dt (A + i theta)) multiplies both the
 *   previous state and the previous-token input, and theta_t is the per-step
 *   angle (it already contains dt).  With theta = 0 and lambda = 1 this is the
 *   Mamba-2 update h = alpha h + dt B x^T (same page, §2.2, and the special
 *   cases listed under eq. (6)).
 *
 *   The state exposed (final_state) is h'_{T-1} in this complex frame.  The
 *   data-dependent RoPE form of Propositions 3.2.2 / 3.2.3 keeps instead
 *   h_t = R(Phi_t)^T h'_t with Phi_t = sum_{i<=t} theta_i; both give the same
 *   y_t.  The RoPE form is written separately in forms.py.
 *
 * Layouts (C-contiguous, fp64):
 *   x     [b, T, h, R, P]      dt, lambda [b, T, h]     A [h]
 *   B, C  [b, T, h, R, N]      theta      [b, T, h, N/2]
 *   h0    [b, h, N, P]         prevB [b, h, R, N]       prevx [b, h, R, P]
 *   y     [b, T, h, R, P]      hT    [b, h, N, P]
 * lambda == NULL means lambda = 1; theta == NULL means theta = 0;
 * h0 / prevB / prevx == NULL mean zero (a prefill from the empty state).
 * Arithmetic is plain fp64 in the order written, one (b, h) pair per OpenMP
 * iteration; nothing is blocked or reordered inside a sequence.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One (b, h) sequence.  hs (N*P) holds the state on entry and on exit; u_prev
 * (N*P) holds the previous token's B X^T on entry and on exit; u is scratch. */
static void run_sequence(int64_t T, int64_t H, int64_t P, int64_t N, int64_t R,
                         int64_t b, int64_t h,
                         const double* x, const double* dt, double A_h,
                         const double* Bm, const double* Cm, const double* lam,
                         const double* theta, double* hs, double* u_prev,
                         double* u, double* y) {
    const int64_t K = N / 2;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t bth = (b * T + t) * H + h;           /* index into [b,T,h] */
        const double d = dt[bth];
        const double l = lam ? lam[bth] : 1.0;
        const double alpha = exp(d * A_h);
        const double beta = (1.0 - l) * d * alpha;
        const double gamma = l * d;

        /* u_t = sum_r B_t[r] x_t[r]^T */
        const double* Bt = Bm + bth * R * N;
        const double* xt = x + bth * R * P;
        for (int64_t n = 0; n < N; ++n)
            for (int64_t p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int64_t r = 0; r < R; ++r) acc += Bt[r * N + n] * xt[r * P + p];
                u[n * P + p] = acc;
            }

        /* h'_t = R(theta_t)(alpha h'_{t-1} + beta u_{t-1}) + gamma u_t */
        for (int64_t k = 0; k < K; ++k) {
            const double phi = theta ? theta[bth * K + k] : 0.0;
            const double c = cos(phi), s = sin(phi);
            double* h0r = hs + (2 * k) * P;
            double* h1r = hs + (2 * k + 1) * P;
            const double* up0 = u_prev + (2 * k) * P;
            const double* up1 = u_prev + (2 * k + 1) * P;
            const double* u0 = u + (2 * k) * P;
            const double* u1 = u + (2 * k + 1) * P;
            for (int64_t p = 0; p < P; ++p) {
                const double z0 = alpha * h0r[p] + beta * up0[p];
                const double z1 = alpha * h1r[p] + beta * up1[p];
                h0r[p] = c * z0 - s * z1 + gamma * u0[p];
                h1r[p] = s * z0 + c * z1 + gamma * u1[p];
            }
        }

        /* y_t[r] = C_t[r]^T h'_t */
        const double* Ct = Cm + bth * R * N;
        double* yt = y + bth * R * P;
        for (int64_t r = 0; r < R; ++r)
            for (int64_t p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) acc += Ct[r * N + n] * hs[n * P + p];
                yt[r * P + p] = acc;
            }

        memcpy(u_prev, u, (size_t)(N * P) * sizeof(double));
    }
}

/* Full scan over all (b, h) sequences.  Returns 0 on success, -1 on bad
 * arguments, -2 on allocation failure.  A decode step is this call with
 * T = 1, h0 = the current state and (prevB, prevx) = the previous token's
 * B and x. */
int oracle_scan_f64(int64_t batch, int64_t T, int64_t H, int64_t P, int64_t N, int64_t R,
                    const double* x, const double* dt, const double* A,
                    const double* Bm, const double* Cm, const double* lam,
                    const double* theta, const double* h0, const double* prevB,
                    const double* prevx, double* y, double* hT, int nthreads) {
    if (batch < 0 || T < 0 || H <= 0 || P <= 0 || N <= 0 || (N % 2) != 0 || R <= 0) return -1;
    if (!dt || !A || !y || !hT || (T > 0 && (!x || !Bm || !Cm))) return -1;
    const int64_t units = batch * H;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t unit = 0; unit < units; ++unit) {
        const int64_t b = unit / H, h = unit % H;
        double* hs = (double*)malloc((size_t)(N * P) * sizeof(double));
        double* up = (double*)malloc((size_t)(N * P) * sizeof(double));
        double* u = (double*)malloc((size_t)(N * P) * sizeof(double));
        if (!hs || !up || !u) {
            failed |= 1;
        } else {
            if (h0) memcpy(hs, h0 + unit * N * P, (size_t)(N * P) * sizeof(double));
            else memset(hs, 0, (size_t)(N * P) * sizeof(double));
            /* u_{-1} = sum_r prevB[r] prevx[r]^T (zero when no carry is given) */
            for (int64_t n = 0; n < N; ++n)
                for (int64_t p = 0; p < P; ++p) {
                    double acc = 0.0;
                    if (prevB && prevx)
                        for (int64_t r = 0; r < R; ++r)
                            acc += prevB[(unit * R + r) * N + n] * prevx[(unit * R + r) * P + p];
                    up[n * P + p] = acc;
                }
            run_sequence(T, H, P, N, R, b, h, x, dt, A[h], Bm, Cm, lam, theta, hs, up, u, y);
            memcpy(hT + unit * N * P, hs, (size_t)(N * P) * sizeof(double));
        }
        free(hs);
        free(up);
        free(u);
    }
    return failed ? -2 : 0;
}
