/*
 * Oracle for the complex SSD forward: a plain O(T) sequential scan in double
 * precision (complex128). TEST INFRASTRUCTURE ONLY: the tests, the package's
 * smoke check and the bench's CPU-baseline leg use it; the product path never
 * links or calls it, and it shares no code with the CUDA path.
 *
 * What it computes (page "Extending -- SSM variants & Triton kernels",
 * Path A, Step 1, the O(T) naive scan; landing page, "03 Chunkwise SSD",
 * the NAIVE line):
 *
 *   A_bar[b,t,h] = exp(softplus(dt[b,t,h]) * A[h])          (complex)
 *   s[b,h]       = s0[b,h]  (zero unless an initial state is given)
 *   for t = 0 .. T-1:
 *       s[n,d] = A_bar[b,t,h] * s[n,d] + B_t[b,t,h,n] * x[b,t,h,d]
 *       y[b,t,h,d] = sum_n C_t[b,t,h,n] * s[n,d]
 *   final_state[b,h] = s after t = T-1
 *
 * Readings taken where the pages are silent: softplus is log(1 + e^x) with
 * beta = 1 (written as max(x,0) + log1p(e^-|x|)); neither product conjugates;
 * the input term B_t x_t is not scaled by the step; the state starts at zero.
 * The initial-state argument exists only so a test can check that scanning
 * [0,T1) then [T1,T) from the carried state equals the whole scan.
 *
 * Layout: every complex array is planar (separate real and imaginary planes),
 * row-major over the shapes given. Inputs are float32 (the configs fix
 * complex64 inputs); all arithmetic and all outputs are double.
 *
 * Parity pins: every function here is pinned by tests that do not call it to
 * get the expected values (brute-force SSD matrix, closed forms, library IIR
 * filter, invariants, chunk-size invariance of an independent chunkwise form).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const float *x_re, *x_im, *A_re, *A_im, *B_re, *B_im, *C_re, *C_im, *dt;
    const double *s0_re, *s0_im; /* optional initial state (B,H,N,D) */
    int64_t Bn, T, H, N, D;
    int64_t t_y; /* y is written for t < t_y only; the state always runs to T */
    double *y_re, *y_im, *s_re, *s_im;
    int64_t next_job;
    pthread_mutex_t lock;
} job_t;

static double softplus(double v) {
    /* log(1 + e^v), stable for both signs */
    return (v > 0.0 ? v : 0.0) + log1p(exp(-fabs(v)));
}

/* One (b,h) sequence: the recurrence above, in order, nothing fused. */
static void scan_one(const job_t *J, int64_t b, int64_t h, double *sr, double *si) {
    const int64_t T = J->T, H = J->H, N = J->N, D = J->D;
    const double ar = J->A_re[h], ai = J->A_im[h];
    if (J->s0_re) {
        const double *r = J->s0_re + ((b * H + h) * N) * D;
        const double *i = J->s0_im + ((b * H + h) * N) * D;
        memcpy(sr, r, sizeof(double) * N * D);
        memcpy(si, i, sizeof(double) * N * D);
    } else {
        memset(sr, 0, sizeof(double) * N * D);
        memset(si, 0, sizeof(double) * N * D);
    }
    for (int64_t t = 0; t < T; ++t) {
        const int64_t bth = (b * T + t) * H + h;
        /* discretisation: A_bar = exp(delta * A), delta = softplus(dt) */
        const double delta = softplus((double)J->dt[bth]);
        const double mag = exp(delta * ar);
        const double abr = mag * cos(delta * ai);
        const double abi = mag * sin(delta * ai);
        const float *xr = J->x_re + bth * D, *xi = J->x_im + bth * D;
        const float *br = J->B_re + bth * N, *bi = J->B_im + bth * N;
        const float *cr = J->C_re + bth * N, *ci = J->C_im + bth * N;
        /* s = A_bar * s + B_t (outer) x_t */
        for (int64_t n = 0; n < N; ++n) {
            const double bnr = br[n], bni = bi[n];
            double *rr = sr + n * D, *ii = si + n * D;
            for (int64_t d = 0; d < D; ++d) {
                const double sr0 = rr[d], si0 = ii[d];
                const double xdr = xr[d], xdi = xi[d];
                rr[d] = (abr * sr0 - abi * si0) + (bnr * xdr - bni * xdi);
                ii[d] = (abr * si0 + abi * sr0) + (bnr * xdi + bni * xdr);
            }
        }
        /* y_t = sum_n C_t[n] * s[n, :] */
        if (t < J->t_y) {
            double *yr = J->y_re + bth * D, *yi = J->y_im + bth * D;
            for (int64_t d = 0; d < D; ++d) {
                double accr = 0.0, acci = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    const double cnr = cr[n], cni = ci[n];
                    accr += cnr * sr[n * D + d] - cni * si[n * D + d];
                    acci += cnr * si[n * D + d] + cni * sr[n * D + d];
                }
                yr[d] = accr;
                yi[d] = acci;
            }
        }
    }
    double *fr = J->s_re + ((b * H + h) * N) * D;
    double *fi = J->s_im + ((b * H + h) * N) * D;
    memcpy(fr, sr, sizeof(double) * N * D);
    memcpy(fi, si, sizeof(double) * N * D);
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    double *sr = (double *)malloc(sizeof(double) * J->N * J->D);
    double *si = (double *)malloc(sizeof(double) * J->N * J->D);
    if (!sr || !si) {
        free(sr);
        free(si);
        return (void *)1;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int64_t j = J->next_job++;
        pthread_mutex_unlock(&J->lock);
        if (j >= J->Bn * J->H) break;
        scan_one(J, j / J->H, j % J->H, sr, si);
    }
    free(sr);
    free(si);
    return NULL;
}

/*
 * Returns 0 on success, -1 on bad arguments, -2 if a thread or buffer could
 * not be created. y must hold B*T*H*D doubles per plane (only t < t_y rows are
 * written), the state B*H*N*D per plane. s0_re/s0_im may be NULL.
 */
int ssd_oracle_naive(const float *x_re, const float *x_im, const float *A_re,
                     const float *A_im, const float *B_re, const float *B_im,
                     const float *C_re, const float *C_im, const float *dt,
                     const double *s0_re, const double *s0_im, int64_t Bn,
                     int64_t T, int64_t H, int64_t N, int64_t D, int64_t t_y,
                     double *y_re, double *y_im, double *s_re, double *s_im,
                     int nthreads) {
    if (Bn <= 0 || T <= 0 || H <= 0 || N <= 0 || D <= 0 || nthreads <= 0) return -1;
    if ((s0_re == NULL) != (s0_im == NULL)) return -1;
    job_t J;
    J.x_re = x_re; J.x_im = x_im; J.A_re = A_re; J.A_im = A_im;
    J.B_re = B_re; J.B_im = B_im; J.C_re = C_re; J.C_im = C_im; J.dt = dt;
    J.s0_re = s0_re; J.s0_im = s0_im;
    J.Bn = Bn; J.T = T; J.H = H; J.N = N; J.D = D;
    J.t_y = t_y < T ? t_y : T;
    J.y_re = y_re; J.y_im = y_im; J.s_re = s_re; J.s_im = s_im;
    J.next_job = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads > Bn * H) nthreads = (int)(Bn * H);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    int rc = 0, started = 0;
    if (!th) rc = -2;
    for (int i = 0; rc == 0 && i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) {
            rc = -2;
            break;
        }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret != NULL) rc = -2;
    }
    if (rc == 0 && started == 0) rc = -2;
    free(th);
    pthread_mutex_destroy(&J.lock);
    return rc;
}
