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
 * ssd_oracle_naive_bwd (end of this file) gives the gradients of that scan
 * with respect to every input, by the adjoint of the same recurrence (the
 * pages' training path; page "Extending -- SSM variants & Triton kernels",
 * Step 3, the autograd wrapper seeded with the true output gradients).
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

/* ------------------------------------------------------------------------
 * Backward pass (gradients) of the scan above, by the adjoint of the
 * recurrence, in double precision. TEST INFRASTRUCTURE ONLY.
 *
 * Convention for complex gradients (the one PyTorch uses for complex
 * tensors): for a real loss L and a complex quantity z, the gradient dz holds
 * dL/dRe(z) in its real part and dL/dIm(z) in its imaginary part. For a
 * holomorphic step w = f(z) this gives dz += conj(f'(z)) * dw.
 *
 * Given dy (B,T,H,D) and d_final_state (B,H,N,D), with g the gradient of the
 * state s_t (N x D):
 *   g = d_final_state
 *   for t = T-1 .. 0:
 *       g[n,d] += conj(C_t[n]) * dy_t[d]                  (y_t = C_t s_t)
 *       dC_t[n]  = sum_d dy_t[d] * conj(s_t[n,d])
 *       dx_t[d]  = sum_n g[n,d] * conj(B_t[n])             (B_t (outer) x_t)
 *       dB_t[n]  = sum_d g[n,d] * conj(x_t[d])
 *       dz_t     = sum_{n,d} g[n,d] * conj(A_bar_t s_{t-1}[n,d])   (also returned)
 *                  (z_t = delta_t A the log-decay, ds_t/dz_t = A_bar_t s_{t-1})
 *       ddt_t    = Re(dz_t * conj(A)) * sigmoid(dt_t)     (delta = softplus(dt))
 *       dA      += delta_t * dz_t                          (summed over b and t)
 *       g        = conj(A_bar_t) * g                       (s_t = A_bar_t s_{t-1} + ...)
 *   d_initial_state = g
 * The states s_t are those of the forward scan, kept for every t.
 * ---------------------------------------------------------------------- */
typedef struct {
    const float *x_re, *x_im, *A_re, *A_im, *B_re, *B_im, *C_re, *C_im, *dt;
    const float *dy_re, *dy_im, *dfs_re, *dfs_im; /* dfs may be NULL: zero */
    const double *s0_re, *s0_im;                  /* may be NULL: zero */
    int64_t Bn, T, H, N, D;
    double *dx_re, *dx_im, *dB_re, *dB_im, *dC_re, *dC_im, *ddt;
    double *dAp_re, *dAp_im; /* per (b,h) partial sums of dA */
    double *ds0_re, *ds0_im; /* (B,H,N,D) */
    double *dz_re, *dz_im;   /* (B,T,H): gradient of the log-decay z_t */
    int64_t next_job;
    pthread_mutex_t lock;
} bjob_t;

static double sigmoid(double v) {
    return v >= 0.0 ? 1.0 / (1.0 + exp(-v)) : exp(v) / (1.0 + exp(v));
}

/* One (b,h) sequence. st holds (T+1) states of N*D complex values:
 * st[0] = s_{-1}, st[t+1] = s_t. */
static void grad_one(const bjob_t *J, int64_t b, int64_t h, double *str, double *sti,
                     double *gr, double *gi) {
    const int64_t T = J->T, H = J->H, N = J->N, D = J->D, ND = N * D;
    const double Ar = J->A_re[h], Ai = J->A_im[h];
    const int64_t bh = b * H + h;
    /* forward, keeping every state */
    if (J->s0_re) {
        memcpy(str, J->s0_re + bh * ND, sizeof(double) * ND);
        memcpy(sti, J->s0_im + bh * ND, sizeof(double) * ND);
    } else {
        memset(str, 0, sizeof(double) * ND);
        memset(sti, 0, sizeof(double) * ND);
    }
    for (int64_t t = 0; t < T; ++t) {
        const int64_t bth = (b * T + t) * H + h;
        const double delta = softplus((double)J->dt[bth]);
        const double mag = exp(delta * Ar);
        const double abr = mag * cos(delta * Ai), abi = mag * sin(delta * Ai);
        const float *xr = J->x_re + bth * D, *xi = J->x_im + bth * D;
        const float *br = J->B_re + bth * N, *bi = J->B_im + bth * N;
        const double *pr = str + t * ND, *pi = sti + t * ND;
        double *qr = str + (t + 1) * ND, *qi = sti + (t + 1) * ND;
        for (int64_t n = 0; n < N; ++n)
            for (int64_t d = 0; d < D; ++d) {
                const int64_t k = n * D + d;
                qr[k] = (abr * pr[k] - abi * pi[k]) + ((double)br[n] * xr[d] - (double)bi[n] * xi[d]);
                qi[k] = (abr * pi[k] + abi * pr[k]) + ((double)br[n] * xi[d] + (double)bi[n] * xr[d]);
            }
    }
    /* backward */
    if (J->dfs_re) {
        for (int64_t k = 0; k < ND; ++k) {
            gr[k] = J->dfs_re[bh * ND + k];
            gi[k] = J->dfs_im[bh * ND + k];
        }
    } else {
        memset(gr, 0, sizeof(double) * ND);
        memset(gi, 0, sizeof(double) * ND);
    }
    double dAr = 0.0, dAi = 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
        const int64_t bth = (b * T + t) * H + h;
        const double delta = softplus((double)J->dt[bth]);
        const double mag = exp(delta * Ar);
        const double abr = mag * cos(delta * Ai), abi = mag * sin(delta * Ai);
        const float *xr = J->x_re + bth * D, *xi = J->x_im + bth * D;
        const float *br = J->B_re + bth * N, *bi = J->B_im + bth * N;
        const float *cr = J->C_re + bth * N, *ci = J->C_im + bth * N;
        const float *yr = J->dy_re + bth * D, *yi = J->dy_im + bth * D;
        const double *sr = str + (t + 1) * ND, *si = sti + (t + 1) * ND; /* s_t */
        const double *pr = str + t * ND, *pi = sti + t * ND;             /* s_{t-1} */
        /* g += conj(C_t) (outer) dy_t */
        for (int64_t n = 0; n < N; ++n)
            for (int64_t d = 0; d < D; ++d) {
                const int64_t k = n * D + d;
                gr[k] += (double)cr[n] * yr[d] + (double)ci[n] * yi[d];
                gi[k] += (double)cr[n] * yi[d] - (double)ci[n] * yr[d];
            }
        /* dC_t[n] = sum_d dy_t[d] conj(s_t[n,d]) */
        for (int64_t n = 0; n < N; ++n) {
            double ar = 0.0, ai = 0.0;
            for (int64_t d = 0; d < D; ++d) {
                const int64_t k = n * D + d;
                ar += yr[d] * sr[k] + yi[d] * si[k];
                ai += yi[d] * sr[k] - yr[d] * si[k];
            }
            J->dC_re[bth * N + n] = ar;
            J->dC_im[bth * N + n] = ai;
        }
        /* dx_t[d] = sum_n g[n,d] conj(B_t[n]) */
        for (int64_t d = 0; d < D; ++d) {
            double ar = 0.0, ai = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const int64_t k = n * D + d;
                ar += gr[k] * br[n] + gi[k] * bi[n];
                ai += gi[k] * br[n] - gr[k] * bi[n];
            }
            J->dx_re[bth * D + d] = ar;
            J->dx_im[bth * D + d] = ai;
        }
        /* dB_t[n] = sum_d g[n,d] conj(x_t[d]) */
        for (int64_t n = 0; n < N; ++n) {
            double ar = 0.0, ai = 0.0;
            for (int64_t d = 0; d < D; ++d) {
                const int64_t k = n * D + d;
                ar += gr[k] * xr[d] + gi[k] * xi[d];
                ai += gi[k] * xr[d] - gr[k] * xi[d];
            }
            J->dB_re[bth * N + n] = ar;
            J->dB_im[bth * N + n] = ai;
        }
        /* dz_t = sum g conj(A_bar_t s_{t-1}) */
        double zr = 0.0, zi = 0.0;
        for (int64_t k = 0; k < ND; ++k) {
            const double ur = abr * pr[k] - abi * pi[k];
            const double ui = abr * pi[k] + abi * pr[k];
            zr += gr[k] * ur + gi[k] * ui;
            zi += gi[k] * ur - gr[k] * ui;
        }
        J->dz_re[bth] = zr;
        J->dz_im[bth] = zi;
        J->ddt[bth] = (zr * Ar + zi * Ai) * sigmoid((double)J->dt[bth]);
        dAr += delta * zr;
        dAi += delta * zi;
        /* g = conj(A_bar_t) g */
        for (int64_t k = 0; k < ND; ++k) {
            const double r = gr[k], i = gi[k];
            gr[k] = abr * r + abi * i;
            gi[k] = abr * i - abi * r;
        }
    }
    J->dAp_re[bh] = dAr;
    J->dAp_im[bh] = dAi;
    if (J->ds0_re) {
        memcpy(J->ds0_re + bh * ND, gr, sizeof(double) * ND);
        memcpy(J->ds0_im + bh * ND, gi, sizeof(double) * ND);
    }
}

static void *grad_worker(void *arg) {
    bjob_t *J = (bjob_t *)arg;
    const size_t ND = (size_t)(J->N * J->D);
    const size_t sts = (size_t)(J->T + 1) * ND;
    double *str = (double *)malloc(sizeof(double) * sts);
    double *sti = (double *)malloc(sizeof(double) * sts);
    double *gr = (double *)malloc(sizeof(double) * ND);
    double *gi = (double *)malloc(sizeof(double) * ND);
    void *ret = NULL;
    if (!str || !sti || !gr || !gi) {
        ret = (void *)1;
    } else {
        for (;;) {
            pthread_mutex_lock(&J->lock);
            const int64_t j = J->next_job++;
            pthread_mutex_unlock(&J->lock);
            if (j >= J->Bn * J->H) break;
            grad_one(J, j / J->H, j % J->H, str, sti, gr, gi);
        }
    }
    free(str);
    free(sti);
    free(gr);
    free(gi);
    return ret;
}

/*
 * Gradients of the scan. Inputs as for ssd_oracle_naive plus dy (B,T,H,D)
 * and d_final_state (B,H,N,D, may be NULL for zero). Outputs (double):
 * dx (B,T,H,D), dA (H), dB and dC (B,T,H,N), ddt (B,T,H), dz (B,T,H), the
 * gradient of each token's log-decay z_t = softplus(dt_t) A, and, when
 * ds0_re / ds0_im are not NULL, d_initial_state (B,H,N,D). dA sums the (b,h)
 * partials in order of b. Returns 0, -1 on bad arguments, -2 when out of threads or
 * memory.
 */
int ssd_oracle_naive_bwd(const float *x_re, const float *x_im, const float *A_re,
                         const float *A_im, const float *B_re, const float *B_im,
                         const float *C_re, const float *C_im, const float *dt,
                         const double *s0_re, const double *s0_im, const float *dy_re,
                         const float *dy_im, const float *dfs_re, const float *dfs_im,
                         int64_t Bn, int64_t T, int64_t H, int64_t N, int64_t D,
                         double *dx_re, double *dx_im, double *dA_re, double *dA_im,
                         double *dB_re, double *dB_im, double *dC_re, double *dC_im,
                         double *ddt, double *ds0_re, double *ds0_im, double *dz_re,
                         double *dz_im, int nthreads) {
    if (Bn <= 0 || T <= 0 || H <= 0 || N <= 0 || D <= 0 || nthreads <= 0) return -1;
    if (dz_re == NULL || dz_im == NULL) return -1;
    if ((s0_re == NULL) != (s0_im == NULL) || (dfs_re == NULL) != (dfs_im == NULL) ||
        (ds0_re == NULL) != (ds0_im == NULL))
        return -1;
    bjob_t J;
    J.x_re = x_re; J.x_im = x_im; J.A_re = A_re; J.A_im = A_im;
    J.B_re = B_re; J.B_im = B_im; J.C_re = C_re; J.C_im = C_im; J.dt = dt;
    J.dy_re = dy_re; J.dy_im = dy_im; J.dfs_re = dfs_re; J.dfs_im = dfs_im;
    J.s0_re = s0_re; J.s0_im = s0_im;
    J.Bn = Bn; J.T = T; J.H = H; J.N = N; J.D = D;
    J.dx_re = dx_re; J.dx_im = dx_im; J.dB_re = dB_re; J.dB_im = dB_im;
    J.dC_re = dC_re; J.dC_im = dC_im; J.ddt = ddt;
    J.ds0_re = ds0_re; J.ds0_im = ds0_im;
    J.dz_re = dz_re; J.dz_im = dz_im;
    J.dAp_re = (double *)calloc((size_t)(Bn * H), sizeof(double));
    J.dAp_im = (double *)calloc((size_t)(Bn * H), sizeof(double));
    J.next_job = 0;
    if (!J.dAp_re || !J.dAp_im) {
        free(J.dAp_re);
        free(J.dAp_im);
        return -2;
    }
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads > Bn * H) nthreads = (int)(Bn * H);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    int rc = 0, started = 0;
    if (!th) rc = -2;
    for (int i = 0; rc == 0 && i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, grad_worker, &J) != 0) {
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
    if (rc == 0) {
        for (int64_t h = 0; h < H; ++h) {
            double ar = 0.0, ai = 0.0;
            for (int64_t b = 0; b < Bn; ++b) {
                ar += J.dAp_re[b * H + h];
                ai += J.dAp_im[b * H + h];
            }
            dA_re[h] = ar;
            dA_im[h] = ai;
        }
    }
    free(th);
    free(J.dAp_re);
    free(J.dAp_im);
    pthread_mutex_destroy(&J.lock);
    return rc;
}
