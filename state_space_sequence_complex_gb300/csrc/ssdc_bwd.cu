// Backward pass of the chunkwise complex SSD in exact fp32 on the SIMT cores
// (page "Extending -- SSM variants & Triton kernels", Step 3: the backward
// recomputes the forward and is seeded with the true output gradients).
//
// Gradient convention: a complex gradient holds dL/dRe in its real part and
// dL/dIm in its imaginary part, so a holomorphic step w = f(z) gives
// dz += conj(f'(z)) dw, and a product w = u v gives du += dw conj(v).
//
// Chunked form. With Acs the in-chunk cumulative log-decay (landing page,
// "03 Chunkwise SSD"), L[t,l] = exp(Acs[t] - Acs[l]) (t >= l),
// dec[l] = exp(Acs[Q-1] - Acs[l]), C'[t] = exp(Acs[t]) C[t], P = (C B^T) o L,
// and R_c the gradient of the state that leaves chunk c:
//   U_c      = C'^H dY                         (gradient of S_in[c] from y)
//   R_{c-1}  = conj(a_c) R_c + U_c,  R_{nc-1} = d_final_state,
//   d_initial_state = conj(a_0) R_0 + U_0
//   W[t,l]   = sum_d dY[t,d] conj(x[l,d]),  V = W o conj(L)
//   dX       = P^H dY + conj(dec o B) R_c
//   dB       = V^T conj(C) + conj(dec) o (conj(x) R_c^T)
//   dC       = V conj(B) + conj(exp(Acs)) o (dY S_in^H)
// and, for the log-decay z_t = softplus(dt_t) A of token t of chunk c,
//   dz_t = <R_c, S_out(c)> + sum_{t' >= t in chunk c} r_t',
//   r_t  = <dC_t, C_t> - <dB_t, B_t>,  <u, v> = sum u conj(v),
// S_out(c) the state leaving chunk c (S_in[c+1], or the final state). This
// follows from dz_t = <g_t, A_bar_t s_{t-1}> = <g_t, s_t> - <dB_t, B_t>, from
// <g_t, s_t> - <g_{t+1}, s_{t+1}> = <dy_t, y_t> - <dB_{t+1}, B_{t+1}> with
// <dy_t, y_t> = <dC_t, C_t>, and from g = R_c + conj(C) (outer) dy at the
// chunk's last token. Anchoring every chunk keeps each sum within Q tokens,
// so fp32 rounding in r_t does not accumulate along the sequence.
//
// Kernels, in launch order after the forward chunk-state kernel and state
// pass have put S_in[c], a_c and the final state in the workspace:
//   ssdc_bwd_chunk_adjoint  grid (nc, H, B)            U_c into the R slots
//   ssdc_adjoint_pass       grid (ceil(N*D/256), B*H)  R_c in place, d_initial_state
//   ssdc_bwd_chunk          grid (nc * ceil(Q/64), H, B) dx, dB_t, dC_t, r_t,
//                                                       <R_c, S_out(c)>
//   ssdc_bwd_dt             grid (H)                   dz -> ddt, dA
#include <cuda_runtime.h>

#include "ssdc_common.cuh"
#include "ssdc_kernels.h"

namespace ssdc {

constexpr int kBwdThreads = 256;
constexpr int kRows = 64;  // token rows per shared-memory block
constexpr int kCols = 64;  // max N, D

struct Plane2 {
    float re[kRows][kCols + 1];  // one float of padding against bank conflicts
    float im[kRows][kCols + 1];
};

__device__ __forceinline__ int chunk_valid(const Problem& p, int64_t t0) {
    return (int)(p.T - t0 < (int64_t)p.Q ? p.T - t0 : (int64_t)p.Q);
}

// Rows [r0, r0 + 64) of one chunk of a (B, T, H, F) plane pair into dst,
// zero past the chunk's valid tokens (`valid`), past F and past the chunk.
// im may be null (a zero imaginary plane).
__device__ __forceinline__ void load_rows(Plane2& dst, const float* __restrict__ re,
                                          const float* __restrict__ im, int64_t bt0, int H, int h,
                                          int F, int r0, int valid) {
    for (int e = threadIdx.x; e < kRows * kCols; e += kBwdThreads) {
        const int r = e / kCols, f = e % kCols;
        float vr = 0.0f, vi = 0.0f;
        if (r0 + r < valid && f < F) {
            const int64_t o = ((bt0 + r0 + r) * H + h) * (int64_t)F + f;
            vr = re[o];
            vi = im != nullptr ? im[o] : 0.0f;
        }
        dst.re[r][f] = vr;
        dst.im[r][f] = vi;
    }
}

// A per-chunk (D, N) state slot [2][D][N] into dst as dst[d][n].
__device__ __forceinline__ void load_state(Plane2& dst, const float* __restrict__ slot, int D, int N) {
    const float* si = slot + (int64_t)D * N;
    for (int e = threadIdx.x; e < kRows * kCols; e += kBwdThreads) {
        const int d = e / kCols, n = e % kCols;
        const bool ok = d < D && n < N;
        dst.re[d][n] = ok ? slot[d * N + n] : 0.0f;
        dst.im[d][n] = ok ? si[d * N + n] : 0.0f;
    }
}

// ---------------------------------------------------------------------------
// U_c^T[d, n] = sum_l dY[l, d] conj(C'[l, n]), C'[l] = exp(Acs[l]) C[l].

struct AdjSmem {
    Acs acs[kMaxQ];
    Plane2 dy, cc;  // dY rows; C' rows
};

__global__ void __launch_bounds__(kBwdThreads)
ssdc_bwd_chunk_adjoint(GradProblem g, Workspace ws, GradWorkspace gw) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    AdjSmem& sm = *reinterpret_cast<AdjSmem*>(smem_raw);
    const Problem& p = g.f;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int Q = p.Q, N = p.N, D = p.D, H = p.H;
    const int64_t t0 = (int64_t)c * Q;
    const int valid = chunk_valid(p, t0);
    const int tid = threadIdx.x;
    const int64_t bt0 = (int64_t)b * p.T + t0;

    if (tid < 32)
        chunk_cumsum_warp(p.dt + bt0 * H + h, H, valid, Q, p.A_re[h], p.A_im[h], sm.acs);

    const int dg = tid / 16, ng = tid % 16;  // micro-tile: d = dg + 16 i, n = ng + 16 j
    float ur[4][4], ui[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) ur[i][j] = ui[i][j] = 0.0f;

    for (int r0 = 0; r0 < Q; r0 += kRows) {
        const int rows = min(kRows, Q - r0);
        __syncthreads();  // the cumsum is written; the previous block's reads are done
        load_rows(sm.dy, g.dy_re, g.dy_im, bt0, H, h, D, r0, valid);
        load_rows(sm.cc, p.C_re, p.C_im, bt0, H, h, N, r0, valid);
        __syncthreads();
        for (int e = tid; e < rows * kCols; e += kBwdThreads) {
            const int r = e / kCols, n = e % kCols;
            if (r0 + r < valid && n < N) {
                const float2 v = cmul(make_float2(sm.cc.re[r][n], sm.cc.im[r][n]),
                                      cexp_exact(acs_value(sm.acs[r0 + r])));
                sm.cc.re[r][n] = v.x;
                sm.cc.im[r][n] = v.y;
            }
        }
        __syncthreads();
        for (int l = 0; l < rows; ++l) {
            float yr[4], yi[4], cr[4], ci[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                yr[i] = sm.dy.re[l][dg + 16 * i];
                yi[i] = sm.dy.im[l][dg + 16 * i];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                cr[j] = sm.cc.re[l][ng + 16 * j];
                ci[j] = sm.cc.im[l][ng + 16 * j];
            }
            // dY conj(C')
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ur[i][j] = fmaf(yr[i], cr[j], fmaf(yi[i], ci[j], ur[i][j]));
                    ui[i][j] = fmaf(yi[i], cr[j], fmaf(-yr[i], ci[j], ui[i][j]));
                }
        }
    }

    const int64_t chunk = ((int64_t)b * H + h) * p.nc + c;
    float* Rr = gw.R + chunk * 2 * D * N;
    float* Ri = Rr + (int64_t)D * N;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = dg + 16 * i, n = ng + 16 * j;
            if (d < D && n < N) {
                Rr[d * N + n] = ur[i][j];
                Ri[d * N + n] = ui[i][j];
            }
        }
}

// ---------------------------------------------------------------------------
// Reverse state pass: one thread per complex (d, n) lane of one (b, h)
// sequence walks the chunks from last to first, replacing U_c in its slot by
// R_c (the gradient of the state leaving chunk c).

constexpr int kAdjAhead = 8;

__global__ void __launch_bounds__(kPassThreads)
ssdc_adjoint_pass(GradProblem g, Workspace ws, GradWorkspace gw) {
    const Problem& p = g.f;
    const int64_t bh = blockIdx.y;
    const int ND = p.N * p.D;
    const int j = blockIdx.x * kPassThreads + threadIdx.x;  // lane = d * N + n
    if (j >= ND) return;
    const int64_t nc = p.nc;
    float* R = gw.R + bh * nc * 2 * ND + j;
    const float* a = ws.a + bh * nc * 2;
    const int d = j / p.N, n = j % p.N;
    const int64_t o = (bh * p.N + n) * p.D + d;  // (b, h, n, d) of the state gradients
    float rr = 0.0f, ri = 0.0f;
    if (g.dfs_re != nullptr) {
        rr = g.dfs_re[o];
        ri = g.dfs_im[o];
    }
    for (int64_t c1 = nc - 1; c1 >= 0; c1 -= kAdjAhead) {
        float ur[kAdjAhead], ui[kAdjAhead], ar[kAdjAhead], ai[kAdjAhead];
#pragma unroll
        for (int k = 0; k < kAdjAhead; ++k) {
            const int64_t c = c1 - k;
            if (c >= 0) {
                const float* s = R + c * 2 * ND;
                ur[k] = __ldcg(s);
                ui[k] = __ldcg(s + ND);
                ar[k] = __ldg(a + 2 * c);
                ai[k] = __ldg(a + 2 * c + 1);
            }
        }
#pragma unroll
        for (int k = 0; k < kAdjAhead; ++k) {
            const int64_t c = c1 - k;
            if (c >= 0) {
                float* s = R + c * 2 * ND;
                __stcg(s, rr);
                __stcg(s + ND, ri);
                // conj(a_c) R_c + U_c
                const float nr = fmaf(ar[k], rr, fmaf(ai[k], ri, ur[k]));
                const float ni = fmaf(ar[k], ri, fmaf(-ai[k], rr, ui[k]));
                rr = nr;
                ri = ni;
            }
        }
    }
    if (g.ds0_re != nullptr) {
        g.ds0_re[o] = rr;
        g.ds0_im[o] = ri;
    }
}

// ---------------------------------------------------------------------------
// dx, dB_t, dC_t and r_t for the 64 token rows of one block `ib` of a chunk.
//   part 1 (rows l of block ib): dX and dB over the token blocks jb >= ib,
//          then the R_c terms;
//   part 2 (rows t of block ib): dC over the blocks jb <= ib, then the S_in
//          term, and r_t.

struct BwdSmem {
    Acs acs[kMaxQ];
    Plane2 own1, own2;  // part 1: B, x of block ib;   part 2: C, dY of block ib
    Plane2 str1, str2;  // part 1: C, dY of block jb;  part 2: B, x of block jb
    Plane2 pv;          // P or V of the block pair, [t][l]
    Plane2 st;          // part 1: R_c^T [d][n];       part 2: S_in^T [d][n]
    float nbb_re[kRows], nbb_im[kRows];  // -<dB_l, B_l> of the rows of block ib
    double anc[kBwdThreads / 32][2];     // per-warp partial sums of <R_c, S_out(c)>
};

__global__ void __launch_bounds__(kBwdThreads)
ssdc_bwd_chunk(GradProblem g, Workspace ws, GradWorkspace gw) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw);
    const Problem& p = g.f;
    const int Q = p.Q, N = p.N, D = p.D, H = p.H;
    const int nb = (Q + kRows - 1) / kRows;
    const int c = blockIdx.x / nb, ib = blockIdx.x % nb;
    const int h = blockIdx.y, b = blockIdx.z;
    const int64_t t0 = (int64_t)c * Q;
    const int valid = chunk_valid(p, t0);
    const int r0 = ib * kRows;
    if (r0 >= valid) return;  // rows entirely past the sequence end
    const int tid = threadIdx.x;
    const int64_t bt0 = (int64_t)b * p.T + t0;
    const int64_t chunk = ((int64_t)b * H + h) * p.nc + c;

    if (tid < 32)
        chunk_cumsum_warp(p.dt + bt0 * H + h, H, valid, Q, p.A_re[h], p.A_im[h], sm.acs);
    load_rows(sm.own1, p.B_re, p.B_im, bt0, H, h, N, r0, valid);
    load_rows(sm.own2, p.x_re, p.x_im, bt0, H, h, D, r0, valid);
    load_state(sm.st, gw.R + chunk * 2 * D * N, D, N);

    const int rg = tid / 16, cg = tid % 16;  // micro-tile: rows rg + 16 i, cols cg + 16 j
    float xr[4][4], xi[4][4], br[4][4], bi[4][4];  // dX[l][d], dB[l][n]
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) xr[i][j] = xi[i][j] = br[i][j] = bi[i][j] = 0.0f;

    // ---- part 1: token blocks jb >= ib (rows t), own rows l
    for (int jb = ib; jb < nb; ++jb) {
        const int s0 = jb * kRows;
        if (s0 >= valid) break;
        const int trows = min(kRows, valid - s0);
        __syncthreads();  // previous pair's reads are done
        load_rows(sm.str1, p.C_re, p.C_im, bt0, H, h, N, s0, valid);
        load_rows(sm.str2, g.dy_re, g.dy_im, bt0, H, h, D, s0, valid);
        __syncthreads();
        // decay factors of the pair: L[t][l] for t = rg + 16 i (block jb), l = cg + 16 j (block ib)
        float lr[4][4], li[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int tt = s0 + rg + 16 * i, ll = r0 + cg + 16 * j;
                float2 v = make_float2(0.0f, 0.0f);
                if (tt >= ll && tt < valid && ll < valid) v = cexp_exact(acs_diff(sm.acs[tt], sm.acs[ll]));
                lr[i][j] = v.x;
                li[i][j] = v.y;
            }
        // P[t][l] = (sum_n C[t,n] B[l,n]) L[t][l]
        {
            float gr[4][4], gi[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) gr[i][j] = gi[i][j] = 0.0f;
            for (int n = 0; n < N; ++n) {
                float cr[4], ci[4], qr[4], qi[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    cr[i] = sm.str1.re[rg + 16 * i][n];
                    ci[i] = sm.str1.im[rg + 16 * i][n];
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    qr[j] = sm.own1.re[cg + 16 * j][n];
                    qi[j] = sm.own1.im[cg + 16 * j][n];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        gr[i][j] = fmaf(cr[i], qr[j], fmaf(-ci[i], qi[j], gr[i][j]));
                        gi[i][j] = fmaf(cr[i], qi[j], fmaf(ci[i], qr[j], gi[i][j]));
                    }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 v = cmul(make_float2(gr[i][j], gi[i][j]), make_float2(lr[i][j], li[i][j]));
                    sm.pv.re[rg + 16 * i][cg + 16 * j] = v.x;
                    sm.pv.im[rg + 16 * i][cg + 16 * j] = v.y;
                }
        }
        __syncthreads();
        // dX[l][d] += sum_t conj(P[t][l]) dY[t][d]
        for (int t = 0; t < trows; ++t) {
            float pr[4], pi[4], yr[4], yi[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                pr[i] = sm.pv.re[t][rg + 16 * i];
                pi[i] = sm.pv.im[t][rg + 16 * i];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                yr[j] = sm.str2.re[t][cg + 16 * j];
                yi[j] = sm.str2.im[t][cg + 16 * j];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    xr[i][j] = fmaf(pr[i], yr[j], fmaf(pi[i], yi[j], xr[i][j]));
                    xi[i][j] = fmaf(pr[i], yi[j], fmaf(-pi[i], yr[j], xi[i][j]));
                }
        }
        __syncthreads();
        // V[t][l] = (sum_d dY[t,d] conj(x[l,d])) conj(L[t][l])
        {
            float wr[4][4], wi[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) wr[i][j] = wi[i][j] = 0.0f;
            for (int d = 0; d < D; ++d) {
                float yr[4], yi[4], qr[4], qi[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    yr[i] = sm.str2.re[rg + 16 * i][d];
                    yi[i] = sm.str2.im[rg + 16 * i][d];
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    qr[j] = sm.own2.re[cg + 16 * j][d];
                    qi[j] = sm.own2.im[cg + 16 * j][d];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        wr[i][j] = fmaf(yr[i], qr[j], fmaf(yi[i], qi[j], wr[i][j]));
                        wi[i][j] = fmaf(yi[i], qr[j], fmaf(-yr[i], qi[j], wi[i][j]));
                    }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 v = cmul(make_float2(wr[i][j], wi[i][j]), make_float2(lr[i][j], -li[i][j]));
                    sm.pv.re[rg + 16 * i][cg + 16 * j] = v.x;
                    sm.pv.im[rg + 16 * i][cg + 16 * j] = v.y;
                }
        }
        __syncthreads();
        // dB[l][n] += sum_t V[t][l] conj(C[t][n])
        for (int t = 0; t < trows; ++t) {
            float vr[4], vi[4], cr[4], ci[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                vr[i] = sm.pv.re[t][rg + 16 * i];
                vi[i] = sm.pv.im[t][rg + 16 * i];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                cr[j] = sm.str1.re[t][cg + 16 * j];
                ci[j] = sm.str1.im[t][cg + 16 * j];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    br[i][j] = fmaf(vr[i], cr[j], fmaf(vi[i], ci[j], br[i][j]));
                    bi[i][j] = fmaf(vi[i], cr[j], fmaf(-vr[i], ci[j], bi[i][j]));
                }
        }
    }

    // R_c terms: dX += conj(dec[l]) sum_n conj(B[l,n]) R[n,d];  dB += conj(dec[l]) sum_d conj(x[l,d]) R[n,d]
    {
        const Acs last = sm.acs[Q - 1];
        float er[4], ei[4];  // conj(dec[l]) of the rows l = rg + 16 i
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 v = cexp_exact(acs_diff(last, sm.acs[min(r0 + rg + 16 * i, Q - 1)]));
            er[i] = v.x;
            ei[i] = -v.y;
        }
        float ar[4][4], ai[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) ar[i][j] = ai[i][j] = 0.0f;
        for (int n = 0; n < N; ++n) {
            float qr[4], qi[4], sr[4], si[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                qr[i] = sm.own1.re[rg + 16 * i][n];
                qi[i] = sm.own1.im[rg + 16 * i][n];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                sr[j] = sm.st.re[cg + 16 * j][n];
                si[j] = sm.st.im[cg + 16 * j][n];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ar[i][j] = fmaf(qr[i], sr[j], fmaf(qi[i], si[j], ar[i][j]));
                    ai[i][j] = fmaf(qr[i], si[j], fmaf(-qi[i], sr[j], ai[i][j]));
                }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 v = cmul(make_float2(er[i], ei[i]), make_float2(ar[i][j], ai[i][j]));
                xr[i][j] += v.x;
                xi[i][j] += v.y;
                ar[i][j] = ai[i][j] = 0.0f;
            }
        for (int d = 0; d < D; ++d) {
            float qr[4], qi[4], sr[4], si[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                qr[i] = sm.own2.re[rg + 16 * i][d];
                qi[i] = sm.own2.im[rg + 16 * i][d];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                sr[j] = sm.st.re[d][cg + 16 * j];
                si[j] = sm.st.im[d][cg + 16 * j];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ar[i][j] = fmaf(qr[i], sr[j], fmaf(qi[i], si[j], ar[i][j]));
                    ai[i][j] = fmaf(qr[i], si[j], fmaf(-qi[i], sr[j], ai[i][j]));
                }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 v = cmul(make_float2(er[i], ei[i]), make_float2(ar[i][j], ai[i][j]));
                br[i][j] += v.x;
                bi[i][j] += v.y;
            }
    }

    // write dX, dB; -<dB_l, B_l> per row into shared memory
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int l = rg + 16 * i;
        const bool row_ok = r0 + l < valid;
        const int64_t tok = (bt0 + r0 + l) * H + h;
        float sr = 0.0f, si = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int f = cg + 16 * j;
            if (row_ok && f < D) {
                g.dx_re[tok * D + f] = xr[i][j];
                if (g.dx_im != nullptr) g.dx_im[tok * D + f] = xi[i][j];
            }
            if (row_ok && f < N) {
                g.dB_re[tok * N + f] = br[i][j];
                g.dB_im[tok * N + f] = bi[i][j];
            }
            // dB conj(B); B is zero past N
            const float qr = sm.own1.re[l][f], qi = sm.own1.im[l][f];
            sr = fmaf(br[i][j], qr, fmaf(bi[i][j], qi, sr));
            si = fmaf(bi[i][j], qr, fmaf(-br[i][j], qi, si));
        }
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) {
            sr += __shfl_xor_sync(0xffffffffu, sr, off);
            si += __shfl_xor_sync(0xffffffffu, si, off);
        }
        if (cg == 0) {
            sm.nbb_re[l] = -sr;
            sm.nbb_im[l] = -si;
        }
    }

    // <R_c, S_out(c)>, once per chunk (row block 0); st holds R_c^T. S_out is the
    // next chunk's S_in ([d][n] slot) or, for the last chunk, the final state (n, d).
    if (ib == 0) {
        const int64_t bh = (int64_t)b * H + h;
        const bool last_chunk = c == p.nc - 1;
        const float* nxt = ws.S + (chunk + 1) * 2 * D * N;
        float ar = 0.0f, ai = 0.0f;
        for (int e = tid; e < D * N; e += kBwdThreads) {
            const int d = e / N, n = e % N;
            float sr, si;
            if (last_chunk) {
                const int64_t o = (bh * N + n) * D + d;
                sr = p.fs_re[o];
                si = p.fs_im[o];
            } else {
                sr = nxt[e];
                si = nxt[(int64_t)D * N + e];
            }
            const float rr = sm.st.re[d][n], ri = sm.st.im[d][n];
            ar = fmaf(rr, sr, fmaf(ri, si, ar));
            ai = fmaf(ri, sr, fmaf(-rr, si, ai));
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            ar += __shfl_xor_sync(0xffffffffu, ar, off);
            ai += __shfl_xor_sync(0xffffffffu, ai, off);
        }
        if ((tid & 31) == 0) {
            sm.anc[tid >> 5][0] = ar;
            sm.anc[tid >> 5][1] = ai;
        }
        __syncthreads();
        if (tid == 0) {
            double sr = 0.0, si = 0.0;
            for (int w = 0; w < kBwdThreads / 32; ++w) {
                sr += sm.anc[w][0];
                si += sm.anc[w][1];
            }
            gw.anchor[2 * chunk] = sr;
            gw.anchor[2 * chunk + 1] = si;
        }
    }

    // ---- part 2: own rows t of block ib, blocks jb <= ib (rows l)
    __syncthreads();
    load_rows(sm.own1, p.C_re, p.C_im, bt0, H, h, N, r0, valid);
    load_rows(sm.own2, g.dy_re, g.dy_im, bt0, H, h, D, r0, valid);
    load_state(sm.st, ws.S + chunk * 2 * D * N, D, N);
    float cr_[4][4], ci_[4][4];  // dC[t][n]
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) cr_[i][j] = ci_[i][j] = 0.0f;
    for (int jb = 0; jb <= ib; ++jb) {
        const int s0 = jb * kRows;
        const int lrows = min(kRows, valid - s0);
        __syncthreads();
        load_rows(sm.str1, p.B_re, p.B_im, bt0, H, h, N, s0, valid);
        load_rows(sm.str2, p.x_re, p.x_im, bt0, H, h, D, s0, valid);
        __syncthreads();
        // V[t][l] = (sum_d dY[t,d] conj(x[l,d])) conj(L[t][l]), t = rg + 16 i (block ib), l = cg + 16 j (block jb)
        {
            float wr[4][4], wi[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) wr[i][j] = wi[i][j] = 0.0f;
            for (int d = 0; d < D; ++d) {
                float yr[4], yi[4], qr[4], qi[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    yr[i] = sm.own2.re[rg + 16 * i][d];
                    yi[i] = sm.own2.im[rg + 16 * i][d];
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    qr[j] = sm.str2.re[cg + 16 * j][d];
                    qi[j] = sm.str2.im[cg + 16 * j][d];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        wr[i][j] = fmaf(yr[i], qr[j], fmaf(yi[i], qi[j], wr[i][j]));
                        wi[i][j] = fmaf(yi[i], qr[j], fmaf(-yr[i], qi[j], wi[i][j]));
                    }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int tt = r0 + rg + 16 * i, ll = s0 + cg + 16 * j;
                    float2 v = make_float2(0.0f, 0.0f);
                    if (tt >= ll && tt < valid && ll < valid) {
                        const float2 L = cexp_exact(acs_diff(sm.acs[tt], sm.acs[ll]));
                        v = cmul(make_float2(wr[i][j], wi[i][j]), make_float2(L.x, -L.y));
                    }
                    sm.pv.re[rg + 16 * i][cg + 16 * j] = v.x;
                    sm.pv.im[rg + 16 * i][cg + 16 * j] = v.y;
                }
        }
        __syncthreads();
        // dC[t][n] += sum_l V[t][l] conj(B[l][n])
        for (int l = 0; l < lrows; ++l) {
            float vr[4], vi[4], qr[4], qi[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                vr[i] = sm.pv.re[rg + 16 * i][l];
                vi[i] = sm.pv.im[rg + 16 * i][l];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                qr[j] = sm.str1.re[l][cg + 16 * j];
                qi[j] = sm.str1.im[l][cg + 16 * j];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    cr_[i][j] = fmaf(vr[i], qr[j], fmaf(vi[i], qi[j], cr_[i][j]));
                    ci_[i][j] = fmaf(vi[i], qr[j], fmaf(-vr[i], qi[j], ci_[i][j]));
                }
        }
    }
    // S_in term: dC[t][n] += conj(exp(Acs[t])) sum_d dY[t,d] conj(S_in[n,d])
    {
        float ar[4][4], ai[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) ar[i][j] = ai[i][j] = 0.0f;
        for (int d = 0; d < D; ++d) {
            float yr[4], yi[4], sr[4], si[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                yr[i] = sm.own2.re[rg + 16 * i][d];
                yi[i] = sm.own2.im[rg + 16 * i][d];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                sr[j] = sm.st.re[d][cg + 16 * j];
                si[j] = sm.st.im[d][cg + 16 * j];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ar[i][j] = fmaf(yr[i], sr[j], fmaf(yi[i], si[j], ar[i][j]));
                    ai[i][j] = fmaf(yi[i], sr[j], fmaf(-yr[i], si[j], ai[i][j]));
                }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 e = cexp_exact(acs_value(sm.acs[min(r0 + rg + 16 * i, Q - 1)]));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 v = cmul(make_float2(e.x, -e.y), make_float2(ar[i][j], ai[i][j]));
                cr_[i][j] += v.x;
                ci_[i][j] += v.y;
            }
        }
    }
    // write dC and r_t = <dC_t, C_t> - <dB_t, B_t>
    const int64_t bh = (int64_t)b * H + h;
    float* rre = gw.r + bh * 2 * p.T;
    float* rim = rre + p.T;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = rg + 16 * i;
        const bool row_ok = r0 + t < valid;
        const int64_t tok = (bt0 + r0 + t) * H + h;
        float sr = 0.0f, si = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = cg + 16 * j;
            if (row_ok && n < N) {
                g.dC_re[tok * N + n] = cr_[i][j];
                g.dC_im[tok * N + n] = ci_[i][j];
            }
            const float qr = sm.own1.re[t][n], qi = sm.own1.im[t][n];
            sr = fmaf(cr_[i][j], qr, fmaf(ci_[i][j], qi, sr));
            si = fmaf(ci_[i][j], qr, fmaf(-cr_[i][j], qi, si));
        }
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) {
            sr += __shfl_xor_sync(0xffffffffu, sr, off);
            si += __shfl_xor_sync(0xffffffffu, si, off);
        }
        if (cg == 0 && row_ok) {
            rre[t0 + r0 + t] = sr + sm.nbb_re[t];
            rim[t0 + r0 + t] = si + sm.nbb_im[t];
        }
    }
}

// ---------------------------------------------------------------------------
// dz_t = <R_c, S_out(c)> + sum_{t' >= t in chunk c} r_t' (fp64), then
// ddt_t = Re(dz_t conj(A)) sigmoid(dt_t) and dA = sum_{b,t} softplus(dt_t) dz_t.
// One CTA per head; its threads take the (b, chunk) pairs of the head in turn.

constexpr int kDtThreads = kBwdDtThreads;

__global__ void __launch_bounds__(kDtThreads)
ssdc_bwd_dt(GradProblem g, Workspace ws, GradWorkspace gw) {
    __shared__ double red[kDtThreads / 32][2];
    const Problem& p = g.f;
    const int h = blockIdx.x, tid = threadIdx.x;
    const int H = p.H, Q = p.Q;
    const int64_t T = p.T, nc = p.nc;
    const float Ar = p.A_re[h], Ai = p.A_im[h];
    double dAr = 0.0, dAi = 0.0;
    for (int64_t k = tid; k < (int64_t)p.B * nc; k += kDtThreads) {
        const int64_t b = k / nc, c = k % nc;
        const int64_t bh = b * H + h;
        const int64_t chunk = bh * nc + c;
        const int64_t t0 = c * Q;
        const int valid = (int)(T - t0 < (int64_t)Q ? T - t0 : (int64_t)Q);
        const float* rre = gw.r + bh * 2 * T;
        const float* rim = rre + T;
        double zr = gw.anchor[2 * chunk], zi = gw.anchor[2 * chunk + 1];
        for (int l = valid - 1; l >= 0; --l) {
            const int64_t t = t0 + l;
            zr += rre[t];
            zi += rim[t];
            const int64_t bth = (b * T + t) * H + h;
            const float v = p.dt[bth];
            const float sig = 1.0f / (1.0f + expf(-v));
            g.ddt[bth] = (float)(zr * Ar + zi * Ai) * sig;
            const double delta = (double)softplus_f(v);
            dAr += delta * zr;
            dAi += delta * zi;
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        dAr += __shfl_xor_sync(0xffffffffu, dAr, off);
        dAi += __shfl_xor_sync(0xffffffffu, dAi, off);
    }
    if ((tid & 31) == 0) {
        red[tid >> 5][0] = dAr;
        red[tid >> 5][1] = dAi;
    }
    __syncthreads();
    if (tid == 0) {
        double sr = 0.0, si = 0.0;
        for (int w = 0; w < kDtThreads / 32; ++w) {
            sr += red[w][0];
            si += red[w][1];
        }
        g.dA_re[h] = (float)sr;
        g.dA_im[h] = (float)si;
    }
}

size_t bwd_adjoint_smem() { return sizeof(AdjSmem); }
size_t bwd_chunk_smem() { return sizeof(BwdSmem); }

}  // namespace ssdc
