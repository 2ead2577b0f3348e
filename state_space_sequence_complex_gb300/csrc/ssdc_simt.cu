// Exact-fp32 SIMT kernels of the chunkwise complex SSD forward (the checking
// variant). Every product and sum is an fp32 FMA on the CUDA cores; decays use
// the accurate expf / sincosf. Landing page, "03 Chunkwise SSD": the CHUNK
// line (L, Y_diag) and the STATE line (per-chunk state).
//
// Launch shapes (one CTA of 256 threads each):
//   ssdc_simt_chunk_state  grid (nc, H, B): S_loc and a_c of one chunk
//   ssdc_simt_chunk_scan   grid (nc * ceil(Q/64), H, B): 64 output rows of a
//                          chunk, Y_diag + Y_off
// Register micro-tiles are 4 x 4 complex outputs per thread.
#include <cuda_runtime.h>

#include "ssdc_common.cuh"
#include "ssdc_kernels.h"

namespace ssdc {

constexpr int kSimtThreads = 256;
constexpr int kBlk = 64;  // rows per smem block along tokens
constexpr int kMaxF = 64;  // max N, D (rows padded by one float against bank conflicts)

// Shared-memory plan of the chunk-state kernel (floats).
struct StateSmem {
    Acs acs[kMaxQ];
    float xr[kBlk][kMaxF + 1], xi[kBlk][kMaxF + 1];  // x rows of one s-block
    float br[kBlk][kMaxF + 1], bi[kBlk][kMaxF + 1];  // dec[s] * B[s, n]
};

// S_loc^T[d, n] = sum_s x[s, d] * dec[s] * B[s, n]; a_c = exp(Acs[Q-1]).
__global__ void __launch_bounds__(kSimtThreads)
ssdc_simt_chunk_state(Problem p, Workspace ws) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    StateSmem& sm = *reinterpret_cast<StateSmem*>(smem_raw);
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int Q = p.Q, N = p.N, D = p.D, H = p.H;
    const int64_t t0 = (int64_t)c * Q;
    const int nvalid = (int)(p.T - t0 < (int64_t)Q ? p.T - t0 : (int64_t)Q);
    const int tid = threadIdx.x;
    if (c == 0 && h == 0 && b == 0 && tid == 0) *ws.status = SSDC_OK;

    if (tid < 32)
        chunk_cumsum_warp(p.dt + ((int64_t)b * p.T + t0) * H + h, H, nvalid, Q,
                          p.A_re[h], p.A_im[h], sm.acs);
    __syncthreads();
    const Acs last = sm.acs[Q - 1];

    // thread micro-tile: d = dg + 16 i, n = ng + 16 j
    const int dg = tid / 16, ng = tid % 16;
    float accr[4][4], acci[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) accr[i][j] = acci[i][j] = 0.0f;

    for (int s0 = 0; s0 < Q; s0 += kBlk) {
        const int rows = min(kBlk, Q - s0);
        // stage x and dec * B for rows [s0, s0 + rows)
        for (int e = tid; e < rows * D; e += kSimtThreads) {
            const int s = e / D, d = e % D;
            const int64_t t = t0 + s0 + s;
            float vr = 0.0f, vi = 0.0f;
            if (s0 + s < nvalid) {
                const int64_t o = ((int64_t)b * p.T + t) * H * D + (int64_t)h * D + d;
                vr = p.x_re[o];
                vi = p.x_im != nullptr ? p.x_im[o] : 0.0f;  // real x: no imaginary plane
            }
            sm.xr[s][d] = vr;
            sm.xi[s][d] = vi;
        }
        for (int e = tid; e < rows * N; e += kSimtThreads) {
            const int s = e / N, n = e % N;
            const int64_t t = t0 + s0 + s;
            float vr = 0.0f, vi = 0.0f;
            if (s0 + s < nvalid) {
                const int64_t o = ((int64_t)b * p.T + t) * H * N + (int64_t)h * N + n;
                const float2 dec = cexp_exact(acs_diff(last, sm.acs[s0 + s]));
                const float2 v = cmul(dec, make_float2(p.B_re[o], p.B_im[o]));
                vr = v.x;
                vi = v.y;
            }
            sm.br[s][n] = vr;
            sm.bi[s][n] = vi;
        }
        __syncthreads();
        for (int s = 0; s < rows; ++s) {
            float xr[4], xi[4], br[4], bi[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int d = dg + 16 * i;
                xr[i] = d < D ? sm.xr[s][d] : 0.0f;
                xi[i] = d < D ? sm.xi[s][d] : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = ng + 16 * j;
                br[j] = n < N ? sm.br[s][n] : 0.0f;
                bi[j] = n < N ? sm.bi[s][n] : 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    accr[i][j] = fmaf(xr[i], br[j], fmaf(-xi[i], bi[j], accr[i][j]));
                    acci[i][j] = fmaf(xr[i], bi[j], fmaf(xi[i], br[j], acci[i][j]));
                }
        }
        __syncthreads();
    }

    const int64_t chunk = ((int64_t)b * H + h) * p.nc + c;
    float* Sr = ws.S + chunk * 2 * D * N;
    float* Si = Sr + (int64_t)D * N;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = dg + 16 * i, n = ng + 16 * j;
            if (d < D && n < N) {
                Sr[d * N + n] = accr[i][j];
                Si[d * N + n] = acci[i][j];
            }
        }
    if (tid == 0) {
        const float2 a = cexp_exact(acs_value(last));
        ws.a[2 * chunk] = a.x;
        ws.a[2 * chunk + 1] = a.y;
    }
}

// Shared-memory plan of the chunk-scan kernel.
struct ScanSmem {
    Acs acs[kMaxQ];
    float cr[kBlk][kMaxF + 1], ci[kBlk][kMaxF + 1];   // C rows of the l-block (later C o exp(Acs))
    float br[kBlk][kMaxF + 1], bi[kBlk][kMaxF + 1];   // B rows of an s-block (later S_in^T)
    float xr[kBlk][kMaxF + 1], xi[kBlk][kMaxF + 1];   // x rows of an s-block
    float pr[kBlk][kBlk + 1], pi[kBlk][kBlk + 1];  // P = (C B^T) o L of the block pair
};

// y[l, :] = sum_{s <= l} P[l, s] x[s, :] + (C o exp(Acs))[l, :] S_in,
// P = (C B^T) o L, for the 64 rows l of one l-block of one chunk.
__global__ void __launch_bounds__(kSimtThreads)
ssdc_simt_chunk_scan(Problem p, Workspace ws) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ScanSmem& sm = *reinterpret_cast<ScanSmem*>(smem_raw);
    const int Q = p.Q, N = p.N, D = p.D, H = p.H;
    const int lblocks = (Q + kBlk - 1) / kBlk;
    const int c = blockIdx.x / lblocks, lb = blockIdx.x % lblocks;
    const int h = blockIdx.y, b = blockIdx.z;
    const int64_t t0 = (int64_t)c * Q;
    const int nvalid = (int)(p.T - t0 < (int64_t)Q ? p.T - t0 : (int64_t)Q);
    const int l0 = lb * kBlk;
    const int lrows = min(kBlk, Q - l0);
    const int tid = threadIdx.x;
    if (l0 >= nvalid) return;  // rows entirely past the sequence end

    if (tid < 32)
        chunk_cumsum_warp(p.dt + ((int64_t)b * p.T + t0) * H + h, H, nvalid, Q,
                          p.A_re[h], p.A_im[h], sm.acs);
    for (int e = tid; e < lrows * N; e += kSimtThreads) {
        const int l = e / N, n = e % N;
        float vr = 0.0f, vi = 0.0f;
        if (l0 + l < nvalid) {
            const int64_t o = ((int64_t)b * p.T + t0 + l0 + l) * H * N + (int64_t)h * N + n;
            vr = p.C_re[o];
            vi = p.C_im[o];
        }
        sm.cr[l][n] = vr;
        sm.ci[l][n] = vi;
    }

    const int rg = tid / 16, cg = tid % 16;  // micro-tile: rows rg + 16 i, cols cg + 16 j
    float yr[4][4], yi[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) yr[i][j] = yi[i][j] = 0.0f;

    for (int sb = 0; sb <= lb; ++sb) {
        const int s0 = sb * kBlk;
        const int srows = min(kBlk, Q - s0);
        __syncthreads();  // previous block's smem reads are done
        for (int e = tid; e < srows * N; e += kSimtThreads) {
            const int s = e / N, n = e % N;
            float vr = 0.0f, vi = 0.0f;
            if (s0 + s < nvalid) {
                const int64_t o = ((int64_t)b * p.T + t0 + s0 + s) * H * N + (int64_t)h * N + n;
                vr = p.B_re[o];
                vi = p.B_im[o];
            }
            sm.br[s][n] = vr;
            sm.bi[s][n] = vi;
        }
        for (int e = tid; e < srows * D; e += kSimtThreads) {
            const int s = e / D, d = e % D;
            float vr = 0.0f, vi = 0.0f;
            if (s0 + s < nvalid) {
                const int64_t o = ((int64_t)b * p.T + t0 + s0 + s) * H * D + (int64_t)h * D + d;
                vr = p.x_re[o];
                vi = p.x_im != nullptr ? p.x_im[o] : 0.0f;  // real x: no imaginary plane
            }
            sm.xr[s][d] = vr;
            sm.xi[s][d] = vi;
        }
        __syncthreads();
        // P[l, s] = (sum_n C[l, n] B[s, n]) * exp(Acs[l] - Acs[s]) for l >= s
        {
            float gr[4][4], gi[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) gr[i][j] = gi[i][j] = 0.0f;
            for (int n = 0; n < N; ++n) {
                float cr[4], ci[4], br[4], bi[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    cr[i] = sm.cr[rg + 16 * i][n];
                    ci[i] = sm.ci[rg + 16 * i][n];
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    br[j] = sm.br[cg + 16 * j][n];
                    bi[j] = sm.bi[cg + 16 * j][n];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        gr[i][j] = fmaf(cr[i], br[j], fmaf(-ci[i], bi[j], gr[i][j]));
                        gi[i][j] = fmaf(cr[i], bi[j], fmaf(ci[i], br[j], gi[i][j]));
                    }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int l = rg + 16 * i, s = cg + 16 * j;
                    float2 v = make_float2(0.0f, 0.0f);
                    if (l0 + l >= s0 + s && l < lrows && s < srows) {
                        const float2 L = cexp_exact(acs_diff(sm.acs[l0 + l], sm.acs[s0 + s]));
                        v = cmul(make_float2(gr[i][j], gi[i][j]), L);
                    }
                    sm.pr[l][s] = v.x;
                    sm.pi[l][s] = v.y;
                }
        }
        __syncthreads();
        // Y += P x
        for (int s = 0; s < srows; ++s) {
            float pr[4], pi[4], xr[4], xi[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                pr[i] = sm.pr[rg + 16 * i][s];
                pi[i] = sm.pi[rg + 16 * i][s];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int d = cg + 16 * j;
                xr[j] = d < D ? sm.xr[s][d] : 0.0f;
                xi[j] = d < D ? sm.xi[s][d] : 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    yr[i][j] = fmaf(pr[i], xr[j], fmaf(-pi[i], xi[j], yr[i][j]));
                    yi[i][j] = fmaf(pr[i], xi[j], fmaf(pi[i], xr[j], yi[i][j]));
                }
        }
    }
    __syncthreads();

    // Y_off: C' = C o exp(Acs[l]) in place, S_in^T into the B buffer
    const int64_t chunk = ((int64_t)b * H + h) * p.nc + c;
    const float* Sr = ws.S + chunk * 2 * D * N;
    const float* Si = Sr + (int64_t)D * N;
    for (int e = tid; e < D * N; e += kSimtThreads) {
        const int d = e / N, n = e % N;
        sm.br[d][n] = Sr[e];
        sm.bi[d][n] = Si[e];
    }
    for (int e = tid; e < lrows * N; e += kSimtThreads) {
        const int l = e / N, n = e % N;
        const float2 g = cexp_exact(acs_value(sm.acs[l0 + l]));
        const float2 v = cmul(make_float2(sm.cr[l][n], sm.ci[l][n]), g);
        sm.cr[l][n] = v.x;
        sm.ci[l][n] = v.y;
    }
    __syncthreads();
    for (int n = 0; n < N; ++n) {
        float cr[4], ci[4], sr[4], si[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            cr[i] = sm.cr[rg + 16 * i][n];
            ci[i] = sm.ci[rg + 16 * i][n];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = cg + 16 * j;
            sr[j] = d < D ? sm.br[d][n] : 0.0f;
            si[j] = d < D ? sm.bi[d][n] : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                yr[i][j] = fmaf(cr[i], sr[j], fmaf(-ci[i], si[j], yr[i][j]));
                yi[i][j] = fmaf(cr[i], si[j], fmaf(ci[i], sr[j], yi[i][j]));
            }
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int l = rg + 16 * i;
        if (l >= lrows || l0 + l >= nvalid) continue;
        const int64_t row = (((int64_t)b * p.T + t0 + l0 + l) * H + h) * D;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = cg + 16 * j;
            if (d < D) {
                p.y_re[row + d] = yr[i][j];
                p.y_im[row + d] = yi[i][j];
            }
        }
    }
}

size_t simt_state_smem() { return sizeof(StateSmem); }
size_t simt_scan_smem() { return sizeof(ScanSmem); }

}  // namespace ssdc
