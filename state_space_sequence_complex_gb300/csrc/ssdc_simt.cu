// Exact-fp32 SIMT kernels of the chunkwise complex SSD forward (the checking
// variant). Every product and sum is an fp32 FMA on the CUDA cores; decays use
// the accurate expf / sincosf. Landing page, "03 Chunkwise SSD": the CHUNK
// line (L, Y_diag) and the STATE line (per-chunk state).
//
// Launches (the state pass between them is csrc/ssdc_pass.cu):
//   ssdc_simt_chunk_state  grid (nc, H, B), 256 threads: S_loc and a_c of one
//                          chunk, 4 x 4 complex register tiles
//   ssdc_simt_chunk_scan   grid (nc * ceil(Q/64), H, B), 512 threads: 64 output
//                          rows of a chunk, Y_diag + Y_off, 4 x 2 complex
//                          register tiles (a warp owns 4 consecutive rows)
// Operands sit in shared memory as interleaved complex tiles (ssdc_tiles.cuh).
// Both kernels are templates on N and D: N = D = 64 compiles with constant
// loop bounds, other sizes read them from the problem.
#include <cuda_runtime.h>

#include "ssdc_common.cuh"
#include "ssdc_kernels.h"
#include "ssdc_tiles.cuh"

namespace ssdc {

constexpr int kStateThreads = 256;
constexpr int kScanThreads = 512;
constexpr int kScanWarps = kScanThreads / 32;

// Shared-memory plan of the chunk-state kernel.
struct StateSmem {
    Acs acs[kMaxQ];
    CTile x, db;  // x rows; dec[s] * B rows
};

// S_loc^T[d, n] = sum_s x[s, d] * dec[s] * B[s, n]; a_c = exp(Acs[Q-1]).
template <int kN, int kD>
__global__ void __launch_bounds__(kStateThreads)
ssdc_simt_chunk_state(Problem p, Workspace ws) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    StateSmem& sm = *reinterpret_cast<StateSmem*>(smem_raw);
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int Q = p.Q, H = p.H;
    const int N = kN > 0 ? kN : p.N, D = kD > 0 ? kD : p.D;
    const int64_t t0 = (int64_t)c * Q;
    const int valid = chunk_valid(p, t0);
    const int tid = threadIdx.x;
    const int64_t bt0 = (int64_t)b * p.T + t0;

    if (tid < 32)
        chunk_cumsum_warp(p.dt + bt0 * H + h, H, valid, Q, p.A_re[h], p.A_im[h], sm.acs);

    const int dg = tid / 16, ng = tid % 16;  // micro-tile: d = dg + 16 i, n = ng + 16 j
    float2 acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

    for (int r0 = 0; r0 < Q; r0 += kRows) {
        const int rows = min(kRows, Q - r0);
        __syncthreads();  // the cumsum is written; the previous block's reads are done
        load_rows<kStateThreads>(sm.x, p.x_re, p.x_im, bt0, H, h, D, r0, valid);
        load_rows<kStateThreads>(sm.db, p.B_re, p.B_im, bt0, H, h, N, r0, valid);
        __syncthreads();
        const Acs last = sm.acs[Q - 1];
        for (int e = tid; e < rows * kCols; e += kStateThreads) {
            const int r = e / kCols, n = e % kCols;
            if (r0 + r < valid && n < N)
                sm.db.v[r][n] = cmul(cexp_exact(acs_diff(last, sm.acs[r0 + r])), sm.db.v[r][n]);
        }
        __syncthreads();
#pragma unroll 4
        for (int s = 0; s < rows; ++s) {
            float2 u[4], w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) u[i] = sm.x.v[s][dg + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = sm.db.v[s][ng + 16 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) cmac(acc[i][j], u[i], w[j]);
        }
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
                Sr[d * N + n] = acc[i][j].x;
                Si[d * N + n] = acc[i][j].y;
            }
        }
    if (tid == 0) {
        const float2 a = cexp_exact(acs_value(sm.acs[Q - 1]));
        ws.a[2 * chunk] = a.x;
        ws.a[2 * chunk + 1] = a.y;
    }
}

// Shared-memory plan of the chunk-scan kernel.
struct ScanSmem {
    Acs acs[kMaxQ];
    CTile cc;  // C rows of the l-block (later C o exp(Acs))
    CTile bb;  // B rows of an s-block
    CTile xx;  // x rows of an s-block
    CTile pv;  // P = (C B^T) o L of the block pair, [l][s]
    CTile st;  // S_in^T [d][n]
};

// y[l, :] = sum_{s <= l} P[l, s] x[s, :] + (C o exp(Acs))[l, :] S_in,
// P = (C B^T) o L, for the 64 rows l of one l-block of one chunk.
template <int kN, int kD>
__global__ void __launch_bounds__(kScanThreads)
ssdc_simt_chunk_scan(Problem p, Workspace ws) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ScanSmem& sm = *reinterpret_cast<ScanSmem*>(smem_raw);
    constexpr int NT = kScanThreads;
    const int Q = p.Q, H = p.H;
    const int N = kN > 0 ? kN : p.N, D = kD > 0 ? kD : p.D;
    const int lblocks = (Q + kRows - 1) / kRows;
    const int c = blockIdx.x / lblocks, lb = blockIdx.x % lblocks;
    const int h = blockIdx.y, b = blockIdx.z;
    const int64_t t0 = (int64_t)c * Q;
    const int valid = chunk_valid(p, t0);
    const int l0 = lb * kRows;
    if (l0 >= valid) return;  // rows entirely past the sequence end
    const int tid = threadIdx.x;
    const int64_t bt0 = (int64_t)b * p.T + t0;
    const int64_t chunk = ((int64_t)b * H + h) * p.nc + c;
    // micro-tile: rows rb + i (i < 4), cols cg + 32 j (j < 2). The warps sharing a
    // scheduler (w mod 4) get strips k, 7-k, 8+k, 15-k, so the causal loop below
    // gives every scheduler the same work.
    const int warp = tid >> 5, cg = tid & 31;
    const int wk = warp & 3, wm = warp >> 2;
    const int rb = 4 * (wm == 0 ? wk : wm == 1 ? 7 - wk : wm == 2 ? 8 + wk : 15 - wk);

    if (tid < 32)
        chunk_cumsum_warp(p.dt + bt0 * H + h, H, valid, Q, p.A_re[h], p.A_im[h], sm.acs);
    load_rows<NT>(sm.cc, p.C_re, p.C_im, bt0, H, h, N, l0, valid);
    load_state<NT>(sm.st, ws.S + chunk * 2 * D * N, D, N);

    float2 y[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) y[i][j] = make_float2(0.0f, 0.0f);

    for (int sb = 0; sb <= lb; ++sb) {
        const int s0 = sb * kRows;
        const int srows = min(kRows, valid - s0);
        __syncthreads();  // previous block's reads are done
        load_rows<NT>(sm.bb, p.B_re, p.B_im, bt0, H, h, N, s0, valid);
        load_rows<NT>(sm.xx, p.x_re, p.x_im, bt0, H, h, D, s0, valid);
        __syncthreads();
        // P[l][s] = (sum_n C[l, n] B[s, n]) L[l][s], l = rb + i, s = cg + 32 j
        {
            float2 G[4][2];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) G[i][j] = make_float2(0.0f, 0.0f);
#pragma unroll 8
            for (int n = 0; n < N; ++n) {
                float2 a[4], q[2];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = sm.cc.v[rb + i][n];
#pragma unroll
                for (int j = 0; j < 2; ++j) q[j] = sm.bb.v[cg + 32 * j][n];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 2; ++j) cmac(G[i][j], a[i], q[j]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int ll = l0 + rb + i, ss = s0 + cg + 32 * j;
                    float2 v = make_float2(0.0f, 0.0f);
                    if (ll >= ss && ll < valid && ss < valid)
                        v = cmul(G[i][j], cexp_exact(acs_diff(sm.acs[ll], sm.acs[ss])));
                    sm.pv.v[rb + i][cg + 32 * j] = v;
                }
        }
        __syncthreads();
        // Y += P x; on the diagonal block pair P[l][s] = 0 for s > l, so a warp stops after
        // its last row
        const int s_hi = sb == lb ? min(srows, rb + 4) : srows;
#pragma unroll 4
        for (int s = 0; s < s_hi; ++s) {
            float2 a[4], q[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = sm.pv.v[rb + i][s];
#pragma unroll
            for (int j = 0; j < 2; ++j) q[j] = sm.xx.v[s][cg + 32 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) cmac(y[i][j], a[i], q[j]);
        }
    }

    // Y_off = (C o exp(Acs)) S_in: sum_n C[l, n] S_in[n, d], scaled by exp(Acs[l]) per row
    {
        float2 acc[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) acc[i][j] = make_float2(0.0f, 0.0f);
#pragma unroll 8
        for (int n = 0; n < N; ++n) {
            float2 a[4], q[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = sm.cc.v[rb + i][n];
#pragma unroll
            for (int j = 0; j < 2; ++j) q[j] = sm.st.v[cg + 32 * j][n];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) cmac(acc[i][j], a[i], q[j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 e = cexp_exact(acs_value(sm.acs[min(l0 + rb + i, Q - 1)]));
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float2 v = cmul(e, acc[i][j]);
                y[i][j].x += v.x;
                y[i][j].y += v.y;
            }
        }
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int l = rb + i;
        if (l0 + l >= valid) continue;
        const int64_t row = ((bt0 + l0 + l) * H + h) * D;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int d = cg + 32 * j;
            if (d < D) {
                p.y_re[row + d] = y[i][j].x;
                p.y_im[row + d] = y[i][j].y;
            }
        }
    }
}

cudaError_t simt_set_smem_attrs() {
    const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e = cudaFuncSetAttribute(ssdc_simt_chunk_state<0, 0>, a, (int)sizeof(StateSmem));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ssdc_simt_chunk_state<64, 64>, a, (int)sizeof(StateSmem));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ssdc_simt_chunk_scan<0, 0>, a, (int)sizeof(ScanSmem));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ssdc_simt_chunk_scan<64, 64>, a, (int)sizeof(ScanSmem));
    return e;
}

void simt_launch_chunk_state(const Problem& p, const Workspace& ws, cudaStream_t stream) {
    const dim3 grid((unsigned)p.nc, (unsigned)p.H, (unsigned)p.B);
    if (p.N == 64 && p.D == 64)
        ssdc_simt_chunk_state<64, 64><<<grid, kStateThreads, sizeof(StateSmem), stream>>>(p, ws);
    else
        ssdc_simt_chunk_state<0, 0><<<grid, kStateThreads, sizeof(StateSmem), stream>>>(p, ws);
}

void simt_launch_chunk_scan(const Problem& p, const Workspace& ws, cudaStream_t stream) {
    const int lblocks = (p.Q + kRows - 1) / kRows;
    const dim3 grid((unsigned)(p.nc * lblocks), (unsigned)p.H, (unsigned)p.B);
    if (p.N == 64 && p.D == 64)
        ssdc_simt_chunk_scan<64, 64><<<grid, kScanThreads, sizeof(ScanSmem), stream>>>(p, ws);
    else
        ssdc_simt_chunk_scan<0, 0><<<grid, kScanThreads, sizeof(ScanSmem), stream>>>(p, ws);
}

}  // namespace ssdc
