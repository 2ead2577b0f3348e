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
// Kernels, in launch order:
//   ssdc_bwd_chunk_states  grid (nc, H, B)             S_loc[c], a_c (the forward's,
//                                                      recomputed) and U_c per chunk
//   ssdc_bwd_passes        grid (2 ceil(N*D/256), B*H) S_in[c] and the final state;
//                                                      R_c and d_initial_state
//   ssdc_bwd_chunk         grid (nc * ceil(Q/64), H, B), 512 threads: dx, dB_t, dC_t, r_t,
//                                                      <R_c, S_out(c)>
//   ssdc_bwd_dt            grid (B*H*nc / 8)           dz -> ddt and each chunk's share of dA
//   ssdc_bwd_dA            grid (H)                    dA
#include <cuda_runtime.h>

#include "ssdc_common.cuh"
#include "ssdc_kernels.h"
#include "ssdc_tiles.cuh"

namespace ssdc {

constexpr int kBwdThreads = 256;

// ---------------------------------------------------------------------------
// Per chunk: the forward's local state S_loc^T[d, n] = sum_s x[s, d] dec[s] B[s, n]
// and a_c = exp(Acs[Q-1]) (recomputed), then U_c^T[d, n] = sum_l dY[l, d]
// conj(C'[l, n]), C'[l] = exp(Acs[l]) C[l]. Two tiles, reused by the two halves.

struct StatesSmem {
    Acs acs[kMaxQ];
    CTile a, b;  // x and dec o B; then dY and C'
};

template <int kN, int kD>
__global__ void __launch_bounds__(kBwdThreads)
ssdc_bwd_chunk_states(GradProblem g, Workspace ws, GradWorkspace gw) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    StatesSmem& sm = *reinterpret_cast<StatesSmem*>(smem_raw);
    const Problem& p = g.f;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int Q = p.Q, H = p.H;
    const int N = kN > 0 ? kN : p.N, D = kD > 0 ? kD : p.D;  // compile-time at the production shape
    const int64_t t0 = (int64_t)c * Q;
    const int valid = chunk_valid(p, t0);
    const int tid = threadIdx.x;
    const int64_t bt0 = (int64_t)b * p.T + t0;
    const int64_t chunk = ((int64_t)b * H + h) * p.nc + c;

    if (tid < 32)
        chunk_cumsum_warp(p.dt + bt0 * H + h, H, valid, Q, p.A_re[h], p.A_im[h], sm.acs);

    const int dg = tid / 16, ng = tid % 16;  // micro-tile: d = dg + 16 i, n = ng + 16 j
    for (int half = 0; half < 2; ++half) {
        // half 0: acc = sum_s x[s] (outer) dec[s] B[s];  half 1: acc = sum_l dY[l] (outer) conj(C'[l])
        float2 acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.0f, 0.0f);
        for (int r0 = 0; r0 < Q; r0 += kRows) {
            const int rows = min(kRows, Q - r0);
            __syncthreads();  // the cumsum is written; the previous tiles' reads are done
            if (half == 0) {
                load_rows(sm.a, p.x_re, p.x_im, bt0, H, h, D, r0, valid);
                load_rows(sm.b, p.B_re, p.B_im, bt0, H, h, N, r0, valid);
            } else {
                load_rows(sm.a, g.dy_re, g.dy_im, bt0, H, h, D, r0, valid);
                load_rows(sm.b, p.C_re, p.C_im, bt0, H, h, N, r0, valid);
            }
            __syncthreads();
            const Acs last = sm.acs[Q - 1];
            for (int e = tid; e < rows * kCols; e += kBwdThreads) {
                const int r = e / kCols, n = e % kCols;
                if (r0 + r < valid && n < N) {
                    // dec[s] = exp(Acs[Q-1] - Acs[s]) or exp(Acs[l]), conjugated for C'
                    const float2 f = half == 0 ? cexp_exact(acs_diff(last, sm.acs[r0 + r]))
                                               : conjf2(cexp_exact(acs_value(sm.acs[r0 + r])));
                    const float2 v = sm.b.v[r][n];
                    sm.b.v[r][n] = half == 0 ? cmul(f, v) : cmul(f, conjf2(v));
                }
            }
            __syncthreads();
#pragma unroll 4
            for (int l = 0; l < rows; ++l) {
                float2 u[4], w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) u[i] = sm.a.v[l][dg + 16 * i];
#pragma unroll
                for (int j = 0; j < 4; ++j) w[j] = sm.b.v[l][ng + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) cmac(acc[i][j], u[i], w[j]);
            }
        }
        float* out = (half == 0 ? ws.S : gw.R) + chunk * 2 * D * N;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int d = dg + 16 * i, n = ng + 16 * j;
                if (d < D && n < N) {
                    out[d * N + n] = acc[i][j].x;
                    out[(int64_t)D * N + d * N + n] = acc[i][j].y;
                }
            }
    }
    if (tid == 0) {
        const float2 a = cexp_exact(acs_value(sm.acs[Q - 1]));
        ws.a[2 * chunk] = a.x;
        ws.a[2 * chunk + 1] = a.y;
    }
}

// ---------------------------------------------------------------------------
// The two chunk recurrences, one thread per complex (d, n) lane of one (b, h)
// sequence; the first half of the grid's x blocks runs the forward one, the
// second half the backward one, concurrently. Forwards, S_loc[c] in its slot
// becomes S_in[c] (the forward's state pass, from the initial state) and the
// final state is written; backwards, U_c in its slot becomes R_c (the
// gradient of the state leaving chunk c) and conj(a_0) R_0 + U_0 is the
// initial-state gradient. Both are chain_walk (ssdc_kernels.h): forwards with
// a_c, backwards with conj(a_c).

__global__ void __launch_bounds__(kPassThreads, 4)
ssdc_bwd_passes(GradProblem g, Workspace ws, GradWorkspace gw) {
    grid_dependency_wait();  // launched as a dependent of the kernel before it
    const Problem& p = g.f;
    const int64_t bh = blockIdx.y;
    const int ND = p.N * p.D;
    const int half_blocks = (ND + kPassThreads - 1) / kPassThreads;
    const bool backwards = (int)blockIdx.x >= half_blocks;
    const int j = (blockIdx.x - (backwards ? half_blocks : 0)) * kPassThreads + threadIdx.x;  // d * N + n
    if (j >= ND) return;
    const int64_t nc = p.nc;
    const float* a = ws.a + bh * nc * 2;
    const int d = j / p.N, n = j % p.N;
    const int64_t o = (bh * p.N + n) * p.D + d;  // (b, h, n, d) of the state arrays
    float* X = (backwards ? gw.R : ws.S) + bh * nc * 2 * ND + j;
    const float* x0r = backwards ? g.dfs_re : p.s0_re;
    const float* x0i = backwards ? g.dfs_im : p.s0_im;
    float xr = 0.0f, xi = 0.0f;
    if (x0r != nullptr) {
        xr = x0r[o];
        xi = x0i[o];
    }
    const float2 xo = chain_walk(X, a, nc, ND, backwards, make_float2(xr, xi));
    xr = xo.x;
    xi = xo.y;
    // the final state, or the initial-state gradient conj(a_0) R_0 + U_0
    float* outr = backwards ? g.ds0_re : p.fs_re;
    float* outi = backwards ? g.ds0_im : p.fs_im;
    if (outr != nullptr) {
        outr[o] = xr;
        outi[o] = xi;
    }
}

// ---------------------------------------------------------------------------
// dx, dB_t, dC_t and r_t for the 64 token rows of one block `ib` of a chunk.
//   part 1 (rows l of block ib): dX and dB over the token blocks jb >= ib,
//          then the R_c terms;
//   part 2 (rows t of block ib): dC over the blocks jb <= ib, then the S_in
//          term, and r_t.
// A chunk of one block (Q <= 64) has a single block pair: part 2 then reuses
// part 1's tiles (C, dY, B) and V instead of loading and forming them again.
// 512 threads: each warp owns a strip of 4 consecutive rows of every 64 x 64
// result and lane c its columns c and c + 32, so on the diagonal block pair,
// where P and V vanish above the diagonal, a warp's row sums start (or stop)
// at its rows.

constexpr int kChunkThreads = kBwdChunkThreads;
constexpr int kChunkWarps = kChunkThreads / 32;

struct BwdSmem {
    Acs acs[kMaxQ];
    CTile own1, own2;  // part 1: B, x of block ib;   part 2: C, dY of block ib
    CTile str1, str2;  // part 1: C, dY of block jb;  part 2: B, x of block jb
    CTile pv;          // P or V of the block pair, [t][l]
    CTile st;          // part 1: R_c^T [d][n];       part 2: S_in^T [d][n]
    float2 nbb[kRows];                // -<dB_l, B_l> of the rows of block ib
    double anc[kChunkWarps][2];       // per-warp partial sums of <R_c, S_out(c)>
};

template <int kN, int kD>
__global__ void __launch_bounds__(kChunkThreads)
ssdc_bwd_chunk(GradProblem g, Workspace ws, GradWorkspace gw) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw);
    constexpr int NT = kChunkThreads;
    const Problem& p = g.f;
    const int Q = p.Q, H = p.H;
    const int N = kN > 0 ? kN : p.N, D = kD > 0 ? kD : p.D;  // compile-time at the production shape
    const int nb = (Q + kRows - 1) / kRows;
    const bool single = nb == 1;
    const int c = blockIdx.x / nb, ib = blockIdx.x % nb;
    const int h = blockIdx.y, b = blockIdx.z;
    const int64_t t0 = (int64_t)c * Q;
    const int valid = chunk_valid(p, t0);
    const int r0 = ib * kRows;
    if (r0 >= valid) return;  // rows entirely past the sequence end
    const int tid = threadIdx.x;
    const int64_t bt0 = (int64_t)b * p.T + t0;
    const int64_t chunk = ((int64_t)b * H + h) * p.nc + c;
    // micro-tile: rows rb + i (i < 4), cols cg + 32 j (j < 2). Warp w owns row strip
    // s(w); the causal loops' length grows (or shrinks) with s, and the strips are
    // dealt so that the four warps w, w+4, w+8, w+12 that share a scheduler
    // (w mod 4) get strips k, 7-k, 8+k, 15-k: equal work per scheduler.
    const int warp = tid >> 5, cg = tid & 31;
    const int wk = warp & 3, wm = warp >> 2;
    const int strip = wm == 0 ? wk : wm == 1 ? 7 - wk : wm == 2 ? 8 + wk : 15 - wk;
    const int rb = 4 * strip;

    if (tid < 32)
        chunk_cumsum_warp(p.dt + bt0 * H + h, H, valid, Q, p.A_re[h], p.A_im[h], sm.acs);
    load_rows<NT>(sm.own1, p.B_re, p.B_im, bt0, H, h, N, r0, valid);
    load_rows<NT>(sm.own2, p.x_re, p.x_im, bt0, H, h, D, r0, valid);
    load_state<NT>(sm.st, gw.R + chunk * 2 * D * N, D, N);
    load_rows<NT>(sm.str1, p.C_re, p.C_im, bt0, H, h, N, r0, valid);  // the first pair's (jb = ib) C, dY
    load_rows<NT>(sm.str2, g.dy_re, g.dy_im, bt0, H, h, D, r0, valid);

    float2 dx[4][2], db[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) dx[i][j] = db[i][j] = make_float2(0.0f, 0.0f);

    // ---- part 1: token blocks jb >= ib (rows t), own rows l
    for (int jb = ib; jb < nb; ++jb) {
        const int s0 = jb * kRows;
        if (s0 >= valid) break;
        const int trows = min(kRows, valid - s0);
        if (jb != ib) {
            __syncthreads();  // previous pair's reads are done
            load_rows<NT>(sm.str1, p.C_re, p.C_im, bt0, H, h, N, s0, valid);
            load_rows<NT>(sm.str2, g.dy_re, g.dy_im, bt0, H, h, D, s0, valid);
        }
        __syncthreads();
        // decay factors of the pair: L[t][l] for t = rb + i (block jb), l = cg + 32 j (block ib)
        float2 L[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int tt = s0 + rb + i, ll = r0 + cg + 32 * j;
                L[i][j] = make_float2(0.0f, 0.0f);
                if (tt >= ll && tt < valid && ll < valid) L[i][j] = cexp_exact(acs_diff(sm.acs[tt], sm.acs[ll]));
            }
        // P[t][l] = (sum_n C[t,n] B[l,n]) L[t][l]
        {
            float2 G[4][2];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) G[i][j] = make_float2(0.0f, 0.0f);
#pragma unroll 8
    #pragma unroll 8
        for (int n = 0; n < N; ++n) {
                float2 a[4], q[2];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = sm.str1.v[rb + i][n];
#pragma unroll
                for (int j = 0; j < 2; ++j) q[j] = sm.own1.v[cg + 32 * j][n];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 2; ++j) cmac(G[i][j], a[i], q[j]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) sm.pv.v[rb + i][cg + 32 * j] = cmul(G[i][j], L[i][j]);
        }
        __syncthreads();
        // dX[l][d] += sum_t conj(P[t][l]) dY[t][d]; on the diagonal pair P[t][l] = 0 for t < l,
        // so a warp starts at its first row
        const int t_lo = jb == ib ? rb : 0;
#pragma unroll 4
        for (int t = t_lo; t < trows; ++t) {
            float2 a[4], y[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = sm.pv.v[t][rb + i];
#pragma unroll
            for (int j = 0; j < 2; ++j) y[j] = sm.str2.v[t][cg + 32 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) cmac_ca(dx[i][j], a[i], y[j]);
        }
        __syncthreads();
        // V[t][l] = (sum_d dY[t,d] conj(x[l,d])) conj(L[t][l])
        {
            float2 W[4][2];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) W[i][j] = make_float2(0.0f, 0.0f);
#pragma unroll 8
    #pragma unroll 8
        for (int d = 0; d < D; ++d) {
                float2 y[4], q[2];
#pragma unroll
                for (int i = 0; i < 4; ++i) y[i] = sm.str2.v[rb + i][d];
#pragma unroll
                for (int j = 0; j < 2; ++j) q[j] = sm.own2.v[cg + 32 * j][d];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 2; ++j) cmac_cb(W[i][j], y[i], q[j]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) sm.pv.v[rb + i][cg + 32 * j] = cmul(W[i][j], conjf2(L[i][j]));
        }
        __syncthreads();
        // dB[l][n] += sum_t V[t][l] conj(C[t][n])  (V[t][l] = 0 for t < l, as P)
#pragma unroll 4
        for (int t = t_lo; t < trows; ++t) {
            float2 v[4], cc[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = sm.pv.v[t][rb + i];
#pragma unroll
            for (int j = 0; j < 2; ++j) cc[j] = sm.str1.v[t][cg + 32 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) cmac_cb(db[i][j], v[i], cc[j]);
        }
    }

    // S_in of the chunk, for part 2: fetched now, stored into st once R_c is no longer read
    StateRegs<NT> sin_regs;
    fetch_state<NT>(sin_regs, ws.S + chunk * 2 * D * N, D, N);

    // R_c terms: dX += conj(dec[l]) sum_n conj(B[l,n]) R[n,d];  dB += conj(dec[l]) sum_d conj(x[l,d]) R[n,d]
    {
        const Acs last = sm.acs[Q - 1];
        float2 e[4];  // conj(dec[l]) of the rows l = rb + i
#pragma unroll
        for (int i = 0; i < 4; ++i) e[i] = conjf2(cexp_exact(acs_diff(last, sm.acs[min(r0 + rb + i, Q - 1)])));
        float2 acc[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) acc[i][j] = make_float2(0.0f, 0.0f);
#pragma unroll 8
        for (int n = 0; n < N; ++n) {
            float2 q[4], r[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) q[i] = sm.own1.v[rb + i][n];
#pragma unroll
            for (int j = 0; j < 2; ++j) r[j] = sm.st.v[cg + 32 * j][n];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) cmac_ca(acc[i][j], q[i], r[j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float2 v = cmul(e[i], acc[i][j]);
                dx[i][j].x += v.x;
                dx[i][j].y += v.y;
                acc[i][j] = make_float2(0.0f, 0.0f);
            }
#pragma unroll 8
        for (int d = 0; d < D; ++d) {
            float2 q[4], r[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) q[i] = sm.own2.v[rb + i][d];
#pragma unroll
            for (int j = 0; j < 2; ++j) r[j] = sm.st.v[d][cg + 32 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) cmac_ca(acc[i][j], q[i], r[j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float2 v = cmul(e[i], acc[i][j]);
                db[i][j].x += v.x;
                db[i][j].y += v.y;
            }
    }

    // write dX, dB; -<dB_l, B_l> per row into shared memory
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int l = rb + i;
        const bool row_ok = r0 + l < valid;
        const int64_t tok = (bt0 + r0 + l) * H + h;
        float2 sum = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int f = cg + 32 * j;
            if (row_ok && f < D) {
                g.dx_re[tok * D + f] = dx[i][j].x;
                if (g.dx_im != nullptr) g.dx_im[tok * D + f] = dx[i][j].y;
            }
            if (row_ok && f < N) {
                g.dB_re[tok * N + f] = db[i][j].x;
                g.dB_im[tok * N + f] = db[i][j].y;
            }
            cmac_cb(sum, db[i][j], sm.own1.v[l][f]);  // dB conj(B); B is zero past N
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            sum.x += __shfl_xor_sync(0xffffffffu, sum.x, off);
            sum.y += __shfl_xor_sync(0xffffffffu, sum.y, off);
        }
        if (cg == 0) sm.nbb[l] = make_float2(-sum.x, -sum.y);
    }

    // <R_c, S_out(c)>, once per chunk (row block 0); st holds R_c^T. S_out is the
    // next chunk's S_in ([d][n] slot) or, for the last chunk, the final state (n, d).
    if (ib == 0) {
        const int64_t bh = (int64_t)b * H + h;
        const bool last_chunk = c == p.nc - 1;
        const float* nxt = ws.S + (chunk + 1) * 2 * D * N;
        float2 acc = make_float2(0.0f, 0.0f);
        for (int e = tid; e < D * N; e += NT) {
            const int d = e / N, n = e % N;
            float2 so;
            if (last_chunk) {
                const int64_t o = (bh * N + n) * D + d;
                so = make_float2(p.fs_re[o], p.fs_im[o]);
            } else {
                so = make_float2(nxt[e], nxt[(int64_t)D * N + e]);
            }
            cmac_cb(acc, sm.st.v[d][n], so);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
            acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
        }
        if (cg == 0) {
            sm.anc[warp][0] = acc.x;
            sm.anc[warp][1] = acc.y;
        }
        __syncthreads();
        if (tid == 0) {
            double sr = 0.0, si = 0.0;
            for (int w = 0; w < kChunkWarps; ++w) {
                sr += sm.anc[w][0];
                si += sm.anc[w][1];
            }
            gw.anchor[2 * chunk] = sr;
            gw.anchor[2 * chunk + 1] = si;
        }
    }

    // ---- part 2: own rows t of block ib, blocks jb <= ib (rows l)
    // With a single block, C and dY of the rows are part 1's str1 / str2, the B rows
    // are own1 and V of the pair is still in pv.
    CTile& Cown = single ? sm.str1 : sm.own1;
    CTile& Yown = single ? sm.str2 : sm.own2;
    CTile& Bsrc = single ? sm.own1 : sm.str1;
    __syncthreads();
    if (!single) {
        load_rows<NT>(sm.own1, p.C_re, p.C_im, bt0, H, h, N, r0, valid);
        load_rows<NT>(sm.own2, g.dy_re, g.dy_im, bt0, H, h, D, r0, valid);
    }
    store_state<NT>(sm.st, sin_regs);
    float2 dc[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) dc[i][j] = make_float2(0.0f, 0.0f);
    for (int jb = 0; jb <= ib; ++jb) {
        const int s0 = jb * kRows;
        const int lrows = min(kRows, valid - s0);
        __syncthreads();
        if (!single) {
            load_rows<NT>(sm.str1, p.B_re, p.B_im, bt0, H, h, N, s0, valid);
            load_rows<NT>(sm.str2, p.x_re, p.x_im, bt0, H, h, D, s0, valid);
            __syncthreads();
            // V[t][l] = (sum_d dY[t,d] conj(x[l,d])) conj(L[t][l]), t = rb + i (block ib),
            // l = cg + 32 j (block jb)
            float2 W[4][2];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) W[i][j] = make_float2(0.0f, 0.0f);
#pragma unroll 8
    #pragma unroll 8
        for (int d = 0; d < D; ++d) {
                float2 y[4], q[2];
#pragma unroll
                for (int i = 0; i < 4; ++i) y[i] = sm.own2.v[rb + i][d];
#pragma unroll
                for (int j = 0; j < 2; ++j) q[j] = sm.str2.v[cg + 32 * j][d];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 2; ++j) cmac_cb(W[i][j], y[i], q[j]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int tt = r0 + rb + i, ll = s0 + cg + 32 * j;
                    float2 v = make_float2(0.0f, 0.0f);
                    if (tt >= ll && tt < valid && ll < valid)
                        v = cmul(W[i][j], conjf2(cexp_exact(acs_diff(sm.acs[tt], sm.acs[ll]))));
                    sm.pv.v[rb + i][cg + 32 * j] = v;
                }
            __syncthreads();
        }
        // dC[t][n] += sum_l V[t][l] conj(B[l][n]); on the diagonal pair V[t][l] = 0 for l > t,
        // so a warp stops after its last row
        const int l_hi = jb == ib ? min(lrows, rb + 4) : lrows;
#pragma unroll 4
        for (int l = 0; l < l_hi; ++l) {
            float2 v[4], q[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = sm.pv.v[rb + i][l];
#pragma unroll
            for (int j = 0; j < 2; ++j) q[j] = Bsrc.v[l][cg + 32 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) cmac_cb(dc[i][j], v[i], q[j]);
        }
    }
    if (single) __syncthreads();  // S_in is in st
    // S_in term: dC[t][n] += conj(exp(Acs[t])) sum_d dY[t,d] conj(S_in[n,d])
    {
        float2 acc[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) acc[i][j] = make_float2(0.0f, 0.0f);
#pragma unroll 8
        for (int d = 0; d < D; ++d) {
            float2 y[4], sv[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) y[i] = Yown.v[rb + i][d];
#pragma unroll
            for (int j = 0; j < 2; ++j) sv[j] = sm.st.v[d][cg + 32 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) cmac_cb(acc[i][j], y[i], sv[j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 e = conjf2(cexp_exact(acs_value(sm.acs[min(r0 + rb + i, Q - 1)])));
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float2 v = cmul(e, acc[i][j]);
                dc[i][j].x += v.x;
                dc[i][j].y += v.y;
            }
        }
    }
    // write dC and r_t = <dC_t, C_t> - <dB_t, B_t>
    const int64_t bh = (int64_t)b * H + h;
    float* rre = gw.r + bh * 2 * p.T;
    float* rim = rre + p.T;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = rb + i;
        const bool row_ok = r0 + t < valid;
        const int64_t tok = (bt0 + r0 + t) * H + h;
        float2 sum = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int n = cg + 32 * j;
            if (row_ok && n < N) {
                g.dC_re[tok * N + n] = dc[i][j].x;
                g.dC_im[tok * N + n] = dc[i][j].y;
            }
            cmac_cb(sum, dc[i][j], Cown.v[t][n]);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            sum.x += __shfl_xor_sync(0xffffffffu, sum.x, off);
            sum.y += __shfl_xor_sync(0xffffffffu, sum.y, off);
        }
        if (cg == 0 && row_ok) {
            rre[t0 + r0 + t] = sum.x + sm.nbb[t].x;
            rim[t0 + r0 + t] = sum.y + sm.nbb[t].y;
        }
    }
}

// ---------------------------------------------------------------------------
// dz_t = <R_c, S_out(c)> + sum_{t' >= t in chunk c} r_t' (fp64), then
// ddt_t = Re(dz_t conj(A)) sigmoid(dt_t) and the chunk's share of
// dA = sum_{b,t} softplus(dt_t) dz_t. One warp per chunk: each lane takes a run
// of consecutive tokens, the runs' totals are suffix-summed across the warp.
// ssdc_bwd_dA then adds the chunk shares of each head in a fixed order.

constexpr int kDtThreads = kBwdDtThreads;
constexpr int kDtWarps = kDtThreads / 32;

__global__ void __launch_bounds__(kDtThreads)
ssdc_bwd_dt(GradProblem g, Workspace ws, GradWorkspace gw) {
    grid_dependency_wait();  // launched as a dependent of the kernel before it
    const Problem& p = g.f;
    const int lane = threadIdx.x & 31;
    const int64_t nc = p.nc;
    const int64_t task = (int64_t)blockIdx.x * kDtWarps + (threadIdx.x >> 5);  // chunk index (b, h, c)
    if (task >= (int64_t)p.B * p.H * nc) return;
    const int H = p.H, Q = p.Q;
    const int64_t T = p.T;
    const int64_t bh = task / nc, c = task % nc;
    const int64_t b = bh / H;
    const int h = (int)(bh % H);
    const int64_t t0 = c * Q;
    const int valid = (int)(T - t0 < (int64_t)Q ? T - t0 : (int64_t)Q);
    const int per = (Q + 31) / 32;  // tokens per lane (Q <= 256: at most 8)
    const int la = min(valid, lane * per), lb = min(valid, la + per);
    const float* rre = gw.r + bh * 2 * T + t0;
    const float* rim = rre + T;
    double tr = 0.0, ti = 0.0;  // this lane's run total
    for (int l = la; l < lb; ++l) {
        tr += rre[l];
        ti += rim[l];
    }
    // inclusive suffix sum of the run totals over the lanes
    double sr = tr, si = ti;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const double ur = __shfl_down_sync(0xffffffffu, sr, off);
        const double ui = __shfl_down_sync(0xffffffffu, si, off);
        if (lane + off < 32) {
            sr += ur;
            si += ui;
        }
    }
    // dz at the end of this lane's run: anchor + the runs after it
    double zr = gw.anchor[2 * task] + (sr - tr), zi = gw.anchor[2 * task + 1] + (si - ti);
    const float Ar = p.A_re[h], Ai = p.A_im[h];
    double dAr = 0.0, dAi = 0.0;
    for (int l = lb - 1; l >= la; --l) {
        zr += rre[l];
        zi += rim[l];
        const int64_t bth = (b * T + t0 + l) * H + h;
        const float v = p.dt[bth];
        const float sig = 1.0f / (1.0f + expf(-v));
        g.ddt[bth] = (float)(zr * Ar + zi * Ai) * sig;
        const double delta = (double)softplus_f(v);
        dAr += delta * zr;
        dAi += delta * zi;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        dAr += __shfl_xor_sync(0xffffffffu, dAr, off);
        dAi += __shfl_xor_sync(0xffffffffu, dAi, off);
    }
    if (lane == 0) {
        gw.dA_part[2 * task] = dAr;
        gw.dA_part[2 * task + 1] = dAi;
    }
}

// dA[h] = sum over b and c of the chunk shares, one CTA per head: each thread
// sums a strided set of chunks, then a fixed-order reduction.
__global__ void __launch_bounds__(kDtThreads)
ssdc_bwd_dA(GradProblem g, Workspace ws, GradWorkspace gw) {
    grid_dependency_wait();  // launched as a dependent of the kernel before it
    __shared__ double red[kDtWarps][2];
    const Problem& p = g.f;
    const int h = blockIdx.x, tid = threadIdx.x;
    const int64_t nc = p.nc, per_head = (int64_t)p.B * nc;
    double sr = 0.0, si = 0.0;
    for (int64_t k = tid; k < per_head; k += kDtThreads) {
        const int64_t b = k / nc, c = k % nc;
        const int64_t task = (b * p.H + h) * nc + c;
        sr += gw.dA_part[2 * task];
        si += gw.dA_part[2 * task + 1];
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        sr += __shfl_xor_sync(0xffffffffu, sr, off);
        si += __shfl_xor_sync(0xffffffffu, si, off);
    }
    if ((tid & 31) == 0) {
        red[tid >> 5][0] = sr;
        red[tid >> 5][1] = si;
    }
    __syncthreads();
    if (tid == 0) {
        double ar = 0.0, ai = 0.0;
        for (int w = 0; w < kDtWarps; ++w) {
            ar += red[w][0];
            ai += red[w][1];
        }
        g.dA_re[h] = (float)ar;
        g.dA_im[h] = (float)ai;
    }
}

// Host side of the two templated kernels: N = D = 64 (the production shape)
// takes the instantiation with compile-time loop bounds.

cudaError_t bwd_set_smem_attrs() {
    const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e = cudaFuncSetAttribute(ssdc_bwd_chunk_states<0, 0>, a, (int)sizeof(StatesSmem));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ssdc_bwd_chunk_states<64, 64>, a, (int)sizeof(StatesSmem));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ssdc_bwd_chunk<0, 0>, a, (int)sizeof(BwdSmem));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ssdc_bwd_chunk<64, 64>, a, (int)sizeof(BwdSmem));
    return e;
}

void bwd_launch_chunk_states(const GradProblem& g, const Workspace& ws, const GradWorkspace& gw,
                             cudaStream_t stream) {
    const Problem& p = g.f;
    const dim3 grid((unsigned)p.nc, (unsigned)p.H, (unsigned)p.B);
    if (p.N == 64 && p.D == 64)
        ssdc_bwd_chunk_states<64, 64><<<grid, kBwdThreads, sizeof(StatesSmem), stream>>>(g, ws, gw);
    else
        ssdc_bwd_chunk_states<0, 0><<<grid, kBwdThreads, sizeof(StatesSmem), stream>>>(g, ws, gw);
}

void bwd_launch_chunk(const GradProblem& g, const Workspace& ws, const GradWorkspace& gw, cudaStream_t stream) {
    const Problem& p = g.f;
    const int nb = (p.Q + kRows - 1) / kRows;
    const dim3 grid((unsigned)(p.nc * nb), (unsigned)p.H, (unsigned)p.B);
    if (p.N == 64 && p.D == 64)
        ssdc_bwd_chunk<64, 64><<<grid, kChunkThreads, sizeof(BwdSmem), stream>>>(g, ws, gw);
    else
        ssdc_bwd_chunk<0, 0><<<grid, kChunkThreads, sizeof(BwdSmem), stream>>>(g, ws, gw);
}

}  // namespace ssdc
