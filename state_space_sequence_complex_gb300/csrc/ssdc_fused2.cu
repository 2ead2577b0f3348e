// Fused single-pass forward of the chunkwise complex SSD scan on the TF32
// tensor cores with the chunk state held in tensor memory (Q = 16, 32 or 64;
// N and D multiples of 8 up to 64).
// One CTA per SM walks whole (b, h) sequences chunk by chunk; every step of
// the chunked decomposition (landing page, "03 Chunkwise SSD": L, Y_diag =
// (C B^T o L) X, the per-chunk state, the pass between chunks, Y_off) runs in
// this one launch, inputs are read from HBM once and y and the final state
// written once.
//
// Transposed output. The kernel accumulates y^T instead of y:
//     Y^T = X^T P^T + S_in^T C'^T,   P = (C B^T) o L,   C' = C o exp(Acs)
//     S_out^T = a_c S_in^T + X^T (dec o B),  a_c = exp(Acs[Q-1])
// so that both A operands of the output MMAs, X^T (rows d, K = s) and S_in^T
// (rows d, K = n), live in TMEM windows, and the state never leaves TMEM: the
// threads read S_loc^T from its accumulator and S_in^T from its window, form
// S_out^T and write it back as the next chunk's window. The B operands are
// shared-memory tiles: P (written by the threads in place of the consumed
// (dec o B)^T), C' (the C tile scaled in place after C B^T has read it) and
// (dec o B)^T (the B tile transposed in place). X^T is written into its window
// straight from the TMA tile by column reads, with no shared-memory transpose.
//
// Complex products are M = 128, N = 128 real MMAs over interleaved planes, as
// in the cluster kernel (ssdc_fused.cu): the A rows interleave the two planes
// in groups of eight (row 16g + 8p + i = plane p of row 8g + i), the B rows
// are stacked or interleaved, and one accumulator holds all four real products
// in TMEM lanes m and m + 8, which the 16x256b access shape hands to one
// thread. Y_off does not wait for anything of its own chunk but C': its state
// was formed at the end of the previous chunk.
//
// Threads: 16 worker warps (phases below), warp 16 issues every MMA in chunk
// order on mbarrier hand-offs, warp 17 issues the TMA loads of the chunk after
// next into the other stage and computes its cumulative log-decay. Each of
// the three tiles of a stage is released as soon as its last reader is done
// (x after its columns are read, C after Y_off, B after Y_diag), so the loads
// of chunk c+2 start during chunk c.
//
// Smaller shapes run on the same 64-row, 64-column tiles. Feature columns past
// N or D are read as zeros by the tensor maps (and never stored), so they add
// nothing to any product. A chunk of Q < 64 tokens fills the first Q rows of
// its tiles; the other rows keep finite values from earlier use (the tiles are
// zeroed at the start), and every product that reads them is masked: the decay
// dec[s] is zero for s >= Q, P is causal, and y rows past Q are not stored
// (the TMA store boxes are Q rows high).
//
// Worker phases of chunk c (stage s):
//   A  decay tables; X^T window from the x tile; (B rows into registers)
//   B  (dec o B)^T in place of B          -> S^T MMA
//   D  y of chunk c-1 from the Y^T accumulator to global memory
//   C  C' in place of C                   -> Y_off MMA (S_in^T window)
//   E  P = (C B^T) o L into the B tile    -> Y_diag MMA
//   F  S_out^T = a_c S_in^T + S_loc^T into the S window (or the final state)
#include <mutex>

#include "fused_io.cuh"

namespace ssdc {
namespace fused2 {
namespace {

using namespace tc;
using namespace fused;

constexpr int kWorkers = 512;  // 16 worker warps
constexpr int kWorkerWarps = kWorkers / 32;
constexpr int kIssuer = kWorkerWarps;        // warp 16: issues the MMAs
constexpr int kProducer = kWorkerWarps + 1;  // warp 17: TMA loads and decays
constexpr int kThreads = kWorkers + 64;
constexpr uint32_t kWorkerBar = 1;  // named barrier of the worker warps
constexpr uint32_t kTmemCols = 512;
// TMEM columns: three 128-column accumulators (C B^T; Y^T; S_loc^T) and two
// 64-column A windows (X^T; S_in^T).
constexpr uint32_t kAccG = 0, kAccY = 128, kAccS = 256, kXwin = 384, kSwin = 448;

struct Smem {
    float c[2][64 * 128];  // [stage] C (interleaved, A of C B^T), then C' in place (B of Y_off)
    float b[2][64 * 128];  // [stage] B (stacked), then (dec o B)^T (stacked, rows n), then P (interleaved)
    float x[2][64 * 128];  // [stage] x (stacked): read into the X^T window
    float2 acs[2][kQ];     // [stage] in-chunk cumulative log-decay
    float2 dec[2][kQ];     // [stage] exp(Acs[Q-1] - Acs[s])
    float2 eacs[2][kQ];    // [stage] exp(Acs[l])
    float2 step[2][kQ];    // [stage] exp(Acs[s] - Acs[s-1]) (s >= 1)
    float2 a_c[2];         // [stage] exp(Acs[Q-1])
    uint64_t full[2];                       // stage loaded (tiles and decays)
    uint64_t free_x[2], free_b[2], free_c[2];  // stage tiles released
    uint64_t xt_ready, bt_ready, c_ready, p_ready, sin_ready;  // worker hand-offs (one arrival per warp)
    uint64_t mma_g, mma_s, mma_yo, mma_y;   // MMA completions, one phase per chunk
    uint32_t tmem;
};

static_assert(sizeof(Smem) <= 232448, "shared-memory plan exceeds the 227 KB a CTA can have");

// Chunk `c` of sequence `q` = b H + h.
struct Pos {
    int q, c, b, h;
};

__device__ __forceinline__ Pos pos_at(int q, int c, int H) {
    Pos p;
    p.q = q;
    p.c = c;
    p.b = (int)((uint32_t)q / (uint32_t)H);
    p.h = q - p.b * H;
    return p;
}

// The items of this CTA, in order: every chunk of sequences blockIdx.x,
// blockIdx.x + gridDim.x, ...
__device__ __forceinline__ Pos pos_next(const Pos& p, int nc, int H) {
    return p.c + 1 < nc ? pos_at(p.q, p.c + 1, H) : pos_at(p.q + (int)gridDim.x, 0, H);
}

// Producer: TMA of one chunk's x (stacked; only the real plane for a real x),
// C (interleaved) or B (stacked) into stage buffers, counted on `bar`.
// A box of Q rows of one 32-column half of one plane is Q x 128 bytes.
__device__ __forceinline__ void load_x(char* dst, const FusedMaps& fm, uint64_t* bar, int h, int t0, int b, int Q,
                                       int lane) {
    if (lane == 0) ptx::mbar_expect_tx(bar, (uint32_t)(Q * 128 * (fm.real_x ? 2 : 4)));
    __syncwarp();
    if (fm.fast & 1) {
        if (lane < 2) ptx::tma_load_5d(dst + stk_row(lane, 0, 0), &fm.x2, bar, 32 * lane, h, t0, 0, b);
    } else {
        const int n = fm.real_x ? 2 : 4;
        if (lane < n) {
            const int half = fm.real_x ? lane : lane >> 1, pl = fm.real_x ? 0 : lane & 1;
            ptx::tma_load_4d(dst + stk_row(half, pl, 0), pl ? &fm.x_im : &fm.x_re, bar, 32 * half, h, t0, b);
        }
    }
}

__device__ __forceinline__ void load_b(char* dst, const FusedMaps& fm, uint64_t* bar, int h, int t0, int b, int Q,
                                       int lane) {
    if (lane == 0) ptx::mbar_expect_tx(bar, (uint32_t)(Q * 128 * 4));
    __syncwarp();
    if ((fm.fast >> 1) & 1) {
        if (lane < 2) ptx::tma_load_5d(dst + stk_row(lane, 0, 0), &fm.B2, bar, 32 * lane, h, t0, 0, b);
    } else if (lane < 4) {
        const int half = lane >> 1, pl = lane & 1;
        ptx::tma_load_4d(dst + stk_row(half, pl, 0), pl ? &fm.B_im : &fm.B_re, bar, 32 * half, h, t0, b);
    }
}

__device__ __forceinline__ void load_c(char* dst, const FusedMaps& fm, uint64_t* bar, int h, int t0, int b, int64_t T,
                                       int Q, int lane) {
    if (lane == 0) ptx::mbar_expect_tx(bar, (uint32_t)(Q * 128 * 4));
    __syncwarp();
    if ((fm.fast >> 2) & 1) {
        if (lane < 2)
            ptx::tma_load_5d(dst + inter_row(lane, 0), &fm.C2, bar, 32 * lane, h, 0, 0, (int)(((int64_t)b * T + t0) >> 3));
    } else {  // rows 8g .. 8g+7 of plane pl, per 32-column half (Q / 8 groups)
        const int ng = Q >> 3;
        if (lane < 4 * ng) {
            const int half = lane / (2 * ng), g = (lane >> 1) % ng, pl = lane & 1;
            ptx::tma_load_4d(dst + inter_row(half, 16 * g + 8 * pl), pl ? &fm.c8_im : &fm.c8_re, bar, 32 * half, h,
                             t0 + 8 * g, b);
        }
    }
}

template <bool kSwapC>
__global__ void __launch_bounds__(kThreads, 1)
fused2_kernel(Problem p, Workspace ws, const __grid_constant__ FusedMaps fm) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H, nc = (int)p.nc, Q = p.Q, N = p.N, D = p.D;
    const int nseq = p.B * H;
    const int nseq_cta = (int)blockIdx.x < nseq ? (nseq - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int nitems = nseq_cta * nc;

    // the swizzled tiles need a 1024-byte aligned base (uniform across the grid)
    if (ptx::smem_addr(smem_raw) & 1023u) {
        if (tid == 0) atomicCAS(ws.status, SSDC_OK, SSDC_ERR_CUDA);
        return;
    }
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&sm.full[s], 1);
            ptx::mbar_init(&sm.free_x[s], 1);
            ptx::mbar_init(&sm.free_b[s], 1);
            ptx::mbar_init(&sm.free_c[s], 1);
        }
        ptx::mbar_init(&sm.xt_ready, kWorkerWarps);
        ptx::mbar_init(&sm.bt_ready, kWorkerWarps);
        ptx::mbar_init(&sm.c_ready, kWorkerWarps);
        ptx::mbar_init(&sm.p_ready, kWorkerWarps);
        ptx::mbar_init(&sm.sin_ready, kWorkerWarps);
        ptx::mbar_init(&sm.mma_g, 1);
        ptx::mbar_init(&sm.mma_s, 1);
        ptx::mbar_init(&sm.mma_yo, 1);
        ptx::mbar_init(&sm.mma_y, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(&sm.tmem, kTmemCols);
        ptx::tmem_relinquish();
    }
    if (Q < kQ) {
        // rows past Q are never loaded: give them finite contents
        float4* z = reinterpret_cast<float4*>(sm.c);
        constexpr int kVecs = 3 * 2 * 64 * 128 / 4;  // the c, b and x tiles of both stages
        for (int i = tid; i < kVecs; i += kThreads) z[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem;

    if (warp == kProducer) {
        // ============ producer warp: TMA loads and cumulative log-decays ============
        bool ok = true;  // false once a wait gave up: later waits are skipped
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (lane == 0 && ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
            __syncwarp();
        };
        Pos ld = pos_at((int)blockIdx.x, 0, H);
        Alog al = {};
        if (nitems > 0) al = load_alog(p, ld.b, ld.h, (int64_t)ld.c * Q, lane, Q);
        for (int j = 0; j < nitems; ++j) {  // item j into stage j & 1
            const int st = j & 1;
            const uint32_t ph = (uint32_t)((j - 2) >> 1) & 1u;
            const int t0 = ld.c * Q;
            if (j >= 2) wait(&sm.free_x[st], ph);
            load_x(reinterpret_cast<char*>(sm.x[st]), fm, &sm.full[st], ld.h, t0, ld.b, Q, lane);
            if (j >= 2) wait(&sm.free_c[st], ph);
            load_c(reinterpret_cast<char*>(sm.c[st]), fm, &sm.full[st], ld.h, t0, ld.b, p.T, Q, lane);
            if (j >= 2) wait(&sm.free_b[st], ph);
            load_b(reinterpret_cast<char*>(sm.b[st]), fm, &sm.full[st], ld.h, t0, ld.b, Q, lane);
            const Alog now = al;
            ld = pos_next(ld, nc, H);
            if (j + 1 < nitems) al = load_alog(p, ld.b, ld.h, (int64_t)ld.c * Q, lane, Q);
            store_acs(sm.acs[st], &sm.full[st], now, lane);
        }
    } else if (warp == kIssuer) {
        // ============ MMA warp: lane 0 issues every MMA in chunk order ============
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
        };
        Pos cur = pos_at((int)blockIdx.x, 0, H);
        for (int it = 0; it < nitems && lane == 0; ++it) {
            const int s = it & 1;
            const uint32_t ph = (uint32_t)it & 1u;
            const bool has_in = cur.c > 0 || p.s0_re != nullptr;
            const uint32_t cs = ptx::smem_addr(sm.c[s]), bs = ptx::smem_addr(sm.b[s]);
            wait(&sm.full[s], (uint32_t)((it >> 1) & 1));
            ptx::tc_fence_after();
            issue_ss128(tmem + kAccG, desc128(cs), desc128(bs));  // C [B_0 | B_1]^T
            ptx::mma_commit(&sm.mma_g);
            wait(&sm.xt_ready, ph);
            wait(&sm.bt_ready, ph);
            ptx::tc_fence_after();
            issue_ts128(tmem + kAccS, tmem + kXwin, desc128(bs), false);  // X^T (dec o B)
            ptx::mma_commit(&sm.mma_s);
            wait(&sm.c_ready, ph);
            wait(&sm.sin_ready, ph);
            ptx::tc_fence_after();
            if (has_in) issue_ts128(tmem + kAccY, tmem + kSwin, desc128(cs), false);  // S_in^T C'^T
            ptx::mma_commit(&sm.mma_yo);
            ptx::mma_commit(&sm.free_c[s]);
            wait(&sm.p_ready, ph);
            ptx::tc_fence_after();
            issue_ts128(tmem + kAccY, tmem + kXwin, desc128(bs), has_in);  // + X^T P^T
            ptx::mma_commit(&sm.mma_y);
            ptx::mma_commit(&sm.free_b[s]);
            cur = pos_next(cur, nc, H);
        }
        __syncwarp();
    } else {
        // ===================== 16 worker warps =====================
        // 16x256b fragment of a warp: TMEM lane quadrant qd, 16-lane block blk, 32-column half
        // kh. Lane i4 of the block holds plane 0 and lane i4 + 8 plane 1 of row
        // rr = 16 qd + 8 blk + i4 (a token l of C B^T; a column d of Y^T, S^T and the windows).
        const int qd = warp & 3, blk = (warp >> 2) & 1, kh = warp >> 3;
        const int i4 = lane >> 2, lq = lane & 3;
        const int rr = 16 * qd + 8 * blk + i4;
        const uint32_t tl = lane_base(tmem, warp) + ((uint32_t)(16 * blk) << 16);
        const int swx = fm.swap & 1, swb = (fm.swap >> 1) & 1;
        constexpr int kCr = kSwapC ? 1 : 0;              // C plane in TMEM lane plane 0 / 1
        constexpr int kRr = 2 * kCr, kRi = 2 - 2 * kCr;  // register offset of the C_r / C_i lanes
        const uint32_t gbr = kAccG + 64 * swb, gbi = kAccG + 64 * (1 - swb);  // B_r / B_i products
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
        };
        // S_in^T[rr, n] of the given sequence's initial state (n = 32 kh + 8 j + 2 lq + e) into
        // the S window, in the 16x256b register order
        auto store_s0 = [&](int q) {
            float w[16];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int j = k >> 1, e = k & 1;
                const int n = 32 * kh + 8 * j + 2 * lq + e;
                const bool in = n < N && rr < D;
                const int64_t o = in ? ((int64_t)q * N + n) * D + rr : 0;
                w[4 * j + e] = in ? p.s0_re[o] : 0.0f;
                w[4 * j + 2 + e] = in ? p.s0_im[o] : 0.0f;
            }
            ptx::tmem_st_16x256b_x4(tl + kSwin + 32 * kh, w);
        };
        // y rows of chunk `pos` from the Y^T accumulator (lanes (d, plane of X), columns
        // 16g + 8p + i = plane p of token 8g + i of P and of C') into the staging tile `buf`
        // (two stacked planes, rows l, the 128-byte swizzle of the TMA boxes; the four rows and
        // eight columns of a warp's store fall on distinct 16-byte positions), then, once every
        // worker has written its part, one thread stores the tile with four TMA copies (rows
        // past T are not written) and commits them as one bulk group.
        auto stage_y = [&](char* buf, const Pos& pos) {
            float v[32];
            ptx::tmem_ld_16x256b_x4(tl + kAccY + 64 * kh, v);
            ptx::tmem_ld_16x256b_x4(tl + kAccY + 64 * kh + 32, v + 16);
            ptx::tmem_wait_ld();
            const uint32_t dofs = (uint32_t)(4 * (rr & 3));
            const int cq = (rr & 31) >> 2;
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int j = 2 * jj;
                        const int l = 32 * kh + 16 * u + 8 * jj + 2 * lq + e;
                        const float a0 = v[16 * u + 4 * j + e], b0 = v[16 * u + 4 * j + 2 + e];
                        const float a1 = v[16 * u + 4 * j + 4 + e], b1 = v[16 * u + 4 * j + 6 + e];
                        const uint32_t o = stk_row(rr >> 5, 0, l) + chunk16(cq, l) + dofs;
                        *reinterpret_cast<float*>(buf + o) = a0 - b1;
                        *reinterpret_cast<float*>(buf + o + kHalfBytes) = a1 + b0;
                    }
            ptx::fence_proxy_async_smem();
            ptx::named_sync(kWorkerBar, kWorkers);
            if (tid == 0) {
                const int t0 = pos.c * Q;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    ptx::tma_store_4d(&fm.y_re, buf + stk_row(half, 0, 0), 32 * half, pos.h, t0, pos.b);
                    ptx::tma_store_4d(&fm.y_im, buf + stk_row(half, 1, 0), 32 * half, pos.h, t0, pos.b);
                }
                ptx::bulk_commit();
            }
        };

        Pos cur = pos_at((int)blockIdx.x, 0, H), prev = cur;
        // the S window of the first item: its initial state, if any
        if (nitems > 0 && p.s0_re != nullptr) {
            store_s0(cur.q);
            ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.sin_ready);

        for (int it = 0; it < nitems; ++it) {
            const int s = it & 1;
            const uint32_t ph = (uint32_t)it & 1u;
            const bool has_in = cur.c > 0 || p.s0_re != nullptr;
            const bool last = cur.c == nc - 1;
            char* xbase = reinterpret_cast<char*>(sm.x[s]);
            char* bbase = reinterpret_cast<char*>(sm.b[s]);
            char* cbase = reinterpret_cast<char*>(sm.c[s]);
            wait(&sm.full[s], (uint32_t)((it >> 1) & 1));
            // the previous chunk's MMAs are complete: its X^T window and Y^T accumulator are free
            if (it > 0) wait(&sm.mma_y, ph ^ 1u);
            ptx::tc_fence_after();

            // ---- A: decay tables; X^T window; B rows into registers
            if (tid < kQ) {  // zero past the chunk's Q tokens (rows holding no token of it)
                sm.dec[s][tid] = tid < Q ? cexp_fast(cdiff(sm.acs[s][kQ - 1], sm.acs[s][tid])) : make_float2(0.0f, 0.0f);
            } else if (tid < 2 * kQ) {
                sm.eacs[s][tid - kQ] = cexp_fast(sm.acs[s][tid - kQ]);
            } else if (tid == 2 * kQ) {
                sm.a_c[s] = cexp_fast(sm.acs[s][kQ - 1]);
            } else if (tid < 3 * kQ) {
                const int t = tid - 2 * kQ;  // 1 .. Q-1
                sm.step[s][t] = cexp_fast(cdiff(sm.acs[s][t], sm.acs[s][t - 1]));
            }
            {
                // X^T rows: TMEM lane 32 qd + lane = plane xp of column xd; columns s of group cg.
                // Plane-1 lanes read row s ^ 4, so that the two planes' rows (8 KB apart, the same
                // banks) fall on different 16-byte positions; the values are put back in order.
                const int xd = 16 * qd + 8 * (lane >> 4) + (lane & 7), xp = (lane >> 3) & 1, cg = warp >> 2;
                float v[16];
                if (xp == 1 && fm.real_x) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) v[k] = 0.0f;
                } else {
                    const char* rowbase = xbase + stk_row(xd >> 5, xp ^ swx, 0) + 4 * (xd & 3);
                    const int cq = (xd & 31) >> 2;
                    float r[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int sr = 16 * cg + (k ^ (4 * xp));
                        r[k] = *reinterpret_cast<const float*>(rowbase + sr * 128 + chunk16(cq, sr));
                    }
#pragma unroll
                    for (int k = 0; k < 16; ++k) v[k] = ptx::to_tf32(xp ? r[k ^ 4] : r[k]);
                }
                ptx::tmem_st16(lane_base(tmem, warp) + kXwin + 16 * cg, v);
            }
            // (dec o B)^T blocks: rows s = 4 bsb + i, columns n = 4 bnb + 2 bjh + {0, 1}, both planes
            const int L0 = lane & 1, L1 = (lane >> 1) & 1, L2 = (lane >> 2) & 1, L3 = (lane >> 3) & 1, L4 = lane >> 4;
            const int bjh = L1;
            const int bsb = L2 + 2 * (warp >> 1), bnb = L0 + 2 * L3 + 4 * L4 + 8 * (warp & 1);
            float2 bv[2][4];
#pragma unroll
            for (int pp = 0; pp < 2; ++pp)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int sr = 4 * bsb + i;
                    bv[pp][i] = *reinterpret_cast<const float2*>(bbase + stk_row(bnb >> 3, pp ^ swb, sr) +
                                                                 chunk16(bnb & 7, sr) + 8 * bjh);
                }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::named_sync(kWorkerBar, kWorkers);
            // every worker has read x; the tile is free at once on the first item, and otherwise
            // once the previous chunk's y, staged in it below, has been read by its TMA stores
            if (tid == 0 && it == 0) ptx::mbar_arrive(&sm.free_x[s]);
            if (lane == 0) ptx::mbar_arrive(&sm.xt_ready);

            // ---- B: (dec o B)^T in place of B (after C B^T has read it)
            wait(&sm.mma_g, ph);
            {
                float2 dv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) dv[i] = sm.dec[s][4 * bsb + i];
#pragma unroll
                for (int j = 0; j < 2; ++j) {  // column n of B -> row n of the output
                    const int nr = 4 * bnb + 2 * bjh + j;
                    float ore[4], oim[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 v = cmul(dv[i], j ? make_float2(bv[0][i].y, bv[1][i].y) : make_float2(bv[0][i].x, bv[1][i].x));
                        ore[i] = ptx::to_tf32(v.x);
                        oim[i] = ptx::to_tf32(v.y);
                    }
                    *reinterpret_cast<float4*>(bbase + stk_row(bsb >> 3, 0, nr) + chunk16(bsb & 7, nr)) =
                        make_float4(ore[0], ore[1], ore[2], ore[3]);
                    *reinterpret_cast<float4*>(bbase + stk_row(bsb >> 3, 1, nr) + chunk16(bsb & 7, nr)) =
                        make_float4(oim[0], oim[1], oim[2], oim[3]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm.bt_ready);
            }

            // ---- D: the previous chunk's y, staged in this chunk's x tile
            if (it > 0) stage_y(xbase, prev);

            // ---- C: C' = C o exp(Acs[l]) in place, plane 0 real. Unit: physical 16-byte chunk j
            // of rows 16g + i (plane 0) and 16g + 8 + i (plane 1) of one half (token l = 8g + i);
            // eight lanes cover the eight chunks of a row.
            {
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int u = tid + kWorkers * k;
                    const int j = u & 7, i = (u >> 3) & 7, g = (u >> 6) & 7, half = u >> 9;
                    char* r0 = cbase + inter_row(half, 16 * g + i) + 16 * j;
                    char* r1 = r0 + 8 * 128;
                    const float2 e = sm.eacs[s][8 * g + i];
                    const float4 v0 = *reinterpret_cast<const float4*>(r0), v1 = *reinterpret_cast<const float4*>(r1);
                    const float4 cr = kSwapC ? v1 : v0, ci = kSwapC ? v0 : v1;
                    using ptx::to_tf32;
                    *reinterpret_cast<float4*>(r0) =
                        make_float4(to_tf32(cr.x * e.x - ci.x * e.y), to_tf32(cr.y * e.x - ci.y * e.y),
                                    to_tf32(cr.z * e.x - ci.z * e.y), to_tf32(cr.w * e.x - ci.w * e.y));
                    *reinterpret_cast<float4*>(r1) =
                        make_float4(to_tf32(cr.x * e.y + ci.x * e.x), to_tf32(cr.y * e.y + ci.y * e.x),
                                    to_tf32(cr.z * e.y + ci.z * e.x), to_tf32(cr.w * e.y + ci.w * e.x));
                }
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();  // the y loads of D precede the Y_off MMA
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm.c_ready);
            }

            // ---- E: P = (C B^T) o L on row rr, columns col, col + 1 (col = 32 kh + 8 j + 2 lq),
            // into the B tile once the S^T MMA has read (dec o B)^T. In the accumulator, one 64-column
            // half holds the products with B_r, the other with B_i; lane plane 0 / 1 of the row holds
            // the products of C's plane 0 / 1 (C_r first unless kSwapC).
            {
                float ga[16], gb[16];
                ptx::tmem_ld_16x256b_x4(tl + gbr + 32 * kh, ga);
                ptx::tmem_ld_16x256b_x4(tl + gbi + 32 * kh, gb);
                ptx::tmem_wait_ld();
                const float2 acs_l = sm.acs[s][rr];
                float2 pv[4][2];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // L[rr, col + 1] from one exponential, L[rr, col] = L[rr, col + 1] exp(-dA[col + 1])
                    const int col = 32 * kh + 8 * j + 2 * lq;
                    // Re G = Cr Br - Ci Bi, Im G = Cr Bi + Ci Br
                    const float2 g0 = make_float2(ga[4 * j + kRr] - gb[4 * j + kRi], gb[4 * j + kRr] + ga[4 * j + kRi]);
                    const float2 g1 = make_float2(ga[4 * j + kRr + 1] - gb[4 * j + kRi + 1],
                                                  gb[4 * j + kRr + 1] + ga[4 * j + kRi + 1]);
                    float2 p0 = make_float2(0.0f, 0.0f), p1 = make_float2(0.0f, 0.0f);
                    if (col + 1 <= rr) {
                        const float2 L1v = cexp_fast(cdiff(acs_l, sm.acs[s][col + 1]));
                        p1 = cmul(g1, L1v);
                        p0 = cmul(g0, cmul(L1v, sm.step[s][col + 1]));
                    } else if (col == rr) {
                        p0 = g0;
                    }
                    pv[j][0] = p0;
                    pv[j][1] = p1;
                }
                wait(&sm.mma_s, ph);
                const int mre = inter_m(rr, 0), mim = inter_m(rr, 1);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    *reinterpret_cast<float2*>(bbase + pair_off(kh, mre, 8 * j + 2 * lq)) =
                        make_float2(ptx::to_tf32(pv[j][0].x), ptx::to_tf32(pv[j][1].x));
                    *reinterpret_cast<float2*>(bbase + pair_off(kh, mim, 8 * j + 2 * lq)) =
                        make_float2(ptx::to_tf32(pv[j][0].y), ptx::to_tf32(pv[j][1].y));
                }
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();  // the C B^T loads precede the next C B^T MMA
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm.p_ready);
            }

            // ---- F: S_out^T = a_c S_in^T + S_loc^T on column d = rr, state rows n = 32 kh + 8 j + 2 lq + e
            {
                float sa[16], sb[16];
                ptx::tmem_ld_16x256b_x4(tl + kAccS + 32 * kh, sa);       // products with (dec o B)_r
                ptx::tmem_ld_16x256b_x4(tl + kAccS + 64 + 32 * kh, sb);  // products with (dec o B)_i
                float w[16];
                if (has_in) ptx::tmem_ld_16x256b_x4(tl + kSwin + 32 * kh, w);
                ptx::tmem_wait_ld();
                const float2 a = sm.a_c[s];
                float outr[8], outi[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int j = k >> 1, e = k & 1;
                    // Re: (x_r (dB)_r)[p0] - (x_i (dB)_i)[p1];  Im: (x_r (dB)_i)[p0] + (x_i (dB)_r)[p1]
                    outr[k] = sa[4 * j + e] - sb[4 * j + 2 + e];
                    outi[k] = sb[4 * j + e] + sa[4 * j + 2 + e];
                    if (has_in) {
                        const float sr = w[4 * j + e], si = w[4 * j + 2 + e];
                        outr[k] += a.x * sr - a.y * si;
                        outi[k] += a.x * si + a.y * sr;
                    }
                }
                // Y_off of this chunk has read the window
                wait(&sm.mma_yo, ph);
                ptx::tc_fence_after();
                const Pos nxt = pos_next(cur, nc, H);
                if (last) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int n = 32 * kh + 8 * (k >> 1) + 2 * lq + (k & 1);
                        if (n < N && rr < D) {
                            const int64_t o = ((int64_t)cur.q * N + n) * D + rr;
                            p.fs_re[o] = outr[k];
                            p.fs_im[o] = outi[k];
                        }
                    }
                    if (it + 1 < nitems && p.s0_re != nullptr) store_s0(nxt.q);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int j = k >> 1, e = k & 1;
                        w[4 * j + e] = outr[k];
                        w[4 * j + 2 + e] = outi[k];
                    }
                    ptx::tmem_st_16x256b_x4(tl + kSwin + 32 * kh, w);
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm.sin_ready);
            }
            if (tid == 0 && it > 0) {  // the y stores have read the x tile
                ptx::bulk_wait_read_all();
                ptx::mbar_arrive(&sm.free_x[s]);
            }
            prev = cur;
            cur = pos_next(cur, nc, H);
        }
        if (nitems > 0) {
            // the last chunk's y, staged in its x tile (read by the last stores, see above)
            wait(&sm.mma_y, (uint32_t)(nitems - 1) & 1u);
            ptx::tc_fence_after();
            ptx::named_sync(kWorkerBar, kWorkers);
            stage_y(reinterpret_cast<char*>(sm.x[(nitems - 1) & 1]), prev);
            if (tid == 0) ptx::bulk_wait_all();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
}

constexpr size_t kSmemBytes = sizeof(Smem);
bool g_attr_set[64] = {};
std::mutex g_mu;

int set_attrs(int dev) {
    std::lock_guard<std::mutex> g(g_mu);
    if (g_attr_set[dev]) return SSDC_OK;
    if (cudaFuncSetAttribute(fused2_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(fused2_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
            cudaSuccess)
        return SSDC_ERR_CUDA;
    g_attr_set[dev] = true;
    return SSDC_OK;
}

}  // namespace
}  // namespace fused2

bool fused2_supported(int N, int D, int Q) {
    return (Q == 16 || Q == 32 || Q == 64) && N >= 8 && N <= 64 && N % 8 == 0 && D >= 8 && D <= 64 && D % 8 == 0;
}

int fused2_launch(const Problem& p, const Workspace& ws, cudaStream_t stream, bool plane_maps) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SSDC_ERR_CUDA;
    int rc = fused2::set_attrs(dev);
    if (rc != SSDC_OK) return rc;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return SSDC_ERR_CUDA;
    fused::FusedMaps fm;
    rc = fused::cached_maps(p, plane_maps, &fm);
    if (rc != SSDC_OK) return rc;
    const int64_t nseq = (int64_t)p.B * p.H;
    const int grid = (int)(nseq < sms ? nseq : sms);
    const dim3 g((unsigned)grid), b(fused2::kThreads);
    if (fm.swap & 4)
        fused2::fused2_kernel<true><<<g, b, fused2::kSmemBytes, stream>>>(p, ws, fm);
    else
        fused2::fused2_kernel<false><<<g, b, fused2::kSmemBytes, stream>>>(p, ws, fm);
    return cudaGetLastError() == cudaSuccess ? 1 : SSDC_ERR_CUDA;
}

}  // namespace ssdc
