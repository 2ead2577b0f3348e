// Fused single-pass forward of the chunkwise complex SSD scan on the TF32
// tensor cores, for chunk size Q = 64 and N = D = 64 (the pages' production
// shape). One launch does every step of the chunked decomposition (landing
// page, "03 Chunkwise SSD": the CHUNK line, L and Y_diag = einsum(C, B, L, X);
// the STATE line, the per-chunk state and the pass between chunks; Y_off):
// inputs are read from HBM once, y and the final state written once, and the
// state passed between chunks never leaves the chip.
//
// Work split. A thread-block cluster of CL CTAs (one CTA per SM) owns one
// (b, h) sequence at a time; CTA rank r takes the chunks c = r, r + CL, ...
// of it, in order. The state entering chunk c+1,
//     S_in[c+1] = exp(Acs_c[Q-1]) S_in[c] + S_loc[c],
// is computed by the CTA of chunk c and copied (cp.async.bulk, 32 KB in four
// 8 KB quarters of rows d) straight into the shared memory of the CTA of
// chunk c+1, rank (r+1) mod CL, where one mbarrier per quarter counts the
// bytes; the receiver frees the buffer by arriving on the sender's mbarrier.
// Each quarter leaves as soon as the four warps that own its rows have it, so
// the quarters of consecutive hops overlap. With CL = 1 the CTA keeps the
// state in its own shared memory. All chunk-local work (C B^T, L, Y_diag,
// S_loc) is independent of the incoming state, so the serial chain per
// sequence is one complex multiply-add per state element and one transfer of
// a quarter of the state per chunk.
//
// Complex products. Planar re/im operands are multiplied as real M=128 MMAs
// whose A operand holds the real and imaginary rows of the left factor
// interleaved in groups of eight (row 16g + 8p + i = plane p of row 8g + i)
// and whose B operand stacks or interleaves the right factor's two planes as
// 128 rows (N = 128). One accumulator then holds, in TMEM lanes m and m + 8,
// all four real products, and
//     Re = (A_r B_r)[lane p=0] - (A_i B_i)[lane p=1]
//     Im = (A_r B_i)[lane p=0] + (A_i B_r)[lane p=1].
// The 16x256b TMEM access shape hands each thread lanes m and m + 8 of the
// same columns, so every thread combines its own values: no exchange between
// lanes. The C tile is loaded in that layout by TMA (one 5-D copy per 32-column
// half, or 8-row boxes); x^T is written in it by a shared-memory transpose. The
// output accumulator takes both P x (Y_diag) and (C o exp(Acs)) S_in (Y_off):
// the two A operands, P and C', are rows written to TMEM.
//
// Threads. 16 worker warps: warp w owns TMEM lane quadrant w % 4, its 16-lane
// block (w / 4) % 2 (8 complex rows) and the 32-column half w / 8, which is a
// contiguous 2 KB of every interleaved tile. They write the transposes, the C'
// and P rows and the state hop, and store y from registers to global memory,
// four lanes per 32-byte run of a row (the previous chunk's y, in the next
// chunk just before its P rows). Warp 16 issues every MMA, in chunk order, on mbarrier hand-offs
// from the workers; warp 17 issues the TMA loads of the next chunk into the
// other stage of a two-stage ring and computes its cumulative log-decay.
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fused_io.cuh"

namespace ssdc {
namespace fused {
namespace {

using namespace tc;

constexpr int kWorkers = 512;               // 16 worker warps
constexpr int kWorkerWarps = kWorkers / 32;
constexpr int kIssuer = kWorkerWarps;        // warp 16: issues the MMAs
constexpr int kProducer = kWorkerWarps + 1;  // warp 17: TMA loads and decays
constexpr int kThreads = kWorkers + 64;
constexpr uint32_t kWorkerBar = 5;           // named barrier of the worker warps (1-4: quadrants)
constexpr uint32_t kTmemCols = 512;
// TMEM columns: three 128-column accumulators and two 64-column A operands.
constexpr uint32_t kAccG = 0, kAccS = 128, kAccY = 256, kPwin = 384, kCwin = 448;
constexpr uint32_t kStageTx = 3 * kTileBytes;     // C, B, x
constexpr uint32_t kStateBytes = kTileBytes;
constexpr uint32_t kQuarterBytes = kStateBytes / 4;  // rows d of one TMEM lane quadrant (4 warps)

struct Smem {
    float c[2][64 * 128];    // [stage] C, interleaved 128 rows (A operand)
    float b[2][64 * 128];    // [stage] B, stacked (rows s); after C B^T, (dec o B)^T stacked (rows n)
    float x[2][64 * 128];    // [stage] x, stacked (rows s); x^T interleaved (rows d); then y staging
    float sin[64 * 128];     // incoming state S_in^T, interleaved rows d, K = n, state layout (st_off)
    float2 acs[2][kQ];       // in-chunk cumulative log-decay, per stage
    float2 dec[kQ];          // exp(Acs[Q-1] - Acs[s])
    float2 eacs[kQ];         // exp(Acs[l])
    float2 a_c;              // exp(Acs[Q-1])
    float2 step[kQ];         // exp(Acs[s] - Acs[s-1]): decay over token s (s >= 1)
    uint64_t full[2], sin_full[4], succ_empty;  // sin_full[q]: rows d in [16q, 16q + 16) of S_in
    uint64_t stage_free;          // workers are done with the previous chunk's stage
    uint64_t xt_ready, bt_ready;  // x^T, (dec o B)^T written (one arrival per worker warp)
    uint64_t p_ready;             // P and C' rows in TMEM (one arrival per worker warp)
    uint64_t mma[3];         // MMA groups C B^T, S_loc^T, y; one phase per chunk
    uint32_t tmem;
};

static_assert(sizeof(Smem) <= 232448, "shared-memory plan exceeds the 227 KB a CTA can have");

// Position of an item: sequence q = b H + h and chunk c (all below 2^31: the
// host limits B H to 65535 and the chunk count to 2^29).
struct Pos {
    int q, c, b, h;
};

// The chunks this CTA processes, in order: for each sequence owned by its
// cluster, the chunks congruent to its rank.
struct Items {
    int nseq, nc;
    uint32_t cl, rank, cluster, nclusters;
    __device__ Items(int nseq_, int nc_)
        : nseq(nseq_), nc(nc_), cl(ptx::cluster_nctarank()), rank(ptx::cluster_ctarank()),
          cluster(ptx::cluster_id_x()), nclusters(ptx::ncluster_x()) {}
    __device__ int count() const {
        const int per_seq = nc > (int)rank ? (nc - 1 - (int)rank) / (int)cl + 1 : 0;
        const int seqs = nseq > (int)cluster ? (nseq - 1 - (int)cluster) / (int)nclusters + 1 : 0;
        return seqs * per_seq;
    }
    __device__ static Pos at(int q, int c, int H) {
        Pos p;
        p.q = q;
        p.c = c;
        p.b = (int)((uint32_t)q / (uint32_t)H);
        p.h = q - p.b * H;
        return p;
    }
    __device__ Pos first(int H) const { return at((int)cluster, (int)rank, H); }
    __device__ Pos next(const Pos& p, int H) const {
        const int c = p.c + (int)cl;
        return c < nc ? at(p.q, c, H) : at(p.q + (int)nclusters, (int)rank, H);
    }
};


// The state tiles (S_in^T and the outgoing state, rows d interleaved, K = n) use
// a 32-byte swizzle instead: 8-row groups of 2 KB holding the eight 32-byte
// K-blocks one after another, so that the per-thread pair accesses of the
// 16x256b fragments hit 16 distinct 8-byte bank positions per half-warp (with
// the 128-byte swizzle two rows of a half-warp share each position), and the
// rows of one TMEM lane quadrant are one contiguous 8 KB.
__device__ __forceinline__ uint32_t st_off(int m, int n) {
    return (uint32_t)((m >> 3) * 2048 + (n >> 3) * 256 + (m & 7) * 32 + ((((n >> 2) ^ (m >> 2)) & 1) << 4) + ((n & 3) << 2));
}
__device__ __forceinline__ uint64_t desc_state(uint32_t base) { return ptx::smem_desc(base, 16u, 2048u, 6u); }

// The same with the B operand in the state layout: K-step k is the next 256-byte block.
__device__ __forceinline__ void issue_ts128_state(uint32_t d, uint32_t a_tmem, uint64_t db) {
#pragma unroll
    for (int k = 0; k < 8; ++k) ptx::mma_tf32_ts(d, a_tmem + 8 * k, db + (uint64_t)(16 * k), kIdesc128, 1u);
}


// Issuer warp: TMA of one chunk's C (re/im interleaved), B and x (stacked)
// into stage `st`, counted on `bar`. The copies are issued by the warp's lanes
// in parallel after lane 0 has announced the bytes.
__device__ __forceinline__ void load_tiles(Smem& sm, int st, const FusedMaps& fm, int h, int t0, int b, int64_t T,
                                           int lane) {
    uint64_t* bar = &sm.full[st];
    // real x: only its real plane is loaded (the workers take the imaginary one as zero)
    if (lane == 0) ptx::mbar_expect_tx(bar, fm.real_x ? kStageTx - kPlaneBytes : kStageTx);
    __syncwarp();
    char* cb = reinterpret_cast<char*>(sm.c[st]);
    char* bb = reinterpret_cast<char*>(sm.b[st]);
    char* xb = reinterpret_cast<char*>(sm.x[st]);
    const bool fx = fm.fast & 1, fb = (fm.fast >> 1) & 1, fc = (fm.fast >> 2) & 1;
    const int nc = fc ? 2 : 32, nb = fb ? 2 : 4, nx = fx ? 2 : fm.real_x ? 2 : 4;
    for (int op = lane; op < nc + nb + nx; op += 32) {
        if (op < nc) {
            if (fc) {
                ptx::tma_load_5d(cb + inter_row(op, 0), &fm.C2, bar, 32 * op, h, 0, 0, (int)(((int64_t)b * T + t0) >> 3));
            } else {  // C rows 8g .. 8g+7 of plane pl
                const int half = op >> 4, g = (op >> 1) & 7, pl = op & 1;
                ptx::tma_load_4d(cb + inter_row(half, 16 * g + 8 * pl), pl ? &fm.c8_im : &fm.c8_re, bar, 32 * half, h,
                                 t0 + 8 * g, b);
            }
        } else {
            const bool isb = op < nc + nb;
            const int k = isb ? op - nc : op - nc - nb;
            char* dst = isb ? bb : xb;
            if (isb ? fb : fx) {
                ptx::tma_load_5d(dst + stk_row(k, 0, 0), isb ? &fm.B2 : &fm.x2, bar, 32 * k, h, t0, 0, b);
            } else {
                // per-plane copies: k = 2 half + plane (for real x, k = half and the real plane only)
                const bool ronly = !isb && fm.real_x;
                const int half = ronly ? k : k >> 1, pl = ronly ? 0 : k & 1;
                const CUtensorMap* m = isb ? (pl ? &fm.B_im : &fm.B_re) : (pl ? &fm.x_im : &fm.x_re);
                ptx::tma_load_4d(dst + stk_row(half, pl, 0), m, bar, 32 * half, h, t0, b);
            }
        }
    }
}


template <bool kSwapC>
__global__ void __launch_bounds__(kThreads, 1)
fused_kernel(Problem p, Workspace ws, const __grid_constant__ FusedMaps fm) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    const Items items(p.B * H, (int)p.nc);
    const int nitems = items.count();
    const uint32_t CL = items.cl, rank = items.rank;
    const uint32_t succ = (rank + 1) % CL, pred = (rank + CL - 1) % CL;

    // the swizzled tiles need a 1024-byte aligned base (uniform across the grid)
    if (ptx::smem_addr(smem_raw) & 1023u) {
        if (tid == 0) atomicCAS(ws.status, SSDC_OK, SSDC_ERR_CUDA);
        return;
    }
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) ptx::mbar_init(&sm.full[s], 1);
        for (int g = 0; g < 3; ++g) ptx::mbar_init(&sm.mma[g], 1);
        for (int k = 0; k < 4; ++k) ptx::mbar_init(&sm.sin_full[k], 1);
        ptx::mbar_init(&sm.stage_free, 1);
        ptx::mbar_init(&sm.xt_ready, kWorkerWarps);
        ptx::mbar_init(&sm.bt_ready, kWorkerWarps);
        ptx::mbar_init(&sm.p_ready, kWorkerWarps);
        ptx::mbar_init(&sm.succ_empty, 1);
        ptx::fence_mbar_init();
        if (CL > 1)  // first transfer
            for (int k = 0; k < 4; ++k) ptx::mbar_arrive_expect_tx(&sm.sin_full[k], kQuarterBytes);
    }
    if (warp == 0) {
        ptx::tmem_alloc(&sm.tmem, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem;

    if (warp == kProducer) {
        // ============ producer warp: TMA loads and cumulative log-decays ============
        bool ok = true;  // false once a wait gave up: later waits are skipped
        // This warp touches no peer's shared memory: it joins the cluster barrier that guards
        // the other warps' first remote accesses with a relaxed arrival, before its first loads
        // (a releasing arrival would wait for them), and completes it later.
        ptx::cluster_arrive_relaxed();
        Pos ld = items.first(H);
        Alog al = {};
        if (nitems > 0) al = load_alog(p, ld.b, ld.h, (int64_t)ld.c * kQ, lane);
        for (int j = 0; j < nitems; ++j) {  // item j into stage j & 1
            if (j == 1) ptx::cluster_wait();
            const int st = j & 1;
            if (j >= 2) {
                // the workers have passed the first barrier of item j - 1: item j - 2 left the stage
                if (lane == 0 && ok && !ptx::mbar_wait(&sm.stage_free, (uint32_t)((j - 2) & 1), kWaitIters)) {
                    fail(ws.status);
                    ok = false;
                }
                __syncwarp();
            }
            load_tiles(sm, st, fm, ld.h, ld.c * kQ, ld.b, p.T, lane);
            const Alog now = al;
            ld = items.next(ld, H);
            if (j + 1 < nitems) al = load_alog(p, ld.b, ld.h, (int64_t)ld.c * kQ, lane);
            store_acs(sm.acs[st], &sm.full[st], now, lane);
        }
        if (nitems <= 1) ptx::cluster_wait();
    } else if (warp == kIssuer) {
        // ============ MMA warp: lane 0 issues every MMA in chunk order ============
        ptx::cluster_sync();  // peers' barriers are initialised before any remote access
        bool ok = true;  // false once a wait gave up: later waits are skipped
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
        };
        const uint32_t pred_empty = ptx::mapa(ptx::smem_addr(&sm.succ_empty), pred);
        const uint32_t sin_saddr = ptx::smem_addr(sm.sin);
        Pos cur = items.first(H);
        bool prev_in = false;
        uint32_t n_recv = 0;
        for (int it = 0; it < nitems && lane == 0; ++it) {
            const int s = it & 1;
            const bool self_fill = cur.c == 0 && p.s0_re != nullptr;  // S_in[0] is the initial state
            const bool has_in = cur.c > 0 || self_fill;
            const uint32_t cs = ptx::smem_addr(sm.c[s]), bs = ptx::smem_addr(sm.b[s]), xs = ptx::smem_addr(sm.x[s]);
            wait(&sm.full[s], (uint32_t)((it >> 1) & 1));
            ptx::tc_fence_after();
            issue_ss128(tmem + kAccG, desc128(cs), desc128(bs));  // [C Br | C Bi]
            ptx::mma_commit(&sm.mma[0]);
            if (it > 0) {
                // the previous chunk's y MMAs are done: its incoming state buffer is free
                wait(&sm.mma[2], (uint32_t)((it - 1) & 1));
                if (prev_in && CL > 1 && ok) {
                    for (int k = 0; k < 4; ++k) ptx::mbar_arrive_expect_tx(&sm.sin_full[k], kQuarterBytes);
                    // the buffer is free for the predecessor's next state, unless this chunk fills
                    // it with an initial state first (then the signal follows that chunk)
                    if (!self_fill) ptx::mbar_arrive_remote(pred_empty);
                }
            }
            wait(&sm.xt_ready, (uint32_t)(it & 1));
            wait(&sm.bt_ready, (uint32_t)(it & 1));
            ptx::tc_fence_after();
            issue_ss128(tmem + kAccS, desc128(xs), desc128(bs));  // [x^T B'r | x^T B'i]
            ptx::mma_commit(&sm.mma[1]);
            wait(&sm.p_ready, (uint32_t)(it & 1));
            ptx::tc_fence_after();
            issue_ts128(tmem + kAccY, tmem + kPwin, desc128(xs), false);  // P x^T (interleaved columns)
            if (has_in) {
                if (CL > 1) {
                    for (int k = 0; k < 4; ++k) wait(&sm.sin_full[k], n_recv & 1);
                    ++n_recv;
                }
                ptx::tc_fence_after();
                issue_ts128_state(tmem + kAccY, tmem + kCwin, desc_state(sin_saddr));  // + C' S_in
            }
            ptx::mma_commit(&sm.mma[2]);
            prev_in = has_in;
            cur = items.next(cur, H);
        }
        __syncwarp();
    } else {
        // ===================== 16 worker warps =====================
        ptx::cluster_sync();  // peers' barriers are initialised before any remote access
        // Fragment of a warp: TMEM lane quadrant qd, 16-lane block blk of it (complex rows
        // rr = 16 qd + 8 blk + i4: lane i4 holds plane 0, lane i4 + 8 plane 1) and the 32-column
        // half kh (column pair n = 32 kh + 8 j + 2 lq + {0, 1}, j = 0 .. 3). In an interleaved
        // tile these are 16 whole 128-byte rows; the four warps of a quadrant hold rows
        // [32 qd, 32 qd + 32) of both halves; in the state layout, the quadrant's contiguous 8 KB.
        const int qd = warp & 3, blk = (warp >> 2) & 1, kh = warp >> 3;
        const int i4 = lane >> 2, lq = lane & 3;
        const int rr = 16 * qd + 8 * blk + i4;
        const int mre = inter_m(rr, 0), mim = inter_m(rr, 1);
        const uint32_t tl = lane_base(tmem, warp) + ((uint32_t)(16 * blk) << 16);
        const bool leader = warp == qd && lane == 0;  // copies the quadrant's rows of the state
        // physical plane order of the x and B tiles, and the C-tile rows and G-accumulator
        // columns that hold the real planes
        const int swx = fm.swap & 1, swb = (fm.swap >> 1) & 1;
        constexpr int kCr = kSwapC ? 1 : 0;                 // C plane in TMEM lane plane 0 / 1
        constexpr int kRr = 2 * kCr, kRi = 2 - 2 * kCr;     // register offset of the C_r / C_i lanes
        const uint32_t gbr = kAccG + 64 * swb, gbi = kAccG + 64 * (1 - swb);  // B_r / B_i products
        uint32_t n_recv = 0, n_send = 0;
        const uint32_t remote_sin = ptx::mapa(ptx::smem_addr(sm.sin), succ);
        const uint32_t remote_sin_full = ptx::mapa(ptx::smem_addr(&sm.sin_full[qd]), succ);
        const uint32_t self_sin = ptx::mapa(ptx::smem_addr(sm.sin), rank);
        const uint32_t self_sin_full = ptx::mapa(ptx::smem_addr(&sm.sin_full[qd]), rank);
        // the successor fills its buffer with an initial state before its first state from here
        const bool succ_self_fills = p.s0_re != nullptr && succ == 0;

        auto wait_mma = [&](int g, int it) {
            if (!ptx::mbar_wait(&sm.mma[g], (uint32_t)(it & 1), kWaitIters)) fail(ws.status);
            ptx::tc_fence_after();
        };
        // this thread's state values S^T[rr, n] in a state tile, index 2 j + e (column pair
        // n = 32 kh + 8 j + 2 lq: K-block 4 kh + j, 256 bytes apart)
        auto for_pairs = [&](char* base, float* vr, float* vi, bool store) {
            const uint32_t soff_re = st_off(mre, 32 * kh + 2 * lq), soff_im = st_off(mim, 32 * kh + 2 * lq);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float2* pr = reinterpret_cast<float2*>(base + soff_re + 256 * j);
                float2* pi = reinterpret_cast<float2*>(base + soff_im + 256 * j);
                if (store) {
                    *pr = make_float2(vr[2 * j], vr[2 * j + 1]);
                    *pi = make_float2(vi[2 * j], vi[2 * j + 1]);
                } else {
                    const float2 a = *pr, b = *pi;
                    vr[2 * j] = a.x;
                    vr[2 * j + 1] = a.y;
                    vi[2 * j] = b.x;
                    vi[2 * j + 1] = b.y;
                }
            }
        };

        // Work left over from the previous chunk, done during the next one (or after the last):
        // (a) at its start, wait for its y MMAs and keep its outgoing state (CL = 1); (b) before
        // the next P x, write its y row straight from the accumulator to global memory, late
        // enough that these stores do not share the SM's outbound link with the state copy that
        // ended the chunk. Column 16g + 8p' + i of the accumulator holds the plane-p' products of
        // column d = 8g + i; four consecutive lanes hold one 32-byte run of a row.
        float outr[8], outi[8];
        // (a) wait for its y MMAs (they read its stage, C' and S_in) and keep its state
        auto finish_wait = [&](int it, bool keep_state) {
            wait_mma(2, it);
            if (keep_state) {
                for_pairs(reinterpret_cast<char*>(sm.sin), outr, outi, true);
                ptx::fence_proxy_async_smem();
            }
        };
        // (b) its y, from the accumulator (free until this chunk's P x)
        auto finish_y = [&](const Pos& pos) {
            float yv[32];
            ptx::tmem_ld_16x256b_x4(tl + kAccY + 64 * kh, yv);
            ptx::tmem_ld_16x256b_x4(tl + kAccY + 64 * kh + 32, yv + 16);
            ptx::tmem_wait_ld();
            const int64_t t = (int64_t)pos.c * kQ + rr;
            const int64_t row = (((int64_t)pos.b * p.T + (t < p.T ? t : 0)) * H + pos.h) * 64;
            const bool odd = lq & 1;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                // this thread's column pairs d0 = 32 kh + 16 u + 2 lq (block dd = 0) and d0 + 8 (dd = 1);
                // Re y = (P_r x_r)[p0] - (P_i x_i)[p1], Im y = (P_r x_i)[p0] + (P_i x_r)[p1]
                float2 re[2], im[2];
#pragma unroll
                for (int dd = 0; dd < 2; ++dd) {
                    const int jr = 16 * u + 8 * dd, ji = jr + 4;  // register blocks of planes x_r, x_i
                    re[dd] = make_float2(yv[jr + 0] - yv[ji + 2], yv[jr + 1] - yv[ji + 3]);
                    im[dd] = make_float2(yv[ji + 0] + yv[jr + 2], yv[ji + 1] + yv[jr + 3]);
                }
                // lanes lq and lq ^ 1 swap one pair each, so that every lane stores 16 bytes: an even
                // lane columns d0 .. d0 + 3 of block 0, an odd lane d0 + 6 .. d0 + 9 of block 1 (its
                // partner's pair, then its own); the four lanes of a row cover 64 contiguous bytes
                const float2 sre = odd ? re[0] : re[1], sim = odd ? im[0] : im[1];
                const float2 rre = make_float2(__shfl_xor_sync(0xffffffffu, sre.x, 1), __shfl_xor_sync(0xffffffffu, sre.y, 1));
                const float2 rim = make_float2(__shfl_xor_sync(0xffffffffu, sim.x, 1), __shfl_xor_sync(0xffffffffu, sim.y, 1));
                const int d = 32 * kh + 16 * u + 2 * lq + (odd ? 6 : 0);
                if (t < p.T) {
                    *reinterpret_cast<float4*>(p.y_re + row + d) =
                        odd ? make_float4(rre.x, rre.y, re[1].x, re[1].y) : make_float4(re[0].x, re[0].y, rre.x, rre.y);
                    if (p.y_im != nullptr)  // absent when only Re(y) is asked for (the head mixer's input)
                        *reinterpret_cast<float4*>(p.y_im + row + d) =
                            odd ? make_float4(rim.x, rim.y, im[1].x, im[1].y) : make_float4(im[0].x, im[0].y, rim.x, rim.y);
                }
            }
        };

        Pos cur = items.first(H), prev = cur;
        bool prev_keep = false;
        for (int it = 0; it < nitems; ++it) {
            const int s = it & 1;
            const bool self_fill = cur.c == 0 && p.s0_re != nullptr;
            const bool has_in = cur.c > 0 || self_fill, last = cur.c == (int)p.nc - 1;
            char* xbase = reinterpret_cast<char*>(sm.x[s]);
            char* bbase = reinterpret_cast<char*>(sm.b[s]);
            char* cbase = reinterpret_cast<char*>(sm.c[s]);
            const uint32_t cs = ptx::smem_addr(cbase);
            if (!ptx::mbar_wait(&sm.full[s], (uint32_t)((it >> 1) & 1), kWaitIters)) fail(ws.status);

            // ---- A: decays; the previous chunk's y; x and B blocks into registers. Lane bits
            // pick the blocks so that a warp's accesses cover all bank groups.
            if (tid < kQ) {
                sm.dec[tid] = cexp_fast(cdiff(sm.acs[s][kQ - 1], sm.acs[s][tid]));
            } else if (tid < 2 * kQ) {
                sm.eacs[tid - kQ] = cexp_fast(sm.acs[s][tid - kQ]);
            } else if (tid == 2 * kQ) {
                sm.a_c = cexp_fast(sm.acs[s][kQ - 1]);
            } else if (tid < 3 * kQ) {
                const int t = tid - 2 * kQ;  // 1 .. Q-1
                sm.step[t] = cexp_fast(cdiff(sm.acs[s][t], sm.acs[s][t - 1]));
            }
            if (it > 0) finish_wait(it - 1, prev_keep);
            // Lane bits L0..L4. 128-bit accesses are served eight lanes at a time, so within
            // each group of eight (L0..L2) the 16-byte chunk positions of both the block loads
            // (rows s, swizzle by s) and the transposed stores (rows d, swizzle by d) are distinct.
            const int L0 = lane & 1, L1 = (lane >> 1) & 1, L2 = (lane >> 2) & 1, L3 = (lane >> 3) & 1, L4 = lane >> 4;
            const int xdb = L0 + 2 * L1 + 4 * L4 + 8 * ((warp >> 2) & 1);
            const int xsb = L2 + 2 * (L1 ^ L3) + 4 * (warp & 3), xp = (warp >> 3) & 1;
            float4 xv[4];
            const bool zero_plane = xp == 1 && fm.real_x;  // the imaginary plane of a real x
#pragma unroll
            for (int i = 0; i < 4; ++i) {  // x block: rows s = 4 xsb + i, columns d = 4 xdb ..
                const int sr = 4 * xsb + i;
                xv[i] = zero_plane ? make_float4(0.0f, 0.0f, 0.0f, 0.0f)
                                   : *reinterpret_cast<const float4*>(xbase + stk_row(xdb >> 3, xp ^ swx, sr) +
                                                                      chunk16(xdb & 7, sr));
            }
            // (dec o B)^T: rows s = 4 bsb + i, columns n = 4 bnb + 2 bjh + {0, 1}, both planes; the
            // 64-bit loads (16 lanes at a time) and the 128-bit stores (8 at a time) are conflict-free
            const int bjh = L1;
            const int bsb = L2 + 2 * (warp >> 1), bnb = L0 + 2 * L3 + 4 * L4 + 8 * (warp & 1);
            float2 bv[2][4];
#pragma unroll
            for (int pp = 0; pp < 2; ++pp)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int sr = 4 * bsb + i;
                    bv[pp][i] = *reinterpret_cast<const float2*>(bbase + stk_row(bnb >> 3, pp ^ swb, sr) + chunk16(bnb & 7, sr) + 8 * bjh);
                }
            // the previous chunk's state copies have read their staging buffer (the
            // other stage's C tile), which the producer's next prefetch overwrites
            if (leader) ptx::bulk_wait_read_all();
            ptx::named_sync(kWorkerBar, kWorkers);
            if (tid == 0 && it >= 1) ptx::mbar_arrive(&sm.stage_free);
            // The decay tables are rewritten at the start of the next chunk, which a warp can
            // reach once every warp has announced its (dec o B)^T block: what is needed after
            // that announcement is read now.
            const float2 a_c = sm.a_c;
            float2 step_j[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) step_j[j] = sm.step[32 * kh + 8 * j + 2 * lq + 1];

            // ---- B: x^T (interleaved rows d) in place of x; C' = C o exp(Acs[l]) rows into TMEM
            {
                using ptx::to_tf32;
                const float4 o[4] = {
                    make_float4(to_tf32(xv[0].x), to_tf32(xv[1].x), to_tf32(xv[2].x), to_tf32(xv[3].x)),
                    make_float4(to_tf32(xv[0].y), to_tf32(xv[1].y), to_tf32(xv[2].y), to_tf32(xv[3].y)),
                    make_float4(to_tf32(xv[0].z), to_tf32(xv[1].z), to_tf32(xv[2].z), to_tf32(xv[3].z)),
                    make_float4(to_tf32(xv[0].w), to_tf32(xv[1].w), to_tf32(xv[2].w), to_tf32(xv[3].w))};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int mm = inter_m(4 * xdb + j, xp);
                    *reinterpret_cast<float4*>(xbase + inter_row(xsb >> 3, mm) + chunk16(xsb & 7, mm)) = o[j];
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm.xt_ready);
            }
            {
                // C'[rr, n] on this thread's eight columns, both planes
                const float2 e = sm.eacs[rr];
                const int cre = inter_m(rr, kCr), cim = inter_m(rr, 1 - kCr);
                float w[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 cr = *reinterpret_cast<const float2*>(cbase + pair_off(kh, cre, 8 * j + 2 * lq));
                    const float2 ci = *reinterpret_cast<const float2*>(cbase + pair_off(kh, cim, 8 * j + 2 * lq));
                    w[4 * j + 0] = ptx::to_tf32(cr.x * e.x - ci.x * e.y);
                    w[4 * j + 1] = ptx::to_tf32(cr.y * e.x - ci.y * e.y);
                    w[4 * j + 2] = ptx::to_tf32(cr.x * e.y + ci.x * e.x);
                    w[4 * j + 3] = ptx::to_tf32(cr.y * e.y + ci.y * e.x);
                }
                ptx::tmem_st_16x256b_x4(tl + kCwin + 32 * kh, w);
            }
            // S_in[0] = the given initial state (N, D) of this sequence, this thread's values in
            // the state layout
            auto load_s0 = [&](float* vr, float* vi) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int n = 32 * kh + 8 * (k >> 1) + 2 * lq + (k & 1);
                    const int64_t o = ((int64_t)cur.q * 64 + n) * 64 + rr;
                    vr[k] = p.s0_re[o];
                    vi[k] = p.s0_im[o];
                }
            };
            if (self_fill && CL == 1) {  // straight into the incoming state tile (read by Y_off after p_ready)
                float vr[8], vi[8];
                load_s0(vr, vi);
                for_pairs(reinterpret_cast<char*>(sm.sin), vr, vi, true);
                ptx::fence_proxy_async_smem();
            }
            wait_mma(0, it);  // C B^T has read B

            // ---- C: (dec o B)^T stacked in place of B (the MMA warp then starts S_loc^T = x^T (dec o B))
            {
                float2 dv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) dv[i] = sm.dec[4 * bsb + i];
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

            if (it > 0) finish_y(prev);  // the previous chunk's y (see finish_y)

            // ---- D: P = (C B^T) o L on this thread's row rr and columns col, col + 1 (col = 32 kh +
            // 8 j + 2 lq); P rows into TMEM (the MMA warp then starts P x). In the accumulator, one
            // 64-column half holds the products with B_r, the other with B_i; lane plane 0 / 1 of
            // the row holds the products of C's plane 0 / 1 (C_r first unless kSwapC).
            {
                float ga[16], gb[16];
                ptx::tmem_ld_16x256b_x4(tl + gbr + 32 * kh, ga);
                ptx::tmem_ld_16x256b_x4(tl + gbi + 32 * kh, gb);
                ptx::tmem_wait_ld();
                const float2 acs_l = sm.acs[s][rr];
                float w[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // L[rr, col + 1] from one exponential, L[rr, col] = L[rr, col + 1] exp(-dA[col + 1])
                    const int col = 32 * kh + 8 * j + 2 * lq;
                    float2 L1 = make_float2(0.0f, 0.0f), L0 = make_float2(0.0f, 0.0f);
                    if (col + 1 <= rr) {
                        L1 = cexp_fast(cdiff(acs_l, sm.acs[s][col + 1]));
                        L0 = cmul(L1, step_j[j]);
                    } else if (col == rr) {
                        L0 = make_float2(1.0f, 0.0f);
                    }
                    // Re G = Cr Br - Ci Bi, Im G = Cr Bi + Ci Br
                    const float2 g0 = make_float2(ga[4 * j + kRr] - gb[4 * j + kRi], gb[4 * j + kRr] + ga[4 * j + kRi]);
                    const float2 g1 = make_float2(ga[4 * j + kRr + 1] - gb[4 * j + kRi + 1],
                                                  gb[4 * j + kRr + 1] + ga[4 * j + kRi + 1]);
                    const float2 p0 = cmul(g0, L0), p1 = cmul(g1, L1);
                    w[4 * j + 0] = ptx::to_tf32(p0.x);
                    w[4 * j + 1] = ptx::to_tf32(p1.x);
                    w[4 * j + 2] = ptx::to_tf32(p0.y);
                    w[4 * j + 3] = ptx::to_tf32(p1.y);
                }
                ptx::tmem_st_16x256b_x4(tl + kPwin + 32 * kh, w);
                // P and C' rows of this warp are in TMEM
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm.p_ready);
            }

            // ---- E: S_loc^T and the state hop  S_out = a_c S_in + S_loc  (row d = rr, this thread's
            // columns n). Each lane quadrant's rows travel to the next CTA as soon as its four warps
            // have them, so the chain of states is pipelined across quadrants.
            wait_mma(1, it);
            {
                float sa[16], sb[16];
                ptx::tmem_ld_16x256b_x4(tl + kAccS + 32 * kh, sa);
                ptx::tmem_ld_16x256b_x4(tl + kAccS + 64 + 32 * kh, sb);
                ptx::tmem_wait_ld();
                // Re: (xr B'r)[p0] - (xi B'i)[p1];  Im: (xr B'i)[p0] + (xi B'r)[p1]
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int j = k >> 1, e = k & 1;
                    outr[k] = sa[4 * j + e] - sb[4 * j + 2 + e];
                    outi[k] = sb[4 * j + e] + sa[4 * j + 2 + e];
                }
            }
            if (self_fill && CL > 1) {
                // With CL > 1 the initial state is staged in the C buffer and copied by the
                // quadrant's leader like a state from a predecessor, so that its arrival is counted
                // on the same barrier. Not before now: a quadrant's 8 KB of the staging buffer holds
                // C rows of other quadrants, and the C B^T MMA reads the whole tile; the S_loc MMA
                // just waited for was issued after C B^T and after every worker had read its C' rows.
                float vr[8], vi[8];
                load_s0(vr, vi);
                for_pairs(cbase, vr, vi, true);
                ptx::fence_proxy_async_smem();
                ptx::named_sync(1 + qd, 128);
                if (leader) {
                    const uint32_t off = (uint32_t)qd * kQuarterBytes;
                    ptx::bulk_copy_to_cluster(self_sin + off, cs + off, kQuarterBytes, self_sin_full);
                    ptx::bulk_commit();
                }
            }
            if (has_in) {
                if (CL > 1) {
                    if (!ptx::mbar_wait(&sm.sin_full[qd], n_recv & 1, kWaitIters)) fail(ws.status);
                    ++n_recv;
                }
                const float2 a = a_c;
                float sr[8], si[8];
                for_pairs(reinterpret_cast<char*>(sm.sin), sr, si, false);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    outr[k] += a.x * sr[k] - a.y * si[k];
                    outi[k] += a.x * si[k] + a.y * sr[k];
                }
            }
            if (last) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int n = 32 * kh + 8 * (k >> 1) + 2 * lq + (k & 1);
                    const int64_t o = ((int64_t)cur.q * 64 + n) * 64 + rr;
                    p.fs_re[o] = outr[k];
                    p.fs_im[o] = outi[k];
                }
            } else if (CL > 1) {
                // stage S_out in the C buffer (C was consumed by C B^T and the C' rows), then the
                // quadrant's leader copies its 8 KB of rows to the next CTA
                for_pairs(cbase, outr, outi, true);
                ptx::fence_proxy_async_smem();
                ptx::named_sync(1 + qd, 128);
                if (leader && cur.c != p.drop_send_chunk) {
                    // send k waits for the successor's k-th buffer release (its (k-1)-th when the
                    // buffer starts out free)
                    const int sig = succ_self_fills ? (int)n_send : (int)n_send - 1;
                    if (sig >= 0 && !ptx::mbar_wait(&sm.succ_empty, (uint32_t)sig & 1, kWaitIters)) fail(ws.status);
                    ++n_send;
                    const uint32_t off = (uint32_t)qd * kQuarterBytes;
                    ptx::bulk_copy_to_cluster(remote_sin + off, cs + off, kQuarterBytes, remote_sin_full);
                    ptx::bulk_commit();
                }
            }
            prev = cur;
            prev_keep = !last && CL == 1;
            cur = items.next(cur, H);
        }
        if (nitems > 0) {
            finish_wait(nitems - 1, false);
            finish_y(prev);
        }
        if (leader) ptx::bulk_wait_all();
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
    ptx::cluster_sync();  // no CTA leaves while a peer may still write to its shared memory
}

constexpr size_t kSmemBytes = sizeof(Smem);
bool g_attr_set[64] = {};


int set_attrs(int dev) {
    if (g_attr_set[dev]) return SSDC_OK;
    if (cudaFuncSetAttribute(fused_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(fused_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
            cudaSuccess)
        return SSDC_ERR_CUDA;
    g_attr_set[dev] = true;
    return SSDC_OK;
}

}  // namespace

namespace {

// Per-call host work is kept off the launch path: the cluster choice is cached
// per (device, sequences, chunks) (the tensor maps per pointer set, in fused_io.cuh).
struct ClusterKey {
    int dev;
    int64_t nseq, nc;
};
struct ClusterChoice {
    ClusterKey key;
    int cl, nclusters;
    double cost;
};
constexpr int kCacheSlots = 16;
std::mutex g_cache_mu;
ClusterChoice g_cluster_cache[kCacheSlots];
int g_cluster_used = 0, g_cluster_next = 0;
}  // namespace

// Choose the cluster size: the one that minimises (waves of clusters) x
// (chunks per CTA, or the serial state chain if that is longer). *cost_out is
// that minimum, in units of one CTA's time for one chunk.
int pick_cluster(const Problem& p, int* cl_out, int* nclusters_out, double* cost_out = nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SSDC_ERR_CUDA;
    const int64_t nseq = (int64_t)p.B * p.H;
    {
        std::lock_guard<std::mutex> g(g_cache_mu);
        for (int i = 0; i < g_cluster_used; ++i) {
            const ClusterChoice& c = g_cluster_cache[i];
            if (c.key.dev == dev && c.key.nseq == nseq && c.key.nc == p.nc) {
                *cl_out = c.cl;
                *nclusters_out = c.nclusters;
                if (cost_out) *cost_out = c.cost;
                return SSDC_OK;
            }
        }
    }
    const int arc = set_attrs(dev);
    if (arc != SSDC_OK) return arc;
    double best = 1e300;
    int best_cl = 1, best_n = 1;
    for (int cl = 1; cl <= 8; cl *= 2) {
        if (cl > 1 && cl > p.nc) break;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cl;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(cl, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, fused_kernel<false>, &cfg) != cudaSuccess || active <= 0) {
            (void)cudaGetLastError();
            continue;
        }
        const int64_t nclusters = nseq < active ? nseq : active;
        const int64_t waves = (nseq + nclusters - 1) / nclusters;
        const double per_cta = (double)((p.nc + cl - 1) / cl);
        // a hop of the state chain costs roughly a quarter of a chunk's local work
        const double chain = cl > 1 ? (double)p.nc / 4.0 : 0.0;
        const double t = (double)waves * (per_cta > chain ? per_cta : chain);
        if (t < best - 1e-9) {
            best = t;
            best_cl = cl;
            best_n = (int)nclusters;
        }
    }
    *cl_out = best_cl;
    *nclusters_out = best_n;
    if (cost_out) *cost_out = best;
    std::lock_guard<std::mutex> g(g_cache_mu);
    g_cluster_cache[g_cluster_next] = ClusterChoice{ClusterKey{dev, nseq, p.nc}, best_cl, best_n, best};
    g_cluster_next = (g_cluster_next + 1) % kCacheSlots;
    if (g_cluster_used < kCacheSlots) ++g_cluster_used;
    return SSDC_OK;
}

}  // namespace fused

bool fused_supported(int N, int D, int Q) { return N == 64 && D == 64 && Q == 64; }

int fused_cluster_choice(const Problem& p, int* cl, double* cost) {
    int n = 1;
    return fused::pick_cluster(p, cl, &n, cost);
}

int fused_launch(const Problem& p, const Workspace& ws, cudaStream_t stream, int force_cluster, bool plane_maps) {
    int cl = 1, nclusters = 1;
    int rc = fused::pick_cluster(p, &cl, &nclusters);
    if (rc != SSDC_OK) return rc;
    if (force_cluster > 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SSDC_ERR_CUDA;
        cl = force_cluster;
        const int64_t nseq = (int64_t)p.B * p.H;
        const int64_t fit = sms / cl > 0 ? sms / cl : 1;
        nclusters = (int)(nseq < fit ? nseq : fit);
    }
    fused::FusedMaps fm;
    rc = fused::cached_maps(p, plane_maps, &fm);
    if (rc != SSDC_OK) return rc;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(cl * nclusters), 1, 1);
    cfg.blockDim = dim3(fused::kThreads, 1, 1);
    cfg.dynamicSmemBytes = fused::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = (fm.swap & 4) ? cudaLaunchKernelEx(&cfg, fused::fused_kernel<true>, p, ws, fm)
                                        : cudaLaunchKernelEx(&cfg, fused::fused_kernel<false>, p, ws, fm);
    return e == cudaSuccess ? 1 : SSDC_ERR_CUDA;
}

}  // namespace ssdc
