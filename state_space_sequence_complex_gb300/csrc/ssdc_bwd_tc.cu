// The backward pass's per-chunk products on the TF32 tensor cores (tcgen05,
// operands staged by TMA, accumulators in tensor memory), for chunks of Q =
// 16, 32 or 64 tokens and N, D multiples of 8 up to 64. The same adjoint as
// the exact kernel of ssdc_bwd.cu (page "Extending -- SSM variants & Triton
// kernels", Step 3: the backward recomputes the forward, seeded with the true
// output gradients; landing page, "03 Chunkwise SSD", for the chunked form):
// with P = (C B^T) o L, W = dY x^H, V = W o conj(L) and R_c the gradient of the
// state leaving the chunk,
//   dX^T = dY^T conj(P) + R_c^T conj(dec o B)^T
//   dB^T = conj(C)^T V + R_c conj(dec o x)^T
//   dC   = V conj(B) + conj(exp(Acs)) o (dY conj(S_in)^T)
// written so that each is a sum of plain products: every conjugation and
// every per-row decay is applied to an operand when it is written (P, V and
// the transposed B as the threads form them; B, x and dY scaled in place once
// the products that read them as loaded are done; the windows as they are
// filled), never in the combine. Then r_t = <dC_t, C_t> - <dB_t, B_t> and the
// chunk's anchor <R_c, S_out(c)>, as in the exact kernel.
//
// One CTA per SM walks chunks blockIdx.x, blockIdx.x + grid, ...; 16 worker
// warps, one warp issuing the MMAs, one loading. The next chunk's tiles load
// while this chunk computes: B once the dX store has read its staging (stage
// W), dY once MMA 4 is done, x once the dB store and -<dB, B> have read it
// (stage C), and C, which stage C still reads, into the other of two stages a
// whole chunk ahead. The load warp also issues the dX and dB stores (TMA), so
// no worker waits on a store's progress.
// Complex products are M = 128, N = 128 real MMAs: the A rows interleave the
// planes in groups of eight (row 16g + 8p + i = plane p of row 8g + i: the C
// and dY tiles as loaded, and the TMEM windows), the B rows are stacked
// (64 rows of plane 0, then plane 1: the B and x tiles as loaded, and the
// tiles the threads write). One accumulator then holds all four real
// products of each complex product, in TMEM lanes m and m + 8 and columns c
// and 64 + c, which the 16x256b access shape hands to one thread.
//
// TMEM: acc0 (C B^T, then dX^T), acc1 (dY x^T, then dB^T), acc2 (dC), and
// two 64-column A windows filled three times. Stages, each ended by a
// hand-off to the MMA warp:
//   loads   C, dY (interleaved), B, x (stacked); the R_c^T window (global)
//   MMA 1   acc0 = C B^T, acc1 = dY x^T
//   P       P from acc0 -> conj(P)^T tile; BT = conj(B)^T; B' = conj(dec o B)
//           in place; the dY^T window
//   MMA 2   acc0 = dY^T conj(P) + R_c^T B'^T                         (dX^T)
//   V       dX staged and stored (TMA); V from acc1 -> V^T tile (over
//           conj(P)^T); x'' = conj(dec o x) in place; dY'' = conj(exp(Acs))
//           o dY in place; windows conj(C)^T and R_c
//   MMA 3   acc1 = conj(C)^T V + R_c x''^T                            (dB^T)
//   W       the V window (from the V^T tile); conj(S_in) tile (over V^T);
//           dB staged and stored, -<dB_l, B_l>
//   MMA 4   acc2 = V BT^T + dY'' conj(S_in)^T                          (dC)
//   C       dC stored, r_t
// Every wait is on a barrier's parity for the chunk (or for the stage's use)
// and bounded (a wait that gives up records SSDC_ERR_TIMEOUT and the later
// waits are skipped).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "fused_io.cuh"

namespace ssdc {
namespace bwdtc {
namespace {

using namespace tc;
using namespace fused;

constexpr int kWorkers = 512;
constexpr int kWorkerWarps = kWorkers / 32;
constexpr int kIssuer = kWorkerWarps;
constexpr int kProducer = kWorkerWarps + 1;
constexpr int kThreads = kWorkers + 64;
constexpr uint32_t kWorkerBar = 1;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcc0 = 0, kAcc1 = 128, kAcc2 = 256, kWa = 384, kWb = 448;

struct Smem {
    float c[2][64 * 128];  // [chunk parity] C, interleaved rows (t, plane)
    float y[64 * 128];     // dY, interleaved rows (t, plane); then dY'' in place
    float b[64 * 128];     // B, stacked rows (l, plane); then B' in place; then the dX staging (rows l)
    float x[64 * 128];     // x, stacked rows (l, plane); then x'' in place; then the dB staging (rows l)
    float bt[64 * 128];    // conj(B)^T, stacked rows (n, plane), K = l
    float pv[64 * 128];    // conj(P)^T, then V^T (stacked rows (l, plane), K = t); then conj(S_in) (rows n,
                           // K = d); once dC is formed, <dC_t, C_t> per 32-column half (float2 [2][64])
    float2 acs[2][64];     // [chunk parity]
    float2 dec[64], eacs[64];
    float2 step[64];       // exp(Acs[t] - Acs[t-1]); from stage W on, -<dB_l, B_l> (written and read by
                           // thread l alone once stage C has begun: its next step[l] is its own)
    float anc[kWorkerWarps][2];
    uint64_t full_b, full_x, full_y, full_c[2];
    uint64_t mma1, mma2, mma3, mma4, p_ready, v_ready, w_ready;
    uint64_t x_free, c_free[2];
    uint32_t tmem;
};

static_assert(sizeof(Smem) <= 232448, "shared-memory plan exceeds the 227 KB a CTA can have");

// Tensor maps of one call: C and dY in 8-row boxes (the interleaved layout),
// B and x in boxes of `rows` rows (stacked), dX and dB for the TMA stores.
struct BwdMaps {
    CUtensorMap c_re, c_im, y_re, y_im, b_re, b_im, x_re, x_im, dx_re, dx_im, db_re, db_im;
    int real_x, real_dy, dx_im_out;
};

// Element (r, k) of a 64-row plane of a stacked or interleaved tile: 32-column
// half k / 32, row r, the 128-byte swizzle.
__device__ __forceinline__ uint32_t elem(int r, int k) {
    return (uint32_t)((k >> 5) * kIntHalf + r * 128) + chunk16((k & 31) >> 2, r) + (uint32_t)(4 * (k & 3));
}
// Stacked: plane p of row r at rows 64 p + r of each half; interleaved: row 16 (r / 8) + 8 p + r % 8.
__device__ __forceinline__ uint32_t stk(int p, int r, int k) { return elem(r, k) + (uint32_t)(p * kHalfBytes); }
__device__ __forceinline__ uint32_t itl(int p, int r, int k) { return elem(inter_m(r, p), k); }
__device__ __forceinline__ float ld(const char* base, uint32_t o) { return *reinterpret_cast<const float*>(base + o); }
__device__ __forceinline__ void st(char* base, uint32_t o, float v) { *reinterpret_cast<float*>(base + o) = v; }

// Four floats at a 16-byte aligned address, read-only for the kernel.
__device__ __forceinline__ float4 ldg4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

// D (+)= A * B over K = 64, both operands in shared memory.
__device__ __forceinline__ void issue_ss(uint32_t d, uint32_t a, uint32_t b, bool accumulate) {
    const uint64_t da = desc128(a), db = desc128(b);
#pragma unroll
    for (int k = 0; k < 8; ++k)
        ptx::mma_tf32_ss(d, desc_k(da, k), desc_k(db, k), kIdesc128, (accumulate || k > 0) ? 1u : 0u);
}

// Zero the 16-byte chunk `i` (< 2048) of a 64-token tile if it holds a row
// that no load writes: a token at or past Q, or plane 1 when `real` (the
// tile's tensor has no imaginary plane). Rows of 128 bytes, 1024 chunks per
// 32-column half; the swizzle only permutes chunks within a row.
__device__ __forceinline__ void zero_unloaded(char* tile, int i, bool interleaved, int Q, bool real) {
    const int row = (i & 1023) >> 3;
    const int plane = interleaved ? (row >> 3) & 1 : row >> 6;
    const int r = interleaved ? 8 * (row >> 4) + (row & 7) : row & 63;
    if (r >= Q || (plane == 1 && real))
        *reinterpret_cast<float4*>(tile + 16 * i) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
}

__global__ void __launch_bounds__(kThreads, 1)
bwd_chunk_tc(GradProblem g, Workspace ws, GradWorkspace gw, const __grid_constant__ BwdMaps bm) {
    grid_dependency_wait();  // launched as a dependent of the state passes
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const Problem& p = g.f;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H, N = p.N, D = p.D, Q = p.Q;
    const int64_t nc = p.nc;
    const int64_t nchunks = (int64_t)p.B * H * nc;
    const int64_t mine = (int64_t)blockIdx.x < nchunks ? (nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int rows = Q < kQ ? Q : kQ;
    // rows that no load writes (tokens past Q, the planes of a real x or dY) must read as zero
    const bool dirty = Q < kQ || bm.real_x || bm.real_dy;

    if (ptx::smem_addr(smem_raw) & 1023u) {
        if (tid == 0) atomicCAS(ws.status, SSDC_OK, SSDC_ERR_CUDA);
        return;
    }
    if (tid == 0) {
        uint64_t* one[] = {&sm.full_b, &sm.full_x, &sm.full_y, &sm.full_c[0], &sm.full_c[1],
                           &sm.mma1,   &sm.mma2,   &sm.mma3,   &sm.mma4,      &sm.c_free[0], &sm.c_free[1]};
        for (uint64_t* bar : one) ptx::mbar_init(bar, 1);
        ptx::mbar_init(&sm.p_ready, kWorkerWarps);
        ptx::mbar_init(&sm.v_ready, kWorkerWarps);
        ptx::mbar_init(&sm.w_ready, kWorkerWarps);
        ptx::mbar_init(&sm.x_free, kWorkerWarps);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(&sm.tmem, kTmemCols);
        ptx::tmem_relinquish();
    }
    if (dirty) {
        float4* z = reinterpret_cast<float4*>(sm.c);
        constexpr int kVecs = 5 * 64 * 128 / 4;  // the two C tiles, dY, B and x
        for (int i = tid; i < kVecs; i += kThreads) z[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem;
    auto chunk_at = [&](int64_t k) { return (int64_t)blockIdx.x + k * gridDim.x; };

    if (warp == kProducer) {
        // ===================== loads, the cumulative log-decay, the stores =====================
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (lane == 0 && ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
            __syncwarp();
        };
        const int ng = rows >> 3;
        // batch b, head h and first token t0 of chunk ch (b H + h) nc + c (every index below 2^31)
        auto coords = [&](int64_t ch, int* b, int* h, int* t0) {
            const uint32_t c32 = (uint32_t)ch, bh = c32 / (uint32_t)nc;
            *b = (int)(bh / (uint32_t)H);
            *h = (int)(bh % (uint32_t)H);
            *t0 = (int)(c32 - bh * (uint32_t)nc) * Q;
        };
        // tile `which` (0: C into stage st, 1: dY, 2: B, 3: x) of chunk ch, counted on `bar`. C and
        // dY: 8-row boxes per plane and half (rows 16 g + 8 pl); B and x: one box per plane and half
        auto load = [&](int which, int st, int64_t ch, uint64_t* bar) {
            int b, h, t0;
            coords(ch, &b, &h, &t0);
            if (which < 2) {
                for (int k = lane; k < 4 * ng; k += 32) {
                    const int half = k / (2 * ng), gg = (k >> 1) % ng, pl = k & 1;
                    if (which == 1 && pl == 1 && bm.real_dy) continue;
                    char* dst = reinterpret_cast<char*>(which ? sm.y : sm.c[st]) + half * kIntHalf + (16 * gg + 8 * pl) * 128;
                    const CUtensorMap* m = which ? (pl ? &bm.y_im : &bm.y_re) : (pl ? &bm.c_im : &bm.c_re);
                    ptx::tma_load_4d(dst, m, bar, 32 * half, h, t0 + 8 * gg, b);
                }
            } else if (lane < 4) {
                const int half = lane >> 1, pl = lane & 1;
                if (!(which == 3 && pl == 1 && bm.real_x)) {
                    char* dst = reinterpret_cast<char*>(which == 3 ? sm.x : sm.b) + half * kIntHalf + pl * kHalfBytes;
                    const CUtensorMap* m = which == 3 ? (pl ? &bm.x_im : &bm.x_re) : (pl ? &bm.b_im : &bm.b_re);
                    ptx::tma_load_4d(dst, m, bar, 32 * half, h, t0, b);
                }
            }
        };
        auto expect = [&](uint64_t* bar, uint32_t planes) {
            if (lane == 0) ptx::mbar_arrive_expect_tx(bar, (uint32_t)rows * 256u * planes);
            __syncwarp();
        };
        // C and Acs of chunk ch into stage st
        auto load_c = [&](int64_t ch, int st) {
            int b, h, t0;
            coords(ch, &b, &h, &t0);
            const Alog al = load_alog(p, b, h, t0, lane, rows);
            if (lane == 0) ptx::mbar_expect_tx(&sm.full_c[st], (uint32_t)rows * 512u);
            __syncwarp();
            load(0, st, ch, &sm.full_c[st]);
            store_acs(sm.acs[st], &sm.full_c[st], al, lane);
        };
        // the dX or dB staging of chunk ch (rows l of the B or x tile) to global memory
        auto store = [&](int64_t ch, const CUtensorMap* re, const CUtensorMap* im, const float* tile) {
            if (lane == 0) {
                int b, h, t0;
                coords(ch, &b, &h, &t0);
                const char* buf = reinterpret_cast<const char*>(tile);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    ptx::tma_store_4d(re, buf + half * kIntHalf, 32 * half, h, t0, b);
                    if (im != nullptr) ptx::tma_store_4d(im, buf + half * kIntHalf + kHalfBytes, 32 * half, h, t0, b);
                }
                ptx::bulk_commit();
            }
            __syncwarp();
        };
        auto stores_read = [&]() {  // every store issued so far has read its staging
            if (lane == 0) ptx::bulk_wait_read_all();
            __syncwarp();
        };
        if (mine > 0) {
            const int64_t ch = chunk_at(0);
            load_c(ch, 0);
            expect(&sm.full_b, 2u);
            load(2, 0, ch, &sm.full_b);
            expect(&sm.full_y, bm.real_dy ? 1u : 2u);
            load(1, 0, ch, &sm.full_y);
            expect(&sm.full_x, bm.real_x ? 1u : 2u);
            load(3, 0, ch, &sm.full_x);
            if (mine > 1) load_c(chunk_at(1), 1);
        }
        // per chunk: its stores, and each tile of the next chunk as soon as this one is done with it
        for (int64_t j = 0; j < mine; ++j) {
            const int64_t ch = chunk_at(j), nx = chunk_at(j + 1);
            const uint32_t ph = (uint32_t)j & 1u;
            const bool more = j + 1 < mine;
            wait(&sm.v_ready, ph);  // dX is staged in the B tile (B' was consumed by MMA 2)
            store(ch, &bm.dx_re, bm.dx_im_out ? &bm.dx_im : nullptr, sm.b);
            if (more) {
                stores_read();
                expect(&sm.full_b, 2u);
                load(2, 0, nx, &sm.full_b);
            }
            wait(&sm.w_ready, ph);  // dB is staged in the x tile (x'' was consumed by MMA 3)
            store(ch, &bm.db_re, &bm.db_im, sm.x);
            if (more) {
                wait(&sm.mma4, ph);  // MMA 4 has read dY''
                expect(&sm.full_y, bm.real_dy ? 1u : 2u);
                load(1, 0, nx, &sm.full_y);
                wait(&sm.x_free, ph);  // -<dB, B> has read the staging
                stores_read();
                expect(&sm.full_x, bm.real_x ? 1u : 2u);
                load(3, 0, nx, &sm.full_x);
            }
            if (j + 2 < mine) {  // C two chunks on, into the stage this chunk used
                wait(&sm.c_free[j & 1], (uint32_t)(j >> 1) & 1u);
                load_c(chunk_at(j + 2), (int)(j & 1));
            }
        }
        if (lane == 0) ptx::bulk_wait_all();  // the stores are complete before the CTA leaves
        __syncwarp();
    } else if (warp == kIssuer) {
        // ===================== MMA issue =====================
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
        };
        const uint32_t ys = ptx::smem_addr(sm.y), bs = ptx::smem_addr(sm.b), xs = ptx::smem_addr(sm.x);
        const uint32_t bts = ptx::smem_addr(sm.bt), pvs = ptx::smem_addr(sm.pv);
        for (int64_t j = 0; j < mine && lane == 0; ++j) {
            const uint32_t ph = (uint32_t)j & 1u;
            const int st = (int)(j & 1);
            wait(&sm.full_c[st], (uint32_t)(j >> 1) & 1u);
            wait(&sm.full_b, ph);
            wait(&sm.full_y, ph);
            wait(&sm.full_x, ph);
            // the unloaded rows are zero again (the accumulators were read before the previous
            // chunk's last hand-off, which this thread waited for)
            if (dirty && j > 0) wait(&sm.c_free[st ^ 1], (uint32_t)((j - 1) >> 1) & 1u);
            ptx::tc_fence_after();
            issue_ss(tmem + kAcc0, ptx::smem_addr(sm.c[st]), bs, false);  // C B^T
            issue_ss(tmem + kAcc1, ys, xs, false);                         // dY x^T
            ptx::mma_commit(&sm.mma1);
            wait(&sm.p_ready, ph);
            ptx::tc_fence_after();
            issue_ts128(tmem + kAcc0, tmem + kWa, desc128(pvs), false);  // dY^T conj(P)
            issue_ts128(tmem + kAcc0, tmem + kWb, desc128(bs), true);    // + R_c^T B'^T
            ptx::mma_commit(&sm.mma2);
            wait(&sm.v_ready, ph);
            ptx::tc_fence_after();
            issue_ts128(tmem + kAcc1, tmem + kWa, desc128(pvs), false);  // conj(C)^T V
            issue_ts128(tmem + kAcc1, tmem + kWb, desc128(xs), true);    // + R_c x''^T
            ptx::mma_commit(&sm.mma3);
            wait(&sm.w_ready, ph);
            ptx::tc_fence_after();
            issue_ts128(tmem + kAcc2, tmem + kWa, desc128(bts), false);  // V conj(B)
            issue_ss(tmem + kAcc2, ys, pvs, true);                       // + dY'' conj(S_in)^T
            ptx::mma_commit(&sm.mma4);
        }
        __syncwarp();
    } else {
        // ===================== 16 worker warps =====================
        // 16x256b fragment: TMEM lane quadrant qd, 16-lane block blk, 32-column half kh; lane i4
        // holds plane 0 and lane i4 + 8 plane 1 of A row rr; columns c = 32 kh + 8 j + 2 lq + e of
        // the B operand's plane 0 (first 64 columns) and plane 1 (next 64).
        const int qd = warp & 3, blk = (warp >> 2) & 1, kh = warp >> 3;
        const int i4 = lane >> 2, lq = lane & 3;
        const int rr = 16 * qd + 8 * blk + i4;
        const uint32_t tl = lane_base(tmem, warp) + ((uint32_t)(16 * blk) << 16);
        // window fill: this lane writes TMEM lane 32 qd + lane = plane wp of row wr, columns 16 wc ..
        const int wr = 16 * qd + 8 * (lane >> 4) + (lane & 7), wp = (lane >> 3) & 1, wc = warp >> 2;
        const uint32_t wl = lane_base(tmem, warp);
        char* yb = reinterpret_cast<char*>(sm.y);
        char* bb = reinterpret_cast<char*>(sm.b);
        char* xb = reinterpret_cast<char*>(sm.x);
        char* btb = reinterpret_cast<char*>(sm.bt);
        char* pvb = reinterpret_cast<char*>(sm.pv);
        float2* dct = reinterpret_cast<float2*>(sm.pv);  // [32-column half][t], after MMA 4
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
        };
        // (values v[k], k < 16, of window columns 16 wc + k) -> TMEM, rounded to TF32
        auto put_window = [&](uint32_t col0, const float* v) {
            float r[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) r[k] = ptx::to_tf32(v[k]);
            ptx::tmem_st16(wl + col0 + 16 * wc, r);
        };
        // Window of a transposed interleaved tile: row wr, column k = plane wp of T[k][wr], T with
        // rows k interleaved (C or dY); plane-1 lanes read row k ^ 4 (rows 8 apart share banks)
        auto window_from_itl = [&](const char* src, float sign1, float* v) {
            float r[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) r[k] = ld(src, itl(wp, 16 * wc + (k ^ (4 * wp)), wr));
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = (wp ? sign1 : 1.0f) * (wp ? r[k ^ 4] : r[k]);
        };
        // The same from a stacked tile with rows k (V^T)
        auto window_from_stk = [&](const char* src, float* v) {
            float r[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) r[k] = ld(src, stk(wp, 16 * wc + (k ^ (4 * wp)), wr));
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = wp ? r[k ^ 4] : r[k];
        };
        // Stage an accumulator whose A rows are features f (lanes) and B rows tokens l (stacked
        // columns) as rows l of a TMA store tile: Re = A0 B0 - A1 B1, Im = A0 B1 + A1 B0.
        auto stage_t = [&](uint32_t acc, char* buf) {
            float v0[16], v1[16];
            ptx::tmem_ld_16x256b_x4(tl + acc + 32 * kh, v0);       // products with B's plane 0
            ptx::tmem_ld_16x256b_x4(tl + acc + 64 + 32 * kh, v1);  // and with its plane 1
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int l = 32 * kh + 8 * j + 2 * lq + e;
                    st(buf, stk(0, l, rr), v0[4 * j + e] - v1[4 * j + 2 + e]);
                    st(buf, stk(1, l, rr), v1[4 * j + e] + v0[4 * j + 2 + e]);
                }
        };

        for (int64_t jc = 0; jc < mine; ++jc) {
            // (the chunk's coordinates are recomputed where they are used: few registers live
            // across the stages)
            const uint32_t ph = (uint32_t)jc & 1u;
            const int stg = (int)(jc & 1);  // the C / Acs stage
            char* cb = reinterpret_cast<char*>(sm.c[stg]);
            const float2* acs = sm.acs[stg];
            auto chunk_of = [&]() { return chunk_at(jc); };  // (b H + h) nc + c
            auto slot = [&](const float* base, int64_t ch) { return base + ch * 2 * (int64_t)D * N; };
            // ---- while the tiles load: the R_c^T window (rows d, K = n; the previous chunk's
            // products that read the windows are done) and the anchor <R_c, S_out(c)>, their loads
            // all in flight together
            {
                const int64_t chunk = chunk_of(), bh = chunk / nc;
                const bool last_chunk = chunk - bh * nc == nc - 1;
                const float* R = slot(gw.R, chunk);  // R_c^T [plane][d][n]
                const float* nxt = slot(ws.S, chunk + 1);
                float v[16];
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {  // four 16-byte loads of the row (N is a multiple of 8)
                    const int n = 16 * wc + 4 * k4;
                    const float4 q = (wr < D && n < N) ? ldg4(R + ((int64_t)wp * D + wr) * N + n)
                                                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    v[4 * k4] = q.x;
                    v[4 * k4 + 1] = q.y;
                    v[4 * k4 + 2] = q.z;
                    v[4 * k4 + 3] = q.w;
                }
                // the anchor's elements e = 8 tid .. 8 tid + 7 (D N <= 4096 is a multiple of 64)
                const int e0 = 8 * tid;
                const bool mine_e = e0 < D * N;
                float4 r4[2][2], s4[2][2];  // [plane][half]
#pragma unroll
                for (int pl = 0; pl < 2; ++pl)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int64_t o = (int64_t)pl * D * N + e0 + 4 * hf;
                        r4[pl][hf] = mine_e ? ldg4(R + o) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        s4[pl][hf] = mine_e && !last_chunk ? ldg4(nxt + o) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    }
                put_window(kWb, v);
                if (last_chunk && mine_e) {  // S_out is the final state, (b, h, n, d)
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int e = e0 + k, d = e / N, n = e - (e / N) * N;
                        const int64_t o = (bh * N + n) * D + d;
                        (&s4[0][k >> 2].x)[k & 3] = p.fs_re[o];
                        (&s4[1][k >> 2].x)[k & 3] = p.fs_im[o];
                    }
                }
                float ar = 0.0f, ai = 0.0f;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const float rr4[4] = {r4[0][hf].x, r4[0][hf].y, r4[0][hf].z, r4[0][hf].w};
                    const float ri4[4] = {r4[1][hf].x, r4[1][hf].y, r4[1][hf].z, r4[1][hf].w};
                    const float sr4[4] = {s4[0][hf].x, s4[0][hf].y, s4[0][hf].z, s4[0][hf].w};
                    const float si4[4] = {s4[1][hf].x, s4[1][hf].y, s4[1][hf].z, s4[1][hf].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        ar += rr4[k] * sr4[k] + ri4[k] * si4[k];  // R conj(S_out)
                        ai += ri4[k] * sr4[k] - rr4[k] * si4[k];
                    }
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) {
                    ar += __shfl_xor_sync(0xffffffffu, ar, off);
                    ai += __shfl_xor_sync(0xffffffffu, ai, off);
                }
                if (lane == 0) {
                    sm.anc[warp][0] = ar;
                    sm.anc[warp][1] = ai;
                }
            }
            wait(&sm.full_c[stg], (uint32_t)(jc >> 1) & 1u);
            // decay tables (thread t writes entry t of each: step[t] was its own -<dB_t, B_t>)
            if (tid < kQ) {
                const int t = tid;
                sm.dec[t] = t < Q ? cexp_fast(cdiff(acs[Q - 1], acs[t])) : make_float2(0.0f, 0.0f);
                sm.eacs[t] = cexp_fast(acs[t]);
                if (t >= 1) sm.step[t] = cexp_fast(cdiff(acs[t], acs[t - 1]));
            }
            ptx::named_sync(kWorkerBar, kWorkers);
            if (warp == 0) {  // the chunk's anchor: the warps' partial sums in a fixed tree
                float sr = lane < kWorkerWarps ? sm.anc[lane][0] : 0.0f;
                float si = lane < kWorkerWarps ? sm.anc[lane][1] : 0.0f;
#pragma unroll
                for (int off = kWorkerWarps / 2; off >= 1; off >>= 1) {
                    sr += __shfl_xor_sync(0xffffffffu, sr, off);
                    si += __shfl_xor_sync(0xffffffffu, si, off);
                }
                if (lane == 0) {
                    gw.anchor[2 * chunk_of()] = sr;
                    gw.anchor[2 * chunk_of() + 1] = si;
                }
            }

            // decay L[rr, col] of a causal pair (t = rr >= l = col), from one exponential per column pair
            auto decay_pair = [&](int col, float2* L0, float2* L1) {
                *L0 = make_float2(0.0f, 0.0f);
                *L1 = make_float2(0.0f, 0.0f);
                if (col + 1 <= rr) {
                    *L1 = cexp_fast(cdiff(acs[rr], acs[col + 1]));
                    *L0 = cmul(*L1, sm.step[col + 1]);
                } else if (col == rr) {
                    *L0 = make_float2(1.0f, 0.0f);
                }
            };

            // ---- stage P (after C B^T and dY x^T)
            wait(&sm.mma1, ph);
            wait(&sm.full_b, ph);  // complete already (the MMA warp waited): the tiles' bytes are visible
            wait(&sm.full_y, ph);
            wait(&sm.full_x, ph);
            ptx::tc_fence_after();
            {
                float ga[16], gb[16];
                ptx::tmem_ld_16x256b_x4(tl + kAcc0 + 32 * kh, ga);
                ptx::tmem_ld_16x256b_x4(tl + kAcc0 + 64 + 32 * kh, gb);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int col = 32 * kh + 8 * j + 2 * lq;
                    float2 L0, L1;
                    decay_pair(col, &L0, &L1);
                    // G = C B^T: Re = Cr Br - Ci Bi, Im = Cr Bi + Ci Br
                    const float2 g0 = make_float2(ga[4 * j] - gb[4 * j + 2], gb[4 * j] + ga[4 * j + 2]);
                    const float2 g1 = make_float2(ga[4 * j + 1] - gb[4 * j + 3], gb[4 * j + 1] + ga[4 * j + 3]);
                    const float2 p0 = cmul(g0, L0), p1 = cmul(g1, L1);
                    // conj(P)^T: row l = col (+1), column t = rr
                    st(pvb, stk(0, col, rr), ptx::to_tf32(p0.x));
                    st(pvb, stk(1, col, rr), ptx::to_tf32(-p0.y));
                    st(pvb, stk(0, col + 1, rr), ptx::to_tf32(p1.x));
                    st(pvb, stk(1, col + 1, rr), ptx::to_tf32(-p1.y));
                }
            }
            {
                // BT = conj(B)^T, then B' = conj(dec o B) in place. Blocks: rows l = 4 bsb + i, columns
                // n = 4 bnb + 2 bjh + {0, 1}; each thread rewrites exactly the B elements it read.
                const int L0b = lane & 1, L1b = (lane >> 1) & 1, L2b = (lane >> 2) & 1, L3b = (lane >> 3) & 1, L4b = lane >> 4;
                const int bjh = L1b, bsb = L2b + 2 * (warp >> 1), bnb = L0b + 2 * L3b + 4 * L4b + 8 * (warp & 1);
                float2 bv[2][4];
#pragma unroll
                for (int pp = 0; pp < 2; ++pp)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        bv[pp][i] = *reinterpret_cast<const float2*>(bb + stk(pp, 4 * bsb + i, 4 * bnb + 2 * bjh));
                using ptx::to_tf32;
#pragma unroll
                for (int jn = 0; jn < 2; ++jn) {  // 16-byte rows of BT: row n, columns l = 4 bsb .. + 3
                    const int n = 4 * bnb + 2 * bjh + jn;
                    float r4[4], i4v[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        r4[i] = to_tf32(jn ? bv[0][i].y : bv[0][i].x);
                        i4v[i] = to_tf32(-(jn ? bv[1][i].y : bv[1][i].x));
                    }
                    *reinterpret_cast<float4*>(btb + stk(0, n, 4 * bsb)) = make_float4(r4[0], r4[1], r4[2], r4[3]);
                    *reinterpret_cast<float4*>(btb + stk(1, n, 4 * bsb)) = make_float4(i4v[0], i4v[1], i4v[2], i4v[3]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int l = 4 * bsb + i, n = 4 * bnb + 2 * bjh;
                    const float2 dv = sm.dec[l];
                    // conj(dec B): Re = dr br - di bi, Im = -(dr bi + di br)
                    *reinterpret_cast<float2*>(bb + stk(0, l, n)) =
                        make_float2(to_tf32(dv.x * bv[0][i].x - dv.y * bv[1][i].x), to_tf32(dv.x * bv[0][i].y - dv.y * bv[1][i].y));
                    *reinterpret_cast<float2*>(bb + stk(1, l, n)) =
                        make_float2(to_tf32(-(dv.x * bv[1][i].x + dv.y * bv[0][i].x)),
                                    to_tf32(-(dv.x * bv[1][i].y + dv.y * bv[0][i].y)));
                }
            }
            {
                float v[16];
                window_from_itl(yb, 1.0f, v);  // dY^T
                put_window(kWa, v);
            }
            ptx::tmem_wait_st();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm.p_ready);

            // ---- stage V (after dX^T). The R_c window's loads are issued before the wait.
            float rwin[16];
            const float* R = slot(gw.R, chunk_of());
#pragma unroll
            for (int k = 0; k < 16; ++k) {  // R_c: rows n, K = d
                const int d = 16 * wc + k;
                rwin[k] = (wr < N && d < D) ? __ldg(R + ((int64_t)wp * D + d) * N + wr) : 0.0f;
            }
            wait(&sm.mma2, ph);
            ptx::tc_fence_after();
            put_window(kWb, rwin);
            ptx::named_sync(kWorkerBar, kWorkers);  // every worker is past its B and dY reads
            stage_t(kAcc0, bb);                     // dX (B' is consumed)
            {
                float ga[16], gb[16];
                ptx::tmem_ld_16x256b_x4(tl + kAcc1 + 32 * kh, ga);
                ptx::tmem_ld_16x256b_x4(tl + kAcc1 + 64 + 32 * kh, gb);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int col = 32 * kh + 8 * j + 2 * lq;
                    float2 L0, L1;
                    decay_pair(col, &L0, &L1);
                    // W = dY conj(x): Re = Yr xr + Yi xi, Im = Yi xr - Yr xi
                    const float2 w0 = make_float2(ga[4 * j] + gb[4 * j + 2], ga[4 * j + 2] - gb[4 * j]);
                    const float2 w1 = make_float2(ga[4 * j + 1] + gb[4 * j + 3], ga[4 * j + 3] - gb[4 * j + 1]);
                    const float2 v0 = cmul(w0, make_float2(L0.x, -L0.y)), v1 = cmul(w1, make_float2(L1.x, -L1.y));
                    st(pvb, stk(0, col, rr), ptx::to_tf32(v0.x));  // V^T
                    st(pvb, stk(1, col, rr), ptx::to_tf32(v0.y));
                    st(pvb, stk(0, col + 1, rr), ptx::to_tf32(v1.x));
                    st(pvb, stk(1, col + 1, rr), ptx::to_tf32(v1.y));
                }
            }
            {
                // x'' = conj(dec o x) in place: same blocks as B (rows l, columns d)
                const int L0b = lane & 1, L1b = (lane >> 1) & 1, L2b = (lane >> 2) & 1, L3b = (lane >> 3) & 1, L4b = lane >> 4;
                const int bjh = L1b, bsb = L2b + 2 * (warp >> 1), bnb = L0b + 2 * L3b + 4 * L4b + 8 * (warp & 1);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int l = 4 * bsb + i, d = 4 * bnb + 2 * bjh;
                    const float2 dv = sm.dec[l];
                    float2* p0 = reinterpret_cast<float2*>(xb + stk(0, l, d));
                    float2* p1 = reinterpret_cast<float2*>(xb + stk(1, l, d));
                    const float2 xr = *p0, xi = *p1;
                    using ptx::to_tf32;
                    *p0 = make_float2(to_tf32(dv.x * xr.x - dv.y * xi.x), to_tf32(dv.x * xr.y - dv.y * xi.y));
                    *p1 = make_float2(to_tf32(-(dv.x * xi.x + dv.y * xr.x)), to_tf32(-(dv.x * xi.y + dv.y * xr.y)));
                }
            }
            {
                // dY'' = conj(exp(Acs[t])) dY in place: rows t = 8 gq + i (planes at rows 16 gq + i, + 8),
                // columns 4 jq .. 4 jq + 3 of half hq; physical 16-byte chunks, the factor per row
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int u = tid + kWorkers * k;
                    const int jq = u & 7, i = (u >> 3) & 7, gq = (u >> 6) & 7, hq = u >> 9;
                    char* r0 = yb + hq * kIntHalf + (16 * gq + i) * 128 + 16 * jq;
                    char* r1 = r0 + 8 * 128;
                    const float2 e = sm.eacs[8 * gq + i];
                    const float4 a = *reinterpret_cast<const float4*>(r0), q = *reinterpret_cast<const float4*>(r1);
                    using ptx::to_tf32;
                    // (er - i ei)(yr + i yi) = er yr + ei yi + i (er yi - ei yr)
                    *reinterpret_cast<float4*>(r0) =
                        make_float4(to_tf32(e.x * a.x + e.y * q.x), to_tf32(e.x * a.y + e.y * q.y),
                                    to_tf32(e.x * a.z + e.y * q.z), to_tf32(e.x * a.w + e.y * q.w));
                    *reinterpret_cast<float4*>(r1) =
                        make_float4(to_tf32(e.x * q.x - e.y * a.x), to_tf32(e.x * q.y - e.y * a.y),
                                    to_tf32(e.x * q.z - e.y * a.z), to_tf32(e.x * q.w - e.y * a.w));
                }
            }
            {
                float v[16];
                window_from_itl(cb, -1.0f, v);  // conj(C)^T
                put_window(kWa, v);
            }
            ptx::fence_proxy_async_smem();
            ptx::named_sync(kWorkerBar, kWorkers);  // the dX staging is written (the load warp stores it)
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm.v_ready);

            // ---- stage W (after dB^T). The S_in loads (8 elements a thread) are issued before the wait.
            float sinr[8], sini[8];
            const float* Sin = slot(ws.S, chunk_of());  // S_in^T [plane][d][n]
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int e = tid + kWorkers * k, d = e >> 6, n = e & 63;
                const bool in = d < D && n < N;
                sinr[k] = in ? __ldg(Sin + (int64_t)d * N + n) : 0.0f;
                sini[k] = in ? __ldg(Sin + (int64_t)D * N + (int64_t)d * N + n) : 0.0f;
            }
            wait(&sm.mma3, ph);
            ptx::tc_fence_after();
            {
                float v[16];
                window_from_stk(pvb, v);  // V: rows t, K = l, from V^T
                put_window(kWa, v);
            }
            ptx::named_sync(kWorkerBar, kWorkers);  // every V^T read is done
            {
                // conj(S_in): rows n, K = d, from S_in^T [plane][d][n]
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int e = tid + kWorkers * k, d = e >> 6, n = e & 63;
                    st(pvb, stk(0, n, d), ptx::to_tf32(sinr[k]));
                    st(pvb, stk(1, n, d), ptx::to_tf32(-sini[k]));
                }
            }
            stage_t(kAcc1, xb);  // dB (x'' is consumed)
            ptx::fence_proxy_async_smem();
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::named_sync(kWorkerBar, kWorkers);
            if (lane == 0) ptx::mbar_arrive(&sm.w_ready);  // (the load warp stores dB)
            {
                // -<dB_l, B_l> = -sum_n dB[l, n] conj(B[l, n]), conj(B[l, n]) = BT[n][l]: 8 threads a row
                const int l = tid >> 3, s8 = tid & 7;
                float sr = 0.0f, si = 0.0f;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int n = 8 * s8 + ((k + s8) & 7);  // rotated: the eight lanes of a row read BT rows of distinct swizzles
                    const float dr = ld(xb, stk(0, l, n)), di = ld(xb, stk(1, l, n));
                    const float br = ld(btb, stk(0, n, l)), bi = ld(btb, stk(1, n, l));
                    sr += dr * br - di * bi;
                    si += dr * bi + di * br;
                }
#pragma unroll
                for (int off = 1; off < 8; off <<= 1) {
                    sr += __shfl_xor_sync(0xffffffffu, sr, off);
                    si += __shfl_xor_sync(0xffffffffu, si, off);
                }
                if (s8 == 0) sm.step[l] = make_float2(-sr, -si);  // every step read was before the last sync
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm.x_free);  // this warp is done with x

            // ---- stage C (after dC)
            wait(&sm.mma4, ph);
            ptx::tc_fence_after();
            {
                float ga[16], gb[16];
                ptx::tmem_ld_16x256b_x4(tl + kAcc2 + 32 * kh, ga);
                ptx::tmem_ld_16x256b_x4(tl + kAcc2 + 64 + 32 * kh, gb);
                ptx::tmem_wait_ld();
                const int64_t chunk = chunk_of(), bh = chunk / nc, t0 = (chunk - bh * nc) * Q;
                const bool row_ok = t0 + rr < p.T && rr < Q;
                const int64_t tok = ((bh / H) * p.T + t0 + rr) * H + bh % H;
                float sr = 0.0f, si = 0.0f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int n = 32 * kh + 8 * j + 2 * lq;
                    const float2 d0 = make_float2(ga[4 * j] - gb[4 * j + 2], gb[4 * j] + ga[4 * j + 2]);
                    const float2 d1 = make_float2(ga[4 * j + 1] - gb[4 * j + 3], gb[4 * j + 1] + ga[4 * j + 3]);
                    if (row_ok && n < N) {  // N is a multiple of 8: n + 1 < N too
                        *reinterpret_cast<float2*>(g.dC_re + tok * N + n) = make_float2(d0.x, d1.x);
                        *reinterpret_cast<float2*>(g.dC_im + tok * N + n) = make_float2(d0.y, d1.y);
                    }
                    // <dC_t, C_t> = sum dC conj(C)
                    const float c0r = ld(cb, itl(0, rr, n)), c0i = ld(cb, itl(1, rr, n));
                    const float c1r = ld(cb, itl(0, rr, n + 1)), c1i = ld(cb, itl(1, rr, n + 1));
                    sr += d0.x * c0r + d0.y * c0i + d1.x * c1r + d1.y * c1i;
                    si += d0.y * c0r - d0.x * c0i + d1.y * c1r - d1.x * c1i;
                }
                sr += __shfl_xor_sync(0xffffffffu, sr, 1);
                si += __shfl_xor_sync(0xffffffffu, si, 1);
                sr += __shfl_xor_sync(0xffffffffu, sr, 2);
                si += __shfl_xor_sync(0xffffffffu, si, 2);
                if (lq == 0) dct[64 * kh + rr] = make_float2(sr, si);  // pv is free: MMA 4 is done
            }
            ptx::named_sync(kWorkerBar, kWorkers);  // every C read is done, dct is written
            if (dirty) {
                // B', x'', dY'' and the stagings wrote rows that the next loads leave alone: zero them
                // (dY, x: MMA 4 and the dB store are done reading; B: the dX store)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = tid + kWorkers * k;
                    zero_unloaded(bb, i, false, Q, false);
                    zero_unloaded(xb, i, false, Q, bm.real_x);
                    zero_unloaded(yb, i, true, Q, bm.real_dy);
                }
                ptx::fence_proxy_async_smem();
                ptx::named_sync(kWorkerBar, kWorkers);
            }
            if (tid == 0) ptx::mbar_arrive(&sm.c_free[stg]);  // C and Acs of this stage are free
            if (tid < 64) {
                const int64_t chunk = chunk_of(), bh = chunk / nc, t0 = (chunk - bh * nc) * Q;
                const float2 a = dct[tid], q = dct[64 + tid], nb = sm.step[tid];
                float* rre = gw.r + bh * 2 * p.T;
                if (tid < Q && t0 + tid < p.T) {
                    rre[t0 + tid] = a.x + q.x + nb.x;
                    rre[p.T + t0 + tid] = a.y + q.y + nb.y;
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
}

constexpr size_t kSmemBytes = sizeof(Smem);
bool g_attr_set[64] = {};

int make_maps(const GradProblem& g, BwdMaps* m) {
    const Problem& p = g.f;
    memset(m, 0, sizeof(*m));
    m->real_x = p.x_im == nullptr;
    m->real_dy = g.dy_im == nullptr;
    m->dx_im_out = g.dx_im != nullptr;
    const int rows = p.Q < kQ ? p.Q : kQ;
    bool ok = encode_feature_map(&m->c_re, p.C_re, p.N, p.H, p.T, p.B, 8) &&
              encode_feature_map(&m->c_im, p.C_im, p.N, p.H, p.T, p.B, 8) &&
              encode_feature_map(&m->y_re, g.dy_re, p.D, p.H, p.T, p.B, 8) &&
              (m->real_dy || encode_feature_map(&m->y_im, g.dy_im, p.D, p.H, p.T, p.B, 8)) &&
              encode_feature_map(&m->b_re, p.B_re, p.N, p.H, p.T, p.B, rows) &&
              encode_feature_map(&m->b_im, p.B_im, p.N, p.H, p.T, p.B, rows) &&
              encode_feature_map(&m->x_re, p.x_re, p.D, p.H, p.T, p.B, rows) &&
              (m->real_x || encode_feature_map(&m->x_im, p.x_im, p.D, p.H, p.T, p.B, rows)) &&
              encode_feature_map(&m->dx_re, g.dx_re, p.D, p.H, p.T, p.B, rows) &&
              (!m->dx_im_out || encode_feature_map(&m->dx_im, g.dx_im, p.D, p.H, p.T, p.B, rows)) &&
              encode_feature_map(&m->db_re, g.dB_re, p.N, p.H, p.T, p.B, rows) &&
              encode_feature_map(&m->db_im, g.dB_im, p.N, p.H, p.T, p.B, rows);
    return ok ? SSDC_OK : SSDC_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Per chunk, on the tensor cores: the forward's local state and the adjoint's
// input of the chunk,
//   S_loc^T = x^T (dec o B)          -> ws.S slot of the chunk, [plane][d][n]
//   U^T     = dY^T conj(C')          -> gw.R slot, C' = exp(Acs) o C
// and a_c = exp(Acs[Q-1]) (the exact kernel's outputs, in the same layouts).
// A operands are TMEM windows (x^T, dY^T) read from the stacked tiles by
// column; B operands are the B and C tiles transposed in place (rows n, K =
// the token), the decay and the conjugation applied as they are written.
//
// One CTA per SM walks chunks blockIdx.x, blockIdx.x + grid, ...: x and dY are
// free once the windows are built (early in a chunk), so the next chunk's x and
// dY load during this chunk's transposes, products and output; B and C, which
// the products read, have two stages, so the next chunk's B and C load during
// this whole chunk. Every wait is on a barrier's parity for the chunk (or the
// stage's use), bounded.

struct StatesSmem {
    float x[64 * 128];  // x, stacked (rows s)
    float y[64 * 128];     // dY, stacked (rows l)
    float b[2][64 * 128];  // [stage] B, stacked; then (dec o B)^T in place (rows n, K = s)
    float c[2][64 * 128];  // [stage] C, stacked; then conj(C')^T in place (rows n, K = l)
    float2 acs[2][64];     // [chunk parity]
    float2 dec[64], eacs[64];
    uint64_t full_xy, xy_free, ready, done, acc_free;
    uint64_t full_bc[2], bc_free[2];  // [stage]
    uint32_t tmem;
};

static_assert(sizeof(StatesSmem) <= 232448, "shared-memory plan exceeds the 227 KB a CTA can have");

struct StatesMaps {
    CUtensorMap x_re, x_im, b_re, b_im, y_re, y_im, c_re, c_im;  // boxes (32, 1, rows, 1)
    int real_x, real_dy;
};

__global__ void __launch_bounds__(kThreads, 1)
bwd_states_tc(GradProblem g, Workspace ws, GradWorkspace gw, const __grid_constant__ StatesMaps sm_maps) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    StatesSmem& sm = *reinterpret_cast<StatesSmem*>(smem_raw);
    const StatesMaps& mp = sm_maps;
    const Problem& p = g.f;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H, N = p.N, D = p.D, Q = p.Q;
    const int64_t nc = p.nc;
    const int64_t nchunks = (int64_t)p.B * H * nc;
    const int64_t mine = (int64_t)blockIdx.x < nchunks ? (nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int rows = Q < kQ ? Q : kQ;
    constexpr uint32_t kS = 0, kU = 128, kWx = 256, kWy = 320;

    if (ptx::smem_addr(smem_raw) & 1023u) {
        if (tid == 0) atomicCAS(ws.status, SSDC_OK, SSDC_ERR_CUDA);
        return;
    }
    if (tid == 0) {
        ptx::mbar_init(&sm.full_xy, 1);
        ptx::mbar_init(&sm.xy_free, kWorkerWarps);
        for (int st = 0; st < 2; ++st) {
            ptx::mbar_init(&sm.full_bc[st], 1);
            ptx::mbar_init(&sm.bc_free[st], 1);
        }
        ptx::mbar_init(&sm.ready, kWorkerWarps);
        ptx::mbar_init(&sm.done, 1);
        ptx::mbar_init(&sm.acc_free, kWorkerWarps);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(&sm.tmem, kTmemCols);
        ptx::tmem_relinquish();
    }
    {
        // rows past Q and the planes of a real x or dY are never loaded: zero (x and dY are only
        // read, so they stay zero; the rows past Q of B and C meet zero window columns)
        float4* z = reinterpret_cast<float4*>(sm.x);
        constexpr int kVecs = 6 * 64 * 128 / 4;  // the six tiles
        for (int i = tid; i < kVecs; i += kThreads) z[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem;
    auto chunk_at = [&](int64_t k) { return (int64_t)blockIdx.x + k * gridDim.x; };

    if (warp == kProducer) {
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (lane == 0 && ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
            __syncwarp();
        };
        // tensor `which` (x, B, dY, C) of chunk (b, h, t0) into its tile (B and C: stage st):
        // lanes (32-column half, plane)
        auto load = [&](int which, int st, int b, int h, int64_t t0) {
            if (lane < 4) {
                const int half = lane >> 1, pl = lane & 1;
                const bool skip = pl == 1 && ((which == 0 && mp.real_x) || (which == 2 && mp.real_dy));
                if (!skip) {
                    float* tiles[4] = {sm.x, sm.b[st], sm.y, sm.c[st]};
                    const CUtensorMap* maps[4][2] = {{&mp.x_re, &mp.x_im}, {&mp.b_re, &mp.b_im},
                                                     {&mp.y_re, &mp.y_im}, {&mp.c_re, &mp.c_im}};
                    char* dst = reinterpret_cast<char*>(tiles[which]) + half * kIntHalf + pl * kHalfBytes;
                    ptx::tma_load_4d(dst, maps[which][pl], which == 0 || which == 2 ? &sm.full_xy : &sm.full_bc[st],
                                     32 * half, h, (int)t0, b);
                }
            }
        };
        for (int64_t k = 0; k < mine; ++k) {
            const int64_t chunk = chunk_at(k);
            const int64_t bh = chunk / nc;
            const int b = (int)(bh / H), h = (int)(bh % H);
            const int64_t t0 = (chunk % nc) * Q;
            const uint32_t pp = (uint32_t)(k - 1) & 1u;  // the previous chunk's parity (x and dY)
            // x and dY: after the previous chunk's windows are built
            if (k > 0) wait(&sm.xy_free, pp);
            const Alog al = load_alog(p, b, h, t0, lane, rows);
            if (lane == 0) {
                const uint32_t planes = 4u - (mp.real_x ? 1u : 0u) - (mp.real_dy ? 1u : 0u);
                ptx::mbar_expect_tx(&sm.full_xy, (uint32_t)rows * 256u * planes);
            }
            __syncwarp();
            load(0, 0, b, h, t0);
            load(2, 0, b, h, t0);
            store_acs(sm.acs[k & 1], &sm.full_xy, al, lane);
            // B and C into stage k & 1: after the products of chunk k - 2, its previous use
            const int st = (int)(k & 1);
            if (k >= 2) wait(&sm.bc_free[st], (uint32_t)((k >> 1) - 1) & 1u);
            if (lane == 0) ptx::mbar_arrive_expect_tx(&sm.full_bc[st], (uint32_t)rows * 256u * 4u);
            __syncwarp();
            load(1, st, b, h, t0);
            load(3, st, b, h, t0);
        }
    } else if (warp == kIssuer) {
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
        };
        for (int64_t k = 0; k < mine && lane == 0; ++k) {
            wait(&sm.ready, (uint32_t)k & 1u);
            if (k > 0) wait(&sm.acc_free, (uint32_t)(k - 1) & 1u);  // the accumulators were read out
            ptx::tc_fence_after();
            const int st = (int)(k & 1);
            issue_ts128(tmem + kS, tmem + kWx, desc128(ptx::smem_addr(sm.b[st])), false);  // x^T (dec o B)
            issue_ts128(tmem + kU, tmem + kWy, desc128(ptx::smem_addr(sm.c[st])), false);  // dY^T conj(C')
            ptx::mma_commit(&sm.done);
            ptx::mma_commit(&sm.bc_free[st]);
        }
        __syncwarp();
    } else {
        const int qd = warp & 3, blk = (warp >> 2) & 1, kh = warp >> 3;
        const int i4 = lane >> 2, lq = lane & 3;
        const int rr = 16 * qd + 8 * blk + i4;
        const uint32_t tl = lane_base(tmem, warp) + ((uint32_t)(16 * blk) << 16);
        const int wr = 16 * qd + 8 * (lane >> 4) + (lane & 7), wp = (lane >> 3) & 1, wc = warp >> 2;
        const uint32_t wl = lane_base(tmem, warp);
        char* xb = reinterpret_cast<char*>(sm.x);
        char* yb = reinterpret_cast<char*>(sm.y);
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
        };
        // windows x^T and dY^T: row wr (d), column k (token) = plane wp of T[k][wr] from a stacked
        // tile; plane-1 lanes read row k ^ 4 (the planes' rows share banks)
        auto window = [&](const char* src, uint32_t col0) {
            float r[16], v[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) r[k] = ld(src, stk(wp, 16 * wc + (k ^ (4 * wp)), wr));
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = ptx::to_tf32(wp ? r[k ^ 4] : r[k]);
            ptx::tmem_st16(wl + col0 + 16 * wc, v);
        };
        const int L0 = lane & 1, L1 = (lane >> 1) & 1, L2 = (lane >> 2) & 1, L3 = (lane >> 3) & 1, L4 = lane >> 4;
        const int bjh = L1, bsb = L2 + 2 * (warp >> 1), bnb = L0 + 2 * L3 + 4 * L4 + 8 * (warp & 1);
        for (int64_t k = 0; k < mine; ++k) {
            const int64_t chunk = chunk_at(k);
            const uint32_t ph = (uint32_t)k & 1u;
            // ---- the chunk's decay tables and windows (the previous chunk's products, which read
            // the windows, are done: this warp waited for them before its output stage)
            wait(&sm.full_xy, ph);
            if (tid < 2 * kQ) {
                const float2* acs = sm.acs[k & 1];
                const int t = tid % kQ;
                if (tid < kQ) sm.dec[t] = t < Q ? cexp_fast(cdiff(acs[Q - 1], acs[t])) : make_float2(0.0f, 0.0f);
                else sm.eacs[t] = cexp_fast(acs[t]);
            }
            window(xb, kWx);
            window(yb, kWy);
            ptx::tmem_wait_st();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm.xy_free);  // this warp is done with x and dY
            // ---- B and C blocks (stage k & 1): rows s = 4 bsb + i, columns n = 4 bnb + 2 bjh + {0, 1}
            const int st = (int)(k & 1);
            char* bb = reinterpret_cast<char*>(sm.b[st]);
            char* cb = reinterpret_cast<char*>(sm.c[st]);
            wait(&sm.full_bc[st], (uint32_t)(k >> 1) & 1u);
            float2 bv[2][4], cv[2][4];
#pragma unroll
            for (int pp = 0; pp < 2; ++pp)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int sr = 4 * bsb + i, n = 4 * bnb + 2 * bjh;
                    bv[pp][i] = make_float2(ld(bb, stk(pp, sr, n)), ld(bb, stk(pp, sr, n + 1)));
                    cv[pp][i] = make_float2(ld(cb, stk(pp, sr, n)), ld(cb, stk(pp, sr, n + 1)));
                }
            ptx::named_sync(kWorkerBar, kWorkers);  // every B and C read is done; the tables are written
#pragma unroll
            for (int jn = 0; jn < 2; ++jn) {  // column n -> row n of the transposed tiles
                const int nr = 4 * bnb + 2 * bjh + jn;
                float br[4], bi[4], cr[4], ci[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int sr = 4 * bsb + i;
                    const float2 bvv = jn ? make_float2(bv[0][i].y, bv[1][i].y) : make_float2(bv[0][i].x, bv[1][i].x);
                    const float2 cvv = jn ? make_float2(cv[0][i].y, cv[1][i].y) : make_float2(cv[0][i].x, cv[1][i].x);
                    const float2 db = cmul(sm.dec[sr], bvv);   // dec o B
                    const float2 ce = cmul(sm.eacs[sr], cvv);  // C' = exp(Acs) o C, conjugated below
                    br[i] = ptx::to_tf32(db.x);
                    bi[i] = ptx::to_tf32(db.y);
                    cr[i] = ptx::to_tf32(ce.x);
                    ci[i] = ptx::to_tf32(-ce.y);
                }
                *reinterpret_cast<float4*>(bb + stk(0, nr, 4 * bsb)) = make_float4(br[0], br[1], br[2], br[3]);
                *reinterpret_cast<float4*>(bb + stk(1, nr, 4 * bsb)) = make_float4(bi[0], bi[1], bi[2], bi[3]);
                *reinterpret_cast<float4*>(cb + stk(0, nr, 4 * bsb)) = make_float4(cr[0], cr[1], cr[2], cr[3]);
                *reinterpret_cast<float4*>(cb + stk(1, nr, 4 * bsb)) = make_float4(ci[0], ci[1], ci[2], ci[3]);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm.ready);
            // ---- output: S_loc^T and U^T rows d = rr: Re = A0 B0 - A1 B1, Im = A0 B1 + A1 B0
            wait(&sm.done, ph);
            ptx::tc_fence_after();
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                float ga[16], gb[16];
                ptx::tmem_ld_16x256b_x4(tl + (which ? kU : kS) + 32 * kh, ga);
                ptx::tmem_ld_16x256b_x4(tl + (which ? kU : kS) + 64 + 32 * kh, gb);
                ptx::tmem_wait_ld();
                float* out = (which ? gw.R : ws.S) + chunk * 2 * (int64_t)D * N;
                if (rr < D) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int n = 32 * kh + 8 * j + 2 * lq;
                        if (n < N) {  // N is a multiple of 8: n + 1 < N too
                            *reinterpret_cast<float2*>(out + rr * N + n) =
                                make_float2(ga[4 * j] - gb[4 * j + 2], ga[4 * j + 1] - gb[4 * j + 3]);
                            *reinterpret_cast<float2*>(out + (int64_t)D * N + rr * N + n) =
                                make_float2(gb[4 * j] + ga[4 * j + 2], gb[4 * j + 1] + ga[4 * j + 3]);
                        }
                    }
                }
            }
            if (tid == 0) {
                const float2 a = sm.eacs[Q - 1];
                ws.a[2 * chunk] = a.x;
                ws.a[2 * chunk + 1] = a.y;
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm.acc_free);  // this warp has read the accumulators
            // the next chunk's tables overwrite dec and eacs: every warp's transposes and a_c are done
            ptx::named_sync(kWorkerBar, kWorkers);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
}

constexpr size_t kStatesSmemBytes = sizeof(StatesSmem);
bool g_states_attr_set[64] = {};

int make_states_maps(const GradProblem& g, StatesMaps* m) {
    const Problem& p = g.f;
    memset(m, 0, sizeof(*m));
    m->real_x = p.x_im == nullptr;
    m->real_dy = g.dy_im == nullptr;
    const int rows = p.Q < kQ ? p.Q : kQ;
    bool ok = encode_feature_map(&m->x_re, p.x_re, p.D, p.H, p.T, p.B, rows) &&
              (m->real_x || encode_feature_map(&m->x_im, p.x_im, p.D, p.H, p.T, p.B, rows)) &&
              encode_feature_map(&m->b_re, p.B_re, p.N, p.H, p.T, p.B, rows) &&
              encode_feature_map(&m->b_im, p.B_im, p.N, p.H, p.T, p.B, rows) &&
              encode_feature_map(&m->y_re, g.dy_re, p.D, p.H, p.T, p.B, rows) &&
              (m->real_dy || encode_feature_map(&m->y_im, g.dy_im, p.D, p.H, p.T, p.B, rows)) &&
              encode_feature_map(&m->c_re, p.C_re, p.N, p.H, p.T, p.B, rows) &&
              encode_feature_map(&m->c_im, p.C_im, p.N, p.H, p.T, p.B, rows);
    return ok ? SSDC_OK : SSDC_ERR_CUDA;
}

}  // namespace
}  // namespace bwdtc

bool bwd_tc_supported(int N, int D, int Q) {
    return (Q == 16 || Q == 32 || Q == 64) && N >= 8 && N <= 64 && N % 8 == 0 && D >= 8 && D <= 64 && D % 8 == 0;
}

int bwd_tc_launch_chunk(const GradProblem& g, const Workspace& ws, const GradWorkspace& gw, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SSDC_ERR_CUDA;
    if (!bwdtc::g_attr_set[dev]) {
        if (cudaFuncSetAttribute(bwdtc::bwd_chunk_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bwdtc::kSmemBytes) != cudaSuccess)
            return SSDC_ERR_CUDA;
        bwdtc::g_attr_set[dev] = true;
    }
    bwdtc::BwdMaps m;
    const int rc = bwdtc::make_maps(g, &m);
    if (rc != SSDC_OK) return rc;
    const Problem& p = g.f;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return SSDC_ERR_CUDA;
    const int64_t chunks = (int64_t)p.B * p.H * p.nc;
    const unsigned grid = (unsigned)(chunks < sms ? chunks : sms);  // one CTA per SM walks the chunks
    if (launch_dependent(bwdtc::bwd_chunk_tc, dim3(grid), dim3(bwdtc::kThreads), bwdtc::kSmemBytes, stream, g, ws,
                         gw, m) != cudaSuccess)
        return SSDC_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? 1 : SSDC_ERR_CUDA;
}

int bwd_tc_launch_chunk_states(const GradProblem& g, const Workspace& ws, const GradWorkspace& gw,
                               cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SSDC_ERR_CUDA;
    if (!bwdtc::g_states_attr_set[dev]) {
        if (cudaFuncSetAttribute(bwdtc::bwd_states_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bwdtc::kStatesSmemBytes) != cudaSuccess)
            return SSDC_ERR_CUDA;
        bwdtc::g_states_attr_set[dev] = true;
    }
    bwdtc::StatesMaps m;
    const int rc = bwdtc::make_states_maps(g, &m);
    if (rc != SSDC_OK) return rc;
    const Problem& p = g.f;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return SSDC_ERR_CUDA;
    const int64_t chunks = (int64_t)p.B * p.H * p.nc;
    const unsigned grid = (unsigned)(chunks < sms ? chunks : sms);  // one CTA per SM walks the chunks
    bwdtc::bwd_states_tc<<<grid, bwdtc::kThreads, bwdtc::kStatesSmemBytes, stream>>>(g, ws, gw, m);
    return cudaGetLastError() == cudaSuccess ? 1 : SSDC_ERR_CUDA;
}

}  // namespace ssdc
