// Fused single-pass forward of the chunkwise complex SSD scan on the TF32
// tensor cores with the chunk state held in tensor memory (Q = 16, 32, 64, 128
// or 256; N and D multiples of 8 up to 64). One CTA per SM walks whole (b, h)
// sequences chunk by chunk; every step of the chunked decomposition (landing
// page, "03 Chunkwise SSD": L, Y_diag = (C B^T o L) X, the per-chunk state,
// the pass between chunks, Y_off) runs in this one launch.
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
// Blocks. Tiles are 64 tokens. A chunk of Q >= 64 tokens is R = Q / 64 row
// tiles r, and its quadratic part the lower-triangular blocks (r, j), j <= r:
//     Y_r^T = sum_{j <= r} X_j^T P_rj^T + S_in^T C'_r^T,
//     P_rj[l, s] = (C_r B_j^T)[l, s] exp(Acs[64 r + l] - Acs[64 j + s])
// (causal inside the diagonal block only), each block a C B^T, a P and a
// Y_diag MMA, with C_r, B_j and x_j loaded for it (the tiles of earlier
// blocks come again from L2). Y_r accumulates over its row's blocks in TMEM;
// the diagonal block also adds its column's share of the chunk state (the
// (dec o B)^T MMA, accumulated over the rows) and row r's Y_off, and the last
// one forms the state leaving the chunk. The items of a CTA are the blocks in
// this order, row by row; for Q <= 64 a chunk is one diagonal block.
//
// Threads: 16 worker warps (phases below), warp 16 issues every MMA in block
// order on mbarrier hand-offs, warp 17 issues the TMA loads of the block after
// next into the other stage and computes each chunk's cumulative log-decay.
// Each of the three tiles of a stage is released as soon as its last reader
// is done (x after its columns are read and the y staged in it is stored, C
// after C B^T or Y_off, B after Y_diag), so the loads of block k+2 start
// during block k.
//
// Smaller shapes run on the same 64-row, 64-column tiles. Feature columns past
// N or D are read as zeros by the tensor maps (and never stored), so they add
// nothing to any product. A chunk of Q < 64 tokens fills the first Q rows of
// its tiles; the other rows keep finite values from earlier use (the tiles are
// zeroed at the start), and every product that reads them is masked: the decay
// dec[s] is zero for s >= Q, P is causal, and y rows past Q are not stored
// (the TMA store boxes are Q rows high).
//
// Worker phases of block (r, j) (stage s):
//   A  the chunk's decay tables (first block); X^T window of x_j; (B_j rows)
//   B  diagonal: (dec o B_j)^T in place of B    -> state MMA
//   D  first block of a row: y of the previous row, staged in this x tile
//   C  diagonal: C'_r in place of C             -> Y_off MMA (S_in^T window)
//   E  P_rj = (C_r B_j^T) o L into the B tile   -> Y_diag MMA
//   F  last block of the chunk: S_out^T = a_c S_in^T + S_loc^T into the S
//      window (or the final state)
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
constexpr int kMaxQc = 256;  // the largest chunk
// TMEM columns: three 128-column accumulators (C B^T; Y^T; S_loc^T) and two
// 64-column A windows (X^T; S_in^T).
constexpr uint32_t kAccG = 0, kAccY = 128, kAccS = 256, kXwin = 384, kSwin = 448;
constexpr int kPlane16 = 64 * 128;  // bytes of one 64-row plane of a bfloat16 tile
constexpr uint32_t kIdescBf16 = ptx::idesc_bf16(128, 128);

// Decay tables, barriers and the TMEM address: the part common to both input types.
struct Tail {
    float2 acs[2][kMaxQc];   // [chunk parity] in-chunk cumulative log-decay
    float2 dec[2][kMaxQc];   // [chunk parity] exp(Acs[Q-1] - Acs[s]), zero past Q
    float2 eacs[2][kMaxQc];  // [chunk parity] exp(Acs[l])
    float2 step[2][kMaxQc];  // [chunk parity] exp(Acs[s] - Acs[s-1]) (s >= 1)
    float2 a_c[2];           // [chunk parity] exp(Acs[Q-1])
    uint64_t full[2];                          // stage loaded (tiles, and a chunk's decays)
    uint64_t free_x[2], free_b[2], free_c[2];  // stage tiles released
    uint64_t xt_ready, bt_ready, c_ready, p_ready, sin_ready;  // worker hand-offs (one arrival per warp)
    uint64_t mma_g, mma_s, mma_yo, mma_y;      // MMA completions
    uint32_t tmem;
    int mix_task;            // fused head mixer: the tile whose share this CTA mixes now, or -1
    int mix_pend;            // fused head mixer: the next tile of the current sequence to mix a share of
    float wmix[16 * 16];     // fused head mixer: W, zero past H
};

template <bool kBf16>
struct Smem;
// fp32 inputs: the stage tiles are also the tiles the threads rewrite.
template <>
struct Smem<false> : Tail {
    alignas(1024) float c[2][64 * 128];  // [stage] C (interleaved, A of C B^T), then C' in place (B of Y_off)
    float b[2][64 * 128];  // [stage] B (stacked), then (dec o B)^T (stacked, rows n), then P (interleaved)
    float x[2][64 * 128];  // [stage] x (stacked): read into the X^T window; then y staging
};
// bfloat16 inputs: 16 KB stage tiles (a 128-byte row of 64 features per token and plane, the
// same row orders as above), read by C B^T and by the threads; what the threads compute goes to
// fp32 work tiles in the fp32 layouts.
template <>
struct Smem<true> : Tail {
    alignas(1024) uint16_t c[2][64 * 128];  // [stage] C (interleaved), A of C B^T
    uint16_t b[2][64 * 128];                // [stage] B (stacked), B of C B^T
    uint16_t x[2][64 * 128];                // [stage] x (stacked)
    alignas(1024) float cw[64 * 128];       // C' (interleaved), B of Y_off
    float bw[64 * 128];                     // (dec o B)^T (stacked, rows n), then P (interleaved)
    float yw[64 * 128];                     // y staging (stacked)
};

static_assert(sizeof(Smem<false>) <= 232448 && sizeof(Smem<true>) <= 232448,
              "shared-memory plan exceeds the 227 KB a CTA can have");

// Block (r, j) of chunk c of sequence q = b H + h.
struct Item {
    int q, c, r, j;
};

__device__ __forceinline__ Item item_at(int q, int c, int r, int j) {
    Item it;
    it.q = q;
    it.c = c;
    it.r = r;
    it.j = j;
    return it;
}

// The items of this CTA, in order: the blocks of every chunk of sequences
// blockIdx.x, blockIdx.x + gridDim.x, ..., row by row. (Without kBlocks every
// chunk is one block, r = j = 0, and the compiler drops the block logic.)
template <bool kBlocks>
__device__ __forceinline__ Item item_next(const Item& p, int R, int nc) {
    if (kBlocks && p.j < p.r) return item_at(p.q, p.c, p.r, p.j + 1);
    if (kBlocks && p.r + 1 < R) return item_at(p.q, p.c, p.r + 1, 0);
    if (p.c + 1 < nc) return item_at(p.q, p.c + 1, 0, 0);
    return item_at(p.q + (int)gridDim.x, 0, 0, 0);
}

// Producer: TMA of one block's C (interleaved) into a stage buffer, counted on
// `bar` (x and B: load_x, load_b of the shared header).
__device__ __forceinline__ void load_c(char* dst, const FusedMaps& fm, uint64_t* bar, int h, int t0, int b, int64_t T,
                                       int rows, int lane) {
    if (lane == 0) ptx::mbar_expect_tx(bar, (uint32_t)(rows * 128 * 4));
    __syncwarp();
    if ((fm.fast >> 2) & 1) {
        if (lane < 2)
            ptx::tma_load_5d(dst + inter_row(lane, 0), &fm.C2, bar, 32 * lane, h, 0, 0, (int)(((int64_t)b * T + t0) >> 3));
    } else {  // rows 8g .. 8g+7 of plane pl, per 32-column half (rows / 8 groups)
        const int ng = rows >> 3;
        if (lane < 4 * ng) {
            const int half = lane / (2 * ng), g = (lane >> 1) % ng, pl = lane & 1;
            ptx::tma_load_4d(dst + inter_row(half, 16 * g + 8 * pl), pl ? &fm.c8_im : &fm.c8_re, bar, 32 * half, h,
                             t0 + 8 * g, b);
        }
    }
}

// The same for bfloat16 inputs: one box of 64 features (one 128-byte row) per
// token and plane; the per-plane maps only.
__device__ __forceinline__ void load_x16(char* dst, const FusedMaps& fm, uint64_t* bar, int h, int t0, int b, int rows,
                                         int lane) {
    const int n = fm.real_x ? 1 : 2;
    if (lane == 0) ptx::mbar_expect_tx(bar, (uint32_t)(rows * 128 * n));
    __syncwarp();
    if (lane < n) ptx::tma_load_4d(dst + lane * kPlane16, lane ? &fm.x_im : &fm.x_re, bar, 0, h, t0, b);
}

__device__ __forceinline__ void load_b16(char* dst, const FusedMaps& fm, uint64_t* bar, int h, int t0, int b, int rows,
                                         int lane) {
    if (lane == 0) ptx::mbar_expect_tx(bar, (uint32_t)(rows * 128 * 2));
    __syncwarp();
    if (lane < 2) ptx::tma_load_4d(dst + lane * kPlane16, lane ? &fm.B_im : &fm.B_re, bar, 0, h, t0, b);
}

__device__ __forceinline__ void load_c16(char* dst, const FusedMaps& fm, uint64_t* bar, int h, int t0, int b, int rows,
                                         int lane) {
    if (lane == 0) ptx::mbar_expect_tx(bar, (uint32_t)(rows * 128 * 2));
    __syncwarp();
    if (lane < 2 * (rows >> 3)) {  // rows 8g .. 8g+7 of plane pl land at rows 16g + 8pl
        const int g = lane >> 1, pl = lane & 1;
        ptx::tma_load_4d(dst + (16 * g + 8 * pl) * 128, pl ? &fm.c8_im : &fm.c8_re, bar, 0, h, t0 + 8 * g, b);
    }
}

// C_r [B_j]^T from the bfloat16 tiles: 4 MMAs of K = 16 (32 bytes of each 128-byte row).
__device__ __forceinline__ void issue_g16(uint32_t d, uint32_t a_base, uint32_t b_base) {
    const uint64_t da = desc128(a_base), db = desc128(b_base);
#pragma unroll
    for (int k = 0; k < 4; ++k) ptx::mma_f16_ss(d, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), kIdescBf16, k > 0 ? 1u : 0u);
}

// Offset of the bfloat16 element (row r, feature f) in a 128-byte swizzled row of a 16-bit tile.
__device__ __forceinline__ uint32_t off16(int r, int f) {
    return (uint32_t)(r * 128) + chunk16(f >> 3, r) + (uint32_t)((f & 7) << 1);
}

// kBlocks: chunks of Q = 128 or 256 tokens, several 64 x 64 blocks each.
// kBf16: x, B_t and C_t in bfloat16. C B^T then multiplies them as they are
// (kind::f16, exact products); x enters the X^T window and B and C the
// threads' products as exact fp32 values, the rest is as for fp32 inputs.
// kMix: the head mixer fused into the epilogue (single-block chunks only).
template <bool kSwapC, bool kBlocks, bool kBf16, bool kMix = false>
__global__ void __launch_bounds__(kThreads, 1)
fused2_kernel(Problem p, Workspace ws, const __grid_constant__ FusedMaps fm) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    Smem<kBf16>& sm = *reinterpret_cast<Smem<kBf16>*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H, nc = (int)p.nc, Q = p.Q, N = p.N, D = p.D;
    const int rows = Q < kQ ? Q : kQ;  // tile rows holding tokens
    const int R = kBlocks ? Q / kQ : 1;  // row tiles per chunk
    const int nseq = p.B * H;
    const int nseq_cta = (int)blockIdx.x < nseq ? (nseq - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int nitems = nseq_cta * nc * (R * (R + 1) / 2);
    const int mix_ntiles = (int)((p.T + rows - 1) / rows);  // fused head mixer: row tiles per sequence
    // The four TMA stores of a staged y tile (two 32-column halves of each plane) leave from lane
    // 0 of worker warps 0-3, one each, in the bfloat16 and the block instances, so that no warp
    // carries all four on its way to the next phase (each then waits for its store to read the
    // tile and releases the x tile); in the fp32 single-block instance thread 0 issues all four,
    // which measured faster there. (tid & kYMask) == 0 selects the issuing threads.
    constexpr int kYWarps = (kBf16 || kBlocks) && !kMix ? 4 : 1;
    constexpr int kYMask = ~((kYWarps - 1) << 5);

    // the swizzled tiles need a 1024-byte aligned base (uniform across the grid)
    if (ptx::smem_addr(smem_raw) & 1023u) {
        if (tid == 0) atomicCAS(ws.status, SSDC_OK, SSDC_ERR_CUDA);
        return;
    }
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&sm.full[s], 1);
            ptx::mbar_init(&sm.free_x[s], kYWarps);
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
    if (kMix && tid == 0) sm.mix_pend = 0;
    if (kMix)
        for (int i = tid; i < 16 * 16; i += kThreads)
            sm.wmix[i] = ((i >> 4) < H && (i & 15) < H) ? p.mix_w[(i >> 4) * H + (i & 15)] : 0.0f;
    if (Q < kQ) {
        // rows past Q are never loaded: give them finite contents
        float4* z = reinterpret_cast<float4*>(sm.c);
        constexpr int kVecs = (int)(3 * sizeof(sm.c) / 16);  // the c, b and x tiles of both stages
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
        Item ld = item_at((int)blockIdx.x, 0, 0, 0);
        int chunks = 0;  // chunks begun by this CTA
        // single-block chunks: the next chunk's dt is read ahead, while this one's tiles load
        Alog al = {};
        if (!kBlocks && nitems > 0) al = load_alog(p, ld.q / H, ld.q % H, 0, lane, Q);
        for (int k = 0; k < nitems; ++k) {  // item k into stage k & 1
            const int st = k & 1;
            const uint32_t ph = (uint32_t)((k - 2) >> 1) & 1u;
            const int tc0 = ld.c * Q, tr = tc0 + kQ * ld.r, tj = tc0 + kQ * ld.j;
            const int bb = ld.q / H, hh = ld.q - bb * H;
            char* xd = reinterpret_cast<char*>(sm.x[st]);
            char* cd = reinterpret_cast<char*>(sm.c[st]);
            char* bd = reinterpret_cast<char*>(sm.b[st]);
            if (k >= 2) wait(&sm.free_x[st], ph);
            if constexpr (kBf16) load_x16(xd, fm, &sm.full[st], hh, tj, bb, rows, lane);
            else load_x(xd, fm, &sm.full[st], hh, tj, bb, rows, lane);
            if (k >= 2) wait(&sm.free_c[st], ph);
            if constexpr (kBf16) load_c16(cd, fm, &sm.full[st], hh, tr, bb, rows, lane);
            else load_c(cd, fm, &sm.full[st], hh, tr, bb, p.T, rows, lane);
            if (k >= 2) wait(&sm.free_b[st], ph);
            if constexpr (kBf16) load_b16(bd, fm, &sm.full[st], hh, tj, bb, rows, lane);
            else load_b(bd, fm, &sm.full[st], hh, tj, bb, rows, lane);
            const Item nx = item_next<kBlocks>(ld, R, nc);
            if (!kBlocks) {  // every block is a chunk and carries its decays
                const Alog now = al;
                if (k + 1 < nitems) {
                    const int nb = nx.q / H;
                    al = load_alog(p, nb, nx.q - nb * H, (int64_t)nx.c * Q, lane, Q);
                }
                store_acs(sm.acs[st], &sm.full[st], now, lane);
            } else {
                if (ld.r == 0 && ld.j == 0) {
                    chunk_acs(p, bb, hh, tc0, Q, lane, sm.acs[chunks & 1]);
                    ++chunks;
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm.full[st]);
            }
            ld = nx;
        }
    } else if (warp == kIssuer) {
        // ============ MMA warp: lane 0 issues every MMA in block order ============
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
        };
        Item cur = item_at((int)blockIdx.x, 0, 0, 0);
        int ndiag = 0, nchunk = 0;  // diagonal blocks and chunks issued
        bool row_acc = false;       // the row's Y^T accumulator holds a product already
        for (int k = 0; k < nitems && lane == 0; ++k) {
            const int s = k & 1;
            const uint32_t ph = (uint32_t)k & 1u, pd = (uint32_t)ndiag & 1u;
            const bool diag = cur.j == cur.r;
            const bool has_in = cur.c > 0 || p.s0_re != nullptr;
            const uint32_t cs = ptx::smem_addr(sm.c[s]), bs = ptx::smem_addr(sm.b[s]);
            uint32_t cw = cs, bw = bs;  // the tiles the threads write: C'; (dec o B)^T and P
            if constexpr (kBf16) {
                cw = ptx::smem_addr(sm.cw);
                bw = ptx::smem_addr(sm.bw);
            }
            if (cur.j == 0) row_acc = false;
            wait(&sm.full[s], (uint32_t)((k >> 1) & 1));
            ptx::tc_fence_after();
            if constexpr (kBf16) issue_g16(tmem + kAccG, cs, bs);  // C_r [B_j0 | B_j1]^T
            else issue_ss128(tmem + kAccG, desc128(cs), desc128(bs));
            ptx::mma_commit(&sm.mma_g);
            if (!diag) ptx::mma_commit(&sm.free_c[s]);  // C is read by C B^T only
            wait(&sm.xt_ready, ph);
            if (diag) {
                wait(&sm.bt_ready, pd);
                ptx::tc_fence_after();
                issue_ts128(tmem + kAccS, tmem + kXwin, desc128(bw), cur.r > 0);  // + X_j^T (dec o B_j)
                ptx::mma_commit(&sm.mma_s);
                wait(&sm.c_ready, pd);
                if (cur.r == 0) wait(&sm.sin_ready, (uint32_t)nchunk & 1u);  // the chunk's incoming state
                ptx::tc_fence_after();
                if (has_in) {
                    issue_ts128(tmem + kAccY, tmem + kSwin, desc128(cw), row_acc);  // S_in^T C'_r^T
                    row_acc = true;
                }
                ptx::mma_commit(&sm.mma_yo);
                ptx::mma_commit(&sm.free_c[s]);
            }
            wait(&sm.p_ready, ph);
            ptx::tc_fence_after();
            issue_ts128(tmem + kAccY, tmem + kXwin, desc128(bw), row_acc);  // + X_j^T P_rj^T
            row_acc = true;
            ptx::mma_commit(&sm.mma_y);
            ptx::mma_commit(&sm.free_b[s]);
            if (diag) ++ndiag;
            if (diag && cur.r == R - 1) ++nchunk;
            cur = item_next<kBlocks>(cur, R, nc);
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
        // Offsets that follow the planes' order in the tiles (fm.swap): held in registers by the
        // fp32 single-block instance and read where they are used by the others, whichever keeps
        // each instance off register spills.
        constexpr bool kSwapAtUse = kBf16 || kBlocks || kMix;
        const int swx0 = fm.swap & 1, swb0 = (fm.swap >> 1) & 1;
        const uint32_t gbr0 = kAccG + 64 * swb0, gbi0 = kAccG + 64 * (1 - swb0);
        auto swx = [&] { return kSwapAtUse ? (fm.swap & 1) : swx0; };
        auto swb = [&] { return kSwapAtUse ? ((fm.swap >> 1) & 1) : swb0; };
        auto gbr = [&] { return kSwapAtUse ? kAccG + 64 * ((fm.swap >> 1) & 1) : gbr0; };  // B_r products
        auto gbi = [&] { return kSwapAtUse ? kAccG + 64 * (1 - ((fm.swap >> 1) & 1)) : gbi0; };  // B_i
        constexpr int kCr = kSwapC ? 1 : 0;              // C plane in TMEM lane plane 0 / 1
        constexpr int kRr = 2 * kCr, kRi = 2 - 2 * kCr;  // register offset of the C_r / C_i lanes
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
        // y rows of the row tile `row` from the Y^T accumulator (lanes (d, plane of X), columns
        // 16g + 8p + i = plane p of token 8g + i of P and of C') into the staging tile `buf`
        // (two stacked planes, rows l, the 128-byte swizzle of the TMA boxes; the four rows and
        // eight columns of a warp's store fall on distinct 16-byte positions), then, once every
        // worker has written its part, the tile leaves in four TMA copies (rows past T are not
        // written) from the threads that kYWarps names, each committing its own bulk group.
        auto stage_y = [&](char* buf, const Item& row) {
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
            if constexpr (kMix) {
                const int t0 = row.c * Q + kQ * row.r, yb = row.q / H, yh = row.q - yb * H;
                // Re(y) only, by every worker with 16-byte stores (rows past T or the chunk skipped),
                // so that a fence of each thread publishes it before the tile is counted
                const int nrow = (int)(p.T - t0 < (int64_t)rows ? p.T - t0 : (int64_t)rows);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int u = tid + kWorkers * k, l = u >> 4, dq = u & 15;
                    if (l < nrow && 4 * dq < D) {
                        const float4 v4 = *reinterpret_cast<const float4*>(buf + stk_row(dq >> 3, 0, l) + chunk16(dq & 7, l));
                        *reinterpret_cast<float4*>(p.y_re + (((int64_t)yb * p.T + t0 + l) * H + yh) * D + 4 * dq) = v4;
                    }
                }
            } else if ((tid & kYMask) == 0) {
                const int t0 = row.c * Q + kQ * row.r, yb = row.q / H, yh = row.q - yb * H;
                // (y_im is absent only with the fused head mixer, which stores above; the fp32
                // instances keep the test, which leaves them without register spills)
                if constexpr (kYWarps == 1) {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        ptx::tma_store_4d(&fm.y_re, buf + stk_row(half, 0, 0), 32 * half, yh, t0, yb);
                        if (kBf16 || fm.y_im_out) ptx::tma_store_4d(&fm.y_im, buf + stk_row(half, 1, 0), 32 * half, yh, t0, yb);
                    }
                } else {
                    const int half = warp & 1, plane = warp >> 1;
                    if (plane == 0) ptx::tma_store_4d(&fm.y_re, buf + stk_row(half, 0, 0), 32 * half, yh, t0, yb);
                    else if (kBf16 || fm.y_im_out) ptx::tma_store_4d(&fm.y_im, buf + stk_row(half, 1, 0), 32 * half, yh, t0, yb);
                }
                ptx::bulk_commit();
            }
        };

        // Fused head mixer (kMix): each CTA stores its sequence's Re(y) tile by tile and counts
        // every stored tile per (batch row, tile). The mixing of a tile, out[t, g, :] =
        // sum_h W[g, h] Re(y)[t, h, :], is shared out by head: the CTA of head h mixes the h-th
        // 1 / H of the tile's tokens, in place, once all H heads have stored the tile. A CTA
        // mixes its ready shares after each tile it stores without waiting, and waits (bounded)
        // only for the shares still open after its sequence's last tile. (Such a wait is for heads
        // whose CTAs are in the same round of sequences, or in the next round after their own;
        // with at least H CTAs no two waits form a cycle.)
        auto mix_share = [&](int mb, int mh, int tile) {
            const int64_t mt0 = (int64_t)tile * rows;
            const int nt = (int)(p.T - mt0 < (int64_t)rows ? p.T - mt0 : (int64_t)rows);
            const int lo = (mh * nt) / H, hi = ((mh + 1) * nt) / H;
            for (int e = tid; e < (hi - lo) * D; e += kWorkers) {
                const int tt = lo + e / D, d = e - (e / D) * D;
                float* col = p.y_re + (((int64_t)mb * p.T + mt0 + tt) * H) * D + d;
                float v[16];
#pragma unroll
                for (int hh = 0; hh < 16; ++hh) v[hh] = hh < H ? __ldcg(col + (int64_t)hh * D) : 0.0f;
#pragma unroll
                for (int g = 0; g < 16; ++g) {
                    if (g < H) {
                        float o = 0.0f;
#pragma unroll
                        for (int hh = 0; hh < 16; ++hh) o = fmaf(sm.wmix[g * 16 + hh], v[hh], o);
                        col[(int64_t)g * D] = o;
                    }
                }
            }
        };
        auto mix_after_store = [&](const Item& row) {
            const int mb = row.q / H, mh = row.q - mb * H;
            const int tile = (row.c * Q + kQ * row.r) / rows;
            const bool last_tile = tile == mix_ntiles - 1;
            int* cnt = p.mix_count + (int64_t)mb * mix_ntiles;
            // every worker's Re(y) stores precede the barrier; the release fence of the counting
            // thread is cumulative over them
            ptx::named_sync(kWorkerBar, kWorkers);
            if (tid == 0) {
                __threadfence();
                atomicAdd(cnt + tile, 1);
            }
            for (;;) {
                if (tid == 0) {
                    int task = -1;
                    const int pend = sm.mix_pend;
                    if (pend <= tile) {
                        volatile int* c = cnt + pend;
                        bool ready = *c >= H;
                        if (!ready && last_tile) {
                            const uint64_t t_start = ptx::globaltimer_ns();
                            while (*c < H) {
                                if (ptx::globaltimer_ns() - t_start > kWaitIters) {
                                    fail(ws.status);
                                    break;
                                }
                                __nanosleep(256);
                            }
                            ready = true;
                        }
                        if (ready) {
                            __threadfence();
                            task = pend;
                            sm.mix_pend = pend + 1;
                        }
                    }
                    sm.mix_task = task;
                }
                ptx::named_sync(kWorkerBar, kWorkers);
                const int task = sm.mix_task;
                ptx::named_sync(kWorkerBar, kWorkers);  // every worker has read the task
                if (task < 0) break;
                mix_share(mb, mh, task);
            }
            if (tid == 0 && last_tile) sm.mix_pend = 0;  // the next sequence starts at its tile 0
        };

        Item cur = item_at((int)blockIdx.x, 0, 0, 0);
        // the S window of the first chunk: its initial state, if any
        if (nitems > 0 && p.s0_re != nullptr) {
            store_s0(cur.q);
            ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.sin_ready);

        int ndiag = 0, nchunk = 0;  // diagonal blocks and chunks begun
        for (int it = 0; it < nitems; ++it) {
            Item mix_row = cur;  // the row tile staged in this item (fused head mixer)
            const int s = it & 1;
            const uint32_t ph = (uint32_t)it & 1u, pd = (uint32_t)ndiag & 1u;
            const bool diag = cur.j == cur.r;
            const bool chunk_first = cur.r == 0 && cur.j == 0, chunk_last = diag && cur.r == R - 1;
            const bool staged = it > 0 && cur.j == 0;  // the previous row's y goes out through this x tile
            const bool has_in = cur.c > 0 || p.s0_re != nullptr;
            const int cp = kBlocks ? (chunk_first ? nchunk : nchunk - 1) & 1 : s;  // the chunk's table parity
            const int orow = kQ * cur.r, ocol = kQ * cur.j;          // token offsets in the chunk
            char* xbase = reinterpret_cast<char*>(sm.x[s]);
            char* bbase = reinterpret_cast<char*>(sm.b[s]);
            char* cbase = reinterpret_cast<char*>(sm.c[s]);
            // where the threads write C', (dec o B)^T and P, and stage y
            char* cwork = cbase;
            char* bwork = bbase;
            char* ystage = xbase;
            if constexpr (kBf16) {
                cwork = reinterpret_cast<char*>(sm.cw);
                bwork = reinterpret_cast<char*>(sm.bw);
                ystage = reinterpret_cast<char*>(sm.yw);
            }
            if (chunk_first) ++nchunk;
            wait(&sm.full[s], (uint32_t)((it >> 1) & 1));
            // the previous block's MMAs are complete: the X^T window and the Y^T accumulator are free
            if (it > 0) wait(&sm.mma_y, ph ^ 1u);
            ptx::tc_fence_after();

            // ---- A: the chunk's decay tables; X^T window; B rows into registers
            if (chunk_first) {
                // over the rows of the chunk's tiles (Q, or 64 for a shorter chunk)
                const float2 last_acs = sm.acs[cp][Q - 1];
                const int Qe = kBlocks ? Q : kQ;
                for (int i = tid; i < 3 * Qe; i += kWorkers) {
                    const int which = i >= 2 * Qe ? 2 : (i >= Qe ? 1 : 0), t = i - which * Qe;
                    if (which == 0) {  // zero past the chunk's Q tokens (rows holding no token of it)
                        sm.dec[cp][t] = t < Q ? cexp_fast(cdiff(last_acs, sm.acs[cp][t])) : make_float2(0.0f, 0.0f);
                    } else if (which == 1) {
                        sm.eacs[cp][t] = cexp_fast(sm.acs[cp][t]);
                    } else if (t >= 1) {
                        sm.step[cp][t] = cexp_fast(cdiff(sm.acs[cp][t], sm.acs[cp][t - 1]));
                    }
                }
                if (tid == 0) sm.a_c[cp] = cexp_fast(last_acs);
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
                } else if constexpr (kBf16) {  // exact in TF32: no rounding
                    const char* planebase = xbase + xp * kPlane16;
                    float r[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int sr = 16 * cg + (k ^ (4 * xp));
                        r[k] = ptx::bf16_lo(*reinterpret_cast<const uint16_t*>(planebase + off16(sr, xd)));
                    }
#pragma unroll
                    for (int k = 0; k < 16; ++k) v[k] = xp ? r[k ^ 4] : r[k];
                } else {
                    const char* rowbase = xbase + stk_row(xd >> 5, xp ^ swx(), 0) + 4 * (xd & 3);
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
            if (diag) {
#pragma unroll
                for (int pp = 0; pp < 2; ++pp)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int sr = 4 * bsb + i;
                        if constexpr (kBf16) {
                            const uint32_t two = *reinterpret_cast<const uint32_t*>(
                                bbase + pp * kPlane16 + off16(sr, 4 * bnb + 2 * bjh));
                            bv[pp][i] = make_float2(ptx::bf16_lo(two), ptx::bf16_hi(two));
                        } else {
                            bv[pp][i] = *reinterpret_cast<const float2*>(bbase + stk_row(bnb >> 3, pp ^ swb(), sr) +
                                                                         chunk16(bnb & 7, sr) + 8 * bjh);
                        }
                    }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::named_sync(kWorkerBar, kWorkers);
            // every worker has read x; the tile is free at once, unless the previous row's y is
            // staged in it below (then once its TMA stores have read it)
            if ((kBf16 || !staged) && (tid & kYMask) == 0) ptx::mbar_arrive(&sm.free_x[s]);
            if (lane == 0) ptx::mbar_arrive(&sm.xt_ready);

            // ---- B: (dec o B_j)^T in place of B (after C B^T has read it)
            wait(&sm.mma_g, ph);
            if (diag) {
                float2 dv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) dv[i] = sm.dec[cp][ocol + 4 * bsb + i];
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
                    *reinterpret_cast<float4*>(bwork + stk_row(bsb >> 3, 0, nr) + chunk16(bsb & 7, nr)) =
                        make_float4(ore[0], ore[1], ore[2], ore[3]);
                    *reinterpret_cast<float4*>(bwork + stk_row(bsb >> 3, 1, nr) + chunk16(bsb & 7, nr)) =
                        make_float4(oim[0], oim[1], oim[2], oim[3]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm.bt_ready);
            }

            // ---- D: the previous row's y, staged in this block's x tile
            if (staged) {  // the row before this one in the CTA's order
                Item row = cur;
                if (cur.r > 0) {
                    row.r = cur.r - 1;
                } else {
                    row.r = R - 1;
                    row.c = cur.c > 0 ? cur.c - 1 : nc - 1;
                    if (cur.c == 0) row.q = cur.q - (int)gridDim.x;
                }
                stage_y(ystage, row);
                mix_row = row;
            }

            // ---- C: C'_r = C_r o exp(Acs[l]) in place, plane 0 real. Unit: physical 16-byte chunk
            // j of rows 16g + i (plane 0) and 16g + 8 + i (plane 1) of one half (token l = 8g + i);
            // eight lanes cover the eight chunks of a row.
            if (diag) {
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int u = tid + kWorkers * k;
                    const int j = u & 7, i = (u >> 3) & 7, g = (u >> 6) & 7, half = u >> 9;
                    char* r0 = cwork + inter_row(half, 16 * g + i) + 16 * j;
                    char* r1 = r0 + 8 * 128;
                    const float2 e = sm.eacs[cp][orow + 8 * g + i];
                    float4 v0, v1;
                    if constexpr (kBf16) {
                        // physical chunk j of row m holds features 32 half + 4 (j ^ (m % 8)) .. + 3
                        const int f = 32 * half + 4 * (j ^ i);
                        const uint2 w0 = *reinterpret_cast<const uint2*>(cbase + off16(16 * g + i, f));
                        const uint2 w1 = *reinterpret_cast<const uint2*>(cbase + off16(16 * g + 8 + i, f));
                        v0 = make_float4(ptx::bf16_lo(w0.x), ptx::bf16_hi(w0.x), ptx::bf16_lo(w0.y), ptx::bf16_hi(w0.y));
                        v1 = make_float4(ptx::bf16_lo(w1.x), ptx::bf16_hi(w1.x), ptx::bf16_lo(w1.y), ptx::bf16_hi(w1.y));
                    } else {
                        v0 = *reinterpret_cast<const float4*>(r0);
                        v1 = *reinterpret_cast<const float4*>(r1);
                    }
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
            } else if (staged) {
                ptx::tc_fence_before();  // the y loads of D precede the next Y^T MMA (after p_ready)
            }

            // ---- E: P_rj = (C_r B_j^T) o L on row rr, columns col, col + 1 (col = 32 kh + 8 j + 2 lq),
            // into the B tile once the state MMA has read (dec o B)^T (or C B^T has read B). In the
            // accumulator, one 64-column half holds the products with B_r, the other with B_i; lane
            // plane 0 / 1 of the row holds the products of C's plane 0 / 1 (C_r first unless kSwapC).
            {
                float ga[16], gb[16];
                ptx::tmem_ld_16x256b_x4(tl + gbr() + 32 * kh, ga);
                ptx::tmem_ld_16x256b_x4(tl + gbi() + 32 * kh, gb);
                ptx::tmem_wait_ld();
                const float2 acs_l = sm.acs[cp][orow + rr];
                float2 pv[4][2];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // L[rr, col + 1] from one exponential, L[rr, col] = L[rr, col + 1] exp(-dA[col + 1]);
                    // causal inside the diagonal block, every pair below it
                    const int col = 32 * kh + 8 * j + 2 * lq;
                    // Re G = Cr Br - Ci Bi, Im G = Cr Bi + Ci Br
                    const float2 g0 = make_float2(ga[4 * j + kRr] - gb[4 * j + kRi], gb[4 * j + kRr] + ga[4 * j + kRi]);
                    const float2 g1 = make_float2(ga[4 * j + kRr + 1] - gb[4 * j + kRi + 1],
                                                  gb[4 * j + kRr + 1] + ga[4 * j + kRi + 1]);
                    float2 p0 = make_float2(0.0f, 0.0f), p1 = make_float2(0.0f, 0.0f);
                    if (!diag || col + 1 <= rr) {
                        const float2 L1v = cexp_fast(cdiff(acs_l, sm.acs[cp][ocol + col + 1]));
                        p1 = cmul(g1, L1v);
                        p0 = cmul(g0, cmul(L1v, sm.step[cp][ocol + col + 1]));
                    } else if (col == rr) {
                        p0 = g0;
                    }
                    pv[j][0] = p0;
                    pv[j][1] = p1;
                }
                if (diag) wait(&sm.mma_s, pd);
                const int mre = inter_m(rr, 0), mim = inter_m(rr, 1);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    *reinterpret_cast<float2*>(bwork + pair_off(kh, mre, 8 * j + 2 * lq)) =
                        make_float2(ptx::to_tf32(pv[j][0].x), ptx::to_tf32(pv[j][1].x));
                    *reinterpret_cast<float2*>(bwork + pair_off(kh, mim, 8 * j + 2 * lq)) =
                        make_float2(ptx::to_tf32(pv[j][0].y), ptx::to_tf32(pv[j][1].y));
                }
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();  // the C B^T loads precede the next C B^T MMA
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm.p_ready);
            }

            // ---- F: S_out^T = a_c S_in^T + S_loc^T on column d = rr, state rows n = 32 kh + 8 j + 2 lq + e
            if (chunk_last) {
                float sa[16], sb[16];
                ptx::tmem_ld_16x256b_x4(tl + kAccS + 32 * kh, sa);       // products with (dec o B)_r
                ptx::tmem_ld_16x256b_x4(tl + kAccS + 64 + 32 * kh, sb);  // products with (dec o B)_i
                float w[16];
                if (has_in) ptx::tmem_ld_16x256b_x4(tl + kSwin + 32 * kh, w);
                ptx::tmem_wait_ld();
                const float2 a = sm.a_c[cp];
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
                // the last Y_off of this chunk has read the window
                wait(&sm.mma_yo, pd);
                ptx::tc_fence_after();
                const Item nxt = item_next<kBlocks>(cur, R, nc);
                if (cur.c == nc - 1) {
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
            if (kMix && staged) {
                // the Re(y) stores read the staging tile before mix_after_store's barrier
                mix_after_store(mix_row);
                if (tid == 0 && !kBf16) ptx::mbar_arrive(&sm.free_x[s]);
            } else if (staged && (tid & kYMask) == 0) {  // its y stores have read the staging tile
                ptx::bulk_wait_read_all();
                if (!kBf16) ptx::mbar_arrive(&sm.free_x[s]);
            }
            if (diag) ++ndiag;
            cur = item_next<kBlocks>(cur, R, nc);
        }
        if (nitems > 0) {
            // the last row's y, staged in the last block's x tile (read by its last stores, above)
            wait(&sm.mma_y, (uint32_t)(nitems - 1) & 1u);
            ptx::tc_fence_after();
            ptx::named_sync(kWorkerBar, kWorkers);
            // the last block of the CTA's last chunk: its last row
            const int qlast = (int)blockIdx.x + (nseq_cta - 1) * (int)gridDim.x;
            char* buf = reinterpret_cast<char*>(sm.x[(nitems - 1) & 1]);
            if constexpr (kBf16) buf = reinterpret_cast<char*>(sm.yw);
            stage_y(buf, item_at(qlast, nc - 1, R - 1, R - 1));
            if (kMix) mix_after_store(item_at(qlast, nc - 1, R - 1, R - 1));
            else if ((tid & kYMask) == 0) ptx::bulk_wait_all();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
}

constexpr size_t kSmemBytes = sizeof(Smem<false>) > sizeof(Smem<true>) ? sizeof(Smem<false>) : sizeof(Smem<true>);
bool g_attr_set[64] = {};
std::mutex g_mu;

int set_attrs(int dev) {
    std::lock_guard<std::mutex> g(g_mu);
    if (g_attr_set[dev]) return SSDC_OK;
    const void* kernels[8] = {
        (const void*)fused2_kernel<false, false, false>,       (const void*)fused2_kernel<true, false, false>,
        (const void*)fused2_kernel<false, true, false>,        (const void*)fused2_kernel<true, true, false>,
        (const void*)fused2_kernel<false, false, true>,        (const void*)fused2_kernel<false, true, true>,
        (const void*)fused2_kernel<false, false, false, true>, (const void*)fused2_kernel<false, false, true, true>};
    for (const void* k : kernels)
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
            return SSDC_ERR_CUDA;
    g_attr_set[dev] = true;
    return SSDC_OK;
}

}  // namespace
}  // namespace fused2

bool fused2_supported(int N, int D, int Q) {
    return (Q == 16 || Q == 32 || Q == 64 || Q == 128 || Q == 256) && N >= 8 && N <= 64 && N % 8 == 0 && D >= 8 &&
           D <= 64 && D % 8 == 0;
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
    const bool swap_c = (fm.swap & 4) != 0, blocks = p.Q > fused2::kQ;
    const size_t sb = fused2::kSmemBytes;
    if (p.mix_w != nullptr) {  // the fused head mixer: Q <= 64, per-plane maps (never swapped)
        if (blocks || swap_c) return SSDC_ERR_UNSUPPORTED;
        if (p.in_bf16)
            fused2::fused2_kernel<false, false, true, true><<<g, b, sb, stream>>>(p, ws, fm);
        else
            fused2::fused2_kernel<false, false, false, true><<<g, b, sb, stream>>>(p, ws, fm);
    } else if (p.in_bf16) {  // bfloat16 inputs take the per-plane maps: never swapped
        if (blocks)
            fused2::fused2_kernel<false, true, true><<<g, b, sb, stream>>>(p, ws, fm);
        else
            fused2::fused2_kernel<false, false, true><<<g, b, sb, stream>>>(p, ws, fm);
    } else if (blocks) {
        if (swap_c)
            fused2::fused2_kernel<true, true, false><<<g, b, sb, stream>>>(p, ws, fm);
        else
            fused2::fused2_kernel<false, true, false><<<g, b, sb, stream>>>(p, ws, fm);
    } else {
        if (swap_c)
            fused2::fused2_kernel<true, false, false><<<g, b, sb, stream>>>(p, ws, fm);
        else
            fused2::fused2_kernel<false, false, false><<<g, b, sb, stream>>>(p, ws, fm);
    }
    return cudaGetLastError() == cudaSuccess ? 1 : SSDC_ERR_CUDA;
}

}  // namespace ssdc
