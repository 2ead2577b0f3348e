// The state a scan leaves behind, without its rows of y: for each (b, h)
// sequence, the chunked decomposition's state side only (landing page, "03
// Chunkwise SSD": the per-chunk states X^T (dec o B) and the pass between
// chunks, the STATE line), with none of the quadratic part or Y_off:
//     S_loc^T(c) = X_c^T (dec_c o B_c),  dec_c[s] = exp(Acs_c[Q-1] - Acs_c[s])
//     S_out^T(c) = a_c S_in^T(c) + S_loc^T(c),  a_c = exp(Acs_c[Q-1])
// from S_in(0) = the initial state (or zero). It reads x, B_t and dt: 1028
// bytes per token-head at N = D = 64, against 2068 for the whole forward. The
// joining of time segments uses it, for the state each segment leaves from
// zero before the segments' incoming states are known.
//
// The tiles, layouts and products are the tensor-memory forward kernel's
// (ssdc_fused2.cu), so the two compute the same final state bit for bit: per
// 64-token tile, the X^T window goes into TMEM by column reads of the TMA x
// tile, (dec o B)^T replaces the B tile in place, and one M = 128, N = 128 TF32
// MMA adds X^T (dec o B) into the S_loc^T accumulator (over a chunk's tiles
// for Q = 128 and 256). At a chunk's last tile the threads form S_out^T from
// the accumulator and S_in^T, which they hold in registers (no MMA reads it):
// 16 values a thread, in the 16x256b order of the accumulator.
//
// One CTA per SM walks whole sequences (sequences blockIdx.x, blockIdx.x +
// grid, ...). 16 worker warps; warp 16 issues the MMAs; warp 17 loads the tiles
// of the tile after next into the other stage and computes each chunk's
// cumulative log-decay. Every wait is bounded (a wait that gives up records
// SSDC_ERR_TIMEOUT in the status word and the later waits are skipped).
#include <mutex>

#include "fused_io.cuh"

namespace ssdc {
namespace state {
namespace {

using namespace tc;
using namespace fused;

constexpr int kWorkers = 512;  // 16 worker warps
constexpr int kWorkerWarps = kWorkers / 32;
constexpr int kIssuer = kWorkerWarps;        // warp 16: issues the MMAs
constexpr int kProducer = kWorkerWarps + 1;  // warp 17: TMA loads and decays
constexpr int kThreads = kWorkers + 64;
constexpr uint32_t kWorkerBar = 1;  // named barrier of the worker warps
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kAccS = 0, kXwin = 128;  // S_loc^T accumulator (128 columns), X^T window (64)
constexpr int kMaxQc = 256;

struct Smem {
    alignas(1024) float b[2][64 * 128];  // [stage] B (stacked), then (dec o B)^T (stacked, rows n)
    float x[2][64 * 128];                // [stage] x (stacked), read into the X^T window
    float2 acs[2][kMaxQc];               // [chunk parity] in-chunk cumulative log-decay
    float2 dec[2][kMaxQc];               // [chunk parity] exp(Acs[Q-1] - Acs[s]), zero past Q
    float2 a_c[2];                       // [chunk parity] exp(Acs[Q-1])
    uint64_t full[2], free_x[2], free_b[2];
    uint64_t xt_ready, bt_ready, mma_s;
    uint32_t tmem;
};
static_assert(sizeof(Smem) <= 232448, "shared-memory plan exceeds the 227 KB a CTA can have");

// Tile j of chunk c of sequence q = b H + h.
struct Tile {
    int q, c, j;
};

__device__ __forceinline__ Tile tile_next(const Tile& t, int R, int nc) {
    Tile n = t;
    if (t.j + 1 < R) {
        ++n.j;
    } else if (t.c + 1 < nc) {
        ++n.c;
        n.j = 0;
    } else {
        n.q += (int)gridDim.x;
        n.c = 0;
        n.j = 0;
    }
    return n;
}

__global__ void __launch_bounds__(kThreads, 1) state_kernel(Problem p, Workspace ws, const __grid_constant__ FusedMaps fm) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H, nc = (int)p.nc, Q = p.Q, N = p.N, D = p.D;
    const int rows = Q < kQ ? Q : kQ;    // tile rows holding tokens
    const int R = Q > kQ ? Q / kQ : 1;   // tiles per chunk
    const int nseq = p.B * H;
    const int nseq_cta = (int)blockIdx.x < nseq ? (nseq - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int ntiles = nseq_cta * nc * R;

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
        }
        ptx::mbar_init(&sm.xt_ready, kWorkerWarps);
        ptx::mbar_init(&sm.bt_ready, kWorkerWarps);
        ptx::mbar_init(&sm.mma_s, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(&sm.tmem, kTmemCols);
        ptx::tmem_relinquish();
    }
    if (Q < kQ) {
        // rows past Q are never loaded: give them finite contents
        float4* z = reinterpret_cast<float4*>(sm.b);
        constexpr int kVecs = (int)(2 * sizeof(sm.b) / 16);  // the b and x tiles of both stages
        for (int i = tid; i < kVecs; i += kThreads) z[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem;

    if (warp == kProducer) {
        // ============ producer warp: TMA loads and cumulative log-decays ============
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (lane == 0 && ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
            __syncwarp();
        };
        Tile ld = {(int)blockIdx.x, 0, 0};
        int chunks = 0;  // chunks begun by this CTA
        // single-tile chunks: the next chunk's dt is read ahead, while this one's tiles load
        Alog al = {};
        if (R == 1 && ntiles > 0) al = load_alog(p, ld.q / H, ld.q % H, 0, lane, Q);
        for (int k = 0; k < ntiles; ++k) {  // tile k into stage k & 1
            const int st = k & 1;
            const uint32_t ph = (uint32_t)((k - 2) >> 1) & 1u;
            const int tc0 = ld.c * Q, tj = tc0 + kQ * ld.j;
            const int bb = ld.q / H, hh = ld.q - bb * H;
            if (k >= 2) wait(&sm.free_x[st], ph);
            load_x(reinterpret_cast<char*>(sm.x[st]), fm, &sm.full[st], hh, tj, bb, rows, lane);
            if (k >= 2) wait(&sm.free_b[st], ph);
            load_b(reinterpret_cast<char*>(sm.b[st]), fm, &sm.full[st], hh, tj, bb, rows, lane);
            const Tile nx = tile_next(ld, R, nc);
            if (R == 1) {  // every tile is a chunk and carries its decays
                const Alog now = al;
                if (k + 1 < ntiles) {
                    const int nb = nx.q / H;
                    al = load_alog(p, nb, nx.q - nb * H, (int64_t)nx.c * Q, lane, Q);
                }
                store_acs(sm.acs[st], &sm.full[st], now, lane);
            } else {
                if (ld.j == 0) {
                    chunk_acs(p, bb, hh, tc0, Q, lane, sm.acs[chunks & 1]);
                    ++chunks;
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm.full[st]);
            }
            ld = nx;
        }
    } else if (warp == kIssuer) {
        // ============ MMA warp: lane 0 issues one MMA per tile ============
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
        };
        Tile cur = {(int)blockIdx.x, 0, 0};
        for (int k = 0; k < ntiles && lane == 0; ++k) {
            const int s = k & 1;
            const uint32_t ph = (uint32_t)k & 1u;
            wait(&sm.xt_ready, ph);
            wait(&sm.bt_ready, ph);
            ptx::tc_fence_after();
            issue_ts128(tmem + kAccS, tmem + kXwin, desc128(ptx::smem_addr(sm.b[s])), cur.j > 0);  // + X^T (dec o B)
            ptx::mma_commit(&sm.mma_s);
            ptx::mma_commit(&sm.free_b[s]);
            cur = tile_next(cur, R, nc);
        }
        __syncwarp();
    } else {
        // ===================== 16 worker warps =====================
        // 16x256b fragment of a warp: TMEM lane quadrant qd, 16-lane block blk, 32-column half
        // kh; lane i4 of the block holds plane 0 and lane i4 + 8 plane 1 of column d = rr of S^T.
        const int qd = warp & 3, blk = (warp >> 2) & 1, kh = warp >> 3;
        const int lq = lane & 3;
        const int rr = 16 * qd + 8 * blk + (lane >> 2);
        const uint32_t tl = lane_base(tmem, warp) + ((uint32_t)(16 * blk) << 16);
        const int swx = fm.swap & 1, swb = (fm.swap >> 1) & 1;
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok && !ptx::mbar_wait(bar, parity, kWaitIters)) {
                fail(ws.status);
                ok = false;
            }
        };
        // S_in^T[rr, n] (n = 32 kh + 8 j + 2 lq + e) at w[4 j + e] (re), w[4 j + 2 + e] (im):
        // the sequence's initial state, or zero
        float w[16];
        auto load_s0 = [&](int q) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int j = k >> 1, e = k & 1;
                const int n = 32 * kh + 8 * j + 2 * lq + e;
                const bool in = p.s0_re != nullptr && n < N && rr < D;
                const int64_t o = in ? ((int64_t)q * N + n) * D + rr : 0;
                w[4 * j + e] = in ? p.s0_re[o] : 0.0f;
                w[4 * j + 2 + e] = in ? p.s0_im[o] : 0.0f;
            }
        };
        Tile cur = {(int)blockIdx.x, 0, 0};
        if (ntiles > 0) load_s0(cur.q);
        int nchunk = 0;  // chunks begun
        for (int k = 0; k < ntiles; ++k) {
            const int s = k & 1;
            const uint32_t ph = (uint32_t)k & 1u;
            const bool chunk_first = cur.j == 0, chunk_last = cur.j == R - 1;
            if (chunk_first) ++nchunk;
            const int cp = R == 1 ? s : (nchunk - 1) & 1;  // the chunk's table parity
            const char* xbase = reinterpret_cast<const char*>(sm.x[s]);
            char* bbase = reinterpret_cast<char*>(sm.b[s]);
            wait(&sm.full[s], (uint32_t)((k >> 1) & 1));
            // the previous tile's MMA is complete: the X^T window is free
            if (k > 0) wait(&sm.mma_s, ph ^ 1u);
            ptx::tc_fence_after();

            // ---- A: the chunk's decays; X^T window; B rows into registers
            if (chunk_first) {
                const float2 last_acs = sm.acs[cp][Q - 1];
                const int Qe = Q > kQ ? Q : kQ;  // the rows of the chunk's tiles
                for (int t = tid; t < Qe; t += kWorkers)  // zero past the chunk's Q tokens
                    sm.dec[cp][t] = t < Q ? cexp_fast(cdiff(last_acs, sm.acs[cp][t])) : make_float2(0.0f, 0.0f);
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
                    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
                } else {
                    const char* rowbase = xbase + stk_row(xd >> 5, xp ^ swx, 0) + 4 * (xd & 3);
                    const int cq = (xd & 31) >> 2;
                    float r[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int sr = 16 * cg + (i ^ (4 * xp));
                        r[i] = *reinterpret_cast<const float*>(rowbase + sr * 128 + chunk16(cq, sr));
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = ptx::to_tf32(xp ? r[i ^ 4] : r[i]);
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
            // every worker has read x and its B rows (and the chunk's decays are written)
            ptx::named_sync(kWorkerBar, kWorkers);
            if (tid == 0) ptx::mbar_arrive(&sm.free_x[s]);
            if (lane == 0) ptx::mbar_arrive(&sm.xt_ready);

            // ---- B: (dec o B)^T in place of B
            {
                float2 dv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) dv[i] = sm.dec[cp][kQ * cur.j + 4 * bsb + i];
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

            // ---- F (the chunk's last tile): S_out^T = a_c S_in^T + S_loc^T on column d = rr,
            // state rows n = 32 kh + 8 j + 2 lq + e
            if (chunk_last) {
                wait(&sm.mma_s, ph);
                ptx::tc_fence_after();
                float sa[16], sb[16];
                ptx::tmem_ld_16x256b_x4(tl + kAccS + 32 * kh, sa);       // products with (dec o B)_r
                ptx::tmem_ld_16x256b_x4(tl + kAccS + 64 + 32 * kh, sb);  // products with (dec o B)_i
                ptx::tmem_wait_ld();
                const bool has_in = cur.c > 0 || p.s0_re != nullptr;
                const float2 a = sm.a_c[cp];
                float outr[8], outi[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int j = i >> 1, e = i & 1;
                    // Re: (x_r (dB)_r)[p0] - (x_i (dB)_i)[p1];  Im: (x_r (dB)_i)[p0] + (x_i (dB)_r)[p1]
                    outr[i] = sa[4 * j + e] - sb[4 * j + 2 + e];
                    outi[i] = sb[4 * j + e] + sa[4 * j + 2 + e];
                    if (has_in) {
                        const float sr = w[4 * j + e], si = w[4 * j + 2 + e];
                        outr[i] += a.x * sr - a.y * si;
                        outi[i] += a.x * si + a.y * sr;
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int j = i >> 1, e = i & 1;
                    w[4 * j + e] = outr[i];
                    w[4 * j + 2 + e] = outi[i];
                }
                if (cur.c == nc - 1) {  // the sequence's final state; the next one starts from its own
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int n = 32 * kh + 8 * (i >> 1) + 2 * lq + (i & 1);
                        if (n < N && rr < D) {
                            const int64_t o = ((int64_t)cur.q * N + n) * D + rr;
                            p.fs_re[o] = outr[i];
                            p.fs_im[o] = outi[i];
                        }
                    }
                    if (k + 1 < ntiles) load_s0(cur.q + (int)gridDim.x);
                }
                ptx::tc_fence_before();  // the accumulator's loads precede the next tile's MMA
            }
            cur = tile_next(cur, R, nc);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
}

// Tensor maps of x and B_t only: both planes in one map where the planes are
// 16-byte spaced and the tiles hold 64 tokens, else one per plane.
int make_state_maps(const Problem& p, bool allow_fast, FusedMaps* fm) {
    memset(fm, 0, sizeof(*fm));
    fm->real_x = p.x_im == nullptr;
    const int rows = p.Q < kQ ? p.Q : kQ;
    const bool pair_ok = allow_fast && rows == kQ;
    bool sw = false;
    if (pair_ok && !fm->real_x && make_pair_map(&fm->x2, p.x_re, p.x_im, p.D, p, &sw))
        fm->fast |= 1, fm->swap |= sw ? 1 : 0;
    if (pair_ok && make_pair_map(&fm->B2, p.B_re, p.B_im, p.N, p, &sw)) fm->fast |= 2, fm->swap |= sw ? 2 : 0;
    bool ok = true;
    if (!(fm->fast & 1))
        ok = ok && tc::encode_feature_map(&fm->x_re, p.x_re, p.D, p.H, p.T, p.B, rows) &&
             (fm->real_x || tc::encode_feature_map(&fm->x_im, p.x_im, p.D, p.H, p.T, p.B, rows));
    if (!(fm->fast & 2))
        ok = ok && tc::encode_feature_map(&fm->B_re, p.B_re, p.N, p.H, p.T, p.B, rows) &&
             tc::encode_feature_map(&fm->B_im, p.B_im, p.N, p.H, p.T, p.B, rows);
    return ok ? SSDC_OK : SSDC_ERR_CUDA;
}

constexpr size_t kSmemBytes = sizeof(Smem);
bool g_attr_set[64] = {};
std::mutex g_mu;

int set_attrs(int dev) {
    std::lock_guard<std::mutex> g(g_mu);
    if (g_attr_set[dev]) return SSDC_OK;
    if (cudaFuncSetAttribute(state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
        cudaSuccess)
        return SSDC_ERR_CUDA;
    g_attr_set[dev] = true;
    return SSDC_OK;
}

}  // namespace
}  // namespace state

bool state_supported(int N, int D, int Q) { return fused2_supported(N, D, Q); }

int state_launch(const Problem& p, const Workspace& ws, cudaStream_t stream, bool plane_maps) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SSDC_ERR_CUDA;
    int rc = state::set_attrs(dev);
    if (rc != SSDC_OK) return rc;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return SSDC_ERR_CUDA;
    fused::FusedMaps fm;
    rc = state::make_state_maps(p, plane_maps, &fm);
    if (rc != SSDC_OK) return rc;
    const int64_t nseq = (int64_t)p.B * p.H;
    const int grid = (int)(nseq < sms ? nseq : sms);
    state::state_kernel<<<grid, state::kThreads, state::kSmemBytes, stream>>>(p, ws, fm);
    return cudaGetLastError() == cudaSuccess ? 1 : SSDC_ERR_CUDA;
}

}  // namespace ssdc
