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
// is computed by the CTA of chunk c and stored (st.async, 32 KB) straight
// into the shared memory of the CTA of chunk c+1, rank (r+1) mod CL, whose
// mbarrier counts the bytes; the receiver frees the buffer by arriving on the
// sender's mbarrier. With CL = 1 the CTA keeps the state in its own shared
// memory. All chunk-local work (C B^T, L, Y_diag, S_loc) is independent of
// the incoming state, so the serial chain per sequence is one complex
// multiply-add per state element and one 32 KB transfer per chunk.
//
// Complex products. Planar re/im operands are multiplied as real M=128 MMAs
// whose A operand holds the real and imaginary rows of the left factor
// interleaved in groups of eight (row 16g + 8p + i = plane p of row 8g + i)
// and whose B operand stacks or interleaves the right factor's two planes as
// 128 rows (N = 128). One accumulator then holds, in TMEM lanes m and m ^ 8
// (the same warp), all four real products, and
//     Re = (A_r B_r)[lane p=0] - (A_i B_i)[lane p=1]
//     Im = (A_r B_i)[lane p=0] + (A_i B_r)[lane p=1]
// is one exchange between partner lanes. The C tile is loaded in that layout
// by TMA (8-row boxes); x^T is written in it by a shared-memory transpose.
// The output accumulator takes both P x (Y_diag) and (C o exp(Acs)) S_in
// (Y_off): the two A operands, P and C', are rows written to TMEM.
//
// Threads. 16 warps; warps w and w + 4k share TMEM lane quadrant w % 4 and
// split a row's 64 columns in quarters (k = w / 4). Worker thread 0 issues
// the MMAs and the TMA stores of y; warp 15 also issues the TMA loads of the
// next chunk's C, B, x tiles into the other stage of a two-stage ring and
// computes its cumulative log-decay.
#include <cuda.h>
#include <cuda_runtime.h>

#include "tc_common.cuh"

namespace ssdc {
namespace fused {
namespace {

using namespace tc;

constexpr int kQ = 64;
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kLoader = kWarps - 1;  // warp that prefetches the next chunk
constexpr uint32_t kTmemCols = 512;
// TMEM columns: three 128-column accumulators and two 64-column A operands.
constexpr uint32_t kAccG = 0, kAccS = 128, kAccY = 256, kPwin = 384, kCwin = 448;
constexpr uint32_t kTileBytes = 2 * kPlaneBytes;  // 32 KB: one complex 64 x 64 tile
constexpr uint32_t kStageTx = 3 * kTileBytes;     // C, B, x
constexpr uint32_t kStateBytes = kTileBytes;
constexpr uint32_t kIntHalf = 16384;  // one 32-column half of a 128-row tile
constexpr uint32_t kIdesc128 = ptx::idesc_tf32(128, 128, 0);  // M = 128, N = 128, B operand K-major

struct Smem {
    float c[2][64 * 128];    // [stage] C, interleaved 128 rows (A operand)
    float b[2][64 * 128];    // [stage] B, stacked (rows s); after C B^T, (dec o B)^T stacked (rows n)
    float x[2][64 * 128];    // [stage] x, stacked (rows s); x^T interleaved (rows d); then y staging
    float sin[64 * 128];     // incoming state S_in^T, interleaved (rows d, n contiguous)
    float2 acs[2][kQ];       // in-chunk cumulative log-decay, per stage
    float2 dec[kQ];          // exp(Acs[Q-1] - Acs[s])
    float2 eacs[kQ];         // exp(Acs[l])
    float2 a_c;              // exp(Acs[Q-1])
    float2 pair[kQ];         // exp(Acs[s+2] - Acs[s]): decay over tokens s+1, s+2
    uint64_t full[2], sin_full, succ_empty;
    uint64_t xt_ready, bt_ready;  // x^T written (all warps), (dec o B)^T written (warps 0-7)
    uint64_t mma[3];         // MMA groups C B^T, S_loc^T, y; one phase per chunk
    uint32_t tmem;
};

static_assert(sizeof(Smem) <= 232448, "shared-memory plan exceeds the 227 KB a CTA can have");

// The chunks this CTA processes, in order: for each sequence owned by its
// cluster, the chunks congruent to its rank.
struct Items {
    int64_t nseq, nc;
    uint32_t cl, rank, cluster, nclusters;
    int64_t per_seq;  // chunks of one sequence owned by this rank
    __device__ Items(int64_t nseq_, int64_t nc_)
        : nseq(nseq_), nc(nc_), cl(ptx::cluster_nctarank()), rank(ptx::cluster_ctarank()),
          cluster(ptx::cluster_id_x()), nclusters(ptx::ncluster_x()) {
        per_seq = nc > (int64_t)rank ? (nc - 1 - rank) / cl + 1 : 0;
    }
    __device__ int64_t count() const {
        const int64_t seqs = nseq > (int64_t)cluster ? (nseq - 1 - cluster) / nclusters + 1 : 0;
        return seqs * per_seq;
    }
    __device__ void get(int64_t i, int64_t& q, int64_t& c) const {
        q = cluster + (i / per_seq) * nclusters;
        c = rank + (i % per_seq) * cl;
    }
};

__device__ __forceinline__ float2 cdiff(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }

// Byte offsets. A "stacked" tile holds two 64 x 64 planes as one K-major
// operand of 128 rows: [32-column half][plane][64 rows][128 B]. An
// "interleaved" tile is [32-column half][128 rows][128 B] with row
// 16g + 8p + i = plane p of row 8g + i. Rows are 128-byte swizzled.
__device__ __forceinline__ uint32_t stk_row(int khalf, int plane, int r) {
    return (uint32_t)(khalf * kIntHalf + plane * kHalfBytes + r * 128);
}
__device__ __forceinline__ uint32_t inter_row(int khalf, int m) { return (uint32_t)(khalf * kIntHalf + m * 128); }
__device__ __forceinline__ uint32_t chunk16(int j, int r) { return (uint32_t)(((j ^ (r & 7)) & 7) << 4); }
__device__ __forceinline__ int inter_m(int r8, int plane) { return 16 * (r8 >> 3) + 8 * plane + (r8 & 7); }

// K-major SW128 descriptor of a 128-row operand; K-step k (8 fp32) adds
// (k / 4) halves and (k % 4) 32-byte steps to the start address.
__device__ __forceinline__ uint64_t desc128(uint32_t base) { return ptx::smem_desc_sw128(base, 16u, 1024u); }
__device__ __forceinline__ uint64_t desc_k(uint64_t d, int k) {
    return d + (uint64_t)((((uint32_t)(k >> 2) * kIntHalf) + (uint32_t)(k & 3) * 32u) >> 4);
}

// D (+)= A * B over K = 64: 8 MMAs of M = 128, N = 128, K = 8.
__device__ __forceinline__ void issue_ss128(uint32_t d, uint64_t da, uint64_t db) {
#pragma unroll
    for (int k = 0; k < 8; ++k) ptx::mma_tf32_ss(d, desc_k(da, k), desc_k(db, k), kIdesc128, k > 0 ? 1u : 0u);
}
__device__ __forceinline__ void issue_ts128(uint32_t d, uint32_t a_tmem, uint64_t db, bool accumulate) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
        ptx::mma_tf32_ts(d, a_tmem + 8 * k, desc_k(db, k), kIdesc128, (accumulate || k > 0) ? 1u : 0u);
}

// Loader warp: TMA of one chunk's C (8-row boxes, re/im interleaved), B and
// x (stacked) into stage `st`, counted on `bar`. The 40 copies are issued by
// the warp's lanes in parallel after lane 0 has announced the bytes.
__device__ __forceinline__ void load_tiles(Smem& sm, int st, const TcMaps& maps, const CUtensorMap& c8_re,
                                           const CUtensorMap& c8_im, int h, int t0, int b, int lane) {
    uint64_t* bar = &sm.full[st];
    if (lane == 0) ptx::mbar_expect_tx(bar, kStageTx);
    __syncwarp();
    char* cb = reinterpret_cast<char*>(sm.c[st]);
    char* bb = reinterpret_cast<char*>(sm.b[st]);
    char* xb = reinterpret_cast<char*>(sm.x[st]);
    for (int op = lane; op < 40; op += 32) {
        const int half = op / 20, k = op % 20, f0 = 32 * half;
        if (k < 16) {  // C rows 8g .. 8g+7 of plane k & 1
            const int g = k >> 1, pl = k & 1;
            ptx::tma_load_4d(cb + inter_row(half, 16 * g + 8 * pl), pl ? &c8_im : &c8_re, bar, f0, h, t0 + 8 * g, b);
        } else {
            const int pl = k & 1;
            const CUtensorMap* m = k < 18 ? (pl ? &maps.B_im : &maps.B_re) : (pl ? &maps.x_im : &maps.x_re);
            ptx::tma_load_4d((k < 18 ? bb : xb) + stk_row(half, pl, 0), m, bar, f0, h, t0, b);
        }
    }
}

// Loader warp: dt of one chunk's 64 tokens (two per lane; tokens past T are
// marked with NaN so that they get zero log-decay), and A of its head. The
// loads are only issued here; their values are first used by store_acs.
struct Alog {
    float dt0, dt1, Ar, Ai;
};
__device__ __forceinline__ Alog load_alog(const Problem& p, int b, int h, int64_t t0, int lane) {
    Alog a;
    const int64_t ta = t0 + 2 * lane, tb = ta + 1;
    a.dt0 = ta < p.T ? p.dt[((int64_t)b * p.T + ta) * p.H + h] : __int_as_float(0x7fffffff);
    a.dt1 = tb < p.T ? p.dt[((int64_t)b * p.T + tb) * p.H + h] : __int_as_float(0x7fffffff);
    a.Ar = p.A_re[h];
    a.Ai = p.A_im[h];
    return a;
}

// Loader warp: discretisation softplus(dt) * A and its inclusive cumulative
// sum into acs, then arrive on the stage barrier (the tile bytes were
// announced by load_tiles). The sum is fp32: its rounding (about 1e-7 of
// |Acs|, so about 1e-5 relative on a decay factor) is far below TF32's.
__device__ __forceinline__ void store_acs(Smem& sm, int st, const Alog& al, int lane) {
    const float sp0 = al.dt0 == al.dt0 ? softplus_f(al.dt0) : 0.0f;
    const float sp1 = al.dt1 == al.dt1 ? softplus_f(al.dt1) : 0.0f;
    const float r0 = sp0 * al.Ar, i0 = sp0 * al.Ai, r1 = sp1 * al.Ar, i1 = sp1 * al.Ai;
    float cr = r0 + r1, ci = i0 + i1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float ur = __shfl_up_sync(0xffffffffu, cr, off);
        const float ui = __shfl_up_sync(0xffffffffu, ci, off);
        if (lane >= off) {
            cr += ur;
            ci += ui;
        }
    }
    const float er = cr - (r0 + r1), ei = ci - (i0 + i1);  // exclusive prefix
    sm.acs[st][2 * lane] = make_float2(er + r0, ei + i0);
    sm.acs[st][2 * lane + 1] = make_float2(cr, ci);
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&sm.full[st]);
}

__global__ void __launch_bounds__(kThreads, 1)
fused_kernel(Problem p, Workspace ws, const __grid_constant__ TcMaps maps, const __grid_constant__ CUtensorMap c8_re,
             const __grid_constant__ CUtensorMap c8_im, const __grid_constant__ CUtensorMap y_re,
             const __grid_constant__ CUtensorMap y_im) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    const Items items((int64_t)p.B * H, p.nc);
    const int64_t nitems = items.count();
    const uint32_t CL = items.cl, rank = items.rank;
    const uint32_t succ = (rank + 1) % CL, pred = (rank + CL - 1) % CL;

    if (tid == 0 && blockIdx.x == 0) *ws.status = SSDC_OK;
    // the swizzled tiles need a 1024-byte aligned base (uniform across the grid)
    if (ptx::smem_addr(smem_raw) & 1023u) {
        if (tid == 0) atomicExch(ws.status, SSDC_ERR_CUDA);
        return;
    }
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) ptx::mbar_init(&sm.full[s], 1);
        for (int g = 0; g < 3; ++g) ptx::mbar_init(&sm.mma[g], 1);
        ptx::mbar_init(&sm.sin_full, 1);
        ptx::mbar_init(&sm.xt_ready, kWarps);
        ptx::mbar_init(&sm.bt_ready, 8);
        ptx::mbar_init(&sm.succ_empty, 1);
        ptx::fence_mbar_init();
        if (CL > 1) ptx::mbar_arrive_expect_tx(&sm.sin_full, kStateBytes);  // first transfer
    }
    if (warp == 0) {
        ptx::tmem_alloc(&sm.tmem, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::cluster_sync();  // peers' barriers are initialised before any remote access
    const uint32_t tmem = sm.tmem;

    // first chunk's tiles and decays
    if (warp == kLoader && nitems > 0) {
        int64_t q0, c0;
        items.get(0, q0, c0);
        const int b0 = (int)(q0 / H), h0 = (int)(q0 % H);
        load_tiles(sm, 0, maps, c8_re, c8_im, h0, (int)(c0 * kQ), b0, lane);
        store_acs(sm, 0, load_alog(p, b0, h0, c0 * kQ, lane), lane);
    }

    const int h4 = warp >> 2;                   // column quarter of this warp
    const int m = (warp & 3) * 32 + lane;       // TMEM lane
    const int r8 = 8 * (m >> 4) + (m & 7);      // complex row (l or d) of this lane
    const int pl = (m >> 3) & 1;                // plane of this lane
    const uint32_t my = lane_base(tmem, warp);
    uint32_t n_recv = 0, n_send = 0;
    bool recv_ok = true;
    const uint32_t sin_saddr = ptx::smem_addr(sm.sin);
    const uint32_t remote_sin = ptx::mapa(sin_saddr, succ);
    const uint32_t remote_sin_full = ptx::mapa(ptx::smem_addr(&sm.sin_full), succ);
    const uint32_t remote_pred_empty = ptx::mapa(ptx::smem_addr(&sm.succ_empty), pred);

    auto wait_mma = [&](int g, int64_t it) {
        if (!ptx::mbar_wait(&sm.mma[g], (uint32_t)(it & 1), kWaitIters)) fail(ws.status);
        ptx::tc_fence_after();
    };
    auto publish = [&]() {  // tcgen05.st and smem writes of all threads -> MMA issue
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
    };

    // dt of chunk it + 1 is loaded during chunk it - 1 and consumed during chunk it
    Alog nal = {};
    if (warp == kLoader && nitems > 1) {
        int64_t q1, c1;
        items.get(1, q1, c1);
        nal = load_alog(p, (int)(q1 / H), (int)(q1 % H), c1 * kQ, lane);
    }
    for (int64_t it = 0; it < nitems; ++it) {
        const int s = (int)(it & 1);
        int64_t q, c;
        items.get(it, q, c);
        const int b = (int)(q / H), h = (int)(q % H);
        const int64_t t0 = c * kQ;
        const bool has_in = c > 0, last = c == p.nc - 1;
        char* xbase = reinterpret_cast<char*>(sm.x[s]);
        char* bbase = reinterpret_cast<char*>(sm.b[s]);
        const char* cbase = reinterpret_cast<const char*>(sm.c[s]);
        const uint32_t cs = ptx::smem_addr(cbase), bs = ptx::smem_addr(bbase), xs = ptx::smem_addr(xbase);
        if (!ptx::mbar_wait(&sm.full[s], (uint32_t)((it >> 1) & 1), kWaitIters)) fail(ws.status);
        if (tid == 0) {
            // C B^T reads only TMA-loaded tiles: issue it first
            ptx::tc_fence_after();
            issue_ss128(tmem + kAccG, desc128(cs), desc128(bs));  // [C Br | C Bi]
            ptx::mma_commit(&sm.mma[0]);
            ptx::bulk_wait_read_all();  // the previous chunk's y store has read its stage
        }

        // ---- A: decays; x and B 4x4 blocks into registers. Lane bits pick the
        // block so that a warp's 16-byte accesses cover all eight bank groups.
        if (tid < kQ) {
            sm.dec[tid] = cexp_fast(cdiff(sm.acs[s][kQ - 1], sm.acs[s][tid]));
        } else if (tid < 2 * kQ) {
            sm.eacs[tid - kQ] = cexp_fast(sm.acs[s][tid - kQ]);
        } else if (tid == 2 * kQ) {
            sm.a_c = cexp_fast(sm.acs[s][kQ - 1]);
        } else if (tid > 2 * kQ && tid <= 3 * kQ - 2) {
            const int t = tid - 2 * kQ - 1;  // 0 .. Q-3
            sm.pair[t] = cexp_fast(cdiff(sm.acs[s][t + 2], sm.acs[s][t]));
        }
        const int blo = lane & 7, bmid = (lane >> 3) & 3;
        const int xsb = bmid + 4 * (warp & 3), xdb = blo + 8 * ((warp >> 2) & 1), xp = (warp >> 3) & 1;
        float4 xv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // x block: rows s = 4 xsb + i, columns d = 4 xdb ..
            const int sr = 4 * xsb + i;
            xv[i] = *reinterpret_cast<const float4*>(xbase + stk_row(xdb >> 3, xp, sr) + chunk16(xdb & 7, sr));
        }
        const bool bwork = warp < 8;  // (dec o B)^T: one block of both planes per thread of warps 0-7
        const int bsb = bmid + 4 * (warp & 3), bnb = blo + 8 * ((warp >> 2) & 1);
        float4 bv[2][4];
        if (bwork) {
#pragma unroll
            for (int pp = 0; pp < 2; ++pp)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int sr = 4 * bsb + i;
                    bv[pp][i] = *reinterpret_cast<const float4*>(bbase + stk_row(bnb >> 3, pp, sr) + chunk16(bnb & 7, sr));
                }
        }
        __syncthreads();
        // the previous chunk's stage is free: prefetch the next chunk into it
        const bool prefetch = it + 1 < nitems;
        int64_t qn = 0, cn = 0;
        if (warp == kLoader && prefetch) items.get(it + 1, qn, cn);

        // ---- B: x^T (interleaved rows d) in place of x; C' = C o exp(Acs[l]) rows into TMEM; C B^T
        {
            const float4 o[4] = {make_float4(xv[0].x, xv[1].x, xv[2].x, xv[3].x), make_float4(xv[0].y, xv[1].y, xv[2].y, xv[3].y),
                                 make_float4(xv[0].z, xv[1].z, xv[2].z, xv[3].z), make_float4(xv[0].w, xv[1].w, xv[2].w, xv[3].w)};
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
            // plane pl of C'[l, n] for n in [16 h4, 16 h4 + 16): row l of both C planes
            const float2 e = sm.eacs[r8];
            const int kh = h4 >> 1, j0 = 4 * (h4 & 1);
            const int mre = inter_m(r8, 0), mim = inter_m(r8, 1);
            float w[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 cr = *reinterpret_cast<const float4*>(cbase + inter_row(kh, mre) + chunk16(j0 + j, mre));
                const float4 ci = *reinterpret_cast<const float4*>(cbase + inter_row(kh, mim) + chunk16(j0 + j, mim));
                const float crv[4] = {cr.x, cr.y, cr.z, cr.w}, civ[4] = {ci.x, ci.y, ci.z, ci.w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    w[4 * j + k] = pl ? (crv[k] * e.y + civ[k] * e.x) : (crv[k] * e.x - civ[k] * e.y);
            }
            ptx::tmem_st16(my + kCwin + 16 * h4, w);
        }
        if (warp == kLoader && prefetch)
            load_tiles(sm, s ^ 1, maps, c8_re, c8_im, (int)(qn % H), (int)(cn * kQ), (int)(qn / H), lane);
        wait_mma(0, it);  // C B^T has read B

        // ---- C: (dec o B)^T stacked in place of B; then S_loc^T = x^T (dec o B), issued by
        // thread 0 once every warp has announced its x^T and (dec o B)^T blocks
        if (bwork) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // column n = 4 bnb + j of B -> row n of the output
                const int nr = 4 * bnb + j;
                float ore[4], oim[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float* r0v = reinterpret_cast<const float*>(&bv[0][i]);
                    const float* r1v = reinterpret_cast<const float*>(&bv[1][i]);
                    const float2 v = cmul(sm.dec[4 * bsb + i], make_float2(r0v[j], r1v[j]));
                    ore[i] = v.x;
                    oim[i] = v.y;
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
        if (tid == 0) {
            if (!ptx::mbar_wait(&sm.xt_ready, (uint32_t)(it & 1), kWaitIters)) fail(ws.status);
            if (!ptx::mbar_wait(&sm.bt_ready, (uint32_t)(it & 1), kWaitIters)) fail(ws.status);
            ptx::tc_fence_after();
            issue_ss128(tmem + kAccS, desc128(xs), desc128(bs));  // [x^T B'r | x^T B'i]
            ptx::mma_commit(&sm.mma[1]);
        }

        // ---- D: P = (C B^T) o L on this thread's columns; P rows into TMEM; then P x
        {
            // columns [8 h4, 8 h4 + 8) and [32 + 8 h4, 32 + 8 h4 + 8), in pairs (e, e + 1)
            float ga[16], gb[16];
            ptx::tmem_ld8(my + kAccG + 8 * h4, ga);
            ptx::tmem_ld8(my + kAccG + 32 + 8 * h4, ga + 8);
            ptx::tmem_ld8(my + kAccG + 64 + 8 * h4, gb);
            ptx::tmem_ld8(my + kAccG + 96 + 8 * h4, gb + 8);
            ptx::tmem_wait_ld();
            const float2 acs_l = sm.acs[s][r8];
            // complex G on this thread's columns: column e + pl of each pair
            float gre[8], gim[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const float ra = __shfl_xor_sync(0xffffffffu, pl ? ga[2 * jj] : ga[2 * jj + 1], 8);
                const float rb = __shfl_xor_sync(0xffffffffu, pl ? gb[2 * jj] : gb[2 * jj + 1], 8);
                // plane-0 products (Cr B) and plane-1 products (Ci B) of this thread's column
                const float ga0 = pl ? ra : ga[2 * jj], gb0 = pl ? rb : gb[2 * jj];
                const float ga1 = pl ? ga[2 * jj + 1] : ra, gb1 = pl ? gb[2 * jj + 1] : rb;
                gre[jj] = ga0 - gb1;
                gim[jj] = gb0 + ga1;
            }
            // L[l, col] for the four columns col = base + 2k + pl of each 8-column range, from
            // the last one with col <= l down: one exponential of a difference of cumulative
            // sums, then L[l, col - 2] = L[l, col] exp(Acs[col] - Acs[col - 2]).
            float pr[8], pim[8];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int base = (rr ? 32 : 0) + 8 * h4 + pl;
                float2 L = make_float2(0.0f, 0.0f);
                bool started = false;
#pragma unroll
                for (int k = 3; k >= 0; --k) {
                    const int col = base + 2 * k, jj = 4 * rr + k;
                    float2 v = make_float2(0.0f, 0.0f);
                    if (col <= r8) {
                        L = started ? cmul(L, sm.pair[col]) : cexp_fast(cdiff(acs_l, sm.acs[s][col]));
                        started = true;
                        v = cmul(make_float2(gre[jj], gim[jj]), L);
                    }
                    pr[jj] = v.x;
                    pim[jj] = v.y;
                }
            }
            float w[16];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                // lane p keeps plane p of P: column e from the p = 0 lane, e + 1 from the p = 1 lane
                const float other = __shfl_xor_sync(0xffffffffu, pl ? pr[jj] : pim[jj], 8);
                w[2 * jj] = pl ? other : pr[jj];
                w[2 * jj + 1] = pl ? pim[jj] : other;
            }
            ptx::tmem_st8(my + kPwin + 8 * h4, w);
            ptx::tmem_st8(my + kPwin + 32 + 8 * h4, w + 8);
        }
        publish();
        if (tid == 0) issue_ts128(tmem + kAccY, tmem + kPwin, desc128(xs), false);  // P x^T (interleaved columns)

        // ---- E: S_loc^T and the state hop  S_out = a_c S_in + S_loc  (row d = r8, n in [16 h4, +16))
        if (warp == kLoader && prefetch) {
            store_acs(sm, s ^ 1, nal, lane);  // next chunk's decays
            if (it + 2 < nitems) {
                int64_t q2, c2;
                items.get(it + 2, q2, c2);
                nal = load_alog(p, (int)(q2 / H), (int)(q2 % H), c2 * kQ, lane);
            }
        }
        wait_mma(1, it);
        float out[16];
        {
            float sa[16], sb[16];
            ptx::tmem_ld16(my + kAccS + 16 * h4, sa);
            ptx::tmem_ld16(my + kAccS + 64 + 16 * h4, sb);
            ptx::tmem_wait_ld();
            if (has_in && CL > 1) {
                if (!ptx::mbar_wait(&sm.sin_full, n_recv & 1, kWaitIters)) {
                    fail(ws.status);
                    recv_ok = false;  // the buffer protocol stops here for this CTA
                }
                ++n_recv;
            }
            const float2 a = sm.a_c;
            const char* sinb = reinterpret_cast<const char*>(sm.sin);
            const int kh = h4 >> 1, j0 = 4 * (h4 & 1);
            const int mre = inter_m(r8, 0), mim = inter_m(r8, 1);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float4 sr = make_float4(0.f, 0.f, 0.f, 0.f), si = sr;
                if (has_in) {
                    sr = *reinterpret_cast<const float4*>(sinb + inter_row(kh, mre) + chunk16(j0 + j, mre));
                    si = *reinterpret_cast<const float4*>(sinb + inter_row(kh, mim) + chunk16(j0 + j, mim));
                }
                const float srv[4] = {sr.x, sr.y, sr.z, sr.w}, siv[4] = {si.x, si.y, si.z, si.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int k = 4 * j + e;
                    const float other = __shfl_xor_sync(0xffffffffu, sb[k], 8);
                    // Re: a S_in + (xr B'r)[p0] - (xi B'i)[p1];  Im: a S_in + (xr B'i)[p0] + (xi B'r)[p1]
                    out[k] = pl ? (a.x * siv[e] + a.y * srv[e] + other + sa[k])
                                : (a.x * srv[e] - a.y * siv[e] + sa[k] - other);
                }
            }
        }
        const int mo = inter_m(r8, pl);
        if (last) {
            float* fs = (pl ? p.fs_im : p.fs_re) + (q * 64) * 64 + r8;
#pragma unroll
            for (int k = 0; k < 16; ++k) fs[(int64_t)(16 * h4 + k) * 64] = out[k];
        } else if (CL > 1) {
            // stage S_out in the C buffer (C was consumed by C B^T and the C' rows);
            // worker thread 0 moves it to the next CTA with one bulk copy
            char* stg = reinterpret_cast<char*>(sm.c[s]);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<float4*>(stg + inter_row(h4 >> 1, mo) + chunk16(4 * (h4 & 1) + j, mo)) =
                    make_float4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
            ptx::fence_proxy_async_smem();
        }

        // ---- F: (C o exp(Acs)) S_in into the same accumulator
        publish();
        if (tid == 0) {
            // the state goes to the next CTA first: it is on the chain's critical path
            if (!last && CL > 1 && c != p.drop_send_chunk) {
                if (n_send > 0 && !ptx::mbar_wait(&sm.succ_empty, (n_send - 1) & 1, kWaitIters)) fail(ws.status);
                ++n_send;
                ptx::bulk_copy_to_cluster(remote_sin, cs, kStateBytes, remote_sin_full);
                ptx::bulk_commit();
            }
            if (has_in) issue_ts128(tmem + kAccY, tmem + kCwin, desc128(sin_saddr), true);
            ptx::mma_commit(&sm.mma[2]);
        }
        wait_mma(2, it);
        if (has_in && CL > 1 && tid == 0 && recv_ok) {
            // the incoming buffer is consumed: re-arm it and free it for the sender
            ptx::mbar_arrive_expect_tx(&sm.sin_full, kStateBytes);
            ptx::mbar_arrive_remote(remote_pred_empty);
        }
        if (!last && CL == 1) {
            // keep the state for this CTA's next chunk
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<float4*>(reinterpret_cast<char*>(sm.sin) + inter_row(h4 >> 1, mo) + chunk16(4 * (h4 & 1) + j, mo)) =
                    make_float4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
            ptx::fence_proxy_async_smem();
        }

        // ---- G: y rows, staged in the x buffer and written by TMA. Columns
        // 16g + 8p' + i of the accumulator hold plane-p' products of column 8g + i.
        {
            float yv[32];
            ptx::tmem_ld16(my + kAccY + 32 * h4, yv);
            ptx::tmem_ld16(my + kAccY + 32 * h4 + 16, yv + 16);
            ptx::tmem_wait_ld();
            float o[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int yi = 16 * (k >> 3) + (k & 7);
                const float ya = yv[yi], yb = yv[yi + 8];
                // Re y = ya[p0] - yb[p1], Im y = yb[p0] + ya[p1]
                const float u = pl ? -yb : ya, v = pl ? ya : yb;
                const float other = __shfl_xor_sync(0xffffffffu, pl ? u : v, 8);
                o[k] = pl ? v + other : u + other;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<float4*>(xbase + stk_row(h4 >> 1, pl, r8) + chunk16(4 * (h4 & 1) + k, r8)) =
                    make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            for (int half = 0; half < 2; ++half) {
                ptx::tma_store_4d(&y_re, xbase + stk_row(half, 0, 0), 32 * half, h, (int)t0, b);
                ptx::tma_store_4d(&y_im, xbase + stk_row(half, 1, 0), 32 * half, h, (int)t0, b);
            }
            ptx::bulk_commit();  // read-complete is awaited before the next prefetch
        }
    }
    if (tid == 0) ptx::bulk_wait_all();

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
    ptx::cluster_sync();  // no CTA leaves while a peer may still write to its shared memory
}

constexpr size_t kSmemBytes = sizeof(Smem);
bool g_attr_set[64] = {};

// (F, H, T, B) fp32 plane as 8-row boxes (32, 1, 8, 1), 128-byte swizzle.
bool make_rows8_map(CUtensorMap* m, const float* base, int H, int64_t T, int B) {
    return tc::encode_feature_map(m, base, 64, H, T, B, 8);
}

}  // namespace

// Choose the cluster size: the one that minimises (waves of clusters) x
// (chunks per CTA, or the serial state chain if that is longer).
int pick_cluster(const Problem& p, int* cl_out, int* nclusters_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SSDC_ERR_CUDA;
    if (!g_attr_set[dev]) {
        if (cudaFuncSetAttribute(fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
            cudaSuccess)
            return SSDC_ERR_CUDA;
        g_attr_set[dev] = true;
    }
    const int64_t nseq = (int64_t)p.B * p.H;
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
        if (cudaOccupancyMaxActiveClusters(&active, fused_kernel, &cfg) != cudaSuccess || active <= 0) {
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
    return SSDC_OK;
}

}  // namespace fused

bool fused_supported(int N, int D, int Q) { return N == 64 && D == 64 && Q == 64; }

int fused_launch(const Problem& p, const Workspace& ws, cudaStream_t stream, int force_cluster) {
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
    tc::TcMaps maps;
    rc = tc::make_maps(p, nullptr, &maps);
    if (rc != SSDC_OK) return rc;
    CUtensorMap c8_re, c8_im, y_re, y_im;
    if (!fused::make_rows8_map(&c8_re, p.C_re, p.H, p.T, p.B) || !fused::make_rows8_map(&c8_im, p.C_im, p.H, p.T, p.B) ||
        !tc::encode_feature_map(&y_re, p.y_re, 64, p.H, p.T, p.B, 64) ||
        !tc::encode_feature_map(&y_im, p.y_im, 64, p.H, p.T, p.B, 64))
        return SSDC_ERR_CUDA;
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
    if (cudaLaunchKernelEx(&cfg, fused::fused_kernel, p, ws, maps, c8_re, c8_im, y_re, y_im) != cudaSuccess) return SSDC_ERR_CUDA;
    return 1;
}

}  // namespace ssdc
