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
// interleaved in groups of eight (row 16g + 8p + i = plane p of row 8g + i).
// Two accumulators, A * Br and A * Bi, then hold in TMEM lanes m and m ^ 8
// (the same warp) all four real products, so
//     Re = (A_r B_r)[lane p=0] - (A_i B_i)[lane p=1]
//     Im = (A_r B_i)[lane p=0] + (A_i B_r)[lane p=1]
// is one exchange between partner lanes. The C tile is loaded in that layout
// by TMA (8-row boxes); x^T is written in it by a shared-memory transpose and
// serves both as an interleaved A operand and, read with a 2 KB group
// stride, as two planar B operands.
//
// Roles in a CTA (288 threads):
//   warps 0-7  workers: transposes, decay mask, state hop, epilogue; worker
//              thread 0 issues the tcgen05 MMAs
//   warp 8     producer: TMA loads of the next chunk's C, B, x tiles into a
//              two-stage ring, dt and the in-chunk cumulative log-decay
// Worker warps w and w + 4 share TMEM lane quadrant w % 4 and split the
// 64 columns of each accumulator row between them (h = w / 4).
#include <cuda.h>
#include <cuda_runtime.h>

#include "tc_common.cuh"

namespace ssdc {
namespace fused {
namespace {

using namespace tc;

constexpr int kQ = 64;
constexpr int kWorkers = 256;
constexpr int kThreads = kWorkers + 32;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: pairs of 64-column accumulators (A * Br | A * Bi) and the
// P operand (64 columns). The C B^T pair is reused for C S_in.
constexpr uint32_t kAccG = 0, kAccS = 128, kAccY = 256, kPwin = 384;
constexpr uint32_t kTileBytes = 2 * kPlaneBytes;  // 32 KB: one complex 64 x 64 tile
constexpr uint32_t kStageTx = 3 * kTileBytes;     // C, B, x
constexpr uint32_t kStateBytes = kTileBytes;
constexpr uint32_t kIntHalf = 16384;  // one 32-column half of a 128-row tile
constexpr uint32_t kIdesc128 = ptx::idesc_tf32(128, 128, 0);  // M = 128, N = 128, B operand K-major
constexpr uint32_t kBarWorkers = 1;   // named barrier id of the worker warps

struct Smem {
    float c[2][64 * 128];    // [stage] C, interleaved 128 rows (A operand)
    float b[2][64 * 128];    // [stage] B, stacked (rows s); after C B^T, (dec o B)^T stacked (rows n)
    float x[2][64 * 128];    // [stage] x, stacked (rows s); x^T interleaved (rows d); then y staging
    float sin[64 * 128];     // incoming state S_in^T, stacked (rows d, n contiguous)
    float2 acs[2][kQ];       // in-chunk cumulative log-decay, per stage
    float2 dec[kQ];          // exp(Acs[Q-1] - Acs[s])
    float2 eacs[kQ];         // exp(Acs[l])
    float2 a_c;              // exp(Acs[Q-1])
    uint64_t full[2], empty[2], sin_full, succ_empty;
    uint64_t mma[4];         // one per MMA group (C B^T, S_loc^T, Y_diag, C S_in), one phase per chunk
    uint32_t tmem;
};

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
// operand of 128 rows: [32-column half][plane][64 rows][128 B], so that a
// descriptor over 128 rows covers plane 0 (rows 0-63) and plane 1 (rows
// 64-127). An "interleaved" tile is [32-column half][128 rows][128 B] with
// row 16g + 8p + i = plane p of row 8g + i. Rows are 128-byte swizzled.
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
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&sm.full[s], 1);
            ptx::mbar_init(&sm.empty[s], 1);
        }
        for (int g = 0; g < 4; ++g) ptx::mbar_init(&sm.mma[g], 1);
        ptx::mbar_init(&sm.sin_full, 1);
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

    if (warp == kWorkers / 32) {
        // ------------------------------------------------------- producer
        for (int64_t it = 0; it < nitems; ++it) {
            const int s = (int)(it & 1);
            if (it >= 2 && !ptx::mbar_wait(&sm.empty[s], (uint32_t)(((it >> 1) & 1) ^ 1), kWaitIters))
                fail(ws.status);
            int64_t q, c;
            items.get(it, q, c);
            const int b = (int)(q / H), h = (int)(q % H);
            const int64_t t0 = c * kQ;
            if (lane == 0) {
                ptx::mbar_expect_tx(&sm.full[s], kStageTx);
                char* cb = reinterpret_cast<char*>(sm.c[s]);
                char* bb = reinterpret_cast<char*>(sm.b[s]);
                char* xb = reinterpret_cast<char*>(sm.x[s]);
                for (int half = 0; half < 2; ++half) {
                    const int f0 = 32 * half;
                    // C as 8-row boxes, re and im groups interleaved
                    for (int g = 0; g < 8; ++g) {
                        ptx::tma_load_4d(cb + inter_row(half, 16 * g), &c8_re, &sm.full[s], f0, h, (int)t0 + 8 * g, b);
                        ptx::tma_load_4d(cb + inter_row(half, 16 * g + 8), &c8_im, &sm.full[s], f0, h, (int)t0 + 8 * g, b);
                    }
                    ptx::tma_load_4d(bb + stk_row(half, 0, 0), &maps.B_re, &sm.full[s], f0, h, (int)t0, b);
                    ptx::tma_load_4d(bb + stk_row(half, 1, 0), &maps.B_im, &sm.full[s], f0, h, (int)t0, b);
                    ptx::tma_load_4d(xb + stk_row(half, 0, 0), &maps.x_re, &sm.full[s], f0, h, (int)t0, b);
                    ptx::tma_load_4d(xb + stk_row(half, 1, 0), &maps.x_im, &sm.full[s], f0, h, (int)t0, b);
                }
            }
            // discretisation and in-chunk inclusive cumulative sum (fp64 accumulation)
            const float Ar = p.A_re[h], Ai = p.A_im[h];
            double r0 = 0.0, i0 = 0.0, r1 = 0.0, i1 = 0.0;
            {
                const int64_t ta = t0 + 2 * lane, tb = ta + 1;
                if (ta < p.T) {
                    const float sp = softplus_f(p.dt[((int64_t)b * p.T + ta) * H + h]);
                    r0 = (double)(sp * Ar);
                    i0 = (double)(sp * Ai);
                }
                if (tb < p.T) {
                    const float sp = softplus_f(p.dt[((int64_t)b * p.T + tb) * H + h]);
                    r1 = (double)(sp * Ar);
                    i1 = (double)(sp * Ai);
                }
            }
            double cr = r0 + r1, ci = i0 + i1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const double ur = __shfl_up_sync(0xffffffffu, cr, off);
                const double ui = __shfl_up_sync(0xffffffffu, ci, off);
                if (lane >= off) {
                    cr += ur;
                    ci += ui;
                }
            }
            const double er = cr - (r0 + r1), ei = ci - (i0 + i1);  // exclusive prefix
            sm.acs[s][2 * lane] = make_float2((float)(er + r0), (float)(ei + i0));
            sm.acs[s][2 * lane + 1] = make_float2((float)(er + r0 + r1), (float)(ei + i0 + i1));
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm.full[s]);
        }
    } else {
        // -------------------------------------------------------- workers
        const int h2 = warp >> 2;                   // column half of this warp
        const int m = (warp & 3) * 32 + lane;       // TMEM lane
        const int r8 = 8 * (m >> 4) + (m & 7);      // complex row (l or d) of this lane
        const int pl = (m >> 3) & 1;                // plane of this lane
        const uint32_t my = lane_base(tmem, warp);
        uint32_t n_recv = 0, n_send = 0;
        const uint32_t sin_saddr = ptx::smem_addr(sm.sin);
        const uint32_t remote_sin = ptx::mapa(sin_saddr, succ);
        const uint32_t remote_sin_full = ptx::mapa(ptx::smem_addr(&sm.sin_full), succ);
        const uint32_t remote_pred_empty = ptx::mapa(ptx::smem_addr(&sm.succ_empty), pred);

        // MMA group g of item `it` completes phase `it` of barrier mma[g]
        auto wait_mma = [&](int g, int64_t it) {
            if (!ptx::mbar_wait(&sm.mma[g], (uint32_t)(it & 1), kWaitIters)) fail(ws.status);
            ptx::tc_fence_after();
        };
        auto publish = [&]() {  // tcgen05.st and smem writes of all workers -> MMA issue
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::named_sync(kBarWorkers, kWorkers);
            ptx::tc_fence_after();
        };

        for (int64_t it = 0; it < nitems; ++it) {
            const int s = (int)(it & 1);
            int64_t q, c;
            items.get(it, q, c);
            const int b = (int)(q / H), h = (int)(q % H);
            const int64_t t0 = c * kQ;
            const bool has_in = c > 0, last = c == p.nc - 1;
            char* cbase = reinterpret_cast<char*>(sm.c[s]);
            char* bbase = reinterpret_cast<char*>(sm.b[s]);
            char* xbase = reinterpret_cast<char*>(sm.x[s]);
            const uint32_t cs = ptx::smem_addr(cbase), bs = ptx::smem_addr(bbase), xs = ptx::smem_addr(xbase);
            if (!ptx::mbar_wait(&sm.full[s], (uint32_t)((it >> 1) & 1), kWaitIters)) fail(ws.status);

            // ---- A: decays; x and B 4x4 blocks into registers. Lane bits pick the
            // block so that the 16-byte loads and stores of a warp spread over all
            // eight bank groups of the swizzled rows.
            if (tid < kQ) {
                sm.dec[tid] = cexp_fast(cdiff(sm.acs[s][kQ - 1], sm.acs[s][tid]));
            } else if (tid < 2 * kQ) {
                sm.eacs[tid - kQ] = cexp_fast(sm.acs[s][tid - kQ]);
            } else if (tid == 2 * kQ) {
                sm.a_c = cexp_fast(sm.acs[s][kQ - 1]);
            }
            const int blo = lane & 7, bmid = (lane >> 3) & 3;
            float4 xv[2][4], bv[2][4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {  // x block: rows s = 4 sbk + i, columns d = 4 dbk ..
                const int wq = warp + 8 * u;
                const int sbk = bmid + 4 * (wq & 3), dbk = blo + 8 * ((wq >> 2) & 1), xp = (wq >> 3) & 1;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int sr = 4 * sbk + i;
                    xv[u][i] = *reinterpret_cast<const float4*>(xbase + stk_row(dbk >> 3, xp, sr) + chunk16(dbk & 7, sr));
                }
            }
            const int bsb = bmid + 4 * (warp & 3), bnb = blo + 8 * ((warp >> 2) & 1);  // rows s = 4 bsb .., columns n = 4 bnb ..
#pragma unroll
            for (int pp = 0; pp < 2; ++pp)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int sr = 4 * bsb + i;
                    bv[pp][i] = *reinterpret_cast<const float4*>(bbase + stk_row(bnb >> 3, pp, sr) + chunk16(bnb & 7, sr));
                }
            ptx::named_sync(kBarWorkers, kWorkers);

            // ---- B: x^T (interleaved rows d) in place of x; then C B^T
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int wq = warp + 8 * u;
                const int sbk = bmid + 4 * (wq & 3), dbk = blo + 8 * ((wq >> 2) & 1), xp = (wq >> 3) & 1;
                const float4 o[4] = {make_float4(xv[u][0].x, xv[u][1].x, xv[u][2].x, xv[u][3].x),
                                     make_float4(xv[u][0].y, xv[u][1].y, xv[u][2].y, xv[u][3].y),
                                     make_float4(xv[u][0].z, xv[u][1].z, xv[u][2].z, xv[u][3].z),
                                     make_float4(xv[u][0].w, xv[u][1].w, xv[u][2].w, xv[u][3].w)};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int mm = inter_m(4 * dbk + j, xp);
                    *reinterpret_cast<float4*>(xbase + inter_row(sbk >> 3, mm) + chunk16(sbk & 7, mm)) = o[j];
                }
            }
            ptx::fence_proxy_async_smem();
            publish();
            if (tid == 0) {
                issue_ss128(tmem + kAccG, desc128(cs), desc128(bs));  // [C Br | C Bi]
                ptx::mma_commit(&sm.mma[0]);
            }
            wait_mma(0, it);

            // ---- C: (dec o B)^T stacked in place of B; then S_loc^T = x^T (dec o B)
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
            publish();
            if (tid == 0) {
                issue_ss128(tmem + kAccS, desc128(xs), desc128(bs));  // [x^T B'r | x^T B'i]
                ptx::mma_commit(&sm.mma[1]);
            }

            // ---- D: P = (C B^T) o L on this thread's columns; P operand rows into TMEM
            {
                float ga[32], gb[32];
                ptx::tmem_ld16(my + kAccG + 16 * h2, ga);
                ptx::tmem_ld16(my + kAccG + 32 + 16 * h2, ga + 16);
                ptx::tmem_ld16(my + kAccG + 64 + 16 * h2, gb);
                ptx::tmem_ld16(my + kAccG + 96 + 16 * h2, gb + 16);
                ptx::tmem_wait_ld();
                const float2 acs_l = sm.acs[s][r8];
                float w[32];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int e = (jj < 8 ? 16 * h2 : 32 + 16 * h2) + 2 * (jj & 7);  // even column of the pair
                    const float ra = __shfl_xor_sync(0xffffffffu, pl ? ga[2 * jj] : ga[2 * jj + 1], 8);
                    const float rb = __shfl_xor_sync(0xffffffffu, pl ? gb[2 * jj] : gb[2 * jj + 1], 8);
                    // plane-0 products (Cr B) and plane-1 products (Ci B) of this thread's column
                    const float ga0 = pl ? ra : ga[2 * jj], gb0 = pl ? rb : gb[2 * jj];
                    const float ga1 = pl ? ga[2 * jj + 1] : ra, gb1 = pl ? gb[2 * jj + 1] : rb;
                    const int col = e + pl;
                    float2 v = make_float2(0.0f, 0.0f);
                    if (col <= r8)
                        v = cmul(make_float2(ga0 - gb1, gb0 + ga1), cexp_fast(cdiff(acs_l, sm.acs[s][col])));
                    // lane p keeps plane p of P: column e from the p = 0 lane, e + 1 from the p = 1 lane
                    const float other = __shfl_xor_sync(0xffffffffu, pl ? v.x : v.y, 8);
                    w[2 * jj] = pl ? other : v.x;
                    w[2 * jj + 1] = pl ? v.y : other;
                }
                ptx::tmem_st16(my + kPwin + 16 * h2, w);
                ptx::tmem_st16(my + kPwin + 32 + 16 * h2, w + 16);
            }
            publish();
            if (tid == 0) {
                // Y_diag: columns 16g + 8p + i hold plane p of P x (row d = 8g + i)
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    ptx::mma_tf32_ts(tmem + kAccY, tmem + kPwin + 8 * k, desc_k(desc128(xs), k), kIdesc128, k > 0);
                ptx::mma_commit(&sm.mma[2]);
            }

            // ---- E: S_loc^T and the state hop  S_out = a_c S_in + S_loc  (row d = r8)
            wait_mma(1, it);  // S_loc^T
            float out[32];
            {
                float sa[32], sb[32];
                ptx::tmem_ld16(my + kAccS + 32 * h2, sa);
                ptx::tmem_ld16(my + kAccS + 16 + 32 * h2, sa + 16);
                ptx::tmem_ld16(my + kAccS + 64 + 32 * h2, sb);
                ptx::tmem_ld16(my + kAccS + 80 + 32 * h2, sb + 16);
                ptx::tmem_wait_ld();
                if (has_in && CL > 1) {
                    if (!ptx::mbar_wait(&sm.sin_full, n_recv & 1, kWaitIters)) fail(ws.status);
                    ++n_recv;
                }
                const float2 a = sm.a_c;
                const char* sinb = reinterpret_cast<const char*>(sm.sin);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float4 sr = make_float4(0.f, 0.f, 0.f, 0.f), si = sr;
                    if (has_in) {
                        sr = *reinterpret_cast<const float4*>(sinb + stk_row(h2, 0, r8) + chunk16(j, r8));
                        si = *reinterpret_cast<const float4*>(sinb + stk_row(h2, 1, r8) + chunk16(j, r8));
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
            if (last) {
                float* fs = (pl ? p.fs_im : p.fs_re) + (q * 64) * 64 + r8;
#pragma unroll
                for (int k = 0; k < 32; ++k) fs[(int64_t)(32 * h2 + k) * 64] = out[k];
            } else if (CL > 1) {
                if (n_send > 0 && !ptx::mbar_wait(&sm.succ_empty, (n_send - 1) & 1, kWaitIters)) fail(ws.status);
                ++n_send;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    ptx::st_async_v4(remote_sin + stk_row(h2, pl, r8) + chunk16(j, r8),
                                     make_float4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]),
                                     remote_sin_full);
            }

            // ---- F: C S_in (reuses the C B^T accumulators)
            publish();
            if (tid == 0) {
                if (has_in) issue_ss128(tmem + kAccG, desc128(cs), desc128(sin_saddr));  // [C Sr | C Si]
                ptx::mma_commit(&sm.mma[3]);
            }
            wait_mma(2, it);  // Y_diag
            wait_mma(3, it);  // C S_in
            if (has_in && CL > 1 && tid == 0) {
                // the incoming buffer is consumed: re-arm it and free it for the sender
                ptx::mbar_arrive_expect_tx(&sm.sin_full, kStateBytes);
                ptx::mbar_arrive_remote(remote_pred_empty);
            }
            if (!last && CL == 1) {
                // keep the state for this CTA's next chunk
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<float4*>(reinterpret_cast<char*>(sm.sin) + stk_row(h2, pl, r8) + chunk16(j, r8)) =
                        make_float4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
                ptx::fence_proxy_async_smem();
            }

            // ---- G: y = Y_diag + exp(Acs[l]) (C S_in), staged in the x buffer
            // (both MMAs reading x^T are done) and written by TMA.
            {
                const float2 e = sm.eacs[r8];
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    const int c0 = 32 * h2 + 16 * pass;  // first column d of this pass
                    float yv[32], za[16], zb[16];
                    ptx::tmem_ld16(my + kAccY + 2 * c0, yv);
                    ptx::tmem_ld16(my + kAccY + 2 * c0 + 16, yv + 16);
                    ptx::tmem_ld16(my + kAccG + c0, za);
                    ptx::tmem_ld16(my + kAccG + 64 + c0, zb);
                    ptx::tmem_wait_ld();
                    float o[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int yi = 16 * (k >> 3) + (k & 7);  // Y column of plane 0; plane 1 is 8 further
                        const float ya = yv[yi], yb = yv[yi + 8];
                        const float zak = has_in ? za[k] : 0.0f, zbk = has_in ? zb[k] : 0.0f;
                        // this lane's share of Re y and Im y (see the header comment)
                        const float u = pl ? (-yb - e.x * zbk - e.y * zak) : (ya + e.x * zak - e.y * zbk);
                        const float v = pl ? (ya + e.x * zak - e.y * zbk) : (yb + e.x * zbk + e.y * zak);
                        const float other = __shfl_xor_sync(0xffffffffu, pl ? u : v, 8);
                        o[k] = pl ? v + other : u + other;
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        *reinterpret_cast<float4*>(xbase + stk_row(h2, pl, r8) + chunk16(4 * pass + k, r8)) =
                            make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_sync(kBarWorkers, kWorkers);
            if (tid == 0) {
                for (int half = 0; half < 2; ++half) {
                    ptx::tma_store_4d(&y_re, xbase + stk_row(half, 0, 0), 32 * half, h, (int)t0, b);
                    ptx::tma_store_4d(&y_im, xbase + stk_row(half, 1, 0), 32 * half, h, (int)t0, b);
                }
                ptx::bulk_commit();
                ptx::bulk_wait_read_all();  // the stage may be refilled once the store has read it
                ptx::mbar_arrive(&sm.empty[s]);
            }
        }
        if (tid == 0) ptx::bulk_wait_all();
    }

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
