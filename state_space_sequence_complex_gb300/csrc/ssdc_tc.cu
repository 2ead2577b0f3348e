// tcgen05 / TMA kernels of the chunkwise complex SSD forward: the chunk
// contractions on the TF32 tensor cores (landing page, "03 Chunkwise SSD":
// the CHUNK line, L and Y_diag = einsum(C, B, L, X), and the STATE line,
// s_chunk = einsum(B, decay, X)).
//
// Complex products as real MMAs. Every complex matrix product here has the
// form R = A * B with A an m x k complex matrix built by the threads and B a
// k x n complex matrix staged in shared memory by TMA (planar: Br, Bi). A is
// written to tensor memory as two 128-row "windows" whose rows interleave the
// real and imaginary parts of A's rows:
//     W1 row 2i = Re A[i,:]     W1 row 2i+1 = Im A[i,:]
//     W2 row 2i = -Im A[i,:]    W2 row 2i+1 = Re A[i,:]
// so that the two M=128 MMAs  D = W1 * Br + W2 * Bi  leave
//     D row 2i = Re R[i,:],  D row 2i+1 = Im R[i,:]
// in TMEM lanes 2i and 2i+1, which belong to adjacent threads of one warp.
// Any complex elementwise step on R (the decay mask L) is then a pair of
// shuffles between neighbour lanes; no shared-memory exchange is needed.
//
// Kernels (128 threads = 4 warps; thread t owns TMEM lane t):
//   tc_chunk_state  grid (nc, H, B): S_loc^T and a_c of one chunk
//   tc_chunk_scan   grid (nc * ceil(Q/64), H, B): 64 output rows of one chunk (Q = 32: the
//                   first 32 rows of a 64-row tile)
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "tc_common.cuh"

namespace ssdc {
namespace tc {
namespace {

constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 256;
// Column offsets inside the CTA's TMEM allocation.
constexpr uint32_t kW1 = 0, kW2 = 64, kAccA = 128, kAccB = 192;

// ------------------------------------------------------------------------
// Chunk state: S_loc[n, d] = sum_s (dec[s] B[s, n]) x[s, d], written as
// S_loc^T (d rows, n contiguous) per plane; a_c = exp(Acs[Q-1]).
// TMEM: W1, W2 (the dec o B^T windows), kAccA = accumulator.
// All threads: make this thread's tcgen05.st visible, then thread 0 may
// issue MMAs reading them.
__device__ __forceinline__ void publish_tmem_writes() {
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
}

struct StateSmem {
    float b[2][64 * 64];  // B block: re, im planes
    float x[2][64 * 64];  // x block: re, im planes
    Acs acs[kMaxQ];
    float2 dec[kMaxQ];
    uint64_t bar_in, bar_mma;
    uint32_t tmem;
};

__global__ void __launch_bounds__(kThreads)
tc_chunk_state(Problem p, Workspace ws, const __grid_constant__ TcMaps maps) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    StateSmem& sm = *reinterpret_cast<StateSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int Q = p.Q, H = p.H;
    const int64_t t0 = (int64_t)c * Q;
    const int nvalid = (int)(p.T - t0 < (int64_t)Q ? p.T - t0 : (int64_t)Q);

    if (tid == 0) {
        ptx::mbar_init(&sm.bar_in, 1);
        ptx::mbar_init(&sm.bar_mma, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(&sm.tmem, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem;
    const uint32_t my = lane_base(tmem, warp);

    const uint32_t sb_re = ptx::smem_addr(sm.b[0]), sb_im = ptx::smem_addr(sm.b[1]);
    const uint32_t sx_re = ptx::smem_addr(sm.x[0]), sx_im = ptx::smem_addr(sm.x[1]);
    const bool real_x = p.x_im == nullptr;  // x real: its imaginary plane stays zero in shared memory
    if (real_x) {
        for (int i = tid; i < 64 * 64; i += kThreads) sm.x[1][i] = 0.0f;
    }
    auto load_block = [&](int s0) {
        ptx::mbar_arrive_expect_tx(&sm.bar_in, (real_x ? 3 : 4) * kPlaneBytes);
        const int t = (int)(t0 + s0);
        for (int half = 0; half < 2; ++half) {
            ptx::tma_load_4d(reinterpret_cast<char*>(sm.b[0]) + half * kHalfBytes, &maps.B_re, &sm.bar_in, 32 * half, h, t, b);
            ptx::tma_load_4d(reinterpret_cast<char*>(sm.b[1]) + half * kHalfBytes, &maps.B_im, &sm.bar_in, 32 * half, h, t, b);
            ptx::tma_load_4d(reinterpret_cast<char*>(sm.x[0]) + half * kHalfBytes, &maps.x_re, &sm.bar_in, 32 * half, h, t, b);
            if (!real_x)
                ptx::tma_load_4d(reinterpret_cast<char*>(sm.x[1]) + half * kHalfBytes, &maps.x_im, &sm.bar_in, 32 * half, h, t, b);
        }
    };
    if (tid == 0) load_block(0);

    if (warp == 0)
        chunk_cumsum_warp(p.dt + ((int64_t)b * p.T + t0) * H + h, H, nvalid, Q, p.A_re[h], p.A_im[h], sm.acs);
    __syncthreads();
    const Acs last = sm.acs[Q - 1];
    for (int s = tid; s < Q; s += kThreads) sm.dec[s] = cexp_fast(acs_diff(last, sm.acs[s]));
    __syncthreads();

    const int n = tid >> 1, part = tid & 1;
    uint32_t ph_in = 0, ph_mma = 0;
    // 64-row blocks of the chunk; with Q = 32 the block's last 32 rows belong to the next chunk
    // and get a zero window (they add nothing to S_loc)
    const int nblocks = (Q + kRows - 1) / kRows;
    for (int sb = 0; sb < nblocks; ++sb) {
        if (!ptx::mbar_wait(&sm.bar_in, ph_in, kWaitIters)) fail(ws.status);
        ph_in ^= 1;
        // windows of A[n, s] = dec[s] * B[s, n]
        float w1[64], w2[64];
#pragma unroll
        for (int s = 0; s < 64; ++s) {
            const float2 bv = make_float2(plane_ld(sm.b[0], s, n), plane_ld(sm.b[1], s, n));
            const int sg = sb * kRows + s;
            const float2 a = sg < Q ? cmul(sm.dec[sg], bv) : make_float2(0.0f, 0.0f);
            w1[s] = part ? a.y : a.x;
            w2[s] = part ? a.x : -a.y;
        }
        tmem_store<64>(my + kW1, w1);
        tmem_store<64>(my + kW2, w2);
        __syncthreads();  // every thread is done reading B
        transpose_tile<kThreads>(sm.x[0], sm.b[0], tid);  // x^T (d rows, s contiguous) into the B buffer
        ptx::fence_proxy_async_smem();
        publish_tmem_writes();
        if (tid == 0) {
            issue_pair(tmem + kAccA, tmem + kW1, tmem + kW2, sb_re, sb_im, sb > 0);
            ptx::mma_commit(&sm.bar_mma);
        }
        if (!ptx::mbar_wait(&sm.bar_mma, ph_mma, kWaitIters)) fail(ws.status);
        ph_mma ^= 1;
        ptx::tc_fence_after();
        if (tid == 0 && sb + 1 < nblocks) {
            ptx::fence_proxy_async_smem();
            load_block((sb + 1) * kRows);
        }
    }

    // epilogue: lane 2n+part holds plane `part` of S_loc[n, 0..63]
    float v[64];
    tmem_load<64>(my + kAccA, v);
    const int64_t chunk = ((int64_t)b * H + h) * p.nc + c;
    float* S = ws.S + (chunk * 2 + part) * 64 * 64;
#pragma unroll
    for (int d = 0; d < 64; ++d) S[d * 64 + n] = v[d];
    if (tid == 0) {
        const float2 a = cexp_fast(acs_value(last));
        ws.a[2 * chunk] = a.x;
        ws.a[2 * chunk + 1] = a.y;
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
    (void)sx_re;
    (void)sx_im;
}

// ------------------------------------------------------------------------
// Chunk scan: rows l0 .. l0+63 of one chunk,
//   y = sum_{s-blocks <= l-block} (G o L) x + (C o exp(Acs)) S_in,  G = C B^T.
// TMEM: W1, W2 (windows of C, then P, then C'), kAccA = G, kAccB = y.
struct ScanSmem {
    float cpl[2][64 * 64];  // C rows of the l-block: re, im
    float b[2][64 * 64];    // B rows of the s-block; later S_in^T (re, im)
    float x[2][64 * 64];    // x rows of the s-block
    Acs acs[kMaxQ];
    uint64_t bar_c, bar_bx, bar_s, bar_mma;
    uint32_t tmem;
};

__global__ void __launch_bounds__(kThreads)
tc_chunk_scan(Problem p, Workspace ws, const __grid_constant__ TcMaps maps) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    ScanSmem& sm = *reinterpret_cast<ScanSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int Q = p.Q, H = p.H;
    // 64-row output blocks; with Q = 32 the block's last 32 rows (the next chunk's) are computed
    // from clamped decays and never stored
    const int lblocks = (Q + kRows - 1) / kRows;
    const int c = blockIdx.x / lblocks, lb = blockIdx.x % lblocks;
    const int h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int64_t t0 = (int64_t)c * Q;
    const int nvalid = (int)(p.T - t0 < (int64_t)Q ? p.T - t0 : (int64_t)Q);
    const int l0 = lb * kRows;
    if (l0 >= nvalid) return;  // whole l-block past the sequence end (uniform)

    if (tid == 0) {
        ptx::mbar_init(&sm.bar_c, 1);
        ptx::mbar_init(&sm.bar_bx, 1);
        ptx::mbar_init(&sm.bar_s, 1);
        ptx::mbar_init(&sm.bar_mma, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(&sm.tmem, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem;
    const uint32_t my = lane_base(tmem, warp);

    const bool real_x = p.x_im == nullptr;  // x real: its imaginary plane stays zero in shared memory
    if (real_x) {
        for (int i = tid; i < 64 * 64; i += kThreads) sm.x[1][i] = 0.0f;
    }
    auto load_bx = [&](int s0) {
        ptx::mbar_arrive_expect_tx(&sm.bar_bx, (real_x ? 3 : 4) * kPlaneBytes);
        const int t = (int)(t0 + s0);
        for (int half = 0; half < 2; ++half) {
            ptx::tma_load_4d(reinterpret_cast<char*>(sm.b[0]) + half * kHalfBytes, &maps.B_re, &sm.bar_bx, 32 * half, h, t, b);
            ptx::tma_load_4d(reinterpret_cast<char*>(sm.b[1]) + half * kHalfBytes, &maps.B_im, &sm.bar_bx, 32 * half, h, t, b);
            ptx::tma_load_4d(reinterpret_cast<char*>(sm.x[0]) + half * kHalfBytes, &maps.x_re, &sm.bar_bx, 32 * half, h, t, b);
            if (!real_x)
                ptx::tma_load_4d(reinterpret_cast<char*>(sm.x[1]) + half * kHalfBytes, &maps.x_im, &sm.bar_bx, 32 * half, h, t, b);
        }
    };
    const int64_t chunk = ((int64_t)b * H + h) * p.nc + c;
    if (tid == 0) {
        ptx::mbar_arrive_expect_tx(&sm.bar_c, 2 * kPlaneBytes);
        const int t = (int)(t0 + l0);
        for (int half = 0; half < 2; ++half) {
            ptx::tma_load_4d(reinterpret_cast<char*>(sm.cpl[0]) + half * kHalfBytes, &maps.C_re, &sm.bar_c, 32 * half, h, t, b);
            ptx::tma_load_4d(reinterpret_cast<char*>(sm.cpl[1]) + half * kHalfBytes, &maps.C_im, &sm.bar_c, 32 * half, h, t, b);
        }
        load_bx(0);
    }
    if (warp == 0)
        chunk_cumsum_warp(p.dt + ((int64_t)b * p.T + t0) * H + h, H, nvalid, Q, p.A_re[h], p.A_im[h], sm.acs);
    __syncthreads();

    const int l = tid >> 1, part = tid & 1;
    const Acs acs_l = sm.acs[l0 + l < Q ? l0 + l : Q - 1];
    const uint32_t sb_re = ptx::smem_addr(sm.b[0]), sb_im = ptx::smem_addr(sm.b[1]);
    const uint32_t sx_re = ptx::smem_addr(sm.x[0]), sx_im = ptx::smem_addr(sm.x[1]);
    uint32_t ph_bx = 0, ph_mma = 0;
    if (!ptx::mbar_wait(&sm.bar_c, 0, kWaitIters)) fail(ws.status);

    for (int sb = 0; sb <= lb; ++sb) {
        const int s0 = sb * kRows;
        if (!ptx::mbar_wait(&sm.bar_bx, ph_bx, kWaitIters)) fail(ws.status);
        ph_bx ^= 1;
        // C windows: row 2l = (Cr | -Ci), row 2l+1 = (Ci | Cr)
        {
            float w1[64], w2[64];
#pragma unroll
            for (int k = 0; k < 64; ++k) {
                const float cr = plane_ld(sm.cpl[0], l, k), ci = plane_ld(sm.cpl[1], l, k);
                w1[k] = part ? ci : cr;
                w2[k] = part ? cr : -ci;
            }
            tmem_store<64>(my + kW1, w1);
            tmem_store<64>(my + kW2, w2);
        }
        publish_tmem_writes();
        if (tid == 0) {
            issue_pair(tmem + kAccA, tmem + kW1, tmem + kW2, sb_re, sb_im, false);
            ptx::mma_commit(&sm.bar_mma);
        }
        if (!ptx::mbar_wait(&sm.bar_mma, ph_mma, kWaitIters)) fail(ws.status);
        ph_mma ^= 1;
        ptx::tc_fence_after();
        // the C B^T MMA has consumed B: x^T (d rows, s contiguous) goes into its buffer
        transpose_tile<kThreads>(sm.x[0], sm.b[0], tid);
        ptx::fence_proxy_async_smem();

        // P = G o L; this thread takes columns s = 2j + part
        float g[64];
        tmem_load<64>(my + kAccA, g);
        float pr[32], pi[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float send = part ? g[2 * j] : g[2 * j + 1];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const float gre = part ? recv : g[2 * j];
            const float gim = part ? g[2 * j + 1] : recv;
            const int s = 2 * j + part;
            float2 v = make_float2(0.0f, 0.0f);
            if (s0 + s <= l0 + l) {
                const float2 L = cexp_fast(acs_diff(acs_l, sm.acs[s0 + s < Q ? s0 + s : Q - 1]));
                v = cmul(make_float2(gre, gim), L);
            }
            pr[j] = v.x;
            pi[j] = v.y;
        }
        // P windows: row 2l = (Pr | -Pi), row 2l+1 = (Pi | Pr)
        {
            float w1[64], w2[64];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float opr = __shfl_xor_sync(0xffffffffu, pr[j], 1);
                const float opi = __shfl_xor_sync(0xffffffffu, pi[j], 1);
                const float re_e = part ? opr : pr[j], im_e = part ? opi : pi[j];  // column 2j
                const float re_o = part ? pr[j] : opr, im_o = part ? pi[j] : opi;  // column 2j+1
                w1[2 * j] = part ? im_e : re_e;
                w1[2 * j + 1] = part ? im_o : re_o;
                w2[2 * j] = part ? re_e : -im_e;
                w2[2 * j + 1] = part ? re_o : -im_o;
            }
            tmem_store<64>(my + kW1, w1);
            tmem_store<64>(my + kW2, w2);
        }
        publish_tmem_writes();
        if (tid == 0) {
            issue_pair(tmem + kAccB, tmem + kW1, tmem + kW2, sb_re, sb_im, sb > 0);
            ptx::mma_commit(&sm.bar_mma);
        }
        if (!ptx::mbar_wait(&sm.bar_mma, ph_mma, kWaitIters)) fail(ws.status);
        ph_mma ^= 1;
        ptx::tc_fence_after();
        if (tid == 0) {
            ptx::fence_proxy_async_smem();
            if (sb < lb) {
                load_bx(s0 + kRows);
            } else {
                // S_in^T of this chunk into the x buffer (x was consumed by the transpose)
                ptx::mbar_arrive_expect_tx(&sm.bar_s, 2 * kPlaneBytes);
                const int row = (int)(chunk * 2 * 64);
                for (int half = 0; half < 2; ++half) {
                    ptx::tma_load_2d(reinterpret_cast<char*>(sm.x[0]) + half * kHalfBytes, &maps.S, &sm.bar_s, 32 * half, row);
                    ptx::tma_load_2d(reinterpret_cast<char*>(sm.x[1]) + half * kHalfBytes, &maps.S, &sm.bar_s, 32 * half, row + 64);
                }
            }
        }
    }

    // Y_off: windows of C' = C o exp(Acs[l]), times S_in (B operand S_in^T, K-major)
    {
        const float2 e = cexp_fast(acs_value(acs_l));
        float w1[64], w2[64];
#pragma unroll
        for (int k = 0; k < 64; ++k) {
            const float2 cv = cmul(make_float2(plane_ld(sm.cpl[0], l, k), plane_ld(sm.cpl[1], l, k)), e);
            w1[k] = part ? cv.y : cv.x;
            w2[k] = part ? cv.x : -cv.y;
        }
        tmem_store<64>(my + kW1, w1);
        tmem_store<64>(my + kW2, w2);
    }
    if (!ptx::mbar_wait(&sm.bar_s, 0, kWaitIters)) fail(ws.status);
    publish_tmem_writes();
    if (tid == 0) {
        issue_pair(tmem + kAccB, tmem + kW1, tmem + kW2, sx_re, sx_im, true);
        ptx::mma_commit(&sm.bar_mma);
    }
    if (!ptx::mbar_wait(&sm.bar_mma, ph_mma, kWaitIters)) fail(ws.status);
    ptx::tc_fence_after();

    float v[64];
    tmem_load<64>(my + kAccB, v);
    if (l0 + l < nvalid) {
        float* yp = (part ? p.y_im : p.y_re) + ((((int64_t)b * p.T + t0 + l0 + l) * H + h) * 64);
        float4* y4 = reinterpret_cast<float4*>(yp);
#pragma unroll
        for (int q = 0; q < 16; ++q) y4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool get_encoder() {
    if (g_encode) return true;
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

}  // namespace

// (F, H, T, B) fp32 plane, box (32, 1, rows, 1), 128-byte swizzle, zero fill.
bool encode_feature_map(CUtensorMap* m, const float* base, int F, int H, int64_t T, int B, int rows) {
    if (!get_encoder()) return false;
    cuuint64_t dims[4] = {(cuuint64_t)F, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)F * 4, (cuuint64_t)F * H * 4, (cuuint64_t)F * H * 4 * (cuuint64_t)T};
    cuuint32_t box[4] = {32, 1, (cuuint32_t)rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// (F, H, T, B) bfloat16 plane, box (64, 1, rows, 1): one 128-byte swizzled row
// of 64 features per token, zero fill past F and T.
bool encode_feature_map_bf16(CUtensorMap* m, const void* base, int F, int H, int64_t T, int B, int rows) {
    if (!get_encoder()) return false;
    cuuint64_t dims[4] = {(cuuint64_t)F, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)F * 2, (cuuint64_t)F * H * 2, (cuuint64_t)F * H * 2 * (cuuint64_t)T};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tiled_f32(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                      const cuuint32_t* box) {
    if (!get_encoder() || rank < 1 || rank > 5) return false;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

bool make_feature_map(CUtensorMap* m, const float* base, int F, int H, int64_t T, int B) {
    return encode_feature_map(m, base, F, H, T, B, 64);
}

// Workspace states as rows of 64 floats, box (32, 64).
bool make_state_map(CUtensorMap* m, const float* base, int64_t rows) {
    cuuint64_t dims[2] = {64, (cuuint64_t)rows};
    cuuint64_t strides[1] = {64 * 4};
    cuuint32_t box[2] = {32, 64};
    cuuint32_t es[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int make_maps(const Problem& p, const float* ws_S, TcMaps* m) {
    if (!get_encoder()) return SSDC_ERR_CUDA;
    bool ok = make_feature_map(&m->x_re, p.x_re, 64, p.H, p.T, p.B) &&
              (p.x_im == nullptr || make_feature_map(&m->x_im, p.x_im, 64, p.H, p.T, p.B)) &&
              make_feature_map(&m->B_re, p.B_re, 64, p.H, p.T, p.B) &&
              make_feature_map(&m->B_im, p.B_im, 64, p.H, p.T, p.B) &&
              // (no C for the chunk states alone: ssd_complex_final_state)
              (p.C_re == nullptr || (make_feature_map(&m->C_re, p.C_re, 64, p.H, p.T, p.B) &&
                                     make_feature_map(&m->C_im, p.C_im, 64, p.H, p.T, p.B))) &&
              (ws_S == nullptr || make_state_map(&m->S, ws_S, (int64_t)p.B * p.H * p.nc * 2 * 64));
    return ok ? SSDC_OK : SSDC_ERR_CUDA;
}

namespace {

constexpr size_t kStateSmem = sizeof(StateSmem) + 1024;
constexpr size_t kScanSmem = sizeof(ScanSmem) + 1024;
// The chunk-state kernel needs little shared memory; ask for enough that at
// most two CTAs share an SM, matching the two 256-column TMEM allocations.
constexpr size_t kStateSmemLaunch = kStateSmem > 80 * 1024 ? kStateSmem : 80 * 1024;

bool g_attr_set[64] = {};

int set_attrs() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SSDC_ERR_CUDA;
    if (g_attr_set[dev]) return SSDC_OK;
    if (cudaFuncSetAttribute(tc_chunk_state, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStateSmemLaunch) !=
            cudaSuccess ||
        cudaFuncSetAttribute(tc_chunk_scan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScanSmem) !=
            cudaSuccess)
        return SSDC_ERR_CUDA;
    g_attr_set[dev] = true;
    return SSDC_OK;
}

}  // namespace
}  // namespace tc

bool tc_supported(int N, int D, int Q) { return N == 64 && D == 64 && (Q == 32 || Q == 64 || Q == 128 || Q == 256); }

int tc_launch_chunk_state(const Problem& p, const Workspace& ws, cudaStream_t stream) {
    int rc = tc::set_attrs();
    if (rc != SSDC_OK) return rc;
    tc::TcMaps maps;
    rc = tc::make_maps(p, ws.S, &maps);
    if (rc != SSDC_OK) return rc;
    const dim3 grid((unsigned)p.nc, (unsigned)p.H, (unsigned)p.B);
    tc::tc_chunk_state<<<grid, tc::kThreads, tc::kStateSmemLaunch, stream>>>(p, ws, maps);
    return 1;
}

int tc_launch_chunk_scan(const Problem& p, const Workspace& ws, cudaStream_t stream) {
    int rc = tc::set_attrs();
    if (rc != SSDC_OK) return rc;
    tc::TcMaps maps;
    rc = tc::make_maps(p, ws.S, &maps);
    if (rc != SSDC_OK) return rc;
    const dim3 grid((unsigned)(p.nc * ((p.Q + tc::kRows - 1) / tc::kRows)), (unsigned)p.H, (unsigned)p.B);
    tc::tc_chunk_scan<<<grid, tc::kThreads, tc::kScanSmem, stream>>>(p, ws, maps);
    return 1;
}

}  // namespace ssdc
