// Pieces shared by the fused TF32 kernels (ssdc_fused.cu, ssdc_fused2.cu):
// the shared-memory tile layouts of the 64 x 64 complex operands, their
// K-major descriptors and M = 128, N = 128 MMA sequences, the tensor maps that
// stage C, B and x by TMA, and the producer's discretisation and in-chunk
// cumulative sum (page "Extending -- SSM variants & Triton kernels", Path A,
// Step 1, for A_bar = exp(softplus(dt) A); landing page, "03 Chunkwise SSD",
// for the chunked form).
#pragma once

#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "tc_common.cuh"

namespace ssdc {
namespace fused {
namespace {

using namespace tc;

constexpr int kQ = 64;
constexpr uint32_t kTileBytes = 2 * kPlaneBytes;  // 32 KB: one complex 64 x 64 tile
constexpr uint32_t kIntHalf = 16384;              // one 32-column half of a 128-row tile
constexpr uint32_t kIdesc128 = ptx::idesc_tf32(128, 128, 0);  // M = 128, N = 128, B operand K-major

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
// Column pair (n, n + 1), n even and below 32, of row m in 32-column half khalf of an interleaved tile.
__device__ __forceinline__ uint32_t pair_off(int khalf, int m, int n) {
    return inter_row(khalf, m) + chunk16(n >> 2, m) + (uint32_t)((n & 3) << 2);
}

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

// Tensor maps of one launch. The fast maps fetch both planes of a tensor in
// one copy per 32-column half, through a "plane" dimension whose stride is the
// distance between the two planes' allocations; the C map also splits time
// into 8-row groups so that its box lands in the interleaved layout. Where a
// fast map cannot be made (planes not 16-byte spaced or too far apart, T not a
// multiple of 8 for C), the per-plane maps are used.
struct FusedMaps {
    CUtensorMap x_re, x_im, B_re, B_im;  // (F, H, T, B), boxes (32, 1, 64, 1)
    CUtensorMap c8_re, c8_im;            // (F, H, T, B), boxes (32, 1, 8, 1)
    CUtensorMap x2, B2;                  // (F, H, T, plane, B), boxes (32, 1, 64, 2, 1)
    CUtensorMap C2;                      // (F, H, T % 8, plane, (B T) / 8), boxes (32, 1, 8, 2, 8)
    CUtensorMap y_re, y_im;              // output planes (D, H, T, B), boxes (32, 1, 64, 1) (TMA stores)
    int fast;                            // bit 0: x2, bit 1: B2, bit 2: C2 in use
    int swap;                            // bit k: the fast map's plane 0 is the imaginary plane (0 x, 1 B, 2 C)
    int real_x;                          // x has no imaginary plane (x_re only)
    int y_im_out;                        // y_im is written (not with the fused head mixer)
};

// Loader warp: dt of one chunk's tokens (two per lane over a 64-row tile; rows
// past the chunk's `rows` tokens or past T are marked with NaN so that they
// get zero log-decay), and A of its head. The loads are only issued here;
// their values are first used by store_acs.
struct Alog {
    float dt0, dt1, Ar, Ai;
};
__device__ __forceinline__ Alog load_alog(const Problem& p, int b, int h, int64_t t0, int lane, int rows = kQ) {
    Alog a;
    const int64_t ta = t0 + 2 * lane, tb = ta + 1;
    a.dt0 = ta < p.T && 2 * lane < rows ? p.dt[((int64_t)b * p.T + ta) * p.H + h] : __int_as_float(0x7fffffff);
    a.dt1 = tb < p.T && 2 * lane + 1 < rows ? p.dt[((int64_t)b * p.T + tb) * p.H + h] : __int_as_float(0x7fffffff);
    a.Ar = p.A_re[h];
    a.Ai = p.A_im[h];
    return a;
}

// Loader warp: discretisation softplus(dt) * A and its inclusive cumulative
// sum into acs, then arrive on the stage barrier `full` (the tile bytes were
// announced with the loads). The sum is fp32: its rounding (about 1e-7 of
// |Acs|, so about 1e-5 relative on a decay factor) is far below TF32's.
__device__ __forceinline__ void store_acs(float2* acs, uint64_t* full, const Alog& al, int lane) {
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
    acs[2 * lane] = make_float2(er + r0, ei + i0);
    acs[2 * lane + 1] = make_float2(cr, ci);
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(full);
}

// Producer: TMA of one 64-token tile of x (stacked; only the real plane for a
// real x) or of B_t (stacked) into a stage buffer, counted on `bar`. A box of
// `rows` rows of one 32-column half of one plane is rows x 128 bytes; both
// planes come in one box per half where the two-plane map is in use.
__device__ __forceinline__ void load_x(char* dst, const FusedMaps& fm, uint64_t* bar, int h, int t0, int b, int rows,
                                       int lane) {
    if (lane == 0) ptx::mbar_expect_tx(bar, (uint32_t)(rows * 128 * (fm.real_x ? 2 : 4)));
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

__device__ __forceinline__ void load_b(char* dst, const FusedMaps& fm, uint64_t* bar, int h, int t0, int b, int rows,
                                       int lane) {
    if (lane == 0) ptx::mbar_expect_tx(bar, (uint32_t)(rows * 128 * 4));
    __syncwarp();
    if ((fm.fast >> 1) & 1) {
        if (lane < 2) ptx::tma_load_5d(dst + stk_row(lane, 0, 0), &fm.B2, bar, 32 * lane, h, t0, 0, b);
    } else if (lane < 4) {
        const int half = lane >> 1, pl = lane & 1;
        ptx::tma_load_4d(dst + stk_row(half, pl, 0), pl ? &fm.B_im : &fm.B_re, bar, 32 * half, h, t0, b);
    }
}


constexpr int kMaxChunkQ = 256;  // the largest chunk

// Producer: the cumulative log-decay of a chunk of Q = 128 or 256 tokens (Q / 32
// consecutive tokens per lane, a warp scan of the lane sums), tokens past T with
// zero log-decay. The sum is fp32: its rounding (about 1e-7 of |Acs|, so about
// 1e-5 relative on a decay factor) is far below TF32's. (Chunks of up to 64
// tokens take load_alog and store_acs, two tokens a lane, which also give the
// rows of a tile past Q zero log-decay.)
__device__ __forceinline__ void chunk_acs(const Problem& p, int b, int h, int64_t t0, int Q, int lane, float2* acs) {
    const int per = Q / 32;
    const float Ar = p.A_re[h], Ai = p.A_im[h];
    float lr[kMaxChunkQ / 32], li[kMaxChunkQ / 32];
    float sr = 0.0f, si = 0.0f;
#pragma unroll
    for (int k = 0; k < kMaxChunkQ / 32; ++k) {
        const int64_t tok = t0 + lane * per + k;
        float ar = 0.0f, ai = 0.0f;
        if (k < per && tok < p.T) {
            const float sp = softplus_f(p.dt[((int64_t)b * p.T + tok) * p.H + h]);
            ar = sp * Ar;
            ai = sp * Ai;
        }
        sr += ar;
        si += ai;
        lr[k] = sr;
        li[k] = si;
    }
    float cr = sr, ci = si;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float ur = __shfl_up_sync(0xffffffffu, cr, off);
        const float ui = __shfl_up_sync(0xffffffffu, ci, off);
        if (lane >= off) {
            cr += ur;
            ci += ui;
        }
    }
    const float er = cr - sr, ei = ci - si;  // exclusive prefix of this lane's tokens
#pragma unroll
    for (int k = 0; k < kMaxChunkQ / 32; ++k)
        if (k < per) acs[lane * per + k] = make_float2(er + lr[k], ei + li[k]);
}

// Plane pair (re, im) as one map dimension: base = the lower address, stride =
// the distance, swap = the imaginary plane comes first.
bool plane_pair(const float* re, const float* im, const float** base, cuuint64_t* stride, bool* swap) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(re), b = reinterpret_cast<uintptr_t>(im);
    if (a == b) return false;
    *swap = b < a;
    *base = reinterpret_cast<const float*>(b < a ? b : a);
    const uint64_t d = b < a ? a - b : b - a;
    if (d % 16 != 0 || d >= (uint64_t(1) << 40)) return false;
    *stride = d;
    return true;
}

// Both planes of an (F, H, T, B) tensor, boxes (32, 1, 64, 2, 1): the stacked
// layout (Q = 64). Feature columns past F (F < 64) are read as zeros.
bool make_pair_map(CUtensorMap* m, const float* re, const float* im, int F, const Problem& p, bool* swap) {
    const float* base;
    cuuint64_t ps;
    if (!plane_pair(re, im, &base, &ps, swap)) return false;
    const cuuint64_t row = (cuuint64_t)F * 4;
    const cuuint64_t dims[5] = {(cuuint64_t)F, (cuuint64_t)p.H, (cuuint64_t)p.T, 2, (cuuint64_t)p.B};
    const cuuint64_t strides[4] = {row, row * p.H, ps, row * p.H * (cuuint64_t)p.T};
    const cuuint32_t box[5] = {32, 1, (cuuint32_t)(p.Q < kQ ? p.Q : kQ), 2, 1};
    return tc::encode_tiled_f32(m, base, 5, dims, strides, box);
}

// Both planes of C, time split into 8-row groups (T a multiple of 8, so that
// batch and group merge into one dimension), boxes (32, 1, 8, 2, rows / 8), rows
// = min(Q, 64): the interleaved layout, row 16g + 8p + i.
bool make_interleaved_map(CUtensorMap* m, const Problem& p, bool* swap) {
    if (p.T % 8 != 0 || p.Q % 8 != 0 || (int64_t)p.B * p.T / 8 >= (int64_t(1) << 31)) return false;
    const float* base;
    cuuint64_t ps;
    if (!plane_pair(p.C_re, p.C_im, &base, &ps, swap)) return false;
    const cuuint64_t row = (cuuint64_t)p.N * 4;
    const cuuint64_t dims[5] = {(cuuint64_t)p.N, (cuuint64_t)p.H, 8, 2, (cuuint64_t)p.B * (cuuint64_t)p.T / 8};
    const cuuint64_t strides[4] = {row, row * p.H, ps, 8 * row * p.H};
    const cuuint32_t box[5] = {32, 1, 8, 2, (cuuint32_t)((p.Q < kQ ? p.Q : kQ) / 8)};
    return tc::encode_tiled_f32(m, base, 5, dims, strides, box);
}

int make_fused_maps(const Problem& p, bool allow_fast, FusedMaps* fm) {
    memset(fm, 0, sizeof(*fm));
    fm->real_x = p.x_im == nullptr;
    if (p.in_bf16) {
        // bfloat16 x, B_t, C_t: one map per plane, boxes of 64 features (one 128-byte row);
        // C in 8-row boxes that land in the interleaved layout
        const int rows16 = p.Q < kQ ? p.Q : kQ;
        bool ok = tc::encode_feature_map_bf16(&fm->x_re, p.x_re, p.D, p.H, p.T, p.B, rows16) &&
                  (fm->real_x || tc::encode_feature_map_bf16(&fm->x_im, p.x_im, p.D, p.H, p.T, p.B, rows16)) &&
                  tc::encode_feature_map_bf16(&fm->B_re, p.B_re, p.N, p.H, p.T, p.B, rows16) &&
                  tc::encode_feature_map_bf16(&fm->B_im, p.B_im, p.N, p.H, p.T, p.B, rows16) &&
                  tc::encode_feature_map_bf16(&fm->c8_re, p.C_re, p.N, p.H, p.T, p.B, 8) &&
                  tc::encode_feature_map_bf16(&fm->c8_im, p.C_im, p.N, p.H, p.T, p.B, 8) &&
                  tc::encode_feature_map(&fm->y_re, p.y_re, p.D, p.H, p.T, p.B, rows16) &&
                  (p.y_im == nullptr || tc::encode_feature_map(&fm->y_im, p.y_im, p.D, p.H, p.T, p.B, rows16));
        fm->y_im_out = p.y_im != nullptr;
        return ok ? SSDC_OK : SSDC_ERR_CUDA;
    }
    bool sw = false;
    // Tiles are 64 rows: a chunk of Q >= 64 tokens is Q / 64 tiles, a smaller chunk fills the
    // first Q rows of one. A two-plane box puts its second plane right after its rows: it lands
    // in the stacked layout (planes 64 rows apart) only for 64-row boxes; smaller chunks take one
    // map per plane.
    const int rows = p.Q < kQ ? p.Q : kQ;
    const bool pair_ok = allow_fast && rows == kQ;
    if (pair_ok && !fm->real_x && make_pair_map(&fm->x2, p.x_re, p.x_im, p.D, p, &sw))
        fm->fast |= 1, fm->swap |= sw ? 1 : 0;
    if (pair_ok && make_pair_map(&fm->B2, p.B_re, p.B_im, p.N, p, &sw)) fm->fast |= 2, fm->swap |= sw ? 2 : 0;
    if (allow_fast && make_interleaved_map(&fm->C2, p, &sw)) fm->fast |= 4, fm->swap |= sw ? 4 : 0;
    bool ok = true;
    if (!(fm->fast & 1))
        ok = ok && tc::encode_feature_map(&fm->x_re, p.x_re, p.D, p.H, p.T, p.B, rows) &&
             (fm->real_x || tc::encode_feature_map(&fm->x_im, p.x_im, p.D, p.H, p.T, p.B, rows));
    if (!(fm->fast & 2))
        ok = ok && tc::encode_feature_map(&fm->B_re, p.B_re, p.N, p.H, p.T, p.B, rows) &&
             tc::encode_feature_map(&fm->B_im, p.B_im, p.N, p.H, p.T, p.B, rows);
    if (!(fm->fast & 4))
        ok = ok && tc::encode_feature_map(&fm->c8_re, p.C_re, p.N, p.H, p.T, p.B, 8) &&
             tc::encode_feature_map(&fm->c8_im, p.C_im, p.N, p.H, p.T, p.B, 8);
    ok = ok && tc::encode_feature_map(&fm->y_re, p.y_re, p.D, p.H, p.T, p.B, rows) &&
         (p.y_im == nullptr || tc::encode_feature_map(&fm->y_im, p.y_im, p.D, p.H, p.T, p.B, rows));
    fm->y_im_out = p.y_im != nullptr;
    return ok ? SSDC_OK : SSDC_ERR_CUDA;
}

// The launch's tensor maps, encoded once per pointer set and size (a small
// cache: per-call host work stays off the launch path).
struct MapKey {
    const void* ptr[8];
    int64_t T;
    int B, H, N, D, Q;
    bool fast, bf16;
};
struct MapEntry {
    MapKey key;
    FusedMaps maps;
};
constexpr int kMapSlots = 16;
std::mutex g_map_mu;
MapEntry g_map_cache[kMapSlots];
int g_map_used = 0, g_map_next = 0;

bool same_map_key(const MapKey& a, const MapKey& b) {
    for (int i = 0; i < 8; ++i)
        if (a.ptr[i] != b.ptr[i]) return false;
    return a.T == b.T && a.B == b.B && a.H == b.H && a.N == b.N && a.D == b.D && a.Q == b.Q && a.fast == b.fast &&
           a.bf16 == b.bf16;
}

int cached_maps(const Problem& p, bool allow_fast, FusedMaps* fm) {
    MapKey k;
    memset(&k, 0, sizeof(k));
    const void* ptrs[8] = {p.x_re, p.x_im, p.B_re, p.B_im, p.C_re, p.C_im, p.y_re, p.y_im};
    for (int i = 0; i < 8; ++i) k.ptr[i] = ptrs[i];
    k.T = p.T;
    k.B = p.B;
    k.H = p.H;
    k.N = p.N;
    k.D = p.D;
    k.Q = p.Q;
    k.fast = allow_fast;
    k.bf16 = p.in_bf16 != 0;
    {
        std::lock_guard<std::mutex> g(g_map_mu);
        for (int i = 0; i < g_map_used; ++i)
            if (same_map_key(g_map_cache[i].key, k)) {
                *fm = g_map_cache[i].maps;
                return SSDC_OK;
            }
    }
    const int rc = make_fused_maps(p, allow_fast, fm);
    if (rc != SSDC_OK) return rc;
    std::lock_guard<std::mutex> g(g_map_mu);
    MapEntry& e = g_map_cache[g_map_next];
    e.key = k;
    e.maps = *fm;
    g_map_next = (g_map_next + 1) % kMapSlots;
    if (g_map_used < kMapSlots) ++g_map_used;
    return SSDC_OK;
}

}  // namespace
}  // namespace fused
}  // namespace ssdc
