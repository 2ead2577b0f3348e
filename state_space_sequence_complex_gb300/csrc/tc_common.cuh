// Helpers shared by the tcgen05 kernels: swizzled 64 x 64 fp32 planes staged
// by TMA, K-major shared-memory descriptors, TMEM row loads/stores and the
// pair of M=128 MMAs that multiplies an interleaved complex window by a
// planar complex operand.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ssdc_common.cuh"
#include "ssdc_kernels.h"

namespace ssdc {
namespace tc {

constexpr int kRows = 64;                      // tokens per block (l or s)
constexpr uint32_t kPlaneBytes = 64 * 64 * 4;  // one 64 x 64 fp32 plane: two 8 KB swizzle halves
constexpr uint32_t kHalfBytes = kPlaneBytes / 2;
constexpr uint64_t kWaitIters = 2000000000ull;  // wait limit: 2 s of wall time
constexpr uint32_t kIdesc = ptx::idesc_tf32(128, 64, 0);  // M = 128, N = 64, B operand K-major

// Byte offset of element (r, c) inside a 64 x 64 fp32 plane staged by TMA as
// two boxes of 64 rows x 32 floats with the 128-byte swizzle (the 16-byte
// chunk index is XORed with row % 8).
__device__ __forceinline__ uint32_t plane_off(int r, int c) {
    const int half = c >> 5, cc = c & 31;
    return (uint32_t)(half * kHalfBytes + r * 128 + ((((cc >> 2) ^ (r & 7)) << 4) | ((cc & 3) << 2)));
}

__device__ __forceinline__ float plane_ld(const float* plane, int r, int c) {
    return *reinterpret_cast<const float*>(reinterpret_cast<const char*>(plane) + plane_off(r, c));
}

__device__ __forceinline__ void plane_st(float* plane, int r, int c, float v) {
    *reinterpret_cast<float*>(reinterpret_cast<char*>(plane) + plane_off(r, c)) = v;
}

// 16-byte chunk j (columns 4j .. 4j+3 of the 32-column half `half`) of row r.
__device__ __forceinline__ float4 plane_ld4(const float* plane, int r, int half, int j) {
    return *reinterpret_cast<const float4*>(reinterpret_cast<const char*>(plane) + half * kHalfBytes + r * 128 +
                                            ((j ^ (r & 7)) << 4));
}

// B operand "K-major": the plane's rows are the MMA's N index, its columns
// the K index (B[n][k]); K-step k covers columns 8k .. 8k+7.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t plane_saddr, int k) {
    const uint32_t start = plane_saddr + (uint32_t)(k >> 2) * kHalfBytes + (uint32_t)(k & 3) * 32u;
    return ptx::smem_desc_sw128(start, 16u, 1024u);
}

// Transpose the two planes of a staged 64 x 64 tile (rows r, columns c) into
// the same swizzled layout with rows and columns exchanged, so that a tile
// whose rows are the contraction index becomes a K-major MMA operand (the
// TF32 MMA takes K-major operands only). Each thread moves 4 x 4 blocks with
// 16-byte loads and stores; the caller synchronises and fences for the MMA.
template <int kNT>
__device__ __forceinline__ void transpose_tile(const float* src, float* dst, int t) {
    for (int blk = t; blk < 2 * 256; blk += kNT) {
        const int plane = blk >> 8, rb = (blk >> 4) & 15, cb = blk & 15;
        const char* sp = reinterpret_cast<const char*>(src) + plane * kPlaneBytes + (cb >> 3) * kHalfBytes;
        char* dp = reinterpret_cast<char*>(dst) + plane * kPlaneBytes + (rb >> 3) * kHalfBytes;
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 4 * rb + i;
            v[i] = *reinterpret_cast<const float4*>(sp + r * 128 + (((cb & 7) ^ (r & 7)) << 4));
        }
        using ptx::to_tf32;  // the tile is an MMA operand: rounded to nearest TF32
        const float4 o[4] = {make_float4(to_tf32(v[0].x), to_tf32(v[1].x), to_tf32(v[2].x), to_tf32(v[3].x)),
                             make_float4(to_tf32(v[0].y), to_tf32(v[1].y), to_tf32(v[2].y), to_tf32(v[3].y)),
                             make_float4(to_tf32(v[0].z), to_tf32(v[1].z), to_tf32(v[2].z), to_tf32(v[3].z)),
                             make_float4(to_tf32(v[0].w), to_tf32(v[1].w), to_tf32(v[2].w), to_tf32(v[3].w))};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = 4 * cb + j;
            *reinterpret_cast<float4*>(dp + r * 128 + (((rb & 7) ^ (r & 7)) << 4)) = o[j];
        }
    }
}

// TMEM address of this warp's 32-lane quadrant (warp w accesses lanes 32 (w % 4) ..).
__device__ __forceinline__ uint32_t lane_base(uint32_t tmem, int warp) {
    return tmem + (((uint32_t)(warp & 3) * 32u) << 16);
}

// Record a wait that gave up. The status word is cleared on the stream before a
// call's first launch; the first error recorded sticks.
__device__ __forceinline__ void fail(int* status) { atomicCAS(status, SSDC_OK, SSDC_ERR_TIMEOUT); }

// Store an MMA A window: every value rounded to nearest TF32 first.
template <int kCols>
__device__ __forceinline__ void tmem_store(uint32_t taddr, const float* v) {
#pragma unroll
    for (int q = 0; q < kCols / 16; ++q) {
        float r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = ptx::to_tf32(v[16 * q + i]);
        ptx::tmem_st16(taddr + 16 * q, r);
    }
}

template <int kCols>
__device__ __forceinline__ void tmem_load(uint32_t taddr, float* v) {
#pragma unroll
    for (int q = 0; q < kCols / 16; ++q) ptx::tmem_ld16(taddr + 16 * q, v + 16 * q);
    ptx::tmem_wait_ld();
}

// Issue D (+)= W1 * B1 + W2 * B2 over K = 64 (8 MMAs of K = 8 each); W1, W2
// are 64-column TMEM windows, B1, B2 K-major 64 x 64 planes in shared memory.
__device__ __forceinline__ void issue_pair(uint32_t d, uint32_t w1, uint32_t w2, uint32_t b1, uint32_t b2,
                                           bool accumulate) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
        ptx::mma_tf32_ts(d, w1 + 8 * k, desc_kmajor(b1, k), kIdesc, (accumulate || k > 0) ? 1u : 0u);
#pragma unroll
    for (int k = 0; k < 8; ++k) ptx::mma_tf32_ts(d, w2 + 8 * k, desc_kmajor(b2, k), kIdesc, 1u);
}

// Tensor maps of one call: the six input planes of x, B_t, C_t as (F, H, T, B)
// boxes of (32, 1, 64, 1), and the workspace states as rows of 64 floats.
struct TcMaps {
    CUtensorMap x_re, x_im, B_re, B_im, C_re, C_im, S;
};

// Host: encode the maps (returns SSDC_OK or SSDC_ERR_CUDA).
int make_maps(const Problem& p, const float* ws_S, TcMaps* m);
// Host: one (F, H, T, B) fp32 plane with boxes of (32, 1, rows, 1).
bool encode_feature_map(CUtensorMap* m, const float* base, int F, int H, int64_t T, int B, int rows);
// Host: one (F, H, T, B) bfloat16 plane with boxes of (64, 1, rows, 1).
bool encode_feature_map_bf16(CUtensorMap* m, const void* base, int F, int H, int64_t T, int B, int rows);
// Host: an fp32 map of any rank (up to 5) with 128-byte swizzle and zero fill;
// strides[i] is the byte stride of dimension i + 1.
bool encode_tiled_f32(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                      const cuuint32_t* box);

}  // namespace tc
}  // namespace ssdc
