// Shared-memory operand tiles of the exact fp32 SIMT kernels (forward chunk
// kernels and backward kernels): 64 token rows of up to 64 complex values,
// filled from the planar (B, T, H, F) arrays or from a per-chunk state slot,
// and the complex multiply-add forms the micro-kernels use.
#pragma once

#include <cuda_runtime.h>

#include "ssdc_common.cuh"
#include "ssdc_kernels.h"

namespace ssdc {

constexpr int kRows = 64;  // token rows per shared-memory block
constexpr int kCols = 64;  // max N, D

// A tile of 64 rows x up to 64 complex values, real and imaginary parts
// interleaved so that one 64-bit shared load fetches a value. Rows are 65
// values long: 16 lanes reading one column of 16 different rows then touch
// all 32 banks once.
struct CTile {
    float2 v[kRows][kCols + 1];
};

// acc += a * b, acc += a * conj(b), acc += conj(a) * b (complex, fp32 FMAs)
__device__ __forceinline__ void cmac(float2& acc, float2 a, float2 b) {
    acc.x = fmaf(a.x, b.x, fmaf(-a.y, b.y, acc.x));
    acc.y = fmaf(a.x, b.y, fmaf(a.y, b.x, acc.y));
}
__device__ __forceinline__ void cmac_cb(float2& acc, float2 a, float2 b) {
    acc.x = fmaf(a.x, b.x, fmaf(a.y, b.y, acc.x));
    acc.y = fmaf(a.y, b.x, fmaf(-a.x, b.y, acc.y));
}
__device__ __forceinline__ void cmac_ca(float2& acc, float2 a, float2 b) {
    acc.x = fmaf(a.x, b.x, fmaf(a.y, b.y, acc.x));
    acc.y = fmaf(a.x, b.y, fmaf(-a.y, b.x, acc.y));
}
__device__ __forceinline__ float2 conjf2(float2 a) { return make_float2(a.x, -a.y); }

__device__ __forceinline__ int chunk_valid(const Problem& p, int64_t t0) {
    return (int)(p.T - t0 < (int64_t)p.Q ? p.T - t0 : (int64_t)p.Q);
}

// Rows [r0, r0 + 64) of one chunk of a (B, T, H, F) plane pair into dst,
// zero past the chunk's valid tokens (`valid`) and past F. F is a multiple
// of 8 and the planes are 16-byte aligned, so every row is read as float4s.
// im may be null (a zero imaginary plane).
template <int NT = 256>
__device__ __forceinline__ void load_rows(CTile& dst, const float* __restrict__ re,
                                          const float* __restrict__ im, int64_t bt0, int H, int h,
                                          int F, int r0, int valid) {
    constexpr int kQuads = kRows * kCols / 4;  // float4 groups of the tile
#pragma unroll
    for (int it = 0; it < kQuads / NT; ++it) {
        const int e = threadIdx.x + it * NT;
        const int r = e / (kCols / 4), f = 4 * (e % (kCols / 4));
        float4 vr = make_float4(0.0f, 0.0f, 0.0f, 0.0f), vi = vr;
        if (r0 + r < valid && f < F) {
            const int64_t o = ((bt0 + r0 + r) * H + h) * (int64_t)F + f;
            vr = __ldg(reinterpret_cast<const float4*>(re + o));
            if (im != nullptr) vi = __ldg(reinterpret_cast<const float4*>(im + o));
        }
        dst.v[r][f] = make_float2(vr.x, vi.x);
        dst.v[r][f + 1] = make_float2(vr.y, vi.y);
        dst.v[r][f + 2] = make_float2(vr.z, vi.z);
        dst.v[r][f + 3] = make_float2(vr.w, vi.w);
    }
}

// A per-chunk (D, N) state slot [2][D][N], fetched into registers (this
// thread's share) and later stored into a tile as dst[d][n].
template <int NT>
struct StateRegs {
    float4 re[kRows * kCols / 4 / NT], im[kRows * kCols / 4 / NT];
};

template <int NT>
__device__ __forceinline__ void fetch_state(StateRegs<NT>& q, const float* __restrict__ slot, int D, int N) {
    const float* si = slot + (int64_t)D * N;
#pragma unroll
    for (int it = 0; it < kRows * kCols / 4 / NT; ++it) {
        const int e = threadIdx.x + it * NT;
        const int d = e / (kCols / 4), n = 4 * (e % (kCols / 4));
        q.re[it] = q.im[it] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (d < D && n < N) {
            q.re[it] = __ldcg(reinterpret_cast<const float4*>(slot + d * N + n));
            q.im[it] = __ldcg(reinterpret_cast<const float4*>(si + d * N + n));
        }
    }
}

template <int NT>
__device__ __forceinline__ void store_state(CTile& dst, const StateRegs<NT>& q) {
#pragma unroll
    for (int it = 0; it < kRows * kCols / 4 / NT; ++it) {
        const int e = threadIdx.x + it * NT;
        const int d = e / (kCols / 4), n = 4 * (e % (kCols / 4));
        dst.v[d][n] = make_float2(q.re[it].x, q.im[it].x);
        dst.v[d][n + 1] = make_float2(q.re[it].y, q.im[it].y);
        dst.v[d][n + 2] = make_float2(q.re[it].z, q.im[it].z);
        dst.v[d][n + 3] = make_float2(q.re[it].w, q.im[it].w);
    }
}

// A per-chunk (D, N) state slot [2][D][N] into dst as dst[d][n].
template <int NT = 256>
__device__ __forceinline__ void load_state(CTile& dst, const float* __restrict__ slot, int D, int N) {
    constexpr int kQuads = kRows * kCols / 4;
    const float* si = slot + (int64_t)D * N;
#pragma unroll
    for (int it = 0; it < kQuads / NT; ++it) {
        const int e = threadIdx.x + it * NT;
        const int d = e / (kCols / 4), n = 4 * (e % (kCols / 4));
        float4 vr = make_float4(0.0f, 0.0f, 0.0f, 0.0f), vi = vr;
        if (d < D && n < N) {
            vr = __ldcg(reinterpret_cast<const float4*>(slot + d * N + n));
            vi = __ldcg(reinterpret_cast<const float4*>(si + d * N + n));
        }
        dst.v[d][n] = make_float2(vr.x, vi.x);
        dst.v[d][n + 1] = make_float2(vr.y, vi.y);
        dst.v[d][n + 2] = make_float2(vr.z, vi.z);
        dst.v[d][n + 3] = make_float2(vr.w, vi.w);
    }
}

}  // namespace ssdc
