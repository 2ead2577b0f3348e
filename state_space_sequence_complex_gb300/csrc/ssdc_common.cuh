// Device helpers shared by the kernels of libssdc: discretisation, in-chunk
// cumulative log-decay and accurate differences of it.
//
// Discretisation (page "Extending -- SSM variants & Triton kernels", Path A,
// Step 1: A_bar = exp(softplus(dt) * A)): the per-token complex log-decay is
//   alog[t] = softplus(dt[t]) * A,   softplus(v) = log(1 + e^v).
// Chunked form (landing page, "03 Chunkwise SSD"): Acs is the inclusive
// cumulative sum of alog inside a chunk and every decay factor is
// exp(Acs[l] - Acs[s]) for l >= s, never exp(Acs[l]) * exp(-Acs[s]).
//
// Precision. |Re Acs| reaches several hundred inside a 256-token chunk, so a
// plain fp32 cumulative sum would put an absolute error of ~1e-5 into every
// difference. The sum is accumulated in fp64 (Q additions per chunk) and kept
// as an unevaluated pair hi + lo of floats; a difference is then
// (hi_l - hi_s) + (lo_l - lo_s), accurate to about one fp32 ulp of the
// difference itself.
#pragma once

#include <cstdint>

#include "../../include/ssdc.h"

namespace ssdc {

constexpr int kMaxQ = 256;

// One token's cumulative log-decay, as two float pairs.
struct Acs {
    float re_hi, re_lo, im_hi, im_lo;
};

__device__ __forceinline__ float softplus_f(float v) {
    return fmaxf(v, 0.0f) + log1pf(expf(-fabsf(v)));
}

__device__ __forceinline__ float2 acs_diff(const Acs& a, const Acs& b) {
    return make_float2((a.re_hi - b.re_hi) + (a.re_lo - b.re_lo),
                       (a.im_hi - b.im_hi) + (a.im_lo - b.im_lo));
}

__device__ __forceinline__ float2 acs_value(const Acs& a) {
    return make_float2(a.re_hi + a.re_lo, a.im_hi + a.im_lo);
}

// exp(z) for complex z, with the library's accurate expf / sincosf.
__device__ __forceinline__ float2 cexp_exact(float2 z) {
    float s, c;
    sincosf(z.y, &s, &c);
    const float m = expf(z.x);
    return make_float2(m * c, m * s);
}

// exp(z) with the hardware approximations. The angle is first reduced to
// [-pi, pi] by Cody and Waite's method (2*pi split into a float head and the
// float nearest to the remainder), where the MUFU sine and cosine are
// accurate to a few 1e-7 absolute.
__device__ __forceinline__ float2 cexp_fast(float2 z) {
    constexpr float kInv2Pi = 0.159154943091895336f;
    constexpr float k2PiHi = 6.28318548202514648f;     // float(2*pi)
    constexpr float k2PiLo = -1.74845553146951715e-7f;  // 2*pi - float(2*pi)
    const float k = rintf(z.y * kInv2Pi);
    float r = fmaf(-k, k2PiHi, z.y);
    r = fmaf(-k, k2PiLo, r);
    float s, c;
    __sincosf(r, &s, &c);
    const float m = __expf(z.x);
    return make_float2(m * c, m * s);
}

__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}

// In-chunk inclusive cumulative sum of alog, computed by ONE warp.
//   dt_chunk  dt of the chunk's first token for this (b, h); token l at
//             dt_chunk[l * dt_stride]
//   nvalid    tokens of the chunk inside the sequence (<= Q); tokens past it
//             get alog = 0 (identity decay), so a partial last chunk carries
//             the state after its last real token.
// Writes acs[0..Q) and returns (to lane 0..31) nothing; caller syncs.
__device__ __forceinline__ void chunk_cumsum_warp(const float* __restrict__ dt_chunk,
                                                  int64_t dt_stride, int nvalid, int Q,
                                                  float A_re, float A_im, Acs* acs) {
    const int lane = threadIdx.x & 31;
    const int per = (Q + 31) / 32;  // tokens per lane, consecutive
    const int l0 = lane * per;
    double sr = 0.0, si = 0.0;
    double loc_r[kMaxQ / 32], loc_i[kMaxQ / 32];
#pragma unroll
    for (int j = 0; j < kMaxQ / 32; ++j) {
        const int l = l0 + j;
        float ar = 0.0f, ai = 0.0f;
        if (j < per && l < Q && l < nvalid) {
            const float sp = softplus_f(__ldg(dt_chunk + (int64_t)l * dt_stride));
            ar = sp * A_re;
            ai = sp * A_im;
        }
        sr += (double)ar;
        si += (double)ai;
        loc_r[j] = sr;
        loc_i[j] = si;
    }
    // exclusive scan of the lane totals
    double incl_r = sr, incl_i = si;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const double ur = __shfl_up_sync(0xffffffffu, incl_r, off);
        const double ui = __shfl_up_sync(0xffffffffu, incl_i, off);
        if (lane >= off) {
            incl_r += ur;
            incl_i += ui;
        }
    }
    const double base_r = incl_r - sr, base_i = incl_i - si;
#pragma unroll
    for (int j = 0; j < kMaxQ / 32; ++j) {
        const int l = l0 + j;
        if (j < per && l < Q) {
            const double vr = base_r + loc_r[j], vi = base_i + loc_i[j];
            Acs a;
            a.re_hi = (float)vr;
            a.re_lo = (float)(vr - (double)a.re_hi);
            a.im_hi = (float)vi;
            a.im_lo = (float)(vi - (double)a.im_hi);
            acs[l] = a;
        }
    }
}

// Workspace layout shared by all kernels of one call.
//   S      [B*H*nc][2][D][N] floats: per chunk the transposed state S^T
//          (d rows, n contiguous), real plane then imaginary plane. The
//          chunk-state kernels write S_loc here; the state pass replaces it
//          in place by S_in (the state entering the chunk).
//   a      [B*H*nc][2] floats: exp(Acs[Q-1]) of each chunk.
//   status one int32: SSDC_OK or a device-detected error.
struct Workspace {
    float* S;
    float* a;
    int* status;
};

__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace ssdc
