// The two steps that join scan segments of one sequence (landing page, "03
// Chunkwise SSD": the STATE line, chunk states passed with the exponential of
// the accumulated decay; applied here to whole segments of the sequence):
//
//   ssd_complex_segment_decay   a_seg[b,h] = exp(sum_t softplus(dt[b,t,h]) A[h]),
//                               the total decay of a segment, the product of its
//                               A_bar_t (page "Extending -- SSM variants & Triton
//                               kernels", Path A, Step 1, for A_bar)
//   ssd_complex_state_combine   s_out = a s_in + s_add per (b, h): the state after
//                               two consecutive segments, from the first's
//                               incoming state and the second's decay and end
//                               state computed from zero
//
// With these a sequence split over ranks (or calls) in time is scanned from
// each segment's true incoming state: (a2, S2) o (a1, S1) = (a2 a1, a2 S1 + S2).
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/ssdc.h"
#include "ssdc_kernels.h"

namespace ssdc {
namespace {

constexpr int kDecayThreads = 256;  // 8 warps, one (b, h) per warp

// The sum of softplus(dt) over a segment in fp64 (T terms), then the complex
// exponential of sum * A in fp64.
__global__ void __launch_bounds__(kDecayThreads) segment_decay_kernel(const float* __restrict__ dt,
                                                                      const float* __restrict__ A_re,
                                                                      const float* __restrict__ A_im, int64_t B,
                                                                      int64_t T, int64_t H, float* out_re,
                                                                      float* out_im) {
    const int lane = threadIdx.x & 31;
    const int64_t q = (int64_t)blockIdx.x * (kDecayThreads / 32) + (threadIdx.x >> 5);
    if (q >= B * H) return;
    const int64_t b = q / H, h = q - b * H;
    double sum = 0.0;
    for (int64_t t = lane; t < T; t += 32) {
        const float v = dt[(b * T + t) * H + h];
        sum += (double)fmaxf(v, 0.0f) + log1p(exp(-(double)fabsf(v)));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) {
        const double zr = sum * (double)A_re[h], zi = sum * (double)A_im[h];
        const double m = exp(zr);
        double s, c;
        sincos(zi, &s, &c);
        out_re[q] = (float)(m * c);
        out_im[q] = (float)(m * s);
    }
}

__global__ void state_combine_kernel(const float* __restrict__ a_re, const float* __restrict__ a_im,
                                     const float* s_in_re, const float* s_in_im, const float* s_add_re,
                                     const float* s_add_im, int64_t nseq, int64_t per_seq, float* out_re,
                                     float* out_im) {
    const int64_t n = nseq * per_seq;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t q = i / per_seq;
        const float ar = a_re[q], ai = a_im[q];
        const float sr = s_in_re ? s_in_re[i] : 0.0f, si = s_in_im ? s_in_im[i] : 0.0f;
        out_re[i] = ar * sr - ai * si + s_add_re[i];
        out_im[i] = ar * si + ai * sr + s_add_im[i];
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ssdc

extern "C" {

int ssd_complex_segment_decay(ssdc_cin A, const float* dt, ssdc_dims dims, ssdc_cout a_seg, cudaStream_t stream) {
    if (dims.B <= 0 || dims.T <= 0 || dims.H <= 0 || dims.B * dims.H > (int64_t(1) << 31)) return SSDC_ERR_INVALID;
    const void* ptrs[] = {A.re, A.im, dt, a_seg.re, a_seg.im};
    for (const void* p : ptrs)
        if (p == nullptr) return SSDC_ERR_INVALID;
    for (const void* p : ptrs)
        if (!ssdc::aligned16(p)) return SSDC_ERR_ALIGN;
    (void)cudaGetLastError();
    const int64_t nseq = dims.B * dims.H;
    const int64_t blocks = (nseq + ssdc::kDecayThreads / 32 - 1) / (ssdc::kDecayThreads / 32);
    ssdc::segment_decay_kernel<<<(unsigned)blocks, ssdc::kDecayThreads, 0, stream>>>(
        dt, A.re, A.im, dims.B, dims.T, dims.H, a_seg.re, a_seg.im);
    if (cudaGetLastError() != cudaSuccess) return SSDC_ERR_CUDA;
    ssdc::set_last_launch_count(1);
    return SSDC_OK;
}

int ssd_complex_state_combine(ssdc_cin a, ssdc_cin s_in, ssdc_cin s_add, ssdc_dims dims, ssdc_cout s_out,
                              cudaStream_t stream) {
    if (dims.B <= 0 || dims.H <= 0 || dims.N <= 0 || dims.D <= 0) return SSDC_ERR_INVALID;
    const void* req[] = {a.re, a.im, s_add.re, s_add.im, s_out.re, s_out.im};
    for (const void* p : req)
        if (p == nullptr) return SSDC_ERR_INVALID;
    if ((s_in.re == nullptr) != (s_in.im == nullptr)) return SSDC_ERR_INVALID;
    const void* all[] = {a.re, a.im, s_add.re, s_add.im, s_out.re, s_out.im, s_in.re, s_in.im};
    for (const void* p : all)
        if (!ssdc::aligned16(p)) return SSDC_ERR_ALIGN;
    (void)cudaGetLastError();
    const int64_t nseq = dims.B * dims.H, per = dims.N * dims.D;
    const int64_t n = nseq * per;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    ssdc::state_combine_kernel<<<(unsigned)blocks, 256, 0, stream>>>(a.re, a.im, s_in.re, s_in.im, s_add.re,
                                                                      s_add.im, nseq, per, s_out.re, s_out.im);
    if (cudaGetLastError() != cudaSuccess) return SSDC_ERR_CUDA;
    ssdc::set_last_launch_count(1);
    return SSDC_OK;
}

}  // extern "C"
