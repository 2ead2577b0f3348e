// MIMO head mixer on the scan's Re(y) (landing page, "02 MIMO Mixer": a fully
// connected H x H mixer across the SSM heads, applied to the Re(y) the block
// consumes), in place over the (B, T, H, D) output:
//
//   out[n, g, d] = sum_h W[g, h] Re(y)[n, h, d]   for every token n = (b, t).
//
// HBM-bound: every element is read once and written once (8 bytes an element,
// 8 H D bytes a token). One thread owns one 8-byte column (two features d) of
// one token: it loads that column from all H heads into registers, then writes
// the H mixed columns back over them. No other thread touches the column, so
// the update in place needs no synchronisation. A warp covers 32 consecutive
// columns: 256 consecutive bytes of each head's row. W sits in shared
// memory (zero past H) and is read as a broadcast. fp32 throughout; the sum runs
// over h in increasing order.
#include <cuda_runtime.h>

#include "ssdc_kernels.h"

namespace ssdc {

namespace {

constexpr int kMixThreads = 256;
constexpr int kMixMaxH = 16;

__global__ void __launch_bounds__(kMixThreads)
ssdc_head_mix(float* y, const float* __restrict__ w, int64_t ntok, int H, int D2) {
    __shared__ float sw[kMixMaxH * kMixMaxH];
    for (int i = threadIdx.x; i < kMixMaxH * kMixMaxH; i += kMixThreads) {
        const int g = i / kMixMaxH, h = i % kMixMaxH;
        sw[i] = (g < H && h < H) ? w[g * H + h] : 0.0f;
    }
    // launched as a programmatic dependent of the scan that writes y: W (written, if at all,
    // before the scan started) is fetched above while the scan finishes; y only after it has
    grid_dependency_wait();
    __syncthreads();
    // one column a thread (a grid-stride loop would let the compiler hold all of W in registers)
    const int64_t i = (int64_t)blockIdx.x * kMixThreads + threadIdx.x;
    if (i < ntok * D2) {
        const int64_t n = i / D2;
        const int d2 = (int)(i - n * D2);
        float2* col = reinterpret_cast<float2*>(y) + n * H * D2 + d2;
        float2 v[kMixMaxH];
#pragma unroll
        for (int h = 0; h < kMixMaxH; ++h)
            if (h < H) v[h] = col[(int64_t)h * D2];
#pragma unroll
        for (int g = 0; g < kMixMaxH; ++g) {
            if (g < H) {
                float2 o = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int h = 0; h < kMixMaxH; ++h) {
                    if (h < H) {
                        const float c = sw[g * kMixMaxH + h];
                        o.x = fmaf(c, v[h].x, o.x);
                        o.y = fmaf(c, v[h].y, o.y);
                    }
                }
                col[(int64_t)g * D2] = o;
            }
        }
    }
}

}  // namespace

int head_mix_launch(float* y, const float* w, int64_t ntok, int H, int D, cudaStream_t stream) {
    if (H < 1 || H > kMixMaxH || D % 2 != 0 || ntok < 0) return SSDC_ERR_UNSUPPORTED;
    if (ntok == 0) return 0;
    const int64_t grid = (ntok * (D / 2) + kMixThreads - 1) / kMixThreads;
    if (grid > 0x7fffffff) return SSDC_ERR_UNSUPPORTED;
    if (launch_dependent(ssdc_head_mix, dim3((unsigned)grid), dim3(kMixThreads), 0, stream, y, w, ntok, H, D / 2) !=
        cudaSuccess)
        return SSDC_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? 1 : SSDC_ERR_CUDA;
}

}  // namespace ssdc
