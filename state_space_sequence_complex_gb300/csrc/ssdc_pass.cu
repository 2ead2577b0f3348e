// Inter-chunk state pass (landing page, "03 Chunkwise SSD", STATE line: the
// chunk states are carried across chunks by the chunk decays).
//
//   S_in[0] = 0 (or the given initial state),
//   S_in[c+1] = a_c * S_in[c] + S_loc[c],  a_c = exp(Acs_c[Q-1])
//   final_state = a_last * S_in[last] + S_loc[last]
//
// This is the sequential form of the pages' "decay_chunk matrix" recurrence.
// One thread owns one complex (d, n) lane of one (b, h) sequence and walks its
// chunks in order, replacing S_loc[c] in the workspace by S_in[c]. The loads
// of S_loc do not depend on the chain, so they are issued a group of chunks
// ahead; only the complex multiply-add is serial. fp32 throughout.
#include <cuda_runtime.h>

#include "ssdc_kernels.h"

namespace ssdc {

constexpr int kPassAhead = 8;

__global__ void __launch_bounds__(kPassThreads)
ssdc_state_pass(Problem p, Workspace ws) {
    const int64_t bh = blockIdx.y;
    const int ND = p.N * p.D;
    const int j = blockIdx.x * kPassThreads + threadIdx.x;  // lane = d * N + n
    if (j >= ND) return;
    const int64_t nc = p.nc;
    float* S = ws.S + bh * nc * 2 * ND + j;
    const float* a = ws.a + bh * nc * 2;
    const int d = j / p.N, n = j % p.N;
    const int64_t o = (bh * p.N + n) * p.D + d;  // (b, h, n, d) of the initial and final states
    float sr = 0.0f, si = 0.0f;
    if (p.s0_re != nullptr) {
        sr = p.s0_re[o];
        si = p.s0_im[o];
    }
    for (int64_t c0 = 0; c0 < nc; c0 += kPassAhead) {
        float lr[kPassAhead], li[kPassAhead], ar[kPassAhead], ai[kPassAhead];
#pragma unroll
        for (int k = 0; k < kPassAhead; ++k) {
            if (c0 + k < nc) {
                const float* s = S + (c0 + k) * 2 * ND;
                lr[k] = __ldcg(s);
                li[k] = __ldcg(s + ND);
                ar[k] = __ldg(a + 2 * (c0 + k));
                ai[k] = __ldg(a + 2 * (c0 + k) + 1);
            }
        }
#pragma unroll
        for (int k = 0; k < kPassAhead; ++k) {
            if (c0 + k < nc) {
                float* s = S + (c0 + k) * 2 * ND;
                __stcg(s, sr);
                __stcg(s + ND, si);
                const float nr = fmaf(ar[k], sr, fmaf(-ai[k], si, lr[k]));
                const float ni = fmaf(ar[k], si, fmaf(ai[k], sr, li[k]));
                sr = nr;
                si = ni;
            }
        }
    }
    p.fs_re[o] = sr;
    p.fs_im[o] = si;
}

}  // namespace ssdc
