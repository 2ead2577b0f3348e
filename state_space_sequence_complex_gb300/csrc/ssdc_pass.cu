// Inter-chunk state pass (landing page, "03 Chunkwise SSD", STATE line: the
// chunk states are carried across chunks by the chunk decays).
//
//   S_in[0] = 0 (or the given initial state),
//   S_in[c+1] = a_c * S_in[c] + S_loc[c],  a_c = exp(Acs_c[Q-1])
//   final_state = a_last * S_in[last] + S_loc[last]
//
// This is the sequential form of the pages' "decay_chunk matrix" recurrence.
// One thread owns one complex (d, n) lane of one (b, h) sequence and walks its
// chunks in order, replacing S_loc[c] in the workspace by S_in[c] (chain_walk:
// the loads of S_loc do not depend on the chain and stay a window of chunks
// ahead; only the complex multiply-add is serial). fp32 throughout.
#include <cuda_runtime.h>

#include "ssdc_kernels.h"

namespace ssdc {

__global__ void __launch_bounds__(kPassThreads, 4)
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
    const float2 so = chain_walk_call(S, a, nc, ND, false, make_float2(sr, si));
    sr = so.x;
    si = so.y;
    p.fs_re[o] = sr;
    p.fs_im[o] = si;
}

}  // namespace ssdc
