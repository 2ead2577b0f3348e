// Internal declarations shared by the host entry points and the kernels.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "ssdc_common.cuh"

namespace ssdc {

// Sizes and device pointers of one forward call (planar complex planes).
struct Problem {
    const float *x_re, *x_im, *A_re, *A_im, *B_re, *B_im, *C_re, *C_im, *dt;
    const float *s0_re, *s0_im;  // initial state (B, H, N, D), or null: zero
    float *y_re, *y_im, *fs_re, *fs_im;
    int64_t T;
    int B, H, N, D, Q;
    int64_t nc;  // chunks per sequence, ceil(T / Q)
    // Test hook of the fused kernel: the CTA of this chunk index does not send
    // the state it computes (-1 = off), so that its successor's bounded wait
    // gives up and reports SSDC_ERR_TIMEOUT.
    int64_t drop_send_chunk;
};

// SIMT (exact fp32) kernels.
__global__ void ssdc_simt_chunk_state(Problem p, Workspace ws);
__global__ void ssdc_simt_chunk_scan(Problem p, Workspace ws);
size_t simt_state_smem();
size_t simt_scan_smem();

// Inter-chunk state pass (fp32, both precisions).
__global__ void ssdc_state_pass(Problem p, Workspace ws);
constexpr int kPassThreads = 256;

// tcgen05 / TMA kernels (TF32 tensor cores). Returns the number of launches
// enqueued, or a negative SSDC_ERR_* code.
int tc_launch_chunk_state(const Problem& p, const Workspace& ws, cudaStream_t stream);
int tc_launch_chunk_scan(const Problem& p, const Workspace& ws, cudaStream_t stream);
bool tc_supported(int N, int D, int Q);

// Fused single-pass TF32 kernel (state passed through distributed shared
// memory inside thread-block clusters). force_cluster = 0 picks the cluster
// size; 1, 2, 4 or 8 forces it. plane_maps = false fetches every plane with
// its own tensor map even where one map could fetch both.
bool fused_supported(int N, int D, int Q);
int fused_launch(const Problem& p, const Workspace& ws, cudaStream_t stream, int force_cluster, bool plane_maps);

// Launch count reported by ssd_complex_last_launch_count() for the calling thread.
void set_last_launch_count(int n);

}  // namespace ssdc
