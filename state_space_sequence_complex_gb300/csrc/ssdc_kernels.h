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
    // x, B_t and C_t hold bfloat16 planes (the pointers above are their
    // addresses, read only through tensor maps); 0: fp32
    int in_bf16 = 0;
    // The MIMO head mixer fused into the epilogue (the tensor-memory kernel): mix_w
    // (H x H, H <= 16) or null; y_re then receives the mixed Re(y) and y_im is null;
    // mix_count: B * ceil(T / min(Q, 64)) counters, zero at launch.
    const float* mix_w = nullptr;
    int* mix_count = nullptr;
    // Test hook of the fused kernel: the CTA of this chunk index does not send
    // the state it computes (-1 = off), so that its successor's bounded wait
    // gives up and reports SSDC_ERR_TIMEOUT.
    int64_t drop_send_chunk;
};

// Sizes and device pointers of one backward call: the forward problem (its
// y is unused; fs points into the backward workspace, where the recomputed
// final state goes) plus the output gradients and the input gradients.
struct GradProblem {
    Problem f;
    const float *dy_re, *dy_im;    // dy_im may be null: zero
    const float *dfs_re, *dfs_im;  // both null: zero
    float *dx_re, *dx_im;          // dx_im may be null: not written
    float *dA_re, *dA_im;
    float *dB_re, *dB_im, *dC_re, *dC_im, *ddt;
    float *ds0_re, *ds0_im;  // both null: not written
};

// Backward workspace beyond the forward one (S, a, status).
//   R  [B*H*nc][2][D][N] floats: U_c, replaced in place by R_c, the gradient
//      of the state leaving chunk c (transposed like S)
//   r  [B*H][2][T] floats: r_t = <dC_t, C_t> - <dB_t, B_t> of every token
//   anchor [B*H*nc][2] doubles: <R_c, S_out(c)>, S_out(c) the state leaving chunk c
//   dA_part [B*H*nc][2] doubles: each chunk's share of dA
struct GradWorkspace {
    float* R;
    float* r;
    double* anchor;
    double* dA_part;
};

// Backward kernels (exact fp32, SIMT).
// The chunk-state/adjoint kernel and the chunk-gradient kernel are templates
// (compile-time N = D = 64, or sizes from the problem); these enqueue the
// right instantiation and set their shared-memory limits.
// The chunk-gradient kernel on the TF32 tensor cores (ssdc_bwd_tc.cu): Q = 16,
// 32 or 64, N and D multiples of 8 up to 64; returns launches or an error.
bool bwd_tc_supported(int N, int D, int Q);
int bwd_tc_launch_chunk(const GradProblem& g, const Workspace& ws, const GradWorkspace& gw, cudaStream_t stream);
// Its chunk-state kernel (S_loc, U_c and a_c per chunk, the outputs of the exact one).
int bwd_tc_launch_chunk_states(const GradProblem& g, const Workspace& ws, const GradWorkspace& gw,
                               cudaStream_t stream);
cudaError_t bwd_set_smem_attrs();
void bwd_launch_chunk_states(const GradProblem& g, const Workspace& ws, const GradWorkspace& gw,
                             cudaStream_t stream);
void bwd_launch_chunk(const GradProblem& g, const Workspace& ws, const GradWorkspace& gw, cudaStream_t stream);
__global__ void ssdc_bwd_passes(GradProblem g, Workspace ws, GradWorkspace gw);
__global__ void ssdc_bwd_dt(GradProblem g, Workspace ws, GradWorkspace gw);
__global__ void ssdc_bwd_dA(GradProblem g, Workspace ws, GradWorkspace gw);
constexpr int kBwdDtThreads = 256;
constexpr int kBwdChunkThreads = 512;  // threads of the chunk-gradient kernel

// SIMT (exact fp32) kernels.
// SIMT kernels are templates (compile-time N = D = 64, or sizes from the
// problem); these enqueue the right instantiation and set their shared-memory
// limits.
cudaError_t simt_set_smem_attrs();
void simt_launch_chunk_state(const Problem& p, const Workspace& ws, cudaStream_t stream);
void simt_launch_chunk_scan(const Problem& p, const Workspace& ws, cudaStream_t stream);

// Inter-chunk state pass (fp32, both precisions).
__global__ void ssdc_state_pass(Problem p, Workspace ws);
constexpr int kPassThreads = 256;

// One lane of a chunk recurrence: x <- a_c x + l_c over the nc chunks of one
// sequence, l_c at X + c * 2 ND (real plane) and + ND (imaginary plane), each
// replaced in its slot by the x entering the step; a_c at a + 2 c. Step k is
// chunk k, or chunk nc - 1 - k with `backwards`, whose coefficient is conj(a_c).
// The loads do not depend on the chain, so kPassAhead chunks' loads stay in
// flight: a slot is refilled, with the chunk kPassAhead steps on (a slot not yet
// written), as soon as its chunk is consumed. x is the incoming value; the
// last is returned.
constexpr int kPassAhead = 8;
__device__ __forceinline__ float2 chain_walk(float* X, const float* a, int64_t nc, int ND, bool backwards,
                                             float2 x) {
    float xr = x.x, xi = x.y;
    const float sg = backwards ? -1.0f : 1.0f;
    auto chunk_of = [&](int64_t k) { return backwards ? nc - 1 - k : k; };
    float lr[kPassAhead], li[kPassAhead], ar[kPassAhead], ai[kPassAhead];
#pragma unroll
    for (int k = 0; k < kPassAhead; ++k)
        if (k < nc) {
            const int64_t c = chunk_of(k);
            lr[k] = __ldcg(X + c * 2 * ND);
            li[k] = __ldcg(X + c * 2 * ND + ND);
            ar[k] = __ldg(a + 2 * c);
            ai[k] = sg * __ldg(a + 2 * c + 1);
        }
#pragma unroll 1
    for (int64_t k0 = 0; k0 < nc; k0 += kPassAhead) {
#pragma unroll
        for (int k = 0; k < kPassAhead; ++k) {
            if (k0 + k < nc) {
                const int64_t c = chunk_of(k0 + k);
                __stcg(X + c * 2 * ND, xr);
                __stcg(X + c * 2 * ND + ND, xi);
                const float nr = fmaf(ar[k], xr, fmaf(-ai[k], xi, lr[k]));
                const float ni = fmaf(ar[k], xi, fmaf(ai[k], xr, li[k]));
                xr = nr;
                xi = ni;
            }
            if (k0 + k + kPassAhead < nc) {
                const int64_t c = chunk_of(k0 + k + kPassAhead);
                lr[k] = __ldcg(X + c * 2 * ND);
                li[k] = __ldcg(X + c * 2 * ND + ND);
                ar[k] = __ldg(a + 2 * c);
                ai[k] = sg * __ldg(a + 2 * c + 1);
            }
        }
    }
    return make_float2(xr, xi);
}
// The same, not inlined, for a caller whose direction is fixed: a direction known
// at compile time let the compiler hold more addresses than registers.
static __device__ __noinline__ float2 chain_walk_call(float* X, const float* a, int64_t nc, int ND, bool backwards,
                                                      float2 x) {
    return chain_walk(X, a, nc, ND, backwards, x);
}

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
// The cluster size the cluster kernel would choose for this problem, and its
// estimated length in chunk-times of one CTA (waves x the longer of a CTA's
// chunks and the state chain).
int fused_cluster_choice(const Problem& p, int* cl, double* cost);
int fused_launch(const Problem& p, const Workspace& ws, cudaStream_t stream, int force_cluster, bool plane_maps);

// Fused TF32 kernel with the chunk state in tensor memory: one CTA per SM walks
// whole sequences. Q in {16, 32, 64, 128, 256}; N, D multiples of 8 up to 64.
bool fused2_supported(int N, int D, int Q);
int fused2_launch(const Problem& p, const Workspace& ws, cudaStream_t stream, bool plane_maps);

// Programmatic dependent launch. A kernel launched with launch_dependent may have its CTAs
// scheduled while the previous kernel on the stream finishes its last CTAs; it must call
// grid_dependency_wait() before it reads anything that kernel writes (or writes anything that
// kernel reads), which holds it until that kernel has completed and its writes are visible.
// Launched the ordinary way, the wait returns at once.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// MIMO head mixer in place over y (ssdc_mix.cu): y[n, g, :] = sum_h w[g * H + h] y[n, h, :]
// for ntok tokens of H x D fp32 (16-byte aligned, D a multiple of 4, H <= 16). Returns the
// launches (0 or 1) or an error.
int head_mix_launch(float* y, const float* w, int64_t ntok, int H, int D, cudaStream_t stream);

// The state side of the same kernel alone (ssdc_state.cu): the final state of
// each sequence from x, B_t and dt, without y (p.C_*, p.y_* unused). The same
// sizes as fused2; returns launches or an error.
bool state_supported(int N, int D, int Q);
int state_launch(const Problem& p, const Workspace& ws, cudaStream_t stream, bool plane_maps);

// Launch count reported by ssd_complex_last_launch_count() for the calling thread.
void set_last_launch_count(int n);

}  // namespace ssdc
