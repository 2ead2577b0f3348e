// Host side of the C ABI declared in include/ssdc.h: argument checks,
// workspace carving and the launch sequences
//   forward:  chunk-state kernel -> state pass -> chunk-scan kernel
//             (or the fused kernel)
//   backward: chunk states and adjoints -> both chunk recurrences -> chunk
//             gradients -> step-size gradients -> per-head dA
// on the caller's stream. No allocation happens in ssd_complex_fwd_ws or
// ssd_complex_bwd.
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include <cuda_runtime.h>

#include "../../include/ssdc.h"
#include "ssdc_kernels.h"

namespace {

thread_local int g_last_launches = 0;
thread_local int g_last_path = -1;

// Process-wide options (ssd_complex_set_option); read on every call, set rarely.
std::atomic<int> g_opt_cluster{0};           // SSDC_OPT_FUSED_CLUSTER: 0 = chosen per call
std::atomic<int> g_opt_plane_maps{1};        // SSDC_OPT_FUSED_PLANE_MAPS
std::atomic<int64_t> g_opt_drop_state_chunk{-1};  // SSDC_OPT_TEST_DROP_STATE_CHUNK: -1 = off
std::atomic<int> g_opt_kernel{0};            // SSDC_OPT_FUSED_KERNEL: 0 = chosen per call
std::atomic<int> g_opt_mimo_fused{0};        // SSDC_OPT_MIMO_FUSED: 0 = scan, then the mixer kernel

// Instrumentation events (see ssd_complex_timing_enable).
constexpr int kMaxTimed = 8;
bool g_timing = false;
int g_timed_launches = 0;
cudaEvent_t g_events[kMaxTimed + 1] = {};
bool g_events_made = false;

int record_event(int i, cudaStream_t stream) {
    if (!g_timing) return SSDC_OK;
    if (i > kMaxTimed) return SSDC_ERR_INVALID;
    return cudaEventRecord(g_events[i], stream) == cudaSuccess ? SSDC_OK : SSDC_ERR_CUDA;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_attr_done[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

int check_sizes(const ssdc_dims& d, int Q) {
    if (d.B <= 0 || d.T <= 0 || d.H <= 0 || d.N <= 0 || d.D <= 0 || Q <= 0) return SSDC_ERR_INVALID;
    if (d.precision != SSDC_PREC_TF32 && d.precision != SSDC_PREC_FP32 && d.precision != SSDC_PREC_TF32_STAGED)
        return SSDC_ERR_INVALID;
    if (d.B > 65535 || d.H > 65535 || d.B * d.H > 65535) return SSDC_ERR_UNSUPPORTED;
    const int64_t nc = ssdc::ceil_div64(d.T, Q);
    if (nc * 4 > INT32_MAX) return SSDC_ERR_UNSUPPORTED;
    // every plane must be indexable
    const int64_t big = d.B * d.T * d.H * (d.N > d.D ? d.N : d.D);
    if (big <= 0 || big > (int64_t(1) << 40)) return SSDC_ERR_UNSUPPORTED;
    if (d.precision == SSDC_PREC_FP32) {
        if (!is_pow2_in(Q, 16, 256)) return SSDC_ERR_UNSUPPORTED;
        if (d.N % 8 || d.D % 8 || d.N > 64 || d.D > 64) return SSDC_ERR_UNSUPPORTED;
    } else if (d.precision == SSDC_PREC_TF32_STAGED) {
        if (!ssdc::tc_supported((int)d.N, (int)d.D, Q)) return SSDC_ERR_UNSUPPORTED;
    } else {
        if (!ssdc::tc_supported((int)d.N, (int)d.D, Q) && !ssdc::fused2_supported((int)d.N, (int)d.D, Q))
            return SSDC_ERR_UNSUPPORTED;
    }
    return SSDC_OK;
}

// TF32 sizes that one of the two fused kernels runs (the others take the staged path).
bool use_fused(const ssdc_dims& d, int Q) {
    return d.precision == SSDC_PREC_TF32 &&
           (ssdc::fused_supported((int)d.N, (int)d.D, Q) || ssdc::fused2_supported((int)d.N, (int)d.D, Q));
}

// The fused head mixer's counters: one per (batch row, row tile of min(Q, 64) tokens).
int64_t mix_counters(const ssdc_dims& d, int Q) { return d.B * ssdc::ceil_div64(d.T, Q < 64 ? Q : 64); }
size_t mix_ws_bytes(const ssdc_dims& d, int Q) {
    return 256 + (((size_t)mix_counters(d, Q) * sizeof(int) + 255) & ~size_t(255));
}

size_t ws_bytes_for(const ssdc_dims& d, int Q) {
    if (use_fused(d, Q)) return 256;  // status word only
    const int64_t nc = ssdc::ceil_div64(d.T, Q);
    const int64_t chunks = d.B * d.H * nc;
    size_t s = (size_t)chunks * 2 * d.N * d.D * sizeof(float);
    s = (s + 255) & ~size_t(255);
    size_t a = (size_t)chunks * 2 * sizeof(float);
    a = (a + 255) & ~size_t(255);
    return s + a + 256;
}

ssdc::Workspace carve(void* ws, const ssdc_dims& d, int Q) {
    // [status word, padded to 256 B][S][a]
    const int64_t nc = ssdc::ceil_div64(d.T, Q);
    const int64_t chunks = d.B * d.H * nc;
    size_t s = (size_t)chunks * 2 * d.N * d.D * sizeof(float);
    s = (s + 255) & ~size_t(255);
    char* base = static_cast<char*>(ws);
    ssdc::Workspace w;
    w.status = reinterpret_cast<int*>(base);
    if (use_fused(d, Q)) {
        w.S = nullptr;
        w.a = nullptr;
    } else {
        w.S = reinterpret_cast<float*>(base + 256);
        w.a = reinterpret_cast<float*>(base + 256 + s);
    }
    return w;
}

int setup_device_attrs() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SSDC_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SSDC_ERR_CUDA;
    if (g_attr_done[dev].load(std::memory_order_acquire)) return SSDC_OK;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return SSDC_ERR_CUDA;
    if (major != 10 || minor != 3) return SSDC_ERR_DEVICE;
    if (ssdc::simt_set_smem_attrs() != cudaSuccess) return SSDC_ERR_CUDA;
    if (ssdc::bwd_set_smem_attrs() != cudaSuccess) return SSDC_ERR_CUDA;
    g_attr_done[dev].store(1, std::memory_order_release);
    return SSDC_OK;
}

// The forward pass behind ssd_complex_fwd_ws, ssd_complex_fwd_init and
// ssd_complex_fwd_bf16: s0 = the initial state's planes, or both null for a zero
// initial state; in_bf16: x, B_t and C_t point to bfloat16 planes.
int fwd_impl(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t, const float* dt, ssdc_cin s0, ssdc_dims dims,
             int chunk_size, ssdc_cout y, ssdc_cout final_state, void* workspace, size_t ws_bytes,
             cudaStream_t stream, bool in_bf16 = false, const float* mix = nullptr);

}  // namespace

extern "C" {

int ssd_complex_fwd_supported(ssdc_dims dims, int chunk_size) { return check_sizes(dims, chunk_size); }

size_t ssd_complex_fwd_workspace_bytes(ssdc_dims dims, int chunk_size) {
    if (check_sizes(dims, chunk_size) != SSDC_OK) return 0;
    return ws_bytes_for(dims, chunk_size);
}

int ssd_complex_fwd_ws(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t, const float* dt,
                       ssdc_dims dims, int chunk_size, ssdc_cout y, ssdc_cout final_state,
                       void* workspace, size_t ws_bytes, cudaStream_t stream) {
    return fwd_impl(x, A, B_t, C_t, dt, ssdc_cin{nullptr, nullptr}, dims, chunk_size, y, final_state, workspace,
                    ws_bytes, stream);
}

int ssd_complex_fwd_init(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t, const float* dt,
                         ssdc_cin initial_state, ssdc_dims dims, int chunk_size, ssdc_cout y,
                         ssdc_cout final_state, void* workspace, size_t ws_bytes, cudaStream_t stream) {
    return fwd_impl(x, A, B_t, C_t, dt, initial_state, dims, chunk_size, y, final_state, workspace, ws_bytes,
                    stream);
}

int ssd_complex_fwd_bf16(ssdc_cin_bf16 x, ssdc_cin A, ssdc_cin_bf16 B_t, ssdc_cin_bf16 C_t, const float* dt,
                         ssdc_cin initial_state, ssdc_dims dims, int chunk_size, ssdc_cout y,
                         ssdc_cout final_state, void* workspace, size_t ws_bytes, cudaStream_t stream) {
    auto as_cin = [](ssdc_cin_bf16 v) {
        return ssdc_cin{reinterpret_cast<const float*>(v.re), reinterpret_cast<const float*>(v.im)};
    };
    return fwd_impl(as_cin(x), A, as_cin(B_t), as_cin(C_t), dt, initial_state, dims, chunk_size, y, final_state,
                    workspace, ws_bytes, stream, true);
}

size_t ssd_complex_fwd_mimo_workspace_bytes(ssdc_dims dims, int chunk_size) {
    if (check_sizes(dims, chunk_size) != SSDC_OK || dims.precision != SSDC_PREC_TF32 || chunk_size > 64 ||
        dims.H > 16 || !ssdc::fused2_supported((int)dims.N, (int)dims.D, chunk_size))
        return 0;
    return mix_ws_bytes(dims, chunk_size);
}

int ssd_complex_fwd_mimo(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t, const float* dt, const float* mix,
                         ssdc_cin initial_state, ssdc_dims dims, int chunk_size, float* out,
                         ssdc_cout final_state, void* workspace, size_t ws_bytes, cudaStream_t stream) {
    if (mix == nullptr) return SSDC_ERR_INVALID;
    return fwd_impl(x, A, B_t, C_t, dt, initial_state, dims, chunk_size, ssdc_cout{out, nullptr}, final_state,
                    workspace, ws_bytes, stream, false, mix);
}

}  // extern "C"

namespace {

int fwd_impl(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t, const float* dt, ssdc_cin s0, ssdc_dims dims,
             int chunk_size, ssdc_cout y, ssdc_cout final_state, void* workspace, size_t ws_bytes,
             cudaStream_t stream, bool in_bf16, const float* mix) {
    int rc = check_sizes(dims, chunk_size);
    if (rc != SSDC_OK) return rc;
    // the fused head mixer runs on the tensor-memory kernel, chunks of up to 64 tokens, H <= 16
    if (mix != nullptr && (dims.precision != SSDC_PREC_TF32 || chunk_size > 64 || dims.H > 16 ||
                           !ssdc::fused2_supported((int)dims.N, (int)dims.D, chunk_size)))
        return SSDC_ERR_UNSUPPORTED;
    // bfloat16 inputs run on the tensor-memory kernel only
    if (in_bf16 && (dims.precision != SSDC_PREC_TF32 ||
                    !ssdc::fused2_supported((int)dims.N, (int)dims.D, chunk_size)))
        return SSDC_ERR_UNSUPPORTED;
    // x.im may be null: a real x (its imaginary plane is zero and is not read); with the fused head
    // mixer y.im is null (only the mixed Re(y) is written) and the matrix is required
    if (mix != nullptr ? y.im != nullptr : y.im == nullptr) return SSDC_ERR_INVALID;
    const void* ptrs[] = {x.re, A.re, A.im, B_t.re, B_t.im, C_t.re, C_t.im, dt,
                          y.re, mix != nullptr ? static_cast<const void*>(mix) : y.im, final_state.re, final_state.im};
    for (const void* q : ptrs)
        if (q == nullptr) return SSDC_ERR_INVALID;
    for (const void* q : ptrs)
        if (!aligned16(q)) return SSDC_ERR_ALIGN;
    if (!aligned16(x.im)) return SSDC_ERR_ALIGN;
    if (x.im == x.re) return SSDC_ERR_INVALID;
    const bool has_s0 = s0.re != nullptr;
    if ((s0.re == nullptr) != (s0.im == nullptr) || (has_s0 && s0.re == s0.im)) return SSDC_ERR_INVALID;
    if (has_s0 && (!aligned16(s0.re) || !aligned16(s0.im))) return SSDC_ERR_ALIGN;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return SSDC_ERR_WORKSPACE;
    if (ws_bytes < (mix != nullptr ? mix_ws_bytes(dims, chunk_size) : ws_bytes_for(dims, chunk_size)))
        return SSDC_ERR_WORKSPACE;

    // outputs must not overlap inputs, the workspace or each other
    const int64_t BTH = dims.B * dims.T * dims.H;
    auto rng = [](const void* p, int64_t n, size_t elem = sizeof(float)) {
        const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        return Range{lo, p == nullptr ? lo : lo + (uintptr_t)n * elem};  // null: empty
    };
    const size_t ie = in_bf16 ? 2 : sizeof(float);  // bytes of an x, B_t or C_t element
    const Range in[] = {rng(x.re, BTH * dims.D, ie), rng(x.im, BTH * dims.D, ie), rng(A.re, dims.H),
                        rng(A.im, dims.H), rng(B_t.re, BTH * dims.N, ie), rng(B_t.im, BTH * dims.N, ie),
                        rng(C_t.re, BTH * dims.N, ie), rng(C_t.im, BTH * dims.N, ie), rng(dt, BTH),
                        Range{reinterpret_cast<uintptr_t>(workspace),
                              reinterpret_cast<uintptr_t>(workspace) + ws_bytes},
                        rng(mix, dims.H * dims.H)};
    const int64_t fsn = dims.B * dims.H * dims.N * dims.D;
    const Range out[] = {rng(y.re, BTH * dims.D), rng(y.im, BTH * dims.D), rng(final_state.re, fsn),
                         rng(final_state.im, fsn)};
    for (const Range& o : out)
        for (const Range& i : in)
            if (overlaps(o, i)) return SSDC_ERR_INVALID;
    for (int i = 0; i < 4; ++i)
        for (int j = i + 1; j < 4; ++j)
            if (overlaps(out[i], out[j])) return SSDC_ERR_INVALID;
    if (has_s0) {
        // the initial state may be the final-state buffer itself (updated in place), plane for
        // plane; it must not otherwise overlap an output or the workspace
        const bool in_place = s0.re == final_state.re && s0.im == final_state.im;
        const Range st[] = {rng(s0.re, fsn), rng(s0.im, fsn)};
        if (overlaps(st[0], st[1])) return SSDC_ERR_INVALID;
        for (const Range& r : st) {
            if (overlaps(r, out[0]) || overlaps(r, out[1]) || overlaps(r, in[9])) return SSDC_ERR_INVALID;
            if (!in_place && (overlaps(r, out[2]) || overlaps(r, out[3]))) return SSDC_ERR_INVALID;
        }
    }

    rc = setup_device_attrs();
    if (rc != SSDC_OK) return rc;

    ssdc::Problem p;
    p.x_re = x.re; p.x_im = x.im; p.A_re = A.re; p.A_im = A.im;
    p.B_re = B_t.re; p.B_im = B_t.im; p.C_re = C_t.re; p.C_im = C_t.im; p.dt = dt;
    p.s0_re = s0.re; p.s0_im = s0.im;
    p.y_re = y.re; p.y_im = y.im; p.fs_re = final_state.re; p.fs_im = final_state.im;
    p.T = dims.T; p.B = (int)dims.B; p.H = (int)dims.H; p.N = (int)dims.N; p.D = (int)dims.D;
    p.Q = chunk_size;
    p.nc = ssdc::ceil_div64(dims.T, chunk_size);
    p.drop_send_chunk = g_opt_drop_state_chunk.load(std::memory_order_relaxed);
    p.in_bf16 = in_bf16 ? 1 : 0;
    ssdc::Workspace w = carve(workspace, dims, chunk_size);
    // the head mixer: fused into the scan's epilogue (SSDC_OPT_MIMO_FUSED), or by default a
    // separate in-place kernel over the Re(y) the scan writes into the output
    const bool mix_fused = mix != nullptr && g_opt_mimo_fused.load(std::memory_order_relaxed) != 0;
    if (mix_fused) {
        p.mix_w = mix;
        p.mix_count = reinterpret_cast<int*>(static_cast<char*>(workspace) + 256);
    }

    (void)cudaGetLastError();  // clear a stale error from unrelated work
    int launches = 0;
    if (record_event(0, stream) != SSDC_OK) return SSDC_ERR_CUDA;
    // the status word starts at SSDC_OK; a kernel's failed wait records the first error (and the
    // fused head mixer's counters start at zero)
    if (cudaMemsetAsync(w.status, 0, mix_fused ? mix_ws_bytes(dims, chunk_size) : sizeof(int), stream) !=
        cudaSuccess)
        return SSDC_ERR_CUDA;
    const dim3 pass_grid((unsigned)ssdc::ceil_div64((int64_t)p.N * p.D, ssdc::kPassThreads),
                         (unsigned)(p.B * p.H));
    int path = SSDC_PATH_STAGED_FP32;
    if (dims.precision == SSDC_PREC_FP32) {
        ssdc::simt_launch_chunk_state(p, w, stream);
        record_event(++launches, stream);
        ssdc::ssdc_state_pass<<<pass_grid, ssdc::kPassThreads, 0, stream>>>(p, w);
        record_event(++launches, stream);
        ssdc::simt_launch_chunk_scan(p, w, stream);
        record_event(++launches, stream);
    } else if (use_fused(dims, chunk_size)) {
        const int force = g_opt_cluster.load(std::memory_order_relaxed);
        const bool plane_maps = g_opt_plane_maps.load(std::memory_order_relaxed) != 0;
        // The cluster kernel takes Q = N = D = 64 only; there it runs when a forced cluster size
        // asks for it, or when its estimated time is the shorter. Estimates, from per-chunk
        // times measured on a GB300 at full occupancy: the tensor-memory kernel walks
        // ceil(sequences / SMs) x chunks at about 3.7 us a chunk; the cluster kernel, its chosen
        // cost at about 4.1 us a chunk with one CTA per sequence and 5.2 us with the state
        // handed between CTAs.
        int kernel = (in_bf16 || mix_fused) ? 2 : g_opt_kernel.load(std::memory_order_relaxed);
        const bool cluster_ok = ssdc::fused_supported(p.N, p.D, p.Q) && !in_bf16 && !mix_fused;
        if (kernel == 0) {
            if (!cluster_ok) {
                kernel = 2;
            } else if (force > 0) {
                kernel = 1;
            } else {
                int cl = 1, dev = 0, sms = 0;
                double cost = 0.0;
                rc = ssdc::fused_cluster_choice(p, &cl, &cost);
                if (rc != SSDC_OK) return rc;
                if (cudaGetDevice(&dev) != cudaSuccess ||
                    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
                    return SSDC_ERR_CUDA;
                const int64_t nseq = (int64_t)p.B * p.H;
                const double t_tmem = 3.7 * (double)((nseq + sms - 1) / sms) * (double)p.nc;
                const double t_cluster = (cl > 1 ? 5.2 : 4.1) * cost;
                kernel = t_tmem <= t_cluster ? 2 : 1;
            }
        }
        if (kernel == 1 && !cluster_ok) return SSDC_ERR_UNSUPPORTED;
        const int n = kernel == 2 ? ssdc::fused2_launch(p, w, stream, plane_maps && !mix_fused)
                                  : ssdc::fused_launch(p, w, stream, force, plane_maps);
        if (n < 0) return n;
        path = kernel == 2 ? SSDC_PATH_FUSED_TMEM : SSDC_PATH_FUSED_CLUSTER;
        launches += n;
        record_event(launches, stream);
        if (mix != nullptr && !mix_fused) {
            const int m = ssdc::head_mix_launch(p.y_re, mix, dims.B * dims.T, p.H, p.D, stream);
            if (m < 0) return m;
            launches += m;
            record_event(launches, stream);
        }
    } else {
        path = SSDC_PATH_STAGED_TF32;
        int n = ssdc::tc_launch_chunk_state(p, w, stream);
        if (n < 0) return n;
        launches += n;
        record_event(launches, stream);
        ssdc::ssdc_state_pass<<<pass_grid, ssdc::kPassThreads, 0, stream>>>(p, w);
        record_event(++launches, stream);
        n = ssdc::tc_launch_chunk_scan(p, w, stream);
        if (n < 0) return n;
        launches += n;
        record_event(launches, stream);
    }
    if (cudaGetLastError() != cudaSuccess) return SSDC_ERR_CUDA;
    g_last_launches = launches;
    g_last_path = path;
    if (g_timing) g_timed_launches = launches;
    return SSDC_OK;
}


// The final state alone (ssd_complex_final_state): the forward's chunk states and
// state pass, with no chunk outputs; C_t and y are not used.
int final_state_impl(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, const float* dt, ssdc_cin s0, ssdc_dims dims,
                     int chunk_size, ssdc_cout final_state, void* workspace, size_t ws_bytes,
                     cudaStream_t stream) {
    int rc = check_sizes(dims, chunk_size);
    if (rc != SSDC_OK) return rc;
    const void* ptrs[] = {x.re, A.re, A.im, B_t.re, B_t.im, dt, final_state.re, final_state.im};
    for (const void* q : ptrs)
        if (q == nullptr) return SSDC_ERR_INVALID;
    for (const void* q : ptrs)
        if (!aligned16(q)) return SSDC_ERR_ALIGN;
    if (!aligned16(x.im)) return SSDC_ERR_ALIGN;
    if (x.im == x.re) return SSDC_ERR_INVALID;
    const bool has_s0 = s0.re != nullptr;
    if ((s0.re == nullptr) != (s0.im == nullptr) || (has_s0 && s0.re == s0.im)) return SSDC_ERR_INVALID;
    if (has_s0 && (!aligned16(s0.re) || !aligned16(s0.im))) return SSDC_ERR_ALIGN;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return SSDC_ERR_WORKSPACE;
    if (ws_bytes < ws_bytes_for(dims, chunk_size)) return SSDC_ERR_WORKSPACE;

    // the final state must not overlap an input, the workspace or its other plane; the
    // initial state may be the final state itself (in place, plane for plane)
    const int64_t BTH = dims.B * dims.T * dims.H;
    auto rng = [](const void* p, int64_t n) {
        const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        return Range{lo, p == nullptr ? lo : lo + (uintptr_t)n * sizeof(float)};  // null: empty
    };
    const int64_t fsn = dims.B * dims.H * dims.N * dims.D;
    const Range in[] = {rng(x.re, BTH * dims.D), rng(x.im, BTH * dims.D), rng(A.re, dims.H), rng(A.im, dims.H),
                        rng(B_t.re, BTH * dims.N), rng(B_t.im, BTH * dims.N), rng(dt, BTH),
                        Range{reinterpret_cast<uintptr_t>(workspace),
                              reinterpret_cast<uintptr_t>(workspace) + ws_bytes}};
    const Range out[] = {rng(final_state.re, fsn), rng(final_state.im, fsn)};
    for (const Range& o : out)
        for (const Range& i : in)
            if (overlaps(o, i)) return SSDC_ERR_INVALID;
    if (overlaps(out[0], out[1])) return SSDC_ERR_INVALID;
    if (has_s0) {
        const bool in_place = s0.re == final_state.re && s0.im == final_state.im;
        const Range st[] = {rng(s0.re, fsn), rng(s0.im, fsn)};
        if (overlaps(st[0], st[1])) return SSDC_ERR_INVALID;
        for (const Range& r : st) {
            if (overlaps(r, in[7])) return SSDC_ERR_INVALID;
            if (!in_place && (overlaps(r, out[0]) || overlaps(r, out[1]))) return SSDC_ERR_INVALID;
        }
    }

    rc = setup_device_attrs();
    if (rc != SSDC_OK) return rc;

    ssdc::Problem p;
    p.x_re = x.re; p.x_im = x.im; p.A_re = A.re; p.A_im = A.im;
    p.B_re = B_t.re; p.B_im = B_t.im; p.C_re = nullptr; p.C_im = nullptr; p.dt = dt;
    p.s0_re = s0.re; p.s0_im = s0.im;
    p.y_re = nullptr; p.y_im = nullptr; p.fs_re = final_state.re; p.fs_im = final_state.im;
    p.T = dims.T; p.B = (int)dims.B; p.H = (int)dims.H; p.N = (int)dims.N; p.D = (int)dims.D;
    p.Q = chunk_size;
    p.nc = ssdc::ceil_div64(dims.T, chunk_size);
    p.drop_send_chunk = -1;
    ssdc::Workspace w = carve(workspace, dims, chunk_size);

    (void)cudaGetLastError();  // clear a stale error from unrelated work
    int launches = 0;
    if (record_event(0, stream) != SSDC_OK) return SSDC_ERR_CUDA;
    if (cudaMemsetAsync(w.status, 0, sizeof(int), stream) != cudaSuccess) return SSDC_ERR_CUDA;
    const dim3 pass_grid((unsigned)ssdc::ceil_div64((int64_t)p.N * p.D, ssdc::kPassThreads),
                         (unsigned)(p.B * p.H));
    int path = SSDC_PATH_STAGED_FP32;
    if (dims.precision == SSDC_PREC_TF32) {
        if (!ssdc::state_supported(p.N, p.D, p.Q)) return SSDC_ERR_UNSUPPORTED;
        const int n = ssdc::state_launch(p, w, stream, g_opt_plane_maps.load(std::memory_order_relaxed) != 0);
        if (n < 0) return n;
        launches += n;
        path = SSDC_PATH_STATE_TMEM;
    } else {
        if (dims.precision == SSDC_PREC_FP32) {
            ssdc::simt_launch_chunk_state(p, w, stream);
            ++launches;
        } else {
            const int n = ssdc::tc_launch_chunk_state(p, w, stream);
            if (n < 0) return n;
            launches += n;
            path = SSDC_PATH_STAGED_TF32;
        }
        record_event(launches, stream);
        ssdc::ssdc_state_pass<<<pass_grid, ssdc::kPassThreads, 0, stream>>>(p, w);
        ++launches;
    }
    record_event(launches, stream);
    if (cudaGetLastError() != cudaSuccess) return SSDC_ERR_CUDA;
    g_last_launches = launches;
    g_last_path = path;
    if (g_timing) g_timed_launches = launches;
    return SSDC_OK;
}

}  // namespace

extern "C" {

size_t ssd_complex_final_state_workspace_bytes(ssdc_dims dims, int chunk_size) {
    return check_sizes(dims, chunk_size) == SSDC_OK ? ws_bytes_for(dims, chunk_size) : 0;
}

int ssd_complex_final_state(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, const float* dt, ssdc_cin initial_state,
                            ssdc_dims dims, int chunk_size, ssdc_cout final_state, void* workspace, size_t ws_bytes,
                            cudaStream_t stream) {
    return final_state_impl(x, A, B_t, dt, initial_state, dims, chunk_size, final_state, workspace, ws_bytes,
                            stream);
}

}  // extern "C"

extern "C" {

int ssd_complex_last_path(void) { return g_last_path; }

int ssd_complex_fwd(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t, const float* dt,
                    ssdc_dims dims, int chunk_size, ssdc_cout y, ssdc_cout final_state,
                    cudaStream_t stream) {
    int rc = check_sizes(dims, chunk_size);
    if (rc != SSDC_OK) return rc;
    const size_t bytes = ws_bytes_for(dims, chunk_size);
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) return SSDC_ERR_CUDA;
    rc = ssd_complex_fwd_ws(x, A, B_t, C_t, dt, dims, chunk_size, y, final_state, ws, bytes, stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && rc == SSDC_OK) rc = SSDC_ERR_CUDA;
    return rc;
}

int ssd_complex_status(void* workspace, cudaStream_t stream) {
    if (workspace == nullptr) return SSDC_ERR_INVALID;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SSDC_ERR_CUDA;
    int status = SSDC_ERR_CUDA;
    if (cudaMemcpy(&status, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SSDC_ERR_CUDA;
    return status;
}

const char* ssd_complex_strerror(int status) {
    switch (status) {
        case SSDC_OK: return "ok";
        case SSDC_ERR_INVALID: return "invalid argument (null pointer, size <= 0, bad precision or overlapping buffers)";
        case SSDC_ERR_UNSUPPORTED: return "unsupported size (chunk_size, N or D outside the supported set)";
        case SSDC_ERR_ALIGN: return "pointer not 16-byte aligned";
        case SSDC_ERR_WORKSPACE: return "workspace null, not 256-byte aligned or too small";
        case SSDC_ERR_CUDA: return "CUDA call or kernel launch failed";
        case SSDC_ERR_TIMEOUT: return "a bounded device wait gave up";
        case SSDC_ERR_DEVICE: return "current device is not a compute capability 10.3 GPU";
        case SSDC_ERR_TOO_LARGE: return "problem needs more workspace than the static no-allocation buffer holds";
        default: return "unknown status";
    }
}

int ssd_complex_last_launch_count(void) { return g_last_launches; }

int ssd_complex_set_option(int option, int64_t value) {
    switch (option) {
        case SSDC_OPT_FUSED_CLUSTER:
            if (value != 0 && value != 1 && value != 2 && value != 4 && value != 8) return SSDC_ERR_INVALID;
            g_opt_cluster.store((int)value);
            return SSDC_OK;
        case SSDC_OPT_FUSED_PLANE_MAPS:
            if (value != 0 && value != 1) return SSDC_ERR_INVALID;
            g_opt_plane_maps.store((int)value);
            return SSDC_OK;
        case SSDC_OPT_FUSED_KERNEL:
            if (value < 0 || value > 2) return SSDC_ERR_INVALID;
            g_opt_kernel.store((int)value);
            return SSDC_OK;
        case SSDC_OPT_MIMO_FUSED:
            if (value != 0 && value != 1) return SSDC_ERR_INVALID;
            g_opt_mimo_fused.store((int)value);
            return SSDC_OK;
        case SSDC_OPT_TEST_DROP_STATE_CHUNK:
            if (value < -1) return SSDC_ERR_INVALID;
            g_opt_drop_state_chunk.store(value);
            return SSDC_OK;
        default: return SSDC_ERR_INVALID;
    }
}

int ssd_complex_timing_enable(int enable) {
    if (enable && !g_events_made) {
        for (int i = 0; i <= kMaxTimed; ++i)
            if (cudaEventCreate(&g_events[i]) != cudaSuccess) return SSDC_ERR_CUDA;
        g_events_made = true;
    }
    g_timing = enable != 0;
    g_timed_launches = 0;
    return SSDC_OK;
}

int ssd_complex_timing_read(float* ms, int n) {
    if (ms == nullptr || n < 0) return SSDC_ERR_INVALID;
    const int k = g_timed_launches;
    if (k == 0) return 0;
    if (cudaEventSynchronize(g_events[k]) != cudaSuccess) return SSDC_ERR_CUDA;
    for (int i = 0; i < k && i < n; ++i)
        if (cudaEventElapsedTime(&ms[i], g_events[i], g_events[i + 1]) != cudaSuccess) return SSDC_ERR_CUDA;
    return k;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward pass: the five kernels of csrc/ssdc_bwd.cu (chunk states and
// adjoints, the two chunk recurrences, chunk gradients, step-size gradients,
// the per-head sum of dA).

namespace {

struct BwdLayout {
    size_t S, a, R, fs, r, anchor, dA_part, total;  // byte offsets (total = size)
};

size_t pad256(size_t v) { return (v + 255) & ~size_t(255); }

// The chunk size the backward's kernels run at: the TF32 chunk kernels take
// chunks of up to 64 tokens, so a longer chunk (128, 256) is worked as 64-token
// chunks. The gradients of the scan do not depend on its chunking (only their
// rounding does), so this changes no result beyond that.
int bwd_chunk(const ssdc_dims& d, int Q) { return d.precision == SSDC_PREC_TF32 && Q > 64 ? 64 : Q; }

BwdLayout bwd_layout(const ssdc_dims& d, int Q) {
    const int64_t nc = ssdc::ceil_div64(d.T, bwd_chunk(d, Q));
    const size_t chunks = (size_t)(d.B * d.H * nc);
    const size_t states = pad256(chunks * 2 * d.N * d.D * sizeof(float));
    BwdLayout l;
    l.S = 256;  // after the status word
    l.a = l.S + states;
    l.R = l.a + pad256(chunks * 2 * sizeof(float));
    l.fs = l.R + states;
    l.r = l.fs + pad256((size_t)(d.B * d.H * d.N * d.D) * 2 * sizeof(float));
    l.anchor = l.r + pad256((size_t)(d.B * d.H * d.T) * 2 * sizeof(float));
    l.dA_part = l.anchor + pad256(chunks * 2 * sizeof(double));
    l.total = l.dA_part + pad256(chunks * 2 * sizeof(double));
    return l;
}

// The exact fp32 backward takes every size the forward does; the TF32 one
// (chunk gradients on the tensor cores) every Q the forward takes (64-token
// chunks for Q = 128, 256) with N, D multiples of 8 up to 64.
int check_bwd_sizes(const ssdc_dims& d, int Q) {
    const int rc = check_sizes(d, Q);
    if (rc != SSDC_OK) return rc;
    if (d.precision == SSDC_PREC_FP32) return SSDC_OK;
    if (d.precision == SSDC_PREC_TF32 && ssdc::bwd_tc_supported((int)d.N, (int)d.D, bwd_chunk(d, Q)))
        return SSDC_OK;
    return SSDC_ERR_UNSUPPORTED;
}

}  // namespace

extern "C" {

size_t ssd_complex_bwd_workspace_bytes(ssdc_dims dims, int chunk_size) {
    if (check_bwd_sizes(dims, chunk_size) != SSDC_OK) return 0;
    return bwd_layout(dims, chunk_size).total;
}

int ssd_complex_bwd(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t, const float* dt,
                    ssdc_cin initial_state, ssdc_cin dy, ssdc_cin d_final_state, ssdc_dims dims,
                    int chunk_size, ssdc_cout dx, ssdc_cout dA, ssdc_cout dB_t, ssdc_cout dC_t,
                    float* ddt, ssdc_cout d_initial_state, void* workspace, size_t ws_bytes,
                    cudaStream_t stream) {
    int rc = check_bwd_sizes(dims, chunk_size);
    if (rc != SSDC_OK) return rc;
    // required pointers; x.im, dy.im and dx.im may be null, the three state pairs both or neither
    const void* req[] = {x.re, A.re, A.im, B_t.re, B_t.im, C_t.re, C_t.im, dt, dy.re,
                         dx.re, dA.re, dA.im, dB_t.re, dB_t.im, dC_t.re, dC_t.im, ddt};
    for (const void* q : req)
        if (q == nullptr) return SSDC_ERR_INVALID;
    const ssdc_cin pairs[] = {initial_state, d_final_state,
                              ssdc_cin{d_initial_state.re, d_initial_state.im}};
    for (const ssdc_cin& q : pairs)
        if ((q.re == nullptr) != (q.im == nullptr) || (q.re != nullptr && q.re == q.im)) return SSDC_ERR_INVALID;
    const void* opt[] = {x.im, dy.im, dx.im, initial_state.re, initial_state.im, d_final_state.re,
                         d_final_state.im, d_initial_state.re, d_initial_state.im};
    for (const void* q : req)
        if (!aligned16(q)) return SSDC_ERR_ALIGN;
    for (const void* q : opt)
        if (!aligned16(q)) return SSDC_ERR_ALIGN;
    if (x.im == x.re || dy.im == dy.re) return SSDC_ERR_INVALID;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return SSDC_ERR_WORKSPACE;
    const BwdLayout lay = bwd_layout(dims, chunk_size);
    if (ws_bytes < lay.total) return SSDC_ERR_WORKSPACE;

    // outputs must not overlap an input, the workspace or each other
    const int64_t BTH = dims.B * dims.T * dims.H;
    const int64_t fsn = dims.B * dims.H * dims.N * dims.D;
    auto rng = [](const void* p, int64_t n) {
        const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        return Range{lo, p == nullptr ? lo : lo + (uintptr_t)n * sizeof(float)};  // null: empty
    };
    const Range in[] = {rng(x.re, BTH * dims.D), rng(x.im, BTH * dims.D), rng(A.re, dims.H),
                        rng(A.im, dims.H), rng(B_t.re, BTH * dims.N), rng(B_t.im, BTH * dims.N),
                        rng(C_t.re, BTH * dims.N), rng(C_t.im, BTH * dims.N), rng(dt, BTH),
                        rng(initial_state.re, fsn), rng(initial_state.im, fsn),
                        rng(dy.re, BTH * dims.D), rng(dy.im, BTH * dims.D),
                        rng(d_final_state.re, fsn), rng(d_final_state.im, fsn),
                        Range{reinterpret_cast<uintptr_t>(workspace),
                              reinterpret_cast<uintptr_t>(workspace) + ws_bytes}};
    const Range out[] = {rng(dx.re, BTH * dims.D), rng(dx.im, BTH * dims.D), rng(dA.re, dims.H),
                         rng(dA.im, dims.H), rng(dB_t.re, BTH * dims.N), rng(dB_t.im, BTH * dims.N),
                         rng(dC_t.re, BTH * dims.N), rng(dC_t.im, BTH * dims.N), rng(ddt, BTH),
                         rng(d_initial_state.re, fsn), rng(d_initial_state.im, fsn)};
    constexpr int kOut = sizeof(out) / sizeof(out[0]);
    for (const Range& o : out)
        for (const Range& i : in)
            if (overlaps(o, i)) return SSDC_ERR_INVALID;
    for (int i = 0; i < kOut; ++i)
        for (int j = i + 1; j < kOut; ++j)
            if (overlaps(out[i], out[j])) return SSDC_ERR_INVALID;

    rc = setup_device_attrs();
    if (rc != SSDC_OK) return rc;

    char* base = static_cast<char*>(workspace);
    ssdc::Workspace w;
    w.status = reinterpret_cast<int*>(base);
    w.S = reinterpret_cast<float*>(base + lay.S);
    w.a = reinterpret_cast<float*>(base + lay.a);
    ssdc::GradWorkspace gw;
    gw.R = reinterpret_cast<float*>(base + lay.R);
    gw.r = reinterpret_cast<float*>(base + lay.r);
    gw.anchor = reinterpret_cast<double*>(base + lay.anchor);
    gw.dA_part = reinterpret_cast<double*>(base + lay.dA_part);
    float* fs = reinterpret_cast<float*>(base + lay.fs);

    ssdc::GradProblem g;
    ssdc::Problem& p = g.f;
    p.x_re = x.re; p.x_im = x.im; p.A_re = A.re; p.A_im = A.im;
    p.B_re = B_t.re; p.B_im = B_t.im; p.C_re = C_t.re; p.C_im = C_t.im; p.dt = dt;
    p.s0_re = initial_state.re; p.s0_im = initial_state.im;
    p.y_re = nullptr; p.y_im = nullptr;  // the forward rows are not needed
    p.fs_re = fs; p.fs_im = fs + fsn;
    p.T = dims.T; p.B = (int)dims.B; p.H = (int)dims.H; p.N = (int)dims.N; p.D = (int)dims.D;
    p.Q = bwd_chunk(dims, chunk_size);
    p.nc = ssdc::ceil_div64(dims.T, p.Q);
    p.drop_send_chunk = -1;
    g.dy_re = dy.re; g.dy_im = dy.im;
    g.dfs_re = d_final_state.re; g.dfs_im = d_final_state.im;
    g.dx_re = dx.re; g.dx_im = dx.im;
    g.dA_re = dA.re; g.dA_im = dA.im;
    g.dB_re = dB_t.re; g.dB_im = dB_t.im; g.dC_re = dC_t.re; g.dC_im = dC_t.im; g.ddt = ddt;
    g.ds0_re = d_initial_state.re; g.ds0_im = d_initial_state.im;

    (void)cudaGetLastError();  // clear a stale error from unrelated work
    int launches = 0;
    if (record_event(0, stream) != SSDC_OK) return SSDC_ERR_CUDA;
    if (cudaMemsetAsync(w.status, 0, sizeof(int), stream) != cudaSuccess) return SSDC_ERR_CUDA;
    const dim3 pass_grid((unsigned)ssdc::ceil_div64((int64_t)p.N * p.D, ssdc::kPassThreads),
                         (unsigned)(p.B * p.H));
    if (dims.precision == SSDC_PREC_TF32) {
        const int n = ssdc::bwd_tc_launch_chunk_states(g, w, gw, stream);
        if (n < 0) return n;
    } else {
        ssdc::bwd_launch_chunk_states(g, w, gw, stream);
    }
    record_event(++launches, stream);
    const dim3 passes_grid(2 * pass_grid.x, pass_grid.y);  // forward and backward chains side by side
    // the passes, the TF32 chunk kernel, dt and dA are launched as programmatic dependents of the
    // kernel before each (their CTAs wait for it in griddepcontrol.wait before touching memory)
    if (ssdc::launch_dependent(ssdc::ssdc_bwd_passes, passes_grid, dim3(ssdc::kPassThreads), 0, stream, g, w, gw) !=
        cudaSuccess)
        return SSDC_ERR_CUDA;
    record_event(++launches, stream);
    if (dims.precision == SSDC_PREC_TF32) {
        const int n = ssdc::bwd_tc_launch_chunk(g, w, gw, stream);
        if (n < 0) return n;
    } else {
        ssdc::bwd_launch_chunk(g, w, gw, stream);
    }
    record_event(++launches, stream);
    const int64_t dt_blocks = ssdc::ceil_div64((int64_t)p.B * p.H * p.nc, ssdc::kBwdDtThreads / 32);
    if (ssdc::launch_dependent(ssdc::ssdc_bwd_dt, dim3((unsigned)dt_blocks), dim3(ssdc::kBwdDtThreads), 0, stream, g,
                               w, gw) != cudaSuccess)
        return SSDC_ERR_CUDA;
    record_event(++launches, stream);
    if (ssdc::launch_dependent(ssdc::ssdc_bwd_dA, dim3((unsigned)p.H), dim3(ssdc::kBwdDtThreads), 0, stream, g, w,
                               gw) != cudaSuccess)
        return SSDC_ERR_CUDA;
    record_event(++launches, stream);
    if (cudaGetLastError() != cudaSuccess) return SSDC_ERR_CUDA;
    g_last_launches = launches;
    if (g_timing) g_timed_launches = launches;
    return SSDC_OK;
}

}  // extern "C"

namespace ssdc {
void set_last_launch_count(int n) { g_last_launches = n; }
}  // namespace ssdc
