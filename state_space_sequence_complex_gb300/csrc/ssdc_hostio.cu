// Forward pass on host buffers (ssd_complex_fwd_host in include/ssdc.h): the
// inputs go to the device, the scan runs, and y and the final state come back.
// The problem is cut into pieces, groups of batch rows and, when the batch is
// small, consecutive segments of the sequence: a segment starts from the final
// state of the previous one (the initial-state form of the forward pass), so
// the scan of a row can begin before the rest of the row has arrived. The
// pieces flow through three internal streams, copy-in -> compute -> copy-out,
// with two device slots in flight, so that host-to-device copies, compute and
// device-to-host copies overlap. The host link, not the compute, then bounds
// the call.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/ssdc.h"
#include "ssdc_kernels.h"

namespace {

constexpr int kSlots = 2;
constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;
constexpr int kMaxPieces = 16;

size_t up(size_t n) { return (n + kAlign - 1) & ~(kAlign - 1); }

// Pieces: batch rows [b0, b0 + Bp) x tokens [t0, t0 + Ts). The first piece's
// copy-in and the last piece's compute and copy-out overlap nothing, so more
// pieces shorten that head and tail; each piece costs one launch (whose time is
// set by the chunk chain of a segment, not by its width) and the setup of its
// copies. Whole-batch-row groups are used when there are enough rows;
// otherwise all rows go together and the sequence is cut into segments of a
// multiple of the chunk size, so that the chunking is that of the whole scan.
struct Plan {
    int64_t Bp, nb;  // rows per group (the last may have fewer), groups
    int64_t Ts, ns;  // tokens per segment (the last may have fewer), segments
};

Plan plan_for(const ssdc_dims& d, int Q) {
    const double io = (double)d.B * d.T * d.H * (2.0 * d.D + 4.0 * d.N + 1.0 + 2.0 * d.D) * 4.0;
    const int64_t want = io <= 512e6 ? 4 : io <= 4e9 ? 8 : kMaxPieces;
    Plan p;
    if (d.B >= want) {
        p.Bp = (d.B + want - 1) / want;
        p.nb = (d.B + p.Bp - 1) / p.Bp;
        p.Ts = d.T;
        p.ns = 1;
    } else {
        p.Bp = d.B;
        p.nb = 1;
        const int64_t nc = (d.T + Q - 1) / Q;
        const int64_t per = (nc + want - 1) / want;  // chunks per segment
        p.Ts = per * Q < d.T ? per * Q : d.T;
        p.ns = (d.T + p.Ts - 1) / p.Ts;
    }
    return p;
}

// Byte offsets of one slot's buffers (a piece of Bp x Ts x H).
struct Slot {
    size_t x, Bt, Ct, dt, A, y, fs, ws, bytes, ws_bytes;
};

Slot slot_for(const ssdc_dims& d, const Plan& p, int Q) {
    Slot s;
    const size_t tok = (size_t)p.Bp * (size_t)p.Ts * (size_t)d.H;
    size_t o = 0;
    s.x = o;
    o += 2 * up(tok * d.D * 4);
    s.Bt = o;
    o += 2 * up(tok * d.N * 4);
    s.Ct = o;
    o += 2 * up(tok * d.N * 4);
    s.dt = o;
    o += up(tok * 4);
    s.A = o;
    o += 2 * up((size_t)d.H * 4);
    s.y = o;
    o += 2 * up(tok * d.D * 4);
    s.fs = o;
    o += 2 * up((size_t)p.Bp * d.H * d.N * d.D * 4);
    s.ws = o;
    ssdc_dims pd = d;
    pd.B = p.Bp;
    pd.T = p.Ts;
    s.ws_bytes = ssd_complex_fwd_workspace_bytes(pd, Q);
    o += up(s.ws_bytes);
    s.bytes = o;
    return s;
}

// Internal streams and events, one set per device, made on first use.
struct Pipe {
    std::mutex mu;
    bool made = false;
    cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in_done[kSlots] = {}, comp_done[kSlots] = {}, out_done[kSlots] = {};
    int* status = nullptr;  // pinned host copy of each piece's device status word
};
Pipe g_pipes[kMaxDevices];

int make_pipe(Pipe& p) {
    if (p.made) return SSDC_OK;
    const unsigned f = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, f) != cudaSuccess || cudaEventCreateWithFlags(&p.end, f) != cudaSuccess)
        return SSDC_ERR_CUDA;
    for (int k = 0; k < kSlots; ++k)
        if (cudaEventCreateWithFlags(&p.in_done[k], f) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.comp_done[k], f) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.out_done[k], f) != cudaSuccess)
            return SSDC_ERR_CUDA;
    if (cudaHostAlloc(&p.status, kMaxPieces * sizeof(int), cudaHostAllocDefault) != cudaSuccess) return SSDC_ERR_CUDA;
    p.made = true;
    return SSDC_OK;
}

// rows x width bytes between row-pitched buffers.
bool copy2d(void* dst, size_t dpitch, const void* src, size_t spitch, size_t width, size_t rows, cudaMemcpyKind kind,
            cudaStream_t st) {
    if (rows == 0 || width == 0) return true;
    if (rows == 1 || (dpitch == width && spitch == width))
        return cudaMemcpyAsync(dst, src, width * rows, kind, st) == cudaSuccess;
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, st) == cudaSuccess;
}

// After a failure with work already enqueued: let it drain, so that no copy
// still reads the caller's buffers or the scratch when the call returns.
int drain(Pipe& p, int rc) {
    cudaStreamSynchronize(p.in);
    cudaStreamSynchronize(p.comp);
    cudaStreamSynchronize(p.out);
    return rc;
}

}  // namespace

extern "C" {

size_t ssd_complex_fwd_host_scratch_bytes(ssdc_dims dims, int chunk_size) {
    if (ssd_complex_fwd_supported(dims, chunk_size) != SSDC_OK) return 0;
    return kSlots * slot_for(dims, plan_for(dims, chunk_size), chunk_size).bytes;
}

int ssd_complex_fwd_host(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t, const float* dt, ssdc_dims dims,
                         int chunk_size, ssdc_cout y, ssdc_cout final_state, void* dev_scratch, size_t scratch_bytes,
                         cudaStream_t stream) {
    int rc = ssd_complex_fwd_supported(dims, chunk_size);
    if (rc != SSDC_OK) return rc;
    const void* ins[] = {x.re, x.im, A.re, A.im, B_t.re, B_t.im, C_t.re, C_t.im, dt, y.re, y.im,
                         final_state.re, final_state.im};
    for (int i = 0; i < 13; ++i)
        if (ins[i] == nullptr && i != 1) return SSDC_ERR_INVALID;  // only x.im may be null: a real x
    const bool real_x = x.im == nullptr;
    if (x.im == x.re) return SSDC_ERR_INVALID;
    {  // host outputs must not overlap the inputs or each other
        const size_t tok = (size_t)dims.B * dims.T * dims.H;
        const size_t ib[] = {tok * dims.D * 4, tok * dims.D * 4, (size_t)dims.H * 4, (size_t)dims.H * 4,
                             tok * dims.N * 4, tok * dims.N * 4, tok * dims.N * 4, tok * dims.N * 4, tok * 4};
        const size_t ob[] = {tok * dims.D * 4, tok * dims.D * 4, (size_t)(dims.B * dims.H * dims.N * dims.D) * 4,
                             (size_t)(dims.B * dims.H * dims.N * dims.D) * 4};
        const void* outs[] = {y.re, y.im, final_state.re, final_state.im};
        auto hit = [](const void* a, size_t na, const void* b, size_t nb) {
            const uintptr_t u = reinterpret_cast<uintptr_t>(a), v = reinterpret_cast<uintptr_t>(b);
            return u < v + nb && v < u + na;
        };
        for (int o = 0; o < 4; ++o) {
            for (int i = 0; i < 9; ++i)
                if (ins[i] != nullptr && hit(outs[o], ob[o], ins[i], ib[i])) return SSDC_ERR_INVALID;
            for (int j = o + 1; j < 4; ++j)
                if (hit(outs[o], ob[o], outs[j], ob[j])) return SSDC_ERR_INVALID;
        }
    }
    const Plan plan = plan_for(dims, chunk_size);
    const Slot sl = slot_for(dims, plan, chunk_size);
    const int npieces = (int)(plan.nb * plan.ns);
    if (dev_scratch == nullptr || (reinterpret_cast<uintptr_t>(dev_scratch) & (kAlign - 1)) != 0 ||
        scratch_bytes < kSlots * sl.bytes)
        return SSDC_ERR_WORKSPACE;
    if (npieces > kMaxPieces) return SSDC_ERR_INVALID;  // unreachable with plan_for's bounds
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSDC_ERR_CUDA;
    Pipe& pipe = g_pipes[dev];
    std::lock_guard<std::mutex> lock(pipe.mu);
    rc = make_pipe(pipe);
    if (rc != SSDC_OK) return rc;

    const int64_t T = dims.T, H = dims.H, N = dims.N, D = dims.D;
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
    // everything starts after the caller's earlier work on `stream`
    if (cudaEventRecord(pipe.start, stream) != cudaSuccess || cudaStreamWaitEvent(pipe.in, pipe.start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(pipe.comp, pipe.start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(pipe.out, pipe.start, 0) != cudaSuccess)
        return SSDC_ERR_CUDA;

    int launches = 0, piece = 0;
    for (int64_t bi = 0; bi < plan.nb; ++bi) {
        for (int64_t si = 0; si < plan.ns; ++si, ++piece) {
            const int k = piece % kSlots;
            char* s = static_cast<char*>(dev_scratch) + (size_t)k * sl.bytes;
            const int64_t b0 = bi * plan.Bp, t0 = si * plan.Ts;
            const int64_t Bp = dims.B - b0 < plan.Bp ? dims.B - b0 : plan.Bp;
            const int64_t Ts = T - t0 < plan.Ts ? T - t0 : plan.Ts;
            const bool first = si == 0, last = si == plan.ns - 1;
            const size_t tokp = (size_t)(Bp * Ts * H);
            float* dx_re = reinterpret_cast<float*>(s + sl.x);
            float* dx_im = reinterpret_cast<float*>(s + sl.x + up(tokp * D * 4));
            float* dB_re = reinterpret_cast<float*>(s + sl.Bt);
            float* dB_im = reinterpret_cast<float*>(s + sl.Bt + up(tokp * N * 4));
            float* dC_re = reinterpret_cast<float*>(s + sl.Ct);
            float* dC_im = reinterpret_cast<float*>(s + sl.Ct + up(tokp * N * 4));
            float* ddt = reinterpret_cast<float*>(s + sl.dt);
            float* dA_re = reinterpret_cast<float*>(s + sl.A);
            float* dA_im = reinterpret_cast<float*>(s + sl.A + up((size_t)H * 4));
            float* dy_re = reinterpret_cast<float*>(s + sl.y);
            float* dy_im = reinterpret_cast<float*>(s + sl.y + up(tokp * D * 4));
            const size_t fsb = up((size_t)plan.Bp * H * N * D * 4);
            float* dfs_re = reinterpret_cast<float*>(s + sl.fs);
            float* dfs_im = reinterpret_cast<float*>(s + sl.fs + fsb);
            // the previous segment of these rows left its final state in the other slot
            const char* ps = static_cast<const char*>(dev_scratch) + (size_t)(1 - k) * sl.bytes;
            const float* ds0_re = first ? nullptr : reinterpret_cast<const float*>(ps + sl.fs);
            const float* ds0_im = first ? nullptr : reinterpret_cast<const float*>(ps + sl.fs + fsb);

            // copy-in, once the slot's previous piece has been copied out: Bp rows of Ts tokens
            if (piece >= kSlots && cudaStreamWaitEvent(pipe.in, pipe.out_done[k], 0) != cudaSuccess)
                return drain(pipe, SSDC_ERR_CUDA);
            const size_t tk0 = (size_t)((b0 * T + t0) * H);            // first (b, t, h) of the piece
            const size_t hrow = (size_t)(T * H), drow = (size_t)(Ts * H);  // tokens per host / device row
            bool ok = copy2d(dx_re, drow * D * 4, x.re + tk0 * D, hrow * D * 4, drow * D * 4, Bp, h2d, pipe.in) &&
                      (real_x ||
                       copy2d(dx_im, drow * D * 4, x.im + tk0 * D, hrow * D * 4, drow * D * 4, Bp, h2d, pipe.in)) &&
                      copy2d(dB_re, drow * N * 4, B_t.re + tk0 * N, hrow * N * 4, drow * N * 4, Bp, h2d, pipe.in) &&
                      copy2d(dB_im, drow * N * 4, B_t.im + tk0 * N, hrow * N * 4, drow * N * 4, Bp, h2d, pipe.in) &&
                      copy2d(dC_re, drow * N * 4, C_t.re + tk0 * N, hrow * N * 4, drow * N * 4, Bp, h2d, pipe.in) &&
                      copy2d(dC_im, drow * N * 4, C_t.im + tk0 * N, hrow * N * 4, drow * N * 4, Bp, h2d, pipe.in) &&
                      copy2d(ddt, drow * 4, dt + tk0, hrow * 4, drow * 4, Bp, h2d, pipe.in) &&
                      cudaMemcpyAsync(dA_re, A.re, H * 4, h2d, pipe.in) == cudaSuccess &&
                      cudaMemcpyAsync(dA_im, A.im, H * 4, h2d, pipe.in) == cudaSuccess &&
                      cudaEventRecord(pipe.in_done[k], pipe.in) == cudaSuccess &&
                      cudaStreamWaitEvent(pipe.comp, pipe.in_done[k], 0) == cudaSuccess;
            if (!ok) return drain(pipe, SSDC_ERR_CUDA);

            // compute on the piece, a dense (Bp, Ts, H) problem; a later segment starts from the
            // previous one's final state (the compute stream runs the pieces in order)
            ssdc_dims pd = dims;
            pd.B = Bp;
            pd.T = Ts;
            rc = ssd_complex_fwd_init(ssdc_cin{dx_re, real_x ? nullptr : dx_im}, ssdc_cin{dA_re, dA_im},
                                      ssdc_cin{dB_re, dB_im},
                                      ssdc_cin{dC_re, dC_im}, ddt, ssdc_cin{ds0_re, ds0_im}, pd, chunk_size,
                                      ssdc_cout{dy_re, dy_im}, ssdc_cout{dfs_re, dfs_im}, s + sl.ws, sl.ws_bytes,
                                      pipe.comp);
            if (rc < 0) return drain(pipe, rc);
            launches += ssd_complex_last_launch_count();

            // copy-out: y of the piece, and the final state after the rows' last segment
            const size_t srow0 = (size_t)(b0 * H);  // first (b, h) of the final state
            const size_t fsn = (size_t)Bp * H * N * D;
            ok = cudaEventRecord(pipe.comp_done[k], pipe.comp) == cudaSuccess &&
                 cudaStreamWaitEvent(pipe.out, pipe.comp_done[k], 0) == cudaSuccess &&
                 // the piece's device status (the slot's next piece resets it only after out_done)
                 cudaMemcpyAsync(pipe.status + piece, s + sl.ws, 4, d2h, pipe.out) == cudaSuccess &&
                 copy2d(y.re + tk0 * D, hrow * D * 4, dy_re, drow * D * 4, drow * D * 4, Bp, d2h, pipe.out) &&
                 copy2d(y.im + tk0 * D, hrow * D * 4, dy_im, drow * D * 4, drow * D * 4, Bp, d2h, pipe.out) &&
                 (!last ||
                  (cudaMemcpyAsync(final_state.re + srow0 * N * D, dfs_re, fsn * 4, d2h, pipe.out) == cudaSuccess &&
                   cudaMemcpyAsync(final_state.im + srow0 * N * D, dfs_im, fsn * 4, d2h, pipe.out) == cudaSuccess)) &&
                 cudaEventRecord(pipe.out_done[k], pipe.out) == cudaSuccess;
            if (!ok) return drain(pipe, SSDC_ERR_CUDA);
        }
    }
    ssdc::set_last_launch_count(launches);
    // the caller's stream continues once every piece is back; the call returns when the
    // outputs are in the host buffers, with the device status of every piece
    if (cudaEventRecord(pipe.end, pipe.out) != cudaSuccess || cudaStreamWaitEvent(stream, pipe.end, 0) != cudaSuccess ||
        cudaStreamSynchronize(pipe.out) != cudaSuccess)
        return drain(pipe, SSDC_ERR_CUDA);
    for (int i = 0; i < npieces; ++i)
        if (pipe.status[i] != SSDC_OK) return pipe.status[i];
    return SSDC_OK;
}

}  // extern "C"
