/*
 * ssdc.h -- C ABI of libssdc.so: forward pass of the complex-valued chunkwise
 * SSD scan (the core scan of a Mamba-3 block) on one GB300 (sm_103a), and
 * its backward pass (ssd_complex_bwd, at the end of this header).
 *
 * The operation (page "Extending -- SSM variants & Triton kernels", Path A,
 * Step 1, the naive O(T) scan and the discretisation it calls; landing page
 * "03 Chunkwise SSD" for the chunked decomposition):
 *
 *   A_bar[b,t,h] = exp(softplus(dt[b,t,h]) * A[h])            (complex)
 *   s_t = A_bar_t * s_{t-1} + B_t (outer) x_t,   s_{-1} = 0     s: (N, D)
 *   y_t = sum_n C_t[n] * s_t[n, :]
 *
 * computed chunk by chunk with chunk size Q (the pages' chunk_size):
 *   Acs     inclusive in-chunk cumulative sum of softplus(dt) * A
 *   L[l,s]  = exp(Acs[l] - Acs[s]) for l >= s, else 0
 *   Y_diag  = (C B^T o L) X
 *   S_loc   = B^T (dec o X),  dec[s] = exp(Acs[Q-1] - Acs[s])
 *   S_in[c+1] = exp(Acs_c[Q-1]) S_in[c] + S_loc[c],  S_in[0] = 0
 *   y       = Y_diag + (C o exp(Acs)) S_in[c]
 *
 * Re(y), the real output the pages' chunkwise function returns, is the real
 * plane of y: no separate buffer is written for it.
 *
 * Layout. Every complex array is PLANAR: two separate float32 device arrays
 * (real plane, imaginary plane), each dense row-major over the shape given:
 *   x      (B, T, H, D)        A (H)          dt (B, T, H)  (real)
 *   B_t    (B, T, H, N)        C_t (B, T, H, N)
 *   y      (B, T, H, D)        final_state (B, H, N, D)
 * All pointers are device pointers, 16-byte aligned. Outputs must not
 * overlap inputs or each other.
 *
 * Real x. x.im may be NULL: x is then real (its imaginary plane is zero and
 * is not read), as in the model, where x is a real H*D slice of the input
 * projection. Every path and entry point accepts it; y and the state stay
 * complex. Any other NULL pointer is SSDC_ERR_INVALID.
 *
 * Ownership. The caller owns every buffer; the library keeps no pointer after
 * a call returns. Work is enqueued on `stream` and runs asynchronously: inputs
 * must stay unchanged, and outputs unread, until the stream reaches that point.
 *
 * Errors. Every entry point returns an int status: 0 (SSDC_OK) or a negative
 * SSDC_ERR_* code. Argument errors are detected on the host before anything
 * is enqueued; nothing aborts, throws or falls back to another path. Errors
 * detected on the device (a bounded wait that gave up) are recorded in the
 * workspace and reported by ssd_complex_status().
 *
 * Precision. SSDC_PREC_TF32 runs the chunk contractions on the tcgen05 tensor
 * cores with TF32 operands and fp32 accumulation, in one fused launch: a
 * kernel whose CTAs each walk whole sequences with the chunk state held in
 * tensor memory (every supported size), or, for fewer sequences than SMs at
 * Q = N = D = 64, one that deals each sequence's chunks over the CTAs of a
 * thread-block cluster and passes the states through distributed shared
 * memory (ssd_complex_last_path() reports which ran). SSDC_PREC_TF32_STAGED
 * is the same arithmetic as three kernels (chunk states, state pass, chunk
 * outputs) with the per-chunk states staged in the workspace. SSDC_PREC_FP32
 * runs every step in exact fp32 on the SIMT cores (the checking variant),
 * staged the same way. The state pass between chunks is fp32 in all three.
 */
#ifndef SSDC_H
#define SSDC_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSDC_OK 0
#define SSDC_ERR_INVALID (-1)     /* null pointer, size <= 0, bad precision, overlap */
#define SSDC_ERR_UNSUPPORTED (-2) /* Q, N or D outside the supported set */
#define SSDC_ERR_ALIGN (-3)       /* a pointer not 16-byte aligned */
#define SSDC_ERR_WORKSPACE (-4)   /* workspace null, misaligned or too small */
#define SSDC_ERR_CUDA (-5)        /* a CUDA call or launch failed */
#define SSDC_ERR_TIMEOUT (-6)     /* a bounded device wait gave up */
#define SSDC_ERR_DEVICE (-7)      /* the current device is not sm_103 */
#define SSDC_ERR_TOO_LARGE (-8)   /* needs more scratch than the static buffer holds */

#define SSDC_PREC_TF32 0
#define SSDC_PREC_FP32 1
#define SSDC_PREC_TF32_STAGED 2

/* Problem sizes: batch B, sequence length T, heads H, complex state size N,
 * complex head dimension D; precision is one of SSDC_PREC_*. */
typedef struct {
    int64_t B, T, H, N, D;
    int32_t precision;
} ssdc_dims;

/* A planar complex input / output: real plane and imaginary plane. */
typedef struct {
    const float *re, *im;
} ssdc_cin;
typedef struct {
    float *re, *im;
} ssdc_cout;

/*
 * Supported sizes.
 *   SSDC_PREC_FP32:        chunk_size in {16, 32, 64, 128, 256};
 *                          N and D multiples of 8 in [8, 64].
 *   SSDC_PREC_TF32:        the same sets.
 *   SSDC_PREC_TF32_STAGED: chunk_size in {32, 64, 128, 256}; N = D = 64.
 * T need not be a multiple of chunk_size: the last chunk is partial.
 */
int ssd_complex_fwd_supported(ssdc_dims dims, int chunk_size);

/* Bytes of device workspace ssd_complex_fwd_ws needs for these sizes (0 on
 * invalid or unsupported sizes). It holds a device status word and, on the
 * staged paths, the per-chunk states and decays. */
size_t ssd_complex_fwd_workspace_bytes(ssdc_dims dims, int chunk_size);

/*
 * Forward pass with a caller-provided workspace (device memory, 256-byte
 * aligned, at least ssd_complex_fwd_workspace_bytes() bytes). The workspace's
 * contents need no initialisation; the call resets its status word. Calls
 * that share one workspace must be ordered on the stream.
 *
 *   x, A, B_t, C_t, dt   inputs (see Layout)
 *   dims, chunk_size     sizes, precision and the chunk length Q
 *   y                    output (B,T,H,D) complex; y.re is Re(y)
 *   final_state          output (B,H,N,D) complex, the state after t = T-1
 *   stream               CUDA stream (0 = legacy default stream)
 */
int ssd_complex_fwd_ws(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t,
                       const float *dt, ssdc_dims dims, int chunk_size,
                       ssdc_cout y, ssdc_cout final_state, void *workspace,
                       size_t ws_bytes, cudaStream_t stream);

/*
 * Forward pass from a given initial state: s_{-1} = initial_state instead of
 * zero. The pages' scan starts from a zero state; this form continues a
 * sequence from the state an earlier call returned, so that a long sequence
 * can be processed in segments: the segment [T1, T) started from the final
 * state of [0, T1) gives the y rows and the final state of the whole scan, up
 * to rounding.
 *
 *   initial_state  (B,H,N,D) complex, planar device arrays, 16-byte aligned.
 *                  Both planes null means a zero initial state (the call is
 *                  then ssd_complex_fwd_ws). It may be the final_state buffer
 *                  itself (an in-place update, plane for plane); otherwise it
 *                  must not overlap an output or the workspace.
 * The other arguments, the workspace, the errors and the precisions are those
 * of ssd_complex_fwd_ws; one null plane is SSDC_ERR_INVALID.
 */
int ssd_complex_fwd_init(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t,
                         const float *dt, ssdc_cin initial_state, ssdc_dims dims,
                         int chunk_size, ssdc_cout y, ssdc_cout final_state,
                         void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * Forward pass with bfloat16 activations: x, B_t and C_t are planar bfloat16
 * arrays (the layouts of ssd_complex_fwd_ws, 2 bytes an element); A, dt, the
 * initial and final states and y stay fp32, and so does every sum and the state
 * (the pages train with BF16 activations around a complex64 state): x, B_t
 * and C_t take 768 bytes per token-head instead of 1536 (1300 in all, instead
 * of 2068, at N = D = 64 and T = 2048). The scan is the same operation on the inputs'
 * values: C B^T multiplies the bfloat16 values as they are (tensor-core BF16
 * products, exact, fp32 sums); every other product takes them as exact fp32
 * (TF32) values, as the TF32 path does its fp32 inputs.
 *
 *   x, B_t, C_t     planar bfloat16, 16-byte aligned; x.im may be null (a real x)
 *   initial_state   as for ssd_complex_fwd_init (both planes null: zero)
 *   dims.precision  must be SSDC_PREC_TF32; N, D multiples of 8 in [8, 64],
 *                   chunk_size in {16, 32, 64, 128, 256} (else SSDC_ERR_UNSUPPORTED)
 * The other arguments, the workspace (ssd_complex_fwd_workspace_bytes), the
 * overlap rules and the errors are those of ssd_complex_fwd_ws. One launch, the
 * fused kernel with the state in tensor memory.
 */
typedef struct {
    const uint16_t *re, *im;
} ssdc_cin_bf16;
int ssd_complex_fwd_bf16(ssdc_cin_bf16 x, ssdc_cin A, ssdc_cin_bf16 B_t, ssdc_cin_bf16 C_t,
                         const float *dt, ssdc_cin initial_state, ssdc_dims dims,
                         int chunk_size, ssdc_cout y, ssdc_cout final_state,
                         void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * Forward pass followed by the MIMO head mixer (landing page, "02 MIMO Mixer":
 * a fully connected mixer across the H SSM heads, H x H, identity-initialised,
 * applied to the Re(y) the block consumes):
 *   out[b, t, g, d] = sum_h mix[g * H + h] Re(y)[b, t, h, d],
 * the same matrix for every feature d. No y.im is written. Two ways, chosen by
 * SSDC_OPT_MIMO_FUSED:
 *   0 (default)  the scan (the fused kernel the library picks, as for
 *                ssd_complex_fwd_ws) writes Re(y) into `out`, then a second
 *                kernel mixes each token's H x D block in place (it reads and
 *                writes `out` once: 8 H D bytes a token), launched as a
 *                programmatic dependent of the scan. Two launches.
 *   1            the mixer in the epilogue of the kernel with the state in
 *                tensor memory: the tiles of Re(y) of one batch row and 64-token
 *                tile from all H heads meet in `out` and are counted there;
 *                once all H are stored, the CTA of head h mixes the h-th 1/H of
 *                the tile's tokens in place. A CTA mixes its ready shares after
 *                each tile it stores, and waits (bounded) only for the shares
 *                still open after its sequence's last tile. One launch; slower
 *                on a GB300 (the exchange lands on the chunk loop's critical path).
 *
 *   mix             (H, H) fp32 device array, row g = output head g; required
 *   out             (B, T, H, D) fp32 device array, 16-byte aligned
 *   initial_state   as for ssd_complex_fwd_init (both planes null: zero)
 *   dims.precision  SSDC_PREC_TF32; H <= 16; N, D multiples of 8 in [8, 64];
 *                   chunk_size 16, 32 or 64 (else SSDC_ERR_UNSUPPORTED)
 *   workspace       ssd_complex_fwd_mimo_workspace_bytes() bytes (a status word
 *                   and one counter per batch row and 64-token tile, which the
 *                   fused epilogue uses), either way
 * The other arguments, the overlap rules and the errors are those of
 * ssd_complex_fwd_ws.
 */
size_t ssd_complex_fwd_mimo_workspace_bytes(ssdc_dims dims, int chunk_size);
int ssd_complex_fwd_mimo(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t, const float *dt,
                         const float *mix, ssdc_cin initial_state, ssdc_dims dims, int chunk_size,
                         float *out, ssdc_cout final_state, void *workspace, size_t ws_bytes,
                         cudaStream_t stream);

/*
 * Joining segments of a sequence split in time (across ranks or calls). The
 * state pass between chunks (landing page "03 Chunkwise SSD", the STATE line:
 * a state carried forward is multiplied by the exponential of the accumulated
 * log-decay) applied to whole segments: a segment with total decay a_seg and
 * end state S_seg (scanned from a zero state) takes the incoming state S_in to
 * a_seg S_in + S_seg, and consecutive segments compose as
 *   (a2, S2) o (a1, S1) = (a2 a1, a2 S1 + S2).
 * A rank that holds segment r of T therefore computes the state its segment
 * leaves from zero (ssd_complex_final_state), gathers the (a_seg, S_seg) of
 * the segments before it, combines them in order into its incoming state, and
 * scans its segment from that state (ssd_complex_fwd_init) for its rows of y
 * and its final state.
 *
 * ssd_complex_segment_decay: a_seg[b,h] = exp(sum_t softplus(dt[b,t,h]) A[h])
 * over the T tokens of dt (B,T,H); the sum and the exponential in fp64.
 *   A       (H) complex;  dt (B,T,H);  a_seg  output (B,H) complex
 * Uses dims.B, T, H; pointers 16-byte aligned device pointers; one launch on
 * `stream`. Errors as for ssd_complex_fwd_ws.
 *
 * ssd_complex_state_combine: s_out = a s_in + s_add, per (b, h) with a[b,h]:
 *   a       (B,H) complex;  s_in, s_add, s_out (B,H,N,D) complex
 *   s_in    both planes NULL for a zero incoming state (s_out = s_add)
 * s_out may be s_in or s_add (element-wise, in place). Uses dims.B, H, N, D;
 * one launch on `stream`.
 */
int ssd_complex_segment_decay(ssdc_cin A, const float *dt, ssdc_dims dims,
                              ssdc_cout a_seg, cudaStream_t stream);
int ssd_complex_state_combine(ssdc_cin a, ssdc_cin s_in, ssdc_cin s_add, ssdc_dims dims,
                              ssdc_cout s_out, cudaStream_t stream);

/*
 * The state a scan leaves behind, without its rows of y: the chunked
 * decomposition's state side alone (landing page "03 Chunkwise SSD": the
 * per-chunk states B^T (decay o X), decay[s] = exp(Acs[Q-1] - Acs[s]), and the
 * pass between chunks, the STATE line), from the given initial state. It gives
 * the final state of ssd_complex_fwd_init on the same arguments, reading only
 * x, B_t and dt (1028 instead of 2068 bytes per token-head at N = D = 64):
 * the end state S_seg of a segment scanned from zero, for the joining above,
 * before the incoming states are known.
 *   x, A, B_t, dt, dims, chunk_size   as for ssd_complex_fwd_ws (x.im may be
 *                   NULL: a real x); the sizes each precision takes are the
 *                   same as for the forward pass
 *   initial_state   as for ssd_complex_fwd_init (both planes NULL: zero); it
 *                   may be final_state itself (updated in place)
 *   final_state     output (B,H,N,D) complex
 *   workspace       ssd_complex_final_state_workspace_bytes(dims, chunk_size)
 *                   bytes, 256-byte aligned; a device-side error is read with
 *                   ssd_complex_status(workspace, stream)
 * SSDC_PREC_TF32 runs one launch with the tensor-memory forward kernel's tiles
 * and products (its final state bit for bit); SSDC_PREC_FP32 and
 * SSDC_PREC_TF32_STAGED run the staged path's chunk-state and state-pass
 * launches. Asynchronous on `stream`; errors as for ssd_complex_fwd_ws.
 */
size_t ssd_complex_final_state_workspace_bytes(ssdc_dims dims, int chunk_size);
int ssd_complex_final_state(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, const float *dt,
                            ssdc_cin initial_state, ssdc_dims dims, int chunk_size,
                            ssdc_cout final_state, void *workspace, size_t ws_bytes,
                            cudaStream_t stream);

/*
 * Forward pass that allocates its workspace on `stream` (cudaMallocAsync /
 * cudaFreeAsync, stream-ordered). A device-side error cannot be queried after
 * it returns; use the _ws form with ssd_complex_status() to read one.
 */
int ssd_complex_fwd(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t,
                    const float *dt, ssdc_dims dims, int chunk_size, ssdc_cout y,
                    ssdc_cout final_state, cudaStream_t stream);

/* Synchronises `stream`, then returns the device status recorded in
 * `workspace` by the last call that used it (SSDC_OK or SSDC_ERR_TIMEOUT), or
 * SSDC_ERR_CUDA if the stream reports an error. */
int ssd_complex_status(void *workspace, cudaStream_t stream);

/* Static, NUL-terminated description of a status code. */
const char *ssd_complex_strerror(int status);

/* Number of kernel launches the last successful forward call enqueued on its
 * stream (from the calling thread). */
int ssd_complex_last_launch_count(void);

/* The path the last successful forward call (or ssd_complex_final_state)
 * took, from the calling thread, or -1 before the first:
 *   SSDC_PATH_STAGED_FP32    exact fp32: chunk states, state pass, chunk outputs
 *                            (the first two for ssd_complex_final_state)
 *   SSDC_PATH_STAGED_TF32    the same launches on the tensor cores
 *   SSDC_PATH_FUSED_CLUSTER  one launch; each sequence's chunks dealt over the
 *                            CTAs of a thread-block cluster, chunk states passed
 *                            through distributed shared memory (Q = N = D = 64)
 *   SSDC_PATH_FUSED_TMEM     one launch; one CTA per SM walks whole sequences,
 *                            the chunk state held in tensor memory (Q = 16 to
 *                            256; N, D multiples of 8 up to 64)
 *   SSDC_PATH_STATE_TMEM     ssd_complex_final_state at SSDC_PREC_TF32: one
 *                            launch, the state side of SSDC_PATH_FUSED_TMEM
 * SSDC_PREC_TF32 takes SSDC_PATH_FUSED_TMEM wherever the sequences fill the GPU
 * one CTA each and SSDC_PATH_FUSED_CLUSTER for fewer sequences at
 * Q = N = D = 64. */
#define SSDC_PATH_STAGED_FP32 0
#define SSDC_PATH_STAGED_TF32 1
#define SSDC_PATH_FUSED_CLUSTER 2
#define SSDC_PATH_FUSED_TMEM 3
#define SSDC_PATH_STATE_TMEM 4
int ssd_complex_last_path(void);

/*
 * Per-kernel timing (instrumentation for benchmarks). While enabled, every
 * forward call records a CUDA event on its stream before its first launch and
 * after each launch. ssd_complex_timing_read() waits for the last call's
 * events and writes the device time of each of its launches, in
 * milliseconds, to ms[0 .. min(n, launches)); it returns the launch count or
 * a negative status. Process-wide state: do not use from several threads.
 */
int ssd_complex_timing_enable(int enable);
int ssd_complex_timing_read(float *ms, int n);

/*
 * Process-wide options (tuning and tests; normal use needs none of them).
 * Each call sets one option for every later forward call, from any thread;
 * returns SSDC_OK, or SSDC_ERR_INVALID for an unknown option or value. The
 * library reads no environment variables.
 *
 *   SSDC_OPT_FUSED_CLUSTER        cluster size of the fused TF32 kernel:
 *                                 0 = chosen per call (default), or 1, 2, 4, 8
 *   SSDC_OPT_FUSED_PLANE_MAPS     1 (default): one tensor map fetches both planes
 *                                 of a tensor where it can; 0: one map per plane
 *   SSDC_OPT_FUSED_KERNEL         fused TF32 kernel: 0 = chosen per call
 *                                 (default), 1 = the cluster kernel, 2 = the
 *                                 kernel with the state in tensor memory
 *   SSDC_OPT_MIMO_FUSED           ssd_complex_fwd_mimo: 0 (default) = the scan writes
 *                                 Re(y) into the output, then a separate kernel mixes
 *                                 it in place; 1 = the mixer fused into the scan's
 *                                 epilogue (one launch)
 *   SSDC_OPT_TEST_DROP_STATE_CHUNK  test hook, -1 = off (default): the fused
 *                                 kernel does not send the state of this chunk
 *                                 index to the next CTA, whose bounded wait then
 *                                 gives up and records SSDC_ERR_TIMEOUT
 */
#define SSDC_OPT_FUSED_CLUSTER 1
#define SSDC_OPT_FUSED_PLANE_MAPS 2
#define SSDC_OPT_TEST_DROP_STATE_CHUNK 3
#define SSDC_OPT_FUSED_KERNEL 4
#define SSDC_OPT_MIMO_FUSED 5
int ssd_complex_set_option(int option, int64_t value);

/*
 * Forward pass that allocates nothing, for callers that cannot allocate
 * device memory when they run the scan (code running inside a memory-pool or
 * allocator hook, latency-critical paths that forbid allocator calls, or
 * embedders with a fixed memory budget). There is no counterpart on the pages;
 * it is an operational variant of the staged path.
 *
 * It runs the staged path (precision SSDC_PREC_FP32 or SSDC_PREC_TF32_STAGED;
 * anything else is SSDC_ERR_UNSUPPORTED) with its workspace in a static device
 * array of SSDC_NOALLOC_SCRATCH_BYTES that the library holds on every GPU that
 * loads it, for the life of the process. Problems whose workspace
 * (ssd_complex_fwd_workspace_bytes) exceeds it return SSDC_ERR_TOO_LARGE
 * before anything is enqueued. Arguments, layout and outputs are those of
 * ssd_complex_fwd_ws; it calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it for the life of the process; make that
 * first call before any stream capture, and do not use the library across a
 * device reset (cudaDeviceReset), which would leave that address stale.
 * All calls share the one array and leave their chunk states in it: calls
 * whose work may overlap on the GPU (different streams, or threads without
 * ordering) race on it and must be serialised by the caller. The array needs
 * no clearing between calls: each call clears the status word at its start,
 * and every chunk state is written before it is read.
 *
 * A device-side error (a bounded wait that gave up) is recorded in the
 * array's status word; ssd_complex_noalloc_status() reads it.
 */
#define SSDC_NOALLOC_SCRATCH_BYTES ((size_t)32 * 1024 * 1024 + (size_t)64 * 1024)
int ssd_complex_fwd_noalloc(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t,
                            const float *dt, ssdc_dims dims, int chunk_size,
                            ssdc_cout y, ssdc_cout final_state, cudaStream_t stream);

/* Synchronises `stream`, then returns the device status the last
 * ssd_complex_fwd_noalloc call on the current device recorded (SSDC_OK or
 * SSDC_ERR_TIMEOUT), or SSDC_ERR_CUDA if the stream reports an error. It
 * allocates nothing: the status word is read from the static array with
 * cudaMemcpyFromSymbol. */
int ssd_complex_noalloc_status(cudaStream_t stream);

/*
 * Forward pass on HOST buffers: the library copies the inputs to the device,
 * runs the forward pass of ssd_complex_fwd_ws and copies y and the final
 * state back. There is no counterpart on the pages; it is the path for callers
 * whose data live in host memory.
 *
 * The problem is cut into pieces (batch rows, and head groups when the batch
 * is small; every (b, h) sequence is independent) that go through internal
 * streams copy-in -> compute -> copy-out with two pieces in flight, so that
 * the host-device copies and the compute overlap. Host buffers should be
 * pinned (cudaHostAlloc / cudaHostRegister) for the copies to be asynchronous
 * and overlap; pageable buffers give the same results, slower.
 *
 *   x, A, B_t, C_t, dt, y, final_state   host pointers, layout as for
 *                                        ssd_complex_fwd_ws
 *   dev_scratch    device memory, 256-byte aligned, at least
 *                  ssd_complex_fwd_host_scratch_bytes(dims, chunk_size) bytes;
 *                  it holds the device copies of two pieces and their
 *                  workspaces (no initialisation needed)
 *   stream         the work starts after the caller's earlier work on
 *                  `stream`, and `stream` continues after the last copy-out
 *
 * The call returns when y and the final state are in the host buffers, with
 * SSDC_OK, a host-side argument error (before anything is enqueued), or the
 * first device status that is not SSDC_OK. Calls on one device are
 * serialised by the library; calls sharing one dev_scratch must not overlap.
 */
size_t ssd_complex_fwd_host_scratch_bytes(ssdc_dims dims, int chunk_size);
int ssd_complex_fwd_host(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t,
                         const float *dt, ssdc_dims dims, int chunk_size,
                         ssdc_cout y, ssdc_cout final_state, void *dev_scratch,
                         size_t scratch_bytes, cudaStream_t stream);

/*
 * Backward pass: the gradients of a real loss L with respect to every input
 * of the forward pass, given the gradients with respect to its outputs. The
 * pages' training path (page "Extending -- SSM variants & Triton kernels",
 * Step 3: the backward recomputes the forward and is seeded with the true
 * output gradients; every differentiated input gets a gradient).
 *
 * Convention. A complex gradient holds dL/dRe(z) in its real plane and
 * dL/dIm(z) in its imaginary plane (PyTorch's convention for complex
 * tensors). With g_t the gradient of the state s_t, the adjoint recurrence is
 *   g_{T-1} = d_final_state + conj(C_{T-1}) (outer) dy_{T-1}
 *   g_{t-1} = conj(A_bar_t) g_t + conj(C_{t-1}) (outer) dy_{t-1}
 *   dx_t[d] = sum_n g_t[n,d] conj(B_t[n])     dB_t[n] = sum_d g_t[n,d] conj(x_t[d])
 *   dC_t[n] = sum_d dy_t[d] conj(s_t[n,d])
 *   dz_t = sum g_t conj(A_bar_t s_{t-1})      (z_t = softplus(dt_t) A)
 *   ddt_t = Re(dz_t conj(A)) sigmoid(dt_t),  dA = sum_{b,t} softplus(dt_t) dz_t
 *   d_initial_state = conj(A_bar_0) g_0
 * The library computes it chunk by chunk: it recomputes the chunk states
 * S_in[c], runs the adjoint state recurrence backwards over the chunks (R_c,
 * the gradient of the state leaving chunk c), forms dx, dB_t and dC_t per
 * chunk, and obtains dz_t for token t of chunk c from the identity
 *   dz_t = <R_c, S_out(c)> + sum_{t' >= t in chunk c} (<dC_t', C_t'> - <dB_t', B_t'>)
 * with <u, v> = sum u conj(v), S_out(c) the state leaving chunk c, and the
 * sums accumulated in fp64. dA is summed over b and t in a fixed order, so
 * repeated calls give bit-identical results.
 *
 *   x, A, B_t, C_t, dt, initial_state   the forward pass's inputs, as for
 *                        ssd_complex_fwd_init (initial_state: both planes null
 *                        for zero; x.im NULL for a real x)
 *   dy                   (B,T,H,D) gradient of y. dy.im may be NULL: a loss of
 *                        Re(y) alone (the pages' model takes Re(y))
 *   d_final_state        (B,H,N,D) gradient of the final state; both planes
 *                        NULL for zero
 *   dx                   output (B,T,H,D). dx.im may be NULL: not written (for
 *                        a real x, dx.re is the gradient of x)
 *   dA                   output (H) complex, summed over b and t
 *   dB_t, dC_t           outputs (B,T,H,N) complex
 *   ddt                  output (B,T,H) real
 *   d_initial_state      output (B,H,N,D) complex; both planes NULL: not
 *                        written
 *   workspace            device memory, 256-byte aligned, at least
 *                        ssd_complex_bwd_workspace_bytes() bytes; no
 *                        initialisation needed
 * All pointers are device pointers, 16-byte aligned. Outputs must not overlap
 * each other, an input or the workspace. One null plane of a pair that must
 * be given together is SSDC_ERR_INVALID.
 *
 * Precision: SSDC_PREC_FP32 is exact fp32 on the SIMT cores (every decay with
 * the accurate expf / sincosf), for the sizes of SSDC_PREC_FP32 in the forward
 * pass. SSDC_PREC_TF32 computes the per-chunk gradient products (dx, dB_t,
 * dC_t) on the TF32 tensor cores, with chunk_size 16, 32, 64, 128 or 256 and
 * N, D multiples of 8 up to 64; at 128 and 256 it works on chunks of 64
 * tokens (the gradients of the scan do not depend on how it is chunked; the
 * workspace size follows). The chunk recurrences and the step-size gradients
 * stay exact fp32. SSDC_PREC_TF32_STAGED returns SSDC_ERR_UNSUPPORTED.
 * Errors, streams and ownership as for ssd_complex_fwd_ws.
 */
size_t ssd_complex_bwd_workspace_bytes(ssdc_dims dims, int chunk_size);
int ssd_complex_bwd(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t, const float *dt,
                    ssdc_cin initial_state, ssdc_cin dy, ssdc_cin d_final_state,
                    ssdc_dims dims, int chunk_size, ssdc_cout dx, ssdc_cout dA,
                    ssdc_cout dB_t, ssdc_cout dC_t, float *ddt, ssdc_cout d_initial_state,
                    void *workspace, size_t ws_bytes, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SSDC_H */
