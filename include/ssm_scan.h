/*
 * ssm_scan.h -- C ABI of a B300 (sm_103a) selective state-space scan library (Mamba "S6").
 *
 * What is computed. For every batch row b, channel d and state n, with the step
 *     dt[b,d,t] = softplus(delta[b,d,t] + delta_bias[d])   (or without softplus / bias)
 * the discretised diagonal system
 *     A_bar = exp(dt * A[d,n]),   B_bar * u = dt * B[b,n,t] * u[b,d,t]
 *     h[b,d,n,t] = A_bar * h[b,d,n,t-1] + dt * B[b,n,t] * u[b,d,t],   h[.,.,.,-1] = 0
 *     y[b,d,t]   = (sum_n C[b,n,t] * h[b,d,n,t] + D[d] * u[b,d,t]) * SiLU(z[b,d,t])
 * This is the per-timestep loop of section 3.2 of "From RNN to Mamba: state-space model
 * principles and long-sequence modelling in practice" (lmnt.cn): A_bar = exp(dt*A),
 * B_bar = dt*B_t, h = A_bar*h + B_bar*x_t, y_t = sum(h*C_t), then y + x*D and the SiLU(z)
 * gate; A diagonal per section 2.2; softplus of a biased projection for dt per section 3.3
 * (softplus(x) = log(1 + e^x): "Mamba architecture principles and industrial long-text
 * practice", jsqmd.com, section 2.2). The recurrent single-token step used at inference
 * (lmnt.cn section 5.3: one fixed-size fp32 state, advanced token by token) is
 * ssm_state_update.
 *
 * Readings the library fixes where the pages are silent:
 *   - B_bar*u = dt*B*u (the page's code); the exact zero-order hold (A_bar-1)/A*B is
 *     available through ssm_selective_scan_fwd_disc / ssm_state_update_disc.
 *   - softplus(v) = v for v > 20, else log(1 + exp(v)) (beta = 1).
 *   - y at t uses the state after the update at t.
 *   - B and C are shared by all channels of a batch row: [batch][dstate][seqlen].
 *
 * Layouts (row-major, last index contiguous; every tensor is dense with no stride gaps):
 *   u, delta, z, y : [batch][dim][seqlen]   io dtype (fp32 or bf16)
 *   B, C           : [batch][dstate][seqlen] io dtype
 *   A              : [dim][dstate]           fp32
 *   D, delta_bias  : [dim]                   fp32
 *   last_state     : [batch][dim][dstate]    fp32
 * Precision: inputs are read in their stored precision, everything is computed in fp32
 * (state, discretisation, readout), and y is rounded once (round-to-nearest-even) to the
 * io dtype. exp uses the hardware base-2 exponential (ex2.approx) on dt*A*log2(e).
 *
 * Ownership: the caller owns every buffer; the library never frees or retains a caller
 * pointer after the call returns. Device pointers must be device memory of the current
 * CUDA device. Alignment: the scan's u, delta, z, y, B, C, last_state and the state
 * update's state and A must be 16-byte aligned; the scan's A, D, delta_bias and the state
 * update's per-token vectors (x, dt, z, y, B, C) and D need only their element alignment.
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default stream)
 * unless stated otherwise.
 *
 * Errors: arguments are checked on the host before anything is launched; on any error
 * nothing is launched and nothing is written. Launch failures return SSM_ERR_CUDA
 * (cudaGetLastError). Errors raised while a kernel runs (the bounded waits of the
 * L-parallel scan) are recorded in a device status word that ssm_stream_status() reads.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif
/* The library is built with hidden symbol visibility; what this header declares is exported. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

typedef enum {
    SSM_OK = 0,
    SSM_ERR_NULL = 1,        /* a required pointer is NULL */
    SSM_ERR_SHAPE = 2,       /* a dimension is negative, dstate < 1, or sizes overflow */
    SSM_ERR_DTYPE = 3,       /* io_dtype is not one of ssm_dtype_t */
    SSM_ERR_ALIGN = 4,       /* a pointer is not aligned as required (see Alignment) */
    SSM_ERR_UNSUPPORTED = 5, /* dstate > SSM_MAX_DSTATE, or no device / wrong architecture */
    SSM_ERR_CUDA = 6,        /* a CUDA runtime call failed */
    SSM_ERR_TIMEOUT = 7,     /* a bounded device-side wait gave up (see ssm_stream_status) */
    SSM_ERR_WORKSPACE = 8,   /* workspace missing or too small */
    SSM_ERR_CHECK = 9        /* checked build only (-DSSM_CHECK): a bounds check on a global or
                                shared-memory access failed and the access was skipped (see
                                ssm_stream_status) */
} ssm_status_t;

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype_t;

/* batch, dim (channels, "d_inner"), seqlen (L) and dstate (N) of a call, and the dtype of
 * u, delta, B, C, z and y (the state, A, D and delta_bias are always fp32). */
typedef struct {
    int64_t batch, dim, seqlen, dstate;
    ssm_dtype_t io_dtype;
} ssm_dims_t;

#define SSM_MAX_DSTATE 128

/*
 * Selective scan forward (lmnt.cn "From RNN to Mamba", section 3.2, the loop; the
 * associative prefix-scan form of section 2.2 and of jsqmd.com section 3.4 lets the GPU
 * split the sequence): computes y (and optionally the final state) as defined above.
 *   dims            batch, dim, seqlen, dstate, io dtype. batch, dim or seqlen may be 0
 *                   (nothing to compute; last_state, if given and seqlen == 0, is zeroed).
 *   u, delta        device, [batch][dim][seqlen], io dtype. delta is the raw step.
 *   A               device, [dim][dstate] fp32 (diagonal of the state matrix; any real).
 *   B, C            device, [batch][dstate][seqlen], io dtype.
 *   D               device, [dim] fp32, or NULL for no skip term.
 *   z               device, [batch][dim][seqlen] io dtype, or NULL for no gate.
 *   delta_bias      device, [dim] fp32 added to delta before the softplus, or NULL.
 *   delta_softplus  nonzero: dt = softplus(delta + bias); zero: dt = delta + bias.
 *   y               device, [batch][dim][seqlen] io dtype, written.
 *   last_state      device, [batch][dim][dstate] fp32, written with h at t = seqlen-1,
 *                   or NULL.
 *   stream          cudaStream_t the work is queued on.
 * Sequences are split into chunks processed in parallel when batch*dim alone cannot fill
 * the GPU; the chunk states then pass through a workspace: the one registered for the
 * current device with ssm_set_workspace if there is one (SSM_ERR_WORKSPACE if it is too
 * small; nothing is allocated then), else one the library allocates stream-ordered
 * (cudaMallocAsync / cudaFreeAsync on `stream`). ssm_selective_scan_fwd_ws takes a
 * workspace per call instead.
 * Rows whose byte length (seqlen * io size) is not a multiple of 16: the default kernel moves
 * rows in 16-byte pieces, so u, delta, z, B and C are first copied to a padded row stride in
 * the workspace and y comes back through a padded buffer (the workspace then also holds
 * those copies). With a workspace too small for them (a registered or caller workspace, or
 * the no-allocation entry's scratch), such rows take the slower element-wise kernel.
 */
ssm_status_t ssm_selective_scan_fwd(const ssm_dims_t *dims, const void *u, const void *delta,
                                    const float *A, const void *B, const void *C,
                                    const float *D, const void *z, const float *delta_bias,
                                    int delta_softplus, void *y, float *last_state,
                                    void *stream);

/* Bytes of device workspace ssm_selective_scan_fwd_ws needs for `dims` (0 if none): the
 * default plan's, including the padded row copies of rows that are not 16-byte multiples. */
size_t ssm_selective_scan_workspace_bytes(const ssm_dims_t *dims);

/* As ssm_selective_scan_fwd, with a caller-owned device workspace (16-byte aligned, at
 * least ssm_selective_scan_workspace_bytes(dims) bytes; it may be NULL when that is 0).
 * The workspace must not be used by anything else until the call has completed on
 * `stream`. Returns SSM_ERR_WORKSPACE if it is too small. */
ssm_status_t ssm_selective_scan_fwd_ws(const ssm_dims_t *dims, const void *u,
                                       const void *delta, const float *A, const void *B,
                                       const void *C, const float *D, const void *z,
                                       const float *delta_bias, int delta_softplus, void *y,
                                       float *last_state, void *workspace,
                                       size_t workspace_bytes, void *stream);

/*
 * Registers a process-wide default workspace for the current CUDA device (the workspace of
 * the split-sequence carries: "Mamba architecture principles and industrial long-text
 * practice", jsqmd.com, section 3.4, a long sequence cut into chunks whose states are passed
 * on; lmnt.cn "From RNN to Mamba" section 5.3 keeps the recurrent state in a fixed buffer).
 *   dev_ptr  device memory of the current device, 16-byte aligned, or NULL to unregister
 *            (the library then allocates stream-ordered again).
 *   bytes    its size; 0 with dev_ptr NULL.
 * Used by ssm_selective_scan_fwd, and by ssm_selective_scan_fwd_disc,
 * ssm_conv_selective_scan_fwd and ssm_selective_scan_bwd when they are given a NULL
 * workspace, for calls on this device: a call that needs more than `bytes` returns
 * SSM_ERR_WORKSPACE before queuing any work, and nothing is allocated while a workspace is
 * registered. ssm_selective_scan_workspace_bytes (and the _conv_ / _bwd_ variants) give
 * the size a call needs.
 * Ownership: the caller keeps the memory; it must stay valid until every call that used it
 * has completed on its stream. The library never frees it.
 * Concurrency: calls that use the registered workspace and overlap on the GPU race on it,
 * whichever streams or host threads issue them: queue them on one stream or order them
 * with events. ssm_selective_scan_fwd_host never uses it.
 * Returns SSM_OK; SSM_ERR_NULL (dev_ptr NULL, bytes > 0); SSM_ERR_WORKSPACE (bytes 0 with a
 * pointer); SSM_ERR_ALIGN; SSM_ERR_CUDA (no current device); SSM_ERR_UNSUPPORTED (device
 * index >= 64). Takes effect for calls made after it returns.
 */
ssm_status_t ssm_set_workspace(void *dev_ptr, size_t bytes);

/* Size of the library's fixed device scratch used by ssm_selective_scan_fwd_noalloc. */
#define SSM_SCRATCH_MAX_BYTES ((size_t)48 * 1024 * 1024)

/*
 * As ssm_selective_scan_fwd, but it never allocates device memory: the chunk carries,
 * the persistent kernel's control words and the prepared B/C live in one fixed scratch
 * array of SSM_SCRATCH_MAX_BYTES per device, compiled into the library. The method has
 * no counterpart on the pages: this is a calling convention, not a step of the scan.
 *
 * For callers that cannot allocate at call time:
 *   - a program whose device memory is held by another allocator (a framework's caching
 *     pool), where a stream-ordered allocation from the driver's default pool can fail for
 *     lack of memory although the framework has free blocks;
 *   - a device or driver configuration without stream-ordered memory pools
 *     (cudaDevAttrMemoryPoolsSupported is 0), where cudaMallocAsync is not available;
 *   - plain C callers with no allocator of their own that cannot size a workspace and
 *     keep it alive until each call has completed on the stream.
 *
 * Scratch size: returns SSM_ERR_WORKSPACE, before any CUDA work is queued, when
 * ssm_selective_scan_workspace_bytes(dims) exceeds SSM_SCRATCH_MAX_BYTES. The default plans
 * keep only chunk carries there (1 x 1536 x 131072 x 64 needs about 41 MiB and fits); a plan
 * that also keeps the whole sequence's B and C there (the persistent time-split kernel,
 * about 65 MiB for that shape) is rejected. Use ssm_selective_scan_fwd_ws for those.
 * Zero state: the control words at the start of the scratch (the persistent kernel's
 * work ticket and per-segment carry flags) must be zero when that kernel starts; every
 * call clears them on `stream` (cudaMemsetAsync) before its launch. Everything else in
 * the scratch is written before it is read within the call.
 * First use: the first call in each device context (and again after the context is reset)
 * resolves the scratch's device address with cudaGetSymbolAddress, which may load the
 * library's module. Make that first call before any stream capture begins. A failure there
 * returns SSM_ERR_CUDA.
 * Concurrency: there is ONE scratch per device. Calls whose GPU work overlaps on the same
 * device race on it, whichever streams or host threads issue them, and give wrong results.
 * Queue such calls on one stream, or order them with events.
 * Arguments, layout and the other status codes are those of ssm_selective_scan_fwd.
 */
ssm_status_t ssm_selective_scan_fwd_noalloc(const ssm_dims_t *dims, const void *u,
                                            const void *delta, const float *A, const void *B,
                                            const void *C, const float *D, const void *z,
                                            const float *delta_bias, int delta_softplus,
                                            void *y, float *last_state, void *stream);

/*
 * Recurrent single-token step (lmnt.cn "From RNN to Mamba", section 5.3; the section 3.2
 * loop body for one timestep), in place on the state:
 *     state[b,d,n] = exp(dt[b,d]*A[d,n]) * state[b,d,n] + dt[b,d]*B[b,n]*x[b,d]
 *     y[b,d]       = (sum_n C[b,n]*state[b,d,n] + D[d]*x[b,d]) * SiLU(z[b,d])
 *   dims        batch, dim, dstate, io dtype (seqlen is ignored).
 *   state       device, [batch][dim][dstate] fp32, read and overwritten.
 *   x, dt       device, [batch][dim] io dtype; dt is the final positive step (no bias,
 *               no softplus applied here).
 *   A           device, [dim][dstate] fp32.   B, C: device, [batch][dstate] io dtype.
 *   D           device, [dim] fp32 or NULL.   z: device, [batch][dim] io dtype or NULL.
 *   y           device, [batch][dim] io dtype, written.
 */
ssm_status_t ssm_state_update(const ssm_dims_t *dims, float *state, const void *x,
                              const void *dt, const float *A, const void *B, const void *C,
                              const float *D, const void *z, void *y, void *stream);

/* Discretisation of B (the A_bar = exp(dt*A) step is the same in both). */
typedef enum {
    SSM_DISC_EULER = 0, /* B_bar = dt*B: the per-timestep loop of lmnt.cn "From RNN to Mamba"
                           section 3.2 (what ssm_selective_scan_fwd and ssm_state_update do) */
    SSM_DISC_ZOH = 1    /* exact zero-order hold B_bar = (exp(dt*A) - 1)/A * B, equal to dt*B
                           where A = 0: jsqmd.com "Mamba architecture principles and industrial
                           long-text practice" section 2.3 */
} ssm_disc_t;

/*
 * ssm_selective_scan_fwd with the discretisation chosen (ssm_disc_t). `workspace` may be
 * NULL (the library then allocates stream-ordered, as ssm_selective_scan_fwd), or a
 * caller-owned buffer as for ssm_selective_scan_fwd_ws. The zero-order hold runs on the
 * default channel-pair kernel; rows that are not 16-byte multiples go through the padded
 * copies described at ssm_selective_scan_fwd, and a workspace too small for them returns
 * SSM_ERR_UNSUPPORTED (as does an unknown `discretization`). B_bar*u is formed as dt*u*B * phi(dt*A), phi(x) = (e^x - 1)/x, with a
 * cubic polynomial for |x| < 1/8 and (exp(x) - 1)/x otherwise: relative error of phi about
 * 2e-6 at most, no extra exponential per element. Other arguments and errors: as
 * ssm_selective_scan_fwd / ssm_selective_scan_fwd_ws.
 */
ssm_status_t ssm_selective_scan_fwd_disc(const ssm_dims_t *dims, const void *u,
                                         const void *delta, const float *A, const void *B,
                                         const void *C, const float *D, const void *z,
                                         const float *delta_bias, int delta_softplus,
                                         int discretization, void *y, float *last_state,
                                         void *workspace, size_t workspace_bytes,
                                         void *stream);

/* ssm_state_update with the discretisation chosen (ssm_disc_t); same arguments and errors,
 * SSM_ERR_UNSUPPORTED for an unknown `discretization`. */
ssm_status_t ssm_state_update_disc(const ssm_dims_t *dims, float *state, const void *x,
                                   const void *dt, const float *A, const void *B,
                                   const void *C, const float *D, const void *z,
                                   int discretization, void *y, void *stream);

/*
 * The conv-to-gate span of the Mamba block fused in front of the scan (lmnt.cn "From RNN to
 * Mamba", sections 3.1-3.2: a depthwise Conv1d with kernel size K and padding K-1, its
 * output cut to the first seqlen steps, then SiLU), per channel:
 *     u[b,d,t] = SiLU(conv_b[d] + sum_{k<K} conv_w[d][k] * x[b,d,t-(K-1)+k]),  x[t < 0] = 0
 * and then exactly ssm_selective_scan_fwd with this u (also in the D skip term). u is formed
 * tile by tile in shared memory and never written to HBM.
 *   x           device, [batch][dim][seqlen] io dtype: the input of the convolution.
 *   conv_w      device, [dim][conv_width] fp32 (the Conv1d weight [dim][1][K] squeezed).
 *   conv_b      device, [dim] fp32, or NULL for no conv bias.
 *   conv_width  K, 1..4 (SSM_ERR_UNSUPPORTED otherwise).
 *   workspace   NULL (stream-ordered allocation by the library) or a caller buffer of at
 *               least ssm_conv_selective_scan_workspace_bytes(dims) bytes.
 * Runs on the channel-pair kernel; rows whose byte length is not a multiple of 16 go through
 * padded copies in the workspace (ssm_conv_selective_scan_workspace_bytes counts them), and
 * a caller or registered workspace too small for them returns SSM_ERR_WORKSPACE. Other
 * arguments, layouts and errors: as ssm_selective_scan_fwd.
 */
ssm_status_t ssm_conv_selective_scan_fwd(const ssm_dims_t *dims, const void *x,
                                         const float *conv_w, const float *conv_b,
                                         int conv_width, const void *delta, const float *A,
                                         const void *B, const void *C, const float *D,
                                         const void *z, const float *delta_bias,
                                         int delta_softplus, void *y, float *last_state,
                                         void *workspace, size_t workspace_bytes,
                                         void *stream);

/* Bytes of device workspace ssm_conv_selective_scan_fwd needs for `dims` (0 if none). */
size_t ssm_conv_selective_scan_workspace_bytes(const ssm_dims_t *dims);

/*
 * Selective scan backward (training differentiates through the recurrence: lmnt.cn "From RNN
 * to Mamba" section 2.2; the loop is section 3.2): gradients of
 *     sum_{b,d,t} y[b,d,t] * dy[b,d,t]  +  sum_{b,d,n} last_state[b,d,n] * dlast_state[b,d,n]
 * with respect to every input of ssm_selective_scan_fwd (Euler discretisation). The forward
 * states are recomputed from checkpoints taken every 8 steps (workspace) and the adjoint
 * recurrence lambda_t = dyhat_t C_t + exp(dt_{t+1} A) lambda_{t+1} is run backwards. Where
 * the batch rows and channels alone would give fewer than two thread blocks per SM, the
 * sequence is also cut into chunks of whole 8-step segments that run in parallel (chunk-local
 * states and adjoint carries, combined between the passes); the workspace then also holds
 * per-segment dt sums and per-chunk states and carries.
 *   u, delta, A, B, C, D, z, delta_bias, delta_softplus: as ssm_selective_scan_fwd.
 *   dy           device, [batch][dim][seqlen] io dtype (gradient of y).
 *   dlast_state  device, [batch][dim][dstate] fp32 gradient of the final state, or NULL.
 *   du, ddelta   device, [batch][dim][seqlen] fp32, written (ddelta: of the raw delta).
 *   dA           device, [dim][dstate] fp32, written (summed over batch and time).
 *   dB, dC       device, [batch][dstate][seqlen] fp32, written (summed over channels).
 *   dD           device, [dim] fp32, or NULL if not wanted.
 *   dz           device, [batch][dim][seqlen] fp32, or NULL (zeros when z is NULL).
 *   ddelta_bias  device, [dim] fp32, or NULL if not wanted.
 *   workspace    NULL (stream-ordered allocation by the library) or a caller buffer of at
 *                least ssm_selective_scan_bwd_workspace_bytes(dims) bytes, 16-byte aligned.
 * Pointers need only their element alignment. Sums over channels, batch rows and time use
 * fp32 atomic additions, so results may differ in the last bits between runs.
 * Returns SSM_OK (with nothing written for an empty batch or channel count; for an empty
 * sequence dA, dD and ddelta_bias are zeroed);
 * SSM_ERR_NULL for a missing required pointer; SSM_ERR_ALIGN for a misaligned pointer or
 * workspace; SSM_ERR_SHAPE / SSM_ERR_DTYPE for bad dims; SSM_ERR_UNSUPPORTED for more than
 * 65535 batch rows or dstate > 128; SSM_ERR_WORKSPACE when a caller or registered workspace
 * is smaller than needed; SSM_ERR_CUDA when a CUDA call fails (ssm_last_cuda_error). The
 * argument checks run before any CUDA call.
 */
ssm_status_t ssm_selective_scan_bwd(const ssm_dims_t *dims, const void *u, const void *delta,
                                    const float *A, const void *B, const void *C,
                                    const float *D, const void *z, const float *delta_bias,
                                    int delta_softplus, const void *dy,
                                    const float *dlast_state, float *du, float *ddelta,
                                    float *dA, float *dB, float *dC, float *dD, float *dz,
                                    float *ddelta_bias, void *workspace,
                                    size_t workspace_bytes, void *stream);

/* Bytes of device workspace ssm_selective_scan_bwd needs for `dims` (0 if none). */
size_t ssm_selective_scan_bwd_workspace_bytes(const ssm_dims_t *dims);

/*
 * Host-buffer scan: the same computation as ssm_selective_scan_fwd, with every array in
 * HOST memory (pinned memory gives the fastest copies). The call copies the inputs to the
 * device, scans, copies y (and last_state) back, and returns when the results are in the
 * host buffers. Device buffers are allocated stream-ordered on `stream` and freed before
 * returning; the work starts after what the caller queued on `stream`. The channels are
 * processed in blocks (up to 32 per call, at least 8 MB of input each) that flow through
 * three streams -- copies in,
 * scans, copies out -- with three buffer sets, so that each block's copies overlap the
 * scans of its neighbours. Same argument meanings and errors as
 * ssm_selective_scan_fwd (alignment is not required of host pointers).
 */
ssm_status_t ssm_selective_scan_fwd_host(const ssm_dims_t *dims, const void *u,
                                         const void *delta, const float *A, const void *B,
                                         const void *C, const float *D, const void *z,
                                         const float *delta_bias, int delta_softplus,
                                         void *y, float *last_state, void *stream);

/* Synchronises `stream` and returns (then clears) the library's device status word:
 * SSM_OK, SSM_ERR_TIMEOUT if a bounded device-side wait gave up since the last check,
 * SSM_ERR_CHECK (checked build) if a bounds check failed, or SSM_ERR_CUDA if the
 * synchronisation itself failed. */
ssm_status_t ssm_stream_status(void *stream);

/*
 * Structured-A fast path of the forward scans (ssm_selective_scan_fwd*, including the
 * conv-front and zero-order-hold variants): where A[d, n] == (n + 1) * A[d, 0] holds
 * exactly in fp32 for every state of a warp's channels (the S4D-real initialisation
 * A_log = log(1..N), lmnt.cn section 3.3, for which A_bar[n] = A_bar[0]^(n+1)), the scan
 * forms the decays of four consecutive states from one exponential and powers of
 * exp(dt * A[d, 0]) instead of one exponential per state. The test runs on the device in
 * every call; warps that fail it (and every warp when dstate is not a multiple of the
 * kernel's state tile) take the general path. The results agree with the general path to
 * fp32 rounding (they are not bitwise identical). enable: nonzero = detect, 0 = always take
 * the general path (the default: the scan's inner loop is limited by instruction issue, not
 * by the exponential unit, so on B300 the power form takes as long as the general path).
 * Process-wide; takes effect for calls queued after it returns. Returns the previous
 * setting (0 or 1). Never fails.
 */
int ssm_set_structured_a(int enable);

/*
 * Launch-plan override: a test and tuning hook, not needed for normal use. The library reads
 * no environment variables; tests and tuning runs that want a particular kernel, lane split
 * or chunk count set it here. Every field 0 means the planner's own choice. Process-wide;
 * takes effect for calls made after it returns (and for ssm_*_workspace_bytes).
 *   kernel                  SSM_KERNEL_AUTO (the planner), SSM_KERNEL_PAIR (the channel-pair
 *                           kernel where the rows allow it), SSM_KERNEL_SEQ (the sequential-
 *                           lane kernel), SSM_KERNEL_TC / SSM_KERNEL_TP (the persistent
 *                           time-split kernels, barrier-phased / pipelined: they keep a
 *                           stretch's decays in tensor memory and chain segment carries
 *                           through release/acquire flags with a bounded wait).
 *   pair_states_per_lane    channel-pair kernel: 4 (dstate <= 16), 8, or 16 (33..64 states).
 *   chunks                  the number of sequence chunks of the channel-pair or sequential-
 *                           lane kernel (clamped to what the sequence length allows).
 *   seq_states_per_lane, seq_lanes_per_channel
 *                           sequential-lane split; both 0, or one of the built pairs (4,1),
 *                           (8,1), (16,1), (4,4), (16,2), (16,4), (16,8).
 *   decode_elementwise      1: the recurrent step reads B and C element by element.
 *   force_timeout           1: the persistent kernels' carry wait watches a flag that nothing
 *                           sets, with a short limit, so that it gives up and records
 *                           SSM_ERR_TIMEOUT (read by ssm_stream_status); tests the failure
 *                           path without faulting anything.
 *   check_probe             checked build (-DSSM_CHECK) only: one thread of each channel-pair
 *                           launch issues a checked load one element past the end of A, which
 *                           the check skips and records as SSM_ERR_CHECK (a test that the
 *                           checks fire). Ignored by the normal build.
 *   bwd_states_per_lane     ssm_selective_scan_bwd: 4 (the default) or 2 states per lane (taken
 *                           for dstate <= 32; more lanes per channel, fewer registers).
 *   bwd_chunks              ssm_selective_scan_bwd: the number of sequence chunks of the time
 *                           split (1 = none; clamped to the number of 8-step segments).
 * ssm_set_plan_override(NULL) restores the planner. Returns SSM_ERR_UNSUPPORTED for an
 * unknown kernel, lane split or states-per-lane value and SSM_ERR_SHAPE for a negative count;
 * the previous override then stays in force.
 */
typedef enum {
    SSM_KERNEL_AUTO = 0,
    SSM_KERNEL_PAIR = 1,
    SSM_KERNEL_SEQ = 2,
    SSM_KERNEL_TC = 3,
    SSM_KERNEL_TP = 4
} ssm_kernel_t;

typedef struct {
    int kernel;
    int pair_states_per_lane;
    int chunks;
    int seq_states_per_lane;
    int seq_lanes_per_channel;
    int decode_elementwise;
    int force_timeout;
    int check_probe;
    int bwd_states_per_lane;
    int bwd_chunks;
} ssm_plan_override_t;

ssm_status_t ssm_set_plan_override(const ssm_plan_override_t *ov);
/* The override in force (all zero when none); SSM_ERR_NULL for a NULL `out`. */
ssm_status_t ssm_get_plan_override(ssm_plan_override_t *out);

/* Human-readable name of a status code (static storage; never NULL). */
const char *ssm_status_string(ssm_status_t status);

/* The CUDA runtime error (a cudaError_t value) behind the most recent SSM_ERR_CUDA that an
 * entry point returned on the calling thread; 0 if none has. Thread-local; not reset by
 * later successful calls. Its text: ssm_cuda_error_string. Callable without a GPU. */
int ssm_last_cuda_error(void);
/* The CUDA runtime's text for error `code` (static storage; never NULL). */
const char *ssm_cuda_error_string(int code);

/* Library ABI version: (major << 16) | minor. */
int ssm_version(void);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif
#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H */
