/*
 * ssm.h -- C ABI of the B300 selective state-space scan library (libssm_b300.so).
 *
 * The library implements the selective state-space model "S6" of
 * "Mamba: Linear-Time Sequence Modeling with Selective State Spaces":
 *
 *   Delta_t   = softplus(delta_raw_t + delta_bias)           (per token, per channel)
 *   dA_t[n]   = exp(Delta_t * A[n])                          (zero-order-hold decay)
 *   h_t[n]    = dA_t[n] * h_{t-1}[n] + Delta_t * B_t[n] * x_t (input term, first order)
 *   y_t       = (sum_n C_t[n] * h_t[n] + D * x_t) * silu(z_t)
 *
 * Passages defining it:
 *   - the state equation h(t+1) = A h(t) + B x(t) and the observation
 *     y(t) = C h(t): "Mamba: Linear-Time Sequence Modeling with Selective
 *     State Spaces" (dhy1.tistory.com), section "0. State Space Models";
 *   - discretisation of (Delta, A, B) by zero-order hold (stage 1) and the
 *     recurrent mode (stage 2), Delta, B and C made input-dependent, A acting
 *     per state dimension: "Mamba的三大创新" (weblog-19d.pages.dev), sections
 *     "S4的4个参数..." and "硬件感知的设计：并行扫描...";
 *   - constant-time recurrent inference over a fixed-size state (the decode
 *     step): the same page, model comparison table (RNN / SSM / Mamba rows).
 * The time index is read so that token t enters its own output (h_t, not
 * h_{t-1}, is read out).  The input term uses Delta*B (the first-order form of
 * the zero-order hold), the skip D*x is added before the gate.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous,
 *     row-major with the last index fastest, and aligned to their element
 *     size (the decode state to 16 bytes when dstate >= 4); a misaligned
 *     pointer is rejected with SSM_ERR_INVALID_ARG.  16-byte aligned tensors
 *     let the scan take its tiled path (see ssm_scan_plan).  The library
 *     never allocates, frees or synchronises; work is enqueued on `stream`
 *     (a cudaStream_t; NULL = the legacy default stream) and runs
 *     asynchronously.  Results are valid once the stream has reached them.
 *   - "io" tensors (x, delta, z, B, C, out) have the dtype `io_dtype`
 *     (fp32 or bf16).  A, D, delta_bias and the states are always fp32, and
 *     the recurrence is always carried in fp32.
 *   - Optional pointers may be NULL: z (no gate), D (no skip), delta_bias
 *     (zero bias), initial_state (zero state), last_state (not written).
 *   - Errors: nothing is enqueued when a call returns other than SSM_OK for an
 *     argument check.  SSM_ERR_CUDA reports a failed launch (the CUDA error is
 *     then available from cudaGetLastError in the caller's runtime).
 */
#ifndef SSM_B300_H
#define SSM_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1,   /* NULL/misaligned pointer, negative size, small workspace */
    SSM_ERR_UNSUPPORTED = 2,   /* valid but not implemented: dstate, dtype, alignment */
    SSM_ERR_CUDA = 3,          /* a kernel launch failed */
    SSM_ERR_TIMEOUT = 4        /* a bounded device-side wait gave up (see ssm_get_device_status) */
} ssm_status;

typedef enum {
    SSM_DTYPE_F32 = 0,
    SSM_DTYPE_BF16 = 1
} ssm_dtype;

/* Problem description shared by the entry points.
 *   batch  : number of sequences (>= 0)
 *   seqlen : tokens per sequence (>= 0; ignored by ssm_state_update)
 *   dim    : channels D (>= 0)
 *   dstate : state size N per channel, one of 1, 2, 4, 8, 16, 32, 64
 *   io_dtype : ssm_dtype of x, delta, z, B, C, out
 *   delta_softplus : 1 = Delta = softplus(delta + delta_bias); 0 = Delta = delta + delta_bias */
typedef struct {
    int64_t batch;
    int64_t seqlen;
    int64_t dim;
    int64_t dstate;
    int32_t io_dtype;
    int32_t delta_softplus;
} ssm_scan_desc;

/* Bytes of device workspace ssm_scan_fwd needs for `desc` (0 when the
 * sequence is not split into chunks).  Returns 0 for an invalid desc. */
SSM_API size_t ssm_scan_workspace_size(const ssm_scan_desc *desc);

/* Selective scan forward over whole sequences (prefill).
 *   x, delta, z, out : (batch, seqlen, dim) io
 *   B, C             : (batch, seqlen, dstate) io, shared by all channels
 *   A                : (dim, dstate) fp32 (the continuous-time diagonal A, normally < 0)
 *   D, delta_bias    : (dim) fp32
 *   initial_state    : (batch, dim, dstate) fp32 state before token 0, or NULL (zeros)
 *   last_state       : (batch, dim, dstate) fp32 state after the last token, or NULL
 *   workspace        : device scratch of at least ssm_scan_workspace_size(desc)
 *                      bytes (may be NULL when that size is 0); its contents on
 *                      entry do not matter and are garbage on exit.
 * `out` must not alias an input.  `last_state` may alias `initial_state`
 * (in-place carry from one call to the next). */
SSM_API ssm_status ssm_scan_fwd(const ssm_scan_desc *desc,
                        const void *x, const void *delta, const float *A,
                        const void *B, const void *C, const float *D,
                        const void *z, const float *delta_bias,
                        void *out, float *last_state, const float *initial_state,
                        void *workspace, size_t workspace_bytes, void *stream);

/* One recurrent step for one new token per sequence (decode).
 * desc->seqlen is ignored (one token).
 *   state            : (batch, dim, dstate) fp32, read and overwritten in place
 *   x, delta, z, out : (batch, dim) io
 *   B, C             : (batch, dstate) io
 *   A                : (dim, dstate) fp32;  D, delta_bias: (dim) fp32
 * Applying it T times equals ssm_scan_fwd over the same T tokens with
 * initial_state = state. */
SSM_API ssm_status ssm_state_update(const ssm_scan_desc *desc, float *state,
                            const void *x, const void *delta, const float *A,
                            const void *B, const void *C, const float *D,
                            const void *z, const float *delta_bias,
                            void *out, void *stream);

/* Discretisation of the input term ("Mamba的三大创新", stage 1, zero-order hold).
 * The decay is exp(Delta A) in both; the input term is
 *   SSM_DISC_EULER : Delta B x                      (the first-order form; ssm_scan_fwd)
 *   SSM_DISC_ZOH   : ((exp(Delta A) - 1) / A) B x   (exact for x held over the step;
 *                                                     Delta B x where A = 0) */
typedef enum { SSM_DISC_EULER = 0, SSM_DISC_ZOH = 1 } ssm_discretization;

/* Options of the _ex entry points; reserved[] must be zero. */
typedef struct {
    int32_t discretization;   /* ssm_discretization */
    int32_t reserved[3];
} ssm_scan_opts;

/* ssm_scan_fwd / ssm_state_update with options (today: the discretisation).
 * Arguments, layouts, workspace and errors are those of the plain calls;
 * opts NULL, an unknown discretisation or non-zero reserved fields return
 * SSM_ERR_INVALID_ARG.  SSM_DISC_ZOH runs in the warp-specialised kernel for
 * dstate 16 and in the general kernel for the other state sizes. */
SSM_API ssm_status ssm_scan_fwd_ex(const ssm_scan_desc *desc, const ssm_scan_opts *opts,
                                   const void *x, const void *delta, const float *A,
                                   const void *B, const void *C, const float *D, const void *z,
                                   const float *delta_bias, void *out, float *last_state,
                                   const float *initial_state, void *workspace,
                                   size_t workspace_bytes, void *stream);
SSM_API ssm_status ssm_state_update_ex(const ssm_scan_desc *desc, const ssm_scan_opts *opts,
                                       float *state, const void *x, const void *delta,
                                       const float *A, const void *B, const void *C,
                                       const float *D, const void *z, const float *delta_bias,
                                       void *out, void *stream);

/* Training pair: the forward also keeps the state before every 16th token,
 * and the backward reads those checkpoints instead of recomputing them.
 *   checkpoints: (batch, ceil(seqlen / 16), dim, dstate) fp32, 16-byte aligned,
 *                ssm_scan_checkpoint_size(desc) bytes; entry j is the state
 *                before token 16 j (entry 0 = initial_state).
 * ssm_scan_fwd_train: ssm_scan_fwd plus the checkpoints (dstate 16 in the
 *   warp-specialised kernel, other sizes in the general one).
 * ssm_scan_bwd_ex: ssm_scan_bwd with checkpoints (NULL: recompute, exactly
 *   ssm_scan_bwd); the inputs must be those of the forward that wrote them.
 *   Workspace: ssm_scan_bwd_ex_workspace_size(desc, with_checkpoints). */
SSM_API size_t ssm_scan_checkpoint_size(const ssm_scan_desc *desc);
SSM_API ssm_status ssm_scan_fwd_train(const ssm_scan_desc *desc, const void *x, const void *delta,
                                      const float *A, const void *B, const void *C,
                                      const float *D, const void *z, const float *delta_bias,
                                      void *out, float *last_state, const float *initial_state,
                                      float *checkpoints, void *workspace, size_t workspace_bytes,
                                      void *stream);
SSM_API size_t ssm_scan_bwd_ex_workspace_size(const ssm_scan_desc *desc, int with_checkpoints);
SSM_API ssm_status ssm_scan_bwd_ex(const ssm_scan_desc *desc, const void *x, const void *delta,
                                   const float *A, const void *B, const void *C, const float *D,
                                   const void *z, const float *delta_bias,
                                   const float *initial_state, const void *dout,
                                   const float *dlast_state, const float *checkpoints, void *dx,
                                   void *ddelta, float *dA, float *dB, float *dC, float *dD,
                                   void *dz, float *ddelta_bias, float *dinitial_state,
                                   void *workspace, size_t workspace_bytes, void *stream);

/* The time-invariant (LTI, S4) model in its convolution mode ("Mamba的三大创新",
 * stage 3).  With a constant per-channel step delta[d] (> 0, used as given:
 * no bias, no softplus) and input-independent per-channel B, C, the
 * recurrence from a zero state is the causal convolution y = K * x with
 *   K[d][k] = sum_n C[d][n] exp(k delta[d] A[d][n]) Bbar[d][n],  k < seqlen,
 * Bbar per opts->discretization (NULL opts: first order).
 *   ssm_lti_kernel  : delta (dim) fp32; A, B, C (dim, dstate) fp32; K out (dim, seqlen) fp32.
 *                     desc->batch and desc->io_dtype are ignored.
 *   ssm_lti_conv_fwd: y[b][t][d] = sum_{k<=t} K[d][k] x[b][t-k][d] + D[d] x[b][t][d],
 *                     gated by silu(z) when z is not NULL.  x, z, out (batch,
 *                     seqlen, dim) io; K (dim, seqlen) fp32; D (dim) fp32 or NULL.
 *                     O(seqlen^2) work per (sequence, channel); desc->dstate and
 *                     desc->delta_softplus are ignored.  out must not alias x.
 *                     bf16 I/O with dim a multiple of 8 and 16-byte aligned x, z,
 *                     out runs on the tensor cores, each tap of K carried as two
 *                     bf16 terms (about 2^-17 of its value); fp32 I/O and other
 *                     shapes run on the CUDA cores in fp32. */
SSM_API ssm_status ssm_lti_kernel(const ssm_scan_desc *desc, const ssm_scan_opts *opts,
                                  const float *delta, const float *A, const float *B,
                                  const float *C, float *K, void *stream);
SSM_API ssm_status ssm_lti_conv_fwd(const ssm_scan_desc *desc, const float *K, const void *x,
                                    const float *D, const void *z, void *out, void *stream);

/* The selection projections of S6 ("Mamba的三大创新", the selection mechanism:
 * Delta, B and C are linear functions of the input), on the tensor cores:
 *   xdbl   = x W_x^T            x (batch*seqlen, dim), W_x (R + 2 dstate, dim)
 *   dt_low = xdbl[:, 0:R]       (batch, seqlen, R)
 *   B, C   = xdbl[:, R:R+N], xdbl[:, R+N:R+2N]   (batch, seqlen, dstate) each
 *   delta  = act(dt_low W_dt^T + delta_bias)     W_dt (dim, R) -> (batch, seqlen, dim)
 * act = softplus when desc->delta_softplus is 1, identity when 0; delta_bias
 * (dim) fp32 or NULL (zero).  With act = softplus, `delta` is the step Delta
 * itself: pass it to ssm_scan_fwd with delta_softplus = 0 and no delta_bias
 * (the scan's prologue work done in this epilogue).  With act = identity and
 * no bias it is the raw step, for ssm_scan_fwd with softplus and bias.
 * All other tensors bf16 (desc->io_dtype must be SSM_DTYPE_BF16), row-major,
 * 16-byte aligned, with dim and R multiples of 8 and R + 2 dstate <= 256;
 * fp32 accumulation, one bf16 rounding per output.  delta may be NULL
 * (x_proj only).  Two tcgen05 GEMM launches. */
typedef struct {
    int32_t dt_rank;      /* R */
    int32_t reserved;     /* must be 0 */
} ssm_proj_desc;

SSM_API ssm_status ssm_selection_proj_fwd(const ssm_scan_desc *desc, const ssm_proj_desc *proj,
                                          const void *x, const void *W_x, const void *W_dt,
                                          const float *delta_bias, void *dt_low, void *B, void *C,
                                          void *delta, void *stream);

/* The scan with the second selection projection fused in front: for every
 * token and channel the raw step delta_raw = dt_low W_dt^T (the selection
 * mechanism of "Mamba的三大创新": Delta computed from the input) is formed
 * inside the scan, a tile of 16 steps x 16 channels at a time, on the tensor
 * cores with fp32 accumulation, and never stored; the scan then proceeds as
 * ssm_scan_fwd with that raw step, softplus and delta_bias.  The pipeline
 * x_proj -> scan needs no dt_proj launch and no (batch, seqlen, dim) delta
 * tensor in memory.
 *   dt_low       (batch, seqlen, R) bf16: the dt_low output of
 *                ssm_selection_proj_fwd (called with delta = NULL)
 *   W_dt         (dim, R) bf16
 *   everything else as ssm_scan_fwd (delta is not an argument).
 * Supported: bf16 I/O, dstate 16, desc->delta_softplus = 1, R = proj->dt_rank
 * of 64 or 128, dim a multiple of 8, every tensor 16-byte aligned; otherwise
 * SSM_ERR_UNSUPPORTED (shape) or SSM_ERR_INVALID_ARG (alignment, NULL).  The
 * raw step is exact fp32 of the bf16 operands (ssm_selection_proj_fwd rounds
 * it to bf16), so results differ from the unfused pipeline by that rounding.
 * Workspace: ssm_scan_workspace_size(desc) bytes. */
SSM_API ssm_status ssm_proj_scan_fwd(const ssm_scan_desc *desc, const ssm_proj_desc *proj,
                                     const void *x, const void *dt_low, const void *W_dt,
                                     const float *A, const void *B, const void *C,
                                     const float *D, const void *z, const float *delta_bias,
                                     void *out, float *last_state, const float *initial_state,
                                     void *workspace, size_t workspace_bytes, void *stream);

/* Gradients of ssm_scan_fwd (the backward half of training; "Mamba的三大创新",
 * stage 2, parallel training of the recurrence).  The states are recomputed
 * from the inputs (stored every 16 steps in the workspace), never kept from
 * the forward call.  With L the loss:
 *   dout          : (batch, seqlen, dim) io, dL/dout
 *   dlast_state   : (batch, dim, dstate) fp32, dL/dlast_state, or NULL (zero)
 * the forward's inputs x, delta, A, B, C, D, z, delta_bias, initial_state as
 * given to ssm_scan_fwd, and outputs (written, never accumulated):
 *   dx, ddelta    : (batch, seqlen, dim) io      -- ddelta is dL/d(delta before
 *                                                   bias and softplus)
 *   dz            : (batch, seqlen, dim) io, or NULL (not computed); NULL when z is NULL
 *   dA            : (dim, dstate) fp32
 *   dB, dC        : (batch, seqlen, dstate) fp32 (sums over the channels)
 *   dD, ddelta_bias : (dim) fp32, or NULL (not computed); computed also when
 *                   D / delta_bias is NULL (the gradient at zero)
 *   dinitial_state: (batch, dim, dstate) fp32, or NULL
 * workspace: ssm_scan_bwd_workspace_size(desc) bytes, 16-byte aligned (about
 * 0.19 x the bytes of (batch, seqlen, dim, dstate) fp32 states, plus the
 * per-CTA dB/dC partials).  Every sum is formed in a fixed order, so results
 * are bit-identical from run to run.  Outputs must not alias inputs.
 * Elements must be aligned to their size; B and C at 4-element alignment take
 * vector loads. */
SSM_API size_t ssm_scan_bwd_workspace_size(const ssm_scan_desc *desc);

/* How ssm_scan_bwd (with_checkpoints = 0) or ssm_scan_bwd_ex with checkpoints
 * (with_checkpoints = 1) will execute `desc` (host-side query, no GPU work).
 *   nchunk    : pieces the time axis is cut into (1 = one reverse sweep per
 *               (sequence, channel block))
 *   warps     : warps per CTA of the reverse sweep, 4 .. 8, chosen so that
 *               the CTAs spread evenly over the 148 SMs
 *   channels  : channels per CTA (warps x 32 / lanes per channel)
 *   ctas      : CTAs of the reverse sweep
 *   workspace : bytes of workspace the call needs
 * Returns SSM_ERR_INVALID_ARG for a NULL `info` and the descriptor checks'
 * status (as ssm_scan_bwd would) for a bad descriptor. */
typedef struct {
    int32_t nchunk;
    int32_t warps;
    int32_t channels;
    int32_t reserved;
    int64_t ctas;
    int64_t workspace;
} ssm_scan_bwd_plan_info;

SSM_API ssm_status ssm_scan_bwd_plan(const ssm_scan_desc *desc, int with_checkpoints,
                                     ssm_scan_bwd_plan_info *info);
SSM_API ssm_status ssm_scan_bwd(const ssm_scan_desc *desc, const void *x, const void *delta,
                                const float *A, const void *B, const void *C, const float *D,
                                const void *z, const float *delta_bias,
                                const float *initial_state, const void *dout,
                                const float *dlast_state, void *dx, void *ddelta, float *dA,
                                float *dB, float *dC, float *dD, void *dz, float *ddelta_bias,
                                float *dinitial_state, void *workspace, size_t workspace_bytes,
                                void *stream);

/* Causal depthwise convolution applied to x before the SSM in the Mamba block
 * ("Mamba的三大创新", simplified-architecture section: a convolution gives each
 * token its neighbours before the SSM; the unite.ai overview: a causal Conv1d
 * layer).  Width K = `width` (1..8), taps w[d][0..K-1] with w[d][K-1] on the
 * current token:
 *   x_conv[t, d] = act(bias[d] + sum_k w[d][k] * x[t - (K-1) + k, d])
 * act = SiLU when `activation` is 1, identity when 0.  Inputs before t = 0
 * come from a conv state (batch, dim, K-1) fp32, oldest first, or are zero
 * when that pointer is NULL; the final state holds the last K-1 inputs. */
typedef struct {
    int32_t width;
    int32_t activation;
} ssm_conv_desc;

/* x_conv = act(causal depthwise conv(x) + bias), standalone.
 *   x, out          : (batch, seqlen, dim) io (desc->io_dtype); out must not alias x
 *   w               : (dim, width) fp32;  bias: (dim) fp32 or NULL
 *   conv_state_in   : (batch, dim, width-1) fp32 or NULL (zeros)
 *   conv_state_out  : (batch, dim, width-1) fp32 or NULL; may not alias conv_state_in
 * desc->dstate and desc->delta_softplus are ignored. */
SSM_API ssm_status ssm_conv1d_fwd(const ssm_scan_desc *desc, const ssm_conv_desc *conv,
                                  const void *x, const float *w, const float *bias,
                                  const float *conv_state_in, void *out,
                                  float *conv_state_out, void *stream);

/* The conv above fused in front of the selective scan: equal to
 * ssm_conv1d_fwd(x) followed by ssm_scan_fwd with x = x_conv (both the input
 * term Delta*x_conv*B and the skip D*x_conv use it), without writing x_conv
 * to memory.  `x` is the raw (pre-conv) input; the other arguments are those
 * of ssm_scan_fwd, with the same workspace size (ssm_scan_workspace_size).
 * conv_state_out may not alias conv_state_in. */
SSM_API ssm_status ssm_conv_scan_fwd(const ssm_scan_desc *desc, const ssm_conv_desc *conv,
                                     const void *x, const float *conv_w, const float *conv_bias,
                                     const float *conv_state_in, float *conv_state_out,
                                     const void *delta, const float *A, const void *B,
                                     const void *C, const float *D, const void *z,
                                     const float *delta_bias, void *out, float *last_state,
                                     const float *initial_state, void *workspace,
                                     size_t workspace_bytes, void *stream);

/* One decode step with the conv in front: x_conv from conv_state and the new
 * raw x, conv_state shifted in place (oldest input dropped, x appended), then
 * ssm_state_update with x = x_conv.  conv_state: (batch, dim, width-1) fp32
 * (may be NULL only when width == 1); the rest as in ssm_state_update. */
SSM_API ssm_status ssm_conv_state_update(const ssm_scan_desc *desc, const ssm_conv_desc *conv,
                                         float *conv_state, const float *conv_w,
                                         const float *conv_bias, float *state, const void *x,
                                         const void *delta, const float *A, const void *B,
                                         const void *C, const float *D, const void *z,
                                         const float *delta_bias, void *out, void *stream);

/* The scan over tensors that live in host memory: the work is cut into
 * slices, and each slice's inputs are copied in, scanned and its outputs
 * copied back in a three-stage pipeline (copies in, the scan, copies out on
 * their own streams, double-buffered), so the host-device transfers overlap
 * one another and the kernels.  A slice is contiguous in host memory:
 *   slice_batch > 0: that many whole sequences;
 *   slice_batch < 0: a run of -slice_batch steps of one sequence, each run
 *     starting from the state the previous run of that sequence ended in
 *     (kept on the device);
 *   slice_batch = 0: whole sequences while one sequence's x is at most
 *     16 MiB, else 16 MiB runs of steps (multiples of 64).
 * Sequences are independent and the state carries across runs, so the
 * result equals one ssm_scan_fwd over the whole batch.
 *   host (pinned for overlap; pageable memory works but serialises):
 *     x, delta, z, out (batch, seqlen, dim) io; B, C (batch, seqlen, dstate) io;
 *     initial_state, last_state (batch, dim, dstate) fp32 (NULL: zeros / not returned)
 *   device: A (dim, dstate), D, delta_bias (dim) fp32
 *   workspace: device memory of ssm_scan_fwd_host_workspace_size(desc,
 *     slice_batch) bytes, 256-byte aligned.
 * Asynchronous on `stream`: when the stream reaches this call's end, every
 * output has landed in host memory. */
SSM_API size_t ssm_scan_fwd_host_workspace_size(const ssm_scan_desc *desc, int64_t slice_batch);
SSM_API ssm_status ssm_scan_fwd_host(const ssm_scan_desc *desc, int64_t slice_batch,
                                     const void *x, const void *delta, const float *A,
                                     const void *B, const void *C, const float *D, const void *z,
                                     const float *delta_bias, void *out, float *last_state,
                                     const float *initial_state, void *workspace,
                                     size_t workspace_bytes, void *stream);

/* Capacity of the fixed scratch buffer used by ssm_scan_fwd_noalloc. */
#define SSM_NOALLOC_SCRATCH_BYTES (8u << 20)

/* ssm_scan_fwd for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point: it exists for library users, not
 * for the method.
 *
 * Some callers cannot call cudaMalloc or hand the library a workspace: a
 * plug-in interface that gives an operator only its input and output
 * buffers and no allocator, or a latency-bound loop that must not call
 * cudaMalloc/cudaFree because those may block and synchronise the device.
 * This variant takes the same arguments as ssm_scan_fwd minus the workspace
 * and allocates nothing: when the plan needs scratch (a long sequence over
 * few channels is cut into chunks), it uses one file-scope device array of
 * SSM_NOALLOC_SCRATCH_BYTES (8 MiB).  Every GPU that loads the library holds
 * that array until the process exits.
 *   - Problems that need more scratch than that return SSM_ERR_UNSUPPORTED
 *     before anything is enqueued (ssm_scan_workspace_size tells the need).
 *   - The first call on a device looks up the array's device address once
 *     (with that device current); make that first call before any stream
 *     capture.
 *   - All calls share the one array, and it keeps the previous call's
 *     contents.  Every value a call reads from it was written earlier in the
 *     same call, so nothing has to start at zero; but two calls that overlap
 *     on the GPU (different streams, or different host threads) race on it
 *     and give wrong results.  Serialise them. */
SSM_API ssm_status ssm_scan_fwd_noalloc(const ssm_scan_desc *desc,
                                        const void *x, const void *delta, const float *A,
                                        const void *B, const void *C, const float *D,
                                        const void *z, const float *delta_bias,
                                        void *out, float *last_state,
                                        const float *initial_state, void *stream);

/* How ssm_scan_fwd will execute `desc` (host-side query, no GPU work).
 *   path        : 0 = general kernel (one thread per channel),
 *                 3 = tiled kernel of one-warp CTAs (dstate 8, 16, 32 or 64)
 *                 (the tiled kernel is used when the io tensors are 16-byte
 *                 aligned; the plan reported assumes they are).  Value 2 (the
 *                 warp-specialised kernel) is what the exact-ZOH scan and the
 *                 fused conv take; value 1 is no longer used.
 *   nchunk      : pieces the time axis is cut into (1 = not cut)
 *   launches    : kernels one ssm_scan_fwd call enqueues
 *   workspace   : bytes of workspace the call needs (= ssm_scan_workspace_size) */
typedef struct {
    int32_t path;
    int32_t nchunk;
    int32_t launches;
    int32_t reserved;
    int64_t workspace;
} ssm_scan_plan_info;

SSM_API ssm_status ssm_scan_plan(const ssm_scan_desc *desc, ssm_scan_plan_info *info);

/* Device-side status of the kernels that ran so far on the current device:
 * SSM_ERR_TIMEOUT if a bounded wait inside a kernel gave up (that launch's
 * outputs are then incomplete), SSM_OK otherwise.  Reading it clears it.
 * Synchronises with the device (it waits for all prior work). */
SSM_API ssm_status ssm_get_device_status(void);

/* The same status, scoped to one stream: waits only for the work already
 * enqueued on `stream` (NULL = the legacy default stream, which itself waits
 * for the device's other blocking streams), then reads and clears the error
 * word.  SSM_ERR_TIMEOUT if a bounded wait gave up, SSM_OK otherwise,
 * SSM_ERR_CUDA if the read failed.  The error word is one per device (a
 * device variable of the library), not one per call: a timeout in one
 * caller's stream is seen, and cleared, by whichever query reads it first.
 * `workspace` is accepted for the form of the boundary's plan (the word in a
 * call's workspace) and is not used; pass NULL or any workspace. */
SSM_API ssm_status ssm_get_async_status(void *workspace, void *stream);

/* Test hook for the timeout path: launches one warp that waits, for at most
 * `limit_ns` nanoseconds (1e3 .. 5e9), on a shared-memory barrier that nothing
 * completes.  The wait gives up, the kernel returns normally, and the next
 * ssm_get_device_status() reports SSM_ERR_TIMEOUT.  No GPU fault or hang is
 * involved.  The pages have no counterpart to this entry point. */
SSM_API ssm_status ssm_selftest_wait_timeout(int64_t limit_ns, void *stream);

/* Static description of a status code (never NULL). */
SSM_API const char *ssm_status_string(ssm_status status);

/* Library version as major*10000 + minor*100 + patch. */
SSM_API int ssm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSM_B300_H */
