/*
 * mamba_ssm.h - C ABI of libmamba_ssm_b300.so, the B300 (sm_103a) selective
 * state-space scan of Mamba, its single-token decode step, the scan with a
 * causal conv1d + SiLU fused in front, and the scan's backward (gradients of
 * every input).
 *
 * The operation (page titles and passages that define it):
 *   "State Space Models and Mamba" (jonathanding.github.io, llm-learning)
 *     §1   continuous system x' = A x + B u, y = C x + D u (D is the skip term);
 *     §1.5 A is diagonal, stored as A_log, A = -exp(A_log);
 *     §2   zero-order hold: Abar = exp(dt A), Bbar = A^-1 (exp(dt A) - I) B,
 *          recurrence x_k = Abar x_{k-1} + Bbar u_k, y_k = C x_k;
 *     §3   recurrence mode: one O(1) state update per token (decode);
 *     §4   selectivity: dt_k = softplus(.), B_k and C_k change per step;
 *          hardware-aware scan (paper §3.3.2): the (B,L,D,N) Abar/Bbar are
 *          never written to memory, only y (B,L,D) is.
 *   "Mamba" paper notes (awesome.papernotes.org, 2023_mamba)
 *     "Design 1: Selective State Space": Bbar = (dt A)^-1 (exp(dt A) - I) dt B,
 *     the selective_ssm sketch (y + D * x) and "Overall framework"
 *     (out = y * SiLU(z)).
 *
 * Per batch b, channel d, state n and step t the scan computes
 *     dt      = softplus(delta[b,t,d] + delta_bias[d])
 *     A       = -exp(A_log[d,n])
 *     h[n]    = exp(dt A) h[n] + (exp(dt A) - 1) / A * B[b,t,n] * u[b,t,d]
 *     y       = sum_n C[b,t,n] h[n] + D[d] u[b,t,d]
 *     out     = y * z / (1 + exp(-z))        (z = z[b,t,d]; no gate if z is NULL)
 * from h = 0 (or from initial_state in the _ex entry point). The decode step
 * is the same body for one token on a state kept in device memory. The
 * backward returns the gradients of sum(dout * out) + sum(dlast * last_state).
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers owned by the caller unless said otherwise;
 *     tensors are contiguous, row-major, in the layouts given per argument.
 *   - Work is enqueued on `stream` and is asynchronous: MAMBA_OK means the
 *     arguments were valid and the kernels were launched. A fault inside a
 *     kernel shows at the caller's next synchronisation, or through
 *     mamba_device_status().
 *   - Stream order holds for every byte read or written. The decode kernels,
 *     and the scan's second kernel when a call launches two, use programmatic
 *     dependent launch: such a kernel may become resident while the kernel
 *     before it in the stream is still running, but each of its threads waits
 *     for that kernel to complete and flush (griddepcontrol.wait) before it
 *     touches memory that kernel may write. The scan and decode kernels also
 *     let the next kernel in the stream launch early; a kernel launched
 *     without the programmatic attribute is not affected by that.
 *   - Validation happens before any launch. Every failure returns a status
 *     and sets a thread-local detail string (mamba_last_error_detail()).
 *     No C++ exception crosses the ABI.
 *   - `out` and `last_state` must not alias any input. The decode `state` is
 *     read and written in place and must not alias any other argument.
 *   - batch == 0, dim == 0 or (scan) seqlen == 0 is valid and empty: nothing
 *     is read; a requested last_state is set to the initial state (zero).
 *   - Input dtype: MAMBA_F32 or MAMBA_BF16 applies to u, delta, z, B, C and
 *     out. A_log, D, delta_bias, states are always fp32. All arithmetic is
 *     fp32 with fp32 state. With MAMBA_F32 inputs the kernels use accurate
 *     expm1/exp/log1p; with MAMBA_BF16 inputs they use the hardware ex2/lg2
 *     approximations, and take exp(dt A) - 1 from a short series wherever
 *     dt |A| is small enough that ex2 - 1 would cancel (the scan reruns a
 *     16-step chunk of a warp with the series when some step of it falls
 *     below dt |A| = 2^-14; the backward takes the series for a whole chunk
 *     of the CTA in that case; the decode step always does), so that Bbar
 *     keeps a relative error near 1e-6 at any dt A.
 *   - |A| = exp(A_log) is floored at 1e-20 inside the kernels. At and below
 *     that floor exp(dt A) and (exp(dt A) - 1) / A equal their A -> 0 limits
 *     (1 and dt) in fp32 for any dt below 1e12, so results are those of the
 *     exact A (the zero-order hold's limit: the state integrates dt B u).
 *     The backward multiplies dA_log = A dloss/dA by the unfloored A.
 *   - dstate (N) may be 1..256 (16, 32, 64 or 128 for the backward).
 */
#ifndef MAMBA_SSM_H
#define MAMBA_SSM_H

#include <stddef.h>
#include <stdint.h>

#if defined(MAMBA_BUILDING_LIBRARY) && defined(__GNUC__)
#define MAMBA_API __attribute__((visibility("default")))
#else
#define MAMBA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t (a CUstream); NULL is the legacy default stream. */
typedef struct CUstream_st *mamba_stream_t;

typedef enum {
    MAMBA_F32 = 0,
    MAMBA_BF16 = 1
} mamba_dtype_t;

typedef enum {
    MAMBA_OK = 0,
    MAMBA_ERR_INVALID_ARG = 1,   /* NULL required pointer, negative size, aliasing */
    MAMBA_ERR_UNSUPPORTED = 2,   /* valid request the library does not implement (e.g. N > 256) */
    MAMBA_ERR_CUDA = 3,          /* a CUDA runtime call failed; detail names it */
    MAMBA_ERR_TIMEOUT = 4        /* a kernel's bounded wait ran out (see mamba_device_status) */
} mamba_status_t;

/*
 * Selective scan, forward.
 *   batch, dim, dstate, seqlen : B, D (= d_inner), N (= d_state), L.
 *   in_dtype   : dtype of u, delta, z, B, C and out.
 *   u          : (B, L, D) input x of the SSM.
 *   delta      : (B, L, D) pre-softplus step (dt = softplus(delta + delta_bias)).
 *   A_log      : (D, N) fp32; A = -exp(A_log).
 *   B, C       : (B, L, N) input and output projections, shared by all D channels of a batch row.
 *   D          : (D,) fp32 skip weights, or NULL for no skip.
 *   z          : (B, L, D) gate input, or NULL for no gate.
 *   delta_bias : (D,) fp32, or NULL for zero.
 *   out        : (B, L, D) written.
 *   last_state : (B, D, N) fp32 written with h after step L-1, or NULL.
 * Splitting long sequences over several CTAs uses a temporary stream-ordered
 * workspace (cudaMallocAsync / cudaFreeAsync on `stream`, about
 * B * D * (N + 1) * 4 bytes per extra segment); MAMBA_ERR_CUDA if it cannot
 * be had.
 */
MAMBA_API mamba_status_t mamba_selective_scan_fwd(
    int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype,
    const void *u, const void *delta, const float *A_log,
    const void *B, const void *C, const float *D, const void *z,
    const float *delta_bias, void *out, float *last_state,
    mamba_stream_t stream);

/*
 * Discretisation of the input matrix.
 *   MAMBA_ZOH        : zero-order hold, Bbar = (exp(dt A) - 1) / A * B - the
 *                      method ("State Space Models and Mamba" §2, "Mamba"
 *                      paper notes, Design 1). The default.
 *   MAMBA_SIMPLIFIED : Bbar = dt * B, the form of the paper notes'
 *                      selective_ssm sketch (first order in dt A); Abar is
 *                      still exp(dt A). About a third fewer FP32 operations.
 */
typedef enum {
    MAMBA_ZOH = 0,
    MAMBA_SIMPLIFIED = 1
} mamba_discretization_t;

/*
 * Plan knobs for mamba_selective_scan_fwd_ex. A zero field means "choose
 * automatically" (or ZOH for discretization). lanes_per_channel, segments
 * and use_tma never change results beyond fp32 rounding order (the tests
 * compare plans against each other and the oracle); discretization selects
 * the input matrix.
 *   lanes_per_channel : threads sharing one channel's N states: a power of
 *                       two from ceil(N / 16) to 16;
 *   segments          : the sequence is cut into this many time segments that
 *                       run in parallel, joined by the two-pass carry (1 = off);
 *   use_tma           : 0 auto, 1 require the TMA tile loader (error if the
 *                       layout does not allow it), 2 force plain loads;
 *   discretization    : a mamba_discretization_t value;
 *   time_lanes        : 0 or 1: each lane walks time sequentially (the default).
 *                       2 or 4: the time-parallel chunk scan: that many lanes
 *                       share a channel, each holding all its states and
 *                       scanning its part of every 16-step chunk; the parts
 *                       are joined by a warp-shuffle scan under the operator
 *                       (a, b) o (a', b') = (a a', a' b + b') and each lane
 *                       fixes its readouts up with the exact state entering
 *                       its part ("State Space Models and Mamba" §4, parallel
 *                       scan). Needs N <= 16, zero-order hold, one segment
 *                       (segments 0 or 1) and lanes_per_channel 0 or 1, and
 *                       is not available with the fused conv1d
 *                       (MAMBA_ERR_UNSUPPORTED / MAMBA_ERR_INVALID_ARG).
 *                       Automatic plans never choose it.
 */
typedef struct {
    int lanes_per_channel;
    int segments;
    int use_tma;
    int discretization;
    int time_lanes;
} mamba_scan_plan_t;

/*
 * As mamba_selective_scan_fwd, plus:
 *   initial_state : (B, D, N) fp32 state to start from, or NULL for zero
 *                   (lets a prefill continue from an earlier chunk or a decode state);
 *   plan          : NULL or knobs above.
 */
MAMBA_API mamba_status_t mamba_selective_scan_fwd_ex(
    int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype,
    const void *u, const void *delta, const float *A_log,
    const void *B, const void *C, const float *D, const void *z,
    const float *delta_bias, const float *initial_state, void *out,
    float *last_state, const mamba_scan_plan_t *plan, mamba_stream_t stream);

/*
 * The scan with the step in front of it in the Mamba block fused in: the
 * input x is passed through a causal depthwise conv1d and SiLU,
 *     u[b,t,d] = SiLU( sum_{k<W} conv_weight[d,k] * x[b, t-(W-1)+k, d] + conv_bias[d] ),
 * x taken as zero before t = 0 ("Mamba" paper notes, Design 3; compassingai
 * "Mamba" §3.3; "State Space Models and Mamba", Mamba Block architecture:
 * kernel size 4, conv then SiLU), and u feeds the scan and its D skip.
 *   x           : (B, L, D) in_dtype, the conv input;
 *   conv_weight : (D, W) fp32; W = conv_width in 1..4 (tap W-1 multiplies x_t);
 *   conv_bias   : (D,) fp32 or NULL for zero.
 * Other arguments as mamba_selective_scan_fwd_ex. Zero-order hold only
 * (plan->discretization must be MAMBA_ZOH): MAMBA_ERR_UNSUPPORTED otherwise,
 * and for W outside 1..4.
 */
MAMBA_API mamba_status_t mamba_conv1d_selective_scan_fwd(
    int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype,
    const void *x, const float *conv_weight, const float *conv_bias, int conv_width,
    const void *delta, const float *A_log, const void *B, const void *C,
    const float *D, const void *z, const float *delta_bias,
    const float *initial_state, void *out, float *last_state,
    const mamba_scan_plan_t *plan, mamba_stream_t stream);

/*
 * Allocation-free variant of mamba_selective_scan_fwd_ex. The pages have no
 * counterpart of this call; it exists for callers that cannot allocate device
 * memory while they run: code inside a custom allocator or a memory-pool
 * callback, or a runtime that forbids allocation after start-up. The regular
 * entry point may take a temporary workspace with cudaMallocAsync; this one
 * never calls cudaMalloc, cudaMallocAsync, cudaFree or any other allocating
 * routine, and uses instead a static device array of
 * MAMBA_NOALLOC_SCRATCH_BYTES (16 MiB) that every device loading the library
 * holds until the process exits. The caller still passes all inputs and
 * outputs.
 *   - The split-sequence workspace of the chosen plan, B * (segments - 1) * D *
 *     (N + 1) * 4 bytes, must fit in the array; larger requests return
 *     MAMBA_ERR_UNSUPPORTED with the byte counts in the detail string (pass a
 *     plan with fewer segments, or segments = 1, which needs no scratch).
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call shares the one array and it keeps the previous call's
 *     contents. Each call writes every scratch value it reads before reading
 *     it, so nothing needs clearing, but calls whose kernels overlap on the GPU
 *     (concurrent streams) race on the array: serialise them.
 * Arguments, results and errors are otherwise those of mamba_selective_scan_fwd_ex.
 */
#define MAMBA_NOALLOC_SCRATCH_BYTES (16u << 20)
MAMBA_API mamba_status_t mamba_selective_scan_fwd_noalloc(
    int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype,
    const void *u, const void *delta, const float *A_log,
    const void *B, const void *C, const float *D, const void *z,
    const float *delta_bias, const float *initial_state, void *out,
    float *last_state, const mamba_scan_plan_t *plan, mamba_stream_t stream);

/*
 * The plan mamba_selective_scan_fwd_ex would use for these sizes on the
 * current device, assuming 16-byte aligned pointers: writes the chosen knobs
 * to *chosen (use_tma = 1 if the TMA loader would be used, else 2) and the
 * number of kernel launches one call makes (1, or 2 with segments > 1) to
 * *kernel_launches. Validation and errors as for the scan itself; the
 * discretization knob is copied through.
 */
MAMBA_API mamba_status_t mamba_selective_scan_plan(
    int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype,
    const mamba_scan_plan_t *plan, mamba_scan_plan_t *chosen, int *kernel_launches);

/*
 * Single-token decode step on a resident state ("State Space Models and
 * Mamba" §3, recurrence mode).
 *   state      : (B, D, N) fp32, read and written in place.
 *   u, delta, z: (B, D) in_dtype (z may be NULL).
 *   A_log      : (D, N) fp32.
 *   B, C       : (B, N) in_dtype.
 *   D, delta_bias : (D,) fp32 or NULL.
 *   out        : (B, D) in_dtype, written.
 * MAMBA_F32 inputs use expf / expm1f / log1pf. MAMBA_BF16 inputs use the
 * hardware ex2 / rcp approximations, with exp(dt A) - 1 from a short series
 * where |dt A| < 1/8 (relative error near 1e-6 at any dt A). With N a power of
 * two from 8 to 256, dim a multiple of 8 and 16-byte aligned pointers, the
 * state is staged through shared memory by bulk copies (the bulk-staged
 * kernel); other shapes take a register-path kernel. batch may be up to 262140.
 */
MAMBA_API mamba_status_t mamba_selective_state_update(
    int batch, int dim, int dstate, mamba_dtype_t in_dtype,
    float *state, const void *u, const void *delta, const float *A_log,
    const void *B, const void *C, const float *D, const void *z,
    const float *delta_bias, void *out, mamba_stream_t stream);

/*
 * As mamba_selective_state_update, with the discretisation of the input
 * matrix (a mamba_discretization_t value; MAMBA_ERR_INVALID_ARG otherwise).
 */
MAMBA_API mamba_status_t mamba_selective_state_update_ex(
    int batch, int dim, int dstate, mamba_dtype_t in_dtype,
    float *state, const void *u, const void *delta, const float *A_log,
    const void *B, const void *C, const float *D, const void *z,
    const float *delta_bias, void *out, int discretization, mamba_stream_t stream);

/*
 * Backward of the scan: the gradients of
 *   loss = sum_{b,t,d} dout[b,t,d] * out[b,t,d] + sum_{b,d,n} dlast_state[b,d,n] * last_state[b,d,n]
 * with respect to every input of mamba_selective_scan_fwd_ex, for the same
 * forward ("State Space Models and Mamba" §2-§4: zero-order hold, or the
 * simplified Bbar = dt B of the "Mamba" paper notes' selective_ssm sketch,
 * chosen by `discretization`; D skip and SiLU gate as in the forward). The
 * forward is recomputed from the inputs: the call needs no saved activations.
 *
 * Inputs (as for the forward; device pointers, row-major, contiguous):
 *   u, delta, z (z may be NULL)      : (B, L, D) in_dtype
 *   A_log                            : (D, N) fp32
 *   B, C                             : (B, L, N) in_dtype
 *   D, delta_bias                    : (D,) fp32 or NULL (= 0)
 *   initial_state                    : (B, D, N) fp32 or NULL (= 0)
 *   dout                             : (B, L, D) in_dtype, the gradient of out
 *   dlast_state                      : (B, D, N) fp32 or NULL (= 0)
 * Outputs (written; none is accumulated into):
 *   du, ddelta                       : (B, L, D) in_dtype, required
 *   dz                               : (B, L, D) in_dtype; must be NULL when z is NULL
 *   dA_log                           : (D, N) fp32, required
 *   dB, dC                           : (B, L, N) fp32, required
 *   dD, ddelta_bias                  : (D,) fp32 or NULL (not computed); computed
 *                                      even when D / delta_bias is NULL
 *   dinitial_state                   : (B, D, N) fp32 or NULL (not computed)
 * dstate must be 16, 32, 64 or 128 (MAMBA_ERR_UNSUPPORTED otherwise); batch
 * <= 65535. The fp32 arrays read or written four at a time (initial_state,
 * dlast_state, dA_log, dB, dC, dinitial_state) must be 16-byte aligned
 * (MAMBA_ERR_UNSUPPORTED otherwise). Outputs may not alias inputs or each
 * other (MAMBA_ERR_INVALID_ARG).
 *
 * Work: the call zeroes dA_log, dB, dC, dD, ddelta_bias on `stream`, then a
 * kernel launch runs the forward over each channel, stores the state every 16
 * steps in a stream-ordered workspace of B * ceil(L/16) * D * N * 4 bytes
 * (cudaMallocAsync / cudaFreeAsync on `stream`), and walks the chunks
 * backwards. When few channel blocks x batch rows would leave SMs idle, the
 * sequence is cut into time segments (see mamba_selective_scan_bwd_ex). dB, dC, dA_log, dD and ddelta_bias are sums over channels or
 * batch rows taken with fp32 atomics, so their last bits may differ from call
 * to call. MAMBA_F32 inputs use expf / expm1f; MAMBA_BF16 inputs use the
 * hardware ex2 / rcp approximations, as the forward does.
 */
MAMBA_API mamba_status_t mamba_selective_scan_bwd(
    int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype, int discretization,
    const void *u, const void *delta, const float *A_log, const void *B, const void *C,
    const float *D, const void *z, const float *delta_bias, const float *initial_state,
    const void *dout, const float *dlast_state,
    void *du, void *ddelta, float *dA_log, float *dB, float *dC,
    float *dD, void *dz, float *ddelta_bias, float *dinitial_state, mamba_stream_t stream);

/*
 * As mamba_selective_scan_bwd, with the number of time segments: 0 chooses
 * automatically (segments only when the channel blocks x batch rows leave SMs
 * idle), 1 runs each channel over the whole sequence, k > 1 cuts the sequence
 * into about k segments of whole 16-step chunks (at most 64). With segments, two
 * extra launches precede the gradient pass: each segment's end state from a zero
 * start, and the adjoint each segment passes back from a zero adjoint; the
 * gradient pass composes them per segment (the split-sequence carry of the
 * forward, run forward and backward in time). The workspace grows by
 * B * segments * D * (2 N + 1) * 4 bytes. segments < 0: MAMBA_ERR_INVALID_ARG.
 */
MAMBA_API mamba_status_t mamba_selective_scan_bwd_ex(
    int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype, int discretization,
    const void *u, const void *delta, const float *A_log, const void *B, const void *C,
    const float *D, const void *z, const float *delta_bias, const float *initial_state,
    const void *dout, const float *dlast_state,
    void *du, void *ddelta, float *dA_log, float *dB, float *dC,
    float *dD, void *dz, float *ddelta_bias, float *dinitial_state, int segments, mamba_stream_t stream);

/* Static description of a status code. */
MAMBA_API const char *mamba_status_string(mamba_status_t s);

/* Detail of the last failure on the calling host thread ("" if none). */
MAMBA_API const char *mamba_last_error_detail(void);

/*
 * Kernel-side status word of the current device. Kernels never trap; a
 * bounded wait that runs out records MAMBA_ERR_TIMEOUT here and the kernel
 * returns early. This call synchronises `stream`, copies the word to
 * *status_out and clears it.
 */
MAMBA_API mamba_status_t mamba_device_status(int *status_out, mamba_stream_t stream);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
MAMBA_API int mamba_version(void);

/*
 * Test setting, process-wide: the limit, in nanoseconds, that the scan and
 * decode launches enqueued after this call give their pipeline's mbarrier
 * waits (default 2000000000, 2 s). 0 makes those waits give up at once, so
 * that a launch that waits on a copy records MAMBA_ERR_TIMEOUT in the device
 * status word and returns early without writing all of its outputs; its
 * copies already in flight are still awaited with the default limit before
 * it exits. This exists to exercise the timeout path on a healthy GPU; leave
 * it at the default otherwise. Returns the previous limit.
 */
MAMBA_API unsigned long long mamba_set_wait_limit_ns(unsigned long long limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_SSM_H */
