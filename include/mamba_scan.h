/*
 * mamba_scan.h -- C ABI of libmamba_scan.so, a B300 (sm_103a) implementation
 * of the Mamba selective scan (forward, backward, single-token decode) and of
 * the causal depthwise conv1d + SiLU that feeds it.
 *
 * Operation (definitions restated from the pages this library follows):
 *   - Discrete state-space recurrence h_t = Abar_t h_{t-1} + Bbar_t u_t,
 *     y_t = C_t h_t + D u_t, started from h = 0 ("图解 Mamba 状态空间模型"
 *     tutorial, "数学基础"; highthink.cn Keras SelectiveSSM listing, where the
 *     scan's initial state is zeros and D*u is added to C.state).
 *   - Diagonal A = -exp(A_log) per (channel, state), Abar = exp(dt*A), and the
 *     small-step form Bbar = dt*B (highthink.cn listing; tutorial step 1, where
 *     Bbar ~ dt*B "when dt is small").
 *   - Input-dependent step dt = softplus(delta + bias) (codechina.net
 *     overview, section 2.1; highthink.cn dt_proj with a bias).
 *   - The result is gated by SiLU(z), the second branch of the Mamba block
 *     (highthink.cn block diagram: x -> SSM, multiplied by the SiLU branch).
 *   - One fused kernel: parameters are read from HBM once, discretisation and
 *     recurrence happen on chip, and only the result is written (codechina.net
 *     overview, section 1 "硬件感知算法" and section 2.2 "核融合").
 *
 * So for every batch b, channel d, time t and state n:
 *   dt      = softplus_flag ? softplus(delta[b,d,t] + bias[d]) : delta[b,d,t] + bias[d]
 *   h[n]    = exp(dt * -exp(A_log[d,n])) * h[n] + dt * B[b,t,n] * u[b,d,t]
 *   out     = (sum_n C[b,t,n] * h[n] + D[d] * u[b,d,t]) * SiLU(z[b,d,t])
 *   y[b,d,t] = out;  last_state[b,d,n] = h[n] after t = seqlen-1.
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers owned by the caller.  Arrays are dense
 *     row-major with the shapes given below.  The library keeps no data
 *     between calls.  Only mamba_selective_scan_fwd (see there and
 *     mamba_selective_scan_fwd_noalloc) and mamba_selective_scan_bwd take
 *     scratch memory, stream-ordered on the call's stream.
 *   - Per device the library caches what it looks up once: the scratch
 *     memory pool, the decode kernel's launch shape (with the shared-memory
 *     attribute it sets) and the no-alloc buffer's address.  A cudaDeviceReset
 *     invalidates them; call the library again only from a fresh process.
 *   - io_dtype (MAMBA_F32 or MAMBA_BF16) is the element type of every
 *     "io" array (u, delta, z, B, C, y; x, dt, z, B, C, out for decode; dout,
 *     du, ddelta, dz for the backward; x, out and the conv state for conv1d).
 *     A_log, D, the bias, the scan state and the parameter gradients are
 *     always fp32.  Arithmetic is fp32;
 *     bf16 results are rounded to nearest even.
 *   - Work is enqueued on `stream` (0 = legacy default stream) and runs
 *     asynchronously; the call does not synchronise.  A non-zero return means
 *     nothing was launched (argument errors) or the launch failed
 *     (MAMBA_ERR_LAUNCH, with the CUDA error left for cudaGetLastError).
 *   - Pointers must be aligned to their element size (4 bytes for fp32, 2 for
 *     bf16), else MAMBA_ERR_ALIGN.  Wider alignment (16 bytes, with row
 *     lengths that keep it) lets the kernels use 128-bit accesses; any other
 *     aligned input takes a scalar path and gives the same results.
 *   - Outputs must not overlap inputs (MAMBA_ERR_ALIAS), except that the
 *     decode state (mamba_selective_state_update) and the conv state
 *     (mamba_causal_conv1d_update) are updated in place by design, and that
 *     mamba_selective_scan_fwd_ex may read h0 from its last_state buffer.
 *   - A required array that has no elements (a zero size) may be NULL.
 */
#ifndef MAMBA_SCAN_H
#define MAMBA_SCAN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that this header needs no CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *mamba_stream_t;

typedef enum { MAMBA_F32 = 0, MAMBA_BF16 = 1 } mamba_dtype_t;

typedef enum {
    MAMBA_OK = 0,
    MAMBA_ERR_NULL = 1,    /* a required pointer is NULL                         */
    MAMBA_ERR_SIZE = 2,    /* a size is negative or the problem is too large     */
    MAMBA_ERR_DSTATE = 3,  /* dstate outside [1, MAMBA_MAX_DSTATE]               */
    MAMBA_ERR_ALIGN = 4,   /* a pointer is not aligned to its element size       */
    MAMBA_ERR_DTYPE = 5,   /* io_dtype is not a mamba_dtype_t                    */
    MAMBA_ERR_LAUNCH = 6,  /* the CUDA launch failed (see cudaGetLastError)      */
    MAMBA_ERR_TIMEOUT = 7, /* a bounded device-side wait gave up (mamba_device_status) */
    MAMBA_ERR_ALIAS = 8,   /* an output overlaps an input                        */
    MAMBA_ERR_SCRATCH = 9  /* _noalloc: the split needs more than its fixed scratch */
} mamba_status_t;

#define MAMBA_MAX_DSTATE 256
/* Largest conv1d width (taps per channel) of mamba_causal_conv1d_*. */
#define MAMBA_MAX_CONV_WIDTH 8

/*
 * Selective scan, forward.
 *
 *   u, delta, z : [batch, dim, seqlen] io_dtype (time contiguous)
 *   B, C        : [batch, seqlen, dstate] io_dtype, shared by all channels
 *   A_log       : [dim, dstate] fp32;  A = -exp(A_log)
 *   D           : [dim] fp32 or NULL (no skip term)
 *   z           : NULL means no gate
 *   delta_bias  : [dim] fp32 or NULL (no bias)
 *   softplus_flag: non-zero applies softplus to delta + bias
 *   y           : [batch, dim, seqlen] io_dtype, written
 *   last_state  : [batch, dim, dstate] fp32 or NULL; receives h after the last
 *                 step (zeros when seqlen == 0)
 *
 * batch, dim, seqlen may be zero (nothing to compute; last_state is still
 * zeroed when seqlen == 0).  Returns MAMBA_OK or an error code as above.
 *
 * Long sequences of few chains (a grid that would leave at least half of the
 * SMs idle) are split along time: a summary pass per segment, a carry pass
 * and the full pass, the three launched on `stream`.  The carried states
 * (batch * dim * segments * (dstate + 1) fp32 values, at most about
 * 256 * SMs * (dstate + 1) * 4 bytes) live in stream-ordered scratch taken
 * on `stream` and returned on `stream` (cudaMallocFromPoolAsync /
 * cudaFreeAsync), so calls on different streams never share it.  The scratch
 * comes from a memory pool the library creates on each device, which keeps
 * freed memory mapped across synchronisation points (up to
 * MAMBA_SCRATCH_RETAIN_MB megabytes; all of it when unset) instead of
 * returning it to the driver as the device's default pool does.  If that
 * allocation fails the scan runs unsplit.  Results of a split and an unsplit
 * scan agree to rounding.
 */
int mamba_selective_scan_fwd(const void *u, const void *delta, const float *A_log,
                             const void *B, const void *C, const float *D, const void *z,
                             const float *delta_bias, int softplus_flag, void *y,
                             float *last_state, int64_t batch, int64_t dim, int64_t seqlen,
                             int64_t dstate, int io_dtype, mamba_stream_t stream);

/*
 * mamba_selective_scan_fwd without any allocation.  This entry point has no
 * counterpart in the pages.  It is for callers that cannot call cudaMalloc or
 * cudaMallocAsync: a framework that hands out all device memory from its own
 * pool and does not let libraries allocate behind its back, or a serving loop
 * that must not enter the driver's allocator mid-request (an allocation can
 * synchronise the device or fail under memory pressure at a moment the caller
 * does not control).
 *
 * Same arguments, same operation and same results as mamba_selective_scan_fwd:
 * bit for bit whenever the allocating entry point obtains its scratch and the
 * planner's split fits the fixed buffer (always, up to about 240 SMs), since
 * the same kernels then run with the same split.  When the scan is split
 * along time, the carried states live in a fixed device buffer of this
 * library (4 MiB per device, a static __device__ array) instead of
 * stream-ordered scratch:
 *   - The buffer's address is looked up per device (cudaGetSymbolAddress) by
 *     the first call on that device, and kept once the look-up succeeds.
 *     Make that first call before any stream capture; it may also be where
 *     the driver loads this library's module on that device.  A failed
 *     look-up returns MAMBA_ERR_LAUNCH, leaves no CUDA error set, and is
 *     tried again by the next call.
 *   - A planned split that would need more than 4 MiB uses fewer segments.
 *     Only a segment count forced through MAMBA_SCAN_SEGMENTS (a testing
 *     switch) that needs more returns MAMBA_ERR_SCRATCH, before anything is
 *     launched.
 *   - Nothing in the buffer has to start at zero.
 *   - Calls that overlap in time on one device (other streams, other host
 *     threads) share the buffer and race.  Calls ordered on one stream are
 *     safe.
 */
int mamba_selective_scan_fwd_noalloc(const void *u, const void *delta, const float *A_log,
                                     const void *B, const void *C, const float *D,
                                     const void *z, const float *delta_bias, int softplus_flag,
                                     void *y, float *last_state, int64_t batch, int64_t dim,
                                     int64_t seqlen, int64_t dstate, int io_dtype,
                                     mamba_stream_t stream);

/*
 * mamba_selective_scan_fwd with a starting state and document boundaries.
 *
 * The pages state that Mamba isolates documents by resetting its hidden state
 * between them (codechina.net overview, section 3.2, point 2 "边界控制"), and
 * recommend processing sequences beyond 1M tokens block by block (the same
 * page's deployment notes), which needs the state at the end of one block as
 * the start of the next.  For every batch b, channel d, state n:
 *
 *   h[n] = h0 ? h0[b,d,n] : 0                       before step 0
 *   at each step t: if (reset && reset[b,t] != 0) h[n] = 0   (token t starts a
 *   new document), then the step of mamba_selective_scan_fwd.
 *
 *   h0    : [batch, dim, dstate] fp32 or NULL (zero start).  It may be the
 *           same buffer as last_state (continue a stream in place); any other
 *           overlap with y or last_state is MAMBA_ERR_ALIAS.  Aligned to 4.
 *   reset : [batch, seqlen] bytes or NULL (no boundaries); shared by all
 *           channels of a batch row; must not overlap y or last_state.
 *
 * Every other argument, layout and error is as for mamba_selective_scan_fwd
 * (including its split of long sequences of few chains and that split's
 * stream-ordered scratch).  With h0 and reset NULL the results equal
 * mamba_selective_scan_fwd's bit for bit.  seqlen == 0 copies h0 (or zeros)
 * to last_state.  Fast path: dstate 16 with 16-byte aligned rows and a reset
 * mask aligned to 4 bytes; other shapes run the register-prefetch kernel.
 */
int mamba_selective_scan_fwd_ex(const void *u, const void *delta, const float *A_log,
                                const void *B, const void *C, const float *D, const void *z,
                                const float *delta_bias, int softplus_flag, const float *h0,
                                const unsigned char *reset, void *y, float *last_state,
                                int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                int io_dtype, mamba_stream_t stream);

/*
 * Gradients of mamba_selective_scan_fwd (zero initial state) for a given
 * output gradient `dout`, by recomputation: no intermediate state is kept by
 * the forward call; this call re-runs the recurrence and takes the adjoint
 * backwards through it (codechina.net overview, section 2.2, third point,
 * gradient recomputation).
 *
 *   u, delta, A_log, B, C, D, z, delta_bias, softplus_flag, batch, dim,
 *   seqlen, dstate, io_dtype : exactly as given to the forward call
 *   dout        : [batch, dim, seqlen] io_dtype, gradient of y
 *   du, ddelta  : [batch, dim, seqlen] io_dtype, written
 *   dz          : [batch, dim, seqlen] io_dtype, written; required when z is
 *                 given, ignored (may be NULL) when z is NULL
 *   dA_log      : [dim, dstate] fp32, written (gradient w.r.t. A_log)
 *   dB, dC      : [batch, seqlen, dstate] fp32, written (summed over dim)
 *   dD          : [dim] fp32 or NULL (not wanted), written
 *   ddelta_bias : [dim] fp32 or NULL (not wanted), written
 *
 * ddelta is the gradient w.r.t. delta (softplus' derivative applied).  The
 * summed outputs (dA_log, dB, dC, dD, ddelta_bias) are zeroed on `stream`
 * and accumulated with atomic adds, so their low bits depend on the order in
 * which blocks finish; du, ddelta and dz are deterministic.  No output may
 * overlap an input or another output (MAMBA_ERR_ALIAS).
 *
 * Scratch: per chain one fp32 state every 16 steps (batch * dim *
 * ceil(seqlen/16) * dstate * 4 bytes), allocated and freed on `stream` in
 * the call (stream-ordered, from the library's pool described at
 * mamba_selective_scan_fwd), where the page's recomputation keeps O(1).
 * Errors as for mamba_selective_scan_fwd.
 */
int mamba_selective_scan_bwd(const void *u, const void *delta, const float *A_log,
                             const void *B, const void *C, const float *D, const void *z,
                             const float *delta_bias, int softplus_flag, const void *dout,
                             void *du, void *ddelta, void *dz, float *dA_log, float *dB,
                             float *dC, float *dD, float *ddelta_bias, int64_t batch,
                             int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype,
                             mamba_stream_t stream);

/*
 * mamba_selective_scan_bwd for the scan of mamba_selective_scan_fwd_ex: from a
 * starting state h0 and with document boundaries (codechina.net overview,
 * section 3.2 point 2: resetting the hidden state isolates documents; the
 * same page's deployment notes on block-by-block processing of long
 * sequences).  Training on packed documents needs these gradients.  A long
 * sequence trained block by block chains them backwards: dh0 of block k + 1
 * is the gradient block k's final state receives, passed to block k as its
 * dlast_state.
 *
 *   h0    : [batch, dim, dstate] fp32 or NULL (zero start), as for the forward
 *   reset : [batch, seqlen] bytes or NULL; non-zero at a token that starts a
 *           document (the state restarts from zero before it): no gradient
 *           flows back across it
 *   dlast_state : [batch, dim, dstate] fp32 or NULL: the gradient of the loss
 *           with respect to last_state (the state after the last step), added
 *           to the adjoint where it enters from the right; NULL means the loss
 *           does not depend on last_state.  It stops at the last document
 *           start of a row, like the output gradients.
 *   dh0   : [batch, dim, dstate] fp32 or NULL (not wanted), written with the
 *           gradient of h0 (of a zero start when h0 is NULL); equal to
 *           dlast_state (or zero) when seqlen == 0
 *
 * Every other argument, layout, scratch rule and error is as for
 * mamba_selective_scan_bwd, which is this call with h0, reset, dlast_state and
 * dh0 NULL (bit for bit).  h0, reset and dlast_state must not overlap any
 * output (MAMBA_ERR_ALIAS); dlast_state must be 4-byte aligned.
 */
int mamba_selective_scan_bwd_ex(const void *u, const void *delta, const float *A_log,
                                const void *B, const void *C, const float *D, const void *z,
                                const float *delta_bias, int softplus_flag, const float *h0,
                                const unsigned char *reset, const void *dout,
                                const float *dlast_state, void *du, void *ddelta, void *dz,
                                float *dA_log, float *dB, float *dC, float *dD,
                                float *ddelta_bias, float *dh0, int64_t batch,
                                int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype,
                                mamba_stream_t stream);

/*
 * Single-token decode step (recurrent inference: each new token touches only
 * the previous state -- tutorial "核心概念"; mhpn.cn article section 3).
 *
 *   state       : [batch, dim, dstate] fp32, read and updated IN PLACE
 *   x, dt, z    : [batch, dim] io_dtype (z may be NULL: no gate)
 *   A_log       : [dim, dstate] fp32
 *   B, C        : [batch, dstate] io_dtype
 *   D, dt_bias  : [dim] fp32 or NULL
 *   out         : [batch, dim] io_dtype, written
 *
 * Same as one step of mamba_selective_scan_fwd started from `state`.
 *
 * Launch: the fast path (dstate a power of two 4..128, dim a multiple of the
 * kernel's tile, 16-byte aligned rows) is launched as a programmatic
 * dependent of the work before it on `stream`: its blocks may become resident
 * while that work drains, and they wait for it to complete, with its memory
 * writes visible, before any access to global memory -- stream order holds
 * for every argument (a decode loop's state is read after the previous step
 * wrote it).  The environment variable MAMBA_DECODE_PDL=0 launches it plainly.
 */
int mamba_selective_state_update(float *state, const void *x, const void *dt,
                                 const float *A_log, const void *B, const void *C,
                                 const float *D, const void *z, const float *dt_bias,
                                 int softplus_flag, void *out, int64_t batch, int64_t dim,
                                 int64_t dstate, int io_dtype, mamba_stream_t stream);

/*
 * Complex-state selective scan, forward (codechina.net overview, section 4.1:
 * the complex version initialises A = -0.5 + i*n, S4D-Lin; section 5.3: a
 * complex state keeps phase information).  For every b, d, t, n:
 *
 *   A[d,n]   = -exp(A_log_re[d,n]) + i * A_im[d,n]
 *   dt       = as for mamba_selective_scan_fwd (softplus of delta + bias)
 *   h[n]     = exp(dt * A[d,n]) * h[n] + dt * B[b,t,n] * u[b,d,t]   (complex)
 *   y[b,d,t] = (Re(sum_n C[b,t,n] * h[n]) + D[d] * u[b,d,t]) * SiLU(z[b,d,t])
 *
 * The pages give only A and the complex state; B and C are read as complex
 * and input-dependent, and the output as the real part (a caller that keeps
 * one state of each conjugate pair scales C by 2).  The state starts at zero.
 *
 *   u, delta, z, y   : [batch, dim, seqlen] io_dtype
 *   B, C             : [batch, seqlen, dstate, 2] io_dtype, (re, im) pairs
 *   A_log_re, A_im   : [dim, dstate] fp32 (S4D-Lin: log 0.5 and n)
 *   D, delta_bias    : [dim] fp32 or NULL
 *   last_state       : [batch, dim, dstate, 2] fp32 (re, im) or NULL, aligned
 *                      to 8 bytes
 *
 * Errors as for mamba_selective_scan_fwd.  Arithmetic is fp32: exp(dt*A) is
 * 2^(dt*Re A*log2 e) times (cos, sin) of dt*Im A reduced to [-pi, pi].
 */
int mamba_selective_scan_complex_fwd(const void *u, const void *delta, const float *A_log_re,
                                     const float *A_im, const void *B, const void *C,
                                     const float *D, const void *z, const float *delta_bias,
                                     int softplus_flag, void *y, float *last_state,
                                     int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                     int io_dtype, mamba_stream_t stream);

/*
 * Causal depthwise conv1d, optionally followed by SiLU: the short per-channel
 * convolution the Mamba block applies to its x branch before the scan
 * (luzhipeng.com tutorial, step 2: Conv1d with kernel_size = d_conv,
 * padding = d_conv - 1, groups = d_model; highthink.cn "Mamba 整体架构":
 * causal Conv1D, then SiLU).  "Causal" keeps the first seqlen outputs of the
 * padded convolution: for every row (b, d) and step t
 *
 *   out[b,d,t] = act(bias[d] + sum_{k<width} weight[d,k] * xin(t - (width-1) + k))
 *   xin(s) = x[b,d,s] for s >= 0, initial_state[b,d,width-1+s] (or 0) for s < 0
 *
 * with act = SiLU if silu_flag, else identity (a cross-correlation, as in
 * PyTorch: weight[d,width-1] multiplies the current input).
 *
 *   x, out        : [batch, dim, seqlen] io_dtype (out must not overlap x)
 *   weight        : [dim, width] fp32;  bias : [dim] fp32 or NULL
 *   initial_state : [batch, dim, width-1] io_dtype or NULL (zeros): the last
 *                   width-1 inputs of the previous block, oldest first
 *   final_state   : [batch, dim, width-1] io_dtype or NULL (not written): the
 *                   last width-1 inputs of xin, for the next block; must not
 *                   overlap initial_state (MAMBA_ERR_ALIAS) -- use two buffers
 *   width         : 1 .. MAMBA_MAX_CONV_WIDTH (Mamba uses 4), else MAMBA_ERR_SIZE
 *
 * Fast path: seqlen a multiple of 8 (bf16) or 4 (fp32), x and out 16-byte
 * aligned and width-1 at most that vector length; other inputs take a scalar
 * path with the same arithmetic.  Errors as for mamba_selective_scan_fwd.
 * The fast path is launched as a programmatic dependent of the work before it
 * on `stream`, with the same ordering guarantee as the decode step
 * (MAMBA_CONV_PDL=0 launches it plainly).
 */
int mamba_causal_conv1d_fwd(const void *x, const float *weight, const float *bias,
                            const void *initial_state, int silu_flag, void *out,
                            void *final_state, int64_t batch, int64_t dim, int64_t seqlen,
                            int64_t width, int io_dtype, mamba_stream_t stream);

/*
 * Decode step of the conv1d: one new token per row.  out[b,d] is
 * mamba_causal_conv1d_fwd of x[b,d] with seqlen 1 and initial state
 * conv_state[b,d,:]; conv_state is then shifted IN PLACE to hold the last
 * width-1 inputs (the oldest drops out, x[b,d] enters at the end).
 *
 *   conv_state : [batch, dim, width-1] io_dtype (may be NULL when width == 1)
 *   x, out     : [batch, dim] io_dtype;  weight [dim, width], bias [dim] as above
 */
int mamba_causal_conv1d_update(void *conv_state, const void *x, const float *weight,
                               const float *bias, int silu_flag, void *out, int64_t batch,
                               int64_t dim, int64_t width, int io_dtype, mamba_stream_t stream);

/*
 * Wait for the work queued on `stream`, then report and clear the device-side
 * error word of this library's kernels on the current device: MAMBA_ERR_TIMEOUT
 * if a bounded on-device wait (for a bulk copy into shared memory) gave up, in
 * which case the outputs of the affected call are not valid.  Returns
 * MAMBA_ERR_LAUNCH if the synchronisation itself reports a CUDA error.
 */
int mamba_device_status(mamba_stream_t stream);

/* Human-readable name of a mamba_status_t; never NULL. */
const char *mamba_status_string(int status);

/* Version of this ABI (major * 10000 + minor * 100 + patch): 1.1.0 adds the
 * backward, the complex-state scan and the causal conv1d entry points. */
int mamba_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_SCAN_H */
