/*
 * ssmscan.h -- C ABI of libssmscan, the selective-scan forward pass of the
 * Mamba S6 selective state-space layer on one NVIDIA B300 (sm_103a).
 *
 * What the library computes
 * -------------------------
 * For every batch row b, channel d and state n, starting from h = 0:
 *
 *   dt        = delta[b,t,d] + delta_bias[d]           (bias optional)
 *   dt        = softplus(dt) = log(1 + exp(dt))        (if softplus_flag)
 *   h[b,d,n]  = exp(dt * A[d,n]) * h[b,d,n] + dt * B[b,t,n] * u[b,t,d]
 *   y[b,t,d]  = sum_n C[b,t,n] * h[b,d,n] + D[d] * u[b,t,d]   (D optional)
 *   y[b,t,d] *= z[b,t,d] / (1 + exp(-z[b,t,d]))          (SiLU gate, optional)
 *   h_last[b,d,n] = h after the last step t = L-1          (optional output)
 *
 * The scan and its shapes follow the "State Space Models (SSM)" summary page,
 * section 3.2 "Selective Scan Algorithm" (u, delta (B,L,D); A (D,N);
 * B, C (B,L,N); zero initial state; deltaA = exp(delta A),
 * deltaB_u = delta B u).  The softplus of (delta + bias), the D skip on the
 * scan input and the SiLU(z) gate after the skip follow the SelectiveSSM /
 * MambaBlock listings of that page (sections 5.1-5.2) and of the youngju.dev
 * page "Mamba와 State Space Model 논문 심층 분석".  B is discretised in the
 * simplified form dt * B that every listing on the pages uses.  The state
 * h_last is the only thing a generation step needs to continue a sequence
 * (Obsidian "Mamba" note, section 4.2).  The expanded (B,L,D,N) state is
 * never written to memory: it lives in registers (itwiki "상태 공간 모델",
 * section "Mamba의 선택 메커니즘"; Obsidian note section 5.1).
 *
 * Layout and ownership
 * --------------------
 * All tensors are dense, row-major, last index fastest, no strides:
 *   u, delta, z, y : (batch, L, dim)      B, C   : (batch, L, N)
 *   A              : (dim, N)  fp32       D, delta_bias : (dim,)  fp32
 *   h_last         : (batch, dim, N)  fp32
 * "dim" is the channel count the pages call D (renamed so it does not clash
 * with the skip vector D).  Every pointer is a DEVICE pointer owned by the
 * caller; the library never allocates, frees or keeps a caller's pointer
 * past the call (the only device address it keeps is that of its own static
 * buffer, see ssm_scan_fwd_bf16_noalloc).  Work is enqueued on `stream` and
 * the call returns without
 * synchronising.  The one exception to "never allocates": when the batch
 * rows and channels alone leave most of the GPU idle (few channels, a long
 * sequence), the sequence is cut into time segments (see below) and the call
 * takes (segments - 1) * batch * dim * (N + 1) * 4 bytes of scratch with
 * cudaMallocAsync on `stream` and returns it with cudaFreeAsync on the same
 * stream; ssm_scan_plan() reports both numbers.  y must not overlap any
 * input.  Optional pointers may be
 * NULL: D (no skip), z (no gate), delta_bias (bias 0), h_last (not written).
 * A required pointer may be NULL only when its tensor has no elements (for
 * example u, delta and y when L = 0, which still writes h_last = 0).
 *
 * Precision: the state h and all arithmetic are fp32.  In the bf16 entry
 * point u, delta, B, C, z and y are bf16 (passed as their 16-bit patterns in
 * uint16_t) while A, D, delta_bias and h_last stay fp32; y is rounded to
 * nearest-even.  Results match an fp64 evaluation to |err| <= 1e-4 (1+|ref|)
 * for fp32 inputs and <= 2e-2 (1+|ref|) for bf16 inputs.
 *
 * Time segments
 * -------------
 * The recurrence h_t = a_t h_{t-1} + b_t composes associatively: two spans
 * (a1, b1) then (a2, b2) act as (a1 a2, a2 b1 + b2) (the scan-operator
 * description on the Obsidian "Mamba" note, section 5.1, "parallel scan").
 * For one state, the product of a_t over a span is exp(A * sum of dt), so a
 * span is summarised by its end state from zero and its sum of dt.  A first
 * pass computes these summaries for every segment but the last; the second
 * pass starts each segment from the fold of the summaries before it and
 * produces y and h_last exactly as the sequential loop defines them (up to
 * fp32 rounding order).
 *
 * Errors
 * ------
 * Host-side argument checks return a nonzero ssm_status and launch nothing.
 * Errors that can only be seen on the device (a bounded wait inside a kernel
 * that ran out) are recorded in a device status word and reported by
 * ssm_scan_last_device_status().  No kernel of this library traps.
 */
#ifndef SSMSCAN_H
#define SSMSCAN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

/* The CUDA runtime's stream handle (same definition as the CUDA headers). */
typedef struct CUstream_st *cudaStream_t;

typedef enum {
    SSM_OK = 0,
    SSM_ERR_NULL = 1,            /* a required pointer is NULL                 */
    SSM_ERR_SIZE = 2,            /* a size is negative, N < 1, or a product    */
                                 /* overflows the index range                  */
    SSM_ERR_ALIGN = 3,           /* a pointer is not aligned to its element    */
    SSM_ERR_UNSUPPORTED_N = 4,   /* N > SSM_MAX_N                              */
    SSM_ERR_LAUNCH = 5,          /* the CUDA runtime refused the launch        */
    SSM_ERR_TIMEOUT = 6,         /* a bounded device-side wait ran out         */
    SSM_ERR_ALIAS = 7,           /* y overlaps an input                        */
    SSM_ERR_ARG = 8,             /* an invalid debug key or value              */
    SSM_ERR_NOMEM = 9,           /* stream-ordered scratch allocation failed   */
    SSM_ERR_SCRATCH = 10         /* reserved: the no-alloc entry point's       */
                                 /* static buffer too small (no longer         */
                                 /* returned; it plans fewer segments)         */
} ssm_status;

/* Largest state size N the kernels are built for. */
#define SSM_MAX_N 128

/*
 * fp32 entry point: every tensor is fp32.
 * Returns SSM_OK once the work is enqueued on `stream`.
 */
SSM_API int ssm_scan_fwd(const float *u, const float *delta, const float *A,
                 const float *B, const float *C, const float *D,
                 const float *z, const float *delta_bias, int softplus_flag,
                 float *y, float *h_last,
                 int64_t batch, int64_t L, int64_t dim, int64_t N,
                 cudaStream_t stream);

/*
 * bf16 entry point: u, delta, B, C, z, y are bf16 bit patterns; A, D,
 * delta_bias and h_last are fp32.  Same argument order and meaning as
 * ssm_scan_fwd.
 */
SSM_API int ssm_scan_fwd_bf16(const uint16_t *u, const uint16_t *delta, const float *A,
                      const uint16_t *B, const uint16_t *C, const float *D,
                      const uint16_t *z, const float *delta_bias, int softplus_flag,
                      uint16_t *y, float *h_last,
                      int64_t batch, int64_t L, int64_t dim, int64_t N,
                      cudaStream_t stream);

/*
 * The scan from a given initial state h0 (batch, dim, N) fp32 instead of
 * zeros: h before step 0 is h0, so a sequence run in two calls, the second
 * with h0 = the first call's h_last, gives the outputs of one call over the
 * whole sequence (up to fp32 rounding order).  This is the state the pages'
 * recurrent inference carries from token to token (Obsidian "Mamba" note,
 * section 4.2).  Same arguments as ssm_scan_fwd / ssm_scan_fwd_bf16 with h0
 * after delta_bias; h0 may be NULL (zero state); it is a device pointer
 * owned by the caller and must not overlap y or h_last (returns
 * SSM_ERR_ALIAS): to continue a sequence in place, alternate two state
 * buffers.
 */
SSM_API int ssm_scan_fwd_h0(const float *u, const float *delta, const float *A,
                    const float *B, const float *C, const float *D,
                    const float *z, const float *delta_bias, const float *h0,
                    int softplus_flag, float *y, float *h_last,
                    int64_t batch, int64_t L, int64_t dim, int64_t N,
                    cudaStream_t stream);
SSM_API int ssm_scan_fwd_bf16_h0(const uint16_t *u, const uint16_t *delta, const float *A,
                    const uint16_t *B, const uint16_t *C, const float *D,
                    const uint16_t *z, const float *delta_bias, const float *h0,
                    int softplus_flag, uint16_t *y, float *h_last,
                    int64_t batch, int64_t L, int64_t dim, int64_t N,
                    cudaStream_t stream);

/*
 * The scan with the exact zero-order-hold discretisation of B (itwiki "상태
 * 공간 모델", section "이산화": Bbar = (dt A)^-1 (exp(dt A) - I) dt B), per
 * state
 *   h[n] = exp(dt A[d,n]) h[n] + (exp(dt A[d,n]) - 1) / A[d,n] * B[b,t,n] u[b,t,d]
 * (dt B u where A[d,n] = 0, the limit), instead of the dt B u of the other
 * entry points.  Arguments as ssm_scan_fwd_h0 (h0 may be NULL).  Runs in the
 * warp-specialised kernel only: rows TMA cannot describe return SSM_ERR_ALIGN.
 */
SSM_API int ssm_scan_fwd_zoh(const float *u, const float *delta, const float *A,
                    const float *B, const float *C, const float *D,
                    const float *z, const float *delta_bias, const float *h0,
                    int softplus_flag, float *y, float *h_last,
                    int64_t batch, int64_t L, int64_t dim, int64_t N,
                    cudaStream_t stream);
SSM_API int ssm_scan_fwd_bf16_zoh(const uint16_t *u, const uint16_t *delta, const float *A,
                    const uint16_t *B, const uint16_t *C, const float *D,
                    const uint16_t *z, const float *delta_bias, const float *h0,
                    int softplus_flag, uint16_t *y, float *h_last,
                    int64_t batch, int64_t L, int64_t dim, int64_t N,
                    cudaStream_t stream);

/*
 * The scan with its input produced in the same kernel by the step before it
 * in the Mamba block: a causal depthwise 1-D convolution of kernel size
 * conv_k (1 .. 4) with bias, then SiLU (the MambaBlock listing of the
 * youngju.dev page, and the SelectiveSSM listing, section 5.1, of the "State
 * Space Models (SSM)" summary page: nn.Conv1d(groups = channels, padding =
 * conv_k - 1), trimmed to the first L outputs):
 *
 *   u[b,t,d] = silu( sum_{k<conv_k} conv_w[d,k] x[b, t-(conv_k-1)+k, d] + conv_b[d] ),
 *
 * x = 0 before t = 0; then the scan of ssm_scan_fwd on u (the D skip uses
 * this u).  x is (batch, L, dim) in place of u; conv_w is (dim, conv_k) fp32;
 * conv_b is (dim,) fp32 or NULL.  Everything else as ssm_scan_fwd /
 * ssm_scan_fwd_bf16.  u is never written to memory.  The prologue needs rows
 * that move by TMA (dim x element size a multiple of 16 bytes, x, delta, z, y
 * 16-byte aligned); otherwise the call returns SSM_ERR_ALIGN.
 */
SSM_API int ssm_conv_scan_fwd(const float *x, const float *conv_w, const float *conv_b,
                      int conv_k, const float *delta, const float *A,
                      const float *B, const float *C, const float *D,
                      const float *z, const float *delta_bias, int softplus_flag,
                      float *y, float *h_last, int64_t batch, int64_t L, int64_t dim,
                      int64_t N, cudaStream_t stream);
SSM_API int ssm_conv_scan_fwd_bf16(const uint16_t *x, const float *conv_w, const float *conv_b,
                      int conv_k, const uint16_t *delta, const float *A,
                      const uint16_t *B, const uint16_t *C, const float *D,
                      const uint16_t *z, const float *delta_bias, int softplus_flag,
                      uint16_t *y, float *h_last, int64_t batch, int64_t L, int64_t dim,
                      int64_t N, cudaStream_t stream);

/*
 * The scan on HOST buffers, for callers whose data lives in host memory: the
 * inputs are copied to the device, the scan runs, and y and h_last are copied
 * back, with the copies of one part of the problem overlapping the scan of
 * another (parts are groups of batch rows; with fewer than 4 rows, pieces of
 * the sequence chained through the state).  Every array argument (u, delta,
 * A, B, C, D, z, delta_bias, y, h_last) is a HOST pointer with the layout of
 * ssm_scan_fwd; page-locked (pinned) memory lets the copies run
 * asynchronously.  workspace is a DEVICE buffer of at least
 * ssm_scan_host_workspace_bytes(batch, L, dim, N, dtype) bytes (dtype 0 =
 * fp32, 1 = bf16), 256-byte aligned, owned by the caller; it must not be in
 * use by another call.  The call enqueues everything behind the work already
 * on `stream` and makes `stream` wait for the last copy back: y and h_last
 * are valid after `stream` synchronises.  The library creates and destroys
 * three streams and some events per call.  Results match ssm_scan_fwd within
 * the tolerances above (a part may be planned differently from the whole).
 * Returns SSM_ERR_SIZE if workspace_bytes is too small.
 */
SSM_API int64_t ssm_scan_host_workspace_bytes(int64_t batch, int64_t L, int64_t dim, int64_t N,
                                              int dtype);
SSM_API int ssm_scan_fwd_host(const float *u, const float *delta, const float *A,
                      const float *B, const float *C, const float *D,
                      const float *z, const float *delta_bias, int softplus_flag,
                      float *y, float *h_last, int64_t batch, int64_t L, int64_t dim,
                      int64_t N, void *workspace, int64_t workspace_bytes,
                      cudaStream_t stream);
SSM_API int ssm_scan_fwd_bf16_host(const uint16_t *u, const uint16_t *delta, const float *A,
                      const uint16_t *B, const uint16_t *C, const float *D,
                      const uint16_t *z, const float *delta_bias, int softplus_flag,
                      uint16_t *y, float *h_last, int64_t batch, int64_t L, int64_t dim,
                      int64_t N, void *workspace, int64_t workspace_bytes,
                      cudaStream_t stream);

/*
 * One recurrent (decode) step for every channel: the scan at L = 1 from the
 * state h, which is updated in place.
 *   u, delta, z, y : (batch, dim)      B, C : (batch, N)
 *   A : (dim, N) fp32    D, delta_bias : (dim,) fp32 (may be NULL)
 *   h : (batch, dim, N) fp32, read and written
 * For each (b, d): dt = softplus(delta + bias) (if softplus_flag);
 *   h[n] = exp(dt A[d,n]) h[n] + dt B[b,n] u;  y = (sum_n C[b,n] h[n] + D u) silu(z).
 * fp32 entry: all of u, delta, B, C, z, y fp32.  bf16 entry: those are bf16
 * (16-bit patterns); A, D, delta_bias and h stay fp32.  y must not overlap an
 * input or h, and h must not overlap an input (SSM_ERR_ALIAS).  z may be NULL
 * (no gate).  Enqueued on `stream`; no allocation.  L steps of this call
 * match one L-step ssm_scan_fwd_h0 from the same state within the tolerances
 * above.
 */
SSM_API int ssm_scan_step(const float *u, const float *delta, const float *A,
                  const float *B, const float *C, const float *D,
                  const float *z, const float *delta_bias, int softplus_flag,
                  float *h, float *y, int64_t batch, int64_t dim, int64_t N,
                  cudaStream_t stream);
SSM_API int ssm_scan_step_bf16(const uint16_t *u, const uint16_t *delta, const float *A,
                  const uint16_t *B, const uint16_t *C, const float *D,
                  const uint16_t *z, const float *delta_bias, int softplus_flag,
                  float *h, uint16_t *y, int64_t batch, int64_t dim, int64_t N,
                  cudaStream_t stream);

/*
 * Backward pass: gradients of y of ssm_scan_fwd (fp32, Euler B, zero initial
 * state) with respect to every input, given dy = dL/dy (batch, L, dim):
 *   du, ddelta, dz : (batch, L, dim)     dB, dC : (batch, L, N)
 *   dA : (dim, N)     dD, ddelta_bias : (dim,)
 * ddelta is the gradient with respect to the raw delta (before bias and
 * softplus).  dz, dD, ddelta_bias are written when z, D, delta_bias are given
 * (they may be NULL otherwise).  The state is recomputed rather than stored
 * (doyouknow.kr Mamba guide, section 3-3): the call keeps the state at every
 * 16th step and per-block partial sums in stream-ordered scratch
 * (cudaMallocAsync / cudaFreeAsync on `stream`, about batch * L * dim * N / 4
 * plus 2 * batch * L * N * ceil(dim / 32) fp32 words; for N > 16, which runs
 * as slices of 16 states, also 3 * ceil(N / 16) * batch * L * dim; with time
 * segments, which the call uses when the batch rows and channels leave most
 * of the GPU idle, also about 2 * segments * batch * dim * N).  Partials are
 * folded in a fixed order, so results are deterministic.  The softplus,
 * SiLU and sigmoid inside the backward are the MUFU forms of the bf16
 * forward (about 1e-7 absolute error) for both entry points, so the bf16
 * entry's gradients are this entry's rounded; the fp32 forward's own
 * softplus is the accurate library form, which differs by at most that
 * much.  N <= 128 (otherwise SSM_ERR_UNSUPPORTED_N).  Outputs must not
 * overlap inputs or each other.
 */
SSM_API int ssm_scan_bwd(const float *u, const float *delta, const float *A,
                 const float *B, const float *C, const float *D,
                 const float *z, const float *delta_bias, int softplus_flag,
                 const float *dy, float *du, float *ddelta, float *dA, float *dB,
                 float *dC, float *dD, float *dz, float *ddelta_bias,
                 int64_t batch, int64_t L, int64_t dim, int64_t N, cudaStream_t stream);

/*
 * The same backward pass for the bf16 forward: u, delta, B, C, z, dy and the
 * gradients du, ddelta, dB, dC, dz are bf16 (bit patterns, 2-byte aligned);
 * A, D, delta_bias and dA, dD, ddelta_bias are fp32.  Inputs are widened to
 * fp32 exactly, every sum runs in fp32 (the checkpointed states, the adjoint
 * and the partials of the shared-parameter gradients), and each bf16
 * gradient is rounded once, to nearest even, when it is written.  Scratch,
 * limits, determinism and errors as for ssm_scan_bwd.
 */
SSM_API int ssm_scan_bwd_bf16(const uint16_t *u, const uint16_t *delta, const float *A,
                 const uint16_t *B, const uint16_t *C, const float *D,
                 const uint16_t *z, const float *delta_bias, int softplus_flag,
                 const uint16_t *dy, uint16_t *du, uint16_t *ddelta, float *dA,
                 uint16_t *dB, uint16_t *dC, float *dD, uint16_t *dz, float *ddelta_bias,
                 int64_t batch, int64_t L, int64_t dim, int64_t N, cudaStream_t stream);

/*
 * The backward pass of a piece of a longer sequence: the scan starts from h0
 * (batch, dim, N; fp32, NULL = zero state, as ssm_scan_fwd*_h0) and the loss
 * also depends on the last state through dh_last = dL/dh_last (batch, dim,
 * N; fp32, NULL = zero).  Besides the gradients of ssm_scan_bwd /
 * ssm_scan_bwd_bf16 (same arguments and types) it writes dh0 = dL/dh0
 * (batch, dim, N; fp32; NULL = not written).  A sequence cut into pieces has
 * the gradients of the whole when each piece runs from the previous piece's
 * last state and takes as dh_last the next piece's dh0 (the adjoint
 * recurrence of doyouknow.kr Mamba guide, section 3-3, carried across the
 * cut).  With L = 0, dh0 = dh_last.  dh0 must not overlap any input or
 * output; scratch, limits and errors as for ssm_scan_bwd.
 */
SSM_API int ssm_scan_bwd_h0(const float *u, const float *delta, const float *A,
                 const float *B, const float *C, const float *D,
                 const float *z, const float *delta_bias, int softplus_flag,
                 const float *dy, float *du, float *ddelta, float *dA, float *dB,
                 float *dC, float *dD, float *dz, float *ddelta_bias,
                 const float *h0, const float *dh_last, float *dh0,
                 int64_t batch, int64_t L, int64_t dim, int64_t N, cudaStream_t stream);
SSM_API int ssm_scan_bwd_bf16_h0(const uint16_t *u, const uint16_t *delta, const float *A,
                 const uint16_t *B, const uint16_t *C, const float *D,
                 const uint16_t *z, const float *delta_bias, int softplus_flag,
                 const uint16_t *dy, uint16_t *du, uint16_t *ddelta, float *dA,
                 uint16_t *dB, uint16_t *dC, float *dD, uint16_t *dz, float *ddelta_bias,
                 const float *h0, const float *dh_last, float *dh0,
                 int64_t batch, int64_t L, int64_t dim, int64_t N, cudaStream_t stream);

/*
 * No-allocation variant of ssm_scan_fwd_bf16 (an engineering addition: the
 * pages describe nothing like it).  Same arguments, same kernels, same
 * results bit for bit; the only difference is where the time-segment
 * summaries live.  Instead of cudaMallocAsync scratch they go to one static
 * device buffer of SSM_NOALLOC_SCRATCH_FLOATS fp32 words (8 MiB) that is part
 * of the library's module image, so the call makes no allocation of any kind.
 *
 * For callers that cannot allocate inside the call: a process that has handed
 * (almost) all device memory to its own caching allocator up front, so the
 * driver's pool has no room for cudaMallocAsync; a latency-critical loop that
 * must not enter an allocator (growing a pool maps new pages); and devices
 * where the stream-ordered allocator is unavailable.
 *
 * Limit: a segmented plan needs (segments - 1) * batch * dim * (N + 1) words
 * of summaries.  This entry point takes at most 1 + SSM_NOALLOC_SCRATCH_FLOATS
 * / (batch * dim * (N + 1)) segments, so the summaries always fit: where the
 * allocating entry point would cut the sequence into more segments, this one
 * uses fewer (a plain one-pass call at the extreme), which changes only the
 * speed and the fp32 rounding order, not the definition.  It never returns
 * SSM_ERR_SCRATCH.  The summary pass writes every word the main pass reads,
 * so nothing in the buffer has to start at zero and the call clears nothing.
 *
 * The buffer is shared by every call on a device: two calls in flight at the
 * same time (other streams, other host threads) race on it and give wrong
 * results.  Calls in one stream are ordered and safe.  The first call on a
 * device (and the first in a new context after a device reset) looks up the
 * buffer's address (cudaGetSymbolAddress, with that device current) and keeps
 * it with the context it belongs to; make that first call before any stream
 * capture.
 */
#define SSM_NOALLOC_SCRATCH_FLOATS 2097152
SSM_API int ssm_scan_fwd_bf16_noalloc(const uint16_t *u, const uint16_t *delta,
                      const float *A, const uint16_t *B, const uint16_t *C,
                      const float *D, const uint16_t *z, const float *delta_bias,
                      int softplus_flag, uint16_t *y, float *h_last,
                      int64_t batch, int64_t L, int64_t dim, int64_t N,
                      cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns SSM_OK, SSM_ERR_TIMEOUT if a kernel gave up a
 * bounded wait since the last call (its outputs are then incomplete), or
 * SSM_ERR_LAUNCH if the CUDA runtime reports an error on the stream.
 */
SSM_API int ssm_scan_last_device_status(cudaStream_t stream);

/* Short English text for a status code (static storage, never NULL). */
SSM_API const char *ssm_status_string(int status);

/*
 * Launch plan the library would use for a problem, without launching.
 * dtype: 0 = fp32, 1 = bf16.  On SSM_OK, plan[0..10] receives:
 *   [0] state groups WS                [1] states per lane NPT
 *   [2] timesteps per chunk            [3] channels per block
 *   [4] threads per block              [5] blocks per time segment
 *   [6] dynamic shared bytes           [7] 1 if tiles move by TMA, else 0
 *   [8] time segments (1: one pass)    [9] scratch bytes taken per call
 *   [10] kernel: 1 = phase kernel (every warp prepares, scans and finishes
 *        each chunk in turn), 2 = warp-specialised kernel (a producer warp,
 *        2 prepare warps, the scan warps and 2 finish warps work on
 *        consecutive chunks at the same time; threads [4] include the 5
 *        warps besides the scan warps)
 * Each channel's N states are split over WS warps (state groups), NPT states
 * per lane (N <= WS * NPT); a lane is a channel.
 */
SSM_API int ssm_scan_plan(int64_t batch, int64_t L, int64_t dim, int64_t N, int dtype,
                  int64_t plan[11]);

/*
 * Process-wide knobs for tests and tuning sweeps (not for production use;
 * not thread-safe against concurrent launches).  Keys:
 *   SSM_KNOB_WAIT_NS        give-up time of every device-side wait, in ns
 *                           (default 2e9; must be >= 1000)
 *   SSM_KNOB_FORCE_TIMEOUT  1: every block first waits on a barrier that
 *                           nothing completes, so the wait runs out, the
 *                           block drains its copies and returns, and
 *                           ssm_scan_last_device_status reports
 *                           SSM_ERR_TIMEOUT.  0 (default): off.
 *   SSM_KNOB_STATE_GROUPS   force WS (1, 2, 4 or 8); 0 = automatic
 *   SSM_KNOB_STAGES         force the TMA ring depth (2, 3 or 4); 0 = automatic
 *   SSM_KNOB_CHUNK          force timesteps per chunk (16 or 32); 0 = automatic
 *   SSM_KNOB_PLAIN_LOADS    1: move tiles with plain loads even when TMA applies
 *   SSM_KNOB_SEGMENTS       force the number of time segments (1 .. 64,
 *                           capped at the number of chunks); 0 = automatic
 *   SSM_KNOB_KERNEL         1: the phase kernel; 2 (or 0, automatic): the
 *                           warp-specialised kernel where tiles move by TMA
 *   SSM_KNOB_BWD_SEGMENTS   force the backward's number of time segments
 *                           (1 .. 64, at most one per 16-step chunk; 0 =
 *                           automatic)
 * A forced combination the library is not built for falls back to automatic.
 * Returns SSM_OK or SSM_ERR_ARG.
 */
enum {
    SSM_KNOB_WAIT_NS = 1,
    SSM_KNOB_FORCE_TIMEOUT = 2,
    SSM_KNOB_STATE_GROUPS = 3,
    SSM_KNOB_CHUNK = 4,
    SSM_KNOB_PLAIN_LOADS = 5,
    SSM_KNOB_STAGES = 6,
    SSM_KNOB_SEGMENTS = 7,
    SSM_KNOB_KERNEL = 8,
    SSM_KNOB_BWD_SEGMENTS = 9
};
SSM_API int ssm_set_knob(int key, int64_t value);

#ifdef __cplusplus
}
#endif

#endif /* SSMSCAN_H */
