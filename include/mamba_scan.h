/*
 * mamba_scan.h -- C ABI of the B300 (sm_103a) selective-scan library
 * (libmambascan.so).
 *
 * The library computes the selective state-space recurrence of Mamba for every
 * batch b, channel d and state n:
 *
 *   Delta_t = softplus(Delta_raw_t + bias_d)        (or Delta_raw_t + bias_d)
 *   A_bar_t = exp(Delta_t * A_{d,n})
 *   h_t     = A_bar_t * h_{t-1} + Delta_t * B_{t,n} * u_t
 *   y_t     = (sum_n C_{t,n} * h_t + D_d * u_t) * SiLU(z_t)      (gate optional)
 *
 * Sources: "Mamba state space model" explainer (fsdata.site) §3.2, the
 * selective_step function (softplus step size, A_bar = exp(dt*A),
 * B_bar = dt*B, h = A_bar*h + B_bar*x, y = C.h + D*x); "Mamba: linear-time
 * sequence modelling with selective state spaces" tutorial (freeguideonline)
 * §4.2 step 2 (Delta bias inside the softplus), §4.3 (each channel owns an
 * independent N-wide state), §2.2 (exact zero-order hold), §5.1 (the scan as
 * an associative combination of step transforms), §4.1 (gate branch);
 * "Mamba: Linear-Time Sequence Modeling with Selective State Spaces" summary
 * (ai.xwebgame.com), PyTorch block (the gate is SiLU of the residual branch).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers on the calling thread's current
 *    CUDA device, owned by the caller.  The library never frees or retains
 *    them.  Outputs must not alias inputs.
 *  - Layouts are dense, row-major, innermost dimension last:
 *        u, delta, z, y     [Bsz][Dch][L]     (time contiguous)
 *        B, C               [Bsz][N][L]       (shared by every channel of b)
 *        A                  [Dch][N]  fp32    (real; negative for decay)
 *        D, delta_bias      [Dch]     fp32
 *        last_state, h0     [Bsz][Dch][N] fp32
 *    "dtype" is the storage type of u, delta, z, B, C and y: MAMBA_F32 or
 *    MAMBA_BF16.  State, A, D and bias are always fp32; arithmetic is fp32.
 *  - D, z, delta_bias, last_state (and h0) may be NULL: NULL means absent
 *    (D = 0, no gate, bias = 0, state not written, zero initial state).
 *  - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  A return of MAMBA_OK means the work was
 *    enqueued; device-side failures surface at the caller's next
 *    synchronisation.  Invalid arguments are rejected on the host before any
 *    CUDA call and nothing is launched.
 *  - No C++ exception crosses this interface.  Pointers that are not 16-byte
 *    aligned, or rows whose byte length is not a multiple of 16, select a
 *    slower scalar-load kernel; they are never an error.
 */
#ifndef MAMBA_SCAN_H
#define MAMBA_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle; binary-compatible with cudaStream_t. */
typedef struct CUstream_st *mamba_stream_t;

/* Storage types (the `dtype` argument). */
enum mamba_dtype { MAMBA_F32 = 0, MAMBA_BF16 = 1 };

/* Status codes. */
enum mamba_status {
    MAMBA_OK = 0,
    MAMBA_ERR_NULL_ARG = -1,        /* a required pointer is NULL */
    MAMBA_ERR_BAD_SHAPE = -2,       /* a size is <= 0 (or too large to index) */
    MAMBA_ERR_UNSUPPORTED_N = -3,   /* N > 64 */
    MAMBA_ERR_BAD_DTYPE = -4,       /* dtype is not MAMBA_F32 / MAMBA_BF16 */
    MAMBA_ERR_ALLOC = -5,           /* stream-ordered workspace allocation failed */
    MAMBA_ERR_LAUNCH = -6,          /* a kernel launch failed (cudaGetLastError) */
    MAMBA_ERR_DEVICE_TIMEOUT = -7,  /* a bounded device-side wait expired (mamba_device_error) */
    MAMBA_ERR_BAD_FLAGS = -8,       /* unknown bit in `flags` */
    MAMBA_ERR_WORKSPACE = -9,       /* caller workspace too small or misaligned */
    MAMBA_ERR_DEVICE = -10,         /* no usable CUDA device / query failed */
    MAMBA_ERR_SCRATCH_LIMIT = -11   /* mamba_selective_scan_fwd_noalloc: the sizes need more
                                       scratch than MAMBA_NOALLOC_SCRATCH_BYTES */
};

/* Flags of mamba_selective_scan_fwd_ex. */
#define MAMBA_FLAG_ZOH 0x1     /* exact zero-order hold: B_bar = (exp(Delta*A) - 1) / A * B
                                  (Delta*B where A == 0); freeguideonline tutorial §2.2 */
#define MAMBA_FLAG_REVERSE 0x2 /* scan t = L-1 down to 0 (the reverse SSM stacked for
                                  bidirectional context; fsdata.site explainer §7 table) */

/*
 * Selective scan forward over a whole sequence, zero initial state.
 *
 *   u, delta, z  [Bsz][Dch][L]   delta is Delta_raw (before bias/softplus)
 *   A [Dch][N] fp32, B, C [Bsz][N][L], D [Dch] fp32, delta_bias [Dch] fp32
 *   softplus_flag  non-zero: Delta = softplus(delta + bias); zero: delta + bias
 *   y            [Bsz][Dch][L]   output, same dtype as u
 *   last_state   [Bsz][Dch][N]   fp32 output h_{L-1} (may be NULL)
 *   Bsz, Dch, L >= 1; 1 <= N <= 64
 *
 * When Bsz*Dch is too small to fill the GPU and L is long, the call runs the
 * sequence-parallel chunked scan (chunk end states, an associative carry over
 * the chunks, then a seeded rescan); its workspace is allocated and freed
 * stream-ordered inside the call (cudaMallocAsync / cudaFreeAsync on
 * `stream`).  Returns MAMBA_OK or a negative mamba_status.
 */
int mamba_selective_scan_fwd(const void *u, const void *delta, const float *A, const void *B,
                             const void *C, const float *D, const void *z, const float *delta_bias,
                             int softplus_flag, void *y, float *last_state, int64_t Bsz,
                             int64_t Dch, int64_t L, int64_t N, int dtype, mamba_stream_t stream);

/*
 * Extended forward scan: everything of mamba_selective_scan_fwd, plus
 *   h0          [Bsz][Dch][N] fp32 initial state (NULL = zero).  With
 *               MAMBA_FLAG_REVERSE it is the state "after" t = L, i.e. the
 *               state the backward-in-time scan starts from.
 *   flags       MAMBA_FLAG_ZOH | MAMBA_FLAG_REVERSE (0 = plain forward scan).
 *               With 16-byte aligned rows and 8 < N <= 64 (fp32: N <= 16) a
 *               flagged call runs on the tensor-memory kernel like a plain
 *               one; otherwise on the general scalar-load kernel (slower).
 *   chunk_len   0: automatic choice between the direct and the chunked scan;
 *               > 0: force the chunked scan with chunks of this many steps
 *                    (rounded up to the kernel's time tile);
 *               < 0: force the direct (single pass) scan.
 *               A call without flags, aligned, 8 < N <= 64 (fp32: N <= 16),
 *               chunk_len a multiple of 32 and no convolution runs the
 *               decay-truncated chunked scan: every chunk once from a zero
 *               state (y, end state), the carry, then y += the entering
 *               state's contribution, decayed with no input, up to where it
 *               falls below 2^-16 (bf16 storage) or 2^-30 (fp32 storage) of
 *               that state, at least 2^7 below the rounding of the stored y
 *               (only when the decay is monotone: softplus on, every
 *               A <= 0).  Other calls, and every
 *               call with the environment variable MAMBA_CHUNKED_SCAN=two-pass
 *               (read on every call), run the two-pass scan: chunk end states
 *               from a zero state, the carry, every chunk again from its
 *               entering state.  Both give the same result up to rounding.
 *   workspace, workspace_bytes
 *               caller-owned device scratch for the chunked scan (256-byte
 *               aligned, at least mamba_scan_workspace_size(...) bytes), or
 *               NULL to let the call allocate it stream-ordered.
 * Returns MAMBA_ERR_WORKSPACE if a non-NULL workspace is too small or not
 * 256-byte aligned, MAMBA_ERR_BAD_FLAGS for unknown flag bits.
 */
int mamba_selective_scan_fwd_ex(const void *u, const void *delta, const float *A, const void *B,
                                const void *C, const float *D, const void *z,
                                const float *delta_bias, int softplus_flag, void *y,
                                float *last_state, const float *h0, int64_t Bsz, int64_t Dch,
                                int64_t L, int64_t N, int dtype, int flags, int64_t chunk_len,
                                void *workspace, size_t workspace_bytes, mamba_stream_t stream);

/*
 * Bytes of device workspace the scan needs for these sizes and chunk_len (same
 * meaning as in _ex), on the current device.  0 means the direct scan runs and
 * needs none.  Returns (size_t)-1 if the sizes are invalid or the device query
 * fails.
 */
size_t mamba_scan_workspace_size(int64_t Bsz, int64_t Dch, int64_t L, int64_t N, int64_t chunk_len,
                                 int dtype);

/*
 * One-token recurrent step (selective_state_update) for every (b, d):
 *   state  [Bsz][Dch][N] fp32, read and overwritten in place with h_t
 *   u, delta, z, y  [Bsz][Dch];  B, C [Bsz][N];  A [Dch][N] fp32;  D, delta_bias [Dch] fp32
 *   y = (C . h_t + D*u) * SiLU(z), same dtype as u.
 * Source: the selective_step function of the fsdata.site explainer §3.2
 * applied to a stored state (inference carries only the fixed-size state,
 * same page, §5 table).  D, z, delta_bias may be NULL.  1 <= N <= 64.
 */
int mamba_state_update(float *state, const void *u, const void *delta, const float *A,
                       const void *B, const void *C, const float *D, const void *z,
                       const float *delta_bias, int softplus_flag, void *y, int64_t Bsz,
                       int64_t Dch, int64_t N, int dtype, mamba_stream_t stream);

/*
 * Backward pass of the forward scan (simple discretisation B_bar = Delta B,
 * forward time, zero initial state): gradients of sum(dy * y), the chain rule
 * of the step in the fsdata.site explainer §3.2 (the pages measure training
 * throughput but print no backward pass).
 *
 *   inputs      u, delta, A, B, C, D, z, delta_bias, softplus_flag as in
 *               mamba_selective_scan_fwd; dy [Bsz][Dch][L] (dtype)
 *   du, ddelta  [Bsz][Dch][L] (dtype): gradients for u and Delta_raw
 *   dz          [Bsz][Dch][L] (dtype), required when z is given (else ignored)
 *   dA [Dch][N], dB, dC [Bsz][N][L], dD [Dch], ddelta_bias [Dch]: fp32 sums,
 *               written from zero by the call (dD, ddelta_bias may be NULL)
 * States are recomputed from checkpoints taken every c steps (c = 16, 8 or 4
 * for N <= 16, 32, 64); this call first sweeps the sequence forwards to take
 * them, in a workspace of mamba_scan_bwd_ckpt_size(...) bytes allocated and
 * freed stream-ordered inside the call (mamba_selective_scan_fwd_save and
 * mamba_selective_scan_bwd_from_ckpt below skip that sweep).  dB and dC receive
 * atomic additions, so their low-order bits may vary between runs.  Returns
 * MAMBA_OK, MAMBA_ERR_NULL_ARG, MAMBA_ERR_BAD_SHAPE, MAMBA_ERR_UNSUPPORTED_N,
 * MAMBA_ERR_BAD_DTYPE, MAMBA_ERR_ALLOC or MAMBA_ERR_LAUNCH.
 */
int mamba_selective_scan_bwd(const void *u, const void *delta, const float *A, const void *B, const void *C,
                             const float *D, const void *z, const float *delta_bias, int softplus_flag,
                             const void *dy, void *du, void *ddelta, float *dA, float *dB, float *dC, float *dD,
                             void *dz, float *ddelta_bias, int64_t Bsz, int64_t Dch, int64_t L, int64_t N,
                             int dtype, mamba_stream_t stream);

/*
 * Training pair: a forward scan that also saves the backward pass's
 * checkpoints, and a backward pass that starts from them instead of sweeping
 * the sequence forwards again (the same gradients as mamba_selective_scan_bwd,
 * up to rounding).  No counterpart on the pages, which measure training
 * throughput but print no backward pass: the checkpoints are this library's
 * layout.
 *
 * mamba_scan_bwd_ckpt_size: bytes of the checkpoint buffer,
 *   Bsz*Dch*K*P*4 with c = 16, 8, 4 steps and P = 16, 32, 64 padded states for
 *   N <= 16, 32, 64, and K = ceil(L / c); 0 for invalid sizes.
 * mamba_selective_scan_fwd_save: mamba_selective_scan_fwd as the direct
 *   (single-pass) scan, plus ckpt [Bsz][Dch][K][P] fp32, caller-owned device
 *   memory, 16-byte aligned: entry k (1 <= k < K) receives the state before
 *   step k*c, zero past N; entry 0 is not written.  On 16-byte aligned rows
 *   with 8 < N <= 64 (fp32: N <= 16) the tensor-memory scan writes them as it
 *   goes; otherwise the scan runs and then one more kernel sweeps the
 *   sequence for them.
 * mamba_selective_scan_bwd_from_ckpt: the arguments of mamba_selective_scan_bwd
 *   plus ckpt as written by mamba_selective_scan_fwd_save for the same inputs
 *   (read only; no workspace is allocated).
 * Both return MAMBA_OK, MAMBA_ERR_NULL_ARG, MAMBA_ERR_BAD_SHAPE (also for a
 * misaligned ckpt), MAMBA_ERR_UNSUPPORTED_N, MAMBA_ERR_BAD_DTYPE or
 * MAMBA_ERR_LAUNCH.
 */
size_t mamba_scan_bwd_ckpt_size(int64_t Bsz, int64_t Dch, int64_t L, int64_t N);
int mamba_selective_scan_fwd_save(const void *u, const void *delta, const float *A, const void *B,
                                  const void *C, const float *D, const void *z, const float *delta_bias,
                                  int softplus_flag, void *y, float *last_state, float *ckpt, int64_t Bsz,
                                  int64_t Dch, int64_t L, int64_t N, int dtype, mamba_stream_t stream);
int mamba_selective_scan_bwd_from_ckpt(const void *u, const void *delta, const float *A, const void *B,
                                       const void *C, const float *D, const void *z, const float *delta_bias,
                                       int softplus_flag, const void *dy, const float *ckpt, void *du,
                                       void *ddelta, float *dA, float *dB, float *dC, float *dD, void *dz,
                                       float *ddelta_bias, int64_t Bsz, int64_t Dch, int64_t L, int64_t N,
                                       int dtype, mamba_stream_t stream);

/*
 * Depthwise causal convolution of width 4 followed by SiLU -- the branch that
 * turns x into the scan's input u (ai.xwebgame.com summary, "running it in
 * PyTorch" block: Conv1d(d_inner, d_inner, kernel_size=4, groups=d_inner,
 * padding=3), first L outputs, then SiLU):
 *   u[b][d][t] = SiLU(conv_bias[d] + sum_{k=0..3} conv_w[d][k] x[b][d][t-3+k]),
 *   x[b][d][s] = 0 for s < 0.
 *
 *   x, u        [Bsz][Dch][L], dtype MAMBA_BF16 or MAMBA_F32 (u may not alias x)
 *   conv_w      [Dch][4] fp32;  conv_bias [Dch] fp32 or NULL (0)
 *   silu_flag   non-zero: apply SiLU; zero: write the convolution itself
 * Caller-owned device memory; nothing is allocated or retained.  Returns
 * MAMBA_OK, MAMBA_ERR_NULL_ARG, MAMBA_ERR_BAD_SHAPE, MAMBA_ERR_BAD_DTYPE or
 * MAMBA_ERR_LAUNCH.
 */
int mamba_causal_conv1d_silu(const void *x, const float *conv_w, const float *conv_bias, int silu_flag, void *u,
                             int64_t Bsz, int64_t Dch, int64_t L, int dtype, mamba_stream_t stream);

/*
 * Selective scan fed by the convolution branch: the scan of
 * mamba_selective_scan_fwd with u = SiLU(causal_conv1d(x)) (the function
 * above), u formed inside the scan kernel from x without a round trip through
 * memory where the tensor-memory kernel runs (bf16, 8 < N <= 16, 16-byte
 * aligned rows, gate given); other cases run the convolution into a
 * stream-ordered temporary and then the scan.  y, last_state, D, z, delta_bias
 * as in mamba_selective_scan_fwd; the D * u term of y uses the convolved u.
 * conv_w [Dch][4] fp32, conv_bias [Dch] fp32 or NULL; x [Bsz][Dch][L] in place
 * of u.  Returns the statuses of mamba_selective_scan_fwd.
 */
int mamba_selective_scan_fwd_conv(const void *x, const float *conv_w, const float *conv_bias, const void *delta,
                                  const float *A, const void *B, const void *C, const float *D, const void *z,
                                  const float *delta_bias, int softplus_flag, void *y, float *last_state,
                                  int64_t Bsz, int64_t Dch, int64_t L, int64_t N, int dtype,
                                  mamba_stream_t stream);

/*
 * Chunked forward scan that allocates no device memory (no counterpart in the
 * pages: this is a deployment variant of the chunked scan above).
 *
 * For callers that cannot allocate device memory while they run the scan --
 * a framework that owns every byte of device memory and hands over only the
 * tensors of the call, or host code under a fixed memory budget that must
 * not call (or synchronise with) the allocator.  The caller still provides
 * every input and output; the chunk end states and step sums live in one
 * file-scope __device__ array of MAMBA_NOALLOC_SCRATCH_BYTES bytes, which
 * every GPU that loads the library holds until the process exits.
 *
 * Arguments are those of mamba_selective_scan_fwd_ex without flags and
 * workspace; chunk_len must be >= 1.  The chunks are c = chunk_len rounded up
 * to the kernel's time tile (16 steps for N <= 8, 32 steps otherwise) long, so
 * there are K = ceil(L / c) of them.  When one chunk covers the sequence the
 * direct scan runs and no scratch is touched.  Otherwise the call needs
 * Bsz*K*Dch*N*4 + Bsz*K*Dch*4 bytes of scratch (each part rounded up to a
 * multiple of 256); larger problems return MAMBA_ERR_SCRATCH_LIMIT before
 * anything is launched.  No cudaMalloc/cudaFree or allocating library call
 * is made.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call shares the one array and it keeps the
 * last call's contents (nothing in it needs to start at zero): calls that
 * overlap on the GPU -- on different streams, or from several host threads --
 * race on it, so order them on one stream.
 */
#define MAMBA_NOALLOC_SCRATCH_BYTES (16u << 20)
int mamba_selective_scan_fwd_noalloc(const void *u, const void *delta, const float *A, const void *B,
                                     const void *C, const float *D, const void *z,
                                     const float *delta_bias, int softplus_flag, void *y,
                                     float *last_state, const float *h0, int64_t Bsz, int64_t Dch,
                                     int64_t L, int64_t N, int dtype, int64_t chunk_len,
                                     mamba_stream_t stream);

/*
 * Reads and clears the library's device error word on the current device
 * (synchronous).  Returns MAMBA_ERR_DEVICE_TIMEOUT if a bounded device-side
 * wait of an earlier kernel gave up (that kernel's outputs are then invalid),
 * MAMBA_OK otherwise, MAMBA_ERR_DEVICE if the query fails.
 *
 * The waits in question are those of the tensor-memory scan kernel (input
 * tiles landed, selector MMA done, buffer released by every compute warp),
 * each limited to about one second of the GPU's global timer.  Test hook:
 * with the environment variable MAMBA_TEST_WAIT_POLLS=0 (read on the host at
 * every call) every such wait gives up after one non-blocking test, so the
 * kernel takes its abort path -- it still waits, with a fixed limit, for its
 * own copies and MMAs in flight before it frees tensor memory and returns --
 * and this function then reports MAMBA_ERR_DEVICE_TIMEOUT.
 */
int mamba_device_error(void);

/* Static, human-readable text for a status code (never NULL). */
const char *mamba_status_string(int status);

/*
 * Microbenchmark of the special-function (MUFU) pipe: launches `blocks` CTAs
 * of `threads` threads, each thread running `iters` rounds of 8 independent
 * ex2.approx.ftz.f32; writes per-CTA elapsed SM clock cycles to
 * cycles[blocks] (int64, device memory) and a checksum to sink[blocks*threads]
 * (fp32, device memory) so nothing is optimised away.  Not part of the scan;
 * it measures the exp throughput that bounds it.
 */
int mamba_bench_ex2(int64_t *cycles, float *sink, int64_t iters, int blocks, int threads,
                    mamba_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_SCAN_H */
