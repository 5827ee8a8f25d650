/*
 * ssm.h -- C ABI of the GB300 (sm_103a) selective state-space scan library.
 *
 * Three operations, each a hand-written CUDA kernel on one GPU:
 *
 *   ssm_scan_fwd     selective scan, per-channel per-state A (Mamba-1 form)
 *   ssd_chunked_fwd  scalar-A-per-head chunked SSD (Mamba-2 form), tensor cores
 *   ssm_decode_step  single-token state update, in place
 *   ssd_mamba3_fwd, ssm_decode_step_mamba3  the same two for Mamba-3 SISO
 *                    (trapezoidal three-term recurrence)
 *   ssd_mamba3_mimo_fwd, ssm_decode_step_mamba3_mimo  Mamba-3 MIMO (rank R)
 *   ssm_mamba3_rope  Mamba-3's data-dependent rotation of B and C
 *   ssm_scan_bwd     gradient of ssm_scan_fwd (reverse mode, every input)
 *   ssm_scan_fwd_host  ssm_scan_fwd on host-resident activations, copies pipelined
 *   ssd_chunked_bwd  gradient of ssd_chunked_fwd, tensor cores
 *   ssd_mamba3_bwd   gradient of ssd_mamba3_fwd (Mamba-3 SISO)
 *   ssd_mamba3_mimo_bwd  gradient of ssd_mamba3_mimo_fwd (Mamba-3 MIMO)
 *
 * Conventions shared by every entry point
 *  - Pointers are DEVICE pointers unless stated otherwise, to dense row-major
 *    (C-contiguous) arrays in the layouts given per function.  The caller owns
 *    every buffer, including the scan's workspace; the library allocates no
 *    device memory.  State it keeps between calls: ssm_scan_fwd_host's copy
 *    streams and events, ssm_scan_fwd_noalloc's fixed scratch array, and the
 *    ssm_debug_set_lookback setting.
 *  - Every base pointer must be 16-byte aligned (any cudaMalloc or PyTorch
 *    allocation is), else SSM_ERR_ALIGN.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Work is only enqueued on it; no entry point synchronises
 *    except ssm_last_device_status.
 *  - Arguments are checked on the host before anything is enqueued; on any
 *    error nothing is launched and the error code is returned.  A launch
 *    failure returns SSM_ERR_CUDA.  Device-side waits are bounded: if one
 *    runs out, the kernel records SSM_ERR_TIMEOUT in the workspace (read it
 *    with ssm_last_device_status) and finishes without hanging; its outputs
 *    are then undefined.  No entry point aborts, prints or traps.
 *  - Outputs must not overlap inputs (SSM_ERR_ALIAS).  Inputs are never
 *    written, except `state` of ssm_decode_step, which is updated in place.
 *  - All state and accumulation is fp32.  `in_dtype` is the type of the
 *    activations (u/delta/z/B/C, or x/B/C); `out_dtype` the type of y.
 *    A, D, delta_bias, dt and every state array are always fp32.
 *
 * Page citations are by page title and section.
 */
#ifndef SSM_GB300_H
#define SSM_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSM_OK = 0,
    SSM_ERR_NULL = 1,        /* a required pointer is NULL */
    SSM_ERR_SHAPE = 2,       /* a size is negative or inconsistent */
    SSM_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
    SSM_ERR_DTYPE = 4,       /* unknown dtype code */
    SSM_ERR_UNSUPPORTED = 5, /* valid, but not a size this library implements */
    SSM_ERR_WORKSPACE = 6,   /* workspace NULL or smaller than required */
    SSM_ERR_TIMEOUT = 7,     /* a bounded device-side wait ran out */
    SSM_ERR_CUDA = 8,        /* a CUDA runtime call or a launch failed */
    SSM_ERR_ALIAS = 9        /* an output overlaps an input */
} ssm_status_t;

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype_t;

/* Version of this ABI (incremented on any incompatible change). */
int ssm_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* ssm_status_string(ssm_status_t status);

/*
 * Bytes of device workspace ssm_scan_fwd needs for this problem (a pure
 * function of its arguments; 0 never returned for a valid problem).
 * Returns 0 if the arguments are invalid.
 */
size_t ssm_scan_workspace_bytes(int batch, int dim, int seqlen, int dstate, int ngroups);

/*
 * Selective scan.
 *   "We brought Mamba to Trainium -- and mapped where custom kernels actually
 *   help", section "Mamba: bringing an unsupported model to the chip, and
 *   writing its missing kernel": h_t = A_t h_{t-1} + B_t x_t, y_t = sum_n C_t h_t.
 *   "Mamba-3 NKI Kernels for AWS Neuron", section "How it works": Phase 0,
 *   dt = softplus(dt + dt_bias) and alpha = exp(dt A); Phase 5, D skip then
 *   silu gate.
 *
 * For every batch b, channel d (group g = d / (dim / ngroups)), step t and
 * state n, in fp32:
 *   dl      = delta[b,d,t] + delta_bias[d];  dl = softplus(dl) if delta_softplus
 *   h[n]    = exp(dl * A[d,n]) * h[n] + dl * B[b,g,n,t] * u[b,d,t]
 *   y[b,d,t] = (sum_n C[b,g,n,t] h[n] + D[d] u[b,d,t]) * silu(z[b,d,t])
 * starting from h = initial_state[b,d,:] (or 0); final_state[b,d,:] = h
 * after the last step.
 *
 * Layouts (in_dtype for u, delta, z, B, C; out_dtype for y):
 *   u, delta, z, y    (batch, dim, seqlen)          seqlen contiguous
 *   A                 (dim, dstate)        fp32
 *   B, C              (batch, ngroups, dstate, seqlen)
 *   D, delta_bias     (dim,)               fp32, each may be NULL (0)
 *   z                 may be NULL (no gate)
 *   initial_state     (batch, dim, dstate) fp32, may be NULL (zero state)
 *   final_state       (batch, dim, dstate) fp32, may be NULL (not written)
 *   workspace         device memory of at least
 *                     ssm_scan_workspace_bytes(...) bytes; its contents on
 *                     entry do not matter; it must not be used by another
 *                     call that may run concurrently.
 * Supported: dstate == 16; dim % ngroups == 0; any batch, dim, seqlen >= 0.
 * seqlen == 0 writes final_state = initial_state (or 0).
 *
 * Two kernels compute it (the same result up to fp32 rounding order):
 *  - batch * dim > 3072: the work-efficient chained scan.  Each channel's 16
 *    states sit in registers and walk the sequence in order (one exp per
 *    element); when the channel blocks outnumber the GPU's resident CTA slots
 *    the sequence is cut into chunks chained through the state.
 *  - batch * dim <= 3072 (too few channels to fill the GPU): the
 *    sequence-parallel scan.  The sequence is cut into 128-step chunks (one
 *    CTA each) and each chunk into 8, 16 or 32 segments (one lane each); a
 *    span of steps acts on the state as h -> P h + q and spans compose by
 *    (P1, q1) o (P2, q2) = (P1 P2, P2 q1 + q2) (the associativity of the first
 *    page's section "We built the parallel scan -- and it taught us something
 *    sharper").  Lanes combine their segments with warp shuffles; chunks
 *    combine through a decoupled look-back in the workspace, each chunk
 *    publishing its aggregate (P, q) before it knows its entry state.  Every
 *    element then costs two exps (one pass from zero, one replay).
 */
ssm_status_t ssm_scan_fwd(const void* u, const void* delta, const float* A,
                          const void* B, const void* C, const float* D, const void* z,
                          const float* delta_bias, int delta_softplus,
                          const float* initial_state, void* y, float* final_state,
                          int batch, int dim, int seqlen, int dstate, int ngroups,
                          ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Chunked SSD, scalar A per head.
 *   "Mamba-3 NKI Kernels for AWS Neuron", section "Kernel details",
 *   mamba3_siso_ssd_kernel (the Mamba-2 SSD structure, chunk 64, stated to be
 *   mathematically equivalent to the recurrence), and section
 *   "Configuration constraints" (seqlen must be divisible by chunk_size).
 *
 * Computes, exactly up to rounding, the recurrence
 *   S[p,n] = exp(dt[b,t,h] A_head[h]) S[p,n] + dt[b,t,h] B[b,t,g,n] x[b,t,h,p]
 *   y[b,t,h,p] = sum_n C[b,t,g,n] S[p,n]
 * from S = initial_state[b,h] (0 when initial_state is NULL; g = h /
 * (nheads / ngroups)); final_state[b,h,p,n] = S after the last step.  dt is
 * taken as given (already discretised).  With initial_state the call resumes
 * a sequence: the SSD over L1 + L2 steps equals the SSD over L1 steps followed
 * by the SSD over L2 steps from its final state.
 *
 * Layouts: x, y (batch, seqlen, nheads, headdim); dt (batch, seqlen, nheads)
 * fp32; A_head (nheads,) fp32; B, C (batch, seqlen, ngroups, dstate);
 * initial_state, final_state (batch, nheads, headdim, dstate) fp32, each may
 * be NULL; initial_state may be the same buffer as final_state (updated in
 * place), any other overlap returns SSM_ERR_ALIAS.
 * Supported: chunk == 64, headdim == 64, dstate == 128, in_dtype == SSM_BF16,
 * seqlen % chunk == 0 (else SSM_ERR_SHAPE), nheads % ngroups == 0.
 * `chunk` is the granularity the call validates (the pages' chunk size and
 * their seqlen % chunk rule); the kernel itself evaluates the chunked form in
 * 128-step blocks, so that every product is an M = 128 tensor-core MMA.  The
 * chunked form equals the recurrence for any block length, so the result does
 * not depend on this choice beyond fp32 rounding.
 * seqlen == 0 writes final_state = initial_state (or 0).
 */
ssm_status_t ssd_chunked_fwd(const void* x, const float* dt, const float* A_head,
                             const void* B, const void* C, int chunk,
                             const float* initial_state, void* y, float* final_state,
                             int batch, int seqlen, int nheads, int headdim, int dstate,
                             int ngroups, ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                             void* stream);

/*
 * Mamba-3 SISO chunked prefill (trapezoidal discretisation), scalar A per head.
 *   "Mamba-3 NKI Kernels for AWS Neuron", section "How it works" (Phase 0:
 *   alpha = exp(dt A), gamma = lambda dt, beta = (dt - gamma) alpha; Eq. 9)
 *   and section "Kernel details", mamba3_siso_ssd_kernel (single-SSD form
 *   with scale = gamma + dt_{t+1} (1 - lambda_{t+1}) and a diagonal
 *   correction, chunk 64).
 *
 * Computes, exactly up to rounding, the recurrence (u_t = B[b,t,g] (x) x[b,t,h])
 *   S = alpha_t S + beta_t u_{t-1} + gamma_t u_t,   y[b,t,h,p] = sum_n C[b,t,g,n] S[p,n]
 * from S = initial_state[b,h] (0 when NULL), where u_{-1} = prev_B[b,g] (x)
 * prev_x[b,h] is the token before the first (both NULL: none).  dt and lam
 * are taken as given (dt after softplus, lambda after sigmoid); rotary
 * position terms on B and C are applied by the caller (B, C are the rotated
 * tensors; per-head rotations use ngroups == nheads).  final_state is S after
 * the last step; with prev_B = B[:, L-1], prev_x = x[:, L-1] a later call
 * (or ssm_decode_step_mamba3) continues the sequence.
 *
 * Layouts as ssd_chunked_fwd; lam (batch, seqlen, nheads) fp32; prev_B
 * (batch, ngroups, dstate) and prev_x (batch, nheads, headdim) in in_dtype.
 * Supported: as ssd_chunked_fwd.  prev_B and prev_x must be both NULL or both
 * given (else SSM_ERR_NULL); lam must be given.  The pages give no
 * counterpart to the resumption inputs: they follow from Eq. 9.
 */
ssm_status_t ssd_mamba3_fwd(const void* x, const float* dt, const float* lam,
                            const float* A_head, const void* B, const void* C, int chunk,
                            const float* initial_state, const void* prev_B, const void* prev_x,
                            void* y, float* final_state,
                            int batch, int seqlen, int nheads, int headdim, int dstate,
                            int ngroups, ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                            void* stream);

/*
 * Mamba-3 MIMO (rank R) chunked prefill.
 *   "Mamba-3 NKI Kernels for AWS Neuron", section "Kernel details",
 *   mamba3_mimo_ssd_kernel (rank flattening: the (step, rank) pairs of a chunk
 *   are taken as chunk * R sub-tokens, with a block-diagonal correction;
 *   chunk 16 for R = 4) and mamba3_mimo_decode_kernel (the rank-R terms).
 *
 * Computes, exactly up to rounding, per (b, h) with BX_t[n,p] = sum_r
 * B[b,t,r,g,n] x[b,t,r,h,p]:
 *   S = alpha_t S + beta_t BX_{t-1} + gamma_t BX_t
 *   y[b,t,r,h,p] = sum_n C[b,t,r,g,n] S[p,n]
 * with the coefficients, initial state and previous token of ssd_mamba3_fwd.
 *
 * Layouts: x, y (batch, seqlen, rank, nheads, headdim); B, C (batch, seqlen,
 * rank, ngroups, dstate); dt, lam (batch, seqlen, nheads) fp32; prev_B (batch,
 * rank, ngroups, dstate) and prev_x (batch, rank, nheads, headdim) in
 * in_dtype; states as ssd_chunked_fwd.  seqlen counts steps.
 * Supported: rank 1, 2 or 4 with chunk * rank == 64; otherwise as
 * ssd_mamba3_fwd (rank 1 is ssd_mamba3_fwd).
 */
ssm_status_t ssd_mamba3_mimo_fwd(const void* x, const float* dt, const float* lam,
                                 const float* A_head, const void* B, const void* C, int chunk,
                                 int rank, const float* initial_state, const void* prev_B,
                                 const void* prev_x, void* y, float* final_state,
                                 int batch, int seqlen, int nheads, int headdim, int dstate,
                                 int ngroups, ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                                 void* stream);

/*
 * One decode step, in place.
 *   "Mamba-3 NKI Kernels for AWS Neuron", section "How it works", decode via
 *   step(), Eq. 9 with lambda = 1 (beta = 0, gamma = dt), and Phase 5 (D skip,
 *   silu gate); section "Kernel details", mamba3_siso_decode_state_kernel.
 *
 *   alpha = exp(dt[b,h] A[h])
 *   state[b,h,p,n] = alpha state[b,h,p,n] + dt[b,h] x[b,h,p] B[b,g,n]
 *   y[b,h,p] = (sum_n C[b,g,n] state[b,h,p,n] + D[h] x[b,h,p]) * silu(z[b,h,p])
 *
 * Layouts: state (batch, nheads, headdim, dstate) fp32, read and written;
 * x, z, y (batch, nheads, headdim) in dtype; dt (batch, nheads) fp32;
 * A, D (nheads,) fp32 (D may be NULL); B, C (batch, ngroups, dstate) in
 * dtype; z may be NULL.  Supported: dstate 16, 32, 64, 128 or 256 (else
 * SSM_ERR_UNSUPPORTED).
 */
ssm_status_t ssm_decode_step(float* state, const void* x, const float* dt,
                             const float* A, const void* B, const void* C,
                             const float* D, const void* z, void* y,
                             int batch, int nheads, int headdim, int dstate, int ngroups,
                             ssm_dtype_t dtype, void* stream);

/*
 * One Mamba-3 SISO decode step, in place.
 *   "Mamba-3 NKI Kernels for AWS Neuron", section "How it works", decode via
 *   step(), Eq. 9 (h_t = alpha h_{t-1} + beta prev_Bx + gamma B_t (x) x_t,
 *   y_t = C_t^T h_t) and Phase 5; section "Kernel details",
 *   mamba3_siso_decode_state_kernel.
 *
 *   alpha = exp(dt A), gamma = lam dt, beta = (dt - gamma) alpha
 *   state = alpha state + beta prev_B (x) prev_x + gamma B (x) x
 *   y = (sum_n C state + D x) * silu(z)
 *
 * Arguments as ssm_decode_step, plus lam (batch, nheads) fp32 (lambda after
 * sigmoid) and the previous token's prev_B (batch, ngroups, dstate) and
 * prev_x (batch, nheads, headdim) in dtype (all required; pass the last
 * prefill token's B and x after ssd_mamba3_fwd, then each step's own).
 */
ssm_status_t ssm_decode_step_mamba3(float* state, const void* prev_B, const void* prev_x,
                                    const void* x, const float* dt, const float* lam,
                                    const float* A, const void* B, const void* C, const float* D,
                                    const void* z, void* y, int batch, int nheads, int headdim,
                                    int dstate, int ngroups, ssm_dtype_t dtype, void* stream);

/*
 * One Mamba-3 MIMO (rank R) decode step, in place.
 *   "Mamba-3 NKI Kernels for AWS Neuron", section "Kernel details",
 *   mamba3_mimo_decode_kernel (BX = sum_r B[n,r] x[p,r]; y[p,r] = sum_n
 *   state[n,p] C[n,r]), with the Eq. 9 coefficients and Phase 5 per rank.
 *
 *   state = alpha state + beta sum_r prev_B[r] (x) prev_x[r] + gamma sum_r B[r] (x) x[r]
 *   y[b,r,h,p] = (sum_n C[b,r,g,n] state[b,h,p,n] + D[h] x[b,r,h,p]) * silu(z[b,r,h,p])
 *
 * Layouts: x, z, y, prev_x (batch, rank, nheads, headdim); B, C, prev_B
 * (batch, rank, ngroups, dstate); others as ssm_decode_step_mamba3.
 * Supported: rank 1 (as ssm_decode_step_mamba3), 2 or 4 with dstate == 128.
 */
ssm_status_t ssm_decode_step_mamba3_mimo(float* state, const void* prev_B, const void* prev_x,
                                         const void* x, const float* dt, const float* lam,
                                         const float* A, const void* B, const void* C,
                                         const float* D, const void* z, void* y, int batch,
                                         int rank, int nheads, int headdim, int dstate,
                                         int ngroups, ssm_dtype_t dtype, void* stream);

/*
 * Mamba-3's data-dependent rotation of B and C.
 *   "Mamba-3 NKI Kernels for AWS Neuron", section "How it works", Phase 1:
 *   the angle cumsum cum_angles = -cumsum(dt * theta), then RoPE applied to B
 *   and C -- the page's "complex-valued state via data-dependent RoPE".
 *
 * For every batch b, head h (group g = h / (nheads / ngroups)), state pair
 * k < dstate / 2, step t and rank r, in fp32:
 *   angle   = angle0[b,h,k] (0 when angle0 is NULL), then per step
 *   angle  -= dt[b,t,h] * theta[b,t,h,k]          (inclusive cumsum)
 *   (B_rot[b,t,r,h,2k], B_rot[b,t,r,h,2k+1]) = the pair (B[b,t,r,g,2k],
 *       B[b,t,r,g,2k+1]) rotated by angle: (x cos - y sin, x sin + y cos);
 *   the same for C;  angle_out[b,h,k] = angle after the last step.
 * The rotated rows are per head, so the SSD and decode entry points take
 * them with ngroups = nheads.  With seqlen = 1 this is the rotation of one
 * decode step (angle0 = the previous step's angle_out; angle_out may be
 * angle0 itself, updated in place).  The angle is carried as a compensated
 * float-float sum (the steps of a tile scanned in segments, the segment sums
 * composed by TwoSum): its error stays near one rounding of its value (about
 * 1e-7 |angle|); angle_out is that sum rounded once to fp32.
 *
 * Layouts (dtype for B, C, B_rot, C_rot; everything else fp32):
 *   B, C            (batch, seqlen, rank, ngroups, dstate)   rank 1 = SISO
 *   dt              (batch, seqlen, nheads)   already discretised (softplus)
 *   theta           (batch, seqlen, nheads, dstate / 2)
 *   angle0, angle_out (batch, nheads, dstate / 2), each may be NULL
 *   B_rot, C_rot    (batch, seqlen, rank, nheads, dstate)
 * Supported: any sizes with dstate even, nheads % ngroups == 0, rank >= 1.
 * Outputs may not overlap inputs (except angle_out == angle0).
 */
ssm_status_t ssm_mamba3_rope(const void* B, const void* C, const float* dt, const float* theta,
                             const float* angle0, void* B_rot, void* C_rot, float* angle_out,
                             int batch, int seqlen, int rank, int nheads, int ngroups, int dstate,
                             ssm_dtype_t dtype, void* stream);

/*
 * Selective scan for callers that cannot allocate device memory.
 *
 * No counterpart on the pages: this is an interface addition of this
 * library.  Some callers of this code cannot call cudaMalloc (or any
 * allocator) when they run the scan: an inference-engine plug-in whose device
 * memory is budgeted once at start-up, a real-time loop that may not take
 * cudaMalloc's implicit device synchronisation or its unbounded latency, or a
 * thin C wrapper that has no handle on the framework's caching allocator.
 * For them this entry point computes exactly what ssm_scan_fwd computes, with
 * the same arguments except that there is no workspace: its scratch lives in
 * a fixed 4 MiB array inside the library's device image, which every GPU that
 * loads the library holds until the process exits.  It allocates nothing.
 *
 *  - Limit: problems whose scratch exceeds 4 MiB are rejected with
 *    SSM_ERR_WORKSPACE before anything is enqueued; ssm_scan_fwd with a
 *    caller-supplied workspace handles them.  The scratch is a 256-byte
 *    header, plus, for the chained scan split into L-chunks on this GPU, one
 *    flag per chunk and channel block and 64 bytes of carried state per
 *    channel and chunk; for the sequence-parallel scan (batch * dim <= 3072,
 *    more than 128 steps), one flag per 128-step chunk and channel block and
 *    192 bytes of aggregate and state per channel and chunk.
 *  - The first call on each device (and the first after a cudaDeviceReset
 *    gave the device a new context) looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - All calls on a device share the one array, which keeps the contents the
 *    last call left; each call clears what must start at zero on its stream.
 *    Calls whose executions overlap on the GPU (different streams, or
 *    different host threads without ordering) race on the array and give
 *    undefined results: serialise them.
 *  - A device-side wait that runs out records SSM_ERR_TIMEOUT in the array's
 *    header, as ssm_scan_fwd does in its workspace: read it with
 *    ssm_noalloc_last_status (ssm_last_device_status has no workspace to
 *    read here).
 */
ssm_status_t ssm_scan_fwd_noalloc(const void* u, const void* delta, const float* A,
                                  const void* B, const void* C, const float* D, const void* z,
                                  const float* delta_bias, int delta_softplus,
                                  const float* initial_state, void* y, float* final_state,
                                  int batch, int dim, int seqlen, int dstate, int ngroups,
                                  ssm_dtype_t in_dtype, ssm_dtype_t out_dtype, void* stream);

/*
 * Waits for `stream` to drain, then returns the device-side status that the
 * last ssm_scan_fwd_noalloc on the current device recorded in its scratch
 * array (SSM_OK or SSM_ERR_TIMEOUT), or SSM_ERR_CUDA if the stream reports an
 * error.  Allocates nothing (the status is copied into a host stack variable).
 * No counterpart on the pages.
 */
ssm_status_t ssm_noalloc_last_status(void* stream);

/*
 * Bytes of the checkpoints ssm_scan_fwd_ckpt keeps: the state entering every
 * 16-step segment, [ceil(seqlen / 16)][batch * dim][16] fp32.  0 if invalid.
 */
size_t ssm_scan_checkpoint_bytes(int batch, int dim, int seqlen, int dstate);

/*
 * ssm_scan_fwd that also keeps, in `checkpoints` (device, at least
 * ssm_scan_checkpoint_bytes(...) bytes, not overlapping anything else), the
 * state entering every 16-step segment -- what ssm_scan_bwd needs, so that a
 * training step does not run the forward recurrence twice.  y and final_state
 * are exactly ssm_scan_fwd's; the same arguments and errors, plus SSM_ERR_NULL
 * for a NULL `checkpoints` when there is work.  (For batch * dim <= 3072,
 * where ssm_scan_fwd runs the sequence-parallel scan, y and final_state come
 * from that scan and the checkpoints from a second, states-only pass of the
 * chained scan.)
 */
ssm_status_t ssm_scan_fwd_ckpt(const void* u, const void* delta, const float* A, const void* B,
                               const void* C, const float* D, const void* z,
                               const float* delta_bias, int delta_softplus,
                               const float* initial_state, void* y, float* final_state,
                               float* checkpoints, int batch, int dim, int seqlen, int dstate,
                               int ngroups, ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace ssm_scan_bwd needs for this problem (a pure
 * function of its arguments).  Returns 0 if the arguments are invalid.
 * About (ceil(seqlen / 16) * batch * dim * 64 + ceil(dim / ngroups / 32) *
 * batch * ngroups * seqlen * 128) bytes plus ssm_scan_workspace_bytes.
 */
size_t ssm_scan_bwd_workspace_bytes(int batch, int dim, int seqlen, int dstate, int ngroups);

/*
 * Gradient of the selective scan.
 *   The forward operation is ssm_scan_fwd's ("We brought Mamba to Trainium --
 *   and mapped where custom kernels actually help", section "Mamba: bringing
 *   an unsupported model to the chip, and writing its missing kernel", with
 *   the discretisation, D skip and gate of "Mamba-3 NKI Kernels for AWS
 *   Neuron", section "How it works").  The second page reports gradient
 *   parity of its mixer (section "Correctness", backward parity through
 *   autograd) but prints no backward formula; this is the exact reverse-mode
 *   derivative of the recurrence.
 *
 * For the scalar loss  sum(dy * y) + sum(dfinal_state * final_state), with y
 * and final_state what ssm_scan_fwd returns for the same inputs, writes the
 * loss's derivative with respect to every input:
 *   du, ddelta            (batch, dim, seqlen)            fp32
 *   dA                    (dim, dstate)                   fp32
 *   dB, dC                (batch, ngroups, dstate, seqlen) fp32
 *   dD, ddelta_bias       (dim,)                          fp32, may be NULL
 *   dz                    (batch, dim, seqlen)            fp32
 *   dinitial_state        (batch, dim, dstate)            fp32, may be NULL
 * ddelta is the derivative with respect to the raw delta (through the
 * softplus when delta_softplus is set).  dD and ddelta_bias are written
 * whenever they are non-NULL, also when D or delta_bias is NULL (then they are
 * the derivative at D = 0 or delta_bias = 0).  dz is required when z is given
 * (SSM_ERR_NULL otherwise) and ignored when z is NULL.  dinitial_state is the
 * derivative with respect to the initial state (zero when initial_state is
 * NULL).
 *
 * Inputs: u, delta, A, B, C, D, z, delta_bias, delta_softplus, initial_state
 * exactly as for ssm_scan_fwd; dy (batch, dim, seqlen) in in_dtype;
 * dfinal_state (batch, dim, dstate) fp32 or NULL (zero); checkpoints: the
 * states ssm_scan_fwd_ckpt kept for the same inputs, or NULL (the call then
 * re-runs the forward recurrence to make them).
 * workspace: at least ssm_scan_bwd_workspace_bytes(...) bytes, contents on
 * entry irrelevant, not shared with a concurrent call.  ssm_last_device_status
 * reads it afterwards like ssm_scan_fwd's (the call runs the forward
 * recurrence once more to store the state every 16 steps, then sweeps
 * backwards; both run on `stream`).
 * Every output must be disjoint from every input, from the other outputs and
 * from the workspace (SSM_ERR_ALIAS).  The sums over channels (dB, dC) and
 * over the batch (dA, dD, ddelta_bias) are added in a fixed order: the result
 * is the same on every run.
 * Supported: dstate == 16; dim % ngroups == 0; any batch, dim, seqlen >= 0.
 * With no steps (seqlen == 0 or batch == 0) dA, dD, ddelta_bias are zeroed and
 * dinitial_state = dfinal_state (or 0); the workspace is not touched then.
 */
ssm_status_t ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B,
                          const void* C, const float* D, const void* z, const float* delta_bias,
                          int delta_softplus, const float* initial_state, const void* dy,
                          const float* dfinal_state, const float* checkpoints, float* du,
                          float* ddelta, float* dA,
                          float* dB, float* dC, float* dD, float* dz, float* ddelta_bias,
                          float* dinitial_state, int batch, int dim, int seqlen, int dstate,
                          int ngroups, ssm_dtype_t in_dtype, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * Bytes of the block states ssd_chunked_fwd_ckpt keeps: the state entering
 * every 128-step block and the final state, [batch * nheads][ceil(seqlen / 128)
 * + 1][headdim][dstate] fp32.  0 if invalid or unsupported.
 */
size_t ssd_chunked_checkpoint_bytes(int batch, int seqlen, int nheads, int headdim, int dstate);

/*
 * ssd_chunked_fwd that also keeps the block states (device, at least
 * ssd_chunked_checkpoint_bytes(...) bytes, not overlapping anything else) for
 * ssd_chunked_bwd, so that a training step runs the forward once.  y and
 * final_state are exactly ssd_chunked_fwd's (y may be NULL: states only); the
 * same arguments and errors, plus SSM_ERR_NULL for a NULL `block_states` when
 * there is work.  With seqlen == 0 nothing is written to block_states.
 */
ssm_status_t ssd_chunked_fwd_ckpt(const void* x, const float* dt, const float* A_head,
                                  const void* B, const void* C, int chunk,
                                  const float* initial_state, void* y, float* final_state,
                                  float* block_states, int batch, int seqlen, int nheads,
                                  int headdim, int dstate, int ngroups, ssm_dtype_t in_dtype,
                                  ssm_dtype_t out_dtype, void* stream);

/*
 * ssd_mamba3_fwd and ssd_mamba3_mimo_fwd that also keep the states their
 * chunked form carries between 128-row blocks (device, at least
 * ssd_chunked_checkpoint_bytes(batch, seqlen * rank, nheads, headdim, dstate)
 * bytes, not overlapping anything else) for ssd_mamba3_bwd /
 * ssd_mamba3_mimo_bwd, so that a training step runs the forward once.  These
 * are the states of S + c_t BX_t (c_t = dt_{t+1} (1 - lambda_{t+1})), the form
 * the gradients walk.  y and final_state are exactly the plain forwards' (y may
 * be NULL: states only); the same arguments and errors, plus SSM_ERR_NULL for a
 * NULL `block_states` when there is work.  The pages have no counterpart: these
 * keep what an autograd training step would save between the forward and the
 * backward pass.
 */
ssm_status_t ssd_mamba3_fwd_ckpt(const void* x, const float* dt, const float* lam,
                                 const float* A_head, const void* B, const void* C, int chunk,
                                 const float* initial_state, const void* prev_B,
                                 const void* prev_x, void* y, float* final_state,
                                 float* block_states, int batch, int seqlen, int nheads,
                                 int headdim, int dstate, int ngroups, ssm_dtype_t in_dtype,
                                 ssm_dtype_t out_dtype, void* stream);
ssm_status_t ssd_mamba3_mimo_fwd_ckpt(const void* x, const float* dt, const float* lam,
                                      const float* A_head, const void* B, const void* C,
                                      int chunk, int rank, const float* initial_state,
                                      const void* prev_B, const void* prev_x, void* y,
                                      float* final_state, float* block_states, int batch,
                                      int seqlen, int nheads, int headdim, int dstate,
                                      int ngroups, ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                                      void* stream);

/*
 * Bytes of device workspace ssd_chunked_bwd needs (a pure function of its
 * arguments; 0 if they are invalid or unsupported).  About batch * nheads *
 * (ceil(seqlen / 128) + 1) * 32 KiB of block states plus 2 * nheads * batch *
 * seqlen * 512 bytes of per-head dB, dC partials.
 */
size_t ssd_chunked_bwd_workspace_bytes(int batch, int seqlen, int nheads, int headdim,
                                       int dstate, int ngroups);

/*
 * Gradient of the chunked SSD.
 *   The forward operation is ssd_chunked_fwd's ("Mamba-3 NKI Kernels for AWS
 *   Neuron", section "Kernel details": the Mamba-2 SSD structure, equal to the
 *   step recurrence S = exp(dt A_h) S + dt B x^T, y = C S).  The same page
 *   reports gradient parity through autograd (section "Correctness") but
 *   prints no backward formula; this is the exact reverse-mode derivative.
 *
 * For the loss sum(dy * y) + sum(dfinal_state * final_state), with y and
 * final_state what ssd_chunked_fwd returns for the same inputs, writes:
 *   dx              (batch, seqlen, nheads, headdim)  fp32
 *   ddt             (batch, seqlen, nheads)           fp32 (dt as given: no softplus)
 *   dA_head         (nheads,)                         fp32
 *   dB, dC          (batch, seqlen, ngroups, dstate)  fp32 (summed over the group's heads)
 *   dinitial_state  (batch, nheads, headdim, dstate)  fp32, may be NULL (not written)
 * Inputs as for ssd_chunked_fwd (x, B, C bf16; dt, A_head, initial_state fp32)
 * plus dy (batch, seqlen, nheads, headdim) in in_dtype, dfinal_state
 * (batch, nheads, headdim, dstate) fp32 or NULL (zero), and block_states: what
 * ssd_chunked_fwd_ckpt kept for the same inputs, or NULL (the call then runs the
 * forward once more to make them).
 * workspace: at least ssd_chunked_bwd_workspace_bytes(...) bytes, contents on
 * entry irrelevant; ssm_last_device_status reads it afterwards.  The call runs
 * the forward kernel once more to store the state entering every 128-step
 * block, then one CTA per (batch, head) walks the blocks in reverse; all on
 * `stream`.  Sums over heads and over the batch are added in a fixed order:
 * the same bits on every run.
 * Every output must be disjoint from every input, from the other outputs and
 * from the workspace (SSM_ERR_ALIAS).
 * Supported: chunk 64, headdim 64, dstate 128, bf16 in_dtype, seqlen % chunk
 * == 0, nheads % ngroups == 0.  With no step (seqlen == 0 or batch == 0)
 * dA_head is zeroed and dinitial_state = dfinal_state (or 0).
 */
ssm_status_t ssd_chunked_bwd(const void* x, const float* dt, const float* A_head, const void* B,
                             const void* C, int chunk, const float* initial_state, const void* dy,
                             const float* dfinal_state, const float* block_states, float* dx,
                             float* ddt, float* dA_head,
                             float* dB, float* dC, float* dinitial_state, int batch, int seqlen,
                             int nheads, int headdim, int dstate, int ngroups,
                             ssm_dtype_t in_dtype, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * Bytes of device workspace ssd_mamba3_bwd needs (a pure function of its
 * arguments; 0 if they are invalid or unsupported): ssd_chunked_bwd's, plus
 * per-step weights and dots and one state per (batch, head).
 */
size_t ssd_mamba3_bwd_workspace_bytes(int batch, int seqlen, int nheads, int headdim,
                                      int dstate, int ngroups);

/*
 * Gradient of the Mamba-3 SISO chunked prefill.
 *   The forward operation is ssd_mamba3_fwd's ("Mamba-3 NKI Kernels for AWS
 *   Neuron", section "How it works", Eq. 9: S = alpha_t S + beta_t u_{t-1} +
 *   gamma_t u_t with alpha = exp(dt A), gamma = lambda dt, beta = (dt - gamma)
 *   alpha; section "Kernel details": the single-SSD form with scale =
 *   gamma + dt_{t+1} (1 - lambda_{t+1}) and a diagonal correction).  The page
 *   reports the mixer's gradients through autograd (section "Correctness")
 *   and prints no backward formula; this is the exact reverse-mode derivative.
 *
 * For the loss sum(dy * y) + sum(dfinal_state * final_state), with y and
 * final_state what ssd_mamba3_fwd returns for the same inputs, writes:
 *   dx, ddt, dA_head, dB, dC, dinitial_state  as ssd_chunked_bwd
 *   dlam     (batch, seqlen, nheads)  fp32 (lambda as given: no sigmoid)
 *   dprev_B  (batch, ngroups, dstate) fp32 (summed over the group's heads) and
 *   dprev_x  (batch, nheads, headdim) fp32, required when prev_B / prev_x are
 *            given, not written otherwise.
 * Inputs as for ssd_mamba3_fwd (x, B, C, prev_B, prev_x bf16; dt, lam, A_head,
 * initial_state fp32), plus dy (batch, seqlen, nheads, headdim) bf16 and
 * dfinal_state (batch, nheads, headdim, dstate) fp32 or NULL (zero), and
 * block_states: what ssd_mamba3_fwd_ckpt kept for the same inputs, or NULL (the
 * call then runs the Mamba-3 forward once more to make them).
 * How: the three-term recurrence is the Mamba-2 SSD recurrence of S + c_t u_t
 * (c_t = dt_{t+1} (1 - lambda_{t+1})) with input weights `scale` and y less
 * c_t (C_t . B_t) x_t, so the call runs the Mamba-3 forward once more for the
 * states entering each 128-step block, the SSD gradient with those weights,
 * then small kernels that take the weights' and the correction's gradients
 * back to dt, lambda, x, B, C and the previous token.  All on `stream`.
 * workspace: at least ssd_mamba3_bwd_workspace_bytes(...) bytes, contents on
 * entry irrelevant; ssm_last_device_status reads it afterwards.  Sums over
 * heads and over the batch are added in a fixed order.
 * Every output must be disjoint from every input, from the other outputs and
 * from the workspace (SSM_ERR_ALIAS).  prev_B and prev_x must be both NULL or
 * both given (else SSM_ERR_NULL).
 * Supported: as ssd_chunked_bwd, with nheads <= 6144.  With no step (seqlen == 0
 * or batch == 0) dA_head is zeroed, dinitial_state = dfinal_state (or 0) and
 * dprev_B, dprev_x are zeroed.
 */
ssm_status_t ssd_mamba3_bwd(const void* x, const float* dt, const float* lam, const float* A_head,
                            const void* B, const void* C, int chunk, const float* initial_state,
                            const void* prev_B, const void* prev_x, const void* dy,
                            const float* dfinal_state, const float* block_states, float* dx,
                            float* ddt, float* dlam,
                            float* dA_head, float* dB, float* dC, float* dinitial_state,
                            float* dprev_B, float* dprev_x, int batch, int seqlen, int nheads,
                            int headdim, int dstate, int ngroups, ssm_dtype_t in_dtype,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace ssd_mamba3_mimo_bwd needs (a pure function of its
 * arguments; 0 if they are invalid or unsupported).
 */
size_t ssd_mamba3_mimo_bwd_workspace_bytes(int batch, int seqlen, int rank, int nheads,
                                           int headdim, int dstate, int ngroups);

/*
 * Gradient of the Mamba-3 MIMO chunked prefill.
 *   The forward operation is ssd_mamba3_mimo_fwd's ("Mamba-3 NKI Kernels for
 *   AWS Neuron", section "Kernel details", mamba3_mimo_ssd_kernel: rank R with
 *   BX_t = sum_r B_{t,r} (x) x_{t,r} in Eq. 9 and y_{t,r} = C_{t,r} . S).  The
 *   page reports the MIMO mixer's gradients through autograd (section
 *   "Correctness"); this is the exact reverse-mode derivative.
 *
 * For the loss sum(dy * y) + sum(dfinal_state * final_state) writes:
 *   dx       (batch, seqlen, rank, nheads, headdim)  fp32
 *   ddt, dlam (batch, seqlen, nheads)                fp32
 *   dA_head  (nheads,)                               fp32
 *   dB, dC   (batch, seqlen, rank, ngroups, dstate)  fp32 (summed over the group's heads)
 *   dinitial_state (batch, nheads, headdim, dstate)  fp32, may be NULL
 *   dprev_B  (batch, rank, ngroups, dstate), dprev_x (batch, rank, nheads, headdim)
 *            fp32, required when prev_B / prev_x are given.
 * Inputs as for ssd_mamba3_mimo_fwd (bf16 x, B, C, prev_B, prev_x), plus dy
 * like x (bf16), dfinal_state fp32 or NULL, and block_states: what
 * ssd_mamba3_mimo_fwd_ckpt kept for the same inputs, or NULL.  The call runs the
 * MIMO forward once more (unless given block_states) for the states entering
 * each 128-row block of sub-tokens, the SSD
 * gradient over the sub-tokens (block-lower-triangular mask, the step's decay
 * on its first sub-token, its scale weight on every one), then elementwise
 * kernels for lambda, the block-diagonal correction and the previous token.
 * workspace, aliasing, determinism and the no-step case as ssd_mamba3_bwd.
 * Supported: rank 1, 2 or 4 with chunk * rank == 64; headdim 64, dstate 128,
 * bf16 in_dtype, seqlen % chunk == 0, nheads % ngroups == 0, and
 * (2 nheads + ngroups) rank^2 <= 12288.
 */
ssm_status_t ssd_mamba3_mimo_bwd(const void* x, const float* dt, const float* lam,
                                 const float* A_head, const void* B, const void* C, int chunk,
                                 int rank, const float* initial_state, const void* prev_B,
                                 const void* prev_x, const void* dy, const float* dfinal_state,
                                 const float* block_states, float* dx, float* ddt, float* dlam,
                                 float* dA_head, float* dB,
                                 float* dC, float* dinitial_state, float* dprev_B,
                                 float* dprev_x, int batch, int seqlen, int nheads, int headdim,
                                 int dstate, int ngroups, ssm_dtype_t in_dtype, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace ssm_scan_fwd_host needs (a pure function of its
 * arguments; 0 if they are invalid).  Four slots, each the largest segment's u,
 * delta, z, B, C, y and states (a segment is at most about 1/8 of the (batch,
 * channel) rows, and at most 3072 rows on long sequences, all steps), plus the
 * largest segment's ssm_scan_workspace_bytes.
 */
size_t ssm_scan_fwd_host_workspace_bytes(int batch, int dim, int seqlen, int dstate, int ngroups,
                                         ssm_dtype_t in_dtype, ssm_dtype_t out_dtype);

/*
 * Selective scan with the activations and results in HOST memory.
 *   Computes exactly what ssm_scan_fwd computes, same arguments and layouts,
 *   but u, delta, z, B, C, initial_state, y and final_state are HOST pointers to
 *   page-locked memory (cudaHostAlloc / cudaMallocHost / cudaHostRegister;
 *   anything else returns SSM_ERR_UNSUPPORTED, except arrays of zero bytes,
 *   which are never touched); A, D, delta_bias and the
 *   workspace are DEVICE pointers.  Every channel's recurrence is independent
 *   of the others, so the (batch, channel) rows are cut into about eight
 *   segments -- whole batches, whole B/C groups of one batch, or part of one
 *   group -- each of whose arrays is one contiguous block of host memory.  A
 *   segment's u, delta, z, its groups' B and C and its initial state are
 *   copied in with one 1-D copy each, scanned on `stream`, and its y and final
 *   state copied back, with the copies of neighbouring segments in flight
 *   during the scan.
 *  - Kernel per segment: where every segment fits the sequence-parallel scan
 *    (at most 3072 channels; on long sequences segments are capped to fit)
 *    while the whole problem does not, every segment takes that scan with one
 *    segments-per-chunk count, so a segment's scan time shrinks with its size
 *    (the chained scan's CTAs each walk the whole sequence).  Each channel's
 *    result is then bit-equal to ssm_scan_fwd run on any channel subset the
 *    sequence-parallel scan takes with the same count, and within the stated
 *    tolerance of the oracle, like either kernel.  Otherwise every segment is
 *    scanned with the kernel and plan ssm_scan_fwd would use for the whole
 *    problem, and the result is bit-equal to ssm_scan_fwd on device copies.
 *
 *  - Asynchronous like every entry point: work is enqueued on `stream` and on
 *    two copy streams of the library's own (created on the first call on a
 *    device and kept until the process exits); `stream` completes only after
 *    every copy of the call.  The host buffers must not be modified (inputs) or
 *    read (outputs) until then.
 *  - workspace: at least ssm_scan_fwd_host_workspace_bytes(...) bytes, not
 *    shared with a concurrent call; ssm_last_device_status reports the first
 *    device-side timeout of any segment (SSM_OK if none).
 *  - Calls on one device are enqueued one at a time (an internal lock).
 */
ssm_status_t ssm_scan_fwd_host(const void* u, const void* delta, const float* A, const void* B,
                               const void* C, const float* D, const void* z,
                               const float* delta_bias, int delta_softplus,
                               const float* initial_state, void* y, float* final_state,
                               int batch, int dim, int seqlen, int dstate, int ngroups,
                               ssm_dtype_t in_dtype, ssm_dtype_t out_dtype, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * Waits for `stream` to drain, then returns the device-side status the last
 * ssm_scan_fwd that used `workspace` recorded (SSM_OK or SSM_ERR_TIMEOUT),
 * or SSM_ERR_CUDA if the stream itself reports an error.
 */
ssm_status_t ssm_last_device_status(const void* workspace, void* stream);

/*
 * Test hook for the scan's bounded look-back waits (every entry point that
 * runs a scan kernel: ssm_scan_fwd, _ckpt, _noalloc, _host and the forward
 * inside ssm_scan_bwd).  The chained scan cuts the sequence into chunks when
 * the channel blocks outnumber the resident CTA slots, and chunk c of a block
 * polls the flag chunk c-1 publishes with its final state.  The
 * sequence-parallel scan always cuts it into 128-step chunks, and chunk c
 * polls the flags of chunks c-1, c-2, ... (aggregate or inclusive state: the
 * decoupled look-back of Merrill and Garland's single-pass prefix scan).  A
 * poll loop that runs out records SSM_ERR_TIMEOUT in the workspace and goes
 * on.
 *  - spin_limit: polls before that happens (0 restores the default, about a
 *    second).
 *  - drop_first_publish: nonzero makes chunk 0 of every block skip its
 *    publish of its final (inclusive) state, so chunk 1 waits until its
 *    limit: a wait on a flag that nothing sets, with no fault.  The scan's
 *    outputs are then undefined.
 *  - Process-wide setting, read when each scan is enqueued; not for use while
 *    other threads enqueue scans.  Always returns SSM_OK.
 */
ssm_status_t ssm_debug_set_lookback(int drop_first_publish, unsigned int spin_limit);

/*
 * Test hook choosing the forward scan's kernel, so that tests can run both on
 * the same problem.  path: 0 as planned (see ssm_scan_fwd), 1 always the
 * chained scan, 2 the sequence-parallel scan wherever batch * dim <= 3072
 * (larger problems keep the chained scan: the workspace size does not cover
 * the other).  segments: the sequence-parallel scan's segments per 128-step
 * chunk, 8, 16 or 32 (0 = planned).  Process-wide, read when each scan is
 * enqueued.  Returns SSM_ERR_SHAPE for other values, else SSM_OK.
 */
ssm_status_t ssm_debug_set_scan_path(int path, int segments);

#ifdef __cplusplus
}
#endif

#endif /* SSM_GB300_H */
