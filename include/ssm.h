/*
 * ssm.h -- C ABI of libssm: the selective state-space (S6) scan on one B300 GPU.
 *
 * What the entry points compute (per batch index b and channel d, time t, state n):
 *
 *   Δ_t  = softplus(delta[b,d,t] + delta_bias[d])   (or without softplus)
 *          -- selection: Δ is a function of the input; "Mamba: Linear-Time
 *             Sequence Modeling" summary page, section 4b, Algorithm 2 and the
 *             parameterisation under it (τ_Δ = softplus of a parameter plus a
 *             projection); SSM/Mamba chapter, section 4.1.
 *   Ā    = exp(Δ_t A[d,n]),  B̄ = (exp(Δ_t A[d,n]) - 1) / A[d,n] * B[b,n,t]
 *          -- zero-order hold for a diagonal A, summary page equation (4);
 *             chapter section 3.2.  A[d,n] = 0 takes the limit B̄ = Δ_t B.
 *   h_t  = Ā h_{t-1} + B̄ u[b,d,t]
 *   y_t  = C[b,:,t] · h_t + D[d] u[b,d,t]
 *          -- recurrence and readout, summary page equations (2a), (2b); the
 *             direct term D from the chapter's section 3.1.
 *   y_t *= z[b,d,t] * sigmoid(z[b,d,t])
 *          -- "SSM output × SiLU(gate)", summary page section 4a shape table.
 *
 * The expanded (batch, d_inner, L, N) state is never written to memory; only
 * y and the final state are.
 *
 * Memory: every pointer is a DEVICE pointer on the current CUDA device (the
 * one exception: ssm_scan_fwd_host takes host buffers and a device
 * workspace), owned by the caller; the library allocates no memory and keeps
 * no pointer after a call returns.  Layouts are dense and row-major (last index fastest):
 *   u, delta, z, y      (batch, dim, seqlen)  in io_dtype (float32 or bfloat16)
 *   B, C                (batch, dstate, seqlen) float32
 *   A                   (dim, dstate) float32
 *   D, delta_bias       (dim) float32
 *   states              (batch, dim, dstate) float32
 * All pointers must be 16-byte aligned (SSM_ERR_ALIGN otherwise).  Any seqlen
 * >= 0 is accepted; rows whose length is not a multiple of 16 bytes take a
 * slower element-wise load path.  Outputs must not overlap inputs.
 *
 * Execution: work is enqueued on the given stream (NULL = the legacy default
 * stream) and the call returns without synchronising.  Argument errors are
 * returned synchronously before anything is enqueued; a failed launch returns
 * SSM_ERR_CUDA (details from cudaGetLastError()).
 */
#ifndef SSM_H
#define SSM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* I/O element types of u, delta, z and y. */
#define SSM_F32 0
#define SSM_BF16 1

/* Bits of the delta_softplus flag word. */
#define SSM_SOFTPLUS 1 /* Δ = softplus(delta + delta_bias) */
#define SSM_EULER_B 2  /* B̄ = Δ B instead of the zero-order hold (A̅ stays exp(Δ A)) */
#define SSM_SAVED_STATES 4 /* ssm_scan_bwd only: its workspace holds the states that
                              ssm_scan_fwd_train saved for these inputs */
#define SSM_LAYOUT_BLD 8   /* scan, training forward, backward and conv1d: the
                              (batch, dim, seqlen) tensors are (batch, seqlen, dim)
                              instead (channels innermost; Algorithm 2's (B, L, D)) */
#define SSM_TEST_STALL 16  /* ssm_scan_fwd_ex only, and only while ssm_set_test_mode is
                              on (SSM_ERR_ARG otherwise): the failure-path test; one
                              block of the call gives up waiting (see ssm_set_test_mode) */

/* Status codes. */
#define SSM_OK 0
#define SSM_ERR_ARG (-1)         /* null required pointer, bad size, bad dtype, overlap */
#define SSM_ERR_ALIGN (-2)       /* a pointer is not 16-byte aligned */
#define SSM_ERR_UNSUPPORTED (-3) /* dstate not in {1, 2, 4, 8, 16, 32, 64, 128} */
#define SSM_ERR_CUDA (-4)        /* a CUDA call or kernel launch failed */
#define SSM_ERR_WORKSPACE (-5)   /* workspace given but too small */
#define SSM_ERR_TIMEOUT (-6)     /* a kernel gave up waiting for its own data (see ssm_status) */

/* Human-readable name of a status code (static string). */
const char* ssm_strerror(int status);

/* Library version, e.g. "0.1.0". */
const char* ssm_version(void);

/*
 * Full-sequence scan (the summary page's Algorithm 2 with the recurrence of
 * equation (2) evaluated as a chunked scan), on the legacy default stream,
 * starting from a zero state.
 *
 *   u, delta      required, (batch, dim, seqlen) io_dtype
 *   delta_bias    optional (NULL = 0), (dim)
 *   A             required, (dim, dstate)
 *   B, C          required, (batch, dstate, seqlen)
 *   D             optional (NULL = 0), (dim)
 *   z             optional (NULL = no gate), (batch, dim, seqlen) io_dtype
 *   delta_softplus  flag word: SSM_SOFTPLUS set: Δ = softplus(delta + bias), else
 *                   Δ = delta + bias; SSM_EULER_B set: B̄ = Δ B (the first-order
 *                   form the summary page gives beside equation (4)) instead of
 *                   the exact zero-order hold; SSM_LAYOUT_BLD set: u, delta,
 *                   z and y are (batch, seqlen, dim); any other bit: SSM_ERR_ARG
 *   y             required output, (batch, dim, seqlen) io_dtype
 *   final_state   optional output (NULL = not written), (batch, dim, dstate) float32
 *
 * batch, dim >= 0 (either 0 is a no-op); seqlen >= 0 (0 writes final_state
 * only); dstate in {1, 2, 4, 8, 16, 32, 64, 128}.
 */
int ssm_scan_fwd(const void* u, const void* delta, const float* delta_bias, const float* A,
                 const float* B, const float* C, const float* D, const void* z,
                 int delta_softplus, void* y, float* final_state,
                 int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype);

/*
 * Bytes of workspace that ssm_scan_fwd_ex may use for these sizes on the
 * current device: a 256-byte header holding the call's device status word
 * (read by ssm_status), then the carry records of a plan that splits the
 * sequence across thread blocks (two passes with a carried float32 state).
 * 256 means the plan does not split; 0 means the sizes are not supported.
 * With no workspace the scan runs one pass per channel and reports its status
 * to the library-wide word.
 */
size_t ssm_scan_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                int io_dtype);

/*
 * Extended scan: as ssm_scan_fwd, plus
 *   init_state      optional (NULL = zeros), (batch, dim, dstate) float32: h_{-1}.
 *                   Passing the final_state of a call over u[..., :L1] as the
 *                   init_state of a call over u[..., L1:] gives the same result
 *                   as one call over the whole sequence (chunk-carried state).
 *                   May equal final_state (read before it is written).
 *   workspace       optional device scratch (NULL = none) of workspace_bytes
 *                   bytes, 16-byte aligned; contents need not be initialised.
 *                   The call zeroes its status word (the first 4 bytes) on
 *                   the stream and a block that gives up waiting sets it, so
 *                   ssm_status(workspace, stream) reports this call until the
 *                   next call on the same workspace.  SSM_ERR_WORKSPACE when
 *                   non-NULL and smaller than ssm_scan_workspace_bytes() (or
 *                   than 256 bytes).  NULL: no split, and the status goes to
 *                   the library-wide word.
 *   stream          cudaStream_t to enqueue on (NULL = legacy default stream).
 * Concurrent calls must not share a workspace.
 */
int ssm_scan_fwd_ex(const void* u, const void* delta, const float* delta_bias, const float* A,
                    const float* B, const float* C, const float* D, const void* z,
                    int delta_softplus, void* y, float* final_state,
                    int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype,
                    const float* init_state, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Scan on strided views: as ssm_scan_fwd_ex, with u, delta, z and y given as
 * views with arbitrary element strides, so that, for instance, u and z can be
 * the two halves of one input projection's output without a copy (the summary
 * page's section 4a shape table splits Linear(2ED) into the SSM input and the
 * gate; Algorithm 2's (B, L, D) with a row stride of 2ED).
 *
 *   strides   12 int64 element strides, (batch, channel, time) for u, delta, z
 *             and y in that order (z's are ignored when z is NULL).  NULL: dense
 *             (batch, dim, seqlen).  Element (b, d, t) of u is
 *             u[b * strides[0] + d * strides[1] + t * strides[2]], and so on.
 *
 * u, delta and z must share one orientation: unit time stride (time-major rows)
 * or unit channel stride (channel-major rows; SSM_ERR_UNSUPPORTED otherwise).
 * Strides are >= 0 and non-zero over extents above one; y's must not map two
 * elements to one place (SSM_ERR_ARG).  Views whose other strides are multiples
 * of 16 bytes are staged by TMA; others take the element-wise path.  y may be
 * any non-overlapping view; with unit time stride and 16-byte aligned rows it is
 * stored in 16-byte vectors.  SSM_LAYOUT_BLD is refused (the strides say the
 * layout); other flags, the workspace and the status word as ssm_scan_fwd_ex.
 * Results equal ssm_scan_fwd_ex's on contiguous copies of the views, bit for
 * bit.  Overlap checks use each view's span (first to last element).
 */
int ssm_scan_fwd_strided(const void* u, const void* delta, const float* delta_bias,
                         const float* A, const float* B, const float* C, const float* D,
                         const void* z, int delta_softplus, void* y, float* final_state,
                         int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                         int io_dtype, const int64_t* strides, const float* init_state,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * The scan on HOST buffers (selective-scan summary page, section 4b equations
 * (2), (4) and Algorithm 2, as ssm_scan_fwd_ex): the copies to and from the
 * device are part of the call.  u, delta, z, y, B, C, A, D, delta_bias,
 * init_state and final_state are host pointers (page-locked memory lets the
 * copies run asynchronously and overlap; pageable memory works but the
 * copies then synchronise), with the layouts, dtypes, flags and nullability
 * of ssm_scan_fwd_ex (SSM_SOFTPLUS, SSM_EULER_B, SSM_LAYOUT_BLD).  workspace is
 * DEVICE memory of at least ssm_scan_fwd_host_workspace_bytes() bytes (the
 * call's status word in its first 256 bytes, read by ssm_status(workspace,
 * stream); the parameters, the unit scans' scratch and three staging slots),
 * 16-byte aligned.
 *
 * The work is cut into units that are contiguous in host memory (a batch row,
 * or a block of a row's channels when batch < 8; a whole row with
 * SSM_LAYOUT_BLD); the copy-in of a unit, the scan of the previous one and
 * the copy-out of the one before run at the same time on two internal copy
 * streams and `stream`.  Results equal ssm_scan_fwd_ex's on the same inputs up
 * to the scan's own plan for the smaller unit (a long unit with few channels
 * may be split along L).  Asynchronous on `stream`: y and final_state are in
 * host memory once `stream` has reached the call's end; work queued earlier
 * on `stream` happens before the first copy.  Errors: as ssm_scan_fwd_ex;
 * SSM_ERR_WORKSPACE when workspace is NULL or too small; outputs may not
 * overlap inputs (final_state may equal init_state exactly).
 */
size_t ssm_scan_fwd_host_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen,
                                         int64_t dstate, int io_dtype, int flags);
int ssm_scan_fwd_host(const void* u, const void* delta, const float* delta_bias, const float* A,
                      const float* B, const float* C, const float* D, const void* z, int flags,
                      void* y, float* final_state, const float* init_state, int64_t batch,
                      int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * Device-side status of scan calls.  The pages have no counterpart: this is the
 * library's failure report.  The scan kernels' only waits are on their own
 * copies into shared memory; a wait that has not completed after 2 s gives up,
 * the block sets the status word, lets its copies in flight land and leaves its
 * outputs unwritten.  The CUDA context stays usable.
 *
 *   workspace  the workspace of a ssm_scan_fwd_ex / ssm_scan_fwd_train /
 *              ssm_scan_fwd_host call: its status word, which the call zeroed,
 *              so the result is that call's (the last call on this workspace;
 *              `stream` must be the stream the call was issued on, or ordered
 *              after it).  NULL: the library-wide word of the calls made without
 *              a workspace (ssm_scan_fwd, ssm_scan_fwd_ex with NULL,
 *              ssm_scan_fwd_noalloc) on the current device since the last
 *              ssm_status(NULL, ·): read and cleared in one atomic step in stream
 *              order, so an error set meanwhile by a kernel on another stream is
 *              kept for the next read.  ssm_status(NULL, ·) calls must not
 *              overlap one another.
 *
 * Synchronises `stream` (NULL = legacy default stream).  Returns SSM_OK,
 * SSM_ERR_TIMEOUT (a block gave up waiting), SSM_ERR_ALIGN (workspace not
 * 16-byte aligned) or SSM_ERR_CUDA (the copy or synchronisation failed).
 */
int ssm_status(const void* workspace, void* stream);

/*
 * Test mode (the pages have no counterpart).  enable = 1 turns it on:
 *   - ssm_scan_fwd_ex accepts SSM_TEST_STALL, which makes the first block (or
 *     warp) of the call's output pass arm the barrier of its second chunk's
 *     copy without issuing the copy, so its waits give up after wait_limit_ns
 *     (1e3 .. 2e9) instead of 2 s; the call's status word then reads
 *     SSM_ERR_TIMEOUT.  It needs a sequence of at least two 16-step chunks with
 *     16-byte rows (the copy path the wait belongs to);
 *   - noalloc_limit_bytes > 0 lowers the scratch limit of ssm_scan_fwd_noalloc
 *     to that many bytes, so that its refusal can be tested;
 *   - scan_kernel picks the forward scan's kernel: 0 = by size (the default),
 *     1 = the block kernel, 2 = the two-warp-block kernel wherever it applies (N = 16,
 *     bf16, zero-order hold, views TMA can stage), so that both can be tested
 *     on small sizes.
 * enable = 0 restores the defaults.  Process-wide; for tests and tuning only.
 * Returns SSM_OK, or SSM_ERR_ARG for an argument out of range.
 */
int ssm_set_test_mode(int enable, int64_t wait_limit_ns, int64_t noalloc_limit_bytes,
                      int scan_kernel);

/*
 * One-token decode: the recurrent mode of the summary page's equation (2)
 * ("O(N) state update per token", section 4b; the efficiency table of 4c),
 * applied in place to a stored state, on the legacy default stream.
 *
 *   state    required in/out, (batch, dim, dstate) float32: h_{t-1} -> h_t
 *   u, delta required, (batch, dim) io_dtype; Δ = delta as given (no bias,
 *            no softplus: the caller passes the step size itself)
 *   A        required, (dim, dstate);  B, C required, (batch, dstate)
 *   D        optional (NULL = 0), (dim);  z optional (NULL = no gate), (batch, dim)
 *   y        required output, (batch, dim) io_dtype
 */
int ssm_state_update(float* state, const void* u, const void* delta, const float* A,
                     const float* B, const float* C, const float* D, const void* z, void* y,
                     int64_t batch, int64_t dim, int64_t dstate, int io_dtype);

/*
 * Extended decode step: as ssm_state_update, plus delta_bias (optional, (dim))
 * and the delta_softplus flag word (as for ssm_scan_fwd: SSM_SOFTPLUS,
 * SSM_EULER_B), on `stream`.
 */
int ssm_state_update_ex(float* state, const void* u, const void* delta, const float* delta_bias,
                        int delta_softplus, const float* A, const float* B, const float* C,
                        const float* D, const void* z, void* y,
                        int64_t batch, int64_t dim, int64_t dstate, int io_dtype, void* stream);

/*
 * Scan without any device allocation by the caller or the library.
 *
 * The paper has no counterpart; this is a deployment aid.  Some callers
 * cannot call cudaMalloc where they run the scan (a process whose device
 * memory is all owned by its own pool, a plug-in host that forbids
 * allocation after start-up, a real-time loop that must not block on the
 * allocator), so they cannot provide the workspace that ssm_scan_fwd_ex uses
 * to split long sequences across blocks.  This entry point takes that
 * scratch from a fixed array of SSM_STATIC_SCRATCH_BYTES compiled into the
 * library; every GPU that loads the library holds the array until the
 * process exits.  The caller still passes all inputs and outputs.
 *
 * Arguments, layouts and results are those of ssm_scan_fwd_ex (no workspace
 * arguments).  Returns SSM_ERR_WORKSPACE when the plan's carry records for
 * these sizes need more than SSM_STATIC_SCRATCH_BYTES (ssm_scan_workspace_bytes()
 * minus its 256-byte header tells in advance); SSM_ERR_ARG when `stream`
 * belongs to another device than the current one (the array used is the
 * current device's: every call needs the stream's device current); other
 * argument errors as ssm_scan_fwd_ex.  Its device status goes to the
 * library-wide word (ssm_status(NULL, stream)).
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress, with the device current) and caches it; make
 * that first call before any stream capture.  A device reset
 * (cudaDeviceReset) while the library is loaded is not supported: the cached
 * address would be stale.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * All calls on a device share the one array, which keeps whatever the last
 * call left in it (every carry record a call reads is written earlier by the
 * same call, so nothing needs clearing).  Calls that can overlap on the GPU
 * (different streams without an ordering between them) race on the array:
 * order them, e.g. on one stream.
 */
#define SSM_STATIC_SCRATCH_BYTES (2u << 20) /* 2 MiB */

int ssm_scan_fwd_noalloc(const void* u, const void* delta, const float* delta_bias,
                         const float* A, const float* B, const float* C, const float* D,
                         const void* z, int delta_softplus, void* y, float* final_state,
                         int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                         int io_dtype, const float* init_state, void* stream);

/*
 * Backward pass (training).  The summary page ("Mamba: Linear-Time Sequence
 * Modeling", section 4c, hardware-aware algorithm) trains the layer with the
 * states recomputed in the backward pass rather than stored; this entry point
 * does that.  It returns the derivatives of
 *
 *     Loss = Σ_{b,d,t} y[b,d,t] dy[b,d,t] + Σ_{b,d,n} final_state[b,d,n] d_final_state[b,d,n]
 *
 * with respect to every input of ssm_scan_fwd_ex, for the same inputs (u,
 * delta, delta_bias, A, B, C, D, z, delta_softplus, init_state as in the
 * forward call; y and final_state need not be kept: the pass recomputes them).
 * The chain rule of equations (2) and (4) with the selection of Algorithm 2
 * (see the kernel source for the formulas).
 *
 * Inputs (device, caller-owned; layouts as above):
 *   dy             (batch, dim, seqlen) io_dtype   dLoss/dy, required
 *   d_final_state  (batch, dim, dstate) float32    nullable (= 0)
 * Outputs (device, caller-owned, written in full, never accumulated into):
 *   du, ddelta     (batch, dim, seqlen) io_dtype   required; ddelta is dLoss/d(delta),
 *                                                  the raw input before bias/softplus
 *   dz             (batch, dim, seqlen) io_dtype   required when z is given; must be
 *                                                  NULL when z is NULL
 *   dA             (dim, dstate) float32           required (summed over the batch)
 *   dB, dC         (batch, dstate, seqlen) float32 required (summed over the channels)
 *   dD, d_delta_bias (dim) float32                 nullable (not written); with D or
 *                                                  delta_bias NULL they hold the
 *                                                  derivative at D = 0 / bias = 0
 *   d_init_state   (batch, dim, dstate) float32    nullable; dLoss/d(init_state)
 *                                                  (init_state NULL = zeros)
 * Workspace: ssm_scan_bwd_workspace_bytes() bytes of device memory (16-byte
 * aligned), required whenever batch, dim and seqlen are all non-zero; it
 * holds the chunk-start states of the recomputation and per-block partial
 * sums, nothing that outlives the call.  Its size depends on the plan for the
 * current device: when the (channel block, batch row) blocks fill less than
 * half a wave of the GPU, the sequence is split into segments run in parallel
 * (the workspace then also holds the segments' forward and adjoint carries and
 * per-segment sums), so size it on the device that runs the call.
 *
 * Precision: fp32 arithmetic; bf16 outputs are rounded to nearest even.  The
 * channel sums (dB, dC), batch sums (dA, dD, d_delta_bias) and segment sums
 * are added in a fixed order, so results are the same from run to run.
 * Errors: as ssm_scan_fwd_ex; outputs may not overlap inputs or each other.
 * A split plan's forward-carry pass stages through TMA with bounded waits; a
 * wait that runs out sets the library-wide status word (ssm_status with a null
 * workspace returns SSM_ERR_TIMEOUT), as for the scans without a workspace.
 * Execution: asynchronous on `stream` (two kernels: the pass and the
 * fixed-order sums; four with a split plan: the forward carries and the
 * adjoint carries first; memsets and a copy instead when a size is zero).
 */
size_t ssm_scan_bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate);

int ssm_scan_bwd(const void* u, const void* delta, const float* delta_bias, const float* A,
                 const float* B, const float* C, const float* D, const void* z,
                 int delta_softplus, const float* init_state, const void* dy,
                 const float* d_final_state, void* du, void* ddelta, float* dA, float* dB,
                 float* dC, float* dD, void* dz, float* d_delta_bias, float* d_init_state,
                 int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Front end of the scan: causal depthwise conv1d followed by SiLU.  The
 * summary page's shape table (section 4a) puts "Conv1d -> SiLU" on the
 * (B, L, ED) path right before the SSM (its output is the scan's u); the
 * configuration page ("2. Mamba 상세") gives the kernel width d_conv = 4.
 * Per channel d with width K = `width` (1..4):
 *
 *     out[b,d,t] = silu(bias[d] + Σ_{k<K} weight[d,k] · x[b,d,t-(K-1)+k])
 *
 * (or the bare sum when bit 1 of `silu` is clear; `silu` may also carry
 * SSM_LAYOUT_BLD: x and out are then (batch, seqlen, dim); the states keep
 * their (batch, dim, width-1) layout).  x[t < 0] comes from conv_state_in, the
 * K-1 inputs before the sequence (NULL = zeros); conv_state_out (nullable)
 * receives the last K-1 inputs of (conv_state_in, x), so a sequence split
 * over calls gives the same outputs as one call.  conv_state_out may be
 * conv_state_in itself (updated in place); no other overlap is allowed.
 *
 * Layouts: x, out (batch, dim, seqlen) io_dtype; weight (dim, width) float32;
 * bias (dim) float32, nullable; conv states (batch, dim, width-1) io_dtype.
 * Arithmetic in fp32; bf16 outputs rounded to nearest even.  Errors as the
 * scan (SSM_ERR_UNSUPPORTED for width outside 1..4).  Asynchronous on stream.
 */
int ssm_conv1d_fwd(const void* x, const float* weight, const float* bias,
                   const void* conv_state_in, int silu, void* out, void* conv_state_out,
                   int64_t batch, int64_t dim, int64_t seqlen, int64_t width, int io_dtype,
                   void* stream);

/*
 * Backward of ssm_conv1d_fwd (the front end of the summary page's section 4a
 * shape table): for a cotangent dout of `out`, with p_t the pre-activation and
 * g_t = dout_t · silu'(p_t), silu'(p) = σ(p)(1 + p(1 - σ(p))) (g = dout when
 * bit 1 of `silu` is clear),
 *
 *     dx[b,d,s]           = Σ_k weight[d,k] g[b,d,s+(K-1)-k]   (s inside the sequence)
 *     d_conv_state_in     = the same sum at the K-1 positions before it
 *     dweight[d,k]        = Σ_{b,t} g[b,d,t] x[b,d,t-(K-1)+k]
 *     dbias[d]            = Σ_{b,t} g[b,d,t]
 *
 * x, conv_state_in, weight, bias, silu (with SSM_LAYOUT_BLD), sizes and
 * layouts as ssm_conv1d_fwd; dout and dx like x (io_dtype); dweight (dim,
 * width) float32, required; dbias (dim) float32 and d_conv_state_in (batch,
 * dim, width-1) float32, nullable.  The sums over the batch and the steps are
 * added in a fixed order (one block per channel), so results repeat bit for
 * bit.  Outputs may not overlap inputs or each other.  Errors as
 * ssm_conv1d_fwd.  Asynchronous on `stream` (one kernel; memsets when a size
 * is zero).
 */
int ssm_conv1d_bwd(const void* x, const float* weight, const float* bias,
                   const void* conv_state_in, int silu, const void* dout, void* dx,
                   float* dweight, float* dbias, float* d_conv_state_in, int64_t batch,
                   int64_t dim, int64_t seqlen, int64_t width, int io_dtype, void* stream);

/*
 * One token of the front end on a rolling state (decode): for every (b, d),
 * window = (conv_state[b,d,0..K-2], x[b,d]); out[b,d] = silu(bias[d] +
 * Σ_k weight[d,k] window[k]); conv_state[b,d] <- window[1..K-1] (in place).
 * x, out (batch, dim) io_dtype; conv_state (batch, dim, width-1) io_dtype
 * (required when width > 1).  Errors and execution as ssm_conv1d_fwd.
 */
int ssm_conv1d_update(void* conv_state, const void* x, const float* weight, const float* bias,
                      int silu, void* out, int64_t batch, int64_t dim, int64_t width,
                      int io_dtype, void* stream);

/*
 * Training forward: ssm_scan_fwd_ex (same arguments, same results) that also
 * saves, in the backward pass's workspace `bwd_workspace` (at least
 * ssm_scan_bwd_workspace_bytes() bytes, 16-byte aligned), the state at the
 * start of every chunk of the sequence.  A following ssm_scan_bwd on the same
 * inputs, with that workspace and SSM_SAVED_STATES in its flag word, then
 * skips its own forward sweep.  Saving applies to dstate <= 16 (the backward's
 * chunk equals the forward's there); for larger dstate nothing is saved and
 * the backward recomputes whatever its flags say.  The workspace must not be
 * used for anything else between the two calls.
 */
int ssm_scan_fwd_train(const void* u, const void* delta, const float* delta_bias, const float* A,
                       const float* B, const float* C, const float* D, const void* z,
                       int delta_softplus, void* y, float* final_state, int64_t batch,
                       int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype,
                       const float* init_state, void* workspace, size_t workspace_bytes,
                       void* bwd_workspace, size_t bwd_workspace_bytes, void* stream);

/*
 * Mamba-2's scalar-A SSM (SSD), chunked.  The chapter page ("14.1 SSM(State
 * Space Models)과 Mamba 아키텍처의 부상", §5.1-5.2) restricts A to a scalar per
 * step times the identity, which makes the SSM the masked product
 * Y = (L ∘ C Bᵀ) X, and computes it chunk by chunk: the quadratic form inside
 * each chunk of 64 steps on the tensor cores, states passed between chunks.
 * Per batch b, head h (P = headdim channels sharing the step; group
 * g = h / (nheads / ngroups)), channel p, state n:
 *
 *   Δ_t   = softplus(dt[b,t,h] + dt_bias[h])   (SSM_SOFTPLUS in flags; else dt + bias)
 *   h_t   = exp(Δ_t A[h]) h_{t-1} + β_t x[b,t,h,p] B[b,t,g,n]
 *           β_t = (exp(Δ_t A[h]) - 1) / A[h]  (zero-order hold), or Δ_t (SSM_EULER_B)
 *   y     = Σ_n C[b,t,g,n] h_t + D[h] x, then · silu(z) when z is given
 *
 * Layouts (dense, row-major): x, z, y (batch, seqlen, nheads, headdim) bf16;
 * dt (batch, seqlen, nheads) bf16; B, C (batch, seqlen, ngroups, dstate) bf16;
 * A, D, dt_bias (nheads) fp32; init_state, final_state (batch, nheads,
 * headdim, dstate) fp32 (nullable).  Supported: headdim 64, dstate 64 or 128,
 * nheads a multiple of ngroups (SSM_ERR_UNSUPPORTED otherwise).  Workspace:
 * ssm_ssd_workspace_bytes() bytes (the states entering each chunk, the
 * chunks' step terms, each chunk's C Bᵀ per group), required when batch,
 * seqlen and nheads are non-zero; the query returns 0 for an unsupported shape.
 * Products in bf16 with fp32 accumulation; the running state is kept in fp32
 * and enters the chunk outputs as bf16.  Errors as the other entry points;
 * asynchronous on `stream` (four kernels).
 */
size_t ssm_ssd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                               int64_t ngroups, int64_t dstate);

int ssm_ssd_fwd(const void* x, const void* dt, const float* dt_bias, const float* A,
                const void* B, const void* C, const float* D, const void* z, int flags, void* y,
                float* final_state, const float* init_state, int64_t batch, int64_t seqlen,
                int64_t nheads, int64_t headdim, int64_t ngroups, int64_t dstate,
                void* workspace, size_t workspace_bytes, void* stream);

/*
 * The selective scan with a complex diagonal A.  The summary page ("Mamba:
 * Linear-Time Sequence Modeling") names a complex S4 only as an ablation row
 * (§5.4) and defines no complex form; this computes the plainest reading of its
 * equations (2) and (4) over complex numbers, per (batch, channel):
 *   Δ_t = softplus(delta_t + bias) (or delta_t + bias), Ā = exp(Δ A_n),
 *   B̄ = (Ā - 1)/A_n (A_n = 0, or the SSM_EULER_B flag: Δ),
 *   h_t = Ā h_{t-1} + B̄ B_{n,t} u_t,  y_t = Re(Σ_n C_{n,t} h_t[n]) + D u_t,
 * then y · silu(z) when z is given.  The real part is taken once: a caller who
 * keeps one state of each conjugate pair doubles C.
 *
 * Layouts: u, delta, z, y (batch, dim, seqlen) in io_dtype; A (dim, dstate),
 * B and C (batch, dstate, seqlen), init_state and final_state (batch, dim,
 * dstate), all complex as interleaved (re, im) fp32 pairs; delta_bias and D
 * (dim) fp32.  Nullable: delta_bias, D, z, final_state, init_state (zeros).
 * Flags: SSM_SOFTPLUS, SSM_EULER_B.  dstate: a power of two up to 64
 * (SSM_ERR_UNSUPPORTED otherwise).  All pointers 16-byte aligned
 * (SSM_ERR_ALIGN).  y must not overlap an input, final_state no input but
 * init_state, which it may equal exactly (an in-place carry).  The arithmetic is
 * the precise flavour (libm expf, expm1f, sincosf) for both I/O dtypes; no
 * workspace; asynchronous on `stream`.
 */
int ssm_scan_fwd_complex(const void* u, const void* delta, const float* delta_bias,
                         const float* A, const float* B, const float* C, const float* D,
                         const void* z, int delta_softplus, void* y, float* final_state,
                         const float* init_state, int64_t batch, int64_t dim, int64_t seqlen,
                         int64_t dstate, int io_dtype, void* stream);

/*
 * Backward of ssm_ssd_fwd (the chapter page's §5.1: SSD is the selective scan
 * of each channel of a head with the scalar A[h] for every state, the head's
 * step shared by its channels and the group's B, C): the derivatives of
 * Σ y·dy + Σ final_state·d_final_state, in the chunked form: the states
 * entering the chunks recomputed by a forward walk (held in fp32), the
 * derivatives reaching the chunks' end states by a reverse walk, then every
 * derivative of a chunk from its 64 steps; the products run on the tensor
 * cores with each fp32 operand split into two bf16 parts (about 16 bits kept),
 * sums and elementwise steps in fp32; sums over a group's heads and over
 * chunks in a fixed order, so results repeat bit for bit.
 *
 * Inputs, layouts, flags and supported shapes as ssm_ssd_fwd; dy (batch,
 * seqlen, nheads, headdim) bf16; d_final_state (batch, nheads, headdim,
 * dstate) fp32, nullable.  Outputs: dx, dz like x (bf16; dz required exactly
 * when z is given), ddt like dt (bf16), dA (nheads) fp32 required, dB, dC like
 * B (fp32, (batch, seqlen, ngroups, dstate)), dD and d_dt_bias (nheads) fp32
 * nullable, d_init_state like init_state (fp32, nullable).  Workspace: device
 * memory of at least ssm_ssd_bwd_workspace_bytes() bytes (the step terms, the
 * fp32 states and state derivatives of every chunk, per-head partial dB and
 * dC).  Errors as ssm_ssd_fwd.
 * Asynchronous on `stream`.
 */
size_t ssm_ssd_bwd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                                   int64_t ngroups, int64_t dstate);
int ssm_ssd_bwd(const void* x, const void* dt, const float* dt_bias, const float* A, const void* B,
                const void* C, const float* D, const void* z, int flags, const float* init_state,
                const void* dy, const float* d_final_state, void* dx, void* ddt, float* dA,
                float* dB, float* dC, float* dD, void* dz, float* d_dt_bias, float* d_init_state,
                int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                int64_t dstate, void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_H */
