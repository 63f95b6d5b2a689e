// Host/device-shared declarations of libssm (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ssm {

// Threads per block of the scan kernel.
constexpr int kScanThreads = 128;

// Arguments of one scan launch.  Pointers are device pointers; see include/ssm.h
// for layouts.  carry_h / carry_s are the per-segment carry records of a
// sequence split across blocks (null when nseg == 1).
struct ScanArgs {
  const void* u;
  const void* delta;
  const void* z;
  const float* bias;
  const float* A;
  const float* B;
  const float* C;
  const float* D;
  void* y;
  float* final_state;
  const float* init_state;
  float* carry_h;  // [nseg-1][batch*dim][N]: segment end state started from zero
  float* carry_s;  // [nseg-1][batch*dim]: sum of Δ over the segment
  int64_t batch, dim, L;
  int64_t seg_len;  // steps per segment, a multiple of the chunk length
  int nseg;
  int softplus;
  int vec_io;       // u/delta/z can be staged by TMA: their strides other than the unit one
                    // are multiples of 16 bytes
  int bld;          // u/delta/z are channel-major (unit channel stride) instead of
                    // time-major (unit time stride)
  // element strides (batch, channel, time) of u, delta, z and y; dense (batch, dim, L)
  // or (batch, L, dim) unless the caller gave others
  int64_t st_u[3], st_d[3], st_z[3], st_y[3];
  int vec_y;        // y has unit time stride and 16-byte aligned rows: vector stores
  int vec_bc;       // rows of B/C are 16-byte aligned
  int force_precise;
  int euler;        // B̄ = Δ B (runs on the precise flavour)
  int use_tma;      // set by the launcher: chunks staged by TMA
  // training forward: the state at the start of every 16-step chunk of the
  // sequence, [batch][ckpt_nch][dim][N] (the backward pass's checkpoints); null
  // when not saving
  float* ckpt;
  int64_t ckpt_nch;
  // device status word that a block which gives up waiting sets to 1 (null: the
  // library-wide word)
  int* status;
  // test of the failure path: block (0, 0, 0) of the output pass arms its
  // second chunk's barrier without issuing the copies, so its wait runs out
  // after test_limit_ns (its other waits use the same limit)
  int test_stall;
  int64_t test_limit_ns;
};

struct ScanPlan {
  int nseg;
  int64_t seg_len;
  size_t workspace_bytes;
  int chunk;  // time steps per chunk
  int chans;  // channels per block
};

// Plan for given sizes on a device with `sm_count` SMs.
ScanPlan scan_plan(int64_t batch, int64_t dim, int64_t L, int64_t N, int io_dtype, int sm_count,
                   bool allow_split);

// Enqueue the scan (one or two kernels). Returns cudaSuccess or the launch error.
cudaError_t scan_launch(const ScanArgs& a, int64_t N, int io_dtype, const ScanPlan& plan,
                        cudaStream_t stream);

// The two-warp-block scan (ssm_scan_fast.cu) for N = 16 and bf16 I/O whose views
// TMA can stage, zero-order hold: whether it applies, whether it is the faster
// choice for these sizes (enough of its warps, one per 8 channels, to give every
// SM 16 of them: below that the block kernel's shared conversion wins), and its
// launch (a.status must point at a device word).
bool scan_fast_applies(const ScanArgs& a, int64_t N, int io_dtype);
bool scan_fast_preferred(const ScanArgs& a);
cudaError_t scan_fast_launch(const ScanArgs& a, cudaStream_t stream);

// Channels per unit of work that the plan sizes the split for (the fast scan's
// warp: 8 channels at N = 16).
constexpr int kFastChannels = 8;

// Arguments of the scan with a complex diagonal A (ssm_scan_complex.cu): A (dim, N),
// B, C (batch, N, L) and the states (batch, dim, N) as (re, im) pairs; u, delta, z,
// y (batch, dim, L) in the I/O dtype.
struct ComplexScanArgs {
  const void* u;
  const void* delta;
  const void* z;
  const float* bias;
  const float2* A;
  const float2* B;
  const float2* C;
  const float* D;
  void* y;
  float2* final_state;
  const float2* init_state;
  int64_t batch, dim, L;
  int softplus;
  int euler;
};

cudaError_t scan_complex_launch(const ComplexScanArgs& a, int64_t N, int io_dtype, cudaStream_t stream);

struct UpdateArgs {
  float* state;
  const void* u;
  const void* delta;
  const void* z;
  const float* bias;
  const float* A;
  const float* B;
  const float* C;
  const float* D;
  void* y;
  int64_t batch, dim;
  int softplus;
  int force_precise;
  int euler;
};

// Reads and clears, in stream order, the library-wide device status word of the
// scans that ran without a workspace (0 = none, 1 = a wait timed out), then
// synchronises `stream`.
cudaError_t scan_library_status(int* code, cudaStream_t stream);

// Bytes at the start of a scan workspace that hold its status word.
constexpr size_t kScanStatusBytes = 256;

// The scan after the C ABI's argument checks (ssm_api.cu), for the entry points
// that manage the workspace themselves: `status` is the device status word (null:
// the library-wide word), zeroed on the stream first when `zero_status`; `carry`
// (carry_bytes) the split plan's scratch (null: the sequence is not split);
// `strides` the 12 element strides (batch, channel, time) of u, delta, z, y (null:
// dense, as the SSM_LAYOUT_BLD flag says).
int scan_fwd_internal(const void* u, const void* delta, const float* delta_bias, const float* A,
                      const float* B, const float* C, const float* D, const void* z, int flags,
                      void* y, float* final_state, int64_t batch, int64_t dim, int64_t seqlen,
                      int64_t dstate, int io_dtype, const float* init_state, int* status,
                      bool zero_status, void* carry, size_t carry_bytes, void* bwd_workspace,
                      size_t bwd_workspace_bytes, bool train, cudaStream_t stream,
                      const int64_t* strides);

// The smaller scratch limit that the failure-path test mode sets for the
// no-allocation scan (0: none).
size_t noalloc_test_limit();

// The scan kernel the test mode asks for: 0 = chosen by size, 1 = the block kernel
// (ssm_scan.cu), 2 = the two-warp-block kernel (ssm_scan_fast.cu) wherever it applies.
int scan_kernel_choice();

// Carry-record bytes of the split plan for these sizes on the current device (0:
// the plan does not split).
size_t scan_carry_bytes(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype);

cudaError_t update_launch(const UpdateArgs& a, int64_t N, int io_dtype, cudaStream_t stream);

// Arguments of the backward pass (device pointers; layouts as in include/ssm.h).
struct BwdArgs {
  const void* u;
  const void* delta;
  const void* z;
  const float* bias;
  const float* A;
  const float* B;
  const float* C;
  const float* D;
  const float* init_state;
  const void* dy;
  const float* d_final_state;
  void* du;
  void* ddelta;
  void* dz;
  float* dA;
  float* dB;
  float* dC;
  float* dD;
  float* d_bias;
  float* d_init_state;
  // workspace parts (see BwdLayout)
  float* ckpt;     // [batch][nch][dim][N]: state at the start of every chunk
  float* ws_B;     // [batch][nblk][N][L]: per-block sums over the block's channels
  float* ws_C;     // [batch][nblk][N][L]
  float* ws_A;     // [nseg][batch][dim][N]: dA per segment and batch row
  float* ws_D;     // [nseg][batch][dim]
  float* ws_bias;  // [nseg][batch][dim]
  int64_t batch, dim, L, nblk;
  int softplus;
  int force_precise;
  int euler;
  int saved;  // ckpt already holds the chunk-start states (a training forward wrote them)
  int bld;    // u/delta/z/dy/du/ddelta/dz are (batch, L, dim)
  // a sequence split into nseg segments of seg_len steps (grid.z), each folding
  // the carries of the others: the forward's end state from zero and ΣΔ of
  // segments 0 .. nseg-2 ([nseg-1][batch*dim][N], [nseg-1][batch*dim]), and the
  // adjoint's value at the start from a zero adjoint at the end and ΣΔ of
  // segments 1 .. nseg-1 (segment k at index k-1, same shapes); ws_A, ws_D,
  // ws_bias hold one slice per segment ([nseg][batch][...])
  int nseg;
  int64_t seg_len;
  float* fcarry_h;
  float* fcarry_s;
  float* acarry_l;
  float* acarry_s;
  int* status;  // device word for the forward carries' bounded waits
};

// Chunk length of the backward pass for state size N (the checkpoint interval).
int bwd_chunk(int64_t N);

// Workspace of the backward pass: byte offsets of its parts (256-byte aligned)
// and the total; nblk = channel blocks per batch row, nch = chunks per sequence.
struct BwdLayout {
  int64_t nblk, nch;
  int nseg;          // segments the sequence is split into (1: none)
  int64_t seg_len;   // steps per segment (a multiple of 16 and of the chunk)
  size_t o_ckpt, o_B, o_C, o_A, o_D, o_bias, o_fh, o_fs, o_al, o_as, bytes;
};

// The plan splits the sequence into segments when its blocks would fill less
// than half a wave on `sm_count` SMs.
BwdLayout bwd_layout(int64_t batch, int64_t dim, int64_t L, int64_t N, int sm_count);

// Enqueue the backward pass: the adjoint's segment carries when the sequence is
// split (the forward's come first, from scan_carries_launch, unless the states
// were saved), the per-block kernel, the fixed-order sums.
cudaError_t bwd_launch(const BwdArgs& a, int64_t N, int io_dtype, cudaStream_t stream);

// The forward scan's first pass alone (the split plan's segment end states from
// zero and ΣΔ into a.carry_h / a.carry_s for segments 0 .. a.nseg-2), with the
// block kernel.
cudaError_t scan_carries_launch(const ScanArgs& a, int64_t N, int io_dtype, cudaStream_t stream);

// Arguments of the conv1d + SiLU front end (device pointers; layouts as in
// include/ssm.h).  For the one-token update, state_out is the in/out state.
struct ConvArgs {
  const void* x;
  const float* w;
  const float* bias;
  const void* state_in;
  void* out;
  void* state_out;
  int64_t batch, dim, L;
  bool silu;
  bool precise;
  bool bld;  // x and out are (batch, L, dim)
};

// Enqueue the conv pass (update = false: over a sequence, then the new state)
// or the one-token update on the rolling state.
cudaError_t conv_launch(const ConvArgs& a, int64_t width, int io_dtype, bool update,
                        cudaStream_t stream);

// Arguments of the conv1d backward: x, dout, dx as the forward's x (io dtype),
// weight (dim, K) fp32, bias (dim) fp32 or null, state_in (batch, dim, K-1) io
// dtype or null; outputs dw (dim, K), dbias (dim) or null, dstate (batch, dim,
// K-1) or null, fp32.
struct ConvBwdArgs {
  const void* x;
  const float* w;
  const float* bias;
  const void* state_in;
  const void* dout;
  void* dx;
  float* dw;
  float* dbias;
  float* dstate;
  int64_t batch, dim, L;
  bool silu;
  bool precise;  // libm exponential and division (float32 I/O)
  bool bld;
};

cudaError_t conv_bwd_launch(const ConvBwdArgs& a, int64_t width, int io_dtype, cudaStream_t stream);

// Arguments of the chunked scalar-A SSM (Mamba-2 SSD).  x, z, y (batch, L, H,
// P) bf16; dt (batch, L, H) bf16; B, C (batch, L, G, N) bf16; A, D, dt_bias (H)
// fp32; states (batch, H, P, N) fp32.  Workspace parts: the states entering
// each chunk [batch][nch][H][P][N] bf16, the chunks' step terms
// [batch][nch][H][s | β | w] (3 x 64 fp32) and the chunks' C Bᵀ per group
// [batch][nch][G][64][64] fp32.
struct SsdArgs {
  const void* x;
  const void* dt;
  const float* dt_bias;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  void* y;
  float* final_state;
  const float* init_state;
  __nv_bfloat16* ws_hin;
  float* ws_terms;
  float* ws_cb;
  int64_t batch, L, H, G, nch;
  int softplus;
  int euler;
  int* status;  // device word set when a bounded wait runs out (the library-wide word)
};

// The chunk length of the SSD kernels and the floats of one (batch, chunk, head)
// record of the step terms [s | β | w] in the workspace.
constexpr int kSsdChunk = 64;
constexpr int kSsdTermsRec = 3 * kSsdChunk;

struct SsdLayout {
  int64_t nch;
  size_t o_hin, o_terms, o_cb, bytes;
};

SsdLayout ssd_layout(int64_t batch, int64_t L, int64_t H, int64_t G, int64_t N);
cudaError_t ssd_launch(const SsdArgs& a, int64_t N, cudaStream_t stream);

// The step terms alone: per (batch, chunk, head) the record [s | β | w] of
// kSsdTermsRec floats in a.ws_terms (reads dt, dt_bias, A, softplus, euler).
cudaError_t ssd_terms_launch(const SsdArgs& a, cudaStream_t stream);

// The chunks' C Bᵀ on the tcgen05 tensor cores (ssm_ssd_tc.cu): one CTA per
// (batch, chunk, group), fp32 rows of 64 into a.ws_cb (tiles on and below the
// diagonal).
cudaError_t ssd_cb_tc_launch(const SsdArgs& a, int64_t N, cudaStream_t stream);

// The chunk outputs y = (mask ∘ C Bᵀ) X + exp(s_t) C Hᵀ + D x, gated, on tcgen05
// (ssm_ssd_tc.cu): persistent CTAs over the (batch, chunk, head) items.
cudaError_t ssd_chunk_tc_launch(const SsdArgs& a, int64_t N, cudaStream_t stream);

// Device address of the library-wide status word on the current device (null on
// error).
int* library_status_word();

}  // namespace ssm
