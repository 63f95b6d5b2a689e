// Host/device-shared declarations of libssm (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
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
  int vec_io;       // rows of u/delta/z/y are 16-byte aligned
  int vec_bc;       // rows of B/C are 16-byte aligned
  int force_precise;
  int use_tma;      // set by the launcher: chunks staged by TMA
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
};

// Synchronises `stream`, then reads and clears the scan kernels' device error
// word (0 = none, 1 = a TMA wait timed out).
cudaError_t scan_device_error(int* code, cudaStream_t stream);

cudaError_t update_launch(const UpdateArgs& a, int64_t N, int io_dtype, cudaStream_t stream);

}  // namespace ssm
