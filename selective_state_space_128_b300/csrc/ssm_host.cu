// Host-buffer entry point of the scan: the copies between host memory and the
// device are part of the call, pipelined against the scan.
//
// The inputs (batch, dim, L) are cut into units that are contiguous in host
// memory: one batch row, or a block of channels of one row when the batch is
// small (a block of channels of a row is a contiguous run of its L-long
// rows); with the (batch, L, dim) layout a unit is always a whole row.  Each
// unit moves through three device slots in turn:
//
//   copy-in stream:   wait until the slot is free, copy u, delta, z, B, C
//                     (and init_state) of unit i into slot i % 3
//   caller's stream:  the scan of unit i on its slot
//   copy-out stream:  copy y and final_state of unit i back to the host, then
//                     mark the slot free
//
// so the copy-in of unit i+1, the scan of unit i and the copy-out of unit i-1
// run at the same time (the two copy directions use separate copy engines).
// The two copy streams and the events are created per call and released when
// their work completes; the caller's stream waits for the last copy-out, so
// the call is asynchronous on `stream` like every other entry point.
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/ssm.h"
#include "ssm_internal.h"

namespace {

constexpr int kSlots = 3;
constexpr int64_t kTargetUnits = 8;  // units per call when the batch is small

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

bool supported_n(int64_t n) {
  return n == 1 || n == 2 || n == 4 || n == 8 || n == 16 || n == 32 || n == 64 || n == 128;
}

struct HostPlan {
  int64_t dchunk = 0;        // channels per unit
  int64_t blocks = 0;        // units per batch row
  size_t io = 0, bc = 0, st = 0;  // bytes of one unit's u (and delta, z, y), B (and C), state
  size_t scan_ws = 0;        // the unit scan's carry scratch
  size_t o_params = 0, o_scan = 0, o_slots = 0, slot = 0, bytes = 0;
};

HostPlan host_plan(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype,
                   bool bld) {
  HostPlan p;
  const size_t esz = io_dtype == SSM_F32 ? 4 : 2;
  p.blocks = (bld || batch >= kTargetUnits) ? 1 : (kTargetUnits + batch - 1) / batch;
  if (p.blocks > dim) p.blocks = dim > 0 ? dim : 1;
  // a multiple of 4 channels, so that a block's slices of D and delta_bias (and
  // of A) start on 16-byte boundaries of the device copies
  p.dchunk = ((dim + p.blocks - 1) / p.blocks + 3) / 4 * 4;
  p.blocks = (dim + p.dchunk - 1) / p.dchunk;
  p.io = up256((size_t)p.dchunk * (size_t)seqlen * esz);
  p.bc = up256((size_t)dstate * (size_t)seqlen * 4);
  p.st = up256((size_t)p.dchunk * (size_t)dstate * 4);
  p.scan_ws = up256(ssm::scan_carry_bytes(1, p.dchunk, seqlen, dstate, io_dtype));
  const size_t params = up256((size_t)dim * (size_t)dstate * 4) + 2 * up256((size_t)dim * 4);
  // the status word first (ssm_status reads it there), then the parameters
  p.o_params = ssm::kScanStatusBytes;
  p.o_scan = p.o_params + params;
  p.o_slots = p.o_scan + p.scan_ws;
  p.slot = 4 * p.io + 2 * p.bc + 2 * p.st;
  p.bytes = p.o_slots + kSlots * p.slot;
  return p;
}

// Device copies of the call, released when their work completes.
struct Pipeline {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, end = nullptr, ready[kSlots] = {}, done[kSlots] = {}, freed[kSlots] = {};
  bool ok = true;
  Pipeline() {
    ok = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking) == cudaSuccess &&
         cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking) == cudaSuccess &&
         cudaEventCreateWithFlags(&start, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&end, cudaEventDisableTiming) == cudaSuccess;
    for (int s = 0; s < kSlots && ok; ++s)
      ok = cudaEventCreateWithFlags(&ready[s], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&done[s], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&freed[s], cudaEventDisableTiming) == cudaSuccess;
  }
  ~Pipeline() {  // destroying streams and events with work pending is allowed
    for (int s = 0; s < kSlots; ++s) {
      if (ready[s]) cudaEventDestroy(ready[s]);
      if (done[s]) cudaEventDestroy(done[s]);
      if (freed[s]) cudaEventDestroy(freed[s]);
    }
    if (start) cudaEventDestroy(start);
    if (end) cudaEventDestroy(end);
    if (in) cudaStreamDestroy(in);
    if (out) cudaStreamDestroy(out);
  }
};

bool copy(void* dst, const void* src, size_t n, cudaStream_t s) {
  return n == 0 || cudaMemcpyAsync(dst, src, n, cudaMemcpyDefault, s) == cudaSuccess;
}

}  // namespace

extern "C" {

size_t ssm_scan_fwd_host_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen,
                                         int64_t dstate, int io_dtype, int flags) {
  if (batch <= 0 || dim <= 0 || seqlen < 0 || batch > 65535) return 0;
  if ((io_dtype != SSM_F32 && io_dtype != SSM_BF16) || !supported_n(dstate)) return 0;
  if ((double)batch * (double)dim * (double)(seqlen > 0 ? seqlen : 1) >= 9.0e18) return 0;
  if (seqlen == 0)  // the status word and a row of zeros
    return ssm::kScanStatusBytes + up256((size_t)dim * (size_t)dstate * 4);
  return host_plan(batch, dim, seqlen, dstate, io_dtype, (flags & SSM_LAYOUT_BLD) != 0).bytes;
}

int ssm_scan_fwd_host(const void* u, const void* delta, const float* delta_bias, const float* A,
                      const float* B, const float* C, const float* D, const void* z, int flags,
                      void* y, float* final_state, const float* init_state, int64_t batch,
                      int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_ARG;
  if ((flags & ~(SSM_SOFTPLUS | SSM_EULER_B | SSM_LAYOUT_BLD)) != 0) return SSM_ERR_ARG;
  if (batch < 0 || dim < 0 || seqlen < 0 || dstate <= 0 || batch > 65535) return SSM_ERR_ARG;
  if ((double)batch * (double)dim * (double)(seqlen > 0 ? seqlen : 1) >= 9.0e18) return SSM_ERR_ARG;
  if (!supported_n(dstate)) return SSM_ERR_UNSUPPORTED;
  if (batch == 0 || dim == 0) return SSM_OK;  // no units
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return SSM_ERR_ALIGN;
  const size_t need = ssm_scan_fwd_host_workspace_bytes(batch, dim, seqlen, dstate, io_dtype, flags);
  if (!workspace || workspace_bytes < need) return SSM_ERR_WORKSPACE;
  cudaStream_t main = static_cast<cudaStream_t>(stream);
  const size_t row_st = (size_t)dim * (size_t)dstate * 4;
  if (seqlen == 0) {
    // no steps: final_state = init_state, or zeros (a device row of zeros copied per row)
    if (cudaMemsetAsync(workspace, 0, sizeof(int), main) != cudaSuccess) return SSM_ERR_CUDA;
    if (!final_state) return SSM_OK;
    if (init_state)
      return cudaMemcpyAsync(final_state, init_state, (size_t)batch * row_st, cudaMemcpyDefault,
                             main) == cudaSuccess
                 ? SSM_OK
                 : SSM_ERR_CUDA;
    unsigned char* zeros = static_cast<unsigned char*>(workspace) + ssm::kScanStatusBytes;
    if (cudaMemsetAsync(workspace, 0, ssm::kScanStatusBytes + row_st, main) != cudaSuccess)
      return SSM_ERR_CUDA;
    for (int64_t b = 0; b < batch; ++b)
      if (cudaMemcpyAsync(reinterpret_cast<unsigned char*>(final_state) + (size_t)b * row_st, zeros,
                          row_st, cudaMemcpyDefault, main) != cudaSuccess)
        return SSM_ERR_CUDA;
    return SSM_OK;
  }
  if (!u || !delta || !A || !B || !C || !y) return SSM_ERR_ARG;
  const bool bld = (flags & SSM_LAYOUT_BLD) != 0;
  const HostPlan pl = host_plan(batch, dim, seqlen, dstate, io_dtype, bld);

  const size_t esz = io_dtype == SSM_F32 ? 4 : 2;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  float* dA = reinterpret_cast<float*>(ws + pl.o_params);
  float* dD = reinterpret_cast<float*>(ws + pl.o_params + up256((size_t)dim * (size_t)dstate * 4));
  float* dBias = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(dD) + up256((size_t)dim * 4));
  void* scan_ws = pl.scan_ws ? ws + pl.o_scan : nullptr;
  // one status word for the whole call: zeroed here, set by any unit's scan
  int* status = reinterpret_cast<int*>(ws);
  if (cudaMemsetAsync(status, 0, sizeof(int), main) != cudaSuccess) return SSM_ERR_CUDA;

  Pipeline pp;
  if (!pp.ok) return SSM_ERR_CUDA;
  // everything earlier on the caller's stream comes first (it may produce the inputs)
  if (cudaEventRecord(pp.start, main) != cudaSuccess ||
      cudaStreamWaitEvent(pp.in, pp.start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(pp.out, pp.start, 0) != cudaSuccess)
    return SSM_ERR_CUDA;
  if (!copy(dA, A, (size_t)dim * (size_t)dstate * 4, pp.in) ||
      (D && !copy(dD, D, (size_t)dim * 4, pp.in)) ||
      (delta_bias && !copy(dBias, delta_bias, (size_t)dim * 4, pp.in)))
    return SSM_ERR_CUDA;

  const int64_t units = batch * pl.blocks;
  for (int64_t i = 0; i < units; ++i) {
    const int s = (int)(i % kSlots);
    const int64_t b = i / pl.blocks, d0 = (i % pl.blocks) * pl.dchunk;
    const int64_t dn = (d0 + pl.dchunk <= dim) ? pl.dchunk : dim - d0;
    unsigned char* slot = ws + pl.o_slots + (size_t)s * pl.slot;
    void* su = slot;
    void* sd = slot + pl.io;
    void* sz = slot + 2 * pl.io;
    void* sy = slot + 3 * pl.io;
    float* sB = reinterpret_cast<float*>(slot + 4 * pl.io);
    float* sC = reinterpret_cast<float*>(slot + 4 * pl.io + pl.bc);
    float* sh0 = reinterpret_cast<float*>(slot + 4 * pl.io + 2 * pl.bc);
    float* sh = reinterpret_cast<float*>(slot + 4 * pl.io + 2 * pl.bc + pl.st);
    // host offsets: (b, d0) of the (batch, dim, L) layout, or row b of (batch, L, dim)
    const size_t io_off = ((size_t)b * (size_t)dim + (size_t)d0) * (size_t)seqlen * esz;
    const size_t io_n = (size_t)dn * (size_t)seqlen * esz;
    const size_t bc_off = (size_t)b * (size_t)dstate * (size_t)seqlen * 4;
    const size_t bc_n = (size_t)dstate * (size_t)seqlen * 4;
    const size_t st_off = ((size_t)b * (size_t)dim + (size_t)d0) * (size_t)dstate * 4;
    const size_t st_n = (size_t)dn * (size_t)dstate * 4;

    if (i >= kSlots && cudaStreamWaitEvent(pp.in, pp.freed[s], 0) != cudaSuccess) return SSM_ERR_CUDA;
    const unsigned char* hu = static_cast<const unsigned char*>(u);
    const unsigned char* hd = static_cast<const unsigned char*>(delta);
    const unsigned char* hz = static_cast<const unsigned char*>(z);
    if (!copy(su, hu + io_off, io_n, pp.in) || !copy(sd, hd + io_off, io_n, pp.in) ||
        (z && !copy(sz, hz + io_off, io_n, pp.in)) ||
        !copy(sB, reinterpret_cast<const unsigned char*>(B) + bc_off, bc_n, pp.in) ||
        !copy(sC, reinterpret_cast<const unsigned char*>(C) + bc_off, bc_n, pp.in) ||
        (init_state && !copy(sh0, reinterpret_cast<const unsigned char*>(init_state) + st_off, st_n, pp.in)))
      return SSM_ERR_CUDA;
    if (cudaEventRecord(pp.ready[s], pp.in) != cudaSuccess ||
        cudaStreamWaitEvent(main, pp.ready[s], 0) != cudaSuccess)
      return SSM_ERR_CUDA;
    const int rc = ssm::scan_fwd_internal(
        su, sd, delta_bias ? dBias + d0 : nullptr, dA + (size_t)d0 * dstate, sB, sC,
        D ? dD + d0 : nullptr, z ? sz : nullptr, flags, sy, final_state ? sh : nullptr, 1, dn,
        seqlen, dstate, io_dtype, init_state ? sh0 : nullptr, status, false, scan_ws, pl.scan_ws,
        nullptr, 0, false, main, nullptr);
    if (rc != SSM_OK) return rc;
    if (cudaEventRecord(pp.done[s], main) != cudaSuccess ||
        cudaStreamWaitEvent(pp.out, pp.done[s], 0) != cudaSuccess)
      return SSM_ERR_CUDA;
    if (!copy(static_cast<unsigned char*>(y) + io_off, sy, io_n, pp.out) ||
        (final_state && !copy(reinterpret_cast<unsigned char*>(final_state) + st_off, sh, st_n, pp.out)))
      return SSM_ERR_CUDA;
    if (cudaEventRecord(pp.freed[s], pp.out) != cudaSuccess) return SSM_ERR_CUDA;
  }
  // the caller's stream completes after the last copy-out
  if (cudaEventRecord(pp.end, pp.out) != cudaSuccess || cudaStreamWaitEvent(main, pp.end, 0) != cudaSuccess)
    return SSM_ERR_CUDA;
  return SSM_OK;
}

}  // extern "C"
