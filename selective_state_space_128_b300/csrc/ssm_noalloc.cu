// ssm_scan_fwd_noalloc: the scan for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run the scan: code running inside a memory-capped process that has
// handed all device memory to its own pool, plug-in hosts that forbid
// allocation after start-up, or real-time loops where an allocation could
// block.  For long sequences with few channels the scan splits the sequence
// across blocks and needs scratch memory for the per-segment carry records;
// this entry point takes that scratch from a fixed array compiled into the
// library instead of from the caller.
//
// The array lives in device global memory of every GPU that loads the
// library, for the life of the process.  Host code may not use the array's
// name as a device address (on the host it names a host-side stand-in), so
// the device address is looked up once per device with cudaGetSymbolAddress,
// with that device current, and cached.  A device reset (cudaDeviceReset)
// while the library is loaded would leave a stale cached address: it is not
// supported.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/ssm.h"
#include "ssm_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_scan_scratch[SSM_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scan_scratch on device `dev`, which is current (nullptr on
// error).
void* scratch_address(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scan_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

namespace ssm {

// Scratch limit of ssm_scan_fwd_noalloc: SSM_STATIC_SCRATCH_BYTES, or a smaller
// one set by the failure-path test mode (ssm_set_test_mode).
size_t noalloc_limit(size_t test_limit) {
  return test_limit > 0 && test_limit < (size_t)SSM_STATIC_SCRATCH_BYTES
             ? test_limit
             : (size_t)SSM_STATIC_SCRATCH_BYTES;
}

}  // namespace ssm

extern "C" int ssm_scan_fwd_noalloc(const void* u, const void* delta, const float* delta_bias,
                                    const float* A, const float* B, const float* C,
                                    const float* D, const void* z, int delta_softplus, void* y,
                                    float* final_state, int64_t batch, int64_t dim,
                                    int64_t seqlen, int64_t dstate, int io_dtype,
                                    const float* init_state, void* stream) {
  // The plan's carry-record need; sizes the scan rejects give 0 here and are
  // reported by the scan below with its own status.
  const size_t need = ssm_scan_workspace_bytes(batch, dim, seqlen, dstate, io_dtype);
  const size_t carry = need > ssm::kScanStatusBytes ? need - ssm::kScanStatusBytes : 0;
  if (carry > ssm::noalloc_limit(ssm::noalloc_test_limit())) return SSM_ERR_WORKSPACE;
  // the scratch is the current device's: the stream must belong to it
  int dev = 0, sdev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (st != nullptr && st != cudaStreamLegacy && st != cudaStreamPerThread) {
    if (cudaStreamGetDevice(st, &sdev) != cudaSuccess) return SSM_ERR_CUDA;
    if (sdev != dev) return SSM_ERR_ARG;
  }
  void* scratch = scratch_address(dev);
  if (!scratch) return SSM_ERR_CUDA;
  // status: the library-wide word (the caller has no workspace to hold one)
  return ssm::scan_fwd_internal(u, delta, delta_bias, A, B, C, D, z, delta_softplus, y,
                                final_state, batch, dim, seqlen, dstate, io_dtype, init_state,
                                nullptr, false, scratch, (size_t)SSM_STATIC_SCRATCH_BYTES, nullptr,
                                0, false, st, nullptr);
}
