// Warp-level tensor-core helpers shared by the SSD state walks (ssm_ssd.cu and
// the backward's walks in ssm_ssd_bwd.cu): ldmatrix, mma.sync m16n8k16 bf16
// with fp32 accumulation, and cp.async staging of bf16 rows into padded
// shared-memory rows.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "ssm_device.cuh"

namespace ssm {

// Four 8x8 bf16 matrices from shared memory (each lane gives one row address:
// lanes 8i..8i+7 the rows of matrix i); the _t form transposes each.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
// d += a (16x16, row-major) * b (16x8, column-major); bf16 in, fp32 accumulate
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 16-byte asynchronous copy global -> shared; with `valid` false nothing is
// read (source size 0) and the destination is zero-filled.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int K> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(K) : "memory");
}

// Issues the copies of ROWS rows of COLS bf16 (a multiple of 8) from global rows
// `gstride` elements apart into shared rows SSTRIDE elements apart, THREADS
// threads sharing them; rows at or past `valid` are zero-filled (their source is
// not read).  Every load is in flight at once; the caller commits the group and
// waits for it.
template <int ROWS, int COLS, int SSTRIDE, int THREADS>
__device__ __forceinline__ void ssd_stage(__nv_bfloat16* dst, const __nv_bfloat16* src,
                                          int64_t gstride, int valid) {
  constexpr int VPR = COLS / 8;  // 16-byte vectors per row
  static_assert((ROWS * VPR) % THREADS == 0, "whole copies per thread");
#pragma unroll
  for (int k = 0; k < ROWS * VPR / THREADS; ++k) {
    const int e = threadIdx.x + k * THREADS;
    const int r = e / VPR, v = e - r * VPR;
    const bool ok = r < valid;
    cp_async16(dst + r * SSTRIDE + v * 8, src + (ok ? r : 0) * gstride + v * 8, ok);
  }
}

}  // namespace ssm
