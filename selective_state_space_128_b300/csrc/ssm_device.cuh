// Device helpers shared by the scan and decode kernels: element I/O for
// float32 / bfloat16, the two arithmetic flavours (fast: MUFU ex2 and packed
// f32x2 math; precise: CUDA libm), and packed-pair arithmetic in inline PTX.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ssm {

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// Element I/O. bfloat16 <-> float conversions are exact widening / RNE narrowing.
// ---------------------------------------------------------------------------
template <typename IO> struct io_traits;
template <> struct io_traits<float> {
  static constexpr int kBytes = 4;
  __device__ static float to_f32(float v) { return v; }
  __device__ static float from_f32(float v) { return v; }
};
template <> struct io_traits<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  __device__ static float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ static __nv_bfloat16 from_f32(float v) { return __float2bfloat16_rn(v); }
};

// ---------------------------------------------------------------------------
// Packed pairs (two fp32 lanes in one 64-bit register): one instruction issue
// for two FP32 operations on sm_100-class SMs.
// ---------------------------------------------------------------------------
struct f2 {
  unsigned long long r;
};

__device__ __forceinline__ f2 pack2(float lo, float hi) {
  f2 v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v.r) : "f"(lo), "f"(hi));
  return v;
}
__device__ __forceinline__ void unpack2(f2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v.r));
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d.r) : "l"(a.r), "l"(b.r));
  return d;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  f2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d.r) : "l"(a.r), "l"(b.r));
  return d;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
  f2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d.r) : "l"(a.r), "l"(b.r));
  return d;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d.r) : "l"(a.r), "l"(b.r), "l"(c.r));
  return d;
}

// Shared-memory accesses of packed pairs (the address must be 8- / 16-byte aligned).
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void lds_pairs(const void* p, f2& a, f2& b) {
  asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a.r), "=l"(b.r) : "r"(smem_u32(p)));
}
__device__ __forceinline__ void lds_pair(const void* p, f2& a) {
  asm volatile("ld.shared.b64 %0, [%1];" : "=l"(a.r) : "r"(smem_u32(p)));
}
__device__ __forceinline__ void sts_pairs(void* p, f2 a, f2 b) {
  asm volatile("st.shared.v2.b64 [%0], {%1, %2};" ::"r"(smem_u32(p)), "l"(a.r), "l"(b.r) : "memory");
}
__device__ __forceinline__ void sts_pair(void* p, f2 a) {
  asm volatile("st.shared.b64 [%0], %1;" ::"r"(smem_u32(p)), "l"(a.r) : "memory");
}

// ---------------------------------------------------------------------------
// mbarrier primitives (inline PTX) and a bounded wait
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for phase `parity` of `bar`, giving up after `limit_ns` (default kWaitLimitNs).
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: every hand-over takes microseconds
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}
// ---------------------------------------------------------------------------
// Fast transcendental pieces (MUFU). ex2.approx.ftz: relative error ~2^-22.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_fast(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_fast(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// softplus(x) = log(1 + e^x).
// Fast flavour: e = 2^(x log2 e) on the MUFU; for x < -4 (e < 0.0184) the
// alternating series e - e^2/2 + e^3/3 - e^4/4 (truncation < e^5/5, relative
// < 4e-10) avoids the rounding of 1 + e; for -4 <= x <= 15 it is
// ln2 * log2(1 + e) (relative error below ~1e-5, from lg2.approx's absolute
// error over log2(1+e) >= 0.026); above 15 it returns x (error < 3e-7).
__device__ __forceinline__ float softplus_fast(float x) {
  float e = ex2_fast(x * kLog2e);
  float series = e * fmaf(e, fmaf(e, fmaf(e, -0.25f, 1.0f / 3.0f), -0.5f), 1.0f);
  float logv = kLn2 * lg2_fast(1.0f + e);
  float r = x < -4.0f ? series : logv;
  return x > 15.0f ? x : r;
}
// Precise flavour: CUDA libm, both branches free of overflow and cancellation.
__device__ __forceinline__ float softplus_precise(float x) {
  return x > 0.0f ? x + log1pf(expf(-x)) : log1pf(expf(x));
}

// E consecutive I/O elements <-> float, as one access of E elements (up to
// 16 bytes) or several 16-byte ones (the caller guarantees the alignment).
template <typename IO, int E> struct vecio;
template <int E> struct vecio<__nv_bfloat16, E> {
  // E consecutive bf16 -> float (E = 1: 2 bytes, 2: 4, 4: 8, 8: 16, 16: 32)
  __device__ static void load(const __nv_bfloat16* p, float (&v)[E]) {
    if constexpr (E == 1) {
      v[0] = __bfloat162float(*p);
    } else {
      uint32_t w[E / 2];
      if constexpr (E == 2) {
        w[0] = *reinterpret_cast<const uint32_t*>(p);
      } else if constexpr (E == 4) {
        const uint2 q = *reinterpret_cast<const uint2*>(p);
        w[0] = q.x; w[1] = q.y;
      } else {
#pragma unroll
        for (int k = 0; k < E / 8; ++k) {
          const uint4 q = reinterpret_cast<const uint4*>(p)[k];
          w[4 * k] = q.x; w[4 * k + 1] = q.y; w[4 * k + 2] = q.z; w[4 * k + 3] = q.w;
        }
      }
#pragma unroll
      for (int i = 0; i < E / 2; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      }
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float (&v)[E]) {
    if constexpr (E == 1) {
      *p = __float2bfloat16_rn(v[0]);
    } else {
      uint32_t w[E / 2];
#pragma unroll
      for (int i = 0; i < E / 2; ++i) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      if constexpr (E == 2) {
        *reinterpret_cast<uint32_t*>(p) = w[0];
      } else if constexpr (E == 4) {
        *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
      } else {
#pragma unroll
        for (int k = 0; k < E / 8; ++k)
          reinterpret_cast<uint4*>(p)[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
      }
    }
  }
};
template <int E> struct vecio<float, E> {
  __device__ static void load(const float* p, float (&v)[E]) {
    if constexpr (E == 1) {
      v[0] = *p;
    } else if constexpr (E == 2) {
      const float2 q = *reinterpret_cast<const float2*>(p);
      v[0] = q.x; v[1] = q.y;
    } else {
#pragma unroll
      for (int k = 0; k < E / 4; ++k) {
        const float4 q = reinterpret_cast<const float4*>(p)[k];
        v[4 * k] = q.x; v[4 * k + 1] = q.y; v[4 * k + 2] = q.z; v[4 * k + 3] = q.w;
      }
    }
  }
  __device__ static void store(float* p, const float (&v)[E]) {
    if constexpr (E == 1) {
      *p = v[0];
    } else if constexpr (E == 2) {
      *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
    } else {
#pragma unroll
      for (int k = 0; k < E / 4; ++k)
        reinterpret_cast<float4*>(p)[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    }
  }
};

// silu(z) = z * sigmoid(z)
__device__ __forceinline__ float silu_fast(float z) {
  return z * rcp_fast(1.0f + ex2_fast(-z * kLog2e));
}
__device__ __forceinline__ float silu_precise(float z) { return z / (1.0f + expf(-z)); }

}  // namespace ssm
