// One-token decode step (recurrent mode) for sm_103a.
//
// The summary page ("Mamba: Linear-Time Sequence Modeling", section 4b, the
// derivation under equation (2), and the efficiency table of section 4c)
// describes inference as the recurrence run one step at a time on a stored
// (batch, d_inner, N) state: h <- Ā h + B̄ u, y = C·h + D u, gated by silu(z),
// with Ā, B̄ from the zero-order hold of equation (4).
//
// The step reads and writes the float32 state once (64 bytes per channel at
// N = 16) and is bound by HBM bandwidth, so the kernel is built to keep many
// bytes in flight with few instructions:
//  * G = 4 lanes share a channel (N <= 16; beyond, G = N/8 lanes of 8 states),
//    each holding N/G contiguous states that it loads and stores as 16-byte
//    vectors, so a warp touches whole channels (512 contiguous bytes per access
//    at N = 16);
//  * each thread handles K channels spaced one warp-width of channels apart
//    and issues all of their loads before any arithmetic, so 64 bytes of
//    state per thread are in flight at once;
//  * the grid is (channel blocks, batch): no integer division per thread, and
//    the block's B/C row is shared by all of its channels.
// The G partial readouts of a channel are summed with two xor-shuffles.  The
// state's 16-byte loads and stores carry streaming cache hints (evict first):
// 40.8 -> 39.0 us per step at batch 256 x d_inner 5120 (the hint on the loads
// alone measured 49.9 us).
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

constexpr int kUpdThreads = 256;
constexpr int kUpdK = 4;  // channels per thread

template <typename IO, int N>
__global__ void __launch_bounds__(kUpdThreads) update_kernel(const UpdateArgs p) {
  // lanes per channel: 4 up to N = 16, then 8 states per lane (8 lanes at N = 64,
  // 16 at N = 128)
  constexpr int G = N <= 16 ? (N >= 4 ? 4 : N) : N / 8;
  constexpr int NPT = N / G;
  constexpr int CPB = kUpdThreads / G;  // channels per block per k
  const int tid = threadIdx.x;
  const int g = tid % G;
  const int64_t b = blockIdx.y;
  const int64_t dbase = (int64_t)blockIdx.x * (CPB * kUpdK) + tid / G;

  // B, C of this batch row for this lane's states (shared by all channels)
  float Bv[NPT], Cv[NPT];
  {
    const float* Bp = p.B + b * N + g * NPT;
    const float* Cp = p.C + b * N + g * NPT;
    if constexpr (NPT % 4 == 0) {
#pragma unroll
      for (int j = 0; j < NPT; j += 4) {
        const float4 b4 = __ldg(reinterpret_cast<const float4*>(Bp + j));
        const float4 c4 = __ldg(reinterpret_cast<const float4*>(Cp + j));
        Bv[j] = b4.x; Bv[j + 1] = b4.y; Bv[j + 2] = b4.z; Bv[j + 3] = b4.w;
        Cv[j] = c4.x; Cv[j + 1] = c4.y; Cv[j + 2] = c4.z; Cv[j + 3] = c4.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < NPT; ++j) { Bv[j] = __ldg(Bp + j); Cv[j] = __ldg(Cp + j); }
    }
  }

  // issue every load of the K channels first
  float st[kUpdK][NPT], Av[kUpdK][NPT], uu[kUpdK], xx[kUpdK], zz[kUpdK], Dd[kUpdK];
  bool ok[kUpdK];
  const IO* gu = static_cast<const IO*>(p.u);
  const IO* gd = static_cast<const IO*>(p.delta);
  const IO* gz = static_cast<const IO*>(p.z);
#pragma unroll
  for (int k = 0; k < kUpdK; ++k) {
    const int64_t d = dbase + (int64_t)k * CPB;
    ok[k] = d < p.dim;
    const int64_t dd = ok[k] ? d : 0;
    const int64_t row = b * p.dim + dd;
    const float* sp = p.state + row * N + g * NPT;
    const float* Ap = p.A + dd * N + g * NPT;
    if constexpr (NPT % 4 == 0) {
#pragma unroll
      for (int j = 0; j < NPT; j += 4) {
        // the state is read once and written once per step: streaming cache hints
        const float4 s4 = __ldcs(reinterpret_cast<const float4*>(sp + j));
        const float4 a4 = __ldg(reinterpret_cast<const float4*>(Ap + j));
        st[k][j] = s4.x; st[k][j + 1] = s4.y; st[k][j + 2] = s4.z; st[k][j + 3] = s4.w;
        Av[k][j] = a4.x; Av[k][j + 1] = a4.y; Av[k][j + 2] = a4.z; Av[k][j + 3] = a4.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < NPT; ++j) { st[k][j] = sp[j]; Av[k][j] = __ldg(Ap + j); }
    }
    uu[k] = io_traits<IO>::to_f32(gu[row]);
    xx[k] = io_traits<IO>::to_f32(gd[row]) + (p.bias ? __ldg(p.bias + dd) : 0.f);
    zz[k] = gz ? io_traits<IO>::to_f32(gz[row]) : 0.f;
    Dd[k] = p.D ? __ldg(p.D + dd) : 0.f;
  }

#pragma unroll
  for (int k = 0; k < kUpdK; ++k) {
    bool precise = p.force_precise != 0 || p.euler != 0;
#pragma unroll
    for (int j = 0; j < NPT; ++j) precise |= (Av[k][j] == 0.f);
    const float x = xx[k];
    const float dt = p.softplus ? (precise ? softplus_precise(x) : softplus_fast(x)) : x;
    float acc = 0.f;
    if (!precise) {
      // h = Ā (h - v) + v with Ā = 2^(Δ A log2 e), v = -B u / A
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const float a = ex2_fast(dt * (Av[k][j] * kLog2e));
        const float nv = Bv[j] * uu[k] * -rcp_fast(Av[k][j]);
        st[k][j] = fmaf(a, st[k][j] - nv, nv);
        acc = fmaf(Cv[j], st[k][j], acc);
      }
    } else {
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const float xa = dt * Av[k][j];
        const float coef = (Av[k][j] != 0.f && !p.euler) ? expm1f(xa) / Av[k][j] : dt;
        st[k][j] = fmaf(expf(xa), st[k][j], coef * (Bv[j] * uu[k]));
        acc = fmaf(Cv[j], st[k][j], acc);
      }
    }
#pragma unroll
    for (int s = G / 2; s >= 1; s /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, s);

    if (!ok[k]) continue;
    const int64_t row = b * p.dim + dbase + (int64_t)k * CPB;
    float* sp = p.state + row * N + g * NPT;
    if constexpr (NPT % 4 == 0) {
#pragma unroll
      for (int j = 0; j < NPT; j += 4)
        __stcs(reinterpret_cast<float4*>(sp + j),
               make_float4(st[k][j], st[k][j + 1], st[k][j + 2], st[k][j + 3]));
    } else {
#pragma unroll
      for (int j = 0; j < NPT; ++j) sp[j] = st[k][j];
    }
    if (g == 0) {
      float yv = fmaf(Dd[k], uu[k], acc);
      if (gz) yv *= precise ? silu_precise(zz[k]) : silu_fast(zz[k]);
      static_cast<IO*>(p.y)[row] = io_traits<IO>::from_f32(yv);
    }
  }
}

template <typename IO, int N>
static cudaError_t upd_typed(const UpdateArgs& a, cudaStream_t stream) {
  constexpr int G = N <= 16 ? (N >= 4 ? 4 : N) : N / 8;
  constexpr int per_block = kUpdThreads / G * kUpdK;
  const dim3 grid((unsigned)((a.dim + per_block - 1) / per_block), (unsigned)a.batch);
  update_kernel<IO, N><<<grid, kUpdThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <typename IO>
static cudaError_t upd_io(const UpdateArgs& a, int64_t N, cudaStream_t stream) {
  switch (N) {
    case 1: return upd_typed<IO, 1>(a, stream);
    case 2: return upd_typed<IO, 2>(a, stream);
    case 4: return upd_typed<IO, 4>(a, stream);
    case 8: return upd_typed<IO, 8>(a, stream);
    case 16: return upd_typed<IO, 16>(a, stream);
    case 32: return upd_typed<IO, 32>(a, stream);
    case 64: return upd_typed<IO, 64>(a, stream);
    case 128: return upd_typed<IO, 128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t update_launch(const UpdateArgs& a, int64_t N, int io_dtype, cudaStream_t stream) {
  if (a.batch == 0 || a.dim == 0) return cudaSuccess;
  if (io_dtype == 0) return upd_io<float>(a, N, stream);
  return upd_io<__nv_bfloat16>(a, N, stream);
}

}  // namespace ssm
