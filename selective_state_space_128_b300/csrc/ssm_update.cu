// One-token decode step (recurrent mode) for sm_103a.
//
// The summary page ("Mamba: Linear-Time Sequence Modeling", section 4b, the
// derivation under equation (2), and the efficiency table of section 4c)
// describes inference as the recurrence run one step at a time on a stored
// (batch, d_inner, N) state: h <- Ā h + B̄ u, y = C·h + D u, gated by silu(z),
// with Ā, B̄ from the zero-order hold of equation (4).
//
// The step reads and writes the float32 state once (64 bytes per channel at
// N = 16) and is bound by HBM bandwidth.  G = 4 lanes share a channel; each
// holds N/4 contiguous states, loaded and stored as 16-byte vectors so that a
// warp touches 8 whole channels (512 contiguous bytes per access).  The G
// partial readouts are summed with two xor-shuffles.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

constexpr int kUpdThreads = 256;

template <typename IO, int N>
__global__ void __launch_bounds__(kUpdThreads) update_kernel(const UpdateArgs p) {
  constexpr int G = N >= 4 ? 4 : N;
  constexpr int NPT = N / G;
  const int64_t gid = (int64_t)blockIdx.x * kUpdThreads + threadIdx.x;
  const int64_t row = gid / G;  // b * dim + d
  const int g = (int)(gid - row * G);
  const int64_t nrows = p.batch * p.dim;
  const bool ok = row < nrows;
  const int64_t rr = ok ? row : 0;
  const int64_t b = rr / p.dim, d = rr - (rr / p.dim) * p.dim;

  float st[NPT], A[NPT], Bv[NPT], Cv[NPT];
  float* sp = p.state + rr * N + g * NPT;
  const float* Ap = p.A + d * N + g * NPT;
  const float* Bp = p.B + b * N + g * NPT;
  const float* Cp = p.C + b * N + g * NPT;
  if (ok) {
    if constexpr (NPT % 4 == 0) {
#pragma unroll
      for (int j = 0; j < NPT; j += 4) {
        const float4 s4 = *reinterpret_cast<const float4*>(sp + j);
        const float4 a4 = __ldg(reinterpret_cast<const float4*>(Ap + j));
        const float4 b4 = __ldg(reinterpret_cast<const float4*>(Bp + j));
        const float4 c4 = __ldg(reinterpret_cast<const float4*>(Cp + j));
        st[j] = s4.x; st[j + 1] = s4.y; st[j + 2] = s4.z; st[j + 3] = s4.w;
        A[j] = a4.x; A[j + 1] = a4.y; A[j + 2] = a4.z; A[j + 3] = a4.w;
        Bv[j] = b4.x; Bv[j + 1] = b4.y; Bv[j + 2] = b4.z; Bv[j + 3] = b4.w;
        Cv[j] = c4.x; Cv[j + 1] = c4.y; Cv[j + 2] = c4.z; Cv[j + 3] = c4.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        st[j] = sp[j]; A[j] = Ap[j]; Bv[j] = Bp[j]; Cv[j] = Cp[j];
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < NPT; ++j) { st[j] = 0.f; A[j] = -1.f; Bv[j] = 0.f; Cv[j] = 0.f; }
  }

  const IO* gu = static_cast<const IO*>(p.u);
  const IO* gd = static_cast<const IO*>(p.delta);
  const IO* gz = static_cast<const IO*>(p.z);
  const float uu = ok ? io_traits<IO>::to_f32(gu[rr]) : 0.f;
  const float x = (ok ? io_traits<IO>::to_f32(gd[rr]) : 0.f) + ((ok && p.bias) ? p.bias[d] : 0.f);
  bool precise = p.force_precise != 0;
#pragma unroll
  for (int j = 0; j < NPT; ++j) precise |= (A[j] == 0.f);
  const float dt = p.softplus ? (precise ? softplus_precise(x) : softplus_fast(x)) : x;

  float acc = 0.f;
  if (!precise) {
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const float a = ex2_fast(dt * (A[j] * kLog2e));
      const float nv = Bv[j] * uu * (-1.f / A[j]);
      st[j] = fmaf(a, st[j] - nv, nv);
      acc = fmaf(Cv[j], st[j], acc);
    }
  } else {
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const float xa = dt * A[j];
      const float coef = A[j] != 0.f ? expm1f(xa) / A[j] : dt;
      st[j] = fmaf(expf(xa), st[j], coef * (Bv[j] * uu));
      acc = fmaf(Cv[j], st[j], acc);
    }
  }
#pragma unroll
  for (int s = G / 2; s >= 1; s /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, s);

  if (!ok) return;
  if constexpr (NPT % 4 == 0) {
#pragma unroll
    for (int j = 0; j < NPT; j += 4)
      *reinterpret_cast<float4*>(sp + j) = make_float4(st[j], st[j + 1], st[j + 2], st[j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < NPT; ++j) sp[j] = st[j];
  }
  if (g == 0) {
    float yv = acc + (p.D ? p.D[d] * uu : 0.f);
    if (gz) {
      const float zz = io_traits<IO>::to_f32(gz[rr]);
      yv *= precise ? silu_precise(zz) : silu_fast(zz);
    }
    static_cast<IO*>(p.y)[rr] = io_traits<IO>::from_f32(yv);
  }
}

template <typename IO, int N>
static cudaError_t upd_typed(const UpdateArgs& a, cudaStream_t stream) {
  constexpr int G = N >= 4 ? 4 : N;
  const int64_t threads = a.batch * a.dim * G;
  const int64_t blocks = (threads + kUpdThreads - 1) / kUpdThreads;
  update_kernel<IO, N><<<(unsigned)blocks, kUpdThreads, 0, stream>>>(a);
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
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t update_launch(const UpdateArgs& a, int64_t N, int io_dtype, cudaStream_t stream) {
  if (a.batch == 0 || a.dim == 0) return cudaSuccess;
  if (io_dtype == 0) return upd_io<float>(a, N, stream);
  return upd_io<__nv_bfloat16>(a, N, stream);
}

}  // namespace ssm
