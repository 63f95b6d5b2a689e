// Front end of the scan for sm_103a: causal depthwise conv1d + SiLU, and its
// one-token form on a rolling state.
//
// The summary page ("Mamba: Linear-Time Sequence Modeling", section 4a shape
// table) puts "Conv1d -> SiLU" on the (B, L, ED) path right before the SSM;
// the configuration page ("2. Mamba 상세") gives the kernel width d_conv = 4.
// Per channel d and width K:
//     out[t] = silu(bias[d] + Σ_k w[d,k] x[t-(K-1)+k]),
// x[t < 0] taken from a carried state of the K-1 previous inputs (zeros when
// absent); the new state is the last K-1 inputs.
//
// The pass moves 2 bytes in and 2 out per element (bf16) for K multiply-adds
// and one exponential: HBM-bound.  A thread produces one 16-byte vector of
// outputs from its own input vector and the tail of the previous one (an L1
// hit: the neighbouring thread loads it too), so every DRAM byte is read once
// and every access is a full 16-byte vector.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

template <typename IO> struct Vec16;
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) { vecio<__nv_bfloat16, 8>::load(p, v); }
  __device__ static void store(__nv_bfloat16* p, const float (&v)[8]) { vecio<__nv_bfloat16, 8>::store(p, v); }
};
template <> struct Vec16<float> {
  static constexpr int n = 4;
  __device__ static void load(const float* p, float (&v)[4]) { vecio<float, 4>::load(p, v); }
  __device__ static void store(float* p, const float (&v)[4]) { vecio<float, 4>::store(p, v); }
};

__device__ __forceinline__ float conv_act(float v, bool silu, bool precise) {
  return silu ? (precise ? silu_precise(v) : silu_fast(v)) : v;
}

// Rows whose length is a multiple of one 16-byte vector.
template <typename IO, int K>
__global__ void __launch_bounds__(256) conv1d_vec_kernel(const ConvArgs p) {
  constexpr int VE = Vec16<IO>::n;
  const int64_t nv = p.L / VE;  // vectors per row
  const int64_t total = p.batch * p.dim * nv;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total;
       v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = v / nv, j = v - row * nv;
    const int64_t d = row % p.dim;
    const IO* xr = static_cast<const IO*>(p.x) + row * p.L;
    float cur[VE], xe[K - 1 + VE];
    Vec16<IO>::load(xr + j * VE, cur);
    if constexpr (K > 1) {
      if (j > 0) {
        float prev[VE];
        Vec16<IO>::load(xr + (j - 1) * VE, prev);
#pragma unroll
        for (int k = 0; k < K - 1; ++k) xe[k] = prev[VE - (K - 1) + k];
      } else {
        const IO* st = p.state_in ? static_cast<const IO*>(p.state_in) + row * (K - 1) : nullptr;
#pragma unroll
        for (int k = 0; k < K - 1; ++k) xe[k] = st ? io_traits<IO>::to_f32(st[k]) : 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < VE; ++i) xe[K - 1 + i] = cur[i];
    float w[K];
#pragma unroll
    for (int k = 0; k < K; ++k) w[k] = __ldg(p.w + d * K + k);
    const float bias = p.bias ? __ldg(p.bias + d) : 0.f;
    float o[VE];
#pragma unroll
    for (int i = 0; i < VE; ++i) {
      float acc = bias;
#pragma unroll
      for (int k = 0; k < K; ++k) acc = fmaf(w[k], xe[i + k], acc);
      o[i] = conv_act(acc, p.silu, p.precise);
    }
    Vec16<IO>::store(static_cast<IO*>(p.out) + row * p.L + j * VE, o);
  }
}

// Rows whose length is a multiple of VPT vectors: a thread produces VPT
// consecutive vectors with every load issued first; the K-1 inputs before its
// first vector come from the neighbouring lane's last vector by shuffles (lane
// 0 loads them).  One thread per VPT vectors, no grid-stride loop, so every
// lane of a warp reaches the shuffles.  VPT = 2 at 8 blocks of 256 threads
// per SM measured best (23 us for 8 x 1536 x 2048 bf16; 4 vectors: 28 us,
// 1 vector: 28 us, a plain 100 MB device copy: 18.6 us).
template <typename IO, int K, int VPT>
__global__ void __launch_bounds__(256, 8) conv1d_wide_kernel(const ConvArgs p) {
  constexpr int VE = Vec16<IO>::n;
  constexpr int TE = VPT * VE;  // elements per thread
  const int64_t nb = p.L / TE;  // threads per row
  const int64_t total = p.batch * p.dim * nb;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool active = gid < total;
  const int64_t id = active ? gid : total - 1;
  const int64_t row = id / nb, jb = id - row * nb;
  const int64_t d = row % p.dim;
  const IO* xr = static_cast<const IO*>(p.x) + row * p.L + jb * TE;
  float xe[K - 1 + TE];
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    float cur[VE];
    Vec16<IO>::load(xr + v * VE, cur);
#pragma unroll
    for (int i = 0; i < VE; ++i) xe[K - 1 + v * VE + i] = cur[i];
  }
  if constexpr (K > 1) {
    const int lane = threadIdx.x & 31;
    float tail[K - 1];
#pragma unroll
    for (int k = 0; k < K - 1; ++k)
      tail[k] = __shfl_up_sync(0xffffffffu, xe[K - 1 + TE - (K - 1) + k], 1);
    if (jb == 0) {
      const IO* st = p.state_in ? static_cast<const IO*>(p.state_in) + row * (K - 1) : nullptr;
#pragma unroll
      for (int k = 0; k < K - 1; ++k) tail[k] = st ? io_traits<IO>::to_f32(st[k]) : 0.f;
    } else if (lane == 0) {
#pragma unroll
      for (int k = 0; k < K - 1; ++k) tail[k] = io_traits<IO>::to_f32(xr[k - (K - 1)]);
    }
#pragma unroll
    for (int k = 0; k < K - 1; ++k) xe[k] = tail[k];
  }
  float w[K];
#pragma unroll
  for (int k = 0; k < K; ++k) w[k] = __ldg(p.w + d * K + k);
  const float bias = p.bias ? __ldg(p.bias + d) : 0.f;
  if (!active) return;
  IO* orow = static_cast<IO*>(p.out) + row * p.L + jb * TE;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    float o[VE];
#pragma unroll
    for (int i = 0; i < VE; ++i) {
      float acc = bias;
#pragma unroll
      for (int k = 0; k < K; ++k) acc = fmaf(w[k], xe[v * VE + i + k], acc);
      o[i] = conv_act(acc, p.silu, p.precise);
    }
    Vec16<IO>::store(orow + v * VE, o);
  }
}

// (batch, L, dim) layout, dim a multiple of one 16-byte vector: a thread
// produces VE consecutive channels of one step from the K input vectors of
// steps t-K+1..t (rows of neighbouring threads overlap: L1 hits).
template <typename IO, int K>
__global__ void __launch_bounds__(256) conv1d_bld_vec_kernel(const ConvArgs p) {
  constexpr int VE = Vec16<IO>::n;
  const int64_t nv = p.dim / VE;  // vectors per step
  const int64_t total = p.batch * p.L * nv;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total;
       v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t bt = v / nv, j = v - bt * nv;
    const int64_t b = bt / p.L, t = bt - b * p.L;
    const int64_t d0 = j * VE;
    float acc[VE];
#pragma unroll
    for (int i = 0; i < VE; ++i) acc[i] = p.bias ? __ldg(p.bias + d0 + i) : 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int64_t s = t - (K - 1) + k;
      float xv[VE];
      if (s >= 0) {
        Vec16<IO>::load(static_cast<const IO*>(p.x) + (b * p.L + s) * p.dim + d0, xv);
      } else {
        const IO* st = static_cast<const IO*>(p.state_in);
#pragma unroll
        for (int i = 0; i < VE; ++i)
          xv[i] = st ? io_traits<IO>::to_f32(st[((b * p.dim) + d0 + i) * (K - 1) + (K - 1 + s)]) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < VE; ++i) acc[i] = fmaf(__ldg(p.w + (d0 + i) * K + k), xv[i], acc[i]);
    }
#pragma unroll
    for (int i = 0; i < VE; ++i) acc[i] = conv_act(acc[i], p.silu, p.precise);
    Vec16<IO>::store(static_cast<IO*>(p.out) + (b * p.L + t) * p.dim + d0, acc);
  }
}

// (batch, L, dim) layout, any dim: one output per thread.
template <typename IO, int K>
__global__ void __launch_bounds__(256) conv1d_bld_scalar_kernel(const ConvArgs p) {
  const int64_t total = p.batch * p.dim * p.L;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t bt = e / p.dim, d = e - bt * p.dim;
    const int64_t b = bt / p.L, t = bt - b * p.L;
    const IO* st = p.state_in ? static_cast<const IO*>(p.state_in) + (b * p.dim + d) * (K - 1)
                              : nullptr;
    float acc = p.bias ? __ldg(p.bias + d) : 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int64_t s = t - (K - 1) + k;
      const float xv = s >= 0 ? io_traits<IO>::to_f32(static_cast<const IO*>(p.x)[(b * p.L + s) * p.dim + d])
                              : (st ? io_traits<IO>::to_f32(st[K - 1 + s]) : 0.f);
      acc = fmaf(__ldg(p.w + d * K + k), xv, acc);
    }
    static_cast<IO*>(p.out)[e] = io_traits<IO>::from_f32(conv_act(acc, p.silu, p.precise));
  }
}

// Any row length: one output per thread.
template <typename IO, int K>
__global__ void __launch_bounds__(256) conv1d_scalar_kernel(const ConvArgs p) {
  const int64_t total = p.batch * p.dim * p.L;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = e / p.L, t = e - row * p.L;
    const int64_t d = row % p.dim;
    const IO* xr = static_cast<const IO*>(p.x) + row * p.L;
    const IO* st = p.state_in ? static_cast<const IO*>(p.state_in) + row * (K - 1) : nullptr;
    float acc = p.bias ? __ldg(p.bias + d) : 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int64_t s = t - (K - 1) + k;
      const float xv = s >= 0 ? io_traits<IO>::to_f32(xr[s])
                              : (st ? io_traits<IO>::to_f32(st[K - 1 + s]) : 0.f);
      acc = fmaf(__ldg(p.w + d * K + k), xv, acc);
    }
    static_cast<IO*>(p.out)[e] = io_traits<IO>::from_f32(conv_act(acc, p.silu, p.precise));
  }
}

// The new state: the last K-1 inputs of (state_in, x).  One thread per row; it
// reads every value before writing, so state_out may be state_in.
template <typename IO, int K>
__global__ void conv1d_state_kernel(const ConvArgs p) {
  const int64_t rows = p.batch * p.dim;
  for (int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; row < rows;
       row += (int64_t)gridDim.x * blockDim.x) {
    // input step s of this row: row * L + s, or (b * L + s) * dim + d in (batch, L, dim)
    const int64_t b = row / p.dim, d = row - b * p.dim;
    const IO* x = static_cast<const IO*>(p.x);
    const IO* st = p.state_in ? static_cast<const IO*>(p.state_in) + row * (K - 1) : nullptr;
    IO v[K > 1 ? K - 1 : 1];
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
      const int64_t s = p.L - (K - 1) + j;
      const int64_t xi = p.bld ? (b * p.L + s) * p.dim + d : row * p.L + s;
      v[j] = s >= 0 ? x[xi] : (st ? st[K - 1 + s] : io_traits<IO>::from_f32(0.f));
    }
    IO* so = static_cast<IO*>(p.state_out) + row * (K - 1);
#pragma unroll
    for (int j = 0; j < K - 1; ++j) so[j] = v[j];
  }
}

// One token per (batch, channel) on the rolling state, in place.
template <typename IO, int K>
__global__ void __launch_bounds__(256) conv1d_update_kernel(const ConvArgs p) {
  const int64_t rows = p.batch * p.dim;
  for (int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; row < rows;
       row += (int64_t)gridDim.x * blockDim.x) {
    const int64_t d = row % p.dim;
    IO* st = static_cast<IO*>(p.state_out) + row * (K - 1);
    float win[K];
#pragma unroll
    for (int k = 0; k < K - 1; ++k) win[k] = io_traits<IO>::to_f32(st[k]);
    const IO xin = static_cast<const IO*>(p.x)[row];
    win[K - 1] = io_traits<IO>::to_f32(xin);
    float acc = p.bias ? __ldg(p.bias + d) : 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) acc = fmaf(__ldg(p.w + d * K + k), win[k], acc);
    static_cast<IO*>(p.out)[row] = io_traits<IO>::from_f32(conv_act(acc, p.silu, p.precise));
#pragma unroll
    for (int k = 0; k + 1 < K - 1; ++k) st[k] = st[k + 1];
    if constexpr (K > 1) st[K - 2] = xin;
  }
}

static unsigned grid_for(int64_t work, int per_block) {
  const int64_t blocks = (work + per_block - 1) / per_block;
  const int64_t cap = 148 * 16;  // grid-stride beyond 16 blocks per SM
  return (unsigned)(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

template <typename IO, int K>
static cudaError_t conv_typed(const ConvArgs& a, bool update, cudaStream_t s) {
  if (update) {
    conv1d_update_kernel<IO, K><<<grid_for(a.batch * a.dim, 256), 256, 0, s>>>(a);
    return cudaGetLastError();
  }
  constexpr int VE = Vec16<IO>::n;
  const int64_t rows = a.batch * a.dim;
  if (a.L > 0 && a.bld) {
    if (a.dim % VE == 0)
      conv1d_bld_vec_kernel<IO, K><<<grid_for(a.batch * a.L * (a.dim / VE), 256), 256, 0, s>>>(a);
    else
      conv1d_bld_scalar_kernel<IO, K><<<grid_for(rows * a.L, 256), 256, 0, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  } else if (a.L > 0) {
    constexpr int VPT = 2;
    if (a.L % (VE * VPT) == 0) {
      const int64_t threads = rows * (a.L / (VE * VPT));
      conv1d_wide_kernel<IO, K, VPT><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(a);
    } else if (a.L % VE == 0)
      conv1d_vec_kernel<IO, K><<<grid_for(rows * (a.L / VE), 256), 256, 0, s>>>(a);
    else
      conv1d_scalar_kernel<IO, K><<<grid_for(rows * a.L, 256), 256, 0, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (K > 1 && a.state_out) {
    conv1d_state_kernel<IO, K><<<grid_for(rows, 256), 256, 0, s>>>(a);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

template <typename IO>
static cudaError_t conv_io(const ConvArgs& a, int64_t K, bool update, cudaStream_t s) {
  switch (K) {
    case 1: return conv_typed<IO, 1>(a, update, s);
    case 2: return conv_typed<IO, 2>(a, update, s);
    case 3: return conv_typed<IO, 3>(a, update, s);
    case 4: return conv_typed<IO, 4>(a, update, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t conv_launch(const ConvArgs& a, int64_t width, int io_dtype, bool update,
                        cudaStream_t stream) {
  if (a.batch == 0 || a.dim == 0) return cudaSuccess;
  if (io_dtype == 0) return conv_io<float>(a, width, update, stream);
  return conv_io<__nv_bfloat16>(a, width, update, stream);
}

}  // namespace ssm
