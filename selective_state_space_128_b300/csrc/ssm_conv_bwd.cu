// Backward of the scan's front end (causal depthwise conv1d + SiLU) for sm_103a.
//
// Forward (summary page "Mamba: Linear-Time Sequence Modeling", section 4a
// shape table: "Conv1d -> SiLU" ahead of the SSM; configuration page "2. Mamba
// 상세": d_conv = 4), per channel d and width K:
//     p_t = bias + Σ_k w[k] x[t-(K-1)+k],   out_t = silu(p_t)  (or p_t)
// Backward, with g_t = dout_t · silu'(p_t) and silu'(p) = σ(p)(1 + p(1 - σ(p))):
//     dx[s]    = Σ_k w[k] g[s+(K-1)-k]    (the K-1 positions before the
//                                          sequence give d conv_state_in)
//     dw[d,k]  = Σ_{b,t} g[b,d,t] x[b,d,t-(K-1)+k],   dbias[d] = Σ_{b,t} g[b,d,t]
//
// One block per channel, walking every batch row of it.  A thread takes 8
// consecutive steps at a time: it recomputes p and g for its steps and the K-1
// after them (their inputs are L1 hits, loaded by the neighbouring thread too),
// writes dx for its steps and accumulates its share of dw and dbias over all
// rows in registers; the block adds the shares in a fixed order, so the
// results repeat bit for bit and no second pass is needed.  The 16-byte x and
// dout vectors of a thread's next unit are in flight while it works on this one.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

constexpr int kConvBwdThreads = 256;
constexpr int kConvBwdSteps = 8;  // steps per thread
// 64 registers a thread, 4 blocks per SM: the pass is bound by memory latency,
// so resident warps matter more than keeping every temporary in a register
// (on an 8 x 1536 x 2048 bf16 input: 97 us at 120 registers and 2 blocks per SM, 70 us here)

// 8 consecutive elements held as raw 16-byte words until they are used.
template <typename IO> struct RawVec8;
template <> struct RawVec8<__nv_bfloat16> {
  uint4 r;
  __device__ void load(const __nv_bfloat16* p) { r = *reinterpret_cast<const uint4*>(p); }
  __device__ void get(float (&v)[8]) const {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};
template <> struct RawVec8<float> {
  float4 a, b;
  __device__ void load(const float* p) {
    a = reinterpret_cast<const float4*>(p)[0];
    b = reinterpret_cast<const float4*>(p)[1];
  }
  __device__ void get(float (&v)[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

template <typename IO, int K>
__global__ void __launch_bounds__(kConvBwdThreads, 4) conv1d_bwd_kernel(const ConvBwdArgs p) {
  constexpr int S = kConvBwdSteps, H = K - 1;
  const int64_t d = blockIdx.x;  // one channel, every batch row
  const int64_t L = p.L;
  const IO* x = static_cast<const IO*>(p.x);
  const IO* dout = static_cast<const IO*>(p.dout);
  IO* dx = static_cast<IO*>(p.dx);
  float w[K];
#pragma unroll
  for (int k = 0; k < K; ++k) w[k] = p.w[d * K + k];
  const float bias = p.bias ? p.bias[d] : 0.f;
  const bool vec = !p.bld && (L * (int64_t)sizeof(IO)) % 16 == 0;
  const int64_t ts = p.bld ? p.dim : 1;

  float dw[K], db = 0.f;
#pragma unroll
  for (int k = 0; k < K; ++k) dw[k] = 0.f;
  // the (row, step-chunk) units of this channel, in order; a thread's 16-byte
  // vectors of x and dout for the next unit are loaded while it works on this one
  const int64_t chunk = (int64_t)kConvBwdThreads * S;
  const int64_t nt = (L + chunk - 1) / chunk;
  const int64_t units = p.batch * nt;
  auto unit_t0 = [&](int64_t i) { return (i % nt) * chunk + (int64_t)threadIdx.x * S; };
  auto unit_base = [&](int64_t i) {
    const int64_t bb = i / nt;
    return p.bld ? bb * L * p.dim + d : (bb * p.dim + d) * L;
  };
  RawVec8<IO> nx, ng;  // the next unit's vectors
  bool nvec = false;
  auto prefetch = [&](int64_t i) {
    nvec = false;
    if (i < units) {
      const int64_t t0 = unit_t0(i);
      if (vec && t0 + S <= L) {
        const int64_t bs = unit_base(i);
        nx.load(x + bs + t0);
        ng.load(dout + bs + t0);
        nvec = true;
      }
    }
  };
  prefetch(0);
  for (int64_t u = 0; u < units; ++u) {
    const RawVec8<IO> cx = nx, cg = ng;
    const bool cvec = nvec;
    prefetch(u + 1);
    const int64_t b = u / nt, t0 = unit_t0(u);
    if (t0 >= L) continue;
    const int64_t row = b * p.dim + d;
    // element t of the row: base + t * ts (ts = 1, or dim in the (batch, L, dim) layout)
    const int64_t base = unit_base(u);
    const IO* st = p.state_in ? static_cast<const IO*>(p.state_in) + row * H : nullptr;
    // input position s in [-(K-1), L): the carried state before the sequence
    auto xin = [&](int64_t s) -> float {
      if (s < 0) return st ? io_traits<IO>::to_f32(st[H + s]) : 0.f;
      return s < L ? io_traits<IO>::to_f32(x[base + s * ts]) : 0.f;
    };
    {
      // inputs at positions t0-(K-1) .. t0+S-1+(K-1), cotangents at t0 .. t0+S-1+(K-1)
      float xs[S + 2 * H], gs[S + H];
      if (cvec) {  // 16-byte accesses (rows of a multiple of 16 bytes)
        float v[S];
        cx.get(v);
#pragma unroll
        for (int i = 0; i < S; ++i) xs[H + i] = v[i];
        cg.get(v);
#pragma unroll
        for (int i = 0; i < S; ++i) gs[i] = v[i];
      } else {
#pragma unroll
        for (int i = 0; i < S; ++i) {
          xs[H + i] = xin(t0 + i);
          gs[i] = t0 + i < L ? io_traits<IO>::to_f32(dout[base + (t0 + i) * ts]) : 0.f;
        }
      }
#pragma unroll
      for (int i = 0; i < H; ++i) {
        xs[i] = xin(t0 - H + i);
        xs[H + S + i] = xin(t0 + S + i);
        gs[S + i] = t0 + S + i < L ? io_traits<IO>::to_f32(dout[base + (t0 + S + i) * ts]) : 0.f;
      }
      // g = dout · silu'(p) at steps t0 .. t0+S-1+(K-1) (zero past the end)
#pragma unroll
      for (int j = 0; j < S + H; ++j) {
        if (p.silu) {
          float pre = bias;
#pragma unroll
          for (int k = 0; k < K; ++k) pre = fmaf(w[k], xs[j + k], pre);
          const float sg = p.precise ? 1.f / (1.f + expf(-pre))
                                     : rcp_fast(1.f + ex2_fast(-pre * kLog2e));
          gs[j] *= sg * fmaf(pre, 1.f - sg, 1.f);
        }
      }
      // dx for this thread's steps; dw, dbias over them
      float dxv[S];
#pragma unroll
      for (int i = 0; i < S; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) acc = fmaf(w[k], gs[i + H - k], acc);
        dxv[i] = acc;
        db += gs[i];
#pragma unroll
        for (int k = 0; k < K; ++k) dw[k] = fmaf(gs[i], xs[i + k], dw[k]);
      }
      if (cvec) {
        vecio<IO, S>::store(dx + base + t0, dxv);
      } else {
#pragma unroll
        for (int i = 0; i < S; ++i)
          if (t0 + i < L) dx[base + (t0 + i) * ts] = io_traits<IO>::from_f32(dxv[i]);
      }
      // the state's positions -(K-1) .. -1 see g[0 .. K-2]
      if (t0 == 0 && p.dstate) {
#pragma unroll
        for (int j = 0; j < H; ++j) {
          float acc = 0.f;
#pragma unroll
          for (int k = 0; k < K; ++k) {
            const int gi = j - k;  // g index of position j - (K-1) through tap k
            if (gi >= 0) acc = fmaf(w[k], gs[gi], acc);
          }
          p.dstate[row * H + j] = acc;
        }
      }
    }
  }

  // the channel's sums: warps by shuffles, then the warps' partials in a fixed order
  __shared__ float red[kConvBwdThreads / 32][K + 1];
  float v[K + 1];
#pragma unroll
  for (int k = 0; k < K; ++k) v[k] = dw[k];
  v[K] = db;
#pragma unroll
  for (int k = 0; k <= K; ++k)
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], s);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0)
#pragma unroll
    for (int k = 0; k <= K; ++k) red[wid][k] = v[k];
  __syncthreads();
  if (threadIdx.x <= K) {
    float s = 0.f;
    for (int i = 0; i < kConvBwdThreads / 32; ++i) s += red[i][threadIdx.x];
    if (threadIdx.x < K) p.dw[d * K + threadIdx.x] = s;
    else if (p.dbias) p.dbias[d] = s;
  }
}

template <typename IO, int K>
static cudaError_t conv_bwd_typed(const ConvBwdArgs& a, cudaStream_t s) {
  conv1d_bwd_kernel<IO, K><<<(unsigned)a.dim, kConvBwdThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename IO>
static cudaError_t conv_bwd_io(const ConvBwdArgs& a, int64_t K, cudaStream_t s) {
  switch (K) {
    case 1: return conv_bwd_typed<IO, 1>(a, s);
    case 2: return conv_bwd_typed<IO, 2>(a, s);
    case 3: return conv_bwd_typed<IO, 3>(a, s);
    case 4: return conv_bwd_typed<IO, 4>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t conv_bwd_launch(const ConvBwdArgs& a, int64_t width, int io_dtype, cudaStream_t stream) {
  return io_dtype == 0 ? conv_bwd_io<float>(a, width, stream)
                       : conv_bwd_io<__nv_bfloat16>(a, width, stream);
}

}  // namespace ssm
