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

// 16-byte asynchronous copy global -> shared; with `valid` false nothing is read
// and the destination is zero-filled.
__device__ __forceinline__ void cp_async16_zfill_g(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(valid ? 16 : 0)
               : "memory");
}
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

// ---------------------------------------------------------------------------
// The same pass with the rows staged through shared memory, for (batch, dim, L)
// rows of a multiple of 16 bytes.  A unit is 2048 steps of one row (8 a thread);
// its x (with the 8 steps on either side) and dout (with the 8 after) are copied
// by 16-byte cp.async into a ring of kRing stages, kRing - 1 units ahead of the
// one being computed, so that a block keeps several units' loads in flight
// instead of one thread-sized vector, and every thread reads its neighbours'
// halo steps from shared memory rather than from global memory.  The arithmetic
// and the order of every sum are the element-wise kernel's, so both give the
// same bits.  Four stages of bf16 (33 KB) or two of float32 (33 KB) a block, four
// blocks an SM.  (Measured on 8 x 1536 x 2048 bf16: taking the neighbour's g
// through shared memory instead of recomputing it, or packing the tap sums into
// f32x2 pairs, was slower: a barrier, and the moves that build the pairs.)
// ---------------------------------------------------------------------------
constexpr int kRingThreads = 256;  // threads of the staged kernel (8 steps each)
template <typename IO> __host__ __device__ constexpr int ring_stages() { return sizeof(IO) == 2 ? 4 : 2; }

template <typename IO> struct RingStage {
  static constexpr int kChunk = 2048;                             // steps of a unit
  static constexpr int kX = 8 + kChunk + 8;                       // x: 8 before, 8 after
  static constexpr int kG = kChunk + 8;                           // dout: 8 after
  static constexpr int kVecElems = 16 / (int)sizeof(IO);          // elements of a 16-byte copy
  IO x[kX];
  IO g[kG];
};

template <typename IO, int K>
__global__ void __launch_bounds__(kRingThreads, kRingThreads == 256 ? 4 : 5)
    conv1d_bwd_ring_kernel(const ConvBwdArgs p) {
  using St = RingStage<IO>;
  constexpr int NT = kRingThreads, S = St::kChunk / NT, H = K - 1;
  constexpr int kChunk = St::kChunk, VE = St::kVecElems, kRing = ring_stages<IO>();
  __shared__ __align__(16) St ring[kRing];
  const int64_t d = blockIdx.x;
  const int64_t L = p.L;
  const int tid = threadIdx.x;
  const IO* x = static_cast<const IO*>(p.x);
  const IO* dout = static_cast<const IO*>(p.dout);
  IO* dx = static_cast<IO*>(p.dx);
  float w[K];
#pragma unroll
  for (int k = 0; k < K; ++k) w[k] = p.w[d * K + k];
  const float bias = p.bias ? p.bias[d] : 0.f;
  const int nt = (int)((L + kChunk - 1) / kChunk);  // units of a row
  const int units = (int)p.batch * nt;

  // copies of the next unit into its stage: 16-byte pieces [s, s + VE) of the row,
  // zero past the row's ends (rows are whole 16-byte pieces).  (ib, itc) walk the
  // units in order: row ib, unit itc of it.
  int issued = 0, ib = 0, itc = 0;
  auto issue = [&]() {
    if (issued < units) {
      St& stg = ring[issued % kRing];
      const int64_t tc0 = (int64_t)itc * kChunk;
      const int64_t base = ((int64_t)ib * p.dim + d) * L;
      const IO* xr = x + base;
      const IO* gr = dout + base;
      constexpr int kPieces = kChunk / VE, kHalo = 8 / VE;
#pragma unroll
      for (int q0 = 0; q0 < kPieces; q0 += NT) {  // x and dout of the unit
        const int q = q0 + tid;
        const int64_t s = tc0 + q * VE;
        const bool ok = s < L;
        cp_async16_zfill_g(stg.x + 8 + q * VE, xr + (ok ? s : 0), ok);
        cp_async16_zfill_g(stg.g + q * VE, gr + (ok ? s : 0), ok);
      }
      if (tid < 3 * kHalo) {  // x of the 8 steps before and after, dout of the 8 after
        const int r = tid % kHalo, which = tid / kHalo;
        const int64_t s = which == 0 ? tc0 - 8 + r * VE : tc0 + kChunk + r * VE;
        IO* dst = which == 0 ? stg.x + r * VE : (which == 1 ? stg.x + 8 + kChunk + r * VE : stg.g + kChunk + r * VE);
        const bool ok = s >= 0 && s < L;
        cp_async16_zfill_g(dst, (which == 2 ? gr : xr) + (ok ? s : 0), ok);
      }
      ++issued;
      if (++itc == nt) { itc = 0; ++ib; }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");  // (empty past the last unit)
  };

  // g = dout · silu'(p) of one step from its K inputs
  auto gate_grad = [&](float gv, const float* xk) {
    if (!p.silu) return gv;
    float pre = bias;
#pragma unroll
    for (int k = 0; k < K; ++k) pre = fmaf(w[k], xk[k], pre);
    const float sg = p.precise ? 1.f / (1.f + expf(-pre)) : rcp_fast(1.f + ex2_fast(-pre * kLog2e));
    return gv * (sg * fmaf(pre, 1.f - sg, 1.f));
  };

  float dw[K], db = 0.f;
#pragma unroll
  for (int k = 0; k < K; ++k) dw[k] = 0.f;
#pragma unroll
  for (int i = 0; i < kRing - 1; ++i) issue();
  int b = 0, tc = 0;  // the unit being computed
  for (int u = 0; u < units; ++u) {
    asm volatile("cp.async.wait_group %0;" ::"n"(kRing - 2) : "memory");
    __syncthreads();                   // unit u is in; unit u - 1's stage is free
    issue();
    const St& stg = ring[u % kRing];
    const int64_t t0 = (int64_t)tc * kChunk + tid * S;
    const int64_t row = (int64_t)b * p.dim + d;
    const bool act = t0 < L;
    // inputs at positions t0-(K-1) .. t0+S-1+(K-1), cotangents at t0 .. t0+S-1+(K-1)
    float xs[S + 2 * H], gs[S + H];
    {
      float v[S];
      vecio<IO, S>::load(stg.x + 8 + tid * S, v);
#pragma unroll
      for (int i = 0; i < S; ++i) xs[H + i] = v[i];
      vecio<IO, S>::load(stg.g + tid * S, v);
#pragma unroll
      for (int i = 0; i < S; ++i) gs[i] = v[i];
    }
    const IO* st = p.state_in ? static_cast<const IO*>(p.state_in) + row * H : nullptr;
#pragma unroll
    for (int i = 0; i < H; ++i) {
      const int64_t sb = t0 - H + i;  // before: the carried state ahead of the sequence
      xs[i] = sb >= 0 ? io_traits<IO>::to_f32(stg.x[8 + tid * S - H + i])
                      : (st ? io_traits<IO>::to_f32(st[H + sb]) : 0.f);
      xs[H + S + i] = io_traits<IO>::to_f32(stg.x[8 + tid * S + S + i]);
    }
    // g at this thread's steps and the K-1 after them (zero past the end)
#pragma unroll
    for (int i = 0; i < H; ++i) gs[S + i] = io_traits<IO>::to_f32(stg.g[tid * S + S + i]);
#pragma unroll
    for (int j = 0; j < S + H; ++j) gs[j] = gate_grad(gs[j], xs + j);
    if (act) {
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
      const int64_t base = row * L;
      if (t0 + S <= L) {
        vecio<IO, S>::store(dx + base + t0, dxv);
      } else {
#pragma unroll
        for (int i = 0; i < S; ++i)
          if (t0 + i < L) dx[base + t0 + i] = io_traits<IO>::from_f32(dxv[i]);
      }
      // the state's positions -(K-1) .. -1 see g[0 .. K-2]
      if (t0 == 0 && p.dstate) {
#pragma unroll
        for (int j = 0; j < H; ++j) {
          float acc = 0.f;
#pragma unroll
          for (int k = 0; k < K; ++k) {
            const int gi = j - k;
            if (gi >= 0) acc = fmaf(w[k], gs[gi], acc);
          }
          p.dstate[row * H + j] = acc;
        }
      }
    }
    if (++tc == nt) { tc = 0; ++b; }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");

  // the channel's sums: warps by shuffles, then the warps' partials in a fixed order
  __shared__ float red[NT / 32][K + 1];
  float v[K + 1];
#pragma unroll
  for (int k = 0; k < K; ++k) v[k] = dw[k];
  v[K] = db;
#pragma unroll
  for (int k = 0; k <= K; ++k)
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], s);
  const int lane = tid & 31, wid = tid >> 5;
  if (lane == 0)
#pragma unroll
    for (int k = 0; k <= K; ++k) red[wid][k] = v[k];
  __syncthreads();
  if (tid <= K) {
    float sum = 0.f;
    for (int i = 0; i < NT / 32; ++i) sum += red[i][tid];
    if (tid < K) p.dw[d * K + tid] = sum;
    else if (p.dbias) p.dbias[d] = sum;
  }
}

template <typename IO, int K>
static cudaError_t conv_bwd_typed(const ConvBwdArgs& a, cudaStream_t s) {
  if (!a.bld && (a.L * (int64_t)sizeof(IO)) % 16 == 0)
    conv1d_bwd_ring_kernel<IO, K><<<(unsigned)a.dim, kRingThreads, 0, s>>>(a);
  else
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
