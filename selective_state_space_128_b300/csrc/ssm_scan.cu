// Selective-scan forward kernel (S6) for sm_103a.
//
// Computes, per (batch b, channel d): Δ_t = softplus(delta + bias), the
// zero-order-hold pair Ā = exp(Δ A), B̄ = (exp(Δ A) - 1)/A · B_t, the recurrence
// h_t = Ā h_{t-1} + B̄ u_t and the readout y_t = (C_t · h_t + D u_t) · silu(z_t)
// ("Mamba: Linear-Time Sequence Modeling" summary page: section 4b equations
// (2), (4) and Algorithm 2; section 4a shape table for the gate; the SSM/Mamba
// chapter's section 3.1 for D).
//
// Design (B300): a block owns CH channels of one batch row and walks the
// sequence in chunks of T steps.  Chunk tiles of u/Δ/z (bf16 or fp32) and of
// B/C (fp32, shared by all channels of the block) are staged into shared
// memory with cp.async (double-buffered), then a cooperative "prep" pass turns
// them into fp32 tiles of Δ (softplus applied once per element), u and the
// gate silu(z), and transposes B/C to [t][n].  Each channel is handled by G
// lanes holding NPT = N/G states each in registers; the state is carried in
// fp32 registers across chunks and the expanded (L, N) state never leaves the
// SM.  Per step and state the fast path costs one MUFU ex2 and six FP32
// operations issued as packed f32x2 pairs; the G partial readouts of a channel
// are combined by a shuffle reduce-scatter so that each lane finishes one time
// step of the block (D term, gate, bf16 rounding), staged to shared memory and
// written back with 16-byte stores.
//
// Long sequences with few channels are split into segments (grid.z): pass 1
// computes each segment's end state from zero and its ΣΔ, pass 0 folds the
// carries of earlier segments (h <- exp(A ΣΔ_k) h + h_k) into its initial state
// and recomputes its segment with outputs.  There is no inter-block waiting.
#include <cuda_pipeline_primitives.h>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

// Per-N tiling: NPT states per lane, G lanes per channel, CH channels per
// block, T steps per chunk.
template <int N> struct ScanCfg {
  static constexpr int NPT = N <= 4 ? N : (N <= 16 ? 4 : N / 4);
  static constexpr int G = N / NPT;
  static constexpr int CH = kScanThreads / G;
  static constexpr int T = (2048 / CH) < 64 ? (2048 / CH) : 64;
  static_assert(G * NPT == N, "tiling");
  static_assert(T % G == 0 && T % 8 == 0, "chunk");
};

constexpr int kPadF = 4;  // fp32 tile row padding (floats)

template <typename IO, int N> struct ScanSmem {
  using Cf = ScanCfg<N>;
  static constexpr int CH = Cf::CH, T = Cf::T;
  static constexpr int RowF = T + kPadF;            // fp32 tile row stride
  static constexpr int RowY = T + 16 / sizeof(IO);  // y tile row stride (elements)
  static constexpr int RowBC = N + 4;               // transposed B/C row stride
  // raw stage (one of two)
  static constexpr size_t kRawIO = (size_t)CH * T * sizeof(IO);
  static constexpr size_t kRawBC = (size_t)N * T * sizeof(float);
  static constexpr size_t kStage = 3 * kRawIO + 2 * kRawBC;
  static constexpr size_t oStage0 = 0;
  static constexpr size_t oStage1 = kStage;
  static constexpr size_t oDt = 2 * kStage;
  static constexpr size_t oU = oDt + (size_t)CH * RowF * 4;
  static constexpr size_t oG = oU + (size_t)CH * RowF * 4;
  static constexpr size_t oB = oG + (size_t)CH * RowF * 4;
  static constexpr size_t oC = oB + (size_t)T * RowBC * 4;
  static constexpr size_t oY = oC + (size_t)T * RowBC * 4;
  static constexpr size_t oBias = oY + (((size_t)CH * RowY * sizeof(IO) + 15) / 16) * 16;
  static constexpr size_t kBytes = oBias + (size_t)CH * 4;
  static_assert(kStage % 16 == 0 && kRawIO % 16 == 0 && kRawBC % 16 == 0, "align");
};

// ---------------------------------------------------------------------------
// Chunk staging
// ---------------------------------------------------------------------------
template <typename IO, int N>
__device__ __forceinline__ void stage_chunk(const ScanArgs& p, unsigned char* stage, int64_t b,
                                            int64_t d0, int64_t t0, int tcount) {
  using S = ScanSmem<IO, N>;
  constexpr int CH = S::CH, T = S::T;
  constexpr int VEC = 16 / sizeof(IO);
  const int tid = threadIdx.x;
  IO* su = reinterpret_cast<IO*>(stage);
  IO* sd = su + CH * T;
  IO* sz = sd + CH * T;
  float* sB = reinterpret_cast<float*>(stage + 3 * S::kRawIO);
  float* sC = sB + N * T;
  const IO* gu = static_cast<const IO*>(p.u);
  const IO* gd = static_cast<const IO*>(p.delta);
  const IO* gz = static_cast<const IO*>(p.z);
  const int nrows = (int)min64(CH, p.dim - d0);
  const int narr = gz ? 3 : 2;
  if (p.vec_io) {
    // tcount is a multiple of VEC here (L and segment starts are)
    const int pieces = tcount / VEC;
    const int per_arr = nrows * pieces;
    for (int i = tid; i < narr * per_arr; i += kScanThreads) {
      const int arr = i / per_arr, rem = i - arr * per_arr;
      const int r = rem / pieces, k = rem - r * pieces;
      const IO* src = arr == 0 ? gu : (arr == 1 ? gd : gz);
      IO* dst = arr == 0 ? su : (arr == 1 ? sd : sz);
      const int64_t off = ((b * p.dim + d0 + r) * p.L + t0) + (int64_t)k * VEC;
      __pipeline_memcpy_async(dst + r * T + k * VEC, src + off, 16);
    }
  } else {
    const int per_arr = nrows * tcount;
    for (int i = tid; i < narr * per_arr; i += kScanThreads) {
      const int arr = i / per_arr, rem = i - arr * per_arr;
      const int r = rem / tcount, k = rem - r * tcount;
      const IO* src = arr == 0 ? gu : (arr == 1 ? gd : gz);
      IO* dst = arr == 0 ? su : (arr == 1 ? sd : sz);
      dst[r * T + k] = src[(b * p.dim + d0 + r) * p.L + t0 + k];
    }
  }
  if (p.vec_bc) {
    const int pieces = tcount / 4;
    const int per_arr = N * pieces;
    for (int i = tid; i < 2 * per_arr; i += kScanThreads) {
      const int arr = i / per_arr, rem = i - arr * per_arr;
      const int n = rem / pieces, k = rem - n * pieces;
      const float* src = arr == 0 ? p.B : p.C;
      float* dst = arr == 0 ? sB : sC;
      __pipeline_memcpy_async(dst + n * T + k * 4, src + (b * N + n) * p.L + t0 + k * 4, 16);
    }
  } else {
    const int per_arr = N * tcount;
    for (int i = tid; i < 2 * per_arr; i += kScanThreads) {
      const int arr = i / per_arr, rem = i - arr * per_arr;
      const int n = rem / tcount, k = rem - n * tcount;
      const float* src = arr == 0 ? p.B : p.C;
      float* dst = arr == 0 ? sB : sC;
      dst[n * T + k] = src[(b * N + n) * p.L + t0 + k];
    }
  }
}

// Turn a raw stage into the fp32 working tiles.  Steps past tcount and rows past
// dim get Δ = 0 and u = 0, which makes them exact no-ops of the recurrence
// (Ā = 1, B̄ u = 0).
template <typename IO, int N, int PASS>
__device__ __forceinline__ void prep_chunk(const ScanArgs& p, const unsigned char* stage,
                                           unsigned char* smem, int64_t d0, int tcount,
                                           bool precise) {
  using S = ScanSmem<IO, N>;
  constexpr int CH = S::CH, T = S::T;
  const int tid = threadIdx.x;
  const IO* su = reinterpret_cast<const IO*>(stage);
  const IO* sd = su + CH * T;
  const IO* sz = sd + CH * T;
  const float* sB = reinterpret_cast<const float*>(stage + 3 * S::kRawIO);
  const float* sC = sB + N * T;
  float* pDt = reinterpret_cast<float*>(smem + S::oDt);
  float* pU = reinterpret_cast<float*>(smem + S::oU);
  float* pG = reinterpret_cast<float*>(smem + S::oG);
  float* pB = reinterpret_cast<float*>(smem + S::oB);
  float* pC = reinterpret_cast<float*>(smem + S::oC);
  const float* sBias = reinterpret_cast<const float*>(smem + S::oBias);
  const int nrows = (int)min64(CH, p.dim - d0);
  const bool has_z = p.z != nullptr;
  for (int e = tid; e < CH * T; e += kScanThreads) {
    const int r = e / T, t = e - r * T;
    const bool ok = r < nrows && t < tcount;
    float dt = 0.f, uu = 0.f, gate = 1.f;
    if (ok) {
      const float x = io_traits<IO>::to_f32(sd[e]) + sBias[r];
      dt = p.softplus ? (precise ? softplus_precise(x) : softplus_fast(x)) : x;
      uu = io_traits<IO>::to_f32(su[e]);
      if (PASS == 0 && has_z) {
        const float zz = io_traits<IO>::to_f32(sz[e]);
        gate = precise ? silu_precise(zz) : silu_fast(zz);
      }
    }
    pDt[r * S::RowF + t] = dt;
    pU[r * S::RowF + t] = uu;
    if (PASS == 0) pG[r * S::RowF + t] = gate;
  }
  for (int e = tid; e < N * T; e += kScanThreads) {
    const int t = e % T, n = e / T;
    const bool ok = t < tcount;
    pB[t * S::RowBC + n] = ok ? sB[n * T + t] : 0.f;
    if (PASS == 0) pC[t * S::RowBC + n] = ok ? sC[n * T + t] : 0.f;
  }
}

// Combine the G partial readouts of a channel: afterwards lane g holds the full
// sum for time step g of the block (shuffle reduce-scatter, log2(G) stages).
template <int G>
__device__ __forceinline__ float reduce_scatter(float (&part)[G], int g) {
#pragma unroll
  for (int s = G / 2; s >= 1; s /= 2) {
    const bool upper = (g & s) != 0;
#pragma unroll
    for (int k = 0; k < s; ++k) {
      const float send = upper ? part[k] : part[k + s];
      const float keep = upper ? part[k + s] : part[k];
      part[k] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return part[0];
}

// ---------------------------------------------------------------------------
// The kernel.  PASS 0: outputs (y, final state).  PASS 1: segment end state
// from a zero start and ΣΔ, for the split plan.
// ---------------------------------------------------------------------------
template <typename IO, int N, int PASS>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(const ScanArgs p) {
  using Cf = ScanCfg<N>;
  using S = ScanSmem<IO, N>;
  constexpr int NPT = Cf::NPT, G = Cf::G, CH = Cf::CH, T = Cf::T;
  constexpr int NP = NPT / 2;  // packed pairs per lane (0 when NPT == 1)
  extern __shared__ __align__(16) unsigned char smem[];

  const int tid = threadIdx.x;
  const int c = tid / G, g = tid - (tid / G) * G;
  const int64_t b = blockIdx.y;
  const int64_t d0 = (int64_t)blockIdx.x * CH;
  const int64_t d = d0 + c;
  const bool chan_ok = d < p.dim;
  const int seg = blockIdx.z;
  const int64_t t_begin = (int64_t)seg * p.seg_len;
  const int64_t t_end = min(p.L, t_begin + p.seg_len);
  const int64_t nchunks = (t_end - t_begin + T - 1) / T;

  // per-row bias into shared memory
  float* sBias = reinterpret_cast<float*>(smem + S::oBias);
  for (int r = tid; r < CH; r += kScanThreads)
    sBias[r] = (p.bias && d0 + r < p.dim) ? p.bias[d0 + r] : 0.f;

  // this lane's states: n = g*NPT + j
  float Aj[NPT];
  bool zeroA = false;
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    Aj[j] = chan_ok ? p.A[d * N + g * NPT + j] : -1.f;
    zeroA |= (Aj[j] == 0.f);
  }
  const bool precise = __syncthreads_or(zeroA) || p.force_precise;

  float h[NPT];
#pragma unroll
  for (int j = 0; j < NPT; ++j) h[j] = 0.f;
  if (PASS == 0 && chan_ok) {
    const int64_t row = b * p.dim + d;
    if (p.init_state) {
#pragma unroll
      for (int j = 0; j < NPT; ++j) h[j] = p.init_state[row * N + g * NPT + j];
    }
    for (int k = 0; k < seg; ++k) {
      const float sk = p.carry_s[(int64_t)k * p.batch * p.dim + row];
      const float* hk = p.carry_h + ((int64_t)k * p.batch * p.dim + row) * N + g * NPT;
#pragma unroll
      for (int j = 0; j < NPT; ++j) h[j] = fmaf(expf(sk * Aj[j]), h[j], hk[j]);
    }
  }
  const float Dd = (PASS == 0 && chan_ok && p.D) ? p.D[d] : 0.f;

  // fast-path constants
  f2 A2p[NP > 0 ? NP : 1], nIp[NP > 0 ? NP : 1], hp[NP > 0 ? NP : 1];
  float A2s = 0.f, nIs = 0.f;
  if constexpr (NPT == 1) {
    A2s = Aj[0] * kLog2e;
    nIs = -1.f / Aj[0];
  } else {
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      A2p[q] = pack2(Aj[2 * q] * kLog2e, Aj[2 * q + 1] * kLog2e);
      nIp[q] = pack2(-1.f / Aj[2 * q], -1.f / Aj[2 * q + 1]);
    }
  }
  float invA[NPT];
#pragma unroll
  for (int j = 0; j < NPT; ++j) invA[j] = Aj[j] != 0.f ? 1.f / Aj[j] : 0.f;

  float sumDt = 0.f;

  unsigned char* stages[2] = {smem + S::oStage0, smem + S::oStage1};
  // prologue: chunks 0 and 1 in flight
  for (int k = 0; k < 2; ++k) {
    if (k < nchunks) {
      const int64_t t0 = t_begin + (int64_t)k * T;
      stage_chunk<IO, N>(p, stages[k], b, d0, t0, (int)min64(T, t_end - t0));
    }
    __pipeline_commit();
  }

  const float* pDt = reinterpret_cast<const float*>(smem + S::oDt) + c * S::RowF;
  const float* pU = reinterpret_cast<const float*>(smem + S::oU) + c * S::RowF;
  const float* pG = reinterpret_cast<const float*>(smem + S::oG) + c * S::RowF;
  const float* pB = reinterpret_cast<const float*>(smem + S::oB) + g * NPT;
  const float* pC = reinterpret_cast<const float*>(smem + S::oC) + g * NPT;
  IO* yT = reinterpret_cast<IO*>(smem + S::oY);

  for (int64_t i = 0; i < nchunks; ++i) {
    const int64_t t0 = t_begin + i * T;
    const int tcount = (int)min64(T, t_end - t0);
    __pipeline_wait_prior(1);
    __syncthreads();
    prep_chunk<IO, N, PASS>(p, stages[i & 1], smem, d0, tcount, precise);
    __syncthreads();
    // the raw stage is consumed: refill it with chunk i + 2
    if (i + 2 < nchunks) {
      const int64_t t2 = t_begin + (i + 2) * T;
      stage_chunk<IO, N>(p, stages[i & 1], b, d0, t2, (int)min64(T, t_end - t2));
    }
    __pipeline_commit();

    const int tround = ((tcount + G - 1) / G) * G;
    if (!precise) {
      if constexpr (NPT > 1) {
#pragma unroll
        for (int q = 0; q < NP; ++q) hp[q] = pack2(h[2 * q], h[2 * q + 1]);
      }
      for (int tb = 0; tb < tround; tb += G) {
        float part[G];
#pragma unroll
        for (int k = 0; k < G; ++k) {
          const int t = tb + k;
          const float dt = pDt[t];
          const float ut = pU[t];
          if (PASS == 1) sumDt += dt;
          if constexpr (NPT == 1) {
            const float a = ex2_fast(dt * A2s);
            const float nv = pB[t * S::RowBC] * ut * nIs;
            h[0] = fmaf(a, h[0] - nv, nv);
            part[k] = PASS == 0 ? pC[t * S::RowBC] * h[0] : 0.f;
          } else {
            const f2 dt2 = pack2(dt, dt);
            const f2 u2 = pack2(ut, ut);
            f2 acc2 = pack2(0.f, 0.f);
            const float* brow = pB + t * S::RowBC;
            const float* crow = pC + t * S::RowBC;
#pragma unroll
            for (int q = 0; q < NP; ++q) {
              const float2 bq = *reinterpret_cast<const float2*>(brow + 2 * q);
              const f2 x = mul2(dt2, A2p[q]);
              float x0, x1;
              unpack2(x, x0, x1);
              const f2 a = pack2(ex2_fast(x0), ex2_fast(x1));
              const f2 nv = mul2(mul2(pack2(bq.x, bq.y), u2), nIp[q]);
              hp[q] = fma2(a, sub2(hp[q], nv), nv);
              if (PASS == 0) {
                const float2 cq = *reinterpret_cast<const float2*>(crow + 2 * q);
                acc2 = fma2(pack2(cq.x, cq.y), hp[q], acc2);
              }
            }
            float lo, hi;
            unpack2(acc2, lo, hi);
            part[k] = lo + hi;
          }
        }
        if (PASS == 0) {
          const float yv = reduce_scatter<G>(part, g);
          const int t = tb + g;
          yT[c * S::RowY + t] = io_traits<IO>::from_f32(fmaf(Dd, pU[t], yv) * pG[t]);
        }
      }
      if constexpr (NPT > 1) {
#pragma unroll
        for (int q = 0; q < NP; ++q) unpack2(hp[q], h[2 * q], h[2 * q + 1]);
      }
    } else {
      for (int tb = 0; tb < tround; tb += G) {
        float part[G];
#pragma unroll
        for (int k = 0; k < G; ++k) {
          const int t = tb + k;
          const float dt = pDt[t];
          const float bu = pU[t];
          if (PASS == 1) sumDt += dt;
          float acc = 0.f;
#pragma unroll
          for (int j = 0; j < NPT; ++j) {
            const float x = dt * Aj[j];
            const float a = expf(x);
            const float coef = Aj[j] != 0.f ? expm1f(x) * invA[j] : dt;
            h[j] = fmaf(a, h[j], coef * (pB[t * S::RowBC + j] * bu));
            if (PASS == 0) acc = fmaf(pC[t * S::RowBC + j], h[j], acc);
          }
          part[k] = acc;
        }
        if (PASS == 0) {
          const float yv = reduce_scatter<G>(part, g);
          const int t = tb + g;
          yT[c * S::RowY + t] = io_traits<IO>::from_f32(fmaf(Dd, pU[t], yv) * pG[t]);
        }
      }
    }
    if (PASS == 0) {
      __syncthreads();
      // write the y tile back
      IO* gy = static_cast<IO*>(p.y);
      const int nrows = (int)min64(CH, p.dim - d0);
      constexpr int VEC = 16 / sizeof(IO);
      if (p.vec_io) {
        const int pieces = tcount / VEC;
        for (int e = tid; e < nrows * pieces; e += kScanThreads) {
          const int r = e / pieces, k = e - r * pieces;
          const uint4 v = *reinterpret_cast<const uint4*>(yT + r * S::RowY + k * VEC);
          *reinterpret_cast<uint4*>(gy + (b * p.dim + d0 + r) * p.L + t0 + k * VEC) = v;
        }
      } else {
        for (int e = tid; e < nrows * tcount; e += kScanThreads) {
          const int r = e / tcount, k = e - r * tcount;
          gy[(b * p.dim + d0 + r) * p.L + t0 + k] = yT[r * S::RowY + k];
        }
      }
    }
  }

  if (!chan_ok) return;
  const int64_t row = b * p.dim + d;
  if (PASS == 0) {
    if (p.final_state && seg == p.nseg - 1) {
#pragma unroll
      for (int j = 0; j < NPT; ++j) p.final_state[row * N + g * NPT + j] = h[j];
    }
  } else {
    float* hk = p.carry_h + ((int64_t)seg * p.batch * p.dim + row) * N + g * NPT;
#pragma unroll
    for (int j = 0; j < NPT; ++j) hk[j] = h[j];
    if (g == 0) p.carry_s[(int64_t)seg * p.batch * p.dim + row] = sumDt;
  }
}

// Writes final_state = init_state (or zeros) for an empty sequence.
__global__ void copy_state_kernel(float* dst, const float* src, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = src ? src[i] : 0.f;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
template <int N> static void cfg_of(int& chans, int& chunk) {
  chans = ScanCfg<N>::CH;
  chunk = ScanCfg<N>::T;
}

static bool cfg_for(int64_t N, int& chans, int& chunk) {
  switch (N) {
    case 1: cfg_of<1>(chans, chunk); return true;
    case 2: cfg_of<2>(chans, chunk); return true;
    case 4: cfg_of<4>(chans, chunk); return true;
    case 8: cfg_of<8>(chans, chunk); return true;
    case 16: cfg_of<16>(chans, chunk); return true;
    case 32: cfg_of<32>(chans, chunk); return true;
    case 64: cfg_of<64>(chans, chunk); return true;
    default: return false;
  }
}

ScanPlan scan_plan(int64_t batch, int64_t dim, int64_t L, int64_t N, int io_dtype, int sm_count,
                   bool allow_split) {
  (void)io_dtype;
  ScanPlan pl{1, L, 0, 64, 32};
  if (!cfg_for(N, pl.chans, pl.chunk)) return pl;
  pl.seg_len = L > 0 ? L : 1;
  if (!allow_split || L <= 0 || batch <= 0 || dim <= 0) return pl;
  const int64_t blocks = ((dim + pl.chans - 1) / pl.chans) * batch;
  const int64_t want = (int64_t)sm_count * 2;  // blocks that keep every SM busy
  if (blocks >= want) return pl;
  int64_t nseg = (want + blocks - 1) / blocks;
  const int64_t max_by_len = L / (8 * (int64_t)pl.chunk);  // at least 8 chunks per segment
  if (nseg > max_by_len) nseg = max_by_len;
  if (nseg > 64) nseg = 64;
  if (nseg < 2) return pl;
  int64_t seg_len = (L + nseg - 1) / nseg;
  seg_len = ((seg_len + pl.chunk - 1) / pl.chunk) * pl.chunk;
  nseg = (L + seg_len - 1) / seg_len;
  if (nseg < 2) return pl;
  pl.nseg = (int)nseg;
  pl.seg_len = seg_len;
  const size_t rows = (size_t)batch * (size_t)dim;
  const size_t hbytes = ((size_t)(nseg - 1) * rows * (size_t)N * 4 + 255) / 256 * 256;
  pl.workspace_bytes = hbytes + (size_t)(nseg - 1) * rows * 4;
  return pl;
}

template <typename IO, int N, int PASS>
static cudaError_t launch_one(const ScanArgs& a, int nz, cudaStream_t stream) {
  using Cf = ScanCfg<N>;
  constexpr size_t bytes = ScanSmem<IO, N>::kBytes;
  auto kern = scan_kernel<IO, N, PASS>;
  static int configured_dev = -1;  // attribute set once per device change
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  dim3 grid((unsigned)((a.dim + Cf::CH - 1) / Cf::CH), (unsigned)a.batch, (unsigned)nz);
  kern<<<grid, kScanThreads, bytes, stream>>>(a);
  return cudaGetLastError();
}

template <typename IO, int N>
static cudaError_t launch_typed(const ScanArgs& a, cudaStream_t stream) {
  if (a.nseg > 1) {
    cudaError_t e = launch_one<IO, N, 1>(a, a.nseg - 1, stream);
    if (e != cudaSuccess) return e;
  }
  return launch_one<IO, N, 0>(a, a.nseg, stream);
}

template <typename IO>
static cudaError_t launch_io(const ScanArgs& a, int64_t N, cudaStream_t stream) {
  switch (N) {
    case 1: return launch_typed<IO, 1>(a, stream);
    case 2: return launch_typed<IO, 2>(a, stream);
    case 4: return launch_typed<IO, 4>(a, stream);
    case 8: return launch_typed<IO, 8>(a, stream);
    case 16: return launch_typed<IO, 16>(a, stream);
    case 32: return launch_typed<IO, 32>(a, stream);
    case 64: return launch_typed<IO, 64>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t scan_launch(const ScanArgs& a, int64_t N, int io_dtype, const ScanPlan& plan,
                        cudaStream_t stream) {
  (void)plan;
  if (a.batch == 0 || a.dim == 0) return cudaSuccess;
  if (a.L == 0) {
    if (!a.final_state) return cudaSuccess;
    const int64_t n = a.batch * a.dim * N;
    copy_state_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(a.final_state, a.init_state, n);
    return cudaGetLastError();
  }
  if (io_dtype == 0) return launch_io<float>(a, N, stream);
  return launch_io<__nv_bfloat16>(a, N, stream);
}

}  // namespace ssm
