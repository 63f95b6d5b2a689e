// Mamba-2's scalar-A state space model (SSD), chunked, for sm_103a.
//
// The chapter page ("14.1 SSM(State Space Models)과 Mamba 아키텍처의 부상",
// §5.1-5.2) restricts A to a scalar per step times the identity, so that per
// head the SSM is the masked product Y = (L ∘ C Bᵀ) X with L the lower-
// triangular matrix of cumulative decays, and computes it in chunks: the
// quadratic form inside a chunk on the tensor cores, states passed between
// chunks.  Per head h (P channels sharing the step Δ_t and the scalar a_h; B,
// C of the head's group), with s_t = Σ_{k<=t in the chunk} Δ_k a_h and the
// input weight β_t = (exp(Δ_t a_h) - 1)/a_h (zero-order hold) or Δ_t (Euler):
//
//   chunk state    S_c = Σ_τ exp(s_end - s_τ) β_τ x_τ ⊗ B_τ                (P x N)
//   state passing  H_c = exp(s_end(c)) H_{c-1} + S_c,  H_{-1} = init_state
//   chunk output   y_t = Σ_{τ<=t} (C_t·B_τ) exp(s_t - s_τ) β_τ x_τ
//                        + exp(s_t) C_t H_{c-1} + D_h x_t       (then · silu(z_t))
//
// Four launches: the chunks' step terms (all chunks in parallel), one walk
// over the chunks that forms each chunk's state contribution on the tensor
// cores and passes the running state on (parallel over heads and slices of the
// state's rows; the state never leaves the registers, only the bf16 copy each
// chunk's outputs read), the chunks' C Bᵀ per group and the chunk outputs (all
// chunks in parallel).  The last two run on the tcgen05 tensor cores with TMEM
// accumulators (ssm_ssd_tc.cu); the walk runs its products as mma.sync
// m16n8k16 bf16 with fp32 accumulation, operands staged in padded
// shared-memory rows (ldmatrix's eight row addresses fall in distinct bank
// groups).  Layouts are Mamba-2's: x, z, y (batch, L, H,
// P); dt (batch, L, H); B, C (batch, L, G, N); states (batch, H, P, N).
#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "ssm_mma.cuh"

namespace ssm {

constexpr int kSsdQ = kSsdChunk;  // chunk length
constexpr int kSsdP = 64;        // head dimension

// ---------------------------------------------------------------------------
// 0. step terms, one warp per (batch, chunk, head): Δ = softplus(dt + bias),
//    the cumulative log decay s_t = Σ_{k<=t in the chunk} Δ_k a_h, the input
//    weight β_t ((exp(Δ a) - 1)/a, or Δ with the Euler flag) and
//    w_t = exp(s_end - s_t) β_t, stored as [s | β | w] (64 floats each) for
//    the two chunk kernels.  Steps past the sequence get Δ = 0 (decay 1,
//    weight 0).  A lane takes two steps; s is a warp prefix sum.
// ---------------------------------------------------------------------------
constexpr int kTermsThreads = 128;
constexpr int kTermsRec = kSsdTermsRec;  // floats per (batch, chunk, head)

__global__ void __launch_bounds__(kTermsThreads) ssd_terms_kernel(const SsdArgs p) {
  constexpr int Q = kSsdQ;
  const int lane = threadIdx.x & 31;
  const int64_t unit = (int64_t)blockIdx.x * (kTermsThreads / 32) + (threadIdx.x >> 5);
  if (unit >= p.batch * p.nch * p.H) return;  // whole warps
  const int h = (int)(unit % p.H);
  const int64_t bc = unit / p.H;
  const int64_t c = bc % p.nch, b = bc / p.nch;
  const float a = p.A[h];
  const float bias = p.dt_bias ? p.dt_bias[h] : 0.f;
  float dA[2], beta[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int64_t t = c * Q + 2 * lane + i;
    dA[i] = 0.f;
    beta[i] = 0.f;
    if (t < p.L) {
      const float x = __bfloat162float(static_cast<const __nv_bfloat16*>(p.dt)[(b * p.L + t) * p.H + h]) + bias;
      const float dt = p.softplus ? softplus_precise(x) : x;
      dA[i] = dt * a;
      beta[i] = p.euler ? dt : (a != 0.f ? expm1f(dA[i]) / a : dt);
    }
  }
  float run = dA[0] + dA[1];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, run, o);
    if (lane >= o) run += n;
  }
  const float s0 = (run - (dA[0] + dA[1])) + dA[0];
  const float s_end = __shfl_sync(0xffffffffu, run, 31);
  float* out = p.ws_terms + unit * kTermsRec + 2 * lane;
  *reinterpret_cast<float2*>(out) = make_float2(s0, run);
  *reinterpret_cast<float2*>(out + Q) = make_float2(beta[0], beta[1]);
  *reinterpret_cast<float2*>(out + 2 * Q) =
      make_float2(__expf(s_end - s0) * beta[0], __expf(s_end - run) * beta[1]);
}

// ---------------------------------------------------------------------------
// 1. chunk states and state passing in one walk over the chunks.  A block
//    owns PR rows p of one head's P x N state; each warp keeps a 16 x N piece
//    of it in mma accumulators (fp32) for the whole sequence.  Per chunk c:
//
//      H_c = exp(s_end) H_{c-1} + Σ_τ w_τ x_τ ⊗ B_τ,   w_τ = exp(s_end - s_τ) β_τ
//
//    with the entering state H_{c-1} stored first (bf16, for the chunk-output
//    products: through a padded shared tile, then 16-byte coalesced stores).
//    The product (w x)ᵀ B runs on the tensor cores.  The next chunk's x slice,
//    B tile and step terms are in flight (cp.async, two stages) while a chunk
//    is used.
// ---------------------------------------------------------------------------
template <int N, int PR> struct SsdStateCfg {
  static constexpr int kWarps = PR / 16;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int RX = PR + 8;  // x slice rows [τ][p]: 80-byte rows
  static constexpr int RB = N + 8;   // B rows [τ][n] and entering-state rows [p][n]
  static constexpr int oB = kSsdQ * RX, oT = oB + kSsdQ * RB;  // bf16 offsets in a stage
  static constexpr int kStage = oT + 2 * kTermsRec;             // bf16 elements per stage
  static constexpr int oH = 2 * kStage;                         // entering-state tile [PR][RB]
  static constexpr size_t kBytes = (size_t)(oH + PR * RB) * 2;
  static constexpr int kTermVecs = kTermsRec * 4 / 16;
  static constexpr int kOutVecs = PR * N / 8;                   // 16-byte vectors of the tile
  static_assert(PR % 16 == 0 && kSsdP % PR == 0, "tiling");
  static_assert(kOutVecs % kThreads == 0, "whole vectors per thread in the state copy-out");
};
constexpr int kWalkRows = 32;  // state rows per block: 2 warps, 2 x 24 x 8 blocks on a 24-head layer

template <int N, int PR>
__global__ void __launch_bounds__(SsdStateCfg<N, PR>::kThreads)
    ssd_state_scan_kernel(const SsdArgs p) {
  using Cf = SsdStateCfg<N, PR>;
  constexpr int Q = kSsdQ, P = kSsdP, RX = Cf::RX, RB = Cf::RB, NT = Cf::kThreads;
  extern __shared__ float4 ssd_state_smem[];
  __nv_bfloat16* tiles = reinterpret_cast<__nv_bfloat16*>(ssd_state_smem);
  __nv_bfloat16* sH = tiles + Cf::oH;
  const int p0 = blockIdx.x * PR, h = blockIdx.y;
  const int64_t b = blockIdx.z;
  const int g = h / (p.H / p.G);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;

  auto stage = [&](int c) {
    __nv_bfloat16* st = tiles + (c & 1) * Cf::kStage;
    const int64_t t0 = (int64_t)c * Q;
    const int valid = (int)min64(Q, p.L - t0);
    ssd_stage<Q, PR, RX, NT>(st, static_cast<const __nv_bfloat16*>(p.x) + ((b * p.L + t0) * p.H + h) * P + p0,
                             p.H * P, valid);
    ssd_stage<Q, N, RB, NT>(st + Cf::oB,
                            static_cast<const __nv_bfloat16*>(p.B) + ((b * p.L + t0) * p.G + g) * N,
                            p.G * N, valid);
    {
      const float* src = p.ws_terms + ((b * p.nch + c) * p.H + h) * kTermsRec;
      for (int e = threadIdx.x; e < Cf::kTermVecs; e += NT)
        cp_async16(reinterpret_cast<float*>(st + Cf::oT) + 4 * e, src + 4 * e, true);
    }
    cp_async_commit();
  };

  // this thread's accumulator elements: rows rl, rl + 8 of the block's slice
  // (head rows p0 + rl, + 8); columns 8j + cc, +1
  const int rl = 16 * w + (lane >> 2), cc = 2 * (lane & 3);
  const int64_t head = (b * p.H + h) * (int64_t)(P * N) + (int64_t)(p0 + rl) * N + cc;
  float acc[N / 8][4];
#pragma unroll
  for (int j = 0; j < N / 8; ++j) {
    if (p.init_state) {
      const float2 u = *reinterpret_cast<const float2*>(p.init_state + head + 8 * j);
      const float2 v = *reinterpret_cast<const float2*>(p.init_state + head + 8 * N + 8 * j);
      acc[j][0] = u.x; acc[j][1] = u.y; acc[j][2] = v.x; acc[j][3] = v.y;
    } else {
      acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    }
  }
  __nv_bfloat16* myH = sH + rl * RB + cc;

  stage(0);
  for (int c = 0; c < p.nch; ++c) {
    const bool more = c + 1 < p.nch;
    if (more) stage(c + 1);
    // the state entering chunk c, into the shared tile
#pragma unroll
    for (int j = 0; j < N / 8; ++j) {
      *reinterpret_cast<uint32_t*>(myH + 8 * j) = pack_bf16(acc[j][0], acc[j][1]);
      *reinterpret_cast<uint32_t*>(myH + 8 * RB + 8 * j) = pack_bf16(acc[j][2], acc[j][3]);
    }
    if (more) cp_async_wait<1>(); else cp_async_wait<0>();
    __syncthreads();  // chunk c's tiles and terms, and the entering-state tile, are visible
    {  // entering state -> workspace [b][c][h][p][n], 16-byte vectors
      constexpr int VPR = N / 8;
      __nv_bfloat16* dst = p.ws_hin + ((b * p.nch + c) * p.H + h) * (int64_t)(P * N) + (int64_t)p0 * N;
#pragma unroll
      for (int k = 0; k < Cf::kOutVecs / NT; ++k) {
        const int v = threadIdx.x + k * NT;
        const int r = v / VPR, c8 = v % VPR;
        *reinterpret_cast<uint4*>(dst + r * N + 8 * c8) =
            *reinterpret_cast<const uint4*>(sH + r * RB + 8 * c8);
      }
    }

    const __nv_bfloat16* sx = tiles + (c & 1) * Cf::kStage;
    const __nv_bfloat16* sb = sx + Cf::oB;
    const float* sT = reinterpret_cast<const float*>(sx + Cf::oT);  // [s | β | w]
    const float* wv = sT + 2 * Q;
    const float decay = __expf(sT[Q - 1]);
#pragma unroll
    for (int j = 0; j < N / 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] *= decay;
#pragma unroll
    for (int ks = 0; ks < Q / 16; ++ks) {
      // A = (w x)ᵀ: rows p, k = τ; x stored [τ][p] -> transposed loads, then each
      // element scaled by its step's w (fp32 product, rounded to bf16)
      uint32_t af[4];
      {
        const int i = lane >> 3;
        ldsm_x4_t(af, sx + (16 * ks + (i >> 1) * 8 + (lane & 7)) * RX + 16 * w + (i & 1) * 8);
        const int tau = 16 * ks + cc;
        const float w0 = wv[tau], w1 = wv[tau + 1], w8 = wv[tau + 8], w9 = wv[tau + 9];
        auto scale = [](uint32_t v, float lo_w, float hi_w) {
          return pack_bf16(__uint_as_float(v << 16) * lo_w, __uint_as_float(v & 0xffff0000u) * hi_w);
        };
        af[0] = scale(af[0], w0, w1);
        af[1] = scale(af[1], w0, w1);
        af[2] = scale(af[2], w8, w9);
        af[3] = scale(af[3], w8, w9);
      }
#pragma unroll
      for (int nn = 0; nn < N / 16; ++nn) {
        // B operand: k = τ, n; stored [τ][n] -> transposed loads, two n8 tiles
        uint32_t bf[4];
        ldsm_x4_t(bf, sb + (16 * ks + (lane & 15)) * RB + 16 * nn + (lane >> 4) * 8);
        mma_bf16(acc[2 * nn], af, bf[0], bf[1]);
        mma_bf16(acc[2 * nn + 1], af, bf[2], bf[3]);
      }
    }
    __syncthreads();  // the next iteration's copies and entering state reuse the tiles
  }
  if (p.final_state) {
#pragma unroll
    for (int j = 0; j < N / 8; ++j) {
      *reinterpret_cast<float2*>(p.final_state + head + 8 * j) = make_float2(acc[j][0], acc[j][1]);
      *reinterpret_cast<float2*>(p.final_state + head + 8 * N + 8 * j) = make_float2(acc[j][2], acc[j][3]);
    }
  }
}

// ---------------------------------------------------------------------------
// 2. the chunks' C Bᵀ, once per (batch, chunk, group): every head of a group
//    shares it.  G[t][τ] = C_t · B_τ, fp32, [t][τ] rows of 64, on the tcgen05
//    tensor cores (ssm_ssd_tc.cu); the chunk outputs read the entries τ <= t.
// ---------------------------------------------------------------------------

// ---------------------------------------------------------------------------
// 3. chunk outputs: y = (mask ∘ C Bᵀ) X + exp(s_t) C Hᵀ + D x, gated, per
//    (batch, chunk, head) on the tcgen05 tensor cores (ssm_ssd_tc.cu).
// ---------------------------------------------------------------------------

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
SsdLayout ssd_layout(int64_t batch, int64_t L, int64_t H, int64_t G, int64_t N) {
  SsdLayout w{};
  w.nch = (L + kSsdQ - 1) / kSsdQ;
  const size_t units = (size_t)batch * (size_t)w.nch * (size_t)H;
  const size_t gunits = (size_t)batch * (size_t)w.nch * (size_t)G;
  w.o_hin = 0;
  w.o_terms = (units * (size_t)kSsdP * (size_t)N * 2 + 255) / 256 * 256;
  w.o_cb = w.o_terms + (units * (size_t)kTermsRec * 4 + 255) / 256 * 256;
  w.bytes = w.o_cb + (gunits * (size_t)kSsdQ * kSsdQ * 4 + 255) / 256 * 256;
  return w;
}

template <int N>
static cudaError_t ssd_walk(const SsdArgs& a, cudaStream_t s) {
  using SC = SsdStateCfg<N, kWalkRows>;
  static int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    const cudaError_t e = cudaFuncSetAttribute(ssd_state_scan_kernel<N, kWalkRows>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SC::kBytes);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  ssd_state_scan_kernel<N, kWalkRows><<<dim3(kSsdP / kWalkRows, (unsigned)a.H, (unsigned)a.batch),
                                        SC::kThreads, SC::kBytes, s>>>(a);
  return cudaGetLastError();
}

cudaError_t ssd_terms_launch(const SsdArgs& a, cudaStream_t s) {
  const int64_t units = a.batch * a.nch * a.H;
  if (units == 0) return cudaSuccess;
  constexpr int kUnitsPerBlock = kTermsThreads / 32;
  ssd_terms_kernel<<<(unsigned)((units + kUnitsPerBlock - 1) / kUnitsPerBlock), kTermsThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <int N>
static cudaError_t ssd_typed(const SsdArgs& a, cudaStream_t s) {
  cudaError_t e = ssd_terms_launch(a, s);
  if (e != cudaSuccess) return e;
  e = ssd_walk<N>(a, s);
  if (e != cudaSuccess) return e;
  e = ssd_cb_tc_launch(a, N, s);
  if (e != cudaSuccess) return e;
  return ssd_chunk_tc_launch(a, N, s);
}

cudaError_t ssd_launch(const SsdArgs& a, int64_t N, cudaStream_t stream) {
  if (a.batch == 0 || a.H == 0 || a.L == 0) return cudaSuccess;
  switch (N) {
    case 64: return ssd_typed<64>(a, stream);
    case 128: return ssd_typed<128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssm
