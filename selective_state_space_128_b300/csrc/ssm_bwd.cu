// Backward pass of the selective scan (S6) for sm_103a.
//
// The summary page ("Mamba: Linear-Time Sequence Modeling", section 4c, the
// hardware-aware algorithm) trains the layer without storing the expanded
// (batch, L, d_inner, N) states: the backward pass recomputes them.  The
// derivatives are the chain rule of the forward definition (equations (2)
// and (4) with the selection of Algorithm 2).  For a loss with dLoss/dy = dy
// and dLoss/dh_{L-1} = dfinal, with g = silu(z), s = C·h + D u, y = s g:
//
//   ds_t = dy_t g_t,           dz_t = dy_t s_t silu'(z_t)
//   λ_t  = ds_t C_t + Ā_{t+1} λ_{t+1}        (λ_{L-1} also receives dfinal)
//   du_t = ds_t D + Σ_n λ B̄ B,               dB_t += λ B̄ u,   dC_t += ds_t h_t
//   dΔ_t = Σ_n Ā λ (A h_{t-1} + B u),        dA += λ (Δ Ā h_{t-1} + B u (Δ Ā - B̄)/A)
//   (the Euler variant B̄ = Δ: dΔ_t = Σ_n λ (A Ā h_{t-1} + B u), and no B u term in dA)
//   dΔraw_t = dΔ_t σ(Δraw_t + bias) (softplus), dbias += dΔraw,  dD += ds u,
//   dh_{-1} = Ā_0 λ_0
// where B̄ = (Ā - 1)/A is the scalar zero-order-hold factor (A = 0: Δ, and
// (Δ Ā - B̄)/A takes its limit Δ²/2).
//
// Design (B300).  A block owns CH channels of one batch row with the same
// lane layout as the forward kernel: G lanes per channel, NPT states per lane
// in registers.  It walks the sequence twice:
//  1. forward, recurrence only, storing the state at the start of every chunk
//     of T steps to a checkpoint workspace (N floats per channel per chunk) --
//     skipped when a training forward (ssm_scan_fwd_train) saved them;
//  2. backward, chunk by chunk from the end: reload the chunk's start state,
//     recompute the T states into shared memory, finalise the gate's
//     derivative from the recomputed readout, then run the adjoint recurrence
//     λ in reverse, reading h_{t-1} from shared memory.  λ and the dA sums
//     stay in registers for the whole sequence.
// Derivatives that are shared by many channels -- dB and dC (per batch, state
// and step), dA, dD and dbias (per channel, summed over the batch) -- are
// first reduced inside the block (over its channels, through shared memory)
// and written as per-block partial sums; a second kernel adds the partials in
// a fixed order, so the result does not depend on scheduling.
#include <cstring>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

constexpr int kBwdThreads = 128;
// Shortest segment of a sequence split across blocks (steps).
constexpr int64_t kBwdMinSeg = 512;

template <int N> struct BwdCfg {
  // states per lane: at most 16 (N = 128 spreads over 8 lanes of a channel)
  static constexpr int NPT = N <= 4 ? N : (N <= 16 ? 4 : (N <= 64 ? N / 4 : 16));
  static constexpr int G = N / NPT;                                // lanes per channel
  static constexpr int CH = kBwdThreads / G;                       // channels per block
  // steps per chunk (at least one channel step per thread in the per-step work)
  static constexpr int T = NPT <= 4 ? 16 : (NPT == 8 ? 8 : (CH >= 32 ? 4 : 8));
  static constexpr int E = CH * T / kBwdThreads;  // channel steps per thread (per-step work)
  static constexpr int TPR = T / E;               // threads per channel row
  static constexpr int VW = NPT < 4 ? NPT : 4;    // floats per shared-memory vector
  static constexpr int QN = NPT / VW;             // vectors per lane
  static constexpr int GW = G < 2 ? G : 2;        // warp layout as in the forward kernel
  static constexpr int CW = 32 / GW;
  static constexpr int WPC = G / GW;
  static constexpr int RowF = T + 1;              // per-channel-step tiles (odd rows)
  static constexpr int RowBC = N < 4 ? N : N + 4; // transposed B/C rows
  static constexpr int NU = T / 4;                // 4-step units of a partial row
  // channel reductions: NV output vectors (step, state group, part); RS threads
  // per vector and RCH channels per thread, or VPT vectors per thread when there
  // are more vectors than threads
  static constexpr int NV = T * G * QN;
  static constexpr int RS = NV >= kBwdThreads ? 1 : kBwdThreads / NV;
  static constexpr int VPT = NV >= kBwdThreads ? NV / kBwdThreads : 1;
  static constexpr int RCH = CH / RS;
  // resident blocks per SM the register budget is sized for (the lanes with 16
  // states, and the 16-step rows of N = 4, need more than a third of the file)
  static constexpr int MINB = (NPT >= 16 || (NPT == 4 && E >= 16)) ? 2 : 3;
  static_assert(G * NPT == N && E >= 1 && TPR <= 8 && RS >= 1 && RCH * RS == CH, "tiling");
  static_assert(VPT * kBwdThreads == NV * RS, "whole reduction vectors per thread");
};

// Shared-memory layout (float offsets).
template <int N> struct BwdSmem {
  using Cf = BwdCfg<N>;
  static constexpr int CH = Cf::CH, T = Cf::T;
  static constexpr int oDT = 0;                              // Δ [CH][RowF]
  static constexpr int oU = oDT + CH * Cf::RowF;             // u [CH][RowF]
  static constexpr int oDS = oU + CH * Cf::RowF;             // ds = dy·g [CH][RowF]
  static constexpr int oBt = (oDS + CH * Cf::RowF + 3) / 4 * 4;  // B [T][RowBC]
  static constexpr int oCt = oBt + T * Cf::RowBC;            // C [T][RowBC]
  // states: slot 0 = state before the chunk, slot t+1 = h_t; overwritten by
  // the adjoint sweep with λ B̄ u of step t.  [T+1][QN][lanes][VW]
  static constexpr int oHs = (oCt + T * Cf::RowBC + 3) / 4 * 4;
  static constexpr int oPa = oHs + (T + 1) * Cf::QN * kBwdThreads * Cf::VW;  // partials [lanes][T]
  static constexpr int oPb = oPa + kBwdThreads * T;
  static constexpr int oBias = oPb + kBwdThreads * T;
  static constexpr int oD = oBias + CH;
  static constexpr int kFloats = oD + CH;
  static constexpr size_t kBytes = (size_t)kFloats * 4;
};

// Partial tile: row = g*CH + c, 4-step units swizzled so that the eight lanes
// of a quarter warp storing a 16-byte unit hit distinct bank groups.
template <int N> __device__ __forceinline__ int bwd_pidx(int row, int t) {
  using Cf = BwdCfg<N>;
  constexpr int NU = Cf::NU;
  const int swz = NU > 1 ? (row / (8 / NU)) & (NU - 1) : 0;
  return row * Cf::T + (((t >> 2) ^ swz) << 2) + (t & 3);
}

template <int N> __device__ __forceinline__ int bwd_lane_of(int c, int g) {
  using Cf = BwdCfg<N>;
  const int wid = (c / Cf::CW) * Cf::WPC + g / Cf::GW;
  const int lid = (g % Cf::GW) * Cf::CW + c % Cf::CW;
  return wid * 32 + lid;
}

__device__ __forceinline__ float sigmoid_fast(float x) { return rcp_fast(1.0f + ex2_fast(-x * kLog2e)); }
__device__ __forceinline__ float sigmoid_precise(float x) { return 1.0f / (1.0f + expf(-x)); }

// K consecutive floats of shared memory, as 16- or 8-byte accesses where K allows
// (every caller's address is aligned to the access).
template <int K> __device__ __forceinline__ void lds_vec(const float* p, float* v) {
  if constexpr (K % 4 == 0) {
#pragma unroll
    for (int i = 0; i < K; i += 4) {
      const float4 x = *reinterpret_cast<const float4*>(p + i);
      v[i] = x.x; v[i + 1] = x.y; v[i + 2] = x.z; v[i + 3] = x.w;
    }
  } else if constexpr (K == 2) {
    const float2 x = *reinterpret_cast<const float2*>(p);
    v[0] = x.x; v[1] = x.y;
  } else {
#pragma unroll
    for (int i = 0; i < K; ++i) v[i] = p[i];
  }
}
template <int K> __device__ __forceinline__ void sts_vec(float* p, const float* v) {
  if constexpr (K % 4 == 0) {
#pragma unroll
    for (int i = 0; i < K; i += 4)
      *reinterpret_cast<float4*>(p + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
  } else if constexpr (K == 2) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
  } else {
#pragma unroll
    for (int i = 0; i < K; ++i) p[i] = v[i];
  }
}

template <typename IO> __device__ __forceinline__ float ld_io(const void* p, int64_t i) {
  return io_traits<IO>::to_f32(static_cast<const IO*>(p)[i]);
}

// Raw global inputs of one thread's share of a chunk (E steps of one channel row;
// PER elements of each of B and C), fetched one chunk ahead so that the loads
// are in flight while the block works on the current chunk.
template <int N> struct BwdPre {
  static constexpr int E = BwdCfg<N>::E;
  static constexpr int PER = (N * BwdCfg<N>::T + kBwdThreads - 1) / kBwdThreads;
  float dl[E], u[E], dy[E], z[E];
  float b[PER], c[PER];
  float h[BwdCfg<N>::NPT];  // the lane's chunk-start state (adjoint sweep)
};

// One recurrence step of a lane, fast flavour, packed pairs:
// h = Ā (h - v) + v with Ā = 2^(Δ A log2 e), v = -B u / A.
template <int NP>
__device__ __forceinline__ void step_pairs(f2 (&hq)[NP], float dt, float u, const f2 (&Bq)[NP],
                                           const f2 (&A2p)[NP], const f2 (&nIp)[NP]) {
  const f2 dt2 = pack2(dt, dt), u2 = pack2(u, u);
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    float x0, x1;
    unpack2(mul2(dt2, A2p[q]), x0, x1);
    const f2 a = pack2(ex2_fast(x0), ex2_fast(x1));
    const f2 v = mul2(mul2(Bq[q], u2), nIp[q]);
    hq[q] = fma2(a, sub2(hq[q], v), v);
  }
}

template <int K> __device__ __forceinline__ void lds_f2(const float* p, f2 (&v)[K]) {
#pragma unroll
  for (int q = 0; q + 1 < K; q += 2) lds_pairs(p + 2 * q, v[q], v[q + 1]);
  if constexpr (K % 2 == 1) lds_pair(p + 2 * (K - 1), v[K - 1]);
}

// ---------------------------------------------------------------------------
// The per-block kernel
// ---------------------------------------------------------------------------
template <typename IO, int N>
__global__ void __launch_bounds__(kBwdThreads, BwdCfg<N>::MINB) scan_bwd_kernel(const BwdArgs p) {
  using Cf = BwdCfg<N>;
  using S = BwdSmem<N>;
  constexpr int NPT = Cf::NPT, CH = Cf::CH, T = Cf::T, E = Cf::E, TPR = Cf::TPR;
  constexpr int VW = Cf::VW, QN = Cf::QN, G = Cf::G;
  constexpr int NP = NPT / 2 > 0 ? NPT / 2 : 1;  // packed pairs per lane (fast flavour)
  constexpr bool PAIRS = NPT % 2 == 0;
  // carry h_t through the adjoint sweep (two more pair registers per pair):
  // only where that stays within the register budget without spills
  constexpr bool kCarryH = PAIRS && NP <= 2 && N >= 8;
  constexpr int PER = BwdPre<N>::PER;
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  float* sDT = sm + S::oDT;
  float* sU = sm + S::oU;
  float* sDS = sm + S::oDS;
  float* sBt = sm + S::oBt;
  float* sCt = sm + S::oCt;
  float* sHs = sm + S::oHs;
  float* sPa = sm + S::oPa;
  float* sPb = sm + S::oPb;
  float* sBias = sm + S::oBias;
  float* sD = sm + S::oD;

  const int tid = threadIdx.x;
  const int wid = tid >> 5, lid = tid & 31;
  const int g = (wid % Cf::WPC) * Cf::GW + lid / Cf::CW;
  const int c = (wid / Cf::WPC) * Cf::CW + lid % Cf::CW;
  const int prow = g * CH + c;
  const int64_t b = blockIdx.y;
  const int blk = blockIdx.x;
  const int64_t d0 = (int64_t)blk * CH;
  const int64_t d = d0 + c;
  const bool chan_ok = d < p.dim;
  const int nrows = (int)min64(CH, p.dim - d0);
  const int64_t L = p.L;
  const int nch = (int)((L + T - 1) / T);
  // this block's segment of the sequence: chunks [k_begin, k_end)
  const int seg = blockIdx.z;
  // (a split plan's segments are whole chunks; the last one ends with the sequence)
  const int k_begin = (int)((int64_t)seg * (p.seg_len / T));
  const int k_end = seg == p.nseg - 1 ? nch : (int)min64(nch, (int64_t)(seg + 1) * (p.seg_len / T));
  // this thread's row and steps in the per-step (cooperative) phases
  const int r = tid / TPR, te = (tid % TPR) * E;
  const bool row_ok = r < nrows;
  // element (this row, step t) of u/Δ/z/dy and their derivatives is at
  // io_row + t * io_ts: rows of L steps, or steps dim apart in (batch, L, dim)
  const bool bld = p.bld != 0;
  const int64_t io_row = bld ? b * L * p.dim + d0 + (row_ok ? r : 0)
                             : (b * p.dim + d0 + (row_ok ? r : 0)) * L;
  const int64_t io_ts = bld ? p.dim : 1;
  // E-step runs as vectors: vecio moves 4 bf16 as 8 bytes and 8 or 16 bf16 (or
  // 4+ floats) as 16-byte accesses, so every row must start on that boundary
  constexpr int kVecBytes = (sizeof(IO) == 2 && E == 4) ? 8 : 16;
  const bool vec = !bld && E % 4 == 0 && (L * (int64_t)sizeof(IO)) % kVecBytes == 0;

  for (int i = tid; i < CH; i += kBwdThreads) {
    const bool ok = d0 + i < p.dim;
    sBias[i] = (p.bias && ok) ? p.bias[d0 + i] : 0.f;
    sD[i] = (p.D && ok) ? p.D[d0 + i] : 0.f;
  }
  float Aj[NPT], invA[NPT];
  f2 A2p[NP], nIp[NP], iAp[NP], Ajp[NP];
  bool zeroA = false;
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    Aj[j] = chan_ok ? p.A[d * N + g * NPT + j] : -1.f;
    zeroA |= Aj[j] == 0.f;
    invA[j] = Aj[j] != 0.f ? 1.f / Aj[j] : 0.f;
  }
  if constexpr (PAIRS) {
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      A2p[q] = pack2(Aj[2 * q] * kLog2e, Aj[2 * q + 1] * kLog2e);
      nIp[q] = pack2(-invA[2 * q], -invA[2 * q + 1]);
      iAp[q] = pack2(invA[2 * q], invA[2 * q + 1]);
      Ajp[q] = pack2(Aj[2 * q], Aj[2 * q + 1]);
    }
  }
  const bool euler = p.euler != 0;  // B̄ = Δ B: runs on the precise flavour
  const bool precise = __syncthreads_or(zeroA) || p.force_precise || euler;
  const bool fast_pairs = PAIRS && !precise;  // block-uniform
  const bool sp = p.softplus != 0;

  // ---- global -> registers (one chunk ahead) ----
  auto fetch = [&](int k, bool full, BwdPre<N>& pr) {
    const int64_t t0 = (int64_t)k * T;
    const int tc = (int)min64(T, L - t0);
    const int64_t gi = io_row + (t0 + te) * io_ts;
    bool done = false;
    if constexpr (E % 4 == 0) {
      if (row_ok && vec && te + E <= tc) {
        vecio<IO, E>::load(static_cast<const IO*>(p.delta) + gi, pr.dl);
        vecio<IO, E>::load(static_cast<const IO*>(p.u) + gi, pr.u);
        if (full) {
          vecio<IO, E>::load(static_cast<const IO*>(p.dy) + gi, pr.dy);
          if (p.z) vecio<IO, E>::load(static_cast<const IO*>(p.z) + gi, pr.z);
        }
        done = true;
      }
    }
    if (!done) {
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const bool ok = row_ok && te + j < tc;
        const int64_t gj = gi + j * io_ts;
        pr.dl[j] = ok ? ld_io<IO>(p.delta, gj) : 0.f;
        pr.u[j] = ok ? ld_io<IO>(p.u, gj) : 0.f;
        if (full) {
          pr.dy[j] = ok ? ld_io<IO>(p.dy, gj) : 0.f;
          pr.z[j] = (ok && p.z) ? ld_io<IO>(p.z, gj) : 0.f;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = tid + i * kBwdThreads;
      const int n = e / T, t = e - n * T;
      const bool ok = (N * T % kBwdThreads == 0 || e < N * T) && t < tc;
      const int64_t bi = (b * N + n) * L + t0 + t;
      pr.b[i] = ok ? p.B[bi] : 0.f;
      if (full) pr.c[i] = ok ? p.C[bi] : 0.f;
    }
    if (full) {
#pragma unroll
      for (int j = 0; j < NPT; ++j) pr.h[j] = chan_ok ? p.ckpt[((b * nch + k) * p.dim + d) * N + g * NPT + j] : 0.f;
    }
  };
  // ---- registers -> shared tiles; Δ, σ, gate, ds per channel step ----
  auto stage = [&](int k, bool full, const BwdPre<N>& pr, float (&dyv)[E], float (&zz)[E],
                   float (&sg)[E]) {
    const int64_t t0 = (int64_t)k * T;
    const int tc = (int)min64(T, L - t0);
    const float bias = sBias[r];
    float dtv[E], dsv[E];
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const bool ok = row_ok && te + j < tc;
      const float x = pr.dl[j] + bias;
      const float dt = sp ? (precise ? softplus_precise(x) : softplus_fast(x)) : x;
      dtv[j] = ok ? dt : 0.f;
      if (full) {
        sg[j] = sp ? (precise ? sigmoid_precise(x) : sigmoid_fast(x)) : 1.f;
        dyv[j] = pr.dy[j];
        zz[j] = pr.z[j];
        const float gate = p.z ? (precise ? silu_precise(zz[j]) : silu_fast(zz[j])) : 1.f;
        dsv[j] = ok ? dyv[j] * gate : 0.f;
      }
    }
    float* rowDT = sDT + r * Cf::RowF + te;
    float* rowU = sU + r * Cf::RowF + te;
    float* rowDS = sDS + r * Cf::RowF + te;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      rowDT[j] = dtv[j];
      rowU[j] = pr.u[j];
      if (full) rowDS[j] = dsv[j];
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = tid + i * kBwdThreads;
      if (N * T % kBwdThreads == 0 || e < N * T) {
        const int n = e / T, t = e - n * T;
        sBt[t * Cf::RowBC + n] = pr.b[i];
        if (full) sCt[t * Cf::RowBC + n] = pr.c[i];
      }
    }
  };
  auto hs_vec = [&](int slot, int q, int lane) {
    return sHs + ((slot * QN + q) * kBwdThreads + lane) * VW;
  };
  // this lane's NPT states of a slot as packed pairs (VW / 2 pairs per vector)
  auto hs_store_pairs = [&](int slot, const f2 (&v)[NP]) {
#pragma unroll
    for (int q = 0; q < QN; ++q) {
      if constexpr (VW == 4) sts_pairs(hs_vec(slot, q, tid), v[2 * q], v[2 * q + 1]);
      else sts_pair(hs_vec(slot, q, tid), v[q]);
    }
  };
  auto hs_load_pairs = [&](int slot, f2 (&v)[NP]) {
#pragma unroll
    for (int q = 0; q < QN; ++q) {
      if constexpr (VW == 4) lds_pairs(hs_vec(slot, q, tid), v[2 * q], v[2 * q + 1]);
      else lds_pair(hs_vec(slot, q, tid), v[q]);
    }
  };

  // ---------------- sweep 1: chunk-start states ----------------
  float h[NPT];
  f2 hq[NP];
#pragma unroll
  for (int j = 0; j < NPT; ++j)
    h[j] = (p.init_state && chan_ok) ? p.init_state[(b * p.dim + d) * N + g * NPT + j] : 0.f;
  if (chan_ok && !p.saved) {
    // earlier segments: h <- exp(A ΣΔ_k) h + (segment k's end state from zero)
    const int64_t row = b * p.dim + d;
    for (int k = 0; k < seg; ++k) {
      const float sk = p.fcarry_s[(int64_t)k * p.batch * p.dim + row];
      const float* hk = p.fcarry_h + ((int64_t)k * p.batch * p.dim + row) * N + g * NPT;
#pragma unroll
      for (int j = 0; j < NPT; ++j) h[j] = fmaf(expf(sk * Aj[j]), h[j], hk[j]);
    }
  }
  if constexpr (PAIRS) {
#pragma unroll
    for (int q = 0; q < NP; ++q) hq[q] = pack2(h[2 * q], h[2 * q + 1]);
  }
  float dyv[E], zz[E], sg[E];
  BwdPre<N> pre;
  const int k1 = p.saved ? k_begin : k_end;  // a training forward already saved them
  if (k_begin < k1) fetch(k_begin, false, pre);
  for (int k = k_begin; k < k1; ++k) {
    if (fast_pairs) {
#pragma unroll
      for (int q = 0; q < NP; ++q) unpack2(hq[q], h[2 * q], h[2 * q + 1]);
    }
    if (chan_ok) {
      float* cp = p.ckpt + ((b * nch + k) * p.dim + d) * N + g * NPT;
      sts_vec<NPT>(cp, h);  // (a global store; sts_vec only packs the vector)
    }
    stage(k, false, pre, dyv, zz, sg);
    if (k + 1 < k1) fetch(k + 1, false, pre);
    __syncthreads();
    const float* rDT = sDT + c * Cf::RowF;
    const float* rU = sU + c * Cf::RowF;
    if (fast_pairs) {
#pragma unroll 4
      for (int t = 0; t < T; ++t) {
        f2 Bq[NP];
        lds_f2<NP>(sBt + t * Cf::RowBC + g * NPT, Bq);
        step_pairs<NP>(hq, rDT[t], rU[t], Bq, A2p, nIp);
      }
    } else {
#pragma unroll 4
      for (int t = 0; t < T; ++t) {
        float Bv[NPT];
        lds_vec<NPT>(sBt + t * Cf::RowBC + g * NPT, Bv);
        const float dt = rDT[t], u = rU[t];
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
          if (!precise) {
            const float a = ex2_fast(dt * Aj[j] * kLog2e);
            const float v = -Bv[j] * u * invA[j];
            h[j] = fmaf(a, h[j] - v, v);
          } else {
            const float x = dt * Aj[j];
            const float bb = (Aj[j] != 0.f && !euler) ? expm1f(x) * invA[j] : dt;
            h[j] = fmaf(expf(x), h[j], bb * (Bv[j] * u));
          }
        }
      }
    }
    __syncthreads();
  }

  // ---------------- sweep 2: adjoint, chunk by chunk from the end ----------------
  float lam[NPT], dAacc[NPT];
  f2 lq[NP], dAq[NP], dA2q[NP];
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    lam[j] = (p.d_final_state && chan_ok) ? p.d_final_state[(b * p.dim + d) * N + g * NPT + j] : 0.f;
    dAacc[j] = 0.f;
  }
  if (chan_ok) {
    // later segments, from the last: λ <- (segment k's adjoint at its start from
    // a zero adjoint at its end) + exp(A ΣΔ_k) λ
    const int64_t row = b * p.dim + d;
    for (int k = p.nseg - 1; k > seg; --k) {
      const float sk = p.acarry_s[(int64_t)(k - 1) * p.batch * p.dim + row];
      const float* lk = p.acarry_l + ((int64_t)(k - 1) * p.batch * p.dim + row) * N + g * NPT;
#pragma unroll
      for (int j = 0; j < NPT; ++j) lam[j] = fmaf(expf(sk * Aj[j]), lam[j], lk[j]);
    }
  }
  if constexpr (PAIRS) {
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      lq[q] = pack2(lam[2 * q], lam[2 * q + 1]);
      dAq[q] = pack2(0.f, 0.f);
      dA2q[q] = pack2(0.f, 0.f);
    }
  }
  float dD_acc = 0.f, dbias_acc = 0.f;
  float* wsB_blk = p.ws_B + ((b * p.nblk + blk) * N) * L;
  float* wsC_blk = p.ws_C + ((b * p.nblk + blk) * N) * L;
  // channel reductions: this thread's output vectors (step rt, state group rg,
  // part rq), VPT of them, and its share `part` of the channels
  const int part = tid % Cf::RS;

  if (k_begin < k_end) fetch(k_end - 1, true, pre);
  for (int k = k_end - 1; k >= k_begin; --k) {
    const int64_t t0 = (int64_t)k * T;
    const int tc = (int)min64(T, L - t0);
    // P1: stage the chunk; the next (earlier) chunk's loads go in flight
    stage(k, true, pre, dyv, zz, sg);
#pragma unroll
    for (int j = 0; j < NPT; ++j) h[j] = pre.h[j];
    if (k > k_begin) fetch(k - 1, true, pre);
    const float* rDT = sDT + c * Cf::RowF;
    const float* rU = sU + c * Cf::RowF;
    const float* rDS = sDS + c * Cf::RowF;
    __syncthreads();

    // P2: recompute the chunk's states into slots 1..T, readout partials
    {
#pragma unroll
      for (int q = 0; q < QN; ++q) sts_vec<VW>(hs_vec(0, q, tid), h + q * VW);
      float acc4[4];
      if (fast_pairs) {
#pragma unroll
        for (int q = 0; q < NP; ++q) hq[q] = pack2(h[2 * q], h[2 * q + 1]);
#pragma unroll 4
        for (int t = 0; t < T; ++t) {
          f2 Bq[NP], Cq[NP];
          lds_f2<NP>(sBt + t * Cf::RowBC + g * NPT, Bq);
          lds_f2<NP>(sCt + t * Cf::RowBC + g * NPT, Cq);
          step_pairs<NP>(hq, rDT[t], rU[t], Bq, A2p, nIp);
          f2 s2 = mul2(Cq[0], hq[0]);
#pragma unroll
          for (int q = 1; q < NP; ++q) s2 = fma2(Cq[q], hq[q], s2);
          float lo, hi;
          unpack2(s2, lo, hi);
          hs_store_pairs(t + 1, hq);
          acc4[t & 3] = lo + hi;
          if ((t & 3) == 3)
            *reinterpret_cast<float4*>(sPa + bwd_pidx<N>(prow, t - 3)) =
                make_float4(acc4[0], acc4[1], acc4[2], acc4[3]);
        }
      } else {
#pragma unroll 4
        for (int t = 0; t < T; ++t) {
          float Bv[NPT], Cv[NPT];
          lds_vec<NPT>(sBt + t * Cf::RowBC + g * NPT, Bv);
          lds_vec<NPT>(sCt + t * Cf::RowBC + g * NPT, Cv);
          const float dt = rDT[t], u = rU[t];
          float s = 0.f;
#pragma unroll
          for (int j = 0; j < NPT; ++j) {
            if (!precise) {
              const float a = ex2_fast(dt * Aj[j] * kLog2e);
              const float v = -Bv[j] * u * invA[j];
              h[j] = fmaf(a, h[j] - v, v);
            } else {
              const float x = dt * Aj[j];
              const float bb = (Aj[j] != 0.f && !euler) ? expm1f(x) * invA[j] : dt;
              h[j] = fmaf(expf(x), h[j], bb * (Bv[j] * u));
            }
            s = fmaf(Cv[j], h[j], s);
          }
#pragma unroll
          for (int q = 0; q < QN; ++q) sts_vec<VW>(hs_vec(t + 1, q, tid), h + q * VW);
          acc4[t & 3] = s;
          if ((t & 3) == 3)
            *reinterpret_cast<float4*>(sPa + bwd_pidx<N>(prow, t - 3)) =
                make_float4(acc4[0], acc4[1], acc4[2], acc4[3]);
        }
      }
    }
    __syncthreads();

    // P3: dz (needs s = Σ_g partials + D u), dD; dC reduced over the block's channels
    {
      float sp_[E];
#pragma unroll
      for (int j = 0; j < E; ++j) sp_[j] = 0.f;
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        if constexpr (E % 4 == 0) {
#pragma unroll
          for (int kq = 0; kq < E / 4; ++kq) {
            const float4 v4 = *reinterpret_cast<const float4*>(sPa + bwd_pidx<N>(gg * CH + r, te + 4 * kq));
            sp_[4 * kq] += v4.x; sp_[4 * kq + 1] += v4.y; sp_[4 * kq + 2] += v4.z; sp_[4 * kq + 3] += v4.w;
          }
        } else {
#pragma unroll
          for (int j = 0; j < E; ++j) sp_[j] += sPa[bwd_pidx<N>(gg * CH + r, te + j)];
        }
      }
      const float Dr = sD[r];
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const int t = te + j;
        const float u = sU[r * Cf::RowF + t];
        const float s = fmaf(Dr, u, sp_[j]);
        dD_acc = fmaf(sDS[r * Cf::RowF + t], u, dD_acc);  // zero past the end
        if (p.z) {
          const float zg = zz[j];
          const float sz = precise ? sigmoid_precise(zg) : sigmoid_fast(zg);
          sp_[j] = dyv[j] * s * sz * fmaf(zg, 1.f - sz, 1.f);
        }
      }
      if (p.z && row_ok) {
        IO* dzp = static_cast<IO*>(p.dz) + io_row + (t0 + te) * io_ts;
        bool done = false;
        if constexpr (E % 4 == 0) {
          if (vec && te + E <= tc) {
            vecio<IO, E>::store(dzp, sp_);
            done = true;
          }
        }
        if (!done) {
#pragma unroll
          for (int j = 0; j < E; ++j)
            if (te + j < tc) dzp[j * io_ts] = io_traits<IO>::from_f32(sp_[j]);
        }
      }
      // dC[t][n] = Σ_c ds[c][t] h_t[c][n]
#pragma unroll
      for (int kv = 0; kv < Cf::VPT; ++kv) {
        const int vid = tid / Cf::RS + kv * (kBwdThreads / Cf::RS);
        const int rt = vid / (G * QN), rg = (vid % (G * QN)) / QN, rq = vid % QN;
        float acc[VW];
#pragma unroll
        for (int v = 0; v < VW; ++v) acc[v] = 0.f;
        const float* dsCol = sDS + rt;
#pragma unroll 4
        for (int i = 0; i < Cf::RCH; ++i) {
          const int cc = part * Cf::RCH + ((i + vid * Cf::RS + part) & (Cf::RCH - 1));
          const float w = dsCol[cc * Cf::RowF];
          float hv[VW];
          lds_vec<VW>(hs_vec(rt + 1, rq, bwd_lane_of<N>(cc, rg)), hv);
#pragma unroll
          for (int v = 0; v < VW; ++v) acc[v] = fmaf(w, hv[v], acc[v]);
        }
#pragma unroll
        for (int s = Cf::RS / 2; s >= 1; s /= 2)
#pragma unroll
          for (int v = 0; v < VW; ++v) acc[v] += __shfl_xor_sync(0xffffffffu, acc[v], s);
        if (part == 0 && rt < tc) {
#pragma unroll
          for (int v = 0; v < VW; ++v)
            wsC_blk[(int64_t)(rg * NPT + rq * VW + v) * L + t0 + rt] = acc[v];
        }
      }
    }
    __syncthreads();

    // P4: the adjoint recurrence over the chunk, from its last step to its first
    {
      float pa4[4], pb4[4];
      if (fast_pairs) {
        // With the zero-order hold, h_t = Ā h_{t-1} + B̄ B u gives exactly
        //   dh_t/dΔ = A h_t + B u   and   dh_t/dA = Δ h_t + B u (Δ - B̄) / A.
        // Where the registers allow (kCarryH), the step uses that form: h_t is
        // the later iteration's h_{t-1} (for the chunk's last step the
        // recompute's final state) and the B u term of dA is summed undivided
        // (dA2q) and divided by A once at the end: 15 paired operations per
        // pair instead of 17.  Elsewhere it uses Ā (A h_{t-1}) + Ā B u.
        f2 htq[NP];
        if constexpr (kCarryH) {
#pragma unroll
          for (int q = 0; q < NP; ++q) htq[q] = hq[q];
        }
#pragma unroll 4
        for (int t = T - 1; t >= 0; --t) {
          const float dt = rDT[t], u = rU[t], ds = rDS[t];
          const f2 dt2 = pack2(dt, dt), u2 = pack2(u, u), ds2 = pack2(ds, ds);
          f2 Bq[NP], Cq[NP], hpq[NP], dbq[NP];
          lds_f2<NP>(sBt + t * Cf::RowBC + g * NPT, Bq);
          lds_f2<NP>(sCt + t * Cf::RowBC + g * NPT, Cq);
          hs_load_pairs(t, hpq);
          f2 du2 = pack2(0.f, 0.f), dd2 = pack2(0.f, 0.f);
#pragma unroll
          for (int q = 0; q < NP; ++q) {
            lq[q] = fma2(ds2, Cq[q], lq[q]);
            float x0, x1;
            unpack2(mul2(dt2, A2p[q]), x0, x1);
            const f2 a = pack2(ex2_fast(x0), ex2_fast(x1));
            const f2 bb = fma2(a, iAp[q], nIp[q]);               // (Ā - 1) / A
            const f2 x2v = mul2(lq[q], mul2(Bq[q], u2));          // λ B u
            const f2 lb = mul2(lq[q], bb);
            du2 = fma2(lb, Bq[q], du2);
            dbq[q] = mul2(lb, u2);
            if constexpr (kCarryH) {
              const f2 x1t = mul2(lq[q], htq[q]);                 // λ h_t
              dd2 = add2(fma2(Ajp[q], x1t, dd2), x2v);            // λ (A h_t + B u)
              dAq[q] = fma2(x1t, dt2, dAq[q]);                    // λ Δ h_t
              dA2q[q] = fma2(x2v, sub2(dt2, bb), dA2q[q]);        // λ B u (Δ - B̄)
              htq[q] = hpq[q];
            } else {
              const f2 da = mul2(dt2, a);                         // Δ Ā
              const f2 w = mul2(sub2(da, bb), iAp[q]);            // (Δ Ā - B̄) / A
              const f2 x1v = mul2(lq[q], hpq[q]);                 // λ h_{t-1}
              dd2 = fma2(a, fma2(Ajp[q], x1v, x2v), dd2);
              dAq[q] = fma2(x2v, w, fma2(x1v, da, dAq[q]));
            }
            lq[q] = mul2(lq[q], a);
          }
          hs_store_pairs(t + 1, dbq);
          float lo, hi;
          unpack2(du2, lo, hi);
          pa4[t & 3] = lo + hi;
          unpack2(dd2, lo, hi);
          pb4[t & 3] = lo + hi;
          if ((t & 3) == 0) {
            *reinterpret_cast<float4*>(sPa + bwd_pidx<N>(prow, t)) =
                make_float4(pa4[0], pa4[1], pa4[2], pa4[3]);
            *reinterpret_cast<float4*>(sPb + bwd_pidx<N>(prow, t)) =
                make_float4(pb4[0], pb4[1], pb4[2], pb4[3]);
          }
        }
      } else {
#pragma unroll 4
        for (int t = T - 1; t >= 0; --t) {
          const float dt = rDT[t], u = rU[t], ds = rDS[t];
          float hp[NPT], dbv[NPT], Bv[NPT], Cv[NPT];
#pragma unroll
          for (int q = 0; q < QN; ++q) lds_vec<VW>(hs_vec(t, q, tid), hp + q * VW);
          lds_vec<NPT>(sBt + t * Cf::RowBC + g * NPT, Bv);
          lds_vec<NPT>(sCt + t * Cf::RowBC + g * NPT, Cv);
          float du_p = 0.f, dd_p = 0.f;
#pragma unroll
          for (int j = 0; j < NPT; ++j) {
            const float Bn = Bv[j];
            lam[j] = fmaf(ds, Cv[j], lam[j]);
            // a = Ā, bb = B̄, w = dB̄/dA, sl = dB̄/dΔ
            float a, bb, w, sl;
            if (!precise) {
              a = ex2_fast(dt * Aj[j] * kLog2e);
              bb = fmaf(a, invA[j], -invA[j]);
              w = (dt * a - bb) * invA[j];
              sl = a;
            } else if (euler) {
              a = expf(dt * Aj[j]);
              bb = dt;
              w = 0.f;
              sl = 1.f;
            } else {
              const float x = dt * Aj[j];
              a = expf(x);
              bb = Aj[j] != 0.f ? expm1f(x) * invA[j] : dt;
              w = Aj[j] != 0.f ? (dt * a - bb) * invA[j] : 0.5f * dt * dt;
              sl = a;
            }
            const float x1 = lam[j] * hp[j];
            const float x2 = lam[j] * (Bn * u);
            const float lb = lam[j] * bb;
            du_p = fmaf(lb, Bn, du_p);
            dbv[j] = lb * u;
            dd_p = fmaf(a * Aj[j], x1, fmaf(sl, x2, dd_p));
            dAacc[j] = fmaf(x2, w, fmaf(x1, dt * a, dAacc[j]));
            lam[j] *= a;
          }
#pragma unroll
          for (int q = 0; q < QN; ++q) sts_vec<VW>(hs_vec(t + 1, q, tid), dbv + q * VW);
          pa4[t & 3] = du_p;
          pb4[t & 3] = dd_p;
          if ((t & 3) == 0) {
            *reinterpret_cast<float4*>(sPa + bwd_pidx<N>(prow, t)) =
                make_float4(pa4[0], pa4[1], pa4[2], pa4[3]);
            *reinterpret_cast<float4*>(sPb + bwd_pidx<N>(prow, t)) =
                make_float4(pb4[0], pb4[1], pb4[2], pb4[3]);
          }
        }
      }
    }
    __syncthreads();

    // P5: du, dΔraw, dbias; dB reduced over the block's channels
    {
      float du_[E], dd_[E];
#pragma unroll
      for (int j = 0; j < E; ++j) du_[j] = dd_[j] = 0.f;
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        if constexpr (E % 4 == 0) {
#pragma unroll
          for (int kq = 0; kq < E / 4; ++kq) {
            const int ix = bwd_pidx<N>(gg * CH + r, te + 4 * kq);
            const float4 a4 = *reinterpret_cast<const float4*>(sPa + ix);
            const float4 b4 = *reinterpret_cast<const float4*>(sPb + ix);
            du_[4 * kq] += a4.x; du_[4 * kq + 1] += a4.y; du_[4 * kq + 2] += a4.z; du_[4 * kq + 3] += a4.w;
            dd_[4 * kq] += b4.x; dd_[4 * kq + 1] += b4.y; dd_[4 * kq + 2] += b4.z; dd_[4 * kq + 3] += b4.w;
          }
        } else {
#pragma unroll
          for (int j = 0; j < E; ++j) {
            du_[j] += sPa[bwd_pidx<N>(gg * CH + r, te + j)];
            dd_[j] += sPb[bwd_pidx<N>(gg * CH + r, te + j)];
          }
        }
      }
      const float Dr = sD[r];
#pragma unroll
      for (int j = 0; j < E; ++j) {
        du_[j] = fmaf(sDS[r * Cf::RowF + te + j], Dr, du_[j]);
        dd_[j] *= sg[j];
        if (te + j < tc) dbias_acc += dd_[j];
      }
      if (row_ok) {
        IO* dup = static_cast<IO*>(p.du) + io_row + (t0 + te) * io_ts;
        IO* ddp = static_cast<IO*>(p.ddelta) + io_row + (t0 + te) * io_ts;
        bool done = false;
        if constexpr (E % 4 == 0) {
          if (vec && te + E <= tc) {
            vecio<IO, E>::store(dup, du_);
            vecio<IO, E>::store(ddp, dd_);
            done = true;
          }
        }
        if (!done) {
#pragma unroll
          for (int j = 0; j < E; ++j) {
            if (te + j < tc) {
              dup[j * io_ts] = io_traits<IO>::from_f32(du_[j]);
              ddp[j * io_ts] = io_traits<IO>::from_f32(dd_[j]);
            }
          }
        }
      }
#pragma unroll
      for (int kv = 0; kv < Cf::VPT; ++kv) {
        const int vid = tid / Cf::RS + kv * (kBwdThreads / Cf::RS);
        const int rt = vid / (G * QN), rg = (vid % (G * QN)) / QN, rq = vid % QN;
        float acc[VW];
#pragma unroll
        for (int v = 0; v < VW; ++v) acc[v] = 0.f;
#pragma unroll 4
        for (int i = 0; i < Cf::RCH; ++i) {
          const int cc = part * Cf::RCH + ((i + vid * Cf::RS + part) & (Cf::RCH - 1));
          float hv[VW];
          lds_vec<VW>(hs_vec(rt + 1, rq, bwd_lane_of<N>(cc, rg)), hv);
#pragma unroll
          for (int v = 0; v < VW; ++v) acc[v] += hv[v];
        }
#pragma unroll
        for (int s = Cf::RS / 2; s >= 1; s /= 2)
#pragma unroll
          for (int v = 0; v < VW; ++v) acc[v] += __shfl_xor_sync(0xffffffffu, acc[v], s);
        if (part == 0 && rt < tc) {
#pragma unroll
          for (int v = 0; v < VW; ++v)
            wsB_blk[(int64_t)(rg * NPT + rq * VW + v) * L + t0 + rt] = acc[v];
        }
      }
    }
    __syncthreads();
  }

  // per-channel results
  if (fast_pairs) {
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      unpack2(lq[q], lam[2 * q], lam[2 * q + 1]);
      unpack2(kCarryH ? fma2(dA2q[q], iAp[q], dAq[q]) : dAq[q], dAacc[2 * q], dAacc[2 * q + 1]);
    }
  }
  // this segment's slices of the per-batch-row sums; d init_state from the first
  const int64_t segoff = (int64_t)seg * p.batch * p.dim;
  if (chan_ok) {
    const int64_t st = (b * p.dim + d) * N + g * NPT;
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      p.ws_A[segoff * N + st + j] = dAacc[j];
      if (p.d_init_state && seg == 0) p.d_init_state[st + j] = lam[j];
    }
  }
#pragma unroll
  for (int s = TPR / 2; s >= 1; s /= 2) {
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, s);
    dbias_acc += __shfl_xor_sync(0xffffffffu, dbias_acc, s);
  }
  if (te == 0 && row_ok) {
    p.ws_D[segoff + b * p.dim + d0 + r] = dD_acc;
    p.ws_bias[segoff + b * p.dim + d0 + r] = dbias_acc;
  }
}

// ---------------------------------------------------------------------------
// Adjoint carries of a split sequence
// ---------------------------------------------------------------------------
// The adjoint is linear in what enters a segment from the right: leaving segment
// k it is (Π_t Ā_t) λ_in + l_k with Π_t Ā_t = exp(A ΣΔ_k), where l_k is what
// leaves when λ_in = 0.  This kernel computes l_k and ΣΔ_k for segments 1 ..
// nseg-1 (index k-1 of acarry_l / acarry_s); the backward kernel of segment s
// starts from d final_state folded through segments nseg-1 .. s+1.  Each step,
// from a segment's last to its first, is the adjoint sweep's own: λ += ds_t C_t,
// then λ *= Ā_t.  A channel's states sit on G lanes of NPT as in the backward
// kernel, in blocks of two warps (64 / G channels); a chunk of TT steps of Δ
// and ds is staged per channel in shared memory, C per step, the next chunk's
// raw inputs in flight in registers meanwhile.
constexpr int kAdjThreads = 64;  // two warps a block: many small blocks keep loads in flight

template <int N> struct AdjCfg {
  using Cf = BwdCfg<N>;
  static constexpr int NPT = Cf::NPT, G = Cf::G, CH = kAdjThreads / G;
  // steps per chunk: at most 8 channel steps of each input and 16 floats of C a thread
  static constexpr int TT = (512 / CH < 1024 / N) ? 512 / CH : 1024 / N;
  static constexpr int E = CH * TT / kAdjThreads;   // channel steps a thread loads
  static constexpr int TPR = TT / E;                // threads per channel row
  static constexpr int PER = (TT * N + kAdjThreads - 1) / kAdjThreads;
  static constexpr int RowF = TT + 1;
  static_assert(CH >= 1 && E >= 1 && E <= 8 && TPR * E == TT && PER <= 16, "tiling");
};

template <typename IO, int N>
__global__ void __launch_bounds__(kAdjThreads) adjoint_carry_kernel(const BwdArgs p) {
  using Cf = AdjCfg<N>;
  constexpr int NPT = Cf::NPT, CH = Cf::CH, TT = Cf::TT, E = Cf::E, TPR = Cf::TPR, PER = Cf::PER;
  __shared__ float sDT[CH * Cf::RowF];
  __shared__ float sDS[CH * Cf::RowF];
  __shared__ float sC[N * (TT + 1)];  // [n][t]: staged along t without bank conflicts
  __shared__ float sBias[CH];

  const int tid = threadIdx.x;
  const int g = tid / CH, c = tid % CH;  // a warp: consecutive channels of one state group
  const int64_t b = blockIdx.y;
  const int64_t d0 = (int64_t)blockIdx.x * CH;
  const int64_t d = d0 + c;
  const bool chan_ok = d < p.dim;
  const int nrows = (int)min64(CH, p.dim - d0);
  const int64_t L = p.L;
  const int seg = blockIdx.z + 1;
  const int64_t s0 = (int64_t)seg * p.seg_len;
  const int64_t s1 = min64(L, s0 + p.seg_len);
  const int nck = (int)((s1 - s0 + TT - 1) / TT);
  // loads: channel rows of L steps (E consecutive steps a thread), or steps dim
  // apart in (batch, L, dim) (consecutive channels across a warp)
  const bool bld = p.bld != 0;
  const int r = bld ? tid % CH : tid / TPR;
  const int te = bld ? (tid / CH) * E : (tid % TPR) * E;
  const bool row_ok = r < nrows;
  const int64_t io_row = bld ? b * L * p.dim + d0 + (row_ok ? r : 0)
                             : (b * p.dim + d0 + (row_ok ? r : 0)) * L;
  const int64_t io_ts = bld ? p.dim : 1;
  constexpr int kVecBytes = (sizeof(IO) == 2 && E == 4) ? 8 : 16;
  const bool vec = !bld && E % 4 == 0 && (L * (int64_t)sizeof(IO)) % kVecBytes == 0;

  for (int i = tid; i < CH; i += kAdjThreads)
    sBias[i] = (p.bias && d0 + i < p.dim) ? p.bias[d0 + i] : 0.f;
  float Aj[NPT], A2[NPT];
  bool zeroA = false;
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    Aj[j] = chan_ok ? p.A[d * N + g * NPT + j] : -1.f;
    A2[j] = Aj[j] * kLog2e;
    zeroA |= Aj[j] == 0.f;
  }
  // the flavour of the backward kernel's adjoint sweep (block-uniform)
  const bool precise = __syncthreads_or(zeroA) || p.force_precise || p.euler;
  const bool sp = p.softplus != 0;

  float rdl[E], rdy[E], rz[E], rc[PER];
  auto fetch = [&](int kk) {
    const int64_t t0 = s0 + (int64_t)kk * TT;
    const int tc = (int)min64(TT, s1 - t0);
    const int64_t gi = io_row + (t0 + te) * io_ts;
    bool done = false;
    if constexpr (E % 4 == 0) {
      if (row_ok && vec && te + E <= tc) {
        vecio<IO, E>::load(static_cast<const IO*>(p.delta) + gi, rdl);
        vecio<IO, E>::load(static_cast<const IO*>(p.dy) + gi, rdy);
        if (p.z) vecio<IO, E>::load(static_cast<const IO*>(p.z) + gi, rz);
        done = true;
      }
    }
    if (!done) {
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const bool ok = row_ok && te + j < tc;
        const int64_t gj = gi + j * io_ts;
        rdl[j] = ok ? ld_io<IO>(p.delta, gj) : 0.f;
        rdy[j] = ok ? ld_io<IO>(p.dy, gj) : 0.f;
        rz[j] = (ok && p.z) ? ld_io<IO>(p.z, gj) : 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = tid + i * kAdjThreads;  // (n, t) of the chunk's C tile
      const int n = e / TT, t = e - n * TT;
      const bool ok = (TT * N % kAdjThreads == 0 || e < TT * N) && t < tc;
      rc[i] = ok ? p.C[(b * N + n) * L + t0 + t] : 0.f;
    }
  };

  float lam[NPT];
#pragma unroll
  for (int j = 0; j < NPT; ++j) lam[j] = 0.f;
  float sdt = 0.f;
  if (nck > 0) fetch(nck - 1);
  for (int kk = nck - 1; kk >= 0; --kk) {
    const int64_t t0 = s0 + (int64_t)kk * TT;
    const int tc = (int)min64(TT, s1 - t0);
    __syncthreads();  // the previous chunk's readers are done
    {
      const float bias = sBias[r];
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const bool ok = row_ok && te + j < tc;
        const float x = rdl[j] + bias;
        const float dt = sp ? (precise ? softplus_precise(x) : softplus_fast(x)) : x;
        const float gate = p.z ? (precise ? silu_precise(rz[j]) : silu_fast(rz[j])) : 1.f;
        sDT[r * Cf::RowF + te + j] = ok ? dt : 0.f;
        sDS[r * Cf::RowF + te + j] = ok ? rdy[j] * gate : 0.f;
      }
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int e = tid + i * kAdjThreads;
        if (TT * N % kAdjThreads == 0 || e < TT * N) {
          const int n = e / TT, t = e - n * TT;
          sC[n * (TT + 1) + t] = rc[i];
        }
      }
    }
    __syncthreads();
    if (kk > 0) fetch(kk - 1);
    const float* rDT = sDT + c * Cf::RowF;
    const float* rDS = sDS + c * Cf::RowF;
    const float* rC = sC + g * NPT * (TT + 1);
    if (precise) {
      for (int t = TT - 1; t >= 0; --t) {
        const float dt = rDT[t], ds = rDS[t];
        sdt += dt;
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
          lam[j] = fmaf(ds, rC[j * (TT + 1) + t], lam[j]);
          lam[j] *= expf(dt * Aj[j]);
        }
      }
    } else {
#pragma unroll 4
      for (int t = TT - 1; t >= 0; --t) {
        const float dt = rDT[t], ds = rDS[t];
        sdt += dt;
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
          lam[j] = fmaf(ds, rC[j * (TT + 1) + t], lam[j]);
          lam[j] *= ex2_fast(dt * A2[j]);
        }
      }
    }
  }
  if (chan_ok) {
    const int64_t row = b * p.dim + d;
    const int64_t o = (int64_t)(seg - 1) * p.batch * p.dim + row;
#pragma unroll
    for (int j = 0; j < NPT; ++j) p.acarry_l[o * N + g * NPT + j] = lam[j];
    if (g == 0) p.acarry_s[o] = sdt;
  }
}

// Adds the per-block partial sums in a fixed order: dB, dC over the channel
// blocks of each batch row; dA, dD, dbias over the segments and the batch.
__global__ void bwd_reduce_kernel(const BwdArgs p, int64_t N) {
  const int64_t nbc = p.batch * N * p.L;
  const int64_t nA = p.dim * N;
  const int64_t total = 2 * nbc + nA + 2 * p.dim;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < 2 * nbc) {
      const bool isC = i >= nbc;
      const int64_t e = isC ? i - nbc : i;        // (b, n, t)
      const int64_t bb = e / (N * p.L), nt = e - bb * N * p.L;
      const float* ws = (isC ? p.ws_C : p.ws_B) + bb * p.nblk * N * p.L + nt;
      float s = 0.f;
      for (int64_t k = 0; k < p.nblk; ++k) s += ws[k * N * p.L];
      (isC ? p.dC : p.dB)[e] = s;
    } else if (i < 2 * nbc + nA) {
      const int64_t e = i - 2 * nbc;              // (d, n)
      float s = 0.f;
      for (int64_t sb = 0; sb < p.nseg * p.batch; ++sb) s += p.ws_A[sb * nA + e];
      p.dA[e] = s;
    } else {
      const int64_t e = i - 2 * nbc - nA;
      const bool isBias = e >= p.dim;
      const int64_t dd = isBias ? e - p.dim : e;
      float* out = isBias ? p.d_bias : p.dD;
      if (!out) continue;
      const float* ws = isBias ? p.ws_bias : p.ws_D;
      float s = 0.f;
      for (int64_t sb = 0; sb < p.nseg * p.batch; ++sb) s += ws[sb * p.dim + dd];
      out[dd] = s;
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
template <int N> static void bwd_geom(int64_t dim, int64_t L, int64_t& nblk, int64_t& nch) {
  nblk = (dim + BwdCfg<N>::CH - 1) / BwdCfg<N>::CH;
  nch = (L + BwdCfg<N>::T - 1) / BwdCfg<N>::T;
}

static bool bwd_geometry(int64_t N, int64_t dim, int64_t L, int64_t& nblk, int64_t& nch) {
  switch (N) {
    case 1: bwd_geom<1>(dim, L, nblk, nch); return true;
    case 2: bwd_geom<2>(dim, L, nblk, nch); return true;
    case 4: bwd_geom<4>(dim, L, nblk, nch); return true;
    case 8: bwd_geom<8>(dim, L, nblk, nch); return true;
    case 16: bwd_geom<16>(dim, L, nblk, nch); return true;
    case 32: bwd_geom<32>(dim, L, nblk, nch); return true;
    case 64: bwd_geom<64>(dim, L, nblk, nch); return true;
    case 128: bwd_geom<128>(dim, L, nblk, nch); return true;
    default: return false;
  }
}

static size_t al256(size_t x) { return (x + 255) / 256 * 256; }

int bwd_chunk(int64_t N) {
  switch (N) {
    case 1: return BwdCfg<1>::T;
    case 2: return BwdCfg<2>::T;
    case 4: return BwdCfg<4>::T;
    case 8: return BwdCfg<8>::T;
    case 16: return BwdCfg<16>::T;
    case 32: return BwdCfg<32>::T;
    case 64: return BwdCfg<64>::T;
    case 128: return BwdCfg<128>::T;
    default: return 0;
  }
}

// Resident backward blocks per SM (the kernel's launch bound).
static int bwd_resident(int64_t N) {
  switch (N) {
    case 1: return BwdCfg<1>::MINB;
    case 2: return BwdCfg<2>::MINB;
    case 4: return BwdCfg<4>::MINB;
    case 8: return BwdCfg<8>::MINB;
    case 16: return BwdCfg<16>::MINB;
    case 32: return BwdCfg<32>::MINB;
    case 64: return BwdCfg<64>::MINB;
    case 128: return BwdCfg<128>::MINB;
    default: return 1;
  }
}

BwdLayout bwd_layout(int64_t batch, int64_t dim, int64_t L, int64_t N, int sm_count) {
  BwdLayout w{};
  if (!bwd_geometry(N, dim, L, w.nblk, w.nch)) return w;
  // Split the sequence when the (channel block, batch row) blocks fill less than
  // half of one wave of resident blocks: as many segments as still fit in one
  // wave (a second, mostly idle wave would cost a whole segment's time), each of
  // at least kBwdMinSeg steps and a multiple of 16 (the forward's and every
  // backward chunk length), at most 64.
  w.nseg = 1;
  w.seg_len = L > 0 ? L : 1;
  const int64_t blocks = w.nblk * batch;
  const int64_t wave = (int64_t)sm_count * bwd_resident(N);
  if (L > 0 && blocks > 0 && 2 * blocks <= wave) {
    int64_t nseg = wave / blocks;
    if (nseg > L / kBwdMinSeg) nseg = L / kBwdMinSeg;
    if (nseg > 64) nseg = 64;
    if (nseg >= 2) {
      int64_t seg_len = (L + nseg - 1) / nseg;
      seg_len = (seg_len + 15) / 16 * 16;
      nseg = (L + seg_len - 1) / seg_len;
      if (nseg >= 2) {
        w.nseg = (int)nseg;
        w.seg_len = seg_len;
      }
    }
  }
  const size_t B_ = (size_t)batch, D_ = (size_t)dim, N_ = (size_t)N, L_ = (size_t)L;
  const size_t S_ = (size_t)w.nseg, rows = B_ * D_;
  w.o_ckpt = 0;
  w.o_B = w.o_ckpt + al256(B_ * (size_t)w.nch * D_ * N_ * 4);
  w.o_C = w.o_B + al256(B_ * (size_t)w.nblk * N_ * L_ * 4);
  w.o_A = w.o_C + al256(B_ * (size_t)w.nblk * N_ * L_ * 4);
  w.o_D = w.o_A + al256(S_ * rows * N_ * 4);
  w.o_bias = w.o_D + al256(S_ * rows * 4);
  w.o_fh = w.o_bias + al256(S_ * rows * 4);
  w.o_fs = w.o_fh + al256((S_ - 1) * rows * N_ * 4);
  w.o_al = w.o_fs + al256((S_ - 1) * rows * 4);
  w.o_as = w.o_al + al256((S_ - 1) * rows * N_ * 4);
  w.bytes = w.o_as + al256((S_ - 1) * rows * 4);
  return w;
}

template <typename IO, int N>
static cudaError_t bwd_typed(const BwdArgs& a, cudaStream_t stream) {
  using Cf = BwdCfg<N>;
  constexpr size_t bytes = BwdSmem<N>::kBytes;
  auto kern = scan_bwd_kernel<IO, N>;
  static int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  const unsigned nblk = (unsigned)((a.dim + Cf::CH - 1) / Cf::CH);
  if (a.nseg > 1) {
    const unsigned ablk = (unsigned)((a.dim + AdjCfg<N>::CH - 1) / AdjCfg<N>::CH);
    adjoint_carry_kernel<IO, N><<<dim3(ablk, (unsigned)a.batch, (unsigned)(a.nseg - 1)), kAdjThreads,
                                  0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(nblk, (unsigned)a.batch, (unsigned)a.nseg);
  kern<<<grid, kBwdThreads, bytes, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t total = 2 * a.batch * N * a.L + a.dim * N + 2 * a.dim;
  const int64_t blocks = (total + 255) / 256;
  bwd_reduce_kernel<<<(unsigned)(blocks < 148 * 16 ? blocks : 148 * 16), 256, 0, stream>>>(a, N);
  return cudaGetLastError();
}

template <typename IO>
static cudaError_t bwd_io(const BwdArgs& a, int64_t N, cudaStream_t stream) {
  switch (N) {
    case 1: return bwd_typed<IO, 1>(a, stream);
    case 2: return bwd_typed<IO, 2>(a, stream);
    case 4: return bwd_typed<IO, 4>(a, stream);
    case 8: return bwd_typed<IO, 8>(a, stream);
    case 16: return bwd_typed<IO, 16>(a, stream);
    case 32: return bwd_typed<IO, 32>(a, stream);
    case 64: return bwd_typed<IO, 64>(a, stream);
    case 128: return bwd_typed<IO, 128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t bwd_launch(const BwdArgs& a, int64_t N, int io_dtype, cudaStream_t stream) {
  if (io_dtype == 0) return bwd_io<float>(a, N, stream);
  return bwd_io<__nv_bfloat16>(a, N, stream);
}

}  // namespace ssm
