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
//   dΔraw_t = dΔ_t σ(Δraw_t + bias) (softplus), dbias += dΔraw,  dD += ds u,
//   dh_{-1} = Ā_0 λ_0
// where B̄ = (Ā - 1)/A is the scalar zero-order-hold factor (A = 0: Δ, and
// (Δ Ā - B̄)/A takes its limit Δ²/2).
//
// Design (B300).  A block owns CH channels of one batch row with the same
// lane layout as the forward kernel: G lanes per channel, NPT states per lane
// in registers.  It walks the sequence twice:
//  1. forward, recurrence only, storing the state at the start of every chunk
//     of T steps to a checkpoint workspace (N floats per channel per chunk);
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

template <int N> struct BwdCfg {
  static constexpr int NPT = N <= 4 ? N : (N <= 16 ? 4 : N / 4);  // states per lane
  static constexpr int G = N / NPT;                                // lanes per channel
  static constexpr int CH = kBwdThreads / G;                       // channels per block
  static constexpr int T = NPT <= 4 ? 16 : (NPT == 8 ? 8 : 4);     // steps per chunk
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
  // channel reductions: threads per reduced vector and channels per thread
  static constexpr int RS = kBwdThreads / (T * G * QN);
  static constexpr int RCH = CH / RS;
  static_assert(G * NPT == N && E >= 1 && TPR <= 4 && RS >= 1 && RCH * RS == CH, "tiling");
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

// ---------------------------------------------------------------------------
// The per-block kernel
// ---------------------------------------------------------------------------
template <typename IO, int N>
__global__ void __launch_bounds__(kBwdThreads, 3) scan_bwd_kernel(const BwdArgs p) {
  using Cf = BwdCfg<N>;
  using S = BwdSmem<N>;
  constexpr int NPT = Cf::NPT, CH = Cf::CH, T = Cf::T, E = Cf::E, TPR = Cf::TPR;
  constexpr int VW = Cf::VW, QN = Cf::QN, G = Cf::G;
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
  // this thread's row and steps in the per-step (cooperative) phases
  const int r = tid / TPR, te = (tid % TPR) * E;
  const bool row_ok = r < nrows;
  const int64_t io_row = (b * p.dim + d0 + (row_ok ? r : 0)) * L;

  for (int i = tid; i < CH; i += kBwdThreads) {
    const bool ok = d0 + i < p.dim;
    sBias[i] = (p.bias && ok) ? p.bias[d0 + i] : 0.f;
    sD[i] = (p.D && ok) ? p.D[d0 + i] : 0.f;
  }
  float Aj[NPT], A2[NPT], invA[NPT];
  bool zeroA = false;
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    Aj[j] = chan_ok ? p.A[d * N + g * NPT + j] : -1.f;
    zeroA |= Aj[j] == 0.f;
    A2[j] = Aj[j] * kLog2e;
    invA[j] = Aj[j] != 0.f ? 1.f / Aj[j] : 0.f;
  }
  const bool precise = __syncthreads_or(zeroA) || p.force_precise;
  const bool sp = p.softplus != 0;

  // one recurrence step of this lane (states in h), for recompute and the checkpoint sweep
  auto lane_step = [&](float (&h)[NPT], float dt, float u, const float* Brow) {
    float Bv[NPT];
    lds_vec<NPT>(Brow, Bv);
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const float Bn = Bv[j];
      if (!precise) {
        const float a = ex2_fast(dt * A2[j]);
        const float v = -Bn * u * invA[j];  // fixed point -B u / A
        h[j] = fmaf(a, h[j] - v, v);
      } else {
        const float x = dt * Aj[j];
        const float bb = Aj[j] != 0.f ? expm1f(x) * invA[j] : dt;
        h[j] = fmaf(expf(x), h[j], bb * (Bn * u));
      }
    }
  };
  // Δ, u (and, with `full`, ds, z, dy, σ) of this thread's E steps of chunk k
  auto load_steps = [&](int k, bool full, float (&dyv)[E], float (&zz)[E], float (&sg)[E]) {
    const int64_t t0 = (int64_t)k * T;
    const int tc = (int)min64(T, L - t0);
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int t = te + j;
      const bool ok = row_ok && t < tc;
      const int64_t gi = io_row + t0 + t;
      float dt = 0.f, u = 0.f, ds = 0.f;
      dyv[j] = 0.f;
      zz[j] = 0.f;
      sg[j] = 1.f;
      if (ok) {
        u = ld_io<IO>(p.u, gi);
        const float x = ld_io<IO>(p.delta, gi) + sBias[r];
        dt = sp ? (precise ? softplus_precise(x) : softplus_fast(x)) : x;
        if (full) {
          if (sp) sg[j] = precise ? sigmoid_precise(x) : sigmoid_fast(x);
          dyv[j] = ld_io<IO>(p.dy, gi);
          float gate = 1.f;
          if (p.z) {
            zz[j] = ld_io<IO>(p.z, gi);
            gate = precise ? silu_precise(zz[j]) : silu_fast(zz[j]);
          }
          ds = dyv[j] * gate;
        }
      }
      sDT[r * Cf::RowF + t] = dt;
      sU[r * Cf::RowF + t] = u;
      if (full) sDS[r * Cf::RowF + t] = ds;
    }
    // B (and C) transposed to [t][n]; zero past the end of the sequence
    for (int e = tid; e < N * T; e += kBwdThreads) {
      const int n = e / T, t = e - n * T;
      const bool ok = t < tc;
      const int64_t bi = (b * N + n) * L + t0 + t;
      sBt[t * Cf::RowBC + n] = ok ? p.B[bi] : 0.f;
      if (full) sCt[t * Cf::RowBC + n] = ok ? p.C[bi] : 0.f;
    }
  };
  auto hs_vec = [&](int slot, int q, int lane) {
    return sHs + ((slot * QN + q) * kBwdThreads + lane) * VW;
  };
  auto ckpt_ptr = [&](int k) {
    return p.ckpt + ((b * nch + k) * p.dim + d) * N + g * NPT;
  };

  // ---------------- sweep 1: chunk-start states ----------------
  float h[NPT];
#pragma unroll
  for (int j = 0; j < NPT; ++j)
    h[j] = (p.init_state && chan_ok) ? p.init_state[(b * p.dim + d) * N + g * NPT + j] : 0.f;
  {
    float dyv[E], zz[E], sg[E];
    for (int k = 0; k < nch; ++k) {
      if (chan_ok) {
        float* cp = ckpt_ptr(k);
#pragma unroll
        for (int j = 0; j < NPT; ++j) cp[j] = h[j];
      }
      load_steps(k, false, dyv, zz, sg);
      __syncthreads();
#pragma unroll 4
      for (int t = 0; t < T; ++t)
        lane_step(h, sDT[c * Cf::RowF + t], sU[c * Cf::RowF + t], sBt + t * Cf::RowBC + g * NPT);
      __syncthreads();
    }
  }

  // ---------------- sweep 2: adjoint, chunk by chunk from the end ----------------
  float lam[NPT], dAacc[NPT];
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    lam[j] = (p.d_final_state && chan_ok) ? p.d_final_state[(b * p.dim + d) * N + g * NPT + j] : 0.f;
    dAacc[j] = 0.f;
  }
  float dD_acc = 0.f, dbias_acc = 0.f;
  float* wsB_blk = p.ws_B + ((b * p.nblk + blk) * N) * L;
  float* wsC_blk = p.ws_C + ((b * p.nblk + blk) * N) * L;

  for (int k = nch - 1; k >= 0; --k) {
    const int64_t t0 = (int64_t)k * T;
    const int tc = (int)min64(T, L - t0);
    // P1: per-step inputs of the chunk; this lane's start state
    float dyv[E], zz[E], sg[E];
    load_steps(k, true, dyv, zz, sg);
    if (chan_ok) {
      const float* cp = ckpt_ptr(k);
#pragma unroll
      for (int j = 0; j < NPT; ++j) h[j] = cp[j];
    } else {
#pragma unroll
      for (int j = 0; j < NPT; ++j) h[j] = 0.f;
    }
    __syncthreads();

    // P2: recompute the chunk's states into slots 1..T, readout partials
    {
#pragma unroll
      for (int q = 0; q < QN; ++q) sts_vec<VW>(hs_vec(0, q, tid), h + q * VW);
      float acc4[4];
#pragma unroll 4
      for (int t = 0; t < T; ++t) {
        const float* Brow = sBt + t * Cf::RowBC + g * NPT;
        const float* Crow = sCt + t * Cf::RowBC + g * NPT;
        lane_step(h, sDT[c * Cf::RowF + t], sU[c * Cf::RowF + t], Brow);
        float Cv[NPT];
        lds_vec<NPT>(Crow, Cv);
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < NPT; ++j) s = fmaf(Cv[j], h[j], s);
#pragma unroll
        for (int q = 0; q < QN; ++q) sts_vec<VW>(hs_vec(t + 1, q, tid), h + q * VW);
        acc4[t & 3] = s;
        if ((t & 3) == 3)
          *reinterpret_cast<float4*>(sPa + bwd_pidx<N>(prow, t - 3)) =
              make_float4(acc4[0], acc4[1], acc4[2], acc4[3]);
      }
    }
    __syncthreads();

    // P3: dz (needs s = Σ_g partials + D u), dD; dC reduced over the block's channels
    {
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const int t = te + j;
        float s = 0.f;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) s += sPa[bwd_pidx<N>(gg * CH + r, t)];
        const float u = sU[r * Cf::RowF + t];
        s = fmaf(sD[r], u, s);
        dD_acc = fmaf(sDS[r * Cf::RowF + t], u, dD_acc);  // zero past the end
        if (p.z && row_ok && t < tc) {
          const float zg = zz[j];
          const float sz = precise ? sigmoid_precise(zg) : sigmoid_fast(zg);
          const float dz = dyv[j] * s * sz * fmaf(zg, 1.f - sz, 1.f);
          static_cast<IO*>(p.dz)[io_row + t0 + t] = io_traits<IO>::from_f32(dz);
        }
      }
      // dC[t][n] = Σ_c ds[c][t] h_t[c][n]
      const int vid = tid / Cf::RS, part = tid % Cf::RS;
      const int t = vid / (G * QN), gq = vid % (G * QN), gg = gq / QN, q = gq % QN;
      float acc[VW];
#pragma unroll
      for (int v = 0; v < VW; ++v) acc[v] = 0.f;
#pragma unroll 4
      for (int i = 0; i < Cf::RCH; ++i) {
        const int cc = part * Cf::RCH + (i + vid * Cf::RS + part) % Cf::RCH;
        const float w = sDS[cc * Cf::RowF + t];
        float hv[VW];
        lds_vec<VW>(hs_vec(t + 1, q, bwd_lane_of<N>(cc, gg)), hv);
#pragma unroll
        for (int v = 0; v < VW; ++v) acc[v] = fmaf(w, hv[v], acc[v]);
      }
#pragma unroll
      for (int s = Cf::RS / 2; s >= 1; s /= 2)
#pragma unroll
        for (int v = 0; v < VW; ++v) acc[v] += __shfl_xor_sync(0xffffffffu, acc[v], s);
      if (part == 0 && t < tc) {
#pragma unroll
        for (int v = 0; v < VW; ++v) wsC_blk[(int64_t)(gg * NPT + q * VW + v) * L + t0 + t] = acc[v];
      }
    }
    __syncthreads();

    // P4: the adjoint recurrence over the chunk, from its last step to its first
    {
      float pa4[4], pb4[4];
#pragma unroll 4
      for (int t = T - 1; t >= 0; --t) {
        const float dt = sDT[c * Cf::RowF + t];
        const float u = sU[c * Cf::RowF + t];
        const float ds = sDS[c * Cf::RowF + t];
        const float* Brow = sBt + t * Cf::RowBC + g * NPT;
        const float* Crow = sCt + t * Cf::RowBC + g * NPT;
        float hp[NPT], dbv[NPT], Bv[NPT], Cv[NPT];
#pragma unroll
        for (int q = 0; q < QN; ++q) lds_vec<VW>(hs_vec(t, q, tid), hp + q * VW);
        lds_vec<NPT>(Brow, Bv);
        lds_vec<NPT>(Crow, Cv);
        float du_p = 0.f, dd_p = 0.f;
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
          const float Bn = Bv[j];
          lam[j] = fmaf(ds, Cv[j], lam[j]);
          float a, bb, w;
          if (!precise) {
            a = ex2_fast(dt * A2[j]);
            bb = fmaf(a, invA[j], -invA[j]);       // (Ā - 1) / A
            w = (dt * a - bb) * invA[j];           // (Δ Ā - B̄) / A
          } else {
            const float x = dt * Aj[j];
            a = expf(x);
            bb = Aj[j] != 0.f ? expm1f(x) * invA[j] : dt;
            w = Aj[j] != 0.f ? (dt * a - bb) * invA[j] : 0.5f * dt * dt;
          }
          const float x1 = lam[j] * hp[j];
          const float x2 = lam[j] * (Bn * u);
          const float lb = lam[j] * bb;
          du_p = fmaf(lb, Bn, du_p);
          dbv[j] = lb * u;
          dd_p = fmaf(a, fmaf(Aj[j], x1, x2), dd_p);
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
    __syncthreads();

    // P5: du, dΔraw, dbias; dB reduced over the block's channels
    {
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const int t = te + j;
        float du = 0.f, dd = 0.f;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          du += sPa[bwd_pidx<N>(gg * CH + r, t)];
          dd += sPb[bwd_pidx<N>(gg * CH + r, t)];
        }
        du = fmaf(sDS[r * Cf::RowF + t], sD[r], du);
        const float dx = dd * sg[j];
        if (row_ok && t < tc) {
          static_cast<IO*>(p.du)[io_row + t0 + t] = io_traits<IO>::from_f32(du);
          static_cast<IO*>(p.ddelta)[io_row + t0 + t] = io_traits<IO>::from_f32(dx);
          dbias_acc += dx;
        }
      }
      const int vid = tid / Cf::RS, part = tid % Cf::RS;
      const int t = vid / (G * QN), gq = vid % (G * QN), gg = gq / QN, q = gq % QN;
      float acc[VW];
#pragma unroll
      for (int v = 0; v < VW; ++v) acc[v] = 0.f;
#pragma unroll 4
      for (int i = 0; i < Cf::RCH; ++i) {
        const int cc = part * Cf::RCH + (i + vid * Cf::RS + part) % Cf::RCH;
        float hv[VW];
        lds_vec<VW>(hs_vec(t + 1, q, bwd_lane_of<N>(cc, gg)), hv);
#pragma unroll
        for (int v = 0; v < VW; ++v) acc[v] += hv[v];
      }
#pragma unroll
      for (int s = Cf::RS / 2; s >= 1; s /= 2)
#pragma unroll
        for (int v = 0; v < VW; ++v) acc[v] += __shfl_xor_sync(0xffffffffu, acc[v], s);
      if (part == 0 && t < tc) {
#pragma unroll
        for (int v = 0; v < VW; ++v) wsB_blk[(int64_t)(gg * NPT + q * VW + v) * L + t0 + t] = acc[v];
      }
    }
    __syncthreads();
  }

  // per-channel results
  if (chan_ok) {
    const int64_t st = (b * p.dim + d) * N + g * NPT;
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      p.ws_A[st + j] = dAacc[j];
      if (p.d_init_state) p.d_init_state[st + j] = lam[j];
    }
  }
#pragma unroll
  for (int s = TPR / 2; s >= 1; s /= 2) {
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, s);
    dbias_acc += __shfl_xor_sync(0xffffffffu, dbias_acc, s);
  }
  if (te == 0 && row_ok) {
    p.ws_D[b * p.dim + d0 + r] = dD_acc;
    p.ws_bias[b * p.dim + d0 + r] = dbias_acc;
  }
}

// Adds the per-block partial sums in a fixed order: dB, dC over the channel
// blocks of each batch row; dA, dD, dbias over the batch.
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
      for (int64_t bb = 0; bb < p.batch; ++bb) s += p.ws_A[bb * nA + e];
      p.dA[e] = s;
    } else {
      const int64_t e = i - 2 * nbc - nA;
      const bool isBias = e >= p.dim;
      const int64_t dd = isBias ? e - p.dim : e;
      float* out = isBias ? p.d_bias : p.dD;
      if (!out) continue;
      const float* ws = isBias ? p.ws_bias : p.ws_D;
      float s = 0.f;
      for (int64_t bb = 0; bb < p.batch; ++bb) s += ws[bb * p.dim + dd];
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
    default: return false;
  }
}

static size_t al256(size_t x) { return (x + 255) / 256 * 256; }

BwdLayout bwd_layout(int64_t batch, int64_t dim, int64_t L, int64_t N) {
  BwdLayout w{};
  if (!bwd_geometry(N, dim, L, w.nblk, w.nch)) return w;
  const size_t B_ = (size_t)batch, D_ = (size_t)dim, N_ = (size_t)N, L_ = (size_t)L;
  w.o_ckpt = 0;
  w.o_B = w.o_ckpt + al256(B_ * (size_t)w.nch * D_ * N_ * 4);
  w.o_C = w.o_B + al256(B_ * (size_t)w.nblk * N_ * L_ * 4);
  w.o_A = w.o_C + al256(B_ * (size_t)w.nblk * N_ * L_ * 4);
  w.o_D = w.o_A + al256(B_ * D_ * N_ * 4);
  w.o_bias = w.o_D + al256(B_ * D_ * 4);
  w.bytes = w.o_bias + al256(B_ * D_ * 4);
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
  const dim3 grid((unsigned)((a.dim + Cf::CH - 1) / Cf::CH), (unsigned)a.batch);
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
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t bwd_launch(const BwdArgs& a, int64_t N, int io_dtype, cudaStream_t stream) {
  if (io_dtype == 0) return bwd_io<float>(a, N, stream);
  return bwd_io<__nv_bfloat16>(a, N, stream);
}

}  // namespace ssm
