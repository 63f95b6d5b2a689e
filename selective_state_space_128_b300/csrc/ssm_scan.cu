// Selective-scan forward kernel (S6) for sm_103a.
//
// Computes, per (batch b, channel d): Δ_t = softplus(delta + bias), the
// zero-order-hold pair Ā = exp(Δ A), B̄ = (exp(Δ A) - 1)/A · B_t, the recurrence
// h_t = Ā h_{t-1} + B̄ u_t and the readout y_t = (C_t · h_t + D u_t) · silu(z_t)
// ("Mamba: Linear-Time Sequence Modeling" summary page: section 4b equations
// (2), (4) and Algorithm 2; section 4a shape table for the gate; the SSM/Mamba
// chapter's section 3.1 for D).
//
// Design (B300).  The work is bound by the SM's FP32 pipe, not by HBM: per
// channel step it moves 8 bytes (bf16 u, Δ, z in, y out) but needs N
// exponentials and about 6N FP32 operations.  So the kernel is organised to
// spend as few issue slots as possible per state update:
//
//  * a block owns CH channels of one batch row; each channel is handled by G
//    lanes holding NPT = N/G states each in fp32 registers for the whole
//    sequence (the expanded (L, N) state never leaves the SM);
//  * chunks of T steps of u/Δ/z (a CH x T box) and of B/C (an N x T box,
//    shared by all channels of the block) are fetched by TMA
//    (cp.async.bulk.tensor, mbarrier completion) into a ring of raw stages,
//    prefetched S chunks ahead;
//  * a cooperative "prep" pass turns a raw stage into fp32 working tiles once
//    per channel step -- Δ (softplus applied once, not once per lane), u, the
//    gate silu(z) -- and transposes B/C to [t][n], so that every lane reads
//    (Δ, Δ, u, u) and its NPT values of B and C with 16-byte shared loads that
//    land directly in packed register pairs;
//  * the state update runs on packed f32x2 pairs (one issue for two lanes of
//    FP32 work) with one MUFU ex2 per state: Ā = 2^(Δ·A·log2 e),
//    v = -B u / A, h = Ā (h - v) + v, which equals Ā h + (Ā - 1)/A · B u;
//  * the G partial readouts of a channel are combined by a shuffle
//    reduce-scatter, after which lane g finishes time step g of each group of
//    G steps (D term, gate, rounding) into a y tile that the block writes back
//    with 16-byte stores.
//
// Long sequences with few channels are split into segments (grid.z): pass 1
// computes each segment's end state from zero and its ΣΔ, pass 0 folds the
// carries of earlier segments (h <- exp(A ΣΔ_k) h + h_k) into its initial state
// and recomputes its segment with outputs.  There is no inter-block waiting.
// The only waits are on the block's own TMA barriers; they give up after a
// time limit, record it in a device error word (read by ssm_status) and end the block.
#include <cuda.h>

#include <cstring>
#include <type_traits>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

// Device-side error word (0 = none).  Read and cleared by scan_device_error().
__device__ int g_scan_error;

// Per-N tiling: NPT states per lane, G lanes per channel, CH channels per
// block, T steps per chunk, S raw stages in flight.
template <int N> struct ScanCfg {
  static constexpr int NPT = N <= 4 ? N : (N <= 16 ? 4 : N / 4);
  static constexpr int G = N / NPT;
  static constexpr int CH = kScanThreads / G;
  static constexpr int T = 32;
  static constexpr int S = 2;
  static_assert(G * NPT == N, "tiling");
  static_assert(T % G == 0 && T % 8 == 0, "chunk");
};

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shared-memory layout of one block.  Raw stages are TMA destinations
// (128-byte aligned); the working tiles are padded so that the lanes of a warp
// hit distinct banks.
template <typename IO, int N> struct ScanSmem {
  using Cf = ScanCfg<N>;
  static constexpr int CH = Cf::CH, T = Cf::T, S = Cf::S;
  static constexpr size_t kRawIO = (size_t)CH * T * sizeof(IO);  // one of u / Δ / z
  static constexpr size_t kRawBC = (size_t)N * T * 4;              // one of B / C
  static constexpr size_t oRawU = 0;
  static constexpr size_t oRawD = align_up(oRawU + kRawIO, 128);
  static constexpr size_t oRawZ = align_up(oRawD + kRawIO, 128);
  static constexpr size_t oRawB = align_up(oRawZ + kRawIO, 128);
  static constexpr size_t oRawC = align_up(oRawB + kRawBC, 128);
  static constexpr size_t kStage = align_up(oRawC + kRawBC, 128);
  static constexpr int RowDU = T + 1;                 // float4 per row (+1 breaks bank aliasing)
  static constexpr int RowG = T + 4;                  // floats per gate row
  static constexpr int RowBC = N + 4;                 // floats per transposed B/C row
  static constexpr int RowY = T + 16 / (int)sizeof(IO);  // elements per y row (16-byte multiple)
  static constexpr size_t oDU = (size_t)S * kStage;
  static constexpr size_t oGate = align_up(oDU + (size_t)CH * RowDU * 16, 16);
  static constexpr size_t oBt = align_up(oGate + (size_t)CH * RowG * 4, 16);
  static constexpr size_t oCt = align_up(oBt + (size_t)T * RowBC * 4, 16);
  static constexpr size_t oY = align_up(oCt + (size_t)T * RowBC * 4, 16);
  static constexpr size_t oBias = align_up(oY + (size_t)CH * RowY * sizeof(IO), 16);
  static constexpr size_t oBar = align_up(oBias + (size_t)CH * 4, 8);
  static constexpr size_t kBytes = oBar + 8 * S;
  static constexpr size_t kLaunchBytes = kBytes + 128;  // room to align the base to 128
};

// ---------------------------------------------------------------------------
// TMA and mbarrier primitives (inline PTX)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
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
// Wait for phase `parity` of `bar`, giving up after kWaitLimitNs.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: a TMA chunk lands in microseconds
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 16-byte shared load into two packed pairs.
__device__ __forceinline__ void lds_pairs(const void* p, f2& a, f2& b) {
  asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a.r), "=l"(b.r) : "r"(smem_u32(p)));
}
__device__ __forceinline__ void lds_pair(const void* p, f2& a) {
  asm volatile("ld.shared.b64 %0, [%1];" : "=l"(a.r) : "r"(smem_u32(p)));
}

// The four tensor maps of a launch (u, Δ, z: box CH x T; B, C: box N x T).
struct ScanMaps {
  CUtensorMap u, d, z, b, c;
};

// ---------------------------------------------------------------------------
// Staging and prep
// ---------------------------------------------------------------------------
template <typename IO> __device__ __forceinline__ void load8(const IO* p, float (&v)[8]);
template <> __device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(ws[i] << 16);
    v[2 * i + 1] = __uint_as_float(ws[i] & 0xffff0000u);
  }
}
template <> __device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Per element of the chunk: Δ (softplus once), u and the gate into the fp32
// working tiles.  Steps past tcount and rows past the channel count get Δ = 0
// and u = 0, exact no-ops of the recurrence (Ā = 1, B̄ u = 0).  The flags are
// template parameters so that the element loop carries no per-element branch.
template <typename IO, int N, int PASS, bool TMA, bool PRECISE, bool SP, bool HZ, bool MASK>
__device__ __forceinline__ void prep_elems(const ScanArgs& p, const unsigned char* stage,
                                           unsigned char* sm, int64_t b, int64_t d0, int64_t t0,
                                           int tcount, int nrows) {
  using S = ScanSmem<IO, N>;
  constexpr int CH = S::CH, T = S::T;
  const int tid = threadIdx.x;
  float4* DU = reinterpret_cast<float4*>(sm + S::oDU);
  float* Gt = reinterpret_cast<float*>(sm + S::oGate);
  const float* sBias = reinterpret_cast<const float*>(sm + S::oBias);
#pragma unroll 1
  for (int e = tid; e < CH * (T / 8); e += kScanThreads) {
    const int r = e / (T / 8), t8 = (e - r * (T / 8)) * 8;
    float dl[8], uu[8], zz[8];
    if (TMA) {
      load8<IO>(reinterpret_cast<const IO*>(stage + S::oRawD) + r * T + t8, dl);
      load8<IO>(reinterpret_cast<const IO*>(stage + S::oRawU) + r * T + t8, uu);
      if (HZ) load8<IO>(reinterpret_cast<const IO*>(stage + S::oRawZ) + r * T + t8, zz);
    } else {
      const int64_t row = (b * p.dim + d0 + r) * p.L + t0 + t8;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const bool ok = r < nrows && t8 + j < tcount;
        dl[j] = ok ? io_traits<IO>::to_f32(static_cast<const IO*>(p.delta)[row + j]) : 0.f;
        uu[j] = ok ? io_traits<IO>::to_f32(static_cast<const IO*>(p.u)[row + j]) : 0.f;
        zz[j] = (ok && HZ) ? io_traits<IO>::to_f32(static_cast<const IO*>(p.z)[row + j]) : 0.f;
      }
    }
    const float bias = sBias[r];
    float gate[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float x = dl[j] + bias;
      float dt = SP ? (PRECISE ? softplus_precise(x) : softplus_fast(x)) : x;
      float u = uu[j];
      if (MASK) {
        const bool ok = r < nrows && t8 + j < tcount;
        dt = ok ? dt : 0.f;
        u = ok ? u : 0.f;
      }
      DU[r * S::RowDU + t8 + j] = make_float4(dt, dt, u, u);
      gate[j] = HZ ? (PRECISE ? silu_precise(zz[j]) : silu_fast(zz[j])) : 1.f;
    }
    if (PASS == 0) {
      float4* g4 = reinterpret_cast<float4*>(Gt + r * S::RowG + t8);
      g4[0] = make_float4(gate[0], gate[1], gate[2], gate[3]);
      g4[1] = make_float4(gate[4], gate[5], gate[6], gate[7]);
    }
  }
}

template <typename IO, int N, int PASS, bool TMA, bool PRECISE>
__device__ __forceinline__ void prep_chunk(const ScanArgs& p, const unsigned char* stage,
                                           unsigned char* sm, int64_t b, int64_t d0, int64_t t0,
                                           int tcount) {
  using S = ScanSmem<IO, N>;
  constexpr int CH = S::CH, T = S::T;
  const int tid = threadIdx.x;
  const int nrows = (int)min64(CH, p.dim - d0);
  const bool mask = tcount < T || nrows < CH;
  const bool hz = PASS == 0 && p.z != nullptr;
#define SSM_PREP(SP, HZ, MASK) \
  prep_elems<IO, N, PASS, TMA, PRECISE, SP, HZ, MASK>(p, stage, sm, b, d0, t0, tcount, nrows)
  if (p.softplus) {
    if (hz) { if (mask) SSM_PREP(true, true, true); else SSM_PREP(true, true, false); }
    else    { if (mask) SSM_PREP(true, false, true); else SSM_PREP(true, false, false); }
  } else {
    if (hz) { if (mask) SSM_PREP(false, true, true); else SSM_PREP(false, true, false); }
    else    { if (mask) SSM_PREP(false, false, true); else SSM_PREP(false, false, false); }
  }
#undef SSM_PREP
  // B / C transposed to [t][n]
  float* Bt = reinterpret_cast<float*>(sm + S::oBt);
  float* Ct = reinterpret_cast<float*>(sm + S::oCt);
  constexpr int NARR = PASS == 0 ? 2 : 1;
#pragma unroll 1
  for (int e = tid; e < NARR * N * (T / 4); e += kScanThreads) {
    const int arr = e / (N * (T / 4));
    const int rem = e - arr * (N * (T / 4));
    const int n = rem / (T / 4), t4 = (rem - n * (T / 4)) * 4;
    float v[4];
    if (TMA) {
      const float4 q = *reinterpret_cast<const float4*>(
          reinterpret_cast<const float*>(stage + (arr == 0 ? S::oRawB : S::oRawC)) + n * T + t4);
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
      const float* src = (arr == 0 ? p.B : p.C) + (b * N + n) * p.L + t0 + t4;
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = t4 + j < tcount ? src[j] : 0.f;
    }
    float* dst = arr == 0 ? Bt : Ct;
#pragma unroll
    for (int j = 0; j < 4; ++j) dst[(t4 + j) * S::RowBC + n] = v[j];
  }
}

// Combine the G partial readouts of a channel: afterwards lane g holds the full
// sum for time step g of the group (shuffle reduce-scatter, log2(G) stages).
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

// Issue the TMA loads of one chunk into a raw stage (one thread).
template <typename IO, int N, int PASS>
__device__ __forceinline__ void issue_chunk(const ScanArgs& p, const ScanMaps& m,
                                            unsigned char* stage, uint64_t* bar, int64_t b,
                                            int64_t d0, int64_t t0) {
  using S = ScanSmem<IO, N>;
  const bool has_z = PASS == 0 && p.z != nullptr;
  const uint32_t bytes = (uint32_t)(S::kRawIO * (has_z ? 3 : 2) + S::kRawBC * (PASS == 0 ? 2 : 1));
  mbar_arrive_expect_tx(bar, bytes);
  const int x = (int)t0, y = (int)d0, z = (int)b;
  tma_load_3d(stage + S::oRawU, &m.u, bar, x, y, z);
  tma_load_3d(stage + S::oRawD, &m.d, bar, x, y, z);
  if (has_z) tma_load_3d(stage + S::oRawZ, &m.z, bar, x, y, z);
  tma_load_3d(stage + S::oRawB, &m.b, bar, x, 0, z);
  if (PASS == 0) tma_load_3d(stage + S::oRawC, &m.c, bar, x, 0, z);
}

// ---------------------------------------------------------------------------
// One chunk of T steps for one lane, fast flavour (MUFU ex2, packed f32x2).
// The step loop is fully unrolled and the Ā / v pairs of step t+1 are formed
// while step t updates the state, so that the serial chain per step is just
// h <- Ā (h - v) + v and the readout.
// ---------------------------------------------------------------------------
template <typename IO, int N, int PASS>
__device__ __forceinline__ void chunk_fast(unsigned char* sm, int c, int g, float Dd,
                                           f2 (&hp)[ScanCfg<N>::NPT / 2],
                                           const f2 (&A2p)[ScanCfg<N>::NPT / 2],
                                           const f2 (&nIp)[ScanCfg<N>::NPT / 2], float& sumDt) {
  using Cf = ScanCfg<N>;
  using S = ScanSmem<IO, N>;
  constexpr int NPT = Cf::NPT, G = Cf::G, T = Cf::T, NP = NPT / 2;
  const float4* DUrow = reinterpret_cast<const float4*>(sm + S::oDU) + c * S::RowDU;
  const float* Grow = reinterpret_cast<const float*>(sm + S::oGate) + c * S::RowG;
  const float* Bt = reinterpret_cast<const float*>(sm + S::oBt) + g * NPT;
  const float* Ct = reinterpret_cast<const float*>(sm + S::oCt) + g * NPT;
  IO* yT = reinterpret_cast<IO*>(sm + S::oY) + c * S::RowY;

  auto load_row = [](const float* row, f2 (&v)[NP]) {
#pragma unroll
    for (int q = 0; q + 1 < NP; q += 2) lds_pairs(row + 2 * q, v[q], v[q + 1]);
    if constexpr (NP % 2 == 1) lds_pair(row + 2 * (NP - 1), v[NP - 1]);
  };
  // Three-deep software pipeline over the fully unrolled steps: the shared
  // loads of step t+2, the exponentials and v of step t+1 and the state
  // update of step t are independent, so their latencies overlap.
  f2 dt_l, u_l, b_l[NP], c_l[NP];      // loaded for step t+1
  f2 a_c[NP], v_c[NP], c_c[NP];        // ready for step t
  auto load_step = [&](int t, f2& dt2, f2& u2, f2 (&bq)[NP], f2 (&cq)[NP]) {
    lds_pairs(DUrow + t, dt2, u2);
    load_row(Bt + t * S::RowBC, bq);
    if (PASS == 0) load_row(Ct + t * S::RowBC, cq);
  };
  auto discretise = [&](const f2& dt2, const f2& u2, const f2 (&bq)[NP], f2 (&ao)[NP],
                        f2 (&vo)[NP]) {
    if (PASS == 1) {
      float lo, hi;
      unpack2(dt2, lo, hi);
      sumDt += lo;
    }
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      const f2 x = mul2(dt2, A2p[q]);
      float x0, x1;
      unpack2(x, x0, x1);
      ao[q] = pack2(ex2_fast(x0), ex2_fast(x1));
      vo[q] = mul2(mul2(bq[q], u2), nIp[q]);
    }
  };

  {
    f2 dt0, u0, b0[NP];
    load_step(0, dt0, u0, b0, c_c);
    discretise(dt0, u0, b0, a_c, v_c);
    load_step(1, dt_l, u_l, b_l, c_l);
  }
  float part[G];
#pragma unroll
  for (int t = 0; t < T; ++t) {
    f2 dt_n, u_n, b_n[NP], c_n[NP], a_n[NP], v_n[NP];
    if (t + 2 < T) load_step(t + 2, dt_n, u_n, b_n, c_n);
    if (t + 1 < T) discretise(dt_l, u_l, b_l, a_n, v_n);
#pragma unroll
    for (int q = 0; q < NP; ++q) hp[q] = fma2(a_c[q], sub2(hp[q], v_c[q]), v_c[q]);
    if (PASS == 0) {
      f2 acc2 = mul2(c_c[0], hp[0]);
#pragma unroll
      for (int q = 1; q < NP; ++q) acc2 = fma2(c_c[q], hp[q], acc2);
      float lo, hi;
      unpack2(acc2, lo, hi);
      part[t % G] = lo + hi;
      if (t % G == G - 1) {
        const float yv = reduce_scatter<G>(part, g);
        const int ty = t - (G - 1) + g;
        yT[ty] = io_traits<IO>::from_f32(fmaf(Dd, DUrow[ty].z, yv) * Grow[ty]);
      }
    }
    if (t + 1 < T) {
#pragma unroll
      for (int q = 0; q < NP; ++q) {
        a_c[q] = a_n[q];
        v_c[q] = v_n[q];
        c_c[q] = c_l[q];
      }
    }
    if (t + 2 < T) {
      dt_l = dt_n;
      u_l = u_n;
#pragma unroll
      for (int q = 0; q < NP; ++q) {
        b_l[q] = b_n[q];
        c_l[q] = c_n[q];
      }
    }
  }
}

// One chunk, one state per lane (N = 1), fast flavour.
template <typename IO, int PASS>
__device__ __forceinline__ void chunk_fast_scalar(unsigned char* sm, int c, float Dd, float& h,
                                                  float A2s, float nIs, float& sumDt) {
  using S = ScanSmem<IO, 1>;
  constexpr int T = ScanCfg<1>::T;
  const float4* DUrow = reinterpret_cast<const float4*>(sm + S::oDU) + c * S::RowDU;
  const float* Grow = reinterpret_cast<const float*>(sm + S::oGate) + c * S::RowG;
  const float* Bt = reinterpret_cast<const float*>(sm + S::oBt);
  const float* Ct = reinterpret_cast<const float*>(sm + S::oCt);
  IO* yT = reinterpret_cast<IO*>(sm + S::oY) + c * S::RowY;
#pragma unroll 8
  for (int t = 0; t < T; ++t) {
    const float4 du = DUrow[t];
    if (PASS == 1) sumDt += du.x;
    const float a = ex2_fast(du.x * A2s);
    const float nv = Bt[t * S::RowBC] * du.z * nIs;
    h = fmaf(a, h - nv, nv);
    if (PASS == 0) yT[t] = io_traits<IO>::from_f32(fmaf(Dd, du.z, Ct[t * S::RowBC] * h) * Grow[t]);
  }
}

// One chunk, precise flavour (CUDA libm expf / expm1f; A = 0 takes the limit).
template <typename IO, int N, int PASS>
__device__ __forceinline__ void chunk_precise(unsigned char* sm, int c, int g, float Dd,
                                              float (&h)[ScanCfg<N>::NPT],
                                              const float (&Aj)[ScanCfg<N>::NPT],
                                              const float (&invA)[ScanCfg<N>::NPT], float& sumDt) {
  using Cf = ScanCfg<N>;
  using S = ScanSmem<IO, N>;
  constexpr int NPT = Cf::NPT, G = Cf::G, T = Cf::T;
  const float4* DUrow = reinterpret_cast<const float4*>(sm + S::oDU) + c * S::RowDU;
  const float* Grow = reinterpret_cast<const float*>(sm + S::oGate) + c * S::RowG;
  const float* Bt = reinterpret_cast<const float*>(sm + S::oBt) + g * NPT;
  const float* Ct = reinterpret_cast<const float*>(sm + S::oCt) + g * NPT;
  IO* yT = reinterpret_cast<IO*>(sm + S::oY) + c * S::RowY;
  for (int tb = 0; tb < T; tb += G) {
    float part[G];
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const int t = tb + k;
      const float4 du = DUrow[t];
      const float dt = du.x, ut = du.z;
      if (PASS == 1) sumDt += dt;
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const float x = dt * Aj[j];
        const float a = expf(x);
        const float coef = Aj[j] != 0.f ? expm1f(x) * invA[j] : dt;
        h[j] = fmaf(a, h[j], coef * (Bt[t * S::RowBC + j] * ut));
        if (PASS == 0) acc = fmaf(Ct[t * S::RowBC + j], h[j], acc);
      }
      part[k] = acc;
    }
    if (PASS == 0) {
      const float yv = reduce_scatter<G>(part, g);
      const int t = tb + g;
      yT[t] = io_traits<IO>::from_f32(fmaf(Dd, DUrow[t].z, yv) * Grow[t]);
    }
  }
}

// The chunk loop of one block: wait for chunk i's TMA stage, prep it, refill
// the stage with chunk i + S, run the steps, write the y tile back.  Returns
// the index of a chunk whose wait timed out, or -1.
template <typename IO, int N, int PASS, bool PRECISE>
__device__ __forceinline__ int64_t run_chunks(
    const ScanArgs& p, const ScanMaps& maps, unsigned char* sm, uint64_t* bars, int64_t b,
    int64_t d0, int64_t t_begin, int64_t t_end, int64_t nchunks, bool use_tma, int c, int g,
    float Dd, float (&h)[ScanCfg<N>::NPT], f2 (&hp)[ScanCfg<N>::NPT / 2 > 0 ? ScanCfg<N>::NPT / 2 : 1],
    const f2 (&A2p)[ScanCfg<N>::NPT / 2 > 0 ? ScanCfg<N>::NPT / 2 : 1],
    const f2 (&nIp)[ScanCfg<N>::NPT / 2 > 0 ? ScanCfg<N>::NPT / 2 : 1], float A2s, float nIs,
    const float (&Aj)[ScanCfg<N>::NPT], const float (&invA)[ScanCfg<N>::NPT], float& sumDt) {
  using Cf = ScanCfg<N>;
  using S = ScanSmem<IO, N>;
  constexpr int NPT = Cf::NPT, CH = Cf::CH, T = Cf::T, NS = Cf::S;
  const int tid = threadIdx.x;
  const IO* yTile = reinterpret_cast<const IO*>(sm + S::oY);
  for (int64_t i = 0; i < nchunks; ++i) {
    const int s = (int)(i % NS);
    const int64_t t0 = t_begin + i * T;
    const int tcount = (int)min64(T, t_end - t0);
    unsigned char* stage = sm + (size_t)s * S::kStage;
    bool ok = true;
    if (use_tma) {
      ok = mbar_wait_bounded(&bars[s], (uint32_t)((i / NS) & 1));
      prep_chunk<IO, N, PASS, true, PRECISE>(p, stage, sm, b, d0, t0, tcount);
    } else {
      prep_chunk<IO, N, PASS, false, PRECISE>(p, stage, sm, b, d0, t0, tcount);
    }
    if (__syncthreads_or(!ok)) return i;
    // the raw stage is consumed: refill it with chunk i + NS
    if (use_tma && tid == 0 && i + NS < nchunks)
      issue_chunk<IO, N, PASS>(p, maps, stage, &bars[s], b, d0, t0 + (int64_t)NS * T);

    if constexpr (PRECISE) {
      chunk_precise<IO, N, PASS>(sm, c, g, Dd, h, Aj, invA, sumDt);
    } else if constexpr (NPT == 1) {
      chunk_fast_scalar<IO, PASS>(sm, c, Dd, h[0], A2s, nIs, sumDt);
    } else {
      chunk_fast<IO, N, PASS>(sm, c, g, Dd, hp, A2p, nIp, sumDt);
    }
    __syncthreads();
    if (PASS == 0) {
      // write the y tile back
      IO* gy = static_cast<IO*>(p.y);
      const int nrows = (int)min64(CH, p.dim - d0);
      constexpr int VEC = 16 / sizeof(IO);
      if (p.vec_io) {
        const int pieces = tcount / VEC;  // tcount is a multiple of VEC here
        for (int e = tid; e < nrows * pieces; e += kScanThreads) {
          const int r = e / pieces, k = e - r * pieces;
          const uint4 v = *reinterpret_cast<const uint4*>(yTile + r * S::RowY + k * VEC);
          *reinterpret_cast<uint4*>(gy + (b * p.dim + d0 + r) * p.L + t0 + k * VEC) = v;
        }
      } else {
        for (int e = tid; e < nrows * tcount; e += kScanThreads) {
          const int r = e / tcount, k = e - r * tcount;
          gy[(b * p.dim + d0 + r) * p.L + t0 + k] = yTile[r * S::RowY + k];
        }
      }
    }
  }
  return -1;
}

// ---------------------------------------------------------------------------
// The kernel.  PASS 0: outputs (y, final state).  PASS 1: segment end state
// from a zero start and ΣΔ, for the split plan.
// ---------------------------------------------------------------------------
template <typename IO, int N, int PASS>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(const ScanArgs p,
                                                            const __grid_constant__ ScanMaps maps) {
  using Cf = ScanCfg<N>;
  using S = ScanSmem<IO, N>;
  constexpr int NPT = Cf::NPT, G = Cf::G, CH = Cf::CH, T = Cf::T, NS = Cf::S;
  constexpr int NP = NPT / 2;  // packed pairs per lane (0 when NPT == 1)
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

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
  const bool use_tma = p.use_tma != 0;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::oBar);
  float* sBias = reinterpret_cast<float*>(sm + S::oBias);
  for (int r = tid; r < CH; r += kScanThreads)
    sBias[r] = (p.bias && d0 + r < p.dim) ? p.bias[d0 + r] : 0.f;
  if (use_tma && tid == 0) {
    prefetch_tmap(&maps.u);
    prefetch_tmap(&maps.d);
    prefetch_tmap(&maps.b);
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }

  // this lane's states: n = g*NPT + j
  float Aj[NPT];
  bool zeroA = false;
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    Aj[j] = chan_ok ? p.A[d * N + g * NPT + j] : -1.f;
    zeroA |= (Aj[j] == 0.f);
  }
  const bool precise = __syncthreads_or(zeroA) || p.force_precise;

  // prologue: the first NS chunks in flight
  if (use_tma && tid == 0) {
    for (int k = 0; k < NS && k < nchunks; ++k)
      issue_chunk<IO, N, PASS>(p, maps, sm + (size_t)k * S::kStage, &bars[k], b, d0,
                               t_begin + (int64_t)k * T);
  }

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

  // fast-path constants: A·log2(e) and -1/A per state, as packed pairs
  f2 A2p[NP > 0 ? NP : 1], nIp[NP > 0 ? NP : 1], hp[NP > 0 ? NP : 1];
  float A2s = 0.f, nIs = 0.f;
  if constexpr (NPT == 1) {
    A2s = Aj[0] * kLog2e;
    nIs = Aj[0] != 0.f ? -1.f / Aj[0] : 0.f;
  } else {
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      A2p[q] = pack2(Aj[2 * q] * kLog2e, Aj[2 * q + 1] * kLog2e);
      nIp[q] = pack2(Aj[2 * q] != 0.f ? -1.f / Aj[2 * q] : 0.f,
                     Aj[2 * q + 1] != 0.f ? -1.f / Aj[2 * q + 1] : 0.f);
      hp[q] = pack2(h[2 * q], h[2 * q + 1]);
    }
  }
  float invA[NPT];
#pragma unroll
  for (int j = 0; j < NPT; ++j) invA[j] = Aj[j] != 0.f ? 1.f / Aj[j] : 0.f;

  float sumDt = 0.f;
  int64_t i = -1;  // chunk whose wait timed out, or -1
  if (precise) {
    i = run_chunks<IO, N, PASS, true>(p, maps, sm, bars, b, d0, t_begin, t_end, nchunks, use_tma,
                                      c, g, Dd, h, hp, A2p, nIp, A2s, nIs, Aj, invA, sumDt);
  } else {
    i = run_chunks<IO, N, PASS, false>(p, maps, sm, bars, b, d0, t_begin, t_end, nchunks,
                                       use_tma, c, g, Dd, h, hp, A2p, nIp, A2s, nIs, Aj, invA,
                                       sumDt);
    if constexpr (NPT > 1) {
#pragma unroll
      for (int q = 0; q < NP; ++q) unpack2(hp[q], h[2 * q], h[2 * q + 1]);
    }
  }
  const bool failed = i >= 0;

  if (failed) {
    // a TMA chunk did not land in time: record it, let the copies still in
    // flight into this block's shared memory finish (bounded), and leave
    // without writing a state
    if (tid == 0) {
      atomicExch(&g_scan_error, 1);
      for (int64_t j = i; j < nchunks && j < i + NS; ++j)
        (void)mbar_wait_bounded(&bars[j % NS], (uint32_t)((j / NS) & 1));
    }
    return;
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
  ScanPlan pl{1, L, 0, 32, 32};
  if (!cfg_for(N, pl.chans, pl.chunk)) return pl;
  pl.seg_len = L > 0 ? L : 1;
  if (!allow_split || L <= 0 || batch <= 0 || dim <= 0) return pl;
  const int64_t blocks = ((dim + pl.chans - 1) / pl.chans) * batch;
  const int64_t want = (int64_t)sm_count * 2;  // blocks that keep every SM busy
  if (blocks >= want) return pl;
  int64_t nseg = (want + blocks - 1) / blocks;
  const int64_t max_by_len = L / (16 * (int64_t)pl.chunk);  // at least 16 chunks per segment
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

// cuTensorMapEncodeTiled, looked up once through the runtime (no link to libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// 3-D map over a (d2, d1, d0) row-major tensor (d0 fastest) with box (1, b1, b0).
static bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, size_t esz,
                     uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !base) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * esz, d0 * d1 * esz};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename IO, int N>
static bool make_maps(ScanMaps& m, const ScanArgs& a) {
  using Cf = ScanCfg<N>;
  const CUtensorMapDataType dt =
      sizeof(IO) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const uint64_t L = (uint64_t)a.L, D = (uint64_t)a.dim, Bt = (uint64_t)a.batch;
  bool ok = make_map(&m.u, a.u, dt, sizeof(IO), L, D, Bt, Cf::T, Cf::CH) &&
            make_map(&m.d, a.delta, dt, sizeof(IO), L, D, Bt, Cf::T, Cf::CH) &&
            make_map(&m.b, a.B, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, L, N, Bt, Cf::T, N) &&
            make_map(&m.c, a.C, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, L, N, Bt, Cf::T, N);
  if (ok && a.z) ok = make_map(&m.z, a.z, dt, sizeof(IO), L, D, Bt, Cf::T, Cf::CH);
  return ok;
}

template <typename IO, int N, int PASS>
static cudaError_t launch_one(const ScanArgs& a, const ScanMaps& m, int nz, cudaStream_t stream) {
  using Cf = ScanCfg<N>;
  constexpr size_t bytes = ScanSmem<IO, N>::kLaunchBytes;
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
  kern<<<grid, kScanThreads, bytes, stream>>>(a, m);
  return cudaGetLastError();
}

template <typename IO, int N>
static cudaError_t launch_typed(ScanArgs a, cudaStream_t stream) {
  ScanMaps m;
  memset(&m, 0, sizeof m);
  // TMA needs 16-byte row strides (rows of u/Δ/z and B/C) and coordinates
  // that fit in int32
  const bool rows16 = a.vec_io && a.vec_bc;
  const bool fits = a.L < (int64_t(1) << 31) && a.dim < (int64_t(1) << 31);
  a.use_tma = rows16 && fits && make_maps<IO, N>(m, a);
  if (a.nseg > 1) {
    cudaError_t e = launch_one<IO, N, 1>(a, m, a.nseg - 1, stream);
    if (e != cudaSuccess) return e;
  }
  return launch_one<IO, N, 0>(a, m, a.nseg, stream);
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

cudaError_t scan_device_error(int* code, cudaStream_t stream) {
  int zero = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(code, g_scan_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_scan_error, &zero, sizeof(int));
}

}  // namespace ssm
