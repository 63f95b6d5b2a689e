// Selective-scan forward for N = 16 states and bf16 I/O: blocks of two warps.
//
// Computes what ssm_scan.cu computes ("Mamba: Linear-Time Sequence Modeling"
// summary page, section 4b equations (2), (4) and Algorithm 2; section 4a shape
// table for the gate; the SSM/Mamba chapter's section 3.1 for D):
//   Δ_t = softplus(delta + bias), Ā = exp(Δ A), B̄ u = (exp(Δ A) - 1)/A · B u,
//   h_t = Ā h_{t-1} + B̄ u_t,  y_t = (C_t · h_t + D u_t) · silu(z_t),
// for the common case (N = 16, bf16 u/Δ/z/y, zero-order hold, views TMA can
// stage, time-major or channel-major).
//
// Design (B300).  The work is bound by instruction issue, shared-memory
// wavefronts and latency, not by HBM: per channel step it needs 16
// exponentials and 6 FP32 operations per state but moves only 8 bytes.  So
// every instruction that is not the recurrence is overhead to cut, and the SMs
// must stay busy to the end of the grid.
//
//  * A block of 64 threads (two warps) owns 16 channels of one batch row over
//    one segment of the sequence, with its own TMA ring (u, Δ, z boxes of
//    T x 16 and the B, C boxes of T x N) and its own buffers; blocks are small,
//    so the block scheduler spreads them evenly over the SMs.
//  * Each channel's 16 states sit on G = 4 threads (4 states each, in fp32
//    registers for the whole segment); warp w holds state groups 2w and 2w + 1
//    of all 16 channels (thread (w, lane l): channel l & 15, group 2w + (l >> 4)),
//    so the warp-wide load of a B or C row touches two 16-byte addresses (two
//    shared-memory wavefronts; four when one warp holds all four groups of 8
//    channels).  A state update is one MUFU ex2 and packed f32x2 arithmetic:
//    Ā = 2^(Δ·A·log2 e), v = -B u / A, h = Ā (h - v) + v (= Ā h + B̄ u); the
//    partial readouts Σ_{its n} C_n h_n of a warp's two groups of a channel are
//    added by a shuffle and written to a partial tile.
//  * Chunks of T = 32 steps for the outputs (16 for the split plan's first
//    pass).  The per-channel-step work that is not per state runs once per
//    channel step, split over the channel's 4 threads (T / 4 steps each): the
//    conversion (Δ = softplus(.) once, u, the gate silu(z) and D u) and the
//    finalisation (y = (Σ partials + D u) · gate, rounded, one 16-byte store
//    per thread and chunk).
//  * B and C are transposed to [t][n] once per chunk (warp 0: B, warp 1: C; 2
//    loads and 8 stores per lane and 16 steps, bank-conflict free), so a
//    thread's 4 values of a step are one 16-byte load.
//  * Two block barriers per chunk: after the conversion and transposition,
//    after the recurrence.
//
// Long sequences with few channels are split into segments exactly as in
// ssm_scan.cu (same carry records): pass 1 computes each segment's end state
// from zero and its ΣΔ, pass 0 folds the carries of earlier segments into its
// initial state and recomputes its segment with outputs.
//
// A block whose channels have some A = 0 runs a plain per-thread loop in the
// precise flavour (CUDA libm expf / expm1f; A = 0 takes the limit Δ B) instead.
// The only waits are on the block's own TMA barriers; they are bounded, and a
// wait that runs out records an error in the call's status word and ends the
// block after its copies in flight have landed.
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kN = 16;    // states
constexpr int kCk = 16;   // steps between the chunk-start states a training forward saves
constexpr int kNSU = 2;   // stages of the u / Δ / z ring (B, C: one stage)

__host__ __device__ constexpr size_t up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct FastMaps {
  CUtensorMap u, d, z, b, c;
};

__device__ __forceinline__ void tma3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                      int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Column of B^T / C^T where state n of step t is stored: the halves of a row are
// swapped for t in 8..15, which spreads the transposition's stores over all 32
// banks and keeps every aligned group of four states contiguous.
__device__ __forceinline__ int bt_col(int t, int n) { return n ^ (((t >> 3) & 1) << 3); }

constexpr int kG = 4;             // state groups (threads per channel)
constexpr int kNPT = kN / kG;     // states per thread
constexpr int kCB = 16;           // channels per block
constexpr int kThreads = 64;
// Chunks: T = 32 steps for the output pass (fewer barriers, waits and pipeline
// fills per step), T = 16 for the split plan's first pass (which has no readout
// and whose 32-step form spills); a thread converts and finalises T / 4 steps.
constexpr int kTOut = 32, kTCarry = 16;

// One thread's view of the launch (the recurrence's mapping).
struct FastLane {
  int lane, c, g;     // lane, channel within the block, state group
  int64_t b, d0, d;   // batch row, first channel of the block, this thread's channel
  bool chan_ok;
};

template <int NPT> struct LaneStates {
  float h[NPT];
};

// The final state (pass 0, last segment) or the segment's carry record (pass 1).
template <int PASS>
__device__ __forceinline__ void write_lane_states(const ScanArgs& p, const FastLane& L, int seg,
                                                  const float* h) {
  constexpr int NPT = kNPT;
  if (!L.chan_ok) return;
  const int64_t row = L.b * p.dim + L.d;
  float* dst = nullptr;
  if (PASS == 0) {
    if (p.final_state && seg == p.nseg - 1) dst = p.final_state + row * kN + L.g * NPT;
  } else {
    dst = p.carry_h + ((int64_t)seg * p.batch * p.dim + row) * kN + L.g * NPT;
  }
  if (dst) {
#pragma unroll
    for (int j = 0; j < NPT; j += 4)
      *reinterpret_cast<float4*>(dst + j) = make_float4(h[j], h[j + 1], h[j + 2], h[j + 3]);
  }
}

// Shared memory of one block (bytes; TMA destinations 128-byte aligned).
template <int T> struct PairSmem {
  static constexpr size_t kRawIO = (size_t)kCB * T * 2;      // one of u / Δ / z (bf16)
  static constexpr size_t kStageU = up(3 * kRawIO, 128);      // u | Δ | z
  static constexpr size_t oStageU = 0;
  static constexpr size_t kRawBC = (size_t)kN * T * 4;        // one of B / C (fp32, [n][t])
  static constexpr size_t oStageBC = kNSU * kStageU;          // B | C
  static constexpr int RowBT = kN + 4;
  static constexpr size_t kBT = (size_t)T * RowBT * 4;        // B^T or C^T [t][n]
  static constexpr size_t oBT = oStageBC + 2 * kRawBC;
  static constexpr size_t oW = oBT + 2 * kBT;                 // (Δ, u) pairs [t][c]
  static constexpr size_t kW = (size_t)T * kCB * 8;
  static constexpr size_t oP = oW + kW;                       // partials [warp][c][t], swizzled
  static constexpr size_t kP = (size_t)2 * kCB * T * 4;       // a warp's two groups pre-added
  static constexpr size_t oBar = up(oP + kP, 8);              // kNSU + 1 mbarriers
  static constexpr size_t kBytes = oBar + 8 * (kNSU + 1);
  static constexpr size_t kLaunch = kBytes + 1024;            // room to align the base
};

// Index (in floats) of steps 4u..4u+3 of partial row (w, c) (4T bytes a row).  The
// 16-byte unit is XOR-swizzled by the channel so that the 8 threads of a quarter
// warp (one warp's groups, 8 consecutive channels) touch 8 distinct bank groups:
// by (c >> 1) & 3 for rows of 4 units (their bank group also depends on c & 1),
// by c & 7 for rows of 8.
template <int T> __device__ __forceinline__ int pair_pidx(int w, int c, int unit) {
  const int sw = T == 16 ? ((c >> 1) & 3) : (c & 7);
  return (w * kCB + c) * T + ((unit ^ sw) << 2);
}

// Precise per-thread loop for blocks with some A = 0 (rare; plain loads through
// the tensors' strides).  The four groups' partial readouts of a step meet in
// `red` (two buffers of 4 x 16 floats, alternating by step: one barrier a step).
template <int PASS>
__device__ __noinline__ void precise_pair(const ScanArgs& p, const FastLane& L, int64_t t_begin,
                                          int64_t t_end, LaneStates<kNPT> hs, float* red) {
  constexpr int NPT = kNPT;
  float* h = hs.h;
  const __nv_bfloat16* u = static_cast<const __nv_bfloat16*>(p.u);
  const __nv_bfloat16* dl = static_cast<const __nv_bfloat16*>(p.delta);
  const __nv_bfloat16* z = static_cast<const __nv_bfloat16*>(p.z);
  __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.y);
  const int64_t dd = L.chan_ok ? L.d : 0;  // threads past dim read channel 0 and store nothing
  const int64_t ou = L.b * p.st_u[0] + dd * p.st_u[1], od = L.b * p.st_d[0] + dd * p.st_d[1];
  const int64_t oz = L.b * p.st_z[0] + dd * p.st_z[1], oy = L.b * p.st_y[0] + dd * p.st_y[1];
  float Aj[NPT], invA[NPT];
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    Aj[j] = p.A[dd * kN + L.g * NPT + j];
    invA[j] = Aj[j] != 0.f ? 1.f / Aj[j] : 0.f;
  }
  const float bias = p.bias ? p.bias[dd] : 0.f;
  const float Dd = p.D ? p.D[dd] : 0.f;
  float sumDt = 0.f;
  for (int64_t t = t_begin; t < t_end; ++t) {
    if (PASS == 0 && p.ckpt != nullptr && ((t - t_begin) % kCk) == 0 && L.chan_ok) {
      float* cp = p.ckpt + ((L.b * p.ckpt_nch + t / kCk) * p.dim + L.d) * kN + L.g * NPT;
#pragma unroll
      for (int j = 0; j < NPT; ++j) cp[j] = h[j];
    }
    const float x = __bfloat162float(dl[od + t * p.st_d[2]]) + bias;
    const float dt = p.softplus ? softplus_precise(x) : x;
    const float ut = __bfloat162float(u[ou + t * p.st_u[2]]);
    sumDt += dt;
    float acc = 0.f;
    const int64_t bc = L.b * kN * p.L + t;
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const int n = L.g * NPT + j;
      const float xa = dt * Aj[j];
      const float coef = Aj[j] != 0.f ? expm1f(xa) * invA[j] : dt;
      h[j] = fmaf(expf(xa), h[j], coef * (p.B[bc + (int64_t)n * p.L] * ut));
      if (PASS == 0) acc = fmaf(p.C[bc + (int64_t)n * p.L], h[j], acc);
    }
    if (PASS == 0) {
      float* r = red + ((t - t_begin) & 1) * (kG * kCB);
      r[L.g * kCB + L.c] = acc;
      __syncthreads();
      if (L.g == 0 && L.chan_ok) {
        const float s = (r[L.c] + r[kCB + L.c]) + (r[2 * kCB + L.c] + r[3 * kCB + L.c]);
        const float gate = z ? silu_precise(__bfloat162float(z[oz + t * p.st_z[2]])) : 1.f;
        y[oy + t * p.st_y[2]] = __float2bfloat16_rn(fmaf(Dd, ut, s) * gate);
      }
    }
  }
  write_lane_states<PASS>(p, L, (int)blockIdx.z, h);
  if (PASS == 1 && L.chan_ok && L.g == 0)
    p.carry_s[(int64_t)blockIdx.z * p.batch * p.dim + L.b * p.dim + L.d] = sumDt;
}

template <int PASS, int T>
__global__ void __launch_bounds__(kThreads, 9)
    scan_pair_kernel(const ScanArgs p, const __grid_constant__ FastMaps maps) {
  using S = PairSmem<T>;
  constexpr int NPT = kNPT, NP = NPT / 2, CB = kCB, TE = T / kG;
  static_assert(TE % 4 == 0 && T % kCk == 0, "whole 16-byte units; whole saved units");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  const int tid = threadIdx.x, warp = tid >> 5;
  FastLane L;
  L.lane = tid & 31;
  L.c = tid & (CB - 1);
  L.g = 2 * warp + (L.lane >> 4);
  L.b = blockIdx.y;
  L.d0 = (int64_t)blockIdx.x * CB;
  L.d = L.d0 + L.c;
  L.chan_ok = L.d < p.dim;
  const int seg = blockIdx.z;
  const int64_t t_begin = (int64_t)seg * p.seg_len;
  const int64_t t_end = min(p.L, t_begin + p.seg_len);
  const int seg_steps = (int)(t_end - t_begin);
  const int nchunks = (seg_steps + T - 1) / T;
  const bool has_z = PASS == 0 && p.z != nullptr;

  // this thread's states n = g*NPT + j: A, and the initial state
  float Aj[NPT];
  bool zeroA = false;
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    Aj[j] = L.chan_ok ? p.A[L.d * kN + L.g * NPT + j] : -1.f;
    zeroA |= Aj[j] == 0.f;
  }
  float h[NPT];
#pragma unroll
  for (int j = 0; j < NPT; ++j) h[j] = 0.f;
  if (PASS == 0 && L.chan_ok) {
    const int64_t row = L.b * p.dim + L.d;
    if (p.init_state) {
#pragma unroll
      for (int j = 0; j < NPT; ++j) h[j] = p.init_state[row * kN + L.g * NPT + j];
    }
    for (int k = 0; k < seg; ++k) {
      const float sk = p.carry_s[(int64_t)k * p.batch * p.dim + row];
      const float* hk = p.carry_h + ((int64_t)k * p.batch * p.dim + row) * kN + L.g * NPT;
#pragma unroll
      for (int j = 0; j < NPT; ++j) h[j] = fmaf(expf(sk * Aj[j]), h[j], hk[j]);
    }
  }
  if (__syncthreads_or(zeroA)) {
    LaneStates<NPT> hs;
#pragma unroll
    for (int j = 0; j < NPT; ++j) hs.h[j] = h[j];
    precise_pair<PASS>(p, L, t_begin, t_end, hs, reinterpret_cast<float*>(sm + S::oP));
    return;
  }

  // ---- the fast path -------------------------------------------------------
  uint64_t* bar_u = reinterpret_cast<uint64_t*>(sm + S::oBar);   // [kNSU]
  uint64_t* bar_bc = bar_u + kNSU;
  const bool stall = PASS == 0 && p.test_stall && blockIdx.x == 0 && blockIdx.y == 0 &&
                     blockIdx.z == 0;
  const uint64_t wlim = stall ? (uint64_t)p.test_limit_ns : kWaitLimitNs;
  const uint32_t bytes_u = (uint32_t)(S::kRawIO * (has_z ? 3 : 2));
  const uint32_t bytes_bc = (uint32_t)(S::kRawBC * (PASS == 0 ? 2 : 1));
  // thread 0: the copies of chunk k (u / Δ / z into stage k % NSU; B / C into the B/C stage)
  auto issue_u = [&](int k) {
    unsigned char* st = sm + S::oStageU + (k % kNSU) * S::kStageU;
    uint64_t* bar = &bar_u[k % kNSU];
    mbar_arrive_expect_tx(bar, bytes_u);
    if (stall && k == 1) return;  // the failure-path test: armed, never copied
    // time-major boxes (T steps, CB channels) or channel-major ones (CB, T)
    const int tk = (int)(t_begin + (int64_t)k * T);
    const int x = p.bld ? (int)L.d0 : tk, y = p.bld ? tk : (int)L.d0, zc = (int)L.b;
    tma3d(st, &maps.u, bar, x, y, zc);
    tma3d(st + S::kRawIO, &maps.d, bar, x, y, zc);
    if (has_z) tma3d(st + 2 * S::kRawIO, &maps.z, bar, x, y, zc);
  };
  auto issue_bc = [&](int k) {
    mbar_arrive_expect_tx(bar_bc, bytes_bc);
    const int x = (int)(t_begin + (int64_t)k * T), zc = (int)L.b;
    tma3d(sm + S::oStageBC, &maps.b, bar_bc, x, 0, zc);
    if (PASS == 0) tma3d(sm + S::oStageBC + S::kRawBC, &maps.c, bar_bc, x, 0, zc);
  };
  // chunks whose u / Δ / z copies were issued and waited for (the same in every thread)
  int issued = min(kNSU, nchunks), consumed = 0;
  if (tid == 0) {
    for (int s = 0; s <= kNSU; ++s) mbar_init(&bar_u[s], 1);
    fence_mbar_init();
    for (int k = 0; k < issued; ++k) issue_u(k);
    if (nchunks > 0) issue_bc(0);
  }
  __syncthreads();

  // per-thread constants: A·log2(e) and -1/A as packed pairs, the channel's bias and D
  f2 A2p[NP], nIp[NP], hp[NP];
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    A2p[q] = pack2(Aj[2 * q] * kLog2e, Aj[2 * q + 1] * kLog2e);
    nIp[q] = pack2(-1.f / Aj[2 * q], -1.f / Aj[2 * q + 1]);
    hp[q] = pack2(h[2 * q], h[2 * q + 1]);
  }
  const float bias = (p.bias && L.chan_ok) ? p.bias[L.d] : 0.f;
  const float Dd = (p.D && L.chan_ok) ? p.D[L.d] : 0.f;
  const bool sp = p.softplus != 0;
  float sumDt = 0.f;
  float2* const W = reinterpret_cast<float2*>(sm + S::oW);
  float* const BT = reinterpret_cast<float*>(sm + S::oBT);
  float* const CT = BT + S::kBT / 4;
  float* const P = reinterpret_cast<float*>(sm + S::oP);
  // this thread's first output of the segment
  __nv_bfloat16* const ybase =
      PASS == 0 ? static_cast<__nv_bfloat16*>(p.y) + L.b * p.st_y[0] +
                      (L.chan_ok ? L.d : 0) * p.st_y[1] + (t_begin + L.g * TE) * p.st_y[2]
                : nullptr;
  bool failed = false;
  for (int i = 0; i < nchunks; ++i) {
    // 1. chunk i's copies; conversion of this thread's TE steps of its channel;
    //    B (warp 0) and C (warp 1) transposed to [t][n]
    const bool ok = mbar_wait_bounded(&bar_u[i % kNSU], (uint32_t)((i / kNSU) & 1), wlim) &&
                    mbar_wait_bounded(bar_bc, (uint32_t)(i & 1), wlim);
    const int tc = min(T, seg_steps - i * T);
    float du[TE], gate[TE];
    {
      const unsigned char* st = sm + S::oStageU + (i % kNSU) * S::kStageU;
      const __nv_bfloat16* su = reinterpret_cast<const __nv_bfloat16*>(st);
      const __nv_bfloat16* sd = reinterpret_cast<const __nv_bfloat16*>(st + S::kRawIO);
      const __nv_bfloat16* sz = reinterpret_cast<const __nv_bfloat16*>(st + 2 * S::kRawIO);
      float dl[TE], uu[TE], zz[TE];
      if (!p.bld) {
        // this thread's steps in a [c][t] box; 32-step rows (64 bytes) arrive with the
        // 16-byte chunks of row c permuted by (c >> 1) & 3
        const int off = L.c * T + (T == 32 ? ((L.g ^ ((L.c >> 1) & 3)) * TE) : L.g * TE);
        vecio<__nv_bfloat16, TE>::load(sd + off, dl);
        vecio<__nv_bfloat16, TE>::load(su + off, uu);
        if (has_z) vecio<__nv_bfloat16, TE>::load(sz + off, zz);
      } else {
        // a [t][c] box: this thread's steps are CB elements apart
#pragma unroll
        for (int j = 0; j < TE; ++j) {
          const int e = (L.g * TE + j) * CB + L.c;
          dl[j] = __bfloat162float(sd[e]);
          uu[j] = __bfloat162float(su[e]);
          if (has_z) zz[j] = __bfloat162float(sz[e]);
        }
      }
      const bool whole = tc == T;
#pragma unroll
      for (int j = 0; j < TE; ++j) {
        const float x = dl[j] + bias;
        float dt = sp ? softplus_fast(x) : x;
        float u = uu[j];
        if (!whole) {  // steps past the segment: exact no-ops (Δ = 0, u = 0)
          const bool in = L.g * TE + j < tc;
          dt = in ? dt : 0.f;
          u = in ? u : 0.f;
        }
        W[(L.g * TE + j) * CB + L.c] = make_float2(dt, u);
        if (PASS == 1) sumDt += dt;  // every thread of the channel sums its own steps
        if (PASS == 0) {
          du[j] = Dd * u;
          gate[j] = has_z ? silu_fast(zz[j]) : 1.f;
        }
      }
      // warp 0: B, warp 1: C, to [t][n]; lane l moves [n = (l >> 2) + 8 r][t = 16 h + 4 (l & 3) .. + 3]
      if (PASS == 0 || warp == 0) {
        const unsigned char* src = sm + S::oStageBC + warp * S::kRawBC;
        float* dst = warp == 0 ? BT : CT;
#pragma unroll
        for (int h16 = 0; h16 < T / 16; ++h16) {
          const int t0 = 16 * h16 + 4 * (L.lane & 3);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int n = (L.lane >> 2) + 8 * r;
            const float4 q = *reinterpret_cast<const float4*>(src + (n * T + t0) * 4);
            const float v[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[(t0 + e) * S::RowBT + bt_col(t0 + e, n)] = v[e];
          }
        }
      }
    }
    // every thread's copies landed (else the block leaves together); the stages
    // just read are free, the (Δ, u) and B^T / C^T tiles complete
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    consumed = i + 1;
    // 2. refill: u / Δ / z of chunk i + NSU into the stage just converted, B / C of i+1
    if (tid == 0) {
      if (issued < nchunks) issue_u(issued);
      if (i + 1 < nchunks) issue_bc(i + 1);
    }
    if (issued < nchunks) ++issued;
    // training forward: the state at the start of chunk i (and below, after every kCk
    // steps inside it), for the backward
    if (PASS == 0 && p.ckpt != nullptr && L.chan_ok) {
      float* cp = p.ckpt + ((L.b * p.ckpt_nch + t_begin / kCk + i * (T / kCk)) * p.dim + L.d) * kN +
                  L.g * NPT;
#pragma unroll
      for (int q = 0; q < NP; q += 2) {
        float a0, a1, a2, a3;
        unpack2(hp[q], a0, a1);
        unpack2(hp[q + 1], a2, a3);
        *reinterpret_cast<float4*>(cp + 2 * q) = make_float4(a0, a1, a2, a3);
      }
    }
    // 3. the recurrence of chunk i
    {
      auto load_row = [&](const float* row, f2 (&v)[NP]) {
#pragma unroll
        for (int q = 0; q < NP; q += 2) {
          const float4 a = *reinterpret_cast<const float4*>(row + 2 * q);
          v[q] = pack2(a.x, a.y);
          v[q + 1] = pack2(a.z, a.w);
        }
      };
      auto load_step = [&](int t, f2& du2, f2 (&bq)[NP], f2 (&cq)[NP]) {
        const float2 w = W[t * CB + L.c];
        du2 = pack2(w.x, w.y);
        const int col = bt_col(t, L.g * NPT);  // NPT >= 4: the group stays contiguous
        load_row(BT + t * S::RowBT + col, bq);
        if (PASS == 0) load_row(CT + t * S::RowBT + col, cq);
      };
      // Ā pairs from Δ·A·log2 e (one packed multiply per pair), v = -B u / A
      auto discretise = [&](f2 du2, const f2 (&bq)[NP], f2 (&ao)[NP], f2 (&vo)[NP]) {
        float dt, u;
        unpack2(du2, dt, u);
        const f2 dt2 = pack2(dt, dt), u2 = pack2(u, u);
#pragma unroll
        for (int q = 0; q < NP; ++q) {
          float x0, x1;
          unpack2(mul2(dt2, A2p[q]), x0, x1);
          ao[q] = pack2(ex2_fast(x0), ex2_fast(x1));
          vo[q] = mul2(mul2(bq[q], u2), nIp[q]);
        }
      };
      f2 du_l;
      f2 b_l[NP], c_l[NP];
      f2 a_c[NP], v_c[NP], c_c[NP];
      {
        f2 du0;
        f2 b0[NP];
        load_step(0, du0, b0, c_c);
        discretise(du0, b0, a_c, v_c);
        load_step(1, du_l, b_l, c_l);
      }
      float acc[4];
#pragma unroll
      for (int t = 0; t < T; ++t) {
        f2 du_n;
        f2 b_n[NP], c_n[NP], a_n[NP], v_n[NP];
        if (t + 2 < T) load_step(t + 2, du_n, b_n, c_n);
        if (t + 1 < T) discretise(du_l, b_l, a_n, v_n);
#pragma unroll
        for (int q = 0; q < NP; ++q) hp[q] = fma2(a_c[q], sub2(hp[q], v_c[q]), v_c[q]);
        if (PASS == 0) {
          f2 acc2 = mul2(c_c[0], hp[0]);
#pragma unroll
          for (int q = 1; q < NP; ++q) acc2 = fma2(c_c[q], hp[q], acc2);
          float lo, hi;
          unpack2(acc2, lo, hi);
          acc[t % 4] = lo + hi;
          if (t % 4 == 3) {  // the warp's two groups of the channel (lanes l, l ^ 16) added
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = __shfl_xor_sync(0xffffffffu, acc[e], 16);
            if (L.lane < 16)
              *reinterpret_cast<float4*>(P + pair_pidx<T>(warp, L.c, t / 4)) =
                  make_float4(acc[0] + o[0], acc[1] + o[1], acc[2] + o[2], acc[3] + o[3]);
          }
        }
        if (PASS == 0 && (t + 1) % kCk == 0 && t + 1 < T && p.ckpt != nullptr && L.chan_ok &&
            i * T + t + 1 < seg_steps) {
          float* cp = p.ckpt + ((L.b * p.ckpt_nch + t_begin / kCk + i * (T / kCk) + (t + 1) / kCk) *
                                    p.dim + L.d) * kN + L.g * NPT;
#pragma unroll
          for (int q = 0; q < NP; q += 2) {
            float a0, a1, a2, a3;
            unpack2(hp[q], a0, a1);
            unpack2(hp[q + 1], a2, a3);
            *reinterpret_cast<float4*>(cp + 2 * q) = make_float4(a0, a1, a2, a3);
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
          du_l = du_n;
#pragma unroll
          for (int q = 0; q < NP; ++q) {
            b_l[q] = b_n[q];
            c_l[q] = c_n[q];
          }
        }
      }
    }
    // the partials are complete; the next chunk's conversion may overwrite the tiles
    __syncthreads();
    // 4. finalise this thread's steps of chunk i (units g TE/4 .. of its channel's rows)
    if (PASS == 0) {
      float y[TE];
#pragma unroll
      for (int u4 = 0; u4 < TE / 4; ++u4) {
        const int unit = L.g * (TE / 4) + u4;
        const float4 s0 = *reinterpret_cast<const float4*>(P + pair_pidx<T>(0, L.c, unit));
        const float4 s1 = *reinterpret_cast<const float4*>(P + pair_pidx<T>(1, L.c, unit));
        const float sv[4] = {s0.x + s1.x, s0.y + s1.y, s0.z + s1.z, s0.w + s1.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) y[4 * u4 + e] = (sv[e] + du[4 * u4 + e]) * gate[4 * u4 + e];
      }
      __nv_bfloat16* dst = ybase + (int64_t)i * T * p.st_y[2];
      if (L.chan_ok) {
        if (p.vec_y && L.g * TE + TE <= tc) {
          vecio<__nv_bfloat16, TE>::store(dst, y);
        } else {
#pragma unroll
          for (int j = 0; j < TE; ++j)
            if (L.g * TE + j < tc) dst[(int64_t)j * p.st_y[2]] = __float2bfloat16_rn(y[j]);
        }
      }
    }
  }
  if (failed) {
    // a wait ran out: record it, let this block's copies still in flight land
    // (bounded) and leave without writing a state
    if (tid == 0) {
      atomicExch(p.status, 1);
      for (int k = consumed; k < issued; ++k)
        (void)mbar_wait_bounded(&bar_u[k % kNSU], (uint32_t)((k / kNSU) & 1), wlim);
      if (consumed < nchunks) (void)mbar_wait_bounded(bar_bc, (uint32_t)(consumed & 1), wlim);
    }
    return;
  }
#pragma unroll
  for (int q = 0; q < NP; ++q) unpack2(hp[q], h[2 * q], h[2 * q + 1]);
  write_lane_states<PASS>(p, L, seg, h);
  if (PASS == 1) {
    // the channel's ΣΔ: each of its G threads summed its own steps
    float* R = P;
    R[L.g * CB + L.c] = sumDt;
    __syncthreads();
    if (L.chan_ok && L.g == 0)
      p.carry_s[(int64_t)seg * p.batch * p.dim + L.b * p.dim + L.d] =
          (R[L.c] + R[CB + L.c]) + (R[2 * CB + L.c] + R[3 * CB + L.c]);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
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

// 3-D map over a (d2, d1, d0) tensor (d0 fastest, unit stride) with element strides
// s1, s2 of d1, d2 (0: dense) and box (1, b1, b0).
bool map3(CUtensorMap* m, const void* base, CUtensorMapDataType dt, size_t esz, uint64_t d0,
          uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1, uint64_t s1 = 0, uint64_t s2 = 0,
          CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !base) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {(s1 ? s1 : d0) * esz, (s2 ? s2 : d0 * d1) * esz};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int PASS, int T>
cudaError_t launch_pair_one(const ScanArgs& a, const FastMaps& m, int nz, cudaStream_t stream) {
  constexpr size_t bytes = PairSmem<T>::kLaunch;
  auto kern = scan_pair_kernel<PASS, T>;
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
  dim3 grid((unsigned)((a.dim + kCB - 1) / kCB), (unsigned)a.batch, (unsigned)nz);
  kern<<<grid, kThreads, bytes, stream>>>(a, m);
  return cudaGetLastError();
}

// Tensor maps of one launch: u / Δ / z boxes of T steps x CW channels, B / C boxes
// of T steps x N states.
bool fast_maps(const ScanArgs& a, uint32_t CW, uint32_t T, FastMaps& m) {
  memset(&m, 0, sizeof m);
  const uint64_t L = (uint64_t)a.L, D = (uint64_t)a.dim, Bt = (uint64_t)a.batch;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                            f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  // u / Δ / z: time-major (L, dim, batch) with (T, CW) boxes, or channel-major
  // (dim, L, batch) with (CW, T) boxes
  const uint64_t i0 = a.bld ? D : L, i1 = a.bld ? L : D;
  const uint32_t b0 = a.bld ? CW : T, b1 = a.bld ? T : CW;
  const int o1 = a.bld ? 2 : 1;
  const CUtensorMapSwizzle sw = (!a.bld && T == 32) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE;
  bool ok = map3(&m.u, a.u, bf, 2, i0, i1, Bt, b0, b1, a.st_u[o1], a.st_u[0], sw) &&
            map3(&m.d, a.delta, bf, 2, i0, i1, Bt, b0, b1, a.st_d[o1], a.st_d[0], sw) &&
            map3(&m.b, a.B, f32, 4, L, kN, Bt, T, kN) && map3(&m.c, a.C, f32, 4, L, kN, Bt, T, kN);
  if (ok && a.z) ok = map3(&m.z, a.z, bf, 2, i0, i1, Bt, b0, b1, a.st_z[o1], a.st_z[0], sw);
  return ok;
}

cudaError_t launch_pair(const ScanArgs& a, cudaStream_t stream) {
  FastMaps m;
  if (a.nseg > 1) {
    if (!fast_maps(a, kCB, kTCarry, m)) return cudaErrorInvalidValue;
    const cudaError_t e = launch_pair_one<1, kTCarry>(a, m, a.nseg - 1, stream);
    if (e != cudaSuccess) return e;
  }
  if (!fast_maps(a, kCB, kTOut, m)) return cudaErrorInvalidValue;
  return launch_pair_one<0, kTOut>(a, m, a.nseg, stream);
}

}  // namespace

bool scan_fast_applies(const ScanArgs& a, int64_t N, int io_dtype) {
  return N == kN && io_dtype == 1 && !a.euler && !a.force_precise && a.vec_io &&
         a.vec_bc && a.L > 0 && a.L < (int64_t(1) << 31) && a.dim < (int64_t(1) << 31) &&
         encode_fn() != nullptr;
}

bool scan_fast_preferred(const ScanArgs& a) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t warps = (a.dim + kCB - 1) / kCB * 2 * a.batch * a.nseg;
  return warps >= (int64_t)sms * 16;
}

cudaError_t scan_fast_launch(const ScanArgs& a, cudaStream_t stream) {
  return launch_pair(a, stream);
}

}  // namespace ssm
