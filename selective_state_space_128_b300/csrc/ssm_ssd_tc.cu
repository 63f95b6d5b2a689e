// C Bᵀ of Mamba-2's chunked SSD on the fifth-generation tensor cores (tcgen05).
//
// The chapter page ("14.1 SSM(State Space Models)과 Mamba 아키텍처의 부상",
// §5.2) computes the SSM chunk by chunk; inside a chunk the quadratic form
// needs G[t][τ] = C_t · B_τ for every pair of steps of the chunk, once per
// (batch, chunk, group) since every head of a group shares B and C.
//
// One CTA of 128 threads per (batch, chunk, group): it stages the chunk's 64
// rows of C and of B (N bf16 each, K-major: the state index n is the
// contraction) in shared memory in the tensor core's canonical no-swizzle
// layout, one thread issues the N/16 tcgen05.mma instructions of D = C Bᵀ
// (M = N_mma = 64, K = N) into a 64-column TMEM accumulator, and after their
// commit arrives on an mbarrier each warp reads its rows back (tcgen05.ld) and
// writes them as fp32 rows of 64, the 16 x 16 tiles on and below the diagonal
// only (the chunk outputs read no others).  With M = 64 the accumulator's row
// 16q + i sits in TMEM lane 32q + i: warp q reads its own lane quarter and its
// first 16 lanes hold rows 16q .. 16q + 15.
//
// Layout in shared memory (both operands): 8-row x 16-byte core matrices, the
// core matrix of rows 8i..8i+7 and columns 8j..8j+7 at (i * N/8 + j) * 128
// bytes, so core matrices adjacent along K are 128 bytes apart (the
// descriptor's leading byte offset) and along M 16 N bytes apart (its stride
// byte offset).  A K = 16 step of the MMA reads two core matrices along K and
// the next step starts 256 bytes further.
//
// The only wait is on the commit's mbarrier and is bounded; the TMEM columns
// are freed on every path.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kQ = kSsdChunk;   // chunk length: the MMA's M and N
constexpr int kTcThreads = 128;

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (all in 16-byte units), descriptor version 1, no
// swizzling.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M x N.
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// One tcgen05.mma (one thread): D (TMEM) = A B (+ D when `accumulate`).
__device__ __forceinline__ void tc_mma(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// 32 consecutive TMEM columns of this warp's 32 lanes (one per thread).
__device__ __forceinline__ void tc_ld32(uint32_t (&r)[32], uint32_t taddr) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 16-byte asynchronous copy global -> shared; with `valid` false nothing is read
// and the destination is zero-filled.
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(valid ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Index (bytes) of element (row, col) of a K-major canonical tile with KB core
// matrices along K (col = the K index), or of an MN-major one with MB core
// matrices along MN (row = the K index, col the MN index).
__device__ __forceinline__ int kmaj_off(int row, int col, int KB) {
  return ((row >> 3) * KB + (col >> 3)) * 128 + (row & 7) * 16 + (col & 7) * 2;
}
__device__ __forceinline__ int mnmaj_off(int krow, int mncol, int MB) {
  return ((krow >> 3) * MB + (mncol >> 3)) * 128 + (krow & 7) * 16 + (mncol & 7) * 2;
}

template <int N> struct CbTcSmem {
  static constexpr size_t kTile = (size_t)kQ * N * 2;  // one operand, bf16
  static constexpr size_t oC = 0, oB = kTile, oBar = 2 * kTile, oSlot = oBar + 8;
  static constexpr size_t kBytes = oSlot + 8;
  static constexpr size_t kLaunch = kBytes + 128;  // room to align the base
};

template <int N>
__global__ void __launch_bounds__(kTcThreads) ssd_cb_tc_kernel(const SsdArgs p) {
  using S = CbTcSmem<N>;
  constexpr int KB = N / 8;  // core matrices along K
  extern __shared__ unsigned char cb_smem_raw[];
  unsigned char* sm = cb_smem_raw + ((128u - (smem_u32(cb_smem_raw) & 127u)) & 127u);
  unsigned char* sC = sm + S::oC;
  unsigned char* sB = sm + S::oB;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + S::oBar);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + S::oSlot);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, g = blockIdx.y;
  const int64_t b = blockIdx.z;
  const int64_t t0 = (int64_t)c * kQ;
  const int valid = (int)min64(kQ, p.L - t0);  // rows past the sequence are zero

  if (warp == 0) {  // the accumulator first: the copies below overlap the allocation
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(kQ));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  // stage C and B: 16-byte vectors (8 states of one step) into their core-matrix
  // rows; thread e's vector is row 8i + (e & 7) of core-matrix column (e >> 3) % KB,
  // so 8 consecutive threads fill one 128-byte core matrix
  const __nv_bfloat16* gC = static_cast<const __nv_bfloat16*>(p.C) + ((b * p.L + t0) * p.G + g) * N;
  const __nv_bfloat16* gB = static_cast<const __nv_bfloat16*>(p.B) + ((b * p.L + t0) * p.G + g) * N;
  for (int e = tid; e < kQ * KB; e += kTcThreads) {
    const int kb = (e >> 3) % KB, r = ((e >> 3) / KB) * 8 + (e & 7);
    const bool ok = r < valid;
    const int64_t src = (int64_t)(ok ? r : 0) * p.G * N + 8 * kb;
    cp_async16_zfill(sC + kmaj_off(r, 8 * kb, KB), gC + src, ok);
    cp_async16_zfill(sB + kmaj_off(r, 8 * kb, KB), gB + src, ok);
  }
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
  // the operands written by threads become visible to the tensor core's (async) proxy
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *slot;

  if (tid == 0) {
    constexpr uint32_t idesc = tc_idesc_bf16(kQ, kQ);
    const uint32_t lbo = 128, sbo = KB * 128;
#pragma unroll
    for (int k = 0; k < N / 16; ++k) {
      const uint64_t ad = tc_desc(smem_u32(sC) + 256u * k, lbo, sbo);
      const uint64_t bd = tc_desc(smem_u32(sB) + 256u * k, lbo, sbo);
      const uint32_t acc = k > 0 ? 1u : 0u;  // the first step overwrites D
      asm volatile(
          "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
          " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
          "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
          : "memory");
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
  }
  const bool ok = mbar_wait_bounded(bar, 0);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (ok) {
    // warp q reads its lane quarter; its lanes 0-15 hold rows t = 16q + lane, whose
    // tiles on and below the diagonal are columns 0 .. 16q + 15
    uint32_t r[32];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(32 * h);
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
          "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
          "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
          : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
            "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
            "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
            "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
            "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
            "=r"(r[30]), "=r"(r[31])
          : "r"(taddr));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      if (lane < 16 && 32 * h <= 16 * warp + 15) {
        float* out = p.ws_cb + ((b * p.nch + c) * p.G + g) * (int64_t)(kQ * kQ) +
                     (int64_t)(16 * warp + lane) * kQ + 32 * h;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (32 * h + 4 * q <= 16 * warp + 15)
            *reinterpret_cast<float4*>(out + 4 * q) =
                make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                            __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
      }
    }
  } else if (tid == 0) {
    atomicExch(p.status, 1);  // the MMA never completed: report it, write nothing
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kQ));
}

// ---------------------------------------------------------------------------
// Chunk outputs on tcgen05: per (batch, chunk, head), with M = 64 rows t,
//   D1 = C Hᵀ            (K = N: the state entering the chunk, [p][n] bf16)
//   D2 = M X,  M[t][τ] = (τ <= t) C_t·B_τ exp(s_t - s_τ) β_τ   (K = τ)
// in two 64-column TMEM accumulators, then y = exp(s_t) D1 + D2 + D x, gated by
// silu(z), through a shared tile and 16-byte stores.  C, H and M are K-major
// operands; X ([τ][p], p contiguous) is the MN-major B operand of D2, whose
// core matrices hold 8 steps x 8 channels and whose descriptor has the K-step
// (1024 bytes) as its leading and the MN-step (128 bytes) as its stride byte
// offset.
// ---------------------------------------------------------------------------
template <int N> struct ChunkTcSmem {
  static constexpr int P = 64;
  static constexpr size_t oC = 0;                                 // [t][n]  K-major
  static constexpr size_t oH = oC + (size_t)kQ * N * 2;           // [p][n]  K-major
  static constexpr size_t oM = oH + (size_t)P * N * 2;            // [t][τ]  K-major
  static constexpr size_t oX = oM + (size_t)kQ * kQ * 2;          // [τ][p]  MN-major
  static constexpr size_t oZ = oX + (size_t)kQ * P * 2;           // [t][p]  rows of 64 + 8
  static constexpr int RZ = P + 8;
  static constexpr size_t oG = oZ + (size_t)kQ * RZ * 2;          // C Bᵀ [t][τ] fp32, rows of 64 + 4
  static constexpr int RG = kQ + 4;
  static constexpr size_t oS = oG + (size_t)kQ * RG * 4;          // s, β
  static constexpr size_t oBar = oS + 2 * kQ * 4;
  static constexpr size_t oSlot = oBar + 8;
  static constexpr size_t kBytes = oSlot + 8;
  static constexpr size_t kLaunch = kBytes + 128;
};

template <int N>
__global__ void __launch_bounds__(kTcThreads) ssd_chunk_tc_kernel(const SsdArgs p) {
  using S = ChunkTcSmem<N>;
  constexpr int P = S::P, KB = N / 8;
  extern __shared__ unsigned char ck_smem_raw[];
  unsigned char* sm = ck_smem_raw + ((128u - (smem_u32(ck_smem_raw) & 127u)) & 127u);
  unsigned char* sC = sm + S::oC;
  unsigned char* sH = sm + S::oH;
  unsigned char* sM = sm + S::oM;
  unsigned char* sX = sm + S::oX;
  __nv_bfloat16* sZ = reinterpret_cast<__nv_bfloat16*>(sm + S::oZ);
  float* sG = reinterpret_cast<float*>(sm + S::oG);
  float* sS = reinterpret_cast<float*>(sm + S::oS);
  float* sBeta = sS + kQ;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + S::oBar);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + S::oSlot);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, h = blockIdx.y;
  const int64_t b = blockIdx.z;
  const int64_t t0 = (int64_t)c * kQ;
  const int valid = (int)min64(kQ, p.L - t0);
  const int g = h / (p.H / p.G);

  if (warp == 0) {  // the accumulators first: the copies below overlap the allocation
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(2 * kQ));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  // copies (16-byte cp.async; thread e's vector is row 8i + (e & 7) of core-matrix
  // column e >> 3, so 8 consecutive threads fill one 128-byte core matrix)
  const __nv_bfloat16* gC = static_cast<const __nv_bfloat16*>(p.C) + ((b * p.L + t0) * p.G + g) * N;
  const __nv_bfloat16* gH = p.ws_hin + ((b * p.nch + c) * p.H + h) * (int64_t)(P * N);
  for (int e = tid; e < kQ * KB; e += kTcThreads) {
    const int kb = (e >> 3) % KB, r = ((e >> 3) / KB) * 8 + (e & 7);
    const bool ok = r < valid;
    cp_async16_zfill(sC + kmaj_off(r, 8 * kb, KB), gC + (int64_t)(ok ? r : 0) * p.G * N + 8 * kb, ok);
    cp_async16_zfill(sH + kmaj_off(r, 8 * kb, KB), gH + (int64_t)r * N + 8 * kb, true);
  }
  const __nv_bfloat16* gX = static_cast<const __nv_bfloat16*>(p.x) + ((b * p.L + t0) * p.H + h) * P;
  const __nv_bfloat16* gZ = static_cast<const __nv_bfloat16*>(p.z) + ((b * p.L + t0) * p.H + h) * P;
  for (int e = tid; e < kQ * (P / 8); e += kTcThreads) {
    const int nb = (e >> 3) % (P / 8), tau = ((e >> 3) / (P / 8)) * 8 + (e & 7);
    const bool ok = tau < valid;
    // X as the MN-major operand: core matrix (τ block, p block), 8 steps of 16 bytes
    cp_async16_zfill(sX + mnmaj_off(tau, 8 * nb, P / 8), gX + (int64_t)(ok ? tau : 0) * p.H * P + 8 * nb, ok);
    if (p.z)
      cp_async16_zfill(sZ + tau * S::RZ + 8 * nb, gZ + (int64_t)(ok ? tau : 0) * p.H * P + 8 * nb, ok);
  }
  const float* gG = p.ws_cb + ((b * p.nch + c) * p.G + g) * (int64_t)(kQ * kQ);
  for (int e = tid; e < kQ * kQ / 4; e += kTcThreads) {
    const int r = e / (kQ / 4), v = e % (kQ / 4);
    if (4 * v <= r)  // the tiles on and below the diagonal were written
      cp_async16_zfill(sG + r * S::RG + 4 * v, gG + r * kQ + 4 * v, true);
  }
  if (tid < 2 * kQ / 4)
    cp_async16_zfill(sS + 4 * tid, p.ws_terms + ((b * p.nch + c) * p.H + h) * kSsdTermsRec + 4 * tid, true);
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
  __syncthreads();
  // M[t][τ] in bf16, K-major: thread e builds 8 consecutive τ of row t
  for (int e = tid; e < kQ * kQ / 8; e += kTcThreads) {
    const int kb = (e >> 3) % 8, t = ((e >> 3) / 8) * 8 + (e & 7);
    const float st = sS[t];
    float m[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int tau = 8 * kb + j;
      m[j] = tau <= t ? sG[t * S::RG + tau] * __expf(st - sS[tau]) * sBeta[tau] : 0.f;
    }
    uint4 v;
    v.x = pack_bf16x2(m[0], m[1]);
    v.y = pack_bf16x2(m[2], m[3]);
    v.z = pack_bf16x2(m[4], m[5]);
    v.w = pack_bf16x2(m[6], m[7]);
    *reinterpret_cast<uint4*>(sM + kmaj_off(t, 8 * kb, 8)) = v;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *slot;
  if (tid == 0) {
    // D1 = C Hᵀ into columns 0..63
    constexpr uint32_t id1 = tc_idesc_bf16(kQ, P);
#pragma unroll
    for (int k = 0; k < N / 16; ++k) {
      const uint64_t ad = tc_desc(smem_u32(sC) + 256u * k, 128, KB * 128);
      const uint64_t bd = tc_desc(smem_u32(sH) + 256u * k, 128, KB * 128);
      tc_mma(tmem, ad, bd, id1, k > 0);
    }
    // D2 = M X into columns 64..127 (X MN-major: bit 16 of the instruction descriptor)
    constexpr uint32_t id2 = tc_idesc_bf16(kQ, P) | (1u << 16);
#pragma unroll
    for (int k = 0; k < kQ / 16; ++k) {
      const uint64_t ad = tc_desc(smem_u32(sM) + 256u * k, 128, 8 * 128);
      const uint64_t bd = tc_desc(smem_u32(sX) + 2u * (P / 8) * 128 * k, (P / 8) * 128, 128);
      tc_mma(tmem + kQ, ad, bd, id2, k > 0);
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
  }
  const bool ok = mbar_wait_bounded(bar, 0);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  // epilogue: warp q's lanes 0-15 hold row t = 16q + lane of both accumulators
  __nv_bfloat16* sY = reinterpret_cast<__nv_bfloat16*>(sC);  // C is no longer read: [t][p] rows of RZ
  const int t = 16 * warp + lane;
  const float Dh = p.D ? p.D[h] : 0.f;
  const float et = lane < 16 ? __expf(sS[t & (kQ - 1)]) : 0.f;
  if (ok) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t r1[32], r2[32];
      tc_ld32(r1, tmem + ((uint32_t)(32 * warp) << 16) + 32 * hh);
      tc_ld32(r2, tmem + ((uint32_t)(32 * warp) << 16) + kQ + 32 * hh);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      if (lane < 16) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int col = 32 * hh + j;
          const __nv_bfloat162 xv =
              *reinterpret_cast<const __nv_bfloat162*>(sX + mnmaj_off(t, col, P / 8));
          float v0 = fmaf(et, __uint_as_float(r1[j]), __uint_as_float(r2[j])) + Dh * __low2float(xv);
          float v1 = fmaf(et, __uint_as_float(r1[j + 1]), __uint_as_float(r2[j + 1])) +
                     Dh * __high2float(xv);
          if (p.z) {
            const __nv_bfloat162 zv = *reinterpret_cast<const __nv_bfloat162*>(sZ + t * S::RZ + col);
            v0 *= silu_precise(__low2float(zv));
            v1 *= silu_precise(__high2float(zv));
          }
          *reinterpret_cast<__nv_bfloat162*>(sY + t * S::RZ + col) = __floats2bfloat162_rn(v0, v1);
        }
      }
    }
  } else if (tid == 0) {
    atomicExch(p.status, 1);  // the MMAs never completed: report it, write nothing
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kQ));
  if (!ok) return;
  __nv_bfloat16* yg = static_cast<__nv_bfloat16*>(p.y) + ((b * p.L + t0) * p.H + h) * P;
  for (int e = tid; e < kQ * (P / 8); e += kTcThreads) {
    const int row = e / (P / 8), c8 = e % (P / 8);
    if (row < valid)
      *reinterpret_cast<uint4*>(yg + (int64_t)row * p.H * P + 8 * c8) =
          *reinterpret_cast<const uint4*>(sY + row * S::RZ + 8 * c8);
  }
}

template <int N>
cudaError_t chunk_tc_typed(const SsdArgs& a, cudaStream_t s) {
  constexpr size_t bytes = ChunkTcSmem<N>::kLaunch;
  static int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    const cudaError_t e = cudaFuncSetAttribute(ssd_chunk_tc_kernel<N>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  ssd_chunk_tc_kernel<N><<<dim3((unsigned)a.nch, (unsigned)a.H, (unsigned)a.batch), kTcThreads, bytes,
                           s>>>(a);
  return cudaGetLastError();
}

template <int N>
cudaError_t cb_tc_typed(const SsdArgs& a, cudaStream_t s) {
  constexpr size_t bytes = CbTcSmem<N>::kLaunch;
  static int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    const cudaError_t e = cudaFuncSetAttribute(ssd_cb_tc_kernel<N>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  ssd_cb_tc_kernel<N><<<dim3((unsigned)a.nch, (unsigned)a.G, (unsigned)a.batch), kTcThreads, bytes,
                        s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t ssd_chunk_tc_launch(const SsdArgs& a, int64_t N, cudaStream_t stream) {
  switch (N) {
    case 64: return chunk_tc_typed<64>(a, stream);
    case 128: return chunk_tc_typed<128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t ssd_cb_tc_launch(const SsdArgs& a, int64_t N, cudaStream_t stream) {
  switch (N) {
    case 64: return cb_tc_typed<64>(a, stream);
    case 128: return cb_tc_typed<128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssm
