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
// silu(z).  C, H and M are K-major operands; X ([τ][p], p contiguous) is the
// MN-major B operand of D2, whose core matrices hold 8 steps x 8 channels and
// whose descriptor has the K-step (1024 bytes) as its leading and the MN-step
// (128 bytes) as its stride byte offset.
//
// Persistent CTAs (as many as fit on every SM) walk contiguous ranges of the
// (batch, chunk, head) items, heads fastest, so that consecutive items of one
// group reuse its C tile (each stage remembers whose C it holds) and its C Bᵀ
// rows (kept in registers).  The operands of the next item (C when its group
// changes, H, X and the step terms) are copied into the other of two stages
// while the current one is computed, its C Bᵀ rows are read into registers
// after the current M is built, and z is read into registers, in the mapping
// of the final store, while the products run.  The
// epilogue reads the accumulators with the 16-lane shape (16x256b: thread i
// holds rows i/4 and i/4 + 8 of its warp's 16, columns 2(i%4) and 2(i%4)+1 of
// each group of 8), so all 32 threads of a warp work on its 16 rows, stages y in
// shared memory, and gates and stores it as 16-byte vectors.
// ---------------------------------------------------------------------------
template <int N> struct ChunkTcSmem {
  static constexpr int P = 64;
  static constexpr int RY = P + 8;                                // y rows: 64 + 8 bf16
  // one stage: the operands of one item
  static constexpr size_t sC = 0;                                 // [t][n]  K-major
  static constexpr size_t sH = sC + (size_t)kQ * N * 2;           // [p][n]  K-major
  static constexpr size_t sX = sH + (size_t)P * N * 2;            // [τ][p]  MN-major
  static constexpr size_t sS = sX + (size_t)kQ * P * 2;           // s, β
  static constexpr size_t kStage = sS + 2 * kQ * 4;
  static constexpr size_t oM = 2 * kStage;                        // [t][τ]  K-major
  static constexpr size_t oY = oM + (size_t)kQ * kQ * 2;          // [t][p]  rows of RY
  static constexpr size_t oBar = oY + (size_t)kQ * RY * 2;
  static constexpr size_t oSlot = oBar + 8;
  static constexpr size_t kBytes = oSlot + 8;
  static constexpr size_t kLaunch = kBytes + 128;
  static_assert(kStage % 128 == 0 && oM % 128 == 0 && oY % 16 == 0 && oBar % 8 == 0, "alignment");
};

// Four 32-bit TMEM columns pairs of 16 lanes (16x256b, one repetition): see above.
__device__ __forceinline__ void tc_ld16x256(uint32_t (&r)[4], uint32_t taddr) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}

// Threads of a chunk-output CTA: two warps per TMEM lane quarter, each taking
// half of the accumulators' columns.
constexpr int kChunkThreads = 256;

struct ChunkItem {
  int64_t b;
  int c, h, g, valid;
  int64_t t0;
};

// (batch, chunk, head) of an item, heads fastest (the item count fits 32 bits:
// the launcher checks)
__device__ __forceinline__ ChunkItem chunk_item(const SsdArgs& p, uint32_t item) {
  ChunkItem it;
  const uint32_t H = (uint32_t)p.H, nch = (uint32_t)p.nch;
  const uint32_t bc = item / H;
  it.h = (int)(item - bc * H);
  const uint32_t b = bc / nch;
  it.c = (int)(bc - b * nch);
  it.b = b;
  it.g = it.h / (int)(p.H / p.G);
  it.t0 = (int64_t)it.c * kQ;
  it.valid = (int)min64(kQ, p.L - it.t0);
  return it;
}

template <int N>
__global__ void __launch_bounds__(kChunkThreads, 2) ssd_chunk_tc_kernel(const SsdArgs p) {
  using S = ChunkTcSmem<N>;
  constexpr int P = S::P, KB = N / 8, RY = S::RY, NT = kChunkThreads;
  constexpr int kMv = kQ * kQ / 8 / NT;      // 8-wide groups of M a thread builds
  constexpr int kVec = kQ * (P / 8) / NT;    // 16-byte vectors of y a thread stores
  extern __shared__ unsigned char ck_smem_raw[];
  unsigned char* sm = ck_smem_raw + ((128u - (smem_u32(ck_smem_raw) & 127u)) & 127u);
  unsigned char* sM = sm + S::oM;
  __nv_bfloat16* sY = reinterpret_cast<__nv_bfloat16*>(sm + S::oY);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + S::oBar);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + S::oSlot);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t total = (uint32_t)(p.batch * p.nch * p.H);
  const int64_t io_step = p.H * P;  // elements between steps of x, z, y

  if (warp == 0) {  // the accumulators first: the copies below overlap the allocation
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(2 * kQ));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }

  // the operands of one item into a stage (16-byte cp.async; thread e's vector is
  // row 8i + (e & 7) of core-matrix column e >> 3, so 8 consecutive threads fill
  // one 128-byte core matrix), as one commit group
  auto copy_stage = [&](const ChunkItem& w, unsigned char* st, bool with_c) {
    const __nv_bfloat16* gC =
        static_cast<const __nv_bfloat16*>(p.C) + ((w.b * p.L + w.t0) * p.G + w.g) * N;
    const __nv_bfloat16* gH = p.ws_hin + ((w.b * p.nch + w.c) * p.H + w.h) * (int64_t)(P * N);
    for (int e = tid; e < kQ * KB; e += NT) {
      const int kb = (e >> 3) % KB, r = ((e >> 3) / KB) * 8 + (e & 7);
      const bool ok = r < w.valid;
      if (with_c)
        cp_async16_zfill(st + S::sC + kmaj_off(r, 8 * kb, KB),
                         gC + (int64_t)(ok ? r : 0) * p.G * N + 8 * kb, ok);
      cp_async16_zfill(st + S::sH + kmaj_off(r, 8 * kb, KB), gH + (int64_t)r * N + 8 * kb, true);
    }
    const __nv_bfloat16* gX =
        static_cast<const __nv_bfloat16*>(p.x) + ((w.b * p.L + w.t0) * p.H + w.h) * P;
    for (int e = tid; e < kQ * (P / 8); e += NT) {
      const int nb = (e >> 3) % (P / 8), tau = ((e >> 3) / (P / 8)) * 8 + (e & 7);
      const bool ok = tau < w.valid;
      cp_async16_zfill(st + S::sX + mnmaj_off(tau, 8 * nb, P / 8),
                       gX + (int64_t)(ok ? tau : 0) * io_step + 8 * nb, ok);
    }
    if (tid < 2 * kQ / 4)
      cp_async16_zfill(st + S::sS + 16 * tid,
                       p.ws_terms + ((w.b * p.nch + w.c) * p.H + w.h) * kSsdTermsRec + 4 * tid, true);
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // C Bᵀ rows of an item for M: thread e's 8 consecutive τ of row t (global, rows
  // of 64 floats; the 16 x 16 tiles on and below the diagonal were written, and
  // every 8-wide group that reaches τ <= t lies in one of them)
  float4 gv[kMv][2];
  float dh_pre = 0.f;  // the item's D
  auto fetch_cb = [&](const ChunkItem& w) {
    const float* gG = p.ws_cb + ((w.b * p.nch + w.c) * p.G + w.g) * (int64_t)(kQ * kQ);
#pragma unroll
    for (int i = 0; i < kMv; ++i) {
      const int e = tid + i * NT, kb = (e >> 3) % 8, t = ((e >> 3) / 8) * 8 + (e & 7);
      if (8 * kb <= t) {
        gv[i][0] = __ldg(reinterpret_cast<const float4*>(gG + t * kQ + 8 * kb));
        gv[i][1] = __ldg(reinterpret_cast<const float4*>(gG + t * kQ + 8 * kb + 4));
      } else {
        gv[i][0] = gv[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  };

  // this CTA's items: a contiguous range (heads fastest), so consecutive items of
  // one (batch, chunk, group) reuse its C tile (kept per stage) and C Bᵀ rows
  const uint32_t beg = (uint32_t)((uint64_t)blockIdx.x * total / gridDim.x);
  const uint32_t end = (uint32_t)((uint64_t)(blockIdx.x + 1) * total / gridDim.x);
  auto group_key = [&](const ChunkItem& w) { return (uint32_t)((w.b * p.nch + w.c) * p.G + w.g); };
  uint32_t ckey0 = 0xffffffffu, ckey1 = 0xffffffffu;  // the group whose C each stage holds
  uint32_t item = beg;
  ChunkItem w = chunk_item(p, item);
  uint32_t gkey = group_key(w);  // the group whose C Bᵀ rows gv holds
  if (item < end) {
    copy_stage(w, sm, true);
    ckey0 = gkey;
    fetch_cb(w);
    dh_pre = p.D ? __ldg(p.D + w.h) : 0.f;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *slot;
  // epilogue share: lane quarter warp % 4, column groups 4 (warp / 4) .. + 3
  const int quarter = warp & 3, jh = 4 * (warp >> 2);
  const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16);
  const int r0 = 16 * quarter + (lane >> 2), cq = 2 * (lane & 3);
  bool ok = true;
  for (int k = 0; item < end; ++k, ++item) {
    const float Dh = dh_pre;
    unsigned char* st = sm + (size_t)(k & 1) * S::kStage;
    const float* sS = reinterpret_cast<const float*>(st + S::sS);
    const float* sBeta = sS + kQ;
    const uint32_t next = item + 1;
    const ChunkItem wn = chunk_item(p, next < end ? next : item);
    const uint32_t nkey = group_key(wn);
    if (next < end) {
      const int ns = (k + 1) & 1;
      copy_stage(wn, sm + (size_t)ns * S::kStage, (ns ? ckey1 : ckey0) != nkey);
      if (ns) ckey1 = nkey;
      else ckey0 = nkey;
      asm volatile("cp.async.wait_group 1;" ::: "memory");  // this item's group
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    // M[t][τ] in bf16, K-major, in packed pairs: G β 2^((s_t - s_τ) log2 e)
#pragma unroll
    for (int i = 0; i < kMv; ++i) {
      const int e = tid + i * NT, kb = (e >> 3) % 8, t = ((e >> 3) / 8) * 8 + (e & 7);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (8 * kb <= t) {
        f2 sq[4], bq[4];
        lds_pairs(sS + 8 * kb, sq[0], sq[1]);
        lds_pairs(sS + 8 * kb + 4, sq[2], sq[3]);
        lds_pairs(sBeta + 8 * kb, bq[0], bq[1]);
        lds_pairs(sBeta + 8 * kb + 4, bq[2], bq[3]);
        const float stt = sS[t];
        const f2 st2 = pack2(stt, stt), l2 = pack2(kLog2e, kLog2e);
        const f2 gq[4] = {pack2(gv[i][0].x, gv[i][0].y), pack2(gv[i][0].z, gv[i][0].w),
                          pack2(gv[i][1].x, gv[i][1].y), pack2(gv[i][1].z, gv[i][1].w)};
        const bool diag = 8 * kb + 7 > t;  // the block holds τ > t: those are zero
        uint32_t* vw = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float x0, x1;
          unpack2(mul2(sub2(st2, sq[q]), l2), x0, x1);
          float m0, m1;
          unpack2(mul2(mul2(gq[q], bq[q]), pack2(ex2_fast(x0), ex2_fast(x1))), m0, m1);
          if (diag) {
            m0 = 8 * kb + 2 * q <= t ? m0 : 0.f;
            m1 = 8 * kb + 2 * q + 1 <= t ? m1 : 0.f;
          }
          vw[q] = pack_bf16x2(m0, m1);
        }
      }
      *reinterpret_cast<uint4*>(sM + kmaj_off(t, 8 * kb, 8)) = v;
    }
    if (next < end) {
      if (nkey != gkey) fetch_cb(wn);  // else gv already holds these rows
      gkey = nkey;
      dh_pre = p.D ? __ldg(p.D + wn.h) : 0.f;
    }
    // z for the final store (row e / 8, channels (e % 8) * 8 .. + 7)
    uint4 zr[kVec];
    const __nv_bfloat16* gZ =
        static_cast<const __nv_bfloat16*>(p.z) + ((w.b * p.L + w.t0) * p.H + w.h) * P;
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const int e = tid + i * NT, row = e >> 3, c8 = e & 7;
      zr[i] = (p.z && row < w.valid)
                  ? __ldg(reinterpret_cast<const uint4*>(gZ + (int64_t)row * io_step + 8 * c8))
                  : make_uint4(0, 0, 0, 0);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (tid == 0) {
      // D1 = C Hᵀ into columns 0..63
      constexpr uint32_t id1 = tc_idesc_bf16(kQ, P);
#pragma unroll
      for (int kk = 0; kk < N / 16; ++kk) {
        const uint64_t ad = tc_desc(smem_u32(st + S::sC) + 256u * kk, 128, KB * 128);
        const uint64_t bd = tc_desc(smem_u32(st + S::sH) + 256u * kk, 128, KB * 128);
        tc_mma(tmem, ad, bd, id1, kk > 0);
      }
      // D2 = M X into columns 64..127 (X MN-major: bit 16 of the instruction descriptor)
      constexpr uint32_t id2 = tc_idesc_bf16(kQ, P) | (1u << 16);
#pragma unroll
      for (int kk = 0; kk < kQ / 16; ++kk) {
        const uint64_t ad = tc_desc(smem_u32(sM) + 256u * kk, 128, 8 * 128);
        const uint64_t bd = tc_desc(smem_u32(st + S::sX) + 2u * (P / 8) * 128 * kk, (P / 8) * 128, 128);
        tc_mma(tmem + kQ, ad, bd, id2, kk > 0);
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                       smem_u32(bar))
                   : "memory");
    }
    ok = mbar_wait_bounded(bar, (uint32_t)(k & 1));
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (__syncthreads_or(!ok)) {  // every thread leaves together
      ok = false;
      break;
    }
    // epilogue: rows 16q + lane/4 and 16q + lane/4 + 8 of quarter q, columns
    // 8j + 2(lane%4) and the next for this warp's four j, of both accumulators
    {
      const unsigned char* sX = st + S::sX;
      uint32_t d1[4][4], d2[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        tc_ld16x256(d1[j], ta + 8 * (jh + j));
        tc_ld16x256(d2[j], ta + kQ + 8 * (jh + j));
      }
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      const f2 dh2 = pack2(Dh, Dh);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int t = r0 + 8 * hf;
        const float et = ex2_fast(sS[t] * kLog2e);
        const f2 et2 = pack2(et, et);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int col = 8 * (jh + j) + cq;
          const float2 xv = __bfloat1622float2(
              *reinterpret_cast<const __nv_bfloat162*>(sX + mnmaj_off(t, col, P / 8)));
          const f2 a = pack2(__uint_as_float(d1[j][2 * hf]), __uint_as_float(d1[j][2 * hf + 1]));
          const f2 c2 = pack2(__uint_as_float(d2[j][2 * hf]), __uint_as_float(d2[j][2 * hf + 1]));
          float v0, v1;
          unpack2(fma2(dh2, pack2(xv.x, xv.y), fma2(et2, a, c2)), v0, v1);
          *reinterpret_cast<uint32_t*>(sY + t * RY + col) = pack_bf16x2(v0, v1);
        }
      }
    }
    // the accumulators are read: the next item's products may overwrite them
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    // gate and store: 16-byte vectors of y
    __nv_bfloat16* yg = static_cast<__nv_bfloat16*>(p.y) + ((w.b * p.L + w.t0) * p.H + w.h) * P;
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const int e = tid + i * NT, row = e >> 3, c8 = e & 7;
      if (row >= w.valid) continue;
      uint4 v = *reinterpret_cast<const uint4*>(sY + row * RY + 8 * c8);
      if (p.z) {
        uint32_t* wv = reinterpret_cast<uint32_t*>(&v);
        const uint32_t* zw = reinterpret_cast<const uint32_t*>(&zr[i]);
        const f2 nl2 = pack2(-kLog2e, -kLog2e), one2 = pack2(1.f, 1.f);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          // y silu(z) = y z / (1 + 2^(-z log2 e)), in packed pairs
          const float2 yv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[q]));
          const float2 zv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&zw[q]));
          const f2 z2 = pack2(zv.x, zv.y);
          float e0, e1;
          unpack2(mul2(z2, nl2), e0, e1);
          float d0, d1;
          unpack2(add2(pack2(ex2_fast(e0), ex2_fast(e1)), one2), d0, d1);
          float o0, o1;
          unpack2(mul2(mul2(pack2(yv.x, yv.y), z2), pack2(rcp_fast(d0), rcp_fast(d1))), o0, o1);
          wv[q] = pack_bf16x2(o0, o1);
        }
      }
      *reinterpret_cast<uint4*>(yg + (int64_t)row * io_step + 8 * c8) = v;
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    w = wn;
  }
  if (!ok && tid == 0) atomicExch(p.status, 1);  // products never completed: the rest is skipped
  asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy outlives the CTA
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kQ));
}

template <int N>
cudaError_t chunk_tc_typed(const SsdArgs& a, cudaStream_t s) {
  constexpr size_t bytes = ChunkTcSmem<N>::kLaunch;
  static int configured_dev = -1, resident = 1, sms = 148;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(ssd_chunk_tc_kernel<N>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(ssd_chunk_tc_kernel<N>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    // CTAs an SM holds: by shared memory (with the per-block reservation) and by
    // registers; 128 TMEM columns a CTA allow at most 4
    int smem_sm = 0, reserved = 0;
    cudaFuncAttributes fa{};
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, ssd_chunk_tc_kernel<N>);
    if (e != cudaSuccess) return e;
    const int by_smem = smem_sm / (int)(bytes + (size_t)reserved);
    const int regs = fa.numRegs > 0 ? fa.numRegs : 255;
    const int by_regs = 65536 / (regs * kChunkThreads);
    resident = by_smem < by_regs ? by_smem : by_regs;
    resident = resident < 1 ? 1 : (resident > 4 ? 4 : resident);
    configured_dev = dev;
  }
  const int64_t total = a.batch * a.nch * a.H;
  if (total >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  const int64_t grid = (int64_t)sms * resident < total ? (int64_t)sms * resident : total;
  if (grid <= 0) return cudaSuccess;
  ssd_chunk_tc_kernel<N><<<(unsigned)grid, kChunkThreads, bytes, s>>>(a);
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
