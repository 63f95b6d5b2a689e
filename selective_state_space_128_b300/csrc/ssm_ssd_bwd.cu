// Backward of Mamba-2's scalar-A SSM (SSD), through the selective scan's
// backward.
//
// The chapter page ("14.1 SSM(State Space Models)과 Mamba 아키텍처의 부상",
// §5.1) restricts A to a scalar per step times the identity: per head h, SSD
// is the selective scan of each of the head's P channels with A[n] = a_h for
// every state n, the head's step Δ_t shared by its channels, and the B, C of
// the head's group.  Its derivatives are therefore the scan backward's
// per-channel derivatives (ssm_scan_bwd: states recomputed per chunk, the
// adjoint in reverse) summed over the channels that share each parameter:
// the head's P channels for dΔ, dA, dD and d dt_bias, every channel of the
// group for dB and dC (the scan backward already sums a batch row's channels).
//
// Per group g the call gathers the group's channels into the scan's layout
// (batch, channels, L) in fp32 (x, the per-channel Δ, z, dy; B, C as (batch, N,
// L); the per-channel A, D, bias tables; the states), runs ssm_scan_bwd with
// float32 I/O (so no derivative is rounded before its sums over channels),
// then scatters dx, dz, dB, dC, d init_state back to SSD's layouts and adds the
// per-head sums in a fixed order.
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/ssm.h"
#include "ssm_device.cuh"

namespace ssm {

struct SsdBwdGlue {
  // SSD side (Mamba-2 layouts)
  const __nv_bfloat16 *x, *dt, *z, *dy, *B, *C;
  const float *A, *D, *dt_bias, *init, *dfin;
  __nv_bfloat16 *dx, *ddt, *dz;
  float *dA, *dB, *dC, *dD, *ddt_bias, *dinit;
  // scan side (one group): (batch, Dc, L) rows, (batch, N, L) B/C, (Dc, N) A
  float *u, *dl, *zz, *dyy, *du, *ddl, *dzz, *Bg, *Cg, *dBg, *dCg, *Ag, *dAg, *Dg, *biasg, *dDg,
      *dbiasg, *initg, *dfing, *dinitg;
  int64_t batch, L, H, P, G, N, hpg, Dc, g;
};

__device__ __forceinline__ float bf(const __nv_bfloat16 v) { return __bfloat162float(v); }

// the group's inputs in the scan's layouts
__global__ void ssd_bwd_gather_kernel(const SsdBwdGlue a) {
  const int64_t HP = a.H * a.P, c0 = a.g * a.hpg * a.P, h0 = a.g * a.hpg;
  const int64_t nrow = a.batch * a.Dc * a.L;      // (b, c, t), t fastest
  const int64_t nbc = a.batch * a.N * a.L;        // (b, n, t)
  const int64_t nst = a.batch * a.Dc * a.N;       // (b, c, n)
  const int64_t ntab = a.Dc * a.N;                // (c, n)
  const int64_t total = nrow + nbc + nst + ntab + a.Dc;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < nrow) {
      const int64_t t = i % a.L, bc = i / a.L, c = bc % a.Dc, b = bc / a.Dc;
      const int64_t src = (b * a.L + t) * HP + c0 + c;
      a.u[i] = bf(a.x[src]);
      a.dyy[i] = bf(a.dy[src]);
      if (a.z) a.zz[i] = bf(a.z[src]);
      a.dl[i] = bf(a.dt[(b * a.L + t) * a.H + h0 + c / a.P]);
    } else if (i < nrow + nbc) {
      const int64_t e = i - nrow;
      const int64_t t = e % a.L, bn = e / a.L, n = bn % a.N, b = bn / a.N;
      const int64_t src = ((b * a.L + t) * a.G + a.g) * a.N + n;
      a.Bg[e] = bf(a.B[src]);
      a.Cg[e] = bf(a.C[src]);
    } else if (i < nrow + nbc + nst) {
      const int64_t e = i - nrow - nbc;
      const int64_t n = e % a.N, bc = e / a.N, c = bc % a.Dc, b = bc / a.Dc;
      const int64_t src = (b * HP + c0 + c) * a.N + n;
      if (a.init) a.initg[e] = a.init[src];
      if (a.dfin) a.dfing[e] = a.dfin[src];
    } else if (i < nrow + nbc + nst + ntab) {
      const int64_t e = i - nrow - nbc - nst;
      a.Ag[e] = a.A[h0 + (e / a.N) / a.P];
    } else {
      const int64_t c = i - nrow - nbc - nst - ntab;
      if (a.D) a.Dg[c] = a.D[h0 + c / a.P];
      if (a.dt_bias) a.biasg[c] = a.dt_bias[h0 + c / a.P];
    }
  }
}

// the group's derivatives back in SSD's layouts; the per-head sums over the
// head's P channels (and, for dA, its N states) in a fixed order
__global__ void ssd_bwd_scatter_kernel(const SsdBwdGlue a) {
  const int64_t HP = a.H * a.P, c0 = a.g * a.hpg * a.P, h0 = a.g * a.hpg;
  const int64_t nrow = a.batch * a.Dc * a.L;      // (b, c, t)
  const int64_t nbc = a.batch * a.N * a.L;        // (b, n, t)
  const int64_t nst = a.batch * a.Dc * a.N;       // (b, c, n)
  const int64_t ndt = a.batch * a.L * a.hpg;      // (b, t, head of the group)
  const int64_t total = nrow + nbc + nst + ndt + a.hpg;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < nrow) {
      const int64_t t = i % a.L, bc = i / a.L, c = bc % a.Dc, b = bc / a.Dc;
      const int64_t dst = (b * a.L + t) * HP + c0 + c;
      a.dx[dst] = __float2bfloat16_rn(a.du[i]);
      if (a.dz) a.dz[dst] = __float2bfloat16_rn(a.dzz[i]);
    } else if (i < nrow + nbc) {
      const int64_t e = i - nrow;
      const int64_t t = e % a.L, bn = e / a.L, n = bn % a.N, b = bn / a.N;
      const int64_t dst = ((b * a.L + t) * a.G + a.g) * a.N + n;
      a.dB[dst] = a.dBg[e];
      a.dC[dst] = a.dCg[e];
    } else if (i < nrow + nbc + nst) {
      const int64_t e = i - nrow - nbc;
      const int64_t n = e % a.N, bc = e / a.N, c = bc % a.Dc, b = bc / a.Dc;
      if (a.dinit) a.dinit[(b * HP + c0 + c) * a.N + n] = a.dinitg[e];
    } else if (i < nrow + nbc + nst + ndt) {
      const int64_t e = i - nrow - nbc - nst;
      const int64_t hl = e % a.hpg, bt = e / a.hpg, t = bt % a.L, b = bt / a.L;
      float s = 0.f;
      for (int64_t p = 0; p < a.P; ++p) s += a.ddl[(b * a.Dc + hl * a.P + p) * a.L + t];
      a.ddt[(b * a.L + t) * a.H + h0 + hl] = __float2bfloat16_rn(s);
    } else {
      const int64_t hl = i - nrow - nbc - nst - ndt;
      float sa = 0.f, sd = 0.f, sb = 0.f;
      for (int64_t p = 0; p < a.P; ++p) {
        const int64_t c = hl * a.P + p;
        for (int64_t n = 0; n < a.N; ++n) sa += a.dAg[c * a.N + n];
        sd += a.dDg[c];
        sb += a.dbiasg[c];
      }
      a.dA[h0 + hl] = sa;
      if (a.dD) a.dD[h0 + hl] = sd;
      if (a.ddt_bias) a.ddt_bias[h0 + hl] = sb;
    }
  }
}

}  // namespace ssm

namespace {

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

struct SsdBwdLayout {
  size_t o[20];  // the group buffers, in SsdBwdGlue's scan-side order
  size_t o_scan, scan_bytes, bytes;
};

SsdBwdLayout ssd_bwd_layout(int64_t batch, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N) {
  SsdBwdLayout w{};
  const size_t Dc = (size_t)(H / G) * (size_t)P;
  const size_t row = up256((size_t)batch * Dc * (size_t)L * 4);
  const size_t bc = up256((size_t)batch * (size_t)N * (size_t)L * 4);
  const size_t tab = up256(Dc * (size_t)N * 4), vec = up256(Dc * 4);
  const size_t st = up256((size_t)batch * Dc * (size_t)N * 4);
  // u dl zz dyy du ddl dzz | Bg Cg dBg dCg | Ag dAg | Dg biasg dDg dbiasg | initg dfing dinitg
  const size_t sizes[20] = {row, row, row, row, row, row, row, bc, bc, bc, bc,
                            tab, tab, vec, vec, vec, vec, st, st, st};
  size_t off = 0;
  for (int k = 0; k < 20; ++k) {
    w.o[k] = off;
    off += sizes[k];
  }
  w.o_scan = off;
  w.scan_bytes = up256(ssm_scan_bwd_workspace_bytes(batch, (int64_t)Dc, L, N));
  w.bytes = off + w.scan_bytes;
  return w;
}

bool ssd_shape_ok(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                  int64_t dstate) {
  if (batch <= 0 || seqlen <= 0 || nheads <= 0 || ngroups <= 0 || nheads % ngroups != 0) return false;
  if (headdim != 64 || (dstate != 64 && dstate != 128) || batch > 65535) return false;
  return (double)batch * (double)nheads * (double)headdim * (double)seqlen < 9.0e18;
}

}  // namespace

extern "C" {

size_t ssm_ssd_bwd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                                   int64_t ngroups, int64_t dstate) {
  if (!ssd_shape_ok(batch, seqlen, nheads, headdim, ngroups, dstate)) return 0;
  return ssd_bwd_layout(batch, seqlen, nheads, headdim, ngroups, dstate).bytes;
}

int ssm_ssd_bwd(const void* x, const void* dt, const float* dt_bias, const float* A, const void* B,
                const void* C, const float* D, const void* z, int flags, const float* init_state,
                const void* dy, const float* d_final_state, void* dx, void* ddt, float* dA,
                float* dB, float* dC, float* dD, void* dz, float* d_dt_bias, float* d_init_state,
                int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                int64_t dstate, void* workspace, size_t workspace_bytes, void* stream) {
  if ((flags & ~(SSM_SOFTPLUS | SSM_EULER_B)) != 0) return SSM_ERR_ARG;
  if (batch < 0 || seqlen < 0 || nheads < 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0)
    return SSM_ERR_ARG;
  if (headdim != 64 || (dstate != 64 && dstate != 128) || (nheads > 0 && nheads % ngroups != 0))
    return SSM_ERR_UNSUPPORTED;
  if (dz && !z) return SSM_ERR_ARG;
  if (batch > 65535) return SSM_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (batch == 0 || nheads == 0 || seqlen == 0) {
    // no step: the head parameters' derivatives are zero and the final state is
    // the initial one, so d init_state = d final_state (zeros without it)
    if (nheads > 0) {
      if (!dA) return SSM_ERR_ARG;
      const size_t nh = (size_t)nheads * 4;
      if (cudaMemsetAsync(dA, 0, nh, st) != cudaSuccess ||
          (dD && cudaMemsetAsync(dD, 0, nh, st) != cudaSuccess) ||
          (d_dt_bias && cudaMemsetAsync(d_dt_bias, 0, nh, st) != cudaSuccess))
        return SSM_ERR_CUDA;
    }
    const size_t nst = (size_t)batch * (size_t)nheads * (size_t)headdim * (size_t)dstate * 4;
    if (d_init_state && nst) {
      const cudaError_t e = d_final_state ? cudaMemcpyAsync(d_init_state, d_final_state, nst,
                                                            cudaMemcpyDeviceToDevice, st)
                                          : cudaMemsetAsync(d_init_state, 0, nst, st);
      if (e != cudaSuccess) return SSM_ERR_CUDA;
    }
    return SSM_OK;
  }
  if (!ssd_shape_ok(batch, seqlen, nheads, headdim, ngroups, dstate)) return SSM_ERR_ARG;
  if (!x || !dt || !A || !B || !C || !dy || !dx || !ddt || !dA || !dB || !dC || (z && !dz))
    return SSM_ERR_ARG;
  const void* ptrs[] = {x, dt, dt_bias, A, B, C, D, z, init_state, dy, d_final_state, dx, ddt, dA,
                        dB, dC, dD, dz, d_dt_bias, d_init_state, workspace};
  for (const void* q : ptrs)
    if (reinterpret_cast<uintptr_t>(q) & 15u) return SSM_ERR_ALIGN;
  const SsdBwdLayout lay = ssd_bwd_layout(batch, seqlen, nheads, headdim, ngroups, dstate);
  if (!workspace || workspace_bytes < lay.bytes) return SSM_ERR_WORKSPACE;

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  auto f = [&](int k) { return reinterpret_cast<float*>(ws + lay.o[k]); };
  ssm::SsdBwdGlue a{};
  a.x = static_cast<const __nv_bfloat16*>(x); a.dt = static_cast<const __nv_bfloat16*>(dt);
  a.z = static_cast<const __nv_bfloat16*>(z); a.dy = static_cast<const __nv_bfloat16*>(dy);
  a.B = static_cast<const __nv_bfloat16*>(B); a.C = static_cast<const __nv_bfloat16*>(C);
  a.A = A; a.D = D; a.dt_bias = dt_bias; a.init = init_state; a.dfin = d_final_state;
  a.dx = static_cast<__nv_bfloat16*>(dx); a.ddt = static_cast<__nv_bfloat16*>(ddt);
  a.dz = static_cast<__nv_bfloat16*>(dz);
  a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD; a.ddt_bias = d_dt_bias; a.dinit = d_init_state;
  a.u = f(0); a.dl = f(1); a.zz = f(2); a.dyy = f(3); a.du = f(4); a.ddl = f(5); a.dzz = f(6);
  a.Bg = f(7); a.Cg = f(8); a.dBg = f(9); a.dCg = f(10); a.Ag = f(11); a.dAg = f(12);
  a.Dg = f(13); a.biasg = f(14); a.dDg = f(15); a.dbiasg = f(16);
  a.initg = f(17); a.dfing = f(18); a.dinitg = f(19);
  a.batch = batch; a.L = seqlen; a.H = nheads; a.P = headdim; a.G = ngroups; a.N = dstate;
  a.hpg = nheads / ngroups; a.Dc = a.hpg * headdim;
  void* scan_ws = ws + lay.o_scan;
  for (int64_t g = 0; g < ngroups; ++g) {
    a.g = g;
    ssm::ssd_bwd_gather_kernel<<<148 * 8, 256, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
    const int rc = ssm_scan_bwd(a.u, a.dl, dt_bias ? a.biasg : nullptr, a.Ag, a.Bg, a.Cg,
                                D ? a.Dg : nullptr, z ? a.zz : nullptr, flags,
                                init_state ? a.initg : nullptr, a.dyy,
                                d_final_state ? a.dfing : nullptr, a.du, a.ddl, a.dAg, a.dBg, a.dCg,
                                a.dDg, z ? a.dzz : nullptr, a.dbiasg, d_init_state ? a.dinitg : nullptr,
                                batch, a.Dc, seqlen, dstate, SSM_F32, scan_ws, lay.scan_bytes, st);
    if (rc != SSM_OK) return rc;
    ssm::ssd_bwd_scatter_kernel<<<148 * 8, 256, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
  }
  return SSM_OK;
}

}  // extern "C"
