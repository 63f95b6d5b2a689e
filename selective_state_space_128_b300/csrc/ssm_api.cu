// C ABI of libssm: argument checks, planning and dispatch.  See include/ssm.h.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/ssm.h"
#include "ssm_internal.h"

namespace {

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_n(int64_t n) {
  return n == 1 || n == 2 || n == 4 || n == 8 || n == 16 || n == 32 || n == 64 || n == 128;
}

// the backward keeps up to 16 states per lane and its recomputed chunk in
// shared memory; it is built for every dstate the forward supports
bool supported_bwd_n(int64_t n) { return supported_n(n); }

// [p, p + bytes) and [q, q + qbytes) intersect (null never does)
bool overlaps(const void* p, size_t bytes, const void* q, size_t qbytes) {
  if (!p || !q || bytes == 0 || qbytes == 0) return false;
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
  return a < b + qbytes && b < a + bytes;
}

int sm_count_current() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

// bytes from the first to one past the last element of a (batch, dim, seqlen)
// tensor with element strides t (0 when empty)
size_t span_bytes(const int64_t* t, int64_t batch, int64_t dim, int64_t seqlen, size_t esz) {
  if (batch <= 0 || dim <= 0 || seqlen <= 0) return 0;
  return (size_t)(1 + (batch - 1) * t[0] + (dim - 1) * t[1] + (seqlen - 1) * t[2]) * esz;
}

// distinct (b, d, t) map to distinct elements: sorted by stride, each stride is at
// least the span of the dimensions with smaller strides
bool strides_injective(const int64_t* t, const int64_t* ext) {
  int idx[3] = {0, 1, 2};
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (t[idx[j]] < t[idx[i]]) { const int q = idx[i]; idx[i] = idx[j]; idx[j] = q; }
  int64_t span = 1;
  for (int i = 0; i < 3; ++i) {
    const int k = idx[i];
    if (ext[k] <= 1) continue;
    if (t[k] < span) return false;
    span = t[k] * (ext[k] - 1) + span;
  }
  return true;
}

// the delta_softplus flag word: SSM_SOFTPLUS | SSM_EULER_B, nothing else
bool flags_ok(int f) { return (f & ~(SSM_SOFTPLUS | SSM_EULER_B)) == 0; }

// failure-path test mode (ssm_set_test_mode): SSM_TEST_STALL is refused unless on
std::atomic<int> g_test_mode{0};
std::atomic<int64_t> g_test_limit_ns{1000000};
std::atomic<int64_t> g_test_noalloc_limit{0};
std::atomic<int> g_test_scan_kernel{0};  // 0: by size, 1: the block kernel, 2: the two-warp-block kernel

bool sizes_ok(int64_t batch, int64_t dim, int64_t seqlen) {
  // every flat index must fit in int64 with room to spare
  if (batch < 0 || dim < 0 || seqlen < 0) return false;
  if (batch > 65535) return false;  // grid.y
  const double total = (double)batch * (double)dim * (double)(seqlen > 0 ? seqlen : 1);
  return total < 9.0e18;
}

}  // namespace

extern "C" {

const char* ssm_strerror(int status) {
  switch (status) {
    case SSM_OK: return "SSM_OK";
    case SSM_ERR_ARG: return "SSM_ERR_ARG: invalid argument";
    case SSM_ERR_ALIGN: return "SSM_ERR_ALIGN: pointer not 16-byte aligned";
    case SSM_ERR_UNSUPPORTED:
      return "SSM_ERR_UNSUPPORTED: dstate not in {1,2,4,8,16,32,64,128}, "
             "or conv width not in 1..4";
    case SSM_ERR_CUDA: return "SSM_ERR_CUDA: CUDA launch failed";
    case SSM_ERR_WORKSPACE: return "SSM_ERR_WORKSPACE: workspace too small";
    case SSM_ERR_TIMEOUT: return "SSM_ERR_TIMEOUT: a kernel gave up waiting for its data";
    default: return "unknown ssm status";
  }
}

const char* ssm_version(void) { return "0.1.0"; }

size_t ssm_scan_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                int io_dtype) {
  if (!supported_n(dstate) || !sizes_ok(batch, dim, seqlen)) return 0;
  return ssm::kScanStatusBytes + ssm::scan_carry_bytes(batch, dim, seqlen, dstate, io_dtype);
}

int ssm_set_test_mode(int enable, int64_t wait_limit_ns, int64_t noalloc_limit_bytes,
                      int scan_kernel) {
  if (enable && (wait_limit_ns < 1000 || wait_limit_ns > 2000000000 || noalloc_limit_bytes < 0 ||
                 scan_kernel < 0 || scan_kernel > 2))
    return SSM_ERR_ARG;
  g_test_limit_ns.store(enable ? wait_limit_ns : 1000000);
  g_test_noalloc_limit.store(enable ? noalloc_limit_bytes : 0);
  g_test_scan_kernel.store(enable ? scan_kernel : 0);
  g_test_mode.store(enable ? 1 : 0);
  return SSM_OK;
}

size_t ssm_ssd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                               int64_t ngroups, int64_t dstate) {
  if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim != 64 || (dstate != 64 && dstate != 128))
    return 0;
  if (ngroups <= 0 || nheads % ngroups != 0) return 0;
  if (!sizes_ok(batch, nheads * headdim, seqlen)) return 0;
  return ssm::ssd_layout(batch, seqlen, nheads, ngroups, dstate).bytes;
}

int ssm_ssd_fwd(const void* x, const void* dt, const float* dt_bias, const float* A,
                const void* B, const void* C, const float* D, const void* z, int flags, void* y,
                float* final_state, const float* init_state, int64_t batch, int64_t seqlen,
                int64_t nheads, int64_t headdim, int64_t ngroups, int64_t dstate,
                void* workspace, size_t workspace_bytes, void* stream) {
  if (!flags_ok(flags)) return SSM_ERR_ARG;
  if (batch < 0 || seqlen < 0 || nheads < 0 || ngroups <= 0 || headdim <= 0 || dstate <= 0)
    return SSM_ERR_ARG;
  if (batch > 65535 || nheads > 65535) return SSM_ERR_ARG;
  if (!sizes_ok(batch, nheads * headdim, seqlen)) return SSM_ERR_ARG;
  if (headdim != 64 || (dstate != 64 && dstate != 128) || nheads % ngroups != 0)
    return SSM_ERR_UNSUPPORTED;
  const bool work = batch > 0 && nheads > 0 && seqlen > 0;
  if (work && (!x || !dt || !A || !B || !C || !y)) return SSM_ERR_ARG;
  const void* ptrs[] = {x, dt, dt_bias, A, B, C, D, z, y, final_state, init_state, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SSM_ERR_ALIGN;
  const size_t nx = (size_t)batch * (size_t)seqlen * (size_t)nheads * (size_t)headdim * 2;
  const size_t ndt = (size_t)batch * (size_t)seqlen * (size_t)nheads * 2;
  const size_t nbc = (size_t)batch * (size_t)seqlen * (size_t)ngroups * (size_t)dstate * 2;
  const size_t nst = (size_t)batch * (size_t)nheads * (size_t)headdim * (size_t)dstate * 4;
  const size_t nh = (size_t)nheads * 4;
  struct Span { const void* p; size_t n; };
  const Span ins[] = {{x, nx}, {dt, ndt}, {dt_bias, nh}, {A, nh}, {B, nbc}, {C, nbc}, {D, nh},
                      {z, nx}, {init_state, nst}};
  for (const Span& in : ins)
    if (overlaps(y, nx, in.p, in.n) || overlaps(final_state, nst, in.p, in.n)) return SSM_ERR_ARG;
  if (overlaps(y, nx, final_state, nst)) return SSM_ERR_ARG;
  const ssm::SsdLayout lay = ssm::ssd_layout(batch, seqlen, nheads, ngroups, dstate);
  if (work) {
    if (!workspace || workspace_bytes < lay.bytes) return SSM_ERR_WORKSPACE;
    for (const Span& in : ins)
      if (overlaps(workspace, lay.bytes, in.p, in.n)) return SSM_ERR_ARG;
    if (overlaps(workspace, lay.bytes, y, nx) || overlaps(workspace, lay.bytes, final_state, nst))
      return SSM_ERR_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!work) {
    // no steps: the final state is the initial one (or zeros)
    if (final_state && nst) {
      const cudaError_t e = init_state ? cudaMemcpyAsync(final_state, init_state, nst,
                                                         cudaMemcpyDeviceToDevice, st)
                                       : cudaMemsetAsync(final_state, 0, nst, st);
      if (e != cudaSuccess) return SSM_ERR_CUDA;
    }
    return SSM_OK;
  }
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  ssm::SsdArgs a{};
  a.x = x; a.dt = dt; a.dt_bias = dt_bias; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.y = y;
  a.final_state = final_state; a.init_state = init_state;
  a.ws_hin = reinterpret_cast<__nv_bfloat16*>(ws + lay.o_hin);
  a.ws_terms = reinterpret_cast<float*>(ws + lay.o_terms);
  a.ws_cb = reinterpret_cast<float*>(ws + lay.o_cb);
  a.batch = batch; a.L = seqlen; a.H = nheads; a.G = ngroups; a.nch = lay.nch;
  a.softplus = (flags & SSM_SOFTPLUS) != 0;
  a.euler = (flags & SSM_EULER_B) != 0;
  a.status = ssm::library_status_word();
  if (!a.status) return SSM_ERR_CUDA;
  const cudaError_t e = ssm::ssd_launch(a, dstate, st);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // extern "C"

namespace ssm {

size_t noalloc_test_limit() { return (size_t)g_test_noalloc_limit.load(); }
int scan_kernel_choice() { return g_test_scan_kernel.load(); }

size_t scan_carry_bytes(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype) {
  return scan_plan(batch, dim, seqlen, dstate, io_dtype, sm_count_current(), true).workspace_bytes;
}

// the scan after the workspace has been resolved into a status word and carry scratch
int scan_fwd_internal(const void* u, const void* delta, const float* delta_bias, const float* A,
                      const float* B, const float* C, const float* D, const void* z,
                      int delta_softplus, void* y, float* final_state, int64_t batch, int64_t dim,
                      int64_t seqlen, int64_t dstate, int io_dtype, const float* init_state,
                      int* status, bool zero_status, void* carry, size_t carry_bytes,
                      void* bwd_workspace, size_t bwd_workspace_bytes, bool train,
                      cudaStream_t stream, const int64_t* strides) {
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_ARG;
  const bool stall = (delta_softplus & SSM_TEST_STALL) != 0;
  if (stall && (!g_test_mode.load() || train)) return SSM_ERR_ARG;
  if (!flags_ok(delta_softplus & ~(SSM_LAYOUT_BLD | SSM_TEST_STALL))) return SSM_ERR_ARG;
  bool bld = (delta_softplus & SSM_LAYOUT_BLD) != 0;
  if (strides && bld) return SSM_ERR_ARG;  // the strides say the layout
  if (!sizes_ok(batch, dim, seqlen) || dstate <= 0) return SSM_ERR_ARG;
  if (!supported_n(dstate)) return SSM_ERR_UNSUPPORTED;
  const bool work = batch > 0 && dim > 0;
  if (work && seqlen > 0 && (!u || !delta || !A || !B || !C || !y)) return SSM_ERR_ARG;
  const void* ptrs[] = {u, delta, delta_bias, A, B, C, D, z, y, final_state, init_state, carry,
                        bwd_workspace, status};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SSM_ERR_ALIGN;
  const size_t esz = io_dtype == SSM_F32 ? 4 : 2;
  // element strides (batch, channel, time) of u, delta, z, y
  int64_t st[4][3];
  for (int k = 0; k < 4; ++k) {
    if (strides) {
      for (int e = 0; e < 3; ++e) st[k][e] = strides[3 * k + e];
    } else {
      st[k][0] = dim * seqlen;
      st[k][1] = bld ? 1 : seqlen;
      st[k][2] = bld ? dim : 1;
    }
  }
  if (strides) {
    const int64_t ext[3] = {batch, dim, seqlen};
    for (int k = 0; k < 4; ++k)
      for (int e = 0; e < 3; ++e)
        if (st[k][e] < 0 || (ext[e] > 1 && st[k][e] == 0)) return SSM_ERR_ARG;
    if (!strides_injective(st[3], ext)) return SSM_ERR_ARG;  // y would write an element twice
    // u, delta (and z) share one orientation: unit time stride, or unit channel stride
    const bool tmaj = st[0][2] == 1 && st[1][2] == 1 && (!z || st[2][2] == 1);
    const bool cmaj = st[0][1] == 1 && st[1][1] == 1 && (!z || st[2][1] == 1);
    if (seqlen > 1 && dim > 1 && !tmaj && !cmaj) return SSM_ERR_UNSUPPORTED;
    bld = !tmaj && cmaj;
  }
  const size_t nio_u = span_bytes(st[0], batch, dim, seqlen, esz);
  const size_t nio_d = span_bytes(st[1], batch, dim, seqlen, esz);
  const size_t nio_z = z ? span_bytes(st[2], batch, dim, seqlen, esz) : 0;
  const size_t nio = span_bytes(st[3], batch, dim, seqlen, esz);  // y
  const size_t nst = (size_t)batch * (size_t)dim * (size_t)dstate * 4;
  const size_t nbc = (size_t)batch * (size_t)dstate * (size_t)seqlen * 4;
  // outputs must not overlap inputs (final_state may equal init_state exactly)
  if (overlaps(y, nio, u, nio_u) || overlaps(y, nio, delta, nio_d) || overlaps(y, nio, z, nio_z))
    return SSM_ERR_ARG;
  if (overlaps(y, nio, B, nbc) || overlaps(y, nio, C, nbc) || overlaps(y, nio, final_state, nst))
    return SSM_ERR_ARG;
  if (final_state && init_state && final_state != init_state &&
      overlaps(final_state, nst, init_state, nst))
    return SSM_ERR_ARG;
  if (overlaps(final_state, nst, u, nio_u) || overlaps(final_state, nst, delta, nio_d) ||
      overlaps(final_state, nst, z, nio_z))
    return SSM_ERR_ARG;
  if (!work) return SSM_OK;

  // A split plan reads init_state in every segment while the last segment
  // writes final_state, so an in-place carry (final_state == init_state)
  // always runs unsplit.
  const bool in_place = final_state != nullptr && final_state == init_state;
  const ssm::ScanPlan plan = ssm::scan_plan(batch, dim, seqlen, dstate, io_dtype,
                                            sm_count_current(), carry != nullptr && !in_place);
  if (carry && carry_bytes < plan.workspace_bytes) return SSM_ERR_WORKSPACE;
  // the training save: the backward's checkpoint part of its workspace
  float* ckpt = nullptr;
  int64_t ckpt_nch = 0;
  if (train && seqlen > 0) {
    const ssm::BwdLayout lay = ssm::bwd_layout(batch, dim, seqlen, dstate, sm_count_current());
    if (!bwd_workspace || bwd_workspace_bytes < lay.bytes) return SSM_ERR_WORKSPACE;
    const void* others[] = {u, delta, z, y, carry, status};
    const size_t sizes[] = {nio_u, nio_d, nio_z, nio, plan.workspace_bytes, sizeof(int)};
    for (int k = 0; k < 6; ++k)
      if (overlaps(bwd_workspace, lay.bytes, others[k], sizes[k])) return SSM_ERR_ARG;
    if (overlaps(bwd_workspace, lay.bytes, final_state, nst) ||
        overlaps(bwd_workspace, lay.bytes, init_state, nst) ||
        overlaps(bwd_workspace, lay.bytes, B, nbc) || overlaps(bwd_workspace, lay.bytes, C, nbc))
      return SSM_ERR_ARG;
    if (ssm::bwd_chunk(dstate) == plan.chunk) {
      ckpt = reinterpret_cast<float*>(static_cast<unsigned char*>(bwd_workspace) + lay.o_ckpt);
      ckpt_nch = lay.nch;
    }
  }
  if (zero_status && status && cudaMemsetAsync(status, 0, sizeof(int), stream) != cudaSuccess)
    return SSM_ERR_CUDA;

  ssm::ScanArgs a{};
  a.ckpt = ckpt;
  a.ckpt_nch = ckpt_nch;
  a.u = u; a.delta = delta; a.z = z; a.bias = delta_bias; a.A = A; a.B = B; a.C = C; a.D = D;
  a.y = y; a.final_state = final_state; a.init_state = init_state;
  a.batch = batch; a.dim = dim; a.L = seqlen;
  a.nseg = plan.nseg; a.seg_len = plan.seg_len;
  a.softplus = (delta_softplus & SSM_SOFTPLUS) != 0;
  a.euler = (delta_softplus & SSM_EULER_B) != 0;
  a.bld = bld;
  a.status = status;
  a.test_stall = stall ? 1 : 0;
  a.test_limit_ns = g_test_limit_ns.load();
  for (int e = 0; e < 3; ++e) {
    a.st_u[e] = st[0][e];
    a.st_d[e] = st[1][e];
    a.st_z[e] = st[2][e];
    a.st_y[e] = st[3][e];
  }
  // staging by TMA: the strides other than the unit one are multiples of 16 bytes
  {
    const int o = bld ? 2 : 1;
    auto m16 = [&](const int64_t* t) { return (t[o] * (int64_t)esz) % 16 == 0 && (t[0] * (int64_t)esz) % 16 == 0; };
    a.vec_io = m16(st[0]) && m16(st[1]) && (!z || m16(st[2]));
    if (bld ? st[0][1] != 1 : st[0][2] != 1) a.vec_io = 0;
  }
  // vector stores of y: unit time stride and 16-byte aligned rows
  a.vec_y = st[3][2] == 1 && (st[3][1] * (int64_t)esz) % 16 == 0 &&
            (st[3][0] * (int64_t)esz) % 16 == 0;
  a.vec_bc = (seqlen * 4) % 16 == 0;
  a.force_precise = io_dtype == SSM_F32;
  if (plan.nseg > 1) {
    const size_t rows = (size_t)batch * (size_t)dim;
    const size_t hbytes = ((size_t)(plan.nseg - 1) * rows * (size_t)dstate * 4 + 255) / 256 * 256;
    a.carry_h = static_cast<float*>(carry);
    a.carry_s = reinterpret_cast<float*>(static_cast<unsigned char*>(carry) + hbytes);
  }
  const cudaError_t e = ssm::scan_launch(a, dstate, io_dtype, plan, stream);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // namespace ssm

namespace {

// A caller's scan workspace: the status word in its first kScanStatusBytes, the
// split plan's carry records after them.
int scan_with_workspace(const void* u, const void* delta, const float* delta_bias, const float* A,
                        const float* B, const float* C, const float* D, const void* z,
                        int delta_softplus, void* y, float* final_state, int64_t batch,
                        int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype,
                        const float* init_state, void* workspace, size_t workspace_bytes,
                        void* bwd_workspace, size_t bwd_workspace_bytes, bool train,
                        void* stream, const int64_t* strides = nullptr) {
  int* status = nullptr;
  void* carry = nullptr;
  size_t carry_bytes = 0;
  if (workspace) {
    if (workspace_bytes < ssm::kScanStatusBytes) return SSM_ERR_WORKSPACE;
    if (!aligned16(workspace)) return SSM_ERR_ALIGN;
    status = static_cast<int*>(workspace);
    carry_bytes = workspace_bytes - ssm::kScanStatusBytes;
    carry = carry_bytes ? static_cast<unsigned char*>(workspace) + ssm::kScanStatusBytes : nullptr;
    // the workspace overlaps no input or output
    const size_t esz = io_dtype == SSM_F32 ? 4 : 2;
    const size_t nst = (size_t)(batch > 0 ? batch : 0) * (size_t)(dim > 0 ? dim : 0) *
                       (size_t)(dstate > 0 ? dstate : 0) * 4;
    const void* io[] = {u, delta, z, y};
    for (int k = 0; k < 4; ++k) {
      int64_t t[3] = {dim * seqlen, seqlen, 1};
      if (strides) {
        for (int e = 0; e < 3; ++e) t[e] = strides[3 * k + e] < 0 ? 0 : strides[3 * k + e];
      } else if (delta_softplus & SSM_LAYOUT_BLD) {
        t[1] = 1;
        t[2] = dim;
      }
      if (overlaps(workspace, workspace_bytes, io[k], span_bytes(t, batch, dim, seqlen, esz)))
        return SSM_ERR_ARG;
    }
    if (overlaps(workspace, workspace_bytes, final_state, nst) ||
        overlaps(workspace, workspace_bytes, init_state, nst))
      return SSM_ERR_ARG;
  }
  return ssm::scan_fwd_internal(u, delta, delta_bias, A, B, C, D, z, delta_softplus, y,
                                final_state, batch, dim, seqlen, dstate, io_dtype, init_state,
                                status, true, carry, carry_bytes, bwd_workspace,
                                bwd_workspace_bytes, train, static_cast<cudaStream_t>(stream),
                                strides);
}

}  // namespace

extern "C" {

int ssm_scan_fwd_ex(const void* u, const void* delta, const float* delta_bias, const float* A,
                    const float* B, const float* C, const float* D, const void* z,
                    int delta_softplus, void* y, float* final_state, int64_t batch, int64_t dim,
                    int64_t seqlen, int64_t dstate, int io_dtype, const float* init_state,
                    void* workspace, size_t workspace_bytes, void* stream) {
  return scan_with_workspace(u, delta, delta_bias, A, B, C, D, z, delta_softplus, y, final_state,
                             batch, dim, seqlen, dstate, io_dtype, init_state, workspace,
                             workspace_bytes, nullptr, 0, false, stream);
}

int ssm_scan_fwd_train(const void* u, const void* delta, const float* delta_bias, const float* A,
                       const float* B, const float* C, const float* D, const void* z,
                       int delta_softplus, void* y, float* final_state, int64_t batch,
                       int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype,
                       const float* init_state, void* workspace, size_t workspace_bytes,
                       void* bwd_workspace, size_t bwd_workspace_bytes, void* stream) {
  return scan_with_workspace(u, delta, delta_bias, A, B, C, D, z, delta_softplus, y, final_state,
                             batch, dim, seqlen, dstate, io_dtype, init_state, workspace,
                             workspace_bytes, bwd_workspace, bwd_workspace_bytes, true, stream);
}

int ssm_scan_fwd_strided(const void* u, const void* delta, const float* delta_bias,
                         const float* A, const float* B, const float* C, const float* D,
                         const void* z, int delta_softplus, void* y, float* final_state,
                         int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                         int io_dtype, const int64_t* strides, const float* init_state,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return scan_with_workspace(u, delta, delta_bias, A, B, C, D, z, delta_softplus, y, final_state,
                             batch, dim, seqlen, dstate, io_dtype, init_state, workspace,
                             workspace_bytes, nullptr, 0, false, stream, strides);
}

int ssm_scan_fwd_complex(const void* u, const void* delta, const float* delta_bias,
                         const float* A, const float* B, const float* C, const float* D,
                         const void* z, int delta_softplus, void* y, float* final_state,
                         const float* init_state, int64_t batch, int64_t dim, int64_t seqlen,
                         int64_t dstate, int io_dtype, void* stream) {
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_ARG;
  if (!flags_ok(delta_softplus)) return SSM_ERR_ARG;
  if (!sizes_ok(batch, dim, seqlen) || dstate <= 0) return SSM_ERR_ARG;
  if (dstate > 64 || (dstate & (dstate - 1)) != 0) return SSM_ERR_UNSUPPORTED;
  const bool work = batch > 0 && dim > 0 && seqlen > 0;
  if (work && (!u || !delta || !A || !B || !C || !y)) return SSM_ERR_ARG;
  const void* ptrs[] = {u, delta, delta_bias, A, B, C, D, z, y, final_state, init_state};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SSM_ERR_ALIGN;
  const size_t esz = io_dtype == SSM_F32 ? 4 : 2;
  const size_t nio = (size_t)batch * (size_t)dim * (size_t)seqlen * esz;
  const size_t nst = (size_t)batch * (size_t)dim * (size_t)dstate * 8;
  const size_t nbc = (size_t)batch * (size_t)dstate * (size_t)seqlen * 8;
  const size_t nA = (size_t)dim * (size_t)dstate * 8, nd = (size_t)dim * 4;
  const void* ins[] = {u, delta, z, B, C, A, delta_bias, D, init_state};
  const size_t in_bytes[] = {nio, nio, nio, nbc, nbc, nA, nd, nd, nst};
  for (int k = 0; k < 9; ++k) {
    if (overlaps(y, nio, ins[k], in_bytes[k])) return SSM_ERR_ARG;
    if (k < 8 && overlaps(final_state, nst, ins[k], in_bytes[k])) return SSM_ERR_ARG;
  }
  if (overlaps(y, nio, final_state, nst)) return SSM_ERR_ARG;
  if (final_state && init_state && final_state != init_state &&
      overlaps(final_state, nst, init_state, nst))
    return SSM_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (batch > 0 && dim > 0 && seqlen == 0) {
    // no step: the final state is the initial one (zeros without it)
    if (!final_state || final_state == init_state) return SSM_OK;
    const cudaError_t e = init_state ? cudaMemcpyAsync(final_state, init_state, nst,
                                                       cudaMemcpyDeviceToDevice, st)
                                     : cudaMemsetAsync(final_state, 0, nst, st);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
  }
  if (!work) return SSM_OK;
  ssm::ComplexScanArgs a{};
  a.u = u; a.delta = delta; a.z = z; a.bias = delta_bias;
  a.A = reinterpret_cast<const float2*>(A);
  a.B = reinterpret_cast<const float2*>(B);
  a.C = reinterpret_cast<const float2*>(C);
  a.D = D; a.y = y;
  a.final_state = reinterpret_cast<float2*>(final_state);
  a.init_state = reinterpret_cast<const float2*>(init_state);
  a.batch = batch; a.dim = dim; a.L = seqlen;
  a.softplus = (delta_softplus & SSM_SOFTPLUS) != 0;
  a.euler = (delta_softplus & SSM_EULER_B) != 0;
  const cudaError_t e = ssm::scan_complex_launch(a, dstate, io_dtype, st);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

int ssm_status(const void* workspace, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int code = 0;
  if (workspace) {
    if (!aligned16(workspace)) return SSM_ERR_ALIGN;
    if (cudaMemcpyAsync(&code, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return SSM_ERR_CUDA;
  } else if (ssm::scan_library_status(&code, st) != cudaSuccess) {
    return SSM_ERR_CUDA;
  }
  return code == 0 ? SSM_OK : SSM_ERR_TIMEOUT;
}

int ssm_scan_fwd(const void* u, const void* delta, const float* delta_bias, const float* A,
                 const float* B, const float* C, const float* D, const void* z,
                 int delta_softplus, void* y, float* final_state, int64_t batch, int64_t dim,
                 int64_t seqlen, int64_t dstate, int io_dtype) {
  return ssm_scan_fwd_ex(u, delta, delta_bias, A, B, C, D, z, delta_softplus, y, final_state,
                         batch, dim, seqlen, dstate, io_dtype, nullptr, nullptr, 0, nullptr);
}

int ssm_state_update_ex(float* state, const void* u, const void* delta, const float* delta_bias,
                        int delta_softplus, const float* A, const float* B, const float* C,
                        const float* D, const void* z, void* y, int64_t batch, int64_t dim,
                        int64_t dstate, int io_dtype, void* stream) {
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_ARG;
  if (!flags_ok(delta_softplus)) return SSM_ERR_ARG;
  if (!sizes_ok(batch, dim, 1) || dstate <= 0) return SSM_ERR_ARG;
  if (!supported_n(dstate)) return SSM_ERR_UNSUPPORTED;
  if (batch > 0 && dim > 0 && (!state || !u || !delta || !A || !B || !C || !y)) return SSM_ERR_ARG;
  const void* ptrs[] = {state, u, delta, delta_bias, A, B, C, D, z, y};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SSM_ERR_ALIGN;
  const size_t esz = io_dtype == SSM_F32 ? 4 : 2;
  const size_t nio = (size_t)batch * (size_t)dim * esz;
  const size_t nst = (size_t)batch * (size_t)dim * (size_t)dstate * 4;
  const size_t nbc = (size_t)batch * (size_t)dstate * 4, nA = (size_t)dim * (size_t)dstate * 4;
  const void* ins[] = {u, delta, z, B, C, A};
  const size_t in_bytes[] = {nio, nio, nio, nbc, nbc, nA};
  for (int k = 0; k < 6; ++k)
    if (overlaps(state, nst, ins[k], in_bytes[k])) return SSM_ERR_ARG;
  if (overlaps(y, nio, state, nst) || overlaps(y, nio, u, nio) || overlaps(y, nio, delta, nio) ||
      overlaps(y, nio, z, nio))
    return SSM_ERR_ARG;
  if (batch == 0 || dim == 0) return SSM_OK;
  ssm::UpdateArgs a{};
  a.state = state; a.u = u; a.delta = delta; a.z = z; a.bias = delta_bias; a.A = A; a.B = B;
  a.C = C; a.D = D; a.y = y; a.batch = batch; a.dim = dim;
  a.softplus = (delta_softplus & SSM_SOFTPLUS) != 0;
  a.euler = (delta_softplus & SSM_EULER_B) != 0;
  a.force_precise = io_dtype == SSM_F32;
  const cudaError_t e = ssm::update_launch(a, dstate, io_dtype, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

int ssm_state_update(float* state, const void* u, const void* delta, const float* A,
                     const float* B, const float* C, const float* D, const void* z, void* y,
                     int64_t batch, int64_t dim, int64_t dstate, int io_dtype) {
  return ssm_state_update_ex(state, u, delta, nullptr, 0, A, B, C, D, z, y, batch, dim, dstate,
                             io_dtype, nullptr);
}

size_t ssm_scan_bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate) {
  if (!supported_bwd_n(dstate) || !sizes_ok(batch, dim, seqlen)) return 0;
  if (batch == 0 || dim == 0 || seqlen == 0) return 0;
  return ssm::bwd_layout(batch, dim, seqlen, dstate, sm_count_current()).bytes;
}

int ssm_scan_bwd(const void* u, const void* delta, const float* delta_bias, const float* A,
                 const float* B, const float* C, const float* D, const void* z,
                 int delta_softplus, const float* init_state, const void* dy,
                 const float* d_final_state, void* du, void* ddelta, float* dA, float* dB,
                 float* dC, float* dD, void* dz, float* d_delta_bias, float* d_init_state,
                 int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype,
                 void* workspace, size_t workspace_bytes, void* stream) {
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_ARG;
  if (!flags_ok(delta_softplus & ~(SSM_SAVED_STATES | SSM_LAYOUT_BLD))) return SSM_ERR_ARG;
  if (!sizes_ok(batch, dim, seqlen) || dstate <= 0) return SSM_ERR_ARG;
  if (!supported_bwd_n(dstate)) return SSM_ERR_UNSUPPORTED;
  if (dz && !z) return SSM_ERR_ARG;
  const bool rows = batch > 0 && dim > 0;
  const bool steps = rows && seqlen > 0;
  if (steps && (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dB || !dC ||
                (z && !dz)))
    return SSM_ERR_ARG;
  if (dim > 0 && !dA) return SSM_ERR_ARG;
  if (batch > 0 && seqlen > 0 && (!dB || !dC)) return SSM_ERR_ARG;
  const void* ptrs[] = {u, delta, delta_bias, A, B, C, D, z, init_state, dy, d_final_state,
                        du, ddelta, dA, dB, dC, dD, dz, d_delta_bias, d_init_state, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SSM_ERR_ALIGN;
  const size_t esz = io_dtype == SSM_F32 ? 4 : 2;
  const size_t nio = (size_t)batch * (size_t)dim * (size_t)seqlen * esz;
  const size_t nst = (size_t)batch * (size_t)dim * (size_t)dstate * 4;
  const size_t nbc = (size_t)batch * (size_t)dstate * (size_t)seqlen * 4;
  const size_t nA = (size_t)dim * (size_t)dstate * 4, nd = (size_t)dim * 4;
  struct Span { const void* p; size_t n; };
  const Span ins[] = {{u, nio}, {delta, nio}, {z, nio}, {dy, nio}, {delta_bias, nd}, {A, nA},
                      {B, nbc}, {C, nbc}, {D, nd}, {init_state, nst}, {d_final_state, nst}};
  const Span outs[] = {{du, nio}, {ddelta, nio}, {dz, nio}, {dA, nA}, {dB, nbc}, {dC, nbc},
                       {dD, nd}, {d_delta_bias, nd}, {d_init_state, nst}};
  for (size_t i = 0; i < sizeof outs / sizeof outs[0]; ++i) {
    for (const Span& in : ins)
      if (overlaps(outs[i].p, outs[i].n, in.p, in.n)) return SSM_ERR_ARG;
    for (size_t j = i + 1; j < sizeof outs / sizeof outs[0]; ++j)
      if (overlaps(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return SSM_ERR_ARG;
  }
  const ssm::BwdLayout lay = ssm::bwd_layout(batch, dim, seqlen, dstate, sm_count_current());
  if (steps) {
    if (!workspace || workspace_bytes < lay.bytes) return SSM_ERR_WORKSPACE;
    for (const Span& q : outs)
      if (overlaps(workspace, lay.bytes, q.p, q.n)) return SSM_ERR_ARG;
    for (const Span& q : ins)
      if (overlaps(workspace, lay.bytes, q.p, q.n)) return SSM_ERR_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!steps) {
    // empty sums are zero; with no steps the initial state passes its
    // derivative through unchanged
    cudaError_t e = cudaSuccess;
    if (dA && nA) e = cudaMemsetAsync(dA, 0, nA, st);
    if (e == cudaSuccess && dD && nd) e = cudaMemsetAsync(dD, 0, nd, st);
    if (e == cudaSuccess && d_delta_bias && nd) e = cudaMemsetAsync(d_delta_bias, 0, nd, st);
    if (e == cudaSuccess && nbc) e = cudaMemsetAsync(dB, 0, nbc, st);
    if (e == cudaSuccess && nbc) e = cudaMemsetAsync(dC, 0, nbc, st);
    if (e == cudaSuccess && d_init_state && nst)
      e = d_final_state ? cudaMemcpyAsync(d_init_state, d_final_state, nst,
                                          cudaMemcpyDeviceToDevice, st)
                        : cudaMemsetAsync(d_init_state, 0, nst, st);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
  }
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  ssm::BwdArgs a{};
  a.u = u; a.delta = delta; a.z = z; a.bias = delta_bias; a.A = A; a.B = B; a.C = C; a.D = D;
  a.init_state = init_state; a.dy = dy; a.d_final_state = d_final_state;
  a.du = du; a.ddelta = ddelta; a.dz = dz; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD;
  a.d_bias = d_delta_bias; a.d_init_state = d_init_state;
  a.ckpt = reinterpret_cast<float*>(ws + lay.o_ckpt);
  a.ws_B = reinterpret_cast<float*>(ws + lay.o_B);
  a.ws_C = reinterpret_cast<float*>(ws + lay.o_C);
  a.ws_A = reinterpret_cast<float*>(ws + lay.o_A);
  a.ws_D = reinterpret_cast<float*>(ws + lay.o_D);
  a.ws_bias = reinterpret_cast<float*>(ws + lay.o_bias);
  a.batch = batch; a.dim = dim; a.L = seqlen; a.nblk = lay.nblk;
  a.bld = (delta_softplus & SSM_LAYOUT_BLD) != 0;
  // saved states are used where the training forward saves them (same chunk length)
  a.saved = (delta_softplus & SSM_SAVED_STATES) != 0 &&
            ssm::bwd_chunk(dstate) ==
                ssm::scan_plan(batch, dim, seqlen, dstate, io_dtype, sm_count_current(), false).chunk;
  a.softplus = (delta_softplus & SSM_SOFTPLUS) != 0;
  a.euler = (delta_softplus & SSM_EULER_B) != 0;
  a.force_precise = io_dtype == SSM_F32;
  a.nseg = lay.nseg;
  a.seg_len = lay.seg_len;
  if (lay.nseg > 1) {
    a.fcarry_h = reinterpret_cast<float*>(ws + lay.o_fh);
    a.fcarry_s = reinterpret_cast<float*>(ws + lay.o_fs);
    a.acarry_l = reinterpret_cast<float*>(ws + lay.o_al);
    a.acarry_s = reinterpret_cast<float*>(ws + lay.o_as);
    if (!a.saved) {
      // the forward's segment carries: the scan's first pass over the same
      // segments (its bounded waits report to the library-wide status word)
      ssm::ScanArgs f{};
      f.u = u; f.delta = delta; f.z = nullptr; f.bias = delta_bias; f.A = A; f.B = B; f.C = C;
      f.batch = batch; f.dim = dim; f.L = seqlen;
      f.nseg = lay.nseg; f.seg_len = lay.seg_len;
      f.carry_h = a.fcarry_h; f.carry_s = a.fcarry_s;
      f.softplus = a.softplus; f.euler = a.euler; f.force_precise = a.force_precise;
      f.bld = a.bld;
      for (int k = 0; k < 4; ++k) {
        int64_t* t = k == 0 ? f.st_u : k == 1 ? f.st_d : k == 2 ? f.st_z : f.st_y;
        t[0] = dim * seqlen;
        t[1] = a.bld ? 1 : seqlen;
        t[2] = a.bld ? dim : 1;
      }
      const int64_t o = a.bld ? dim : seqlen;  // the stride other than the unit one
      f.vec_io = (o * (int64_t)esz) % 16 == 0 && (dim * seqlen * (int64_t)esz) % 16 == 0;
      f.vec_bc = (seqlen * 4) % 16 == 0;
      f.test_limit_ns = 0;
      const cudaError_t ef = ssm::scan_carries_launch(f, dstate, io_dtype, st);
      if (ef != cudaSuccess) return SSM_ERR_CUDA;
    }
  }
  const cudaError_t e = ssm::bwd_launch(a, dstate, io_dtype, st);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

int ssm_conv1d_fwd(const void* x, const float* weight, const float* bias,
                   const void* conv_state_in, int silu, void* out, void* conv_state_out,
                   int64_t batch, int64_t dim, int64_t seqlen, int64_t width, int io_dtype,
                   void* stream) {
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_ARG;
  if ((silu & ~(1 | SSM_LAYOUT_BLD)) != 0) return SSM_ERR_ARG;
  if (!sizes_ok(batch, dim, seqlen) || width <= 0) return SSM_ERR_ARG;
  if (width > 4) return SSM_ERR_UNSUPPORTED;
  const bool rows = batch > 0 && dim > 0;
  if (rows && seqlen > 0 && (!x || !weight || !out)) return SSM_ERR_ARG;
  if (rows && conv_state_out && !weight) return SSM_ERR_ARG;
  const void* ptrs[] = {x, weight, bias, conv_state_in, out, conv_state_out};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SSM_ERR_ALIGN;
  const size_t esz = io_dtype == SSM_F32 ? 4 : 2;
  const size_t nio = (size_t)batch * (size_t)dim * (size_t)seqlen * esz;
  const size_t nst = (size_t)batch * (size_t)dim * (size_t)(width - 1) * esz;
  const size_t nw = (size_t)dim * (size_t)width * 4, nb = (size_t)dim * 4;
  if (overlaps(out, nio, x, nio) || overlaps(out, nio, weight, nw) || overlaps(out, nio, bias, nb) ||
      overlaps(out, nio, conv_state_in, nst) || overlaps(out, nio, conv_state_out, nst))
    return SSM_ERR_ARG;
  if (conv_state_out && (overlaps(conv_state_out, nst, x, nio) ||
                         overlaps(conv_state_out, nst, weight, nw) ||
                         overlaps(conv_state_out, nst, bias, nb) ||
                         (conv_state_out != conv_state_in &&
                          overlaps(conv_state_out, nst, conv_state_in, nst))))
    return SSM_ERR_ARG;
  if (!rows) return SSM_OK;
  ssm::ConvArgs a{};
  a.x = x; a.w = weight; a.bias = bias; a.state_in = conv_state_in; a.out = out;
  a.state_out = width > 1 ? conv_state_out : nullptr;
  a.batch = batch; a.dim = dim; a.L = seqlen;
  a.silu = (silu & 1) != 0;
  a.bld = (silu & SSM_LAYOUT_BLD) != 0;
  a.precise = io_dtype == SSM_F32;
  const cudaError_t e = ssm::conv_launch(a, width, io_dtype, false, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

int ssm_conv1d_bwd(const void* x, const float* weight, const float* bias,
                   const void* conv_state_in, int silu, const void* dout, void* dx,
                   float* dweight, float* dbias, float* d_conv_state_in, int64_t batch,
                   int64_t dim, int64_t seqlen, int64_t width, int io_dtype, void* stream) {
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_ARG;
  if ((silu & ~(1 | SSM_LAYOUT_BLD)) != 0) return SSM_ERR_ARG;
  if (!sizes_ok(batch, dim, seqlen) || width <= 0) return SSM_ERR_ARG;
  if (width > 4) return SSM_ERR_UNSUPPORTED;
  if (dim > 0 && !dweight) return SSM_ERR_ARG;
  const bool rows = batch > 0 && dim > 0;
  if (rows && seqlen > 0 && (!x || !weight || !dout || !dx)) return SSM_ERR_ARG;
  const void* ptrs[] = {x, weight, bias, conv_state_in, dout, dx, dweight, dbias, d_conv_state_in};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SSM_ERR_ALIGN;
  const size_t esz = io_dtype == SSM_F32 ? 4 : 2;
  const size_t nio = (size_t)batch * (size_t)dim * (size_t)seqlen * esz;
  const size_t nst = (size_t)batch * (size_t)dim * (size_t)(width - 1);
  const size_t nw = (size_t)dim * (size_t)width * 4, nb = (size_t)dim * 4;
  // outputs overlap no input and no other output
  const void* ins[] = {x, weight, bias, conv_state_in, dout};
  const size_t insz[] = {nio, nw, nb, nst * esz, nio};
  const void* outs[] = {dx, dweight, dbias, d_conv_state_in};
  const size_t outsz[] = {nio, nw, nb, nst * 4};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 5; ++j)
      if (overlaps(outs[i], outsz[i], ins[j], insz[j])) return SSM_ERR_ARG;
    for (int j = i + 1; j < 4; ++j)
      if (overlaps(outs[i], outsz[i], outs[j], outsz[j])) return SSM_ERR_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!rows || seqlen == 0) {
    // no step: every derivative is zero
    if (dim > 0 && cudaMemsetAsync(dweight, 0, nw, st) != cudaSuccess) return SSM_ERR_CUDA;
    if (dim > 0 && dbias && cudaMemsetAsync(dbias, 0, nb, st) != cudaSuccess) return SSM_ERR_CUDA;
    if (d_conv_state_in && nst && cudaMemsetAsync(d_conv_state_in, 0, nst * 4, st) != cudaSuccess)
      return SSM_ERR_CUDA;
    return SSM_OK;
  }
  ssm::ConvBwdArgs a{};
  a.x = x; a.w = weight; a.bias = bias; a.state_in = conv_state_in; a.dout = dout; a.dx = dx;
  a.dw = dweight; a.dbias = dbias; a.dstate = width > 1 ? d_conv_state_in : nullptr;
  a.batch = batch; a.dim = dim; a.L = seqlen;
  a.silu = (silu & 1) != 0;
  a.precise = io_dtype == SSM_F32;
  a.bld = (silu & SSM_LAYOUT_BLD) != 0;
  const cudaError_t e = ssm::conv_bwd_launch(a, width, io_dtype, st);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

int ssm_conv1d_update(void* conv_state, const void* x, const float* weight, const float* bias,
                      int silu, void* out, int64_t batch, int64_t dim, int64_t width,
                      int io_dtype, void* stream) {
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_ARG;
  if (!sizes_ok(batch, dim, 1) || width <= 0) return SSM_ERR_ARG;
  if (width > 4) return SSM_ERR_UNSUPPORTED;
  const bool rows = batch > 0 && dim > 0;
  if (rows && (!x || !weight || !out || (width > 1 && !conv_state))) return SSM_ERR_ARG;
  const void* ptrs[] = {conv_state, x, weight, bias, out};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SSM_ERR_ALIGN;
  const size_t esz = io_dtype == SSM_F32 ? 4 : 2;
  const size_t nio = (size_t)batch * (size_t)dim * esz;
  const size_t nst = (size_t)batch * (size_t)dim * (size_t)(width - 1) * esz;
  const size_t nw = (size_t)dim * (size_t)width * 4, nb = (size_t)dim * 4;
  if (overlaps(out, nio, x, nio) || overlaps(out, nio, conv_state, nst) ||
      overlaps(out, nio, weight, nw) || overlaps(out, nio, bias, nb) ||
      overlaps(conv_state, nst, x, nio) || overlaps(conv_state, nst, weight, nw) ||
      overlaps(conv_state, nst, bias, nb))
    return SSM_ERR_ARG;
  if (!rows) return SSM_OK;
  ssm::ConvArgs a{};
  a.x = x; a.w = weight; a.bias = bias; a.out = out; a.state_out = conv_state;
  a.batch = batch; a.dim = dim; a.L = 1;
  a.silu = silu != 0;
  a.precise = io_dtype == SSM_F32;
  const cudaError_t e = ssm::conv_launch(a, width, io_dtype, true, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // extern "C"
