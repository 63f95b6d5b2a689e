/*
 * fp64 CPU oracle for the selective state-space (S6) scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the bench's CPU
 * baseline do.  It shares no code with the CUDA library.
 *
 * What it computes is the plain definition, evaluated sequentially in double
 * precision, one (batch, channel) unit at a time:
 *
 *   Selection (Mamba summary page, section 4b, Algorithm 2 "SSM + Selection
 *   (S6)" and the parameterisation under it; the SSM/Mamba chapter, 4.1):
 *       Δ_t = softplus(Δraw_t + bias_d)      (bias absent = 0; softplus optional)
 *   Zero-order-hold discretisation (summary page, section 4b, equation (4);
 *   chapter section 3.2), per state n of the diagonal A:
 *       Ā = exp(Δ A_n),   B̄ = (ΔA_n)^-1 (exp(ΔA_n) - 1) Δ B_{n,t}
 *         = expm1(Δ A_n) / A_n * B_{n,t}      (A_n = 0: the limit Δ B_{n,t})
 *   Recurrence and readout (summary page, equations (2a), (2b); the chapter's
 *   section 3.1 adds the direct term D):
 *       h_t = Ā h_{t-1} + B̄ u_t,      y_t = C_t · h_t + D u_t
 *   Gate (summary page, section 4a shape table, "SSM output × SiLU(gate)"):
 *       y_t <- y_t * z_t * sigmoid(z_t)       (z absent = no gate)
 *
 * Variant (the `mode` bit 2, "Euler"): B̄ = Δ B_{n,t}, the first-order form the
 * summary page gives beside equation (4) as the small-Δ limit of the ZOH.
 * The `mode` argument of every entry point: bit 1 = softplus on Δ, bit 2 = Euler.
 *
 * Readings where the pages leave a step open: h_{-1} = 0 unless an initial
 * state is given; y_t reads the state after the update at t; D sits inside
 * the gate; Δ_raw + bias with softplus off is used as Δ directly.
 *
 * bfloat16 inputs are decoded exactly (bits << 16) to float and then double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double in_val(const void* p, int bf16, int64_t i) {
  if (bf16) {
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return (double)((const float*)p)[i];
}

static double softplus(double x) {
  /* log(1 + e^x), written so that neither branch overflows or cancels */
  return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));
}

/* One unit (one batch index b, one channel d) over L steps. */
static void scan_unit(int64_t L, int64_t N, int bf16,
                      const void* u, const void* delta, const void* z, int64_t row,
                      double bias, const float* A_row, const float* B_b, const float* C_b,
                      int64_t bc_ld, double Dd, int mode,
                      const double* h0, int64_t y_stride, double* y_row, double* h_out) {
  const int softplus_on = mode & 1, euler = (mode & 2) != 0;
  double h[512];
  for (int64_t n = 0; n < N; ++n) h[n] = h0 ? h0[n] : 0.0;
  for (int64_t t = 0; t < L; ++t) {
    double ut = in_val(u, bf16, row * L + t);
    double x = in_val(delta, bf16, row * L + t) + bias;
    double dt = softplus_on ? softplus(x) : x;
    double acc = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      double An = (double)A_row[n];
      double dA = dt * An;
      double abar = exp(dA);
      double bbar = euler ? dt : ((An != 0.0) ? expm1(dA) / An : dt);   /* times B below */
      h[n] = abar * h[n] + bbar * (double)B_b[n * bc_ld + t] * ut;
      acc += (double)C_b[n * bc_ld + t] * h[n];
    }
    double yv = acc + Dd * ut;
    if (z) {
      double zt = in_val(z, bf16, row * L + t);
      yv *= zt / (1.0 + exp(-zt));
    }
    if (y_row && (t % y_stride) == 0) y_row[t / y_stride] = yv;
  }
  if (h_out)
    for (int64_t n = 0; n < N; ++n) h_out[n] = h[n];
}

/*
 * Scan U independent units.  Unit i reads row i of u / delta / z (each row L
 * contiguous elements; float32, or bfloat16 bits when io_bf16), batch
 * unit_b[i] of B and C (element (b, n, t) at B[(b*N + n)*bc_ld + t]) and
 * channel unit_d[i] of A (dim x N), D (dim) and delta_bias (dim).
 * y (optional) receives y_t for t = 0, y_stride, 2*y_stride, ... as rows of
 * ceil(L / y_stride) doubles; final_state (optional) receives h_{L-1} as U x N
 * doubles; init_state (optional) is U x N doubles.  Returns 0, or -1 when N
 * exceeds the fixed state buffer (512).
 */
int ssm_oracle_scan(int64_t U, int64_t L, int64_t N, int io_bf16,
                    const void* u, const void* delta, const void* z,
                    const int64_t* unit_b, const int64_t* unit_d,
                    const float* delta_bias, const float* A, const float* B, const float* C,
                    int64_t bc_ld, const float* D, int delta_softplus,
                    const double* init_state, int64_t y_stride, double* y,
                    double* final_state, int nthreads) {
  if (N > 512 || N < 1 || L < 0 || U < 0 || y_stride < 1) return -1;
  int64_t ny = (L + y_stride - 1) / y_stride;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < U; ++i) {
    int64_t b = unit_b[i], d = unit_d[i];
    scan_unit(L, N, io_bf16, u, delta, z, i, delta_bias ? (double)delta_bias[d] : 0.0,
              A + d * N, B + b * N * bc_ld, C + b * N * bc_ld, bc_ld, D ? (double)D[d] : 0.0,
              delta_softplus, init_state ? init_state + i * N : 0, y_stride,
              y ? y + i * ny : 0, final_state ? final_state + i * N : 0);
  }
  return 0;
}

/*
 * One recurrent (decode) step, the summary page's "recurrent mode" of
 * equation (2): state[i] <- Ā state[i] + B̄ u, y = C·state + D u, gated.
 * Unit i reads element i of u / delta / z, row unit_b[i] of B and C
 * (batch x N), channel unit_d[i] of A / D / delta_bias.  state is U x N
 * doubles, updated in place; y is U doubles.
 */
int ssm_oracle_step(int64_t U, int64_t N, int io_bf16, const void* u, const void* delta,
                    const void* z, const int64_t* unit_b, const int64_t* unit_d,
                    const float* delta_bias, const float* A, const float* B, const float* C,
                    const float* D, int delta_softplus, double* state, double* y, int nthreads) {
  if (N > 512 || N < 1 || U < 0) return -1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < U; ++i) {
    int64_t b = unit_b[i], d = unit_d[i];
    /* a single step is the scan over one time step (bc_ld = 1, L = 1) */
    scan_unit(1, N, io_bf16, u, delta, z, i, delta_bias ? (double)delta_bias[d] : 0.0,
              A + d * N, B + b * N, C + b * N, 1, D ? (double)D[d] : 0.0, delta_softplus,
              state + i * N, 1, y + i, state + i * N);
  }
  return 0;
}

/*
 * Backward pass (reverse-mode derivative) of the scan above.
 *
 * The summary page ("Mamba: Linear-Time Sequence Modeling", section 4c,
 * "hardware-aware algorithm") trains the layer by recomputing the states in
 * the backward pass instead of storing the expanded (B, L, D, N) tensor; it
 * gives no formula for the gradients.  This oracle takes them from the chain
 * rule applied to the forward definition, one unit at a time, in double
 * precision.  For a loss with upstream derivatives dy_t = dLoss/dy_t and
 * dfinal = dLoss/dh_{L-1}:
 *
 *   g_t  = silu(z_t) (1 without a gate),   s_t = C_t·h_t + D u_t,  y_t = s_t g_t
 *   ds_t = dy_t g_t,   dz_t = dy_t s_t silu'(z_t),  silu'(z) = σ(z)(1 + z(1 - σ(z)))
 *   λ_t  = dLoss/dh_t = ds_t C_t + Ā_{t+1} λ_{t+1},  λ_{L-1} = ds_{L-1} C_{L-1} + dfinal
 *   with h_t = Ā_t h_{t-1} + B̄_t B_t u_t (B̄_t here the scalar factor expm1(ΔA)/A):
 *   du_t    = ds_t D + Σ_n λ_{t,n} B̄_{t,n} B_{t,n}
 *   dB_{t,n} += λ_{t,n} B̄_{t,n} u_t           (summed over the channels of a batch)
 *   dC_{t,n} += ds_t h_{t,n}                  (summed over the channels of a batch)
 *   dΔ_t    = Σ_n λ_{t,n} (h_{t-1,n} A_n Ā_{t,n} + B_{t,n} u_t Ā_{t,n})
 *             [dĀ/dΔ = A Ā, d(expm1(ΔA)/A)/dΔ = Ā; Euler B̄ = Δ: 1 and 0]
 *   dA_n   += λ_{t,n} (h_{t-1,n} Δ_t Ā_{t,n} + B_{t,n} u_t (Δ_t Ā_{t,n} - B̄_{t,n}) / A_n)
 *             [A_n = 0: the limit Δ_t^2 / 2 for the second factor]
 *   dΔraw_t = dΔ_t σ(Δraw_t + bias) with softplus, else dΔ_t;  dbias += dΔraw_t
 *   dD     += ds_t u_t;   dh_{-1} = Ā_0 λ_0
 */
static double sigmoid(double x) {
  return x >= 0.0 ? 1.0 / (1.0 + exp(-x)) : exp(x) / (1.0 + exp(x));
}

/* One unit.  dB_b / dC_b: this unit's batch slice of the accumulators
 * (element (n, t) at [n * L + t]).  Scratch: L*N doubles for the states and L
 * doubles each for Δ, Δraw + bias and s. */
static void scan_bwd_unit(int64_t L, int64_t N, int bf16, const void* u, const void* delta,
                          const void* z, int64_t row, double bias, const float* A_row,
                          const float* B_b, const float* C_b, int64_t bc_ld, double Dd,
                          int mode, const double* h0, const double* dy_row,
                          const double* dfinal, double* du_row, double* ddelta_row,
                          double* dz_row, double* dA_out, double* dD_out, double* dbias_out,
                          double* dinit_out, double* dB_b, double* dC_b, double* hs,
                          double* dts, double* xs, double* ss) {
  const int softplus_on = mode & 1, euler = (mode & 2) != 0;
  /* forward, keeping every state h_t (hs[t*N + n]), Δ_t, Δraw_t + bias and s_t */
  for (int64_t t = 0; t < L; ++t) {
    double ut = in_val(u, bf16, row * L + t);
    double x = in_val(delta, bf16, row * L + t) + bias;
    double dt = softplus_on ? softplus(x) : x;
    double acc = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      double An = (double)A_row[n];
      double prev = t > 0 ? hs[(t - 1) * N + n] : (h0 ? h0[n] : 0.0);
      double abar = exp(dt * An);
      double bbar = euler ? dt : ((An != 0.0) ? expm1(dt * An) / An : dt);
      double h = abar * prev + bbar * (double)B_b[n * bc_ld + t] * ut;
      hs[t * N + n] = h;
      acc += (double)C_b[n * bc_ld + t] * h;
    }
    dts[t] = dt;
    xs[t] = x;
    ss[t] = acc + Dd * ut;
  }
  /* reverse */
  double lam[512];
  for (int64_t n = 0; n < N; ++n) {
    lam[n] = dfinal ? dfinal[n] : 0.0;
    dA_out[n] = 0.0;
  }
  double dD = 0.0, dbias = 0.0;
  for (int64_t t = L - 1; t >= 0; --t) {
    double ut = in_val(u, bf16, row * L + t);
    double dt = dts[t];
    double g = 1.0;
    if (z) {
      double zt = in_val(z, bf16, row * L + t);
      double sg = sigmoid(zt);
      g = zt * sg;
      if (dz_row) dz_row[t] = dy_row[t] * ss[t] * sg * (1.0 + zt * (1.0 - sg));
    }
    double ds = dy_row[t] * g;
    dD += ds * ut;
    double du = ds * Dd;
    double ddt = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      double An = (double)A_row[n];
      double Bn = (double)B_b[n * bc_ld + t];
      double Cn = (double)C_b[n * bc_ld + t];
      double prev = t > 0 ? hs[(t - 1) * N + n] : (h0 ? h0[n] : 0.0);
      double abar = exp(dt * An);
      double bbar = euler ? dt : ((An != 0.0) ? expm1(dt * An) / An : dt);
      /* d B̄/dA and d B̄/dΔ: ZOH (A = 0: the limit), Euler: 0 and 1 */
      double dbbar_dA = euler ? 0.0 : ((An != 0.0) ? (dt * abar - bbar) / An : 0.5 * dt * dt);
      double dbbar_ddt = euler ? 1.0 : abar;
      lam[n] += ds * Cn;
      dC_b[n * L + t] += ds * hs[t * N + n];
      dB_b[n * L + t] += lam[n] * bbar * ut;
      du += lam[n] * bbar * Bn;
      ddt += lam[n] * (prev * An * abar + Bn * ut * dbbar_ddt);
      dA_out[n] += lam[n] * (prev * dt * abar + Bn * ut * dbbar_dA);
      lam[n] *= abar;
    }
    du_row[t] = du;
    double dx = softplus_on ? ddt * sigmoid(xs[t]) : ddt;
    ddelta_row[t] = dx;
    dbias += dx;
  }
  *dD_out = dD;
  *dbias_out = dbias;
  if (dinit_out)
    for (int64_t n = 0; n < N; ++n) dinit_out[n] = lam[n];
}

/*
 * Backward of ssm_oracle_scan over U units (same input conventions).  dy is
 * U x L doubles; dfinal (optional) U x N.  Outputs: du, ddelta (U x L), dz
 * (U x L, optional; only with z), per-unit dA (U x N), dD (U), dbias (U) and
 * dinit (U x N, optional); dB and dC (nbatch x N x L) receive the sums over
 * the units of each batch (they are overwritten, not accumulated into).
 * Returns 0, -1 on bad sizes, -2 when scratch memory runs out.
 */
int ssm_oracle_scan_bwd(int64_t U, int64_t L, int64_t N, int io_bf16, const void* u,
                        const void* delta, const void* z, const int64_t* unit_b,
                        const int64_t* unit_d, const float* delta_bias, const float* A,
                        const float* B, const float* C, int64_t bc_ld, const float* D,
                        int delta_softplus, const double* init_state, const double* dy,
                        const double* dfinal, double* du, double* ddelta, double* dz,
                        double* dA, double* dD, double* dbias, double* dinit, int64_t nbatch,
                        double* dB, double* dC, int nthreads) {
  if (N > 512 || N < 1 || L < 0 || U < 0 || nbatch < 1) return -1;
  for (int64_t i = 0; i < U; ++i)
    if (unit_b[i] < 0 || unit_b[i] >= nbatch) return -1;
  const int64_t nbc = nbatch * N * L;
  memset(dB, 0, sizeof(double) * (size_t)nbc);
  memset(dC, 0, sizeof(double) * (size_t)nbc);
  int failed = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel
  {
    double* acc = (double*)calloc((size_t)(2 * nbc), sizeof(double));
    double* scratch = (double*)malloc(sizeof(double) * (size_t)(L * N + 3 * L + 1));
    const int ok = acc && scratch;
    if (!ok) {
#pragma omp atomic write
      failed = 1;
    }
    /* every thread reaches the loop (a work-sharing construct); one without
       scratch skips its units and the call reports the failure */
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < U; ++i) {
      if (!ok) continue;
      int64_t b = unit_b[i], d = unit_d[i];
      scan_bwd_unit(L, N, io_bf16, u, delta, z, i, delta_bias ? (double)delta_bias[d] : 0.0,
                    A + d * N, B + b * N * bc_ld, C + b * N * bc_ld, bc_ld,
                    D ? (double)D[d] : 0.0, delta_softplus, init_state ? init_state + i * N : 0,
                    dy + i * L, dfinal ? dfinal + i * N : 0, du + i * L, ddelta + i * L,
                    (z && dz) ? dz + i * L : 0, dA + i * N, dD + i, dbias + i,
                    dinit ? dinit + i * N : 0, acc + b * N * L, acc + nbc + b * N * L,
                    scratch, scratch + L * N, scratch + L * N + L, scratch + L * N + 2 * L);
    }
    if (ok) {
#pragma omp critical
      {
        for (int64_t k = 0; k < nbc; ++k) {
          dB[k] += acc[k];
          dC[k] += acc[nbc + k];
        }
      }
    }
    free(acc);
    free(scratch);
  }
  return failed ? -2 : 0;
}

/*
 * Front end of the scan: causal depthwise convolution over time followed by
 * SiLU.  The summary page's shape table (section 4a, "Conv1d -> SiLU" on
 * (B, L, ED): local features and a non-linearity ahead of the SSM) and the
 * configuration-framework page's d_conv = 4 (the kernel width) fix the
 * operation; per channel d, with width K,
 *
 *     v[t]   = bias[d] + Σ_{k=0}^{K-1} w[d, k] · x[t - (K-1) + k]
 *     out[t] = silu(v[t]) = v[t] σ(v[t])          (or v[t] with silu off)
 *
 * where x[t] for t < 0 comes from the carried state (the K-1 inputs before
 * the sequence; zeros when absent).  The new state is the last K-1 inputs of
 * the extended sequence (state, x).
 */
int ssm_oracle_conv1d(int64_t U, int64_t L, int64_t K, int io_bf16, const void* x,
                      const int64_t* unit_d, const float* w, const float* bias,
                      const double* state_in, int silu_on, double* out, double* state_out,
                      int nthreads) {
  if (K < 1 || K > 64 || L < 0 || U < 0) return -1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < U; ++i) {
    const int64_t d = unit_d[i];
    /* xe[j] = x[j - (K-1)] for j >= K-1, the state for j < K-1 */
    for (int64_t t = 0; t < L; ++t) {
      double v = bias ? (double)bias[d] : 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const int64_t s = t - (K - 1) + k;  /* input time */
        double xv;
        if (s >= 0) xv = in_val(x, io_bf16, i * L + s);
        else xv = state_in ? state_in[i * (K - 1) + (K - 1 + s)] : 0.0;
        v += (double)w[d * K + k] * xv;
      }
      out[i * L + t] = silu_on ? v / (1.0 + exp(-v)) : v;
    }
    if (state_out) {
      for (int64_t j = 0; j < K - 1; ++j) {
        const int64_t s = L - (K - 1) + j;  /* input time of state slot j */
        double xv;
        if (s >= 0) xv = in_val(x, io_bf16, i * L + s);
        else xv = state_in ? state_in[i * (K - 1) + (K - 1 + s)] : 0.0;
        state_out[i * (K - 1) + j] = xv;
      }
    }
  }
  return 0;
}

/* Threads OpenMP will use (the CPU baseline reports it). */
int ssm_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
