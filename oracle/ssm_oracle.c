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
 * Readings where the pages leave a step open: h_{-1} = 0 unless an initial
 * state is given; y_t reads the state after the update at t; D sits inside
 * the gate; Δ_raw + bias with softplus off is used as Δ directly.
 *
 * bfloat16 inputs are decoded exactly (bits << 16) to float and then double.
 */
#include <math.h>
#include <stdint.h>
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
                      int64_t bc_ld, double Dd, int softplus_on,
                      const double* h0, int64_t y_stride, double* y_row, double* h_out) {
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
      double bbar = (An != 0.0) ? expm1(dA) / An : dt;   /* times B below */
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

/* Threads OpenMP will use (the CPU baseline reports it). */
int ssm_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
