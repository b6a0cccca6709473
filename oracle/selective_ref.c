/*
 * Float64 CPU oracle for the Mamba-1 selective scan.  TEST INFRASTRUCTURE ONLY:
 * nothing on the product path may link, load or call this file; only the tests,
 * the smoke check and the CPU-baseline leg of the bench use it.
 *
 * "3.3 Hardware-aware algorithm and GPU memory hierarchy" (booiljung.github.io),
 * section 2.1: the parameters (delta, A, B, C) and the input x are read, the
 * continuous parameters are discretised by the zero-order hold
 *     Abar = exp(delta A),      Bbar = (delta A)^-1 (exp(delta A) - I) delta B,
 * the recurrence runs, and only y is written out; section 3 lists the fused
 * steps (load, discretise, scan, multiply the state by C); section 4.1 writes
 * the update as the first-order linear recurrence h_t = Abar_t h_{t-1} +
 * Bbar_t x_t.  A is diagonal per channel, so for channel d and state n
 *     h_t[d,n] = exp(delta_t[d] A[d,n]) h_{t-1}[d,n]
 *                + (exp(delta_t[d] A[d,n]) - 1) / A[d,n] * B_t[n] * x_t[d]
 * (the factor is delta_t[d] B_t[n] x_t[d] where A[d,n] = 0, its limit), and
 *     y_t[d] = sum_n C_t[n] h_t[d,n]  (+ Dskip[d] x_t[d] when Dskip is given).
 * y_t reads the state after token t's update.  Written plainly: one channel at a
 * time, one token at a time, no blocking or reordering.
 *
 * Shapes: x, delta, y (b, L, D); B, C (b, L, N); A (D, N); Dskip (D);
 * init / final state (b, D, N).  x, delta, B, C are float32 or bfloat16 bit
 * patterns (uint16), widened exactly to double; A, Dskip, init are float32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double sel_widen(const void* base, int64_t i, int is_bf16) {
  if (is_bf16) {
    uint32_t bits = ((uint32_t)((const uint16_t*)base)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return (double)((const float*)base)[i];
}

/*
 * Returns 0 on success, -1 on bad arguments.  y: b x L x D (may be NULL);
 * hfinal: b x D x N (may be NULL), the state after the last token.
 */
int ssd_ref_selective_scan(int64_t batch, int64_t L, int64_t D, int64_t N, int io_bf16,
                           const void* x, const void* delta, const float* A, const void* Bm,
                           const void* Cm, const float* Dskip, const float* init, double* y,
                           double* hfinal) {
  if (batch <= 0 || L < 0 || D <= 0 || N <= 0 || !x || !delta || !A || !Bm || !Cm) return -1;
#pragma omp parallel for collapse(2) schedule(dynamic, 16)
  for (int64_t b = 0; b < batch; ++b) {
    for (int64_t d = 0; d < D; ++d) {
      double* h = (double*)malloc(sizeof(double) * (size_t)N);
      for (int64_t n = 0; n < N; ++n) h[n] = init ? (double)init[(b * D + d) * N + n] : 0.0;
      const double skip = Dskip ? (double)Dskip[d] : 0.0;
      for (int64_t t = 0; t < L; ++t) {
        const int64_t row = (b * L + t) * D + d;
        const double dv = sel_widen(delta, row, io_bf16);
        const double xv = sel_widen(x, row, io_bf16);
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
          const double a = (double)A[d * N + n];
          const double w = dv * a;
          const double abar = exp(w);
          const double coef = a == 0.0 ? dv : expm1(w) / a;  /* (exp(delta A) - 1) / A */
          const double bv = sel_widen(Bm, (b * L + t) * N + n, io_bf16);
          const double cv = sel_widen(Cm, (b * L + t) * N + n, io_bf16);
          h[n] = abar * h[n] + coef * bv * xv;
          acc += cv * h[n];
        }
        if (y) y[row] = acc + skip * xv;
      }
      if (hfinal) memcpy(hfinal + (b * D + d) * N, h, sizeof(double) * (size_t)N);
      free(h);
    }
  }
  return 0;
}
