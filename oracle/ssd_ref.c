/*
 * Float64 CPU oracle for the Mamba-2 SSD forward scan.  TEST INFRASTRUCTURE ONLY:
 * nothing on the product path may link, load or call this file; only the tests,
 * the smoke check and the CPU-baseline leg of the bench use it.
 *
 * What it computes is the plain token-by-token definition of the layer, per
 * (batch, head) pair, with no chunking, blocking or reordering:
 *
 *     h_0  = init_state[b,h]            (zeros when absent)
 *     h_t  = exp(dt_t * A_h) * h_{t-1} + dt_t * outer(x_t, B_t)        (P x N)
 *     y_t  = h_t @ C_t + D_h * x_t                                     (length P)
 *
 * "Mamba-2 cuda-tile forward pass kernels" (devotd.net), section 1: Mamba-2
 * keeps a fixed-size hidden state that each token updates, and section 2 names
 * the state entering every chunk and the state after the last chunk as the
 * second kernel's outputs; the update and the read-out above are the Mamba-2
 * recurrence those sections describe (Mamba-2 discretises B by dt, not by the
 * Mamba-1 zero-order hold that "3.3 Hardware-aware algorithm and GPU memory
 * hierarchy" section 2.1 prints).  y_t reads the state after token t's update
 * (inclusive).  Head h reads B/C group g = h / (H / G).
 *
 * Inputs x, B, C arrive either as IEEE float32 or as bfloat16 bit patterns
 * (uint16, the top half of a float32); both widen to double exactly.  dt, A,
 * D and the init state are float32.  All arithmetic is double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int64_t batch, seqlen, nheads, headdim, dstate, ngroups, chunk;
} ssd_ref_dims;

static double widen(const void* base, int64_t i, int is_bf16) {
  if (is_bf16) {
    uint32_t bits = ((uint32_t)((const uint16_t*)base)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return (double)((const float*)base)[i];
}

static int dims_ok(const ssd_ref_dims* d) {
  if (!d) return 0;
  if (d->batch <= 0 || d->seqlen < 0 || d->nheads <= 0 || d->headdim <= 0 || d->dstate <= 0 ||
      d->ngroups <= 0 || d->chunk <= 0)
    return 0;
  if (d->nheads % d->ngroups) return 0;
  return 1;
}

/*
 * Runs the recurrence for the selected (batch, head) pairs.
 *   pairs      : nsel x 2 int64 (b, h)
 *   y          : nsel x L x P        (may be NULL)
 *   hfinal     : nsel x P x N        (may be NULL)   state after the last token
 *   hchunk_in  : nsel x nc x P x N   (may be NULL)   state entering chunk c,
 *                                                    i.e. h after token c*Q-1
 * Returns 0 on success, -1 on bad arguments.
 */
int ssd_ref_recurrence(const ssd_ref_dims* d, int io_bf16, const void* x, const float* dt,
                       const float* A, const void* Bm, const void* Cm, const float* D,
                       const float* init, const int64_t* pairs, int64_t nsel, double* y,
                       double* hfinal, double* hchunk_in) {
  if (!dims_ok(d) || !x || !dt || !A || !Bm || !Cm || !pairs || nsel < 0) return -1;
  const int64_t L = d->seqlen, H = d->nheads, P = d->headdim, N = d->dstate, G = d->ngroups;
  const int64_t Q = d->chunk, nc = (L + Q - 1) / Q, heads_per_group = H / G;
  for (int64_t s = 0; s < nsel; ++s)
    if (pairs[2 * s] < 0 || pairs[2 * s] >= d->batch || pairs[2 * s + 1] < 0 || pairs[2 * s + 1] >= H)
      return -1;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t s = 0; s < nsel; ++s) {
    const int64_t b = pairs[2 * s], h = pairs[2 * s + 1], g = h / heads_per_group;
    double* st = (double*)malloc(sizeof(double) * (size_t)(P * N));
    double* bt = (double*)malloc(sizeof(double) * (size_t)N);
    double* ct = (double*)malloc(sizeof(double) * (size_t)N);
    for (int64_t i = 0; i < P * N; ++i)
      st[i] = init ? (double)init[((b * H + h) * P) * N + i] : 0.0;
    const double a_h = (double)A[h];
    const double d_h = D ? (double)D[h] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
      if (hchunk_in && t % Q == 0)
        memcpy(hchunk_in + ((s * nc + t / Q) * P) * N, st, sizeof(double) * (size_t)(P * N));
      const double dtv = (double)dt[(b * L + t) * H + h];
      const double decay = exp(dtv * a_h);
      const int64_t bc = ((b * L + t) * G + g) * N;
      for (int64_t n = 0; n < N; ++n) {
        bt[n] = widen(Bm, bc + n, io_bf16);
        ct[n] = widen(Cm, bc + n, io_bf16);
      }
      for (int64_t p = 0; p < P; ++p) {
        const double xv = widen(x, ((b * L + t) * H + h) * P + p, io_bf16);
        const double u = dtv * xv;
        double* row = st + p * N;
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
          row[n] = decay * row[n] + u * bt[n];
          acc += row[n] * ct[n];
        }
        if (y) y[(s * L + t) * P + p] = acc + d_h * xv;
      }
    }
    if (hfinal) memcpy(hfinal + s * P * N, st, sizeof(double) * (size_t)(P * N));
    free(st);
    free(bt);
    free(ct);
  }
  return 0;
}

/*
 * Per-chunk end state started from zero ("chunk state"): for every selected
 * (b, h) and chunk c, runs the same recurrence over tokens [cQ, min(L,(c+1)Q))
 * from h = 0 and stores the state after the chunk's last token.
 *   S : nsel x nc x P x N
 */
int ssd_ref_chunk_states(const ssd_ref_dims* d, int io_bf16, const void* x, const float* dt,
                         const float* A, const void* Bm, const int64_t* pairs, int64_t nsel,
                         double* S) {
  if (!dims_ok(d) || !x || !dt || !A || !Bm || !pairs || !S || nsel < 0) return -1;
  const int64_t L = d->seqlen, H = d->nheads, P = d->headdim, N = d->dstate, G = d->ngroups;
  const int64_t Q = d->chunk, nc = (L + Q - 1) / Q, heads_per_group = H / G;
  for (int64_t s = 0; s < nsel; ++s)
    if (pairs[2 * s] < 0 || pairs[2 * s] >= d->batch || pairs[2 * s + 1] < 0 || pairs[2 * s + 1] >= H)
      return -1;

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int64_t s = 0; s < nsel; ++s) {
    for (int64_t c = 0; c < nc; ++c) {
      const int64_t b = pairs[2 * s], h = pairs[2 * s + 1], g = h / heads_per_group;
      double* st = S + ((s * nc + c) * P) * N;
      for (int64_t i = 0; i < P * N; ++i) st[i] = 0.0;
      const double a_h = (double)A[h];
      const int64_t t1 = (c + 1) * Q < L ? (c + 1) * Q : L;
      for (int64_t t = c * Q; t < t1; ++t) {
        const double dtv = (double)dt[(b * L + t) * H + h];
        const double decay = exp(dtv * a_h);
        const int64_t bc = ((b * L + t) * G + g) * N;
        for (int64_t p = 0; p < P; ++p) {
          const double u = dtv * widen(x, ((b * L + t) * H + h) * P + p, io_bf16);
          double* row = st + p * N;
          for (int64_t n = 0; n < N; ++n) row[n] = decay * row[n] + u * widen(Bm, bc + n, io_bf16);
        }
      }
    }
  }
  return 0;
}

/* Number of OpenMP threads the oracle will use (for the CPU-baseline report). */
int ssd_ref_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
