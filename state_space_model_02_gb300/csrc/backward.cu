// backward -- the element-wise and reduction steps of the SSD backward pass.
//
// The forward ("Mamba-2 cuda-tile forward pass kernels", sections 1-2) is the recurrence
//     h_t = a_t h_{t-1} + dt_t x_t (x) B_t,  a_t = exp(dt_t A),  y_t = h_t C_t + D x_t.
// Its adjoint state g_t = dL/dh_t runs backwards in time, g_t = dy_t (x) C_t + a_{t+1} g_{t+1}
// (g_{L-1} starts from dL/dfinal) -- the same kind of scan in reversed time, with the decay of
// the following token and inputs not scaled by dt.  The gradients are then
//     dx_t  = dt_t (g_t B_t) + D dy_t                    (reverse scan read out with B)
//     dB_t  = sum_h dt_t (g_t^T x_t)                      (reverse scan, x and C roles swapped)
//     dC_t  = sum_h h_t^T dy_t                            (forward scan, x and B roles swapped)
//     dD    = sum <dy_t, x_t>,   dinit = a_0 g_0
// and, with cs_t the running sum of A dt (every decay is exp(cs_t - cs_s)),
//     dL/dcs_t = <dy_t, y_t - D x_t> - dt_t <x_t, g_t B_t>  (+ <dfinal, final> at t = L-1)
//     ddt_t    = <x_t, g_t B_t> + A sum_{s >= t} dL/dcs_s,  dA = sum_t dt_t sum_{s >= t} dL/dcs_s.
// The scans run through the forward kernels; this file holds the steps between them: the
// time flips, group expansions and float32 widenings of their inputs, the shifted decays, the
// per-token combinations and the reverse cumulative sum.  The two scans whose outputs meet in
// dL/dcs (the forward again and the adjoint scan) run in float32 whatever the I/O dtype: that
// difference cancels heavily, and bf16-rounded operands would leave dA with bf16-sized
// errors relative to a much smaller result.
#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

__device__ __forceinline__ float ldf(const float* p, int64_t i) { return __ldg(p + i); }
__device__ __forceinline__ float ldf(const uint16_t* p, int64_t i) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(p + i)) << 16);
}
__device__ __forceinline__ void stf(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void stf(uint16_t* p, int64_t i, float v) {
  p[i] = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu);
}

// The layout kernels below run one block per (batch, token) row group: the block index gives
// (b, t) once per thread, and the positions inside the group split with 32-bit arithmetic
// (a shift when the divisor is a power of two) instead of 64-bit division per element.
struct RowSplit {
  uint32_t d;
  int sh;  // log2(d) when d is a power of two, else -1
  __device__ __forceinline__ uint32_t div(uint32_t n) const { return sh >= 0 ? n >> sh : n / d; }
};
inline RowSplit row_split(int64_t d) {
  RowSplit r{static_cast<uint32_t>(d), -1};
  if (d > 0 && (d & (d - 1)) == 0) {
    r.sh = 0;
    while ((int64_t(1) << r.sh) < d) ++r.sh;
  }
  return r;
}
constexpr int kRowThreads = 128;

// dst[b, t, h, :] = src[b, flip ? L-1-t : t, h / rep, v0 : v0 + vec_dst], in 16-byte vectors
// (source rows of vec_src vectors, destination rows of vec_dst)
__global__ void __launch_bounds__(kRowThreads) flip_expand_kernel(
    const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t L, int64_t Hsrc, int64_t Hdst,
    int64_t vec_src, int64_t vec_dst, int64_t v0, bool flip, RowSplit by_vec, RowSplit by_rep) {
  const int64_t bt = blockIdx.x, b = bt / L, t = bt - b * L;
  const int64_t ts = flip ? L - 1 - t : t;
  const uint4* srow = src + (b * L + ts) * Hsrc * vec_src + v0;
  uint4* drow = dst + bt * Hdst * vec_dst;
  const uint32_t n = static_cast<uint32_t>(Hdst * vec_dst);
  for (uint32_t j = threadIdx.x; j < n; j += kRowThreads) {
    const uint32_t h = by_vec.div(j), v = j - h * static_cast<uint32_t>(vec_dst);
    drow[j] = __ldg(srow + int64_t(by_rep.div(h)) * vec_src + v);
  }
}

// float32 copy: dst[b, t, h, f] = src[b, flip ? L-1-t : t, h / rep, f], src float32 or bf16;
// four consecutive f per thread (F a multiple of 4)
template <typename IN>
__global__ void __launch_bounds__(kRowThreads) widen_flip_expand_kernel(
    const IN* __restrict__ src, float* __restrict__ dst, int64_t L, int64_t Hsrc, int64_t Hdst, int64_t F,
    bool flip, RowSplit by_quads, RowSplit by_rep) {
  const int64_t bt = blockIdx.x, b = bt / L, t = bt - b * L;
  const int64_t ts = flip ? L - 1 - t : t;
  const IN* srow = src + (b * L + ts) * Hsrc * F;
  float* drow = dst + bt * Hdst * F;
  const uint32_t quads = static_cast<uint32_t>(F / 4), n = static_cast<uint32_t>(Hdst) * quads;
  for (uint32_t j = threadIdx.x; j < n; j += kRowThreads) {
    const uint32_t h = by_quads.div(j), f = 4 * (j - h * quads);
    const IN* sp = srow + int64_t(by_rep.div(h)) * F + f;
    float4 o;
    if constexpr (sizeof(IN) == 2) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(sp));
      o = make_float4(bf16lo_to_f32(w.x), bf16hi_to_f32(w.x), bf16lo_to_f32(w.y), bf16hi_to_f32(w.y));
    } else {
      o = __ldg(reinterpret_cast<const float4*>(sp));
    }
    *reinterpret_cast<float4*>(drow + int64_t(h) * F + f) = o;
  }
}

// the decay steps of the reversed scan: step t of the reversed sequence decays by dt of
// original token L - t (the token after it in forward time); nothing decays at t = 0
__global__ void reverse_decay_kernel(const float* __restrict__ dt, float* __restrict__ out, int64_t L,
                                     int64_t H, int64_t total) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int64_t h = i % H, bt = i / H, t = bt % L, b = bt / L;
  out[i] = t == 0 ? 0.f : __ldg(dt + (b * L + (L - t)) * H + h);
}

// (rows, P, N) -> (rows, Nk, P) for the columns n0 .. n0 + Nk - 1, float32
__global__ void transpose_state_kernel(const float* __restrict__ src, float* __restrict__ dst, int64_t P,
                                       int64_t N, int64_t n0, int64_t Nk, int64_t total) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int64_t n = i % Nk, pr = i / Nk, p = pr % P, r = pr / P;
  dst[(r * Nk + n) * P + p] = __ldg(src + (r * P + p) * N + n0 + n);
}

// one warp per (b, t, h): dx, dL/dcs, <x, g B> and <dy, x> from dy, x, y (without the skip
// term) and the reverse scan's output g B (stored time-reversed)
template <typename IO>
__global__ void combine_kernel(const IO* __restrict__ dy, const IO* __restrict__ x, const float* __restrict__ yssm,
                               const float* __restrict__ gB_rev, const float* __restrict__ dt,
                               const float* __restrict__ D, IO* __restrict__ dx, float* __restrict__ dcs,
                               float* __restrict__ xgB, float* __restrict__ dyx, int64_t L, int64_t H, int64_t P,
                               int64_t rows) {
  const int64_t row = int64_t(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int64_t h = row % H, bt = row / H, t = bt % L, b = bt / L;
  const int64_t rrow = (b * L + (L - 1 - t)) * H + h;
  const float d = __ldg(dt + row), dsk = D ? __ldg(D + h) : 0.f;
  float s_dy = 0.f, s_xg = 0.f, s_dx = 0.f;
  for (int64_t p = lane; p < P; p += 32) {
    const float g = ldf(gB_rev, rrow * P + p), xv = ldf(x, row * P + p), dyv = ldf(dy, row * P + p);
    s_dy = fmaf(dyv, ldf(yssm, row * P + p), s_dy);
    s_xg = fmaf(xv, g, s_xg);
    s_dx = fmaf(dyv, xv, s_dx);
    stf(dx, row * P + p, fmaf(d, g, dsk * dyv));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    s_dy += __shfl_xor_sync(0xffffffffu, s_dy, off);
    s_xg += __shfl_xor_sync(0xffffffffu, s_xg, off);
    s_dx += __shfl_xor_sync(0xffffffffu, s_dx, off);
  }
  if (lane == 0) {
    dcs[row] = s_dy - d * s_xg;
    xgB[row] = s_xg;
    dyx[row] = s_dx;
  }
}

// one block per (b, h): dL/dcs at the last token gains <dfinal, final>
__global__ void final_dot_kernel(const float* __restrict__ dfinal, const float* __restrict__ fin,
                                 float* __restrict__ dcs, int64_t L, int64_t H, int64_t PN) {
  __shared__ float red[32];
  const int64_t bh = blockIdx.x, b = bh / H, h = bh % H;
  float s = 0.f;
  for (int64_t i = threadIdx.x; i < PN; i += blockDim.x) s = fmaf(__ldg(dfinal + bh * PN + i), __ldg(fin + bh * PN + i), s);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    s = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (threadIdx.x == 0) dcs[(b * L + L - 1) * H + h] += s;
  }
}

// one warp per (b, h): the reverse cumulative sum r_t = sum_{s >= t} dL/dcs_s, in rounds of 32
// tokens from the end; ddt_t = <x, g B>_t + A r_t, and this (b, h)'s shares of dA (sum dt_t r_t)
// and of dD (sum <dy_t, x_t>)
__global__ void reverse_cumsum_kernel(const float* __restrict__ dcs, const float* __restrict__ xgB,
                                      const float* __restrict__ dyx, const float* __restrict__ dt,
                                      const float* __restrict__ A, float* __restrict__ ddt,
                                      float* __restrict__ dA_part, float* __restrict__ dD_part, int64_t L,
                                      int64_t H, int64_t BH) {
  const int64_t bh = int64_t(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (bh >= BH) return;
  const int64_t b = bh / H, h = bh % H;
  const float a = __ldg(A + h);
  float carry = 0.f, acc = 0.f, accd = 0.f;
  for (int64_t top = L - 1; top >= 0; top -= 32) {
    const int64_t t = top - lane;  // lane 0 takes the latest token of the round
    const int64_t i = (b * L + t) * H + h;
    float v = t >= 0 ? __ldg(dcs + i) : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += o;
    }
    const float r = carry + v;
    if (t >= 0) {
      const float d = __ldg(dt + i);
      ddt[i] = fmaf(a, r, __ldg(xgB + i));
      acc = fmaf(d, r, acc);
      accd += __ldg(dyx + i);
    }
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    acc += __shfl_xor_sync(0xffffffffu, acc, off);
    accd += __shfl_xor_sync(0xffffffffu, accd, off);
  }
  if (lane == 0) {
    dA_part[bh] = acc;
    dD_part[bh] = accd;
  }
}

// out[h] = sum_b part[b, h]
__global__ void sum_batches_kernel(const float* __restrict__ part, float* __restrict__ out, int64_t nb, int64_t H) {
  const int64_t h = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (h >= H) return;
  float s = 0.f;
  for (int64_t b = 0; b < nb; ++b) s += __ldg(part + b * H + h);
  out[h] = s;
}

// out[b, t, g, n] = sum over the heads h of group g of scale(b, t, h) y[b, t', h, n], with
// t' = L-1-t when flip and scale = dt when given (else 1)
// (y has Nk columns per row; out has N, of which n0 .. n0 + Nk - 1 are written); one block per
// (b, t)
template <typename IO>
__global__ void __launch_bounds__(kRowThreads) group_sum_kernel(
    const IO* __restrict__ y, const float* __restrict__ dt, IO* __restrict__ out, int64_t L, int64_t H, int64_t G,
    int64_t N, int64_t n0, int64_t Nk, bool flip, RowSplit by_nk) {
  const int64_t bt = blockIdx.x, b = bt / L, t = bt - b * L;
  const int64_t ts = flip ? L - 1 - t : t;
  const int64_t hpg = H / G;
  const IO* yrow = y + (b * L + ts) * H * Nk;
  const float* drow = dt ? dt + bt * H : nullptr;
  const uint32_t n_out = static_cast<uint32_t>(G * Nk);
  for (uint32_t j = threadIdx.x; j < n_out; j += kRowThreads) {
    const uint32_t g = by_nk.div(j), n = j - g * static_cast<uint32_t>(Nk);
    float s = 0.f;
    for (int64_t k = 0; k < hpg; ++k) {
      const int64_t h = g * hpg + k;
      const float sc = drow ? __ldg(drow + h) : 1.f;
      s = fmaf(sc, ldf(yrow, h * Nk + n), s);
    }
    stf(out, (bt * G + g) * N + n0 + n, s);
  }
}

// dinit = a_0 g_0 = exp(A dt_0) times the reverse scan's final state
__global__ void dinit_kernel(const float* __restrict__ g0, const float* __restrict__ dt, const float* __restrict__ A,
                             float* __restrict__ dinit, int64_t L, int64_t H, int64_t PN, int64_t total) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int64_t bh = i / PN, b = bh / H, h = bh % H;
  dinit[i] = expf(__ldg(A + h) * __ldg(dt + (b * L) * H + h)) * __ldg(g0 + i);
}

inline unsigned blocks_for(int64_t n, int per) { return static_cast<unsigned>((n + per - 1) / per); }

}  // namespace

cudaError_t launch_flip_expand(const void* src, void* dst, int64_t b, int64_t L, int64_t Hsrc, int64_t Hdst,
                               int64_t src_row_bytes, int64_t col_byte0, int64_t dst_row_bytes, bool flip,
                               cudaStream_t st) {
  const int64_t vec_dst = dst_row_bytes / 16;
  if (b * L == 0 || Hdst * vec_dst == 0) return cudaSuccess;
  flip_expand_kernel<<<static_cast<unsigned>(b * L), kRowThreads, 0, st>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), L, Hsrc, Hdst, src_row_bytes / 16, vec_dst,
      col_byte0 / 16, flip, row_split(vec_dst), row_split(Hdst / Hsrc));
  return cudaGetLastError();
}

cudaError_t launch_reverse_decay(const float* dt, float* out, int64_t b, int64_t L, int64_t H, cudaStream_t st) {
  const int64_t total = b * L * H;
  reverse_decay_kernel<<<blocks_for(total, 256), 256, 0, st>>>(dt, out, L, H, total);
  return cudaGetLastError();
}

cudaError_t launch_transpose_state(const float* src, float* dst, int64_t rows, int64_t P, int64_t N, int64_t n0,
                                   int64_t Nk, cudaStream_t st) {
  const int64_t total = rows * P * Nk;
  transpose_state_kernel<<<blocks_for(total, 256), 256, 0, st>>>(src, dst, P, N, n0, Nk, total);
  return cudaGetLastError();
}

cudaError_t launch_bwd_combine(const Problem& p, const void* dy, const void* x, const float* yssm, const float* gB_rev,
                               const float* dt, const float* D, void* dx, float* dcs, float* xgB, float* dyx,
                               cudaStream_t st) {
  const int64_t rows = p.b * p.L * p.H;
  const unsigned grid = blocks_for(rows, 8);
  if (p.io_bf16)
    combine_kernel<uint16_t><<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(dy), static_cast<const uint16_t*>(x),
                                                   yssm, gB_rev, dt, D, static_cast<uint16_t*>(dx), dcs, xgB, dyx,
                                                   p.L, p.H, p.P, rows);
  else
    combine_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(dy), static_cast<const float*>(x), yssm,
                                                gB_rev, dt, D, static_cast<float*>(dx), dcs, xgB, dyx, p.L, p.H,
                                                p.P, rows);
  return cudaGetLastError();
}

cudaError_t launch_widen_flip_expand(const void* src, float* dst, int64_t b, int64_t L, int64_t Hsrc, int64_t Hdst,
                                     int64_t F, bool flip, bool src_bf16, cudaStream_t st) {
  if (b * L == 0 || Hdst * F == 0) return cudaSuccess;
  if (F % 4 != 0) return cudaErrorInvalidValue;  // headdim and dstate are multiples of 16 here
  const unsigned grid = static_cast<unsigned>(b * L);
  if (src_bf16)
    widen_flip_expand_kernel<uint16_t><<<grid, kRowThreads, 0, st>>>(
        static_cast<const uint16_t*>(src), dst, L, Hsrc, Hdst, F, flip, row_split(F / 4), row_split(Hdst / Hsrc));
  else
    widen_flip_expand_kernel<float><<<grid, kRowThreads, 0, st>>>(
        static_cast<const float*>(src), dst, L, Hsrc, Hdst, F, flip, row_split(F / 4), row_split(Hdst / Hsrc));
  return cudaGetLastError();
}

cudaError_t launch_bwd_scalars(const Problem& p, const float* dfinal, const float* fin, const float* xgB,
                               const float* dyx, const float* dt, const float* A, float* dcs, float* ddt,
                               float* part, float* dA, float* dD, cudaStream_t st) {
  if (dfinal) final_dot_kernel<<<static_cast<unsigned>(p.b * p.H), 256, 0, st>>>(dfinal, fin, dcs, p.L, p.H, p.P * p.N);
  const int64_t BH = p.b * p.H;
  reverse_cumsum_kernel<<<blocks_for(BH, 8), 256, 0, st>>>(dcs, xgB, dyx, dt, A, ddt, part, part + BH, p.L, p.H, BH);
  sum_batches_kernel<<<blocks_for(p.H, 128), 128, 0, st>>>(part, dA, p.b, p.H);
  if (dD) sum_batches_kernel<<<blocks_for(p.H, 128), 128, 0, st>>>(part + BH, dD, p.b, p.H);
  return cudaGetLastError();
}

cudaError_t launch_group_sum(const Problem& p, const void* y, const float* dt, void* out, int64_t n0, int64_t Nk,
                             bool flip, cudaStream_t st) {
  if (p.b * p.L == 0 || p.G * Nk == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(p.b * p.L);
  if (p.io_bf16)
    group_sum_kernel<uint16_t><<<grid, kRowThreads, 0, st>>>(
        static_cast<const uint16_t*>(y), dt, static_cast<uint16_t*>(out), p.L, p.H, p.G, p.N, n0, Nk, flip,
        row_split(Nk));
  else
    group_sum_kernel<float><<<grid, kRowThreads, 0, st>>>(
        static_cast<const float*>(y), dt, static_cast<float*>(out), p.L, p.H, p.G, p.N, n0, Nk, flip, row_split(Nk));
  return cudaGetLastError();
}

cudaError_t launch_dinit(const Problem& p, const float* g0, const float* dt, const float* A, float* dinit,
                         cudaStream_t st) {
  const int64_t total = p.b * p.H * p.P * p.N;
  dinit_kernel<<<blocks_for(total, 256), 256, 0, st>>>(g0, dt, A, dinit, p.L, p.H, p.P * p.N, total);
  return cudaGetLastError();
}

}  // namespace ssd
