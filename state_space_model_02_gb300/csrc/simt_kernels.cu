// CUDA-core (FFMA) versions of chunk_state and chunk_scan.
//
// These serve every shape, in float32 or bf16 I/O, with float32 arithmetic throughout
// (no bf16 rounding of intermediates), which is what the float32 workload needs to stay
// within 1e-4 of the float64 oracle.  The tensor-core kernels (chunk_state_tc.cu,
// chunk_scan_tc.cu) replace them on the shapes those support.
//
// chunk_state ("Mamba-2 cuda-tile forward pass kernels", section 2, fwd_pass_state):
//     S[b,c,h,p,n] = sum_{t in chunk} 2^{cs2_last - cs2_t} dt_t x[t,p] B[t,n]
// chunk_scan (same section, compute_out):
//     y[i,p] = sum_{j<=i} 2^{cs2_i - cs2_j} dt_j (C_i . B_j) x[j,p]
//              + 2^{cs2_i} (C_i . hprev[p,:]) + D_h x[i,p]
// cs2 is the log2-domain in-chunk cumsum written by chunk_cumsum; rows past the sequence end
// read as zero (dt = 0 there, so they contribute nothing).
#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

__device__ __forceinline__ float ld_io(const float* p, int64_t i) { return __ldg(p + i); }
__device__ __forceinline__ float ld_io(const uint16_t* p, int64_t i) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(p + i)) << 16);
}
__device__ __forceinline__ void st_io(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_io(uint16_t* p, int64_t i, float v) {
  p[i] = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu);
}

constexpr int T = 32;  // tile edge

// grid: x = p-tile * n_tiles + n-tile, y = h, z = b * nc + c.  256 threads, 32x32 outputs.
template <typename IO>
__global__ void __launch_bounds__(256) chunk_state_simt_kernel(
    const IO* __restrict__ x, const IO* __restrict__ Bm, const float* __restrict__ cs2,
    const float* __restrict__ dtT, IO* __restrict__ S, int64_t L, int64_t H, int64_t P,
    int64_t N, int64_t G, int64_t Q, int64_t nc) {
  __shared__ float xs[T][T + 1];
  __shared__ float bs[T][T + 1];
  const int tid = threadIdx.x, tx = tid % T, ty = tid / T;  // ty in 0..7
  const int64_t n_tiles = (N + T - 1) / T;
  const int64_t p0 = (blockIdx.x / n_tiles) * T, n0 = (blockIdx.x % n_tiles) * T;
  const int64_t h = blockIdx.y, bc = blockIdx.z, b = bc / nc, c = bc % nc;
  const int64_t g = h / (H / G);
  const float* csr = cs2 + ((b * H + h) * nc + c) * Q;
  const float* dtr = dtT + ((b * H + h) * nc + c) * Q;
  const float last = csr[Q - 1];
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int64_t t0 = 0; t0 < Q; t0 += T) {
    // xs[t][p] = w_t * x[t, p], bs[t][n] = B[t, n]
    for (int e = tid; e < T * T; e += 256) {
      const int tt = e / T, cc = e % T;
      const int64_t t = t0 + tt, tok = c * Q + t;
      float xv = 0.f, bv = 0.f;
      if (tok < L) {
        const float w = ex2(last - csr[t]) * dtr[t];
        if (p0 + cc < P) xv = w * ld_io(x, ((b * L + tok) * H + h) * P + p0 + cc);
        if (n0 + cc < N) bv = ld_io(Bm, ((b * L + tok) * G + g) * N + n0 + cc);
      }
      xs[tt][cc] = xv;
      bs[tt][cc] = bv;
    }
    __syncthreads();
#pragma unroll 8
    for (int tt = 0; tt < T; ++tt) {
      const float bv = bs[tt][tx];
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] = fmaf(xs[tt][ty + 8 * k], bv, acc[k]);
    }
    __syncthreads();
  }
  IO* out = S + (((b * nc + c) * H + h) * P) * N;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int64_t p = p0 + ty + 8 * k, n = n0 + tx;
    if (p < P && n < N) st_io(out, p * N + n, acc[k]);
  }
}

// grid: x = row tile (32 rows of the chunk), y = h, z = b * nc + c.  256 threads.
// Dynamic shared memory: Gs[32][Q] (masked, decayed C.B^T rows).
template <typename IO, typename HT>
__global__ void __launch_bounds__(256) chunk_scan_simt_kernel(
    const IO* __restrict__ x, const IO* __restrict__ Bm, const IO* __restrict__ Cm,
    const float* __restrict__ D, const float* __restrict__ cs2, const float* __restrict__ dtT,
    const HT* __restrict__ hprev, IO* __restrict__ y, int64_t L, int64_t H, int64_t P, int64_t N,
    int64_t G, int64_t Q, int64_t nc) {
  extern __shared__ float Gs[];  // [T][Q]
  __shared__ float cs_s[T], e_s[T];
  __shared__ float ta[T][T + 1];
  __shared__ float tb[T][T + 1];
  const int tid = threadIdx.x, tx = tid % T, ty = tid / T;
  const int64_t i0 = int64_t(blockIdx.x) * T;
  const int64_t h = blockIdx.y, bc = blockIdx.z, b = bc / nc, c = bc % nc;
  const int64_t g = h / (H / G);
  const float* csr = cs2 + ((b * H + h) * nc + c) * Q;
  const float* dtr = dtT + ((b * H + h) * nc + c) * Q;
  const int64_t jmax = i0 + T;  // columns j < jmax can be causal for these rows
  if (tid < T) {
    cs_s[tid] = csr[i0 + tid];
    e_s[tid] = ex2(csr[i0 + tid]);
  }

  // Phase 1: Gs[i][j] = C_i . B_j for rows i0..i0+31 and j < jmax, then mask and decay.
  for (int64_t j0 = 0; j0 < jmax; j0 += T) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t n0 = 0; n0 < N; n0 += T) {
      for (int e = tid; e < T * T; e += 256) {
        const int r = e / T, cc = e % T;
        const int64_t ti = c * Q + i0 + r, tj = c * Q + j0 + r, n = n0 + cc;
        ta[r][cc] = (ti < L && n < N) ? ld_io(Cm, ((b * L + ti) * G + g) * N + n) : 0.f;
        tb[r][cc] = (tj < L && n < N) ? ld_io(Bm, ((b * L + tj) * G + g) * N + n) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int nn = 0; nn < T; ++nn) {
        const float bv = tb[tx][nn];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = fmaf(ta[ty + 8 * k][nn], bv, acc[k]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int il = ty + 8 * k;
      const int64_t i = i0 + il, j = j0 + tx;
      float v = 0.f;
      if (j <= i) v = acc[k] * ex2(cs_s[il] - csr[j]) * dtr[j];
      Gs[il * Q + j] = v;
    }
  }
  __syncthreads();

  // Phase 2: y[i][p] for p tiles of 32.
  const float Dh = D ? D[h] : 0.f;
  for (int64_t p0 = 0; p0 < P; p0 += T) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float acc2[4] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t j0 = 0; j0 < jmax; j0 += T) {
      for (int e = tid; e < T * T; e += 256) {
        const int r = e / T, cc = e % T;
        const int64_t tj = c * Q + j0 + r;
        ta[r][cc] = (tj < L && p0 + cc < P) ? ld_io(x, ((b * L + tj) * H + h) * P + p0 + cc) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int jj = 0; jj < T; ++jj) {
        const float xv = ta[jj][tx];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = fmaf(Gs[(ty + 8 * k) * Q + j0 + jj], xv, acc[k]);
      }
      __syncthreads();
    }
    const HT* hp = hprev + (((b * nc + c) * H + h) * P) * N;
    for (int64_t n0 = 0; n0 < N; n0 += T) {
      for (int e = tid; e < T * T; e += 256) {
        const int r = e / T, cc = e % T;
        const int64_t ti = c * Q + i0 + r, n = n0 + cc;
        ta[r][cc] = (ti < L && n < N) ? ld_io(Cm, ((b * L + ti) * G + g) * N + n) : 0.f;
        tb[r][cc] = (p0 + r < P && n < N) ? ld_io(hp, (p0 + r) * N + n) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int nn = 0; nn < T; ++nn) {
        const float hv = tb[tx][nn];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc2[k] = fmaf(ta[ty + 8 * k][nn], hv, acc2[k]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int il = ty + 8 * k;
      const int64_t ti = c * Q + i0 + il, p = p0 + tx;
      if (ti < L && p < P) {
        const int64_t off = ((b * L + ti) * H + h) * P + p;
        st_io(y, off, acc[k] + e_s[il] * acc2[k] + Dh * ld_io(x, off));
      }
    }
  }
}

}  // namespace

cudaError_t launch_chunk_state_simt(const Problem& p, const void* x, const void* B, const float* cs2,
                                    const float* dtT, void* S, cudaStream_t st) {
  const int64_t tiles = ((p.P + T - 1) / T) * ((p.N + T - 1) / T);
  const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(p.H),
                  static_cast<unsigned>(p.b * p.nc));
  if (p.io_bf16)
    chunk_state_simt_kernel<uint16_t><<<grid, 256, 0, st>>>(
        static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(B), cs2, dtT,
        static_cast<uint16_t*>(S), p.L, p.H, p.P, p.N, p.G, p.Q, p.nc);
  else
    chunk_state_simt_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(x),
                                                         static_cast<const float*>(B), cs2, dtT,
                                                         static_cast<float*>(S), p.L, p.H, p.P, p.N,
                                                         p.G, p.Q, p.nc);
  return cudaGetLastError();
}

cudaError_t launch_chunk_scan_simt(const Problem& p, const void* x, const void* B, const void* C,
                                   const float* D, const float* cs2, const float* dtT,
                                   const void* hprev, void* y, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(p.Q / T), static_cast<unsigned>(p.H),
                  static_cast<unsigned>(p.b * p.nc));
  const size_t smem = static_cast<size_t>(T) * p.Q * sizeof(float);
  if (p.io_bf16) {
    auto k = chunk_scan_simt_kernel<uint16_t, uint16_t>;
    k<<<grid, 256, smem, st>>>(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(B),
                               static_cast<const uint16_t*>(C), D, cs2, dtT,
                               static_cast<const uint16_t*>(hprev), static_cast<uint16_t*>(y), p.L,
                               p.H, p.P, p.N, p.G, p.Q, p.nc);
  } else {
    auto k = chunk_scan_simt_kernel<float, float>;
    k<<<grid, 256, smem, st>>>(static_cast<const float*>(x), static_cast<const float*>(B),
                               static_cast<const float*>(C), D, cs2, dtT,
                               static_cast<const float*>(hprev), static_cast<float*>(y), p.L, p.H,
                               p.P, p.N, p.G, p.Q, p.nc);
  }
  return cudaGetLastError();
}

}  // namespace ssd
