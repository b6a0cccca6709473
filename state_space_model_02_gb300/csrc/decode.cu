// decode -- the recurrent form over a short run of tokens (autoregressive decoding).
//
// "Compiler-First State Space Duality and Portable O(1) Autoregressive Caching for Inference"
// (gist.science), technical summary section 2: during autoregressive decoding the fixed-size
// state is the whole cache, and its per-token update runs inside an on-device loop rather than
// a host loop, so no host-device round trip happens per token; section 4 measures the decode
// phase as bound by HBM bandwidth.  One launch here advances the state over the shape's seqlen
// tokens, in place:
//     h <- exp(dt_t A_h) h + dt_t outer(x_t, B_t),     y_t = h C_t + D_h x_t
// The state is read once and written once per launch, whatever the number of tokens.
//
// One CTA per (batch, head) with P * N / 64 threads: thread t keeps 64 consecutive state
// elements of row p = t / (N / 64) in registers for the whole run.  Per token, B_t and C_t of
// the head's group are staged in shared memory; each thread updates its 64 elements, forms its
// part of y_t[p], and the N / 64 parts of a row (adjacent lanes of one warp) are summed with
// shuffles.  The recurrence runs in float32 throughout; exp(dt A) is 2^(dt A log2 e) on the
// MUFU unit.
// Requirements (decode_ok): N a multiple of 64 with N / 64 <= 32, P * N / 64 a multiple of 32
// and at most 512 (so that a thread's 64 state elements stay in registers).
#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ld_io(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ld_io(const uint16_t* p) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(p)) << 16);
}
__device__ __forceinline__ void st_io(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_io(uint16_t* p, float v) {
  *p = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu);
}

template <typename IO>
__global__ void __launch_bounds__(512) decode_kernel(
    const IO* __restrict__ x, const float* __restrict__ dt, const float* __restrict__ A,
    const IO* __restrict__ Bm, const IO* __restrict__ Cm, const float* __restrict__ D,
    float* __restrict__ state, IO* __restrict__ y, int64_t T, int64_t H, int64_t P, int64_t N,
    int64_t G) {
  extern __shared__ float bc[];  // [2][N]: B_t then C_t of this head's group
  const int64_t bh = blockIdx.x, b = bh / H, h = bh % H, g = h / (H / G);
  const int tid = threadIdx.x;
  const int per_row = static_cast<int>(N / 64);
  const int p = tid / per_row, n0 = (tid % per_row) * 64;
  grid_dep_wait();  // the state may come from the previous launch

  float* srow = state + (bh * P + p) * N + n0;
  float hv[64];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float4 v = *reinterpret_cast<const float4*>(srow + 4 * i);
    hv[4 * i] = v.x;
    hv[4 * i + 1] = v.y;
    hv[4 * i + 2] = v.z;
    hv[4 * i + 3] = v.w;
  }
  const float a = __ldg(A + h) * kLog2e;
  const float dh = D ? __ldg(D + h) : 0.f;
  for (int64_t t = 0; t < T; ++t) {
    const int64_t bt = b * T + t;
    for (int64_t i = tid; i < 2 * N; i += blockDim.x) {
      const int64_t n = i % N;
      bc[i] = ld_io((i < N ? Bm : Cm) + (bt * G + g) * N + n);
    }
    const float d = __ldg(dt + bt * H + h);
    const float xp = ld_io(x + (bt * H + h) * P + p);
    __syncthreads();
    const float decay = ex2(d * a), u = d * xp;
    const float* Bs = bc + n0;
    const float* Cs = bc + N + n0;
    float ypart = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float4 bv = *reinterpret_cast<const float4*>(Bs + 4 * i);
      const float4 cv = *reinterpret_cast<const float4*>(Cs + 4 * i);
      hv[4 * i] = fmaf(decay, hv[4 * i], u * bv.x);
      hv[4 * i + 1] = fmaf(decay, hv[4 * i + 1], u * bv.y);
      hv[4 * i + 2] = fmaf(decay, hv[4 * i + 2], u * bv.z);
      hv[4 * i + 3] = fmaf(decay, hv[4 * i + 3], u * bv.w);
      ypart = fmaf(hv[4 * i], cv.x, ypart);
      ypart = fmaf(hv[4 * i + 1], cv.y, ypart);
      ypart = fmaf(hv[4 * i + 2], cv.z, ypart);
      ypart = fmaf(hv[4 * i + 3], cv.w, ypart);
    }
    // the row's parts sit in per_row adjacent lanes of one warp
    for (int off = 1; off < per_row; off <<= 1) ypart += __shfl_xor_sync(0xffffffffu, ypart, off);
    if (tid % per_row == 0) st_io(y + (bt * H + h) * P + p, fmaf(dh, xp, ypart));
    __syncthreads();  // bc is refilled for the next token
  }
#pragma unroll
  for (int i = 0; i < 16; ++i)
    *reinterpret_cast<float4*>(srow + 4 * i) = make_float4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
  grid_dep_launch();
}

}  // namespace

bool decode_ok(const Problem& p) {
  const int64_t per_row = p.N / 64;
  return p.N % 64 == 0 && per_row <= 32 && (p.P * per_row) % 32 == 0 && p.P * per_row <= 512 &&
         p.b * p.H <= int64_t(0x7fffffff);
}

cudaError_t launch_decode(const Problem& p, const void* x, const float* dt, const float* A,
                          const void* B, const void* C, const float* D, float* state, void* y,
                          cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(p.b * p.H)), block(static_cast<unsigned>(p.P * (p.N / 64)));
  const size_t smem = static_cast<size_t>(2 * p.N) * sizeof(float);
  if (p.io_bf16)
    return launch_pdl(decode_kernel<uint16_t>, grid, block, smem, st, static_cast<const uint16_t*>(x),
                      dt, A, static_cast<const uint16_t*>(B), static_cast<const uint16_t*>(C), D,
                      state, static_cast<uint16_t*>(y), p.L, p.H, p.P, p.N, p.G);
  return launch_pdl(decode_kernel<float>, grid, block, smem, st, static_cast<const float*>(x), dt, A,
                    static_cast<const float*>(B), static_cast<const float*>(C), D, state,
                    static_cast<float*>(y), p.L, p.H, p.P, p.N, p.G);
}

}  // namespace ssd
