// chunk_cumsum -- step 1 of the SSD forward scan.
//
// "Mamba-2 cuda-tile forward pass kernels" (devotd.net), section 2: the first kernel
// accumulates (decay rate x time step) inside each chunk and stores it for the two later
// kernels; its listing loads a (1, chunk, head-tile) tile of dt with zero padding and the
// per-head A, takes the cumulative sum along the chunk axis and scales it by log2(e).
// Section 3 relays the decay cumsum and dt out so later reads are contiguous; here both
// leave this kernel as (b, H, nc, Q) float32 rows, one contiguous row per (head, chunk).
//
// One CTA = (chunk c, batch b, tile of 8 heads); one warp per head.  The (Q x 8) dt tile is
// staged through shared memory with all loads in flight; each warp then scans its head's Q
// values in rounds of 32 tokens (a warp-shuffle Kogge-Stone scan per round plus a running
// carry), so each round writes one contiguous 128-byte row of cs2 and of dtT.
#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kHeadsPerCta = 8;
constexpr float kLog2e = 1.4426950408889634f;

// unit_scale: dtT holds 1 for every token of the sequence (0 past its end) instead of dt --
// the scan whose inputs are not scaled by the step, which the backward pass runs.
template <int Q>
__global__ void __launch_bounds__(256) chunk_cumsum_kernel(const float* __restrict__ dt,
                                                           const float* __restrict__ A,
                                                           float* __restrict__ cs2,
                                                           float* __restrict__ dtT, int64_t L,
                                                           int64_t H, int64_t nc, bool unit_scale) {
  constexpr int R = Q / 32;                 // tokens per lane
  constexpr int ROW = Q + Q / 32;           // padded row (t + t/32) for the staging writes
  __shared__ float tile[kHeadsPerCta][ROW];
  const int64_t c = blockIdx.x, b = blockIdx.y, h0 = int64_t(blockIdx.z) * kHeadsPerCta;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  grid_dep_wait();    // cs2 / dtT may still be read by the previous step's kernels
  grid_dep_launch();

  // all loads of the tile are issued before any is consumed (Q/32 per thread in flight)
  constexpr int kPer = Q * kHeadsPerCta / 256;
  float v[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = tid + 256 * i, t = e / kHeadsPerCta, k = e % kHeadsPerCta;
    const int64_t tok = c * Q + t, h = h0 + k;
    v[i] = 0.f;  // zero padding past the sequence end and past the last head
    if (tok < L && h < H) v[i] = __ldg(dt + (b * L + tok) * H + h);
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = tid + 256 * i, t = e / kHeadsPerCta, k = e % kHeadsPerCta;
    tile[k][t + t / 32] = v[i];
  }
  __syncthreads();

  const int64_t h = h0 + warp;
  if (h >= H) return;
  const float a = __ldg(A + h);
  float* out_cs = cs2 + ((b * H + h) * nc + c) * Q;
  float* out_dt = dtT + ((b * H + h) * nc + c) * Q;
  // round r covers tokens 32r .. 32r+31, one per lane: a warp-shuffle inclusive scan plus the
  // running total of the earlier rounds; every store is one coalesced 128-byte row
  float carry = 0.f;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int t = 32 * r + lane;
    const float d = tile[warp][t + t / 32];
    float incl = a * d;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    out_cs[t] = (carry + incl) * kLog2e;
    out_dt[t] = unit_scale ? (c * Q + t < L ? 1.f : 0.f) : d;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
}

}  // namespace

cudaError_t launch_chunk_cumsum(const Problem& p, const float* dt, const float* A, float* cs2,
                                float* dtT, cudaStream_t st, bool unit_scale) {
  const dim3 grid(static_cast<unsigned>(p.nc), static_cast<unsigned>(p.b),
                  static_cast<unsigned>((p.H + kHeadsPerCta - 1) / kHeadsPerCta));
  switch (p.Q) {
    case 64:
      return launch_pdl(chunk_cumsum_kernel<64>, grid, dim3(256), 0, st, dt, A, cs2, dtT, p.L, p.H, p.nc, unit_scale);
    case 128:
      return launch_pdl(chunk_cumsum_kernel<128>, grid, dim3(256), 0, st, dt, A, cs2, dtT, p.L, p.H, p.nc, unit_scale);
    case 256:
      return launch_pdl(chunk_cumsum_kernel<256>, grid, dim3(256), 0, st, dt, A, cs2, dtT, p.L, p.H, p.nc, unit_scale);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace ssd
