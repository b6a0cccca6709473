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
// staged through shared memory with coalesced loads, then each lane sums Q/32 consecutive
// tokens and a warp-shuffle (Kogge-Stone) scan combines the lane totals.
#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kHeadsPerCta = 8;
constexpr float kLog2e = 1.4426950408889634f;

template <int Q>
__global__ void __launch_bounds__(256) chunk_cumsum_kernel(const float* __restrict__ dt,
                                                           const float* __restrict__ A,
                                                           float* __restrict__ cs2,
                                                           float* __restrict__ dtT, int64_t L,
                                                           int64_t H, int64_t nc) {
  constexpr int R = Q / 32;                 // tokens per lane
  constexpr int ROW = Q + Q / 32;           // padded row: index t + t/32 is bank-conflict free
  __shared__ float tile[kHeadsPerCta][ROW];
  const int64_t c = blockIdx.x, b = blockIdx.y, h0 = int64_t(blockIdx.z) * kHeadsPerCta;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int e = tid; e < Q * kHeadsPerCta; e += 256) {
    const int t = e / kHeadsPerCta, k = e % kHeadsPerCta;
    const int64_t tok = c * Q + t, h = h0 + k;
    float v = 0.f;  // zero padding past the sequence end and past the last head
    if (tok < L && h < H) v = __ldg(dt + (b * L + tok) * H + h);
    tile[k][t + t / 32] = v;
  }
  __syncthreads();

  const int64_t h = h0 + warp;
  if (h >= H) return;
  const float a = __ldg(A + h);
  float d[R], run = 0.f;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int t = lane * R + r;
    d[r] = tile[warp][t + t / 32];
    run += a * d[r];
    // keep the running in-lane prefix; the lane offset is added after the warp scan
    tile[warp][t + t / 32] = run;
  }
  // inclusive warp scan of the lane totals
  float incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  const float excl = incl - run;
  float* out_cs = cs2 + ((b * H + h) * nc + c) * Q + lane * R;
  float* out_dt = dtT + ((b * H + h) * nc + c) * Q + lane * R;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int t = lane * R + r;
    out_cs[r] = (excl + tile[warp][t + t / 32]) * kLog2e;
    out_dt[r] = d[r];
  }
}

}  // namespace

cudaError_t launch_chunk_cumsum(const Problem& p, const float* dt, const float* A, float* cs2,
                                float* dtT, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(p.nc), static_cast<unsigned>(p.b),
                  static_cast<unsigned>((p.H + kHeadsPerCta - 1) / kHeadsPerCta));
  switch (p.Q) {
    case 64:
      chunk_cumsum_kernel<64><<<grid, 256, 0, st>>>(dt, A, cs2, dtT, p.L, p.H, p.nc);
      break;
    case 128:
      chunk_cumsum_kernel<128><<<grid, 256, 0, st>>>(dt, A, cs2, dtT, p.L, p.H, p.nc);
      break;
    case 256:
      chunk_cumsum_kernel<256><<<grid, 256, 0, st>>>(dt, A, cs2, dtT, p.L, p.H, p.nc);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace ssd
