// chunk_cumsum -- step 1 of the SSD forward scan.
//
// "Mamba-2 cuda-tile forward pass kernels" (devotd.net), section 2: the first kernel
// accumulates (decay rate x time step) inside each chunk and stores it for the two later
// kernels; its listing loads a (1, chunk, head-tile) tile of dt with zero padding and the
// per-head A, takes the cumulative sum along the chunk axis and scales it by log2(e).
// Section 3 relays the decay cumsum and dt out so later reads are contiguous; here both
// leave this kernel as (b, H, nc, Q) float32 rows, one contiguous row per (head, chunk).
//
// One CTA = (chunk c, batch b, tile of HEADS heads), 8 warps.  The (Q x HEADS) dt tile is
// staged through shared memory with all loads in flight; each warp then scans its heads' Q
// values in rounds of 32 tokens (a warp-shuffle Kogge-Stone scan per round plus a running
// carry), so each round writes one contiguous 128-byte row of cs2 and of dtT.  HEADS = 8 (one
// head per warp) in general; HEADS = 32 (four per warp) when H is a multiple of 32 and the
// grid stays large, so that each warp-wide load reads whole 128-byte rows of dt (32 heads of
// one token) instead of 32-byte pieces of four rows.
#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;

// unit_scale: dtT holds 1 for every token of the sequence (0 past its end) instead of dt --
// the scan whose inputs are not scaled by the step, which the backward pass runs.
template <int Q, int HEADS>
__global__ void __launch_bounds__(256) chunk_cumsum_kernel(const float* __restrict__ dt,
                                                           const float* __restrict__ A,
                                                           float* __restrict__ cs2,
                                                           float* __restrict__ dtT, int64_t L,
                                                           int64_t H, int64_t nc, bool unit_scale) {
  constexpr int R = Q / 32;                 // tokens per lane
  // padded rows for the transposing staging writes: with 8 heads a warp writes 4 tokens x 8
  // heads (column t + t/32 spreads them over the banks); with 32 heads it writes one token
  // of 32 heads (a row pitch of Q + 1 puts the 32 rows in 32 banks)
  constexpr int ROW = HEADS == 32 ? Q + 1 : Q + Q / 32;
  __shared__ float tile[HEADS][ROW];
  auto col = [](int t) { return HEADS == 32 ? t : t + t / 32; };
  const int64_t c = blockIdx.x, b = blockIdx.y, h0 = int64_t(blockIdx.z) * HEADS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  grid_dep_wait();    // cs2 / dtT may still be read by the previous step's kernels
  grid_dep_launch();

  // all loads of the tile are issued before any is consumed (Q/32 per thread in flight)
  constexpr int kPer = Q * HEADS / 256;
  float v[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = tid + 256 * i, t = e / HEADS, k = e % HEADS;
    const int64_t tok = c * Q + t, h = h0 + k;
    v[i] = 0.f;  // zero padding past the sequence end and past the last head
    if (tok < L && h < H) v[i] = __ldg(dt + (b * L + tok) * H + h);
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = tid + 256 * i, t = e / HEADS, k = e % HEADS;
    tile[k][col(t)] = v[i];
  }
  __syncthreads();

  for (int hl = warp; hl < HEADS; hl += kWarps) {
    const int64_t h = h0 + hl;
    if (h >= H) return;
    const float a = __ldg(A + h);
    float* out_cs = cs2 + ((b * H + h) * nc + c) * Q;
    float* out_dt = dtT + ((b * H + h) * nc + c) * Q;
    // round r covers tokens 32r .. 32r+31, one per lane: a warp-shuffle inclusive scan plus the
    // running total of the earlier rounds; every store is one coalesced 128-byte row.  Tokens
    // past the sequence end repeat the last token's value bit for bit: each lane's prefix comes
    // from its own tree of additions, so summing the padding's zeros would not reproduce it, and
    // the chunk-end value is the reference every decay of the chunk is taken against.
    float carry = 0.f, last = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int t = 32 * r + lane;
      const float d = tile[hl][col(t)];
      float incl = a * d;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      float v = (carry + incl) * kLog2e;
      const int64_t valid = L - (c * Q + 32 * r);  // tokens of this round inside the sequence
      if (valid < 32) {                            // uniform over the warp
        const float lastv = __shfl_sync(0xffffffffu, v, valid > 0 ? int(valid) - 1 : 0);
        if (lane >= valid) v = valid > 0 ? lastv : last;
      }
      last = __shfl_sync(0xffffffffu, v, 31);
      out_cs[t] = v;
      out_dt[t] = unit_scale ? (c * Q + t < L ? 1.f : 0.f) : d;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
}

template <int HEADS>
cudaError_t launch_heads(const Problem& p, const float* dt, const float* A, float* cs2, float* dtT,
                         cudaStream_t st, bool unit_scale) {
  const dim3 grid(static_cast<unsigned>(p.nc), static_cast<unsigned>(p.b),
                  static_cast<unsigned>((p.H + HEADS - 1) / HEADS));
  switch (p.Q) {
    case 64:
      return launch_pdl(chunk_cumsum_kernel<64, HEADS>, grid, dim3(256), 0, st, dt, A, cs2, dtT, p.L, p.H, p.nc, unit_scale);
    case 128:
      return launch_pdl(chunk_cumsum_kernel<128, HEADS>, grid, dim3(256), 0, st, dt, A, cs2, dtT, p.L, p.H, p.nc, unit_scale);
    case 256:
      return launch_pdl(chunk_cumsum_kernel<256, HEADS>, grid, dim3(256), 0, st, dt, A, cs2, dtT, p.L, p.H, p.nc, unit_scale);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_chunk_cumsum(const Problem& p, const float* dt, const float* A, float* cs2,
                                float* dtT, cudaStream_t st, bool unit_scale) {
  int sms = num_sms_current_device();
  if (sms <= 0) sms = 1;
  if (p.H % 32 == 0 && p.nc * p.b * (p.H / 32) >= 2 * int64_t(sms))
    return launch_heads<32>(p, dt, A, cs2, dtT, st, unit_scale);
  return launch_heads<8>(p, dt, A, cs2, dtT, st, unit_scale);
}

}  // namespace ssd
