// selective_scan -- the Mamba-1 selective scan, fused: load, discretise, scan, read out.
//
// "3.3 Hardware-aware algorithm and GPU memory hierarchy" (booiljung.github.io):
// section 2.1 -- the parameters (delta, A, B, C) and x come in from HBM, the discretisation
// by zero-order hold (Abar = exp(delta A), Bbar = (delta A)^-1 (exp(delta A) - I) delta B) and
// the recurrence run on chip, and only y goes back; the expanded state (b, L, D, N) is never
// stored.  Section 3 fuses the four steps into one kernel; section 4.1 writes the update as
// the first-order linear recurrence h_t = Abar_t h_{t-1} + Bbar_t x_t.  With A diagonal per
// channel d and state n:
//     h[d,n] <- exp(delta[d] A[d,n]) h[d,n] + (exp(delta[d] A[d,n]) - 1) / A[d,n] B[n] x[d]
//     y[d]    = sum_n C[n] h[d,n] + Dskip[d] x[d]
//
// The work is one exponential per (channel, state, token), so the kernel is bound by the
// arithmetic pipes, not by HBM (about 10 instruction slots and one MUFU ex2 per element
// against 4 bytes of x, delta and y per channel and token).  The b * D * N chains are
// independent, so no parallel scan over tokens is needed: each lane owns two states of one
// channel for the whole sequence and walks the tokens in order (the sequence order keeps
// the chain exact; the parallelism is across chains).
//
// One warp per CTA.  Lane l holds states (2p, 2p + 1), p = l mod N/2, of channel
// d0 + l / (N/2) in registers.  Every 32 tokens, lane t stages token t's inputs for the
// warp -- delta and x of the warp's 64/N channels, B and C -- widened to float32 in shared
// memory (the next block's loads are issued before the current block is processed).  Per
// token each lane reads one float4 (its B and C pair) and one float2 (its channel's delta,
// x).  The state-independent work of N tokens -- z = delta A log2 e, Abar = 2^z (MUFU), the
// zero-order-hold factor (exp(w) - 1) / A with w = z ln 2, taken as delta (1 + w/2 + w^2/6)
// for |w| < 1/64 (where exp(w) - 1 would cancel) and as (Abar - 1) / A above, and
// u = factor B x -- is done first, on float32 pairs (fma.rn.f32x2), so that N independent
// chains hide the MUFU and shared-memory latencies; then the N dependent updates
// h <- Abar h + u and the read-out shares C . h follow.  Each lane's two shares are summed,
// and the N / 2 lanes of a channel reduce N / 2 tokens at a time with a recursive-halving
// exchange that leaves one token's y in each lane.
#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr float kLog2eSel = 1.4426950408889634f;
constexpr int kSelTokens = 32;  // tokens staged per block (one per lane)

template <int N>
struct SelGeom {
  static constexpr int kW = N / 2;                 // lanes per channel
  static constexpr int kCW = 32 / kW;              // channels per warp
  // staged token row (floats): N/2 float4 (B pair, C pair), then kCW float2 (delta, x),
  // padded to 16 bytes and then to an odd number of 16-byte chunks: lane t writes row t, and
  // an odd row stride puts the 8 lanes of each 16-byte store phase on 8 different bank quads
  // (an even one paired them up, two accesses per bank: 162 -> 154 us on the 130M layer)
  static constexpr int kBC = 0;
  static constexpr int kDX = 2 * N;
  static constexpr int kRow0 = (2 * N + 2 * kCW + 3) / 4 * 4;
  static constexpr int kRow = (kRow0 / 4) % 2 == 0 ? kRow0 + 4 : kRow0;
};

template <typename IO, int CNT>
struct RawVec {
  static constexpr int kBytes = CNT * int(sizeof(IO));
  static constexpr int kWords = kBytes >= 4 ? kBytes / 4 : 1;
  uint32_t w[kWords];
};

template <typename IO, int CNT>
__device__ __forceinline__ void load_raw(RawVec<IO, CNT>& r, const IO* src) {
  constexpr int B = RawVec<IO, CNT>::kBytes;
  if constexpr (B % 16 == 0) {
#pragma unroll
    for (int k = 0; k < B / 16; ++k) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + k);
      r.w[4 * k] = v.x; r.w[4 * k + 1] = v.y; r.w[4 * k + 2] = v.z; r.w[4 * k + 3] = v.w;
    }
  } else if constexpr (B == 8) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
    r.w[0] = v.x; r.w[1] = v.y;
  } else if constexpr (B == 4) {
    r.w[0] = __ldg(reinterpret_cast<const uint32_t*>(src));
  } else {
    static_assert(B == 2, "unexpected vector size");
    r.w[0] = __ldg(reinterpret_cast<const uint16_t*>(src));
  }
}

template <typename IO, int CNT>
__device__ __forceinline__ float raw_elem(const RawVec<IO, CNT>& r, int k) {
  if constexpr (sizeof(IO) == 4) {
    return __uint_as_float(r.w[k]);
  } else {
    return (k & 1) ? bf16hi_to_f32(r.w[k >> 1]) : bf16lo_to_f32(r.w[k >> 1]);
  }
}

template <typename IO, int N>
struct TokenRaw {
  RawVec<IO, SelGeom<N>::kCW> dl, x;
  RawVec<IO, N> b, c;
};

__device__ __forceinline__ void st_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_out(uint16_t* p, float v) {
  *p = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu);
}

// Recursive-halving reduce-scatter within aligned groups of W lanes (V = W values): on
// return a[0] holds the group total of value number `idx` (the return value).
template <int W>
__device__ __forceinline__ int reduce_scatter_group(float (&a)[W], int lane) {
  int idx = 0;
#pragma unroll
  for (int half = W / 2; half >= 1; half /= 2) {
    const bool up = (lane & half) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = up ? a[k] : a[k + half];
      const float keep = up ? a[k + half] : a[k];
      a[k] = keep + __shfl_xor_sync(0xffffffffu, send, half);
    }
    if (up) idx += half;
  }
  return idx;
}

template <typename IO, int N>
__global__ void __launch_bounds__(32) selective_scan_kernel(
    const IO* __restrict__ x, const IO* __restrict__ delta, const float* __restrict__ A,
    const IO* __restrict__ Bm, const IO* __restrict__ Cm, const float* __restrict__ Dskip,
    const float* __restrict__ init, float* __restrict__ final_state, IO* __restrict__ y, int64_t L,
    int64_t D) {
  using Geo = SelGeom<N>;
  constexpr int W = Geo::kW, CW = Geo::kCW, TB = kSelTokens, RF = Geo::kRow;
  __shared__ __align__(16) float stage[2][TB * RF];
  const int lane = threadIdx.x;
  const int64_t warps_per_batch = D / CW;
  const int64_t b = blockIdx.x / warps_per_batch, d0 = (blockIdx.x % warps_per_batch) * CW;
  const int c = lane / W, p = lane % W;
  const int64_t d = d0 + c;
  grid_dep_wait();  // inputs may come from the previous kernel in the stream

  const float2 Av = *reinterpret_cast<const float2*>(A + d * N + 2 * p);
  const float2 invA = make_float2(1.f / Av.x, 1.f / Av.y);  // unused where A = 0 (|w| < 1/64)
  float2 h = make_float2(0.f, 0.f);
  if (init) h = *reinterpret_cast<const float2*>(init + (b * D + d) * N + 2 * p);
  const float dsk = (Dskip && p == 0) ? __ldg(Dskip + d) : 0.f;

  // staging: lane t loads token t of a block and writes its row in float32
  auto load_token = [&](TokenRaw<IO, N>& r, int64_t tok) {
    const int64_t row = (b * L + tok) * D + d0;
    load_raw(r.dl, delta + row);
    load_raw(r.x, x + row);
    load_raw(r.b, Bm + (b * L + tok) * N);
    load_raw(r.c, Cm + (b * L + tok) * N);
  };
  auto store_token = [&](const TokenRaw<IO, N>& r, float* rowp) {
#pragma unroll
    for (int q = 0; q < N / 2; ++q)
      *reinterpret_cast<float4*>(rowp + Geo::kBC + 4 * q) =
          make_float4(raw_elem(r.b, 2 * q), raw_elem(r.b, 2 * q + 1), raw_elem(r.c, 2 * q),
                      raw_elem(r.c, 2 * q + 1));
#pragma unroll
    for (int k = 0; k < CW; ++k)
      *reinterpret_cast<float2*>(rowp + Geo::kDX + 2 * k) = make_float2(raw_elem(r.dl, k), raw_elem(r.x, k));
  };

  {
    TokenRaw<IO, N> r;
    if (lane < L) {
      load_token(r, lane);
      store_token(r, &stage[0][lane * RF]);
    }
  }
  __syncwarp();

  const float2 ninvA = make_float2(-invA.x, -invA.y);
  const float2 a2z = make_float2(Av.x * kLog2eSel, Av.y * kLog2eSel);  // exp(delta A) = 2^(delta a2z)
  // the hold's factor for small |w| as a polynomial in z = w log2 e: 1 + (ln2/2) z + (ln2^2/6) z^2
  const float2 one = make_float2(1.f, 1.f);
  const float2 k1z = make_float2(0.34657359027997264f, 0.34657359027997264f);
  const float2 k2z = make_float2(0.08007410688212759f, 0.08007410688212759f);
  constexpr float kZSmall = 0.022541950359959f;  // |w| < 1/64

  // the state-independent work of a token: Abar and u = Bbar x for the lane's two states, its
  // C pair and the skip term
  struct Pre {
    float2 ab, u, cc;
    float sx;
  };
  auto prepare = [&](const float* rowp) -> Pre {
    const float4 bc = *reinterpret_cast<const float4*>(rowp + Geo::kBC + 4 * p);
    const float2 dx = *reinterpret_cast<const float2*>(rowp + Geo::kDX + 2 * c);
    const float2 dl2 = make_float2(dx.x, dx.x);
    const float2 z = mul_f32x2(dl2, a2z);
    const float2 ab = make_float2(ex2(z.x), ex2(z.y));
    const float2 e = fma_f32x2(z, fma_f32x2(z, k2z, k1z), one);
    const float2 cs = mul_f32x2(dl2, e);
    const float2 cl = fma_f32x2(ab, invA, ninvA);
    const float2 cf = make_float2(fabsf(z.x) < kZSmall ? cs.x : cl.x, fabsf(z.y) < kZSmall ? cs.y : cl.y);
    const float2 u = mul_f32x2(cf, mul_f32x2(make_float2(bc.x, bc.y), make_float2(dx.y, dx.y)));
    Pre r;
    r.ab = ab;
    r.u = u;
    r.cc = make_float2(bc.z, bc.w);
    r.sx = dsk * dx.y;  // Dskip x enters once per channel (lane p = 0)
    return r;
  };

  // the sequential part: h <- Abar h + u, and the lane's share of y_t
  auto advance = [&](const Pre& r) -> float {
    h = fma_f32x2(r.ab, h, r.u);
    const float2 yc = mul_f32x2(r.cc, h);
    return r.sx + (yc.x + yc.y);
  };
  auto step = [&](const float* rowp) -> float { return advance(prepare(rowp)); };

  for (int64_t t0 = 0, blk = 0; t0 < L; t0 += TB, ++blk) {
    const int nt = static_cast<int>(L - t0 < TB ? L - t0 : TB);
    const bool has_next = t0 + TB < L;
    TokenRaw<IO, N> nxt;
    const bool mine = has_next && t0 + TB + lane < L;
    if (mine) load_token(nxt, t0 + TB + lane);
    const float* rows = stage[blk & 1];

    // full groups of 2W tokens: branch-free, so the per-token work that does not depend on
    // h (loads, exponentials, the hold's factor) overlaps across tokens; two reductions in
    // flight at once
    int tb = 0;
    for (; tb + 2 * W <= nt; tb += 2 * W) {
      // the state-independent work of all 2W tokens first, then the dependent updates
      float pa[W], pb[W];
      Pre pr[2 * W];
#pragma unroll
      for (int k = 0; k < 2 * W; ++k) pr[k] = prepare(rows + (tb + k) * RF);
#pragma unroll
      for (int k = 0; k < W; ++k) pa[k] = advance(pr[k]);
#pragma unroll
      for (int k = 0; k < W; ++k) pb[k] = advance(pr[W + k]);
      const int ia = reduce_scatter_group<W>(pa, lane);
      const int ib = reduce_scatter_group<W>(pb, lane);
      st_out(y + (b * L + t0 + tb + ia) * D + d, pa[0]);
      st_out(y + (b * L + t0 + tb + W + ib) * D + d, pb[0]);
    }
    for (; tb < nt; tb += W) {  // ragged tail of the sequence
      float part[W];
#pragma unroll
      for (int k = 0; k < W; ++k) part[k] = tb + k < nt ? step(rows + (tb + k) * RF) : 0.f;
      const int idx = reduce_scatter_group<W>(part, lane);
      if (tb + idx < nt) st_out(y + (b * L + t0 + tb + idx) * D + d, part[0]);
    }
    if (mine) store_token(nxt, &stage[(blk + 1) & 1][lane * RF]);
    __syncwarp();
  }
  if (final_state) *reinterpret_cast<float2*>(final_state + (b * D + d) * N + 2 * p) = h;
  grid_dep_launch();
}

template <typename IO, int N>
cudaError_t launch_sel(const SelProblem& p, const void* x, const void* delta, const float* A,
                       const void* B, const void* C, const float* Dskip, const float* init,
                       float* final_state, void* y, cudaStream_t st) {
  const int64_t warps = p.b * p.D / SelGeom<N>::kCW;
  return launch_pdl(selective_scan_kernel<IO, N>, dim3(static_cast<unsigned>(warps)), dim3(32), 0, st,
                    static_cast<const IO*>(x), static_cast<const IO*>(delta), A,
                    static_cast<const IO*>(B), static_cast<const IO*>(C), Dskip, init, final_state,
                    static_cast<IO*>(y), p.L, p.D);
}

}  // namespace

bool selective_ok(const SelProblem& p) {
  if (p.N != 8 && p.N != 16 && p.N != 32 && p.N != 64) return false;
  const int64_t cw = 64 / p.N;
  return p.D % cw == 0 && p.b * p.D / cw <= int64_t(0x7fffffff);
}

cudaError_t launch_selective_scan(const SelProblem& p, const void* x, const void* delta, const float* A,
                                  const void* B, const void* C, const float* Dskip, const float* init,
                                  float* final_state, void* y, cudaStream_t st) {
#define SSD_SEL_CASE(NN)                                                                          \
  case NN:                                                                                       \
    return p.io_bf16 ? launch_sel<uint16_t, NN>(p, x, delta, A, B, C, Dskip, init, final_state, y, st) \
                     : launch_sel<float, NN>(p, x, delta, A, B, C, Dskip, init, final_state, y, st);
  switch (p.N) {
    SSD_SEL_CASE(8)
    SSD_SEL_CASE(16)
    SSD_SEL_CASE(32)
    SSD_SEL_CASE(64)
    default:
      return cudaErrorInvalidValue;
  }
#undef SSD_SEL_CASE
}

}  // namespace ssd
