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
// Two kernels, both float32 throughout, exp(dt A) as 2^(dt A log2 e) on the MUFU unit:
//
// decode_rows_kernel (N in {64, 128, 256, 512}, P a multiple of 8): the state is streamed
// with every warp instruction covering 512 consecutive bytes.  A warp owns 128 * CH
// consecutive floats of one head's state -- whole rows -- and lane l holds the float4s at
// offsets 128 i + 4 l (i < CH) in registers for the whole run, so the load and the store of the
// state are 16-byte accesses fully coalesced across the warp, with no shared memory and no
// block barrier.  Lane l's columns are 128 j + 4 l (N >= 128) or 4 (l mod N/4) (N = 64), so
// per token it needs only 4 N/128 (at least 4) elements of B_t and C_t, which it reads
// directly, together with x_t of the warp's rows; the next token's inputs are fetched before
// the current token is processed.  The row sums y_t[p] = sum_n h[p, n] C_t[n] are spread over
// the lanes that share a row: each lane first folds its own partial sums per row, then a
// recursive-halving exchange (reduce-scatter) leaves every row's total in one lane, V values
// over W lanes in V - 1 + log2(W / V) shuffles instead of V log2 W.
//
// decode_kernel (the other sizes, N = 64 * 2^k up to 2048): one CTA per (batch, head) with
// P * N / 64 threads; thread t keeps 64 consecutive state elements of row p = t / (N / 64)
// in registers.  Per token, B_t and C_t of the head's group are staged in shared memory;
// each thread updates its 64 elements, forms its part of y_t[p], and the N / 64 parts of a
// row (adjacent lanes of one warp) are summed with shuffles.
// Requirements of decode_kernel: N / 64 a power of two up to 32, P * N / 64 a multiple of 32
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

// ------------------------------------------------------------------ row-streaming kernel

// Recursive-halving reduce-scatter over the W lanes of a group (W a power of two, V <= W,
// groups are aligned blocks of W lanes): on return a[0] holds, in every lane, the total over
// the group of value number `idx` (the return value); the lanes of a group that agree in
// their bits above W / V - 1 hold the same value.
template <int V, int W>
__device__ __forceinline__ int reduce_scatter(float (&a)[V], int lane) {
  int idx = 0;
#pragma unroll
  for (int half = V / 2, m = W / 2; half >= 1; half /= 2, m /= 2) {
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = up ? a[k] : a[k + half];
      const float keep = up ? a[k + half] : a[k];
      a[k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
    if (up) idx += half;
  }
#pragma unroll
  for (int m = W / (2 * V); m >= 1; m /= 2) a[0] += __shfl_xor_sync(0xffffffffu, a[0], m);
  return idx;
}

// 32-bit words of IO data -> float element k
__device__ __forceinline__ float word_elem(const uint32_t* w, int k, float*) { return __uint_as_float(w[k]); }
__device__ __forceinline__ float word_elem(const uint32_t* w, int k, uint16_t*) {
  return (k & 1) ? bf16hi_to_f32(w[k >> 1]) : bf16lo_to_f32(w[k >> 1]);
}

// Loads `WORDS` 32-bit words from a 4 * WORDS-byte aligned address, widest access first.
template <int WORDS>
__device__ __forceinline__ void load_words(uint32_t (&w)[WORDS], const void* src) {
  if constexpr (WORDS % 4 == 0) {
#pragma unroll
    for (int k = 0; k < WORDS / 4; ++k) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + k);
      w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
    }
  } else if constexpr (WORDS % 2 == 0) {
#pragma unroll
    for (int k = 0; k < WORDS / 2; ++k) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(src) + k);
      w[2 * k] = v.x; w[2 * k + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int k = 0; k < WORDS; ++k) w[k] = __ldg(reinterpret_cast<const uint32_t*>(src) + k);
  }
}

template <typename IO, int N, int CH>
struct RowsGeom {
  static constexpr int kWarpFloats = 128 * CH;               // floats of state per warp
  static constexpr int kRows = kWarpFloats / N;              // rows per warp
  static constexpr int kSets = N >= 128 ? N / 128 : 1;       // float4 column sets per lane
  static constexpr int kV = N >= 128 ? kRows : CH;           // row partial sums per lane
  static constexpr int kW = N >= 128 ? 32 : N / 4;           // lanes that share a row
  static constexpr int kXWords = kRows * int(sizeof(IO)) / 4;        // x of the warp's rows
  static constexpr int kBWords = kSets * 4 * int(sizeof(IO)) / 4;    // B_t (or C_t) of a lane
  static_assert(kWarpFloats % N == 0 && kXWords >= 1, "a warp owns whole rows");
};

// One token's inputs of a warp, as raw 32-bit words (converted at use).
template <typename IO, int N, int CH>
struct TokenIn {
  using G = RowsGeom<IO, N, CH>;
  float dt;
  uint32_t x[G::kXWords];
  uint32_t b[G::kBWords];
  uint32_t c[G::kBWords];
  // depth of the prefetch ring: the next token's inputs load while one is processed (deeper
  // rings measured no faster: a run of tokens is bound by instruction issue, not by latency)
  static constexpr int kRing = 2;
};

template <typename IO, int N, int CH>
__device__ __forceinline__ void load_token(TokenIn<IO, N, CH>& in, const IO* x, const float* dt,
                                           const IO* Bm, const IO* Cm, int64_t bt, int64_t H,
                                           int64_t P, int64_t G, int64_t h, int64_t g, int row0,
                                           int lane) {
  using Geo = RowsGeom<IO, N, CH>;
  in.dt = __ldg(dt + bt * H + h);
  load_words(in.x, x + (bt * H + h) * P + row0);
  const int64_t bc = (bt * G + g) * N;
#pragma unroll
  for (int j = 0; j < Geo::kSets; ++j) {
    const int col = N >= 128 ? 128 * j + 4 * lane : 4 * (lane % Geo::kW);
    constexpr int kPer = 4 * int(sizeof(IO)) / 4;   // words per 4 elements
    uint32_t wb[kPer], wc[kPer];
    load_words(wb, Bm + bc + col);
    load_words(wc, Cm + bc + col);
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      in.b[j * kPer + k] = wb[k];
      in.c[j * kPer + k] = wc[k];
    }
  }
}

template <typename IO, int N, int CH, int K>
__global__ void __launch_bounds__(128) decode_rows_kernel(
    const IO* __restrict__ x, const float* __restrict__ dt, const float* __restrict__ A,
    const IO* __restrict__ Bm, const IO* __restrict__ Cm, const float* __restrict__ D,
    float* __restrict__ state, IO* __restrict__ y, int64_t T, int64_t H, int64_t P, int64_t G,
    int64_t nwarps) {
  using Geo = RowsGeom<IO, N, CH>;
  constexpr int V = Geo::kV, W = Geo::kW;
  const int lane = threadIdx.x & 31;
  const int64_t gw = int64_t(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  if (gw >= nwarps) return;  // no block barrier below: idle warps may leave
  const int64_t off = gw * Geo::kWarpFloats, PN = P * N;
  const int64_t bh = off / PN, b = bh / H, h = bh % H, g = h / (H / G);
  const int row0 = static_cast<int>((off % PN) / N);
  const int grp = N >= 128 ? 0 : lane / W;  // row of an instruction this lane is on (N = 64)
  float* sp = state + off + 4 * lane;
  grid_dep_wait();  // the state may come from the previous launch

  float4 hv[CH];
#pragma unroll
  for (int i = 0; i < CH; ++i) hv[i] = *reinterpret_cast<const float4*>(sp + 128 * i);
  const float a = __ldg(A + h) * kLog2e;
  const float dh = D ? __ldg(D + h) : 0.f;

  // x of partial-sum slot v: row v of the warp (N >= 128), or row 2 v + grp (N = 64)
  auto xval = [grp](const TokenIn<IO, N, CH>& in, int v) -> float {
    if constexpr (N >= 128) {
      return word_elem(in.x, v, static_cast<IO*>(nullptr));
    } else {
      const int r = (128 / N) * v;
      return grp ? word_elem(in.x, r + 1, static_cast<IO*>(nullptr))
                 : word_elem(in.x, r, static_cast<IO*>(nullptr));
    }
  };

  // one token: update the warp's rows, then form and store y_t of each row
  auto token = [&](const TokenIn<IO, N, CH>& in, int64_t bt) {
    const float d = in.dt, decay = ex2(d * a);
    const float2 dec2 = make_float2(decay, decay);
    // element pairs go through the packed float32x2 pipe: per pair one multiply (u B), one
    // fused update and one fused accumulation of h C
    float2 acc2[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc2[v] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      // this instruction's row (as a partial-sum slot) and column set
      const int v = N >= 128 ? i / Geo::kSets : i;
      const int j = N >= 128 ? i % Geo::kSets : 0;
      const float u = d * xval(in, v);
      const float2 u2 = make_float2(u, u);
      const float2 b01 = make_float2(word_elem(in.b, 4 * j, static_cast<IO*>(nullptr)),
                                     word_elem(in.b, 4 * j + 1, static_cast<IO*>(nullptr)));
      const float2 b23 = make_float2(word_elem(in.b, 4 * j + 2, static_cast<IO*>(nullptr)),
                                     word_elem(in.b, 4 * j + 3, static_cast<IO*>(nullptr)));
      const float2 c01 = make_float2(word_elem(in.c, 4 * j, static_cast<IO*>(nullptr)),
                                     word_elem(in.c, 4 * j + 1, static_cast<IO*>(nullptr)));
      const float2 c23 = make_float2(word_elem(in.c, 4 * j + 2, static_cast<IO*>(nullptr)),
                                     word_elem(in.c, 4 * j + 3, static_cast<IO*>(nullptr)));
      const float2 h01 = fma_f32x2(dec2, make_float2(hv[i].x, hv[i].y), mul_f32x2(u2, b01));
      const float2 h23 = fma_f32x2(dec2, make_float2(hv[i].z, hv[i].w), mul_f32x2(u2, b23));
      hv[i] = make_float4(h01.x, h01.y, h23.x, h23.y);
      acc2[v] = fma_f32x2(h23, c23, fma_f32x2(h01, c01, acc2[v]));
    }
    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = acc2[v].x + acc2[v].y;
    // D x enters each row's total once, through the first lane of the row's group
    if ((lane % W) == 0) {
#pragma unroll
      for (int v = 0; v < V; ++v) acc[v] = fmaf(dh, xval(in, v), acc[v]);
    }
    const int idx = reduce_scatter<V, W>(acc, lane);
    if ((lane & (W / V - 1)) == 0) {
      const int row = row0 + (N >= 128 ? idx : (128 / N) * idx + grp);
      st_io(y + (bt * H + h) * P + row, acc[0]);
    }
  };

  // the inputs of the next K - 1 tokens are in flight while a token is processed (a ring of
  // K register sets, indexed statically by unrolling the token loop K times)
  TokenIn<IO, N, CH> ring[K];
  const int64_t bt0 = b * T;
#pragma unroll
  for (int k = 0; k < K; ++k)
    if (k < T) load_token<IO, N, CH>(ring[k], x, dt, Bm, Cm, bt0 + k, H, P, G, h, g, row0, lane);
  for (int64_t t0 = 0; t0 < T; t0 += K) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int64_t t = t0 + k;
      if (t < T) {
        token(ring[k], bt0 + t);
        if (t + K < T) load_token<IO, N, CH>(ring[k], x, dt, Bm, Cm, bt0 + t + K, H, P, G, h, g, row0, lane);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < CH; ++i) *reinterpret_cast<float4*>(sp + 128 * i) = hv[i];
  grid_dep_launch();
}

constexpr int kRowsCH = 8;  // float4s of state per lane

template <typename IO, int N>
cudaError_t launch_rows(const Problem& p, const void* x, const float* dt, const float* A,
                        const void* B, const void* C, const float* D, float* state, void* y,
                        cudaStream_t st) {
  const int64_t nwarps = p.b * p.H * p.P * N / RowsGeom<IO, N, kRowsCH>::kWarpFloats;
  const dim3 grid(static_cast<unsigned>((nwarps + 3) / 4)), block(128);
  // one token per launch (the common decoding step) needs no prefetch ring and keeps more
  // warps resident; longer runs keep several tokens' inputs in flight
  constexpr int K = TokenIn<IO, N, kRowsCH>::kRing;
  auto kern = p.L == 1 ? decode_rows_kernel<IO, N, kRowsCH, 1> : decode_rows_kernel<IO, N, kRowsCH, K>;
  return launch_pdl(kern, grid, block, 0, st, static_cast<const IO*>(x),
                    dt, A, static_cast<const IO*>(B), static_cast<const IO*>(C), D, state,
                    static_cast<IO*>(y), p.L, p.H, p.P, p.G, nwarps);
}

bool rows_ok(const Problem& p) {
  const int64_t wf = 128 * kRowsCH;
  return (p.N == 64 || p.N == 128 || p.N == 256 || p.N == 512) && p.P % 8 == 0 &&
         (p.P * p.N) % wf == 0 && (p.b * p.H * p.P * p.N / wf + 3) / 4 <= int64_t(0x7fffffff);
}

}  // namespace

bool decode_ok(const Problem& p) {
  if (rows_ok(p)) return true;
  // the parts of a row are summed by xor-shuffles within a warp: N / 64 a power of two
  const int64_t per_row = p.N / 64;
  return p.N % 64 == 0 && per_row <= 32 && (per_row & (per_row - 1)) == 0 &&
         (p.P * per_row) % 32 == 0 && p.P * per_row <= 512 && p.b * p.H <= int64_t(0x7fffffff);
}

cudaError_t launch_decode(const Problem& p, const void* x, const float* dt, const float* A,
                          const void* B, const void* C, const float* D, float* state, void* y,
                          cudaStream_t st) {
  if (rows_ok(p)) {
    switch (p.N) {
      case 64:
        return p.io_bf16 ? launch_rows<uint16_t, 64>(p, x, dt, A, B, C, D, state, y, st)
                         : launch_rows<float, 64>(p, x, dt, A, B, C, D, state, y, st);
      case 128:
        return p.io_bf16 ? launch_rows<uint16_t, 128>(p, x, dt, A, B, C, D, state, y, st)
                         : launch_rows<float, 128>(p, x, dt, A, B, C, D, state, y, st);
      case 256:
        return p.io_bf16 ? launch_rows<uint16_t, 256>(p, x, dt, A, B, C, D, state, y, st)
                         : launch_rows<float, 256>(p, x, dt, A, B, C, D, state, y, st);
      default:
        return p.io_bf16 ? launch_rows<uint16_t, 512>(p, x, dt, A, B, C, D, state, y, st)
                         : launch_rows<float, 512>(p, x, dt, A, B, C, D, state, y, st);
    }
  }
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
