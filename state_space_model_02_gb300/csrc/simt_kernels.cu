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

// Both kernels are tiled matrix products on 64 x 64 output tiles: 256 threads, thread
// (tx, ty) = (tid % 16, tid / 16) owns rows 4 ty .. 4 ty + 3 and columns 4 tx .. 4 tx + 3, and
// every k step reads one float4 of each operand from shared memory (operands staged k-major,
// 16 k values at a time) for 16 fused multiply-adds.
constexpr int TM = 64;  // tile edge
constexpr int KT = 16;  // k values staged per step
constexpr int GS = TM + 4;  // row stride of the masked-matrix buffer (keeps float4 alignment)
constexpr float kMaxFactorSpan = 64.f;  // widest factored decay span inside a diagonal block

__device__ __forceinline__ void mma4x4(float (&acc)[4][4], const float4 a, const float4 b) {
  const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
}

// grid: x = p-tile * n_tiles + n-tile, y = h, z = b * nc + c.  S tile (64 p x 64 n) =
// sum over the chunk's tokens t of (w_t x[t, p]) B[t, n].
template <typename IO>
__global__ void __launch_bounds__(256, 3) chunk_state_simt_kernel(
    const IO* __restrict__ x, const IO* __restrict__ Bm, const float* __restrict__ cs2,
    const float* __restrict__ dtT, IO* __restrict__ S, int64_t L, int64_t H, int64_t P,
    int64_t N, int64_t G, int64_t Q, int64_t nc) {
  __shared__ __align__(16) float As[KT][TM];  // As[k][p] = w x[t0 + k, p0 + p]
  __shared__ __align__(16) float Bs[KT][TM];  // Bs[k][n] = B[t0 + k, n0 + n]
  __shared__ float wsm[256];                  // the chunk's decay weights (Q <= 256)
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int64_t n_tiles = (N + TM - 1) / TM;
  const int64_t p0 = (blockIdx.x / n_tiles) * TM, n0 = (blockIdx.x % n_tiles) * TM;
  const int64_t h = blockIdx.y, bc = blockIdx.z, b = bc / nc, c = bc % nc;
  const int64_t g = h / (H / G);
  const float* csr = cs2 + ((b * H + h) * nc + c) * Q;
  const float* dtr = dtT + ((b * H + h) * nc + c) * Q;
  const float last = csr[Q - 1];
  for (int t = tid; t < Q; t += 256) wsm[t] = c * Q + t < L ? ex2(last - csr[t]) * dtr[t] : 0.f;
  // the next tile's x and B values are loaded into registers while the current tile's
  // products run; element e = tid + 256 i of a tile is (k = e / TM, col = e % TM)
  constexpr int kPer = KT * TM / 256;
  float xr[kPer], br[kPer];
  auto load_tile = [&](int64_t t0) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + 256 * i, k = e / TM, col = e % TM;
      const int64_t tok = c * Q + t0 + k;
      xr[i] = 0.f;
      br[i] = 0.f;
      if (tok < L) {
        if (p0 + col < P) xr[i] = ld_io(x, ((b * L + tok) * H + h) * P + p0 + col);
        if (n0 + col < N) br[i] = ld_io(Bm, ((b * L + tok) * G + g) * N + n0 + col);
      }
    }
  };
  float acc[4][4] = {};
  load_tile(0);
  __syncthreads();  // weights ready
  for (int64_t t0 = 0; t0 < Q; t0 += KT) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + 256 * i, k = e / TM, col = e % TM;
      As[k][col] = wsm[t0 + k] * xr[i];
      Bs[k][col] = br[i];
    }
    __syncthreads();
    if (t0 + KT < Q) load_tile(t0 + KT);
#pragma unroll
    for (int k = 0; k < KT; ++k)
      mma4x4(acc, *reinterpret_cast<const float4*>(&As[k][4 * ty]), *reinterpret_cast<const float4*>(&Bs[k][4 * tx]));
    __syncthreads();
  }
  IO* out = S + (((b * nc + c) * H + h) * P) * N;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const int64_t p = p0 + 4 * ty + r, n = n0 + 4 * tx + cc;
      if (p < P && n < N) st_io(out, p * N + n, acc[r][cc]);
    }
}

// grid: x = b * nc + c, y = 64-row tile of the chunk, z = group * head_split + part.  The
// CTA computes the tile's causal C_i . B_j (j <= i, j < jmax) once -- it is the same for every
// head of the group -- into dynamic shared memory, transposed (CBs[j][i]), then runs the heads
// [part * per, (part + 1) * per) of the group.  Per head the decay 2^{cs2_i - cs2_j} dt_j is
// applied in blocks of KT columns [j0, j1], j1 = j0 + KT - 1: 2^{cs2_j1 - cs2_j} dt_j scales the
// staged x rows and 2^{cs2_i - cs2_j1} (0 for rows above the block) scales the block's partial
// sums, so no per-head matrix is formed.  With decaying steps (dt A <= 0) both factors are
// <= 1 for every row i >= j1, whatever the step sizes; only rows inside the block see a row
// factor above 1, bounded by 2^{cs2_j0 - cs2_j1}.  A block that holds such rows and decays by
// more than kMaxFactorSpan (log2 units) takes each weight as one exp2 of its own instead.
template <typename IO, typename HT>
__global__ void __launch_bounds__(256, 2) chunk_scan_simt_kernel(
    const IO* __restrict__ x, const IO* __restrict__ Bm, const IO* __restrict__ Cm,
    const float* __restrict__ D, const float* __restrict__ cs2, const float* __restrict__ dtT,
    const HT* __restrict__ hprev, IO* __restrict__ y, int64_t L, int64_t H, int64_t P, int64_t N,
    int64_t G, int64_t Q, int64_t nc, int64_t head_split) {
  extern __shared__ __align__(16) float CBs[];  // [jmax][GS]
  // padded rows: the C / B / hprev fills write a column k at a time (stride GS, not TM, keeps
  // those transposing stores from all landing in one bank)
  __shared__ __align__(16) float As[KT][GS];
  __shared__ __align__(16) float Bs[KT][GS];
  __shared__ float cs_i[TM], e_i[TM];
  __shared__ float csq[256], dtq[256];  // the current head's cs2 and dt rows of the chunk (Q <= 256)
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int64_t i0 = int64_t(blockIdx.y) * TM;
  const int64_t bc = blockIdx.x, b = bc / nc, c = bc % nc;
  const int64_t g = blockIdx.z / head_split, part = blockIdx.z % head_split;
  const int64_t hpg = H / G, per = (hpg + head_split - 1) / head_split;
  const int64_t h_begin = g * hpg + part * per, h_end = min(g * hpg + hpg, h_begin + per);
  const int64_t jmax = i0 + TM < Q ? i0 + TM : Q;  // columns j < jmax can be causal for these rows
  auto row_ok = [&](int64_t i_chunk) { return i_chunk < Q && c * Q + i_chunk < L; };
  // Every operand tile is 16 x 64 values, four per thread.  The loops below run over flat
  // sequences of tiles, and the next tile's global loads go into registers before the current
  // tile's products, so their latency overlaps the products.  For the C-major fills
  // (k = state column, consecutive threads read consecutive columns) element e = tid + 256 m is
  // (row e / KT, k = e % KT); for the x fill it is (k = e / TM, column e % TM).
  constexpr int kPer = KT * TM / 256;
  float ra[kPer], rb[kPer];
  auto load_c_rows = [&](int64_t n0) {  // ra: C rows of the tile, transposed on the store
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int e = tid + 256 * m, r = e / KT, k = e % KT;
      const int64_t n = n0 + k, ti = i0 + r;
      ra[m] = (row_ok(ti) && n < N) ? ld_io(Cm, ((b * L + c * Q + ti) * G + g) * N + n) : 0.f;
    }
  };
  auto store_rows = [&]() {  // ra -> As, rb -> Bs, both transposed (k-major)
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int e = tid + 256 * m, r = e / KT, k = e % KT;
      As[k][r] = ra[m];
      Bs[k][r] = rb[m];
    }
  };

  // Phase 1: the causal C . B^T of the tile's rows, head-independent; (j0, n0) tiles in order
  const int64_t nn = (N + KT - 1) / KT, n_cb = ((jmax + TM - 1) / TM) * nn;
  auto load_cb = [&](int64_t t) {
    const int64_t j0 = (t / nn) * TM, n0 = (t % nn) * KT;
    load_c_rows(n0);
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int e = tid + 256 * m, r = e / KT, k = e % KT;
      const int64_t n = n0 + k, tj = j0 + r;
      rb[m] = (row_ok(tj) && n < N) ? ld_io(Bm, ((b * L + c * Q + tj) * G + g) * N + n) : 0.f;
    }
  };
  {
    float acc[4][4] = {};
    load_cb(0);
    for (int64_t t = 0; t < n_cb; ++t) {
      store_rows();
      __syncthreads();
      if (t + 1 < n_cb) load_cb(t + 1);
#pragma unroll
      for (int k = 0; k < KT; ++k)
        mma4x4(acc, *reinterpret_cast<const float4*>(&As[k][4 * ty]), *reinterpret_cast<const float4*>(&Bs[k][4 * tx]));
      __syncthreads();
      if (t % nn == nn - 1) {
        const int64_t j0 = (t / nn) * TM;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int64_t j = j0 + 4 * tx + cc;
          if (j < jmax) {
            float v[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) v[r] = (j <= i0 + 4 * ty + r) ? acc[r][cc] : 0.f;
            *reinterpret_cast<float4*>(&CBs[j * GS + 4 * ty]) = make_float4(v[0], v[1], v[2], v[3]);
          }
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[r][cc] = 0.f;
        }
      }
    }
  }

  // Phase 2: per head and 64-column p tile, n1 tiles of Y1 = (L o CB) x (x rows j0 .. j0 + KT)
  // then n2 tiles of Y2 = C hprev^T (state columns n0 .. n0 + KT), one flat sequence over the
  // CTA's heads
  const int64_t np = (P + TM - 1) / TM, n1 = (jmax + KT - 1) / KT, n2 = nn;
  const int64_t per_tile = n1 + n2, per_head = np * per_tile, n_all = (h_end - h_begin) * per_head;
  auto load_tile = [&](int64_t t) {
    const int64_t h = h_begin + t / per_head, rem = t % per_head;
    const int64_t p0 = (rem / per_tile) * TM, q = rem % per_tile;
    if (q < n1) {
      const int64_t j0 = q * KT;
#pragma unroll
      for (int m = 0; m < kPer; ++m) {
        const int e = tid + 256 * m, k = e / TM, col = e % TM;
        const int64_t tj = j0 + k;
        ra[m] = (row_ok(tj) && p0 + col < P) ? ld_io(x, ((b * L + c * Q + tj) * H + h) * P + p0 + col) : 0.f;
      }
    } else {
      const int64_t n0 = (q - n1) * KT;
      load_c_rows(n0);
      const HT* hp = hprev + (((b * nc + c) * H + h) * P) * N;
#pragma unroll
      for (int m = 0; m < kPer; ++m) {
        const int e = tid + 256 * m, r = e / KT, k = e % KT;
        const int64_t n = n0 + k;
        rb[m] = (p0 + r < P && n < N) ? ld_io(hp, (p0 + r) * N + n) : 0.f;
      }
    }
  };
  float acc1[4][4], acc2[4][4];
  if (n_all > 0) load_tile(0);
  for (int64_t t = 0; t < n_all; ++t) {
    const int64_t h = h_begin + t / per_head, rem = t % per_head;
    const int64_t p0 = (rem / per_tile) * TM, q = rem % per_tile;
    if (rem == 0) {
      // a new head: its cs2 / dt rows (the previous head's epilogue has read e_i)
      const float* csr = cs2 + ((b * H + h) * nc + c) * Q;
      const float* dtr = dtT + ((b * H + h) * nc + c) * Q;
      __syncthreads();
      if (tid < TM) {
        const bool in = i0 + tid < Q;
        cs_i[tid] = in ? csr[i0 + tid] : 0.f;
        e_i[tid] = in ? ex2(csr[i0 + tid]) : 0.f;
      }
      for (int64_t j = tid; j < Q; j += 256) {
        csq[j] = csr[j];
        dtq[j] = dtr[j];
      }
      __syncthreads();
    }
    if (q == 0) {
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) acc1[r][cc] = acc2[r][cc] = 0.f;
    }
    if (q < n1) {
      const int64_t j0 = q * KT;
      const float cj1 = csq[j0 + KT - 1];
      // uniform over the CTA: a block left of every row of the tile (j0 < i0) always factors
      const bool factored = j0 < i0 || fabsf(csq[j0] - cj1) <= kMaxFactorSpan;
#pragma unroll
      for (int m = 0; m < kPer; ++m) {
        const int e = tid + 256 * m, k = e / TM, col = e % TM;
        const int tj = int(j0) + k;
        Bs[k][col] = ra[m] * (factored ? ex2(cj1 - csq[tj]) * dtq[tj] : dtq[tj]);
      }
      __syncthreads();
      if (t + 1 < n_all) load_tile(t + 1);
      if (factored) {
        float part_acc[4][4] = {};
#pragma unroll
        for (int k = 0; k < KT; ++k)
          mma4x4(part_acc, *reinterpret_cast<const float4*>(&CBs[(j0 + k) * GS + 4 * ty]),
                 *reinterpret_cast<const float4*>(&Bs[k][4 * tx]));
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int il = 4 * ty + r;
          const float rf = (j0 <= i0 + il) ? ex2(cs_i[il] - cj1) : 0.f;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) acc1[r][cc] = fmaf(rf, part_acc[r][cc], acc1[r][cc]);
        }
      } else {
        // every weight 2^{cs2_i - cs2_j} (j <= i) on its own; CBs is already zero for j > i
#pragma unroll 4
        for (int k = 0; k < KT; ++k) {
          const int64_t j = j0 + k;
          const float cjk = csq[j];
          const float4 cb = *reinterpret_cast<const float4*>(&CBs[j * GS + 4 * ty]);
          const float4 xv = *reinterpret_cast<const float4*>(&Bs[k][4 * tx]);
          const float cbv[4] = {cb.x, cb.y, cb.z, cb.w}, xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int il = 4 * ty + r;
            const float a = j <= i0 + il ? cbv[r] * ex2(cs_i[il] - cjk) : 0.f;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) acc1[r][cc] = fmaf(a, xw[cc], acc1[r][cc]);
          }
        }
      }
      __syncthreads();
    } else {
      store_rows();
      __syncthreads();
      if (t + 1 < n_all) load_tile(t + 1);
#pragma unroll
      for (int k = 0; k < KT; ++k)
        mma4x4(acc2, *reinterpret_cast<const float4*>(&As[k][4 * ty]), *reinterpret_cast<const float4*>(&Bs[k][4 * tx]));
      __syncthreads();
    }
    if (q == per_tile - 1) {
      const float Dh = D ? D[h] : 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int il = 4 * ty + r;
        const int64_t ti = i0 + il;
        if (!row_ok(ti)) continue;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int64_t p = p0 + 4 * tx + cc;
          if (p < P) {
            const int64_t off = ((b * L + c * Q + ti) * H + h) * P + p;
            st_io(y, off, acc1[r][cc] + e_i[il] * acc2[r][cc] + Dh * ld_io(x, off));
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_chunk_state_simt(const Problem& p, const void* x, const void* B, const float* cs2,
                                    const float* dtT, void* S, cudaStream_t st) {
  const int64_t tiles = ((p.P + TM - 1) / TM) * ((p.N + TM - 1) / TM);
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
  // split a group's heads over CTAs: more CTAs fill the SMs' resident slots, but a partial
  // last wave costs as much as a full one and every CTA computes its own C.B^T
  const int64_t row_tiles = (p.Q + TM - 1) / TM, base = row_tiles * p.b * p.nc * p.G;
  int sms = num_sms_current_device();
  if (sms <= 0) sms = 1;
  const size_t smem = static_cast<size_t>(p.Q) * GS * sizeof(float);
  cudaError_t e;
  const auto kb = chunk_scan_simt_kernel<uint16_t, uint16_t>;
  const auto kf = chunk_scan_simt_kernel<float, float>;
  e = cudaFuncSetAttribute(p.io_bf16 ? reinterpret_cast<const void*>(kb) : reinterpret_cast<const void*>(kf),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, p.io_bf16 ? reinterpret_cast<const void*>(kb) : reinterpret_cast<const void*>(kf), 256, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  // cost of a split s ~ waves x (heads per CTA + the CTA's own C.B^T)
  const int64_t slots = int64_t(per_sm) * sms;
  int64_t split = 1, best = -1;
  for (int64_t s = 1; s <= p.hpg; ++s) {
    const int64_t waves = (base * s + slots - 1) / slots;
    const int64_t cost = waves * ((p.hpg + s - 1) / s + 1);
    if (best < 0 || cost < best) {
      best = cost;
      split = s;
    }
  }
  if (p.G * split > 65535) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(p.b * p.nc), static_cast<unsigned>(row_tiles),
                  static_cast<unsigned>(p.G * split));
  if (p.io_bf16) {
    auto k = kb;
    k<<<grid, 256, smem, st>>>(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(B),
                               static_cast<const uint16_t*>(C), D, cs2, dtT,
                               static_cast<const uint16_t*>(hprev), static_cast<uint16_t*>(y), p.L,
                               p.H, p.P, p.N, p.G, p.Q, p.nc, split);
  } else {
    auto k = kf;
    k<<<grid, 256, smem, st>>>(static_cast<const float*>(x), static_cast<const float*>(B),
                               static_cast<const float*>(C), D, cs2, dtT,
                               static_cast<const float*>(hprev), static_cast<float*>(y), p.L, p.H,
                               p.P, p.N, p.G, p.Q, p.nc, split);
  }
  return cudaGetLastError();
}

}  // namespace ssd
