// chunk_cumsum -- step 1 of the SSD forward scan.
//
// "Mamba-2 cuda-tile forward pass kernels" (devotd.net), section 2: the first kernel
// accumulates (decay rate x time step) inside each chunk and stores it for the two later
// kernels; its listing loads a (1, chunk, head-tile) tile of dt with zero padding and the
// per-head A, takes the cumulative sum along the chunk axis and scales it by log2(e).
// Section 3 relays the decay cumsum and dt out so later reads are contiguous; here both
// leave this kernel as (b, H, nc, Q) float32 rows, one contiguous row per (head, chunk).
//
// A tile = (chunk c, batch b, HT heads), scanned by 8 warps, each owning Q/8 consecutive tokens
// of the chunk.  A lane owns one head and a run of R consecutive tokens (32/HT lanes per head
// split the warp's tokens), so it reads its head's column of the (token, head) tile as dt lays it
// out.  The scan has three levels: the lane's run in registers (sequential in groups of 8
// tokens, then the groups' running totals), a warp-shuffle scan across the lanes of a head, and
// the warps' totals through shared memory.  Tokens past the sequence end read dt = 0 and then
// take the last token's cs2 bit for bit (it is the reference every decay of the chunk is taken
// against), copied through shared memory in the last chunk.
//
// Two kernels.  When dt's rows are 16-byte aligned (H a multiple of 4) and there are at least four
// tiles per SM, persistent CTAs walk the tiles strided by the grid: TMA copies each (token, head) tile of dt into one of two shared-
// memory stages while the previous tile is scanned; the lanes write their cs2 and dt runs as
// 16-byte vectors into head-major staging tiles (128-byte rows of 32 tokens, 16-byte chunks
// XOR-swizzled by head so that 8 lanes of different heads hit 8 different bank groups), and TMA
// stores send the staged rows out, so every global access is a whole tile (one load box and one
// store box per output).  Otherwise one CTA per tile loads dt and stores cs2 / dt from the lanes'
// registers directly.
#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;

// Tile geometry shared by both kernels.
template <int Q, int HT>
struct Geo {
  static constexpr int TL = 32 / HT;        // lanes per head in a warp
  static constexpr int TW = Q / kWarps;     // tokens per warp
  static constexpr int R = TW / TL;         // tokens per lane
  static constexpr int SG = R < 8 ? R : 8;  // sequential group inside a lane's run
  static constexpr int NSG = R / SG;
  static_assert(R >= 2 && R % SG == 0, "unsupported chunk / head-tile combination");
};

// Stores N (2 or a multiple of 4) consecutive floats from registers to a 4N-byte-aligned row.
template <int N>
__device__ __forceinline__ void store_run(float* dst, const float (&v)[N]) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int k = 0; k < N; k += 4)
      *reinterpret_cast<float4*>(dst + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
  } else {
    static_assert(N == 2, "runs are 2 tokens or a multiple of 4");
    *reinterpret_cast<float2*>(dst) = make_float2(v[0], v[1]);
  }
}

// Turns this lane's run of a * dt (in v, zero past the sequence end and for heads past H) into
// cs2.  Every thread of the CTA calls it: it holds one __syncthreads, two in the last chunk of a
// ragged sequence.  warp_total holds kWarps * HT floats, last_cs HT.
template <int Q, int HT>
__device__ __forceinline__ void scan_core(float (&v)[Geo<Q, HT>::R], int64_t c, int64_t L, int t0,
                                          float* warp_total, float* last_cs) {
  using G = Geo<Q, HT>;
  constexpr int R = G::R, SG = G::SG, NSG = G::NSG, TL = G::TL;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = lane % HT, tl = lane / HT;
  // the lane's run: sequential sums in groups of SG, then the groups' running totals
#pragma unroll
  for (int g = 0; g < NSG; ++g)
#pragma unroll
    for (int k = 1; k < SG; ++k) v[g * SG + k] += v[g * SG + k - 1];
  if constexpr (NSG > 1) {
    float tot[NSG];
#pragma unroll
    for (int g = 0; g < NSG; ++g) tot[g] = v[g * SG + SG - 1];
    float run = tot[0];
#pragma unroll
    for (int g = 1; g < NSG; ++g) {
#pragma unroll
      for (int k = 0; k < SG; ++k) v[g * SG + k] += run;
      run += tot[g];
    }
  }
  // across the TL lanes of a head (lanes hl, hl + HT, ...): inclusive scan of the run totals
  float incl = v[R - 1];
#pragma unroll
  for (int off = 1; off < TL; off <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, incl, off * HT);
    if (tl >= off) incl += o;
  }
  const float up = __shfl_up_sync(0xffffffffu, incl, TL > 1 ? HT : 0);
  const float lane_prefix = tl > 0 ? up : 0.f;
  if (tl == TL - 1) warp_total[warp * HT + hl] = incl;
  __syncthreads();
  float prefix = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps - 1; ++w)
    if (w < warp) prefix += warp_total[w * HT + hl];
  prefix += lane_prefix;
#pragma unroll
  for (int r = 0; r < R; ++r) v[r] = (prefix + v[r]) * kLog2e;

  // last chunk of a ragged sequence: padded tokens repeat the last token's value exactly
  const int64_t in_chunk = L - c * Q;  // valid tokens of this chunk (uniform over the CTA)
  if (in_chunk < Q) {
    const int tlast = int(in_chunk) - 1;
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (t0 + r == tlast) last_cs[hl] = v[r];
    __syncthreads();
    const float lv = last_cs[hl];
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (t0 + r > tlast) v[r] = lv;
  }
}

// One CTA per tile; each lane loads its column of the tile straight from dt and stores its runs.
// unit_scale: dtT holds 1 for every token of the sequence (0 past its end) instead of dt -- the
// scan whose inputs are not scaled by the step, which the backward pass runs.
template <int Q, int HT>
__global__ void __launch_bounds__(256) chunk_cumsum_kernel(const float* __restrict__ dt,
                                                           const float* __restrict__ A,
                                                           float* __restrict__ cs2,
                                                           float* __restrict__ dtT, int64_t L,
                                                           int64_t H, int64_t nc, bool unit_scale) {
  using G = Geo<Q, HT>;
  constexpr int R = G::R;
  __shared__ float warp_total[kWarps * HT];
  __shared__ float last_cs[HT];
  const int64_t c = blockIdx.x, b = blockIdx.y, h0 = int64_t(blockIdx.z) * HT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = lane % HT, tl = lane / HT;
  const int64_t h = h0 + hl;
  const bool head_ok = h < H;
  const int t0 = warp * G::TW + tl * R;              // first token of the run, inside the chunk
  const int64_t tok0 = c * Q + t0;
  const int64_t left = L - tok0;                     // tokens of the run inside the sequence
  const int nvalid = left >= R ? R : left > 0 ? int(left) : 0;
  grid_dep_wait();    // dt may come from the previous kernel; cs2 / dtT may still be read by it
  grid_dep_launch();

  float v[R];
  {
    const float* src = dt + (b * L + tok0) * H + h;
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = head_ok && r < nvalid ? __ldg(src + int64_t(r) * H) : 0.f;
  }
  const int64_t row = ((b * H + h) * nc + c) * Q + t0;
  if (head_ok) {
    if (unit_scale) {
      float one[R];
#pragma unroll
      for (int r = 0; r < R; ++r) one[r] = r < nvalid ? 1.f : 0.f;
      store_run<R>(dtT + row, one);
    } else {
      store_run<R>(dtT + row, v);
    }
  }
  const float a = head_ok ? __ldg(A + h) : 0.f;
#pragma unroll
  for (int r = 0; r < R; ++r) v[r] *= a;
  scan_core<Q, HT>(v, c, L, t0, warp_total, last_cs);
  if (head_ok) store_run<R>(cs2 + row, v);
}

constexpr int kTmaStages = 2;

// Shared memory of the TMA kernel: two dt stages ((Q tokens x HT heads) float32, token-major as
// dt lays it out) and two output slots, each a cs2 tile and a dt tile in the swizzled head-major
// layout the TMA stores read: Q/32 boxes of HT rows x 128 bytes (32 tokens of one head).
template <int Q, int HT>
struct TmaSmem {
  static constexpr uint32_t kTile = Q * HT * 4;
  static constexpr uint32_t kBox = HT * 128;  // one store box: 32 tokens of every head
  static constexpr uint32_t kIn = 0;
  static constexpr uint32_t kOut = kTmaStages * kTile;  // slot o: cs2 at kOut + 2 o kTile, dt after
  static constexpr uint32_t kAlloc = kOut + 4 * kTile + 1024;  // + slack for 1024-byte alignment
  static_assert(kBox % 1024 == 0, "store boxes must stay 1024-byte aligned for the 128-byte swizzle");
};

// Byte offset of (head hl, tokens t..t+3) in a swizzled output tile: box t / 32, row hl, 16-byte
// chunk (t % 32) / 4 XOR (hl % 8) -- the 128-byte swizzle pattern of the store's tensor map.
template <int HT>
__device__ __forceinline__ uint32_t out_offset(int hl, int t) {
  return uint32_t(t >> 5) * (HT * 128) + uint32_t(hl) * 128 + (uint32_t(((t & 31) >> 2) ^ (hl & 7)) << 4);
}

// Persistent CTAs; tile t = (c, b, head tile z), c fastest; CTA k takes t = k, k + grid, ...
// Thread 0 keeps the next tile's copy in flight in the other dt stage, refilling a stage once
// every thread has read it, and issues the stores of a tile's staged outputs; a slot's staging is
// rewritten two tiles later, after thread 0 has seen that slot's stores finish reading it.
// Waits are bounded: on expiry the status word records SSD_ERR_TIMEOUT and the CTA runs its loop
// to the end without copying or storing anything more.
template <int Q, int HT>
__global__ void __launch_bounds__(256) chunk_cumsum_tma_kernel(const __grid_constant__ CUtensorMap tm_dt,
                                                               const __grid_constant__ CUtensorMap tm_cs,
                                                               const __grid_constant__ CUtensorMap tm_dtT,
                                                               const float* __restrict__ A, int64_t L,
                                                               int64_t H, int64_t nc, int64_t nb,
                                                               bool unit_scale, bool one_box,
                                                               uint32_t* status, uint64_t wait_ns) {
  using G = Geo<Q, HT>;
  using SM = TmaSmem<Q, HT>;
  constexpr int R = G::R;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  __shared__ __align__(8) uint64_t full[kTmaStages];
  __shared__ float warp_total[2][kWarps * HT];  // by tile parity: a fast warp may start the next
  __shared__ float last_cs[HT];
  __shared__ uint32_t abort_word;
  volatile uint32_t* abort_flag = &abort_word;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = lane % HT, tl = lane / HT;
  const int t0 = warp * G::TW + tl * R;
  const int64_t nz = (H + HT - 1) / HT, ntiles = nc * nb * nz;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTmaStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    *abort_flag = 0u;
    fence_mbar_init();
    prefetch_tmap(&tm_dt);
    prefetch_tmap(&tm_cs);
    prefetch_tmap(&tm_dtT);
  }
  __syncthreads();
  const WaitCtl ctl{wait_ns, abort_flag, status};
  grid_dep_wait();    // dt may come from the previous kernel; cs2 / dtT may still be read by it
  grid_dep_launch();

  uint32_t pend = 0u, ph = 0u;  // thread 0, bit s: stage s has a copy not yet seen complete / its parity
  auto issue = [&](int64_t t, int s, uint32_t parity) {
    const int64_t c = t % nc, rest = t / nc, b = rest % nb, z = rest / nb;
    mbar_arrive_expect_tx(smem_u32(&full[s]), SM::kTile);
    tma_load_3d(sb + SM::kIn + s * SM::kTile, &tm_dt, smem_u32(&full[s]), int32_t(z * HT), int32_t(c * Q),
                int32_t(b));
    pend |= 1u << s;
    ph = (ph & ~(1u << s)) | (parity << s);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTmaStages; ++s)
      if (blockIdx.x + int64_t(s) * gridDim.x < ntiles) issue(blockIdx.x + int64_t(s) * gridDim.x, s, 0u);
  }
  int k = 0;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++k) {
    const int s = k % kTmaStages, o = k & 1;
    const uint32_t parity = uint32_t(k / kTmaStages) & 1u;
    const int64_t c = t % nc, rest = t / nc, b = rest % nb, z = rest / nb;
    const int64_t h = z * HT + hl;
    const bool ok = mbar_wait(smem_u32(&full[s]), parity, ctl) && !*abort_flag;
    if (threadIdx.x == 0 && ok) pend &= ~(1u << s);
    // rows past L and heads past H arrive as zeros (the copy's out-of-bounds fill)
    const float* tile = reinterpret_cast<const float*>(smem + SM::kIn + s * SM::kTile);
    const float a = h < H ? __ldg(A + h) : 0.f;
    float v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = ok ? tile[(t0 + r) * HT + hl] * a : 0.f;
    // slot o's stores of two tiles ago must have read their staging before it is rewritten;
    // the scan's barrier publishes that to every thread
    if (threadIdx.x == 0) bulk_wait_read<1>();
    scan_core<Q, HT>(v, c, L, t0, warp_total[k & 1], last_cs);
    if (ok) {
      uint8_t* out_cs = smem + SM::kOut + 2 * o * SM::kTile;
      uint8_t* out_dt = out_cs + SM::kTile;
      const int64_t left = L - (c * Q + t0);
      float d[R];
#pragma unroll
      for (int r = 0; r < R; ++r) d[r] = unit_scale ? (r < left ? 1.f : 0.f) : tile[(t0 + r) * HT + hl];
      if constexpr (R % 4 == 0) {
#pragma unroll
        for (int r = 0; r < R; r += 4) {
          const uint32_t off = out_offset<HT>(hl, t0 + r);
          *reinterpret_cast<float4*>(out_cs + off) = make_float4(v[r], v[r + 1], v[r + 2], v[r + 3]);
          *reinterpret_cast<float4*>(out_dt + off) = make_float4(d[r], d[r + 1], d[r + 2], d[r + 3]);
        }
      } else {  // runs of 2 tokens: the lower or upper half of a 16-byte chunk
        static_assert(R == 2, "runs are 2 tokens or a multiple of 4");
        const uint32_t off = out_offset<HT>(hl, t0 & ~3) + uint32_t(t0 & 3) * 4;
        *reinterpret_cast<float2*>(out_cs + off) = make_float2(v[0], v[1]);
        *reinterpret_cast<float2*>(out_dt + off) = make_float2(d[0], d[1]);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();  // staging written, stage s read by every thread
    if (threadIdx.x == 0 && !*abort_flag) {
      const uint32_t out_cs = sb + SM::kOut + 2 * o * SM::kTile, out_dt = out_cs + SM::kTile;
      if (one_box) {  // the whole staged tile as one box of the 5-D view
        tma_store_5d(&tm_cs, out_cs, 0, int32_t(z * HT), 0, int32_t(c), int32_t(b));
        tma_store_5d(&tm_dtT, out_dt, 0, int32_t(z * HT), 0, int32_t(c), int32_t(b));
      } else {
        for (int tb = 0; tb < Q / 32; ++tb) {
          tma_store_4d(&tm_cs, out_cs + tb * SM::kBox, tb * 32, int32_t(c), int32_t(z * HT), int32_t(b));
          tma_store_4d(&tm_dtT, out_dt + tb * SM::kBox, tb * 32, int32_t(c), int32_t(z * HT), int32_t(b));
        }
      }
      bulk_commit();
      if (t + int64_t(kTmaStages) * gridDim.x < ntiles) issue(t + int64_t(kTmaStages) * gridDim.x, s, parity ^ 1u);
    }
  }
  // every copy issued must have landed, and every store completed, before the CTA exits
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTmaStages; ++s)
      if ((pend >> s) & 1u) (void)mbar_drain(smem_u32(&full[s]), (ph >> s) & 1u, kWaitLimitNs);
    bulk_wait0();
  }
}

template <int HT>
cudaError_t launch_heads(const Problem& p, const float* dt, const float* A, float* cs2, float* dtT,
                         cudaStream_t st, bool unit_scale) {
  const dim3 grid(static_cast<unsigned>(p.nc), static_cast<unsigned>(p.b),
                  static_cast<unsigned>((p.H + HT - 1) / HT));
  switch (p.Q) {
    case 64:
      return launch_pdl(chunk_cumsum_kernel<64, HT>, grid, dim3(256), 0, st, dt, A, cs2, dtT, p.L, p.H, p.nc, unit_scale);
    case 128:
      return launch_pdl(chunk_cumsum_kernel<128, HT>, grid, dim3(256), 0, st, dt, A, cs2, dtT, p.L, p.H, p.nc, unit_scale);
    case 256:
      return launch_pdl(chunk_cumsum_kernel<256, HT>, grid, dim3(256), 0, st, dt, A, cs2, dtT, p.L, p.H, p.nc, unit_scale);
    default:
      return cudaErrorInvalidValue;
  }
}

struct TmaMaps {
  CUtensorMap dt, cs, dtT;
  bool one_box;  // cs / dtT are the 5-D view storing a whole tile per box (else 4-D, a box per 32 tokens)
};

template <int Q, int HT>
cudaError_t launch_tma_q(const Problem& p, const TmaMaps& m, const float* A, bool unit_scale,
                         uint32_t* status, cudaStream_t st, int sms) {
  using SM = TmaSmem<Q, HT>;
  auto kern = chunk_cumsum_tma_kernel<Q, HT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kAlloc);
  if (e != cudaSuccess) return e;
  static const int per_sm = [&] {
    int n = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 256, SM::kAlloc) == cudaSuccess && n > 0 ? n : 1;
  }();
  const int64_t tiles = p.nc * p.b * ((p.H + HT - 1) / HT);
  const int64_t grid = tiles < int64_t(sms) * per_sm ? tiles : int64_t(sms) * per_sm;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(256), SM::kAlloc, st, m.dt, m.cs, m.dtT, A,
                    p.L, p.H, p.nc, p.b, unit_scale, m.one_box, status, kWaitLimitNs);
}

template <int HT>
cudaError_t launch_tma(const Problem& p, const float* dt, const float* A, float* cs2, float* dtT,
                       bool unit_scale, uint32_t* status, cudaStream_t st, int sms) {
  TmaMaps m;
  {
    // dt (b, L, H) float32; a load box is (HT heads, Q tokens) of one batch
    const uint64_t dims[3] = {uint64_t(p.H), uint64_t(p.L), uint64_t(p.b)};
    const uint64_t strides[2] = {uint64_t(p.H * 4), uint64_t(p.L * p.H * 4)};
    const uint32_t box[3] = {uint32_t(HT), uint32_t(p.Q), 1u};
    if (!encode_tmap(&m.dt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dt, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE, nullptr))
      return cudaErrorInvalidValue;
  }
  // cs2 and dtT (b, H, nc, Q) float32, stored from the staging layout: rows of 128 bytes (32
  // tokens of one head, 128-byte swizzle), head rows inside token blocks.  Preferred view: 5-D
  // (token in block, head, token block, chunk, batch), whose (32, HT, Q/32, 1, 1) box is a whole
  // staged tile; else 4-D (token, chunk, head, batch) with a box per 32-token block.  Heads past
  // H are not written.
  {
    const uint64_t dims[5] = {32u, uint64_t(p.H), uint64_t(p.Q / 32), uint64_t(p.nc), uint64_t(p.b)};
    const uint64_t strides[4] = {uint64_t(p.nc * p.Q * 4), 128u, uint64_t(p.Q * 4), uint64_t(p.H * p.nc * p.Q * 4)};
    const uint32_t box[5] = {32u, uint32_t(HT), uint32_t(p.Q / 32), 1u, 1u};
    m.one_box = encode_tmap(&m.cs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, cs2, dims, strides, box,
                            CU_TENSOR_MAP_SWIZZLE_128B, nullptr) &&
                encode_tmap(&m.dtT, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, dtT, dims, strides, box,
                            CU_TENSOR_MAP_SWIZZLE_128B, nullptr);
  }
  if (!m.one_box) {
    const uint64_t dims[4] = {uint64_t(p.Q), uint64_t(p.nc), uint64_t(p.H), uint64_t(p.b)};
    const uint64_t strides[3] = {uint64_t(p.Q * 4), uint64_t(p.nc * p.Q * 4), uint64_t(p.H * p.nc * p.Q * 4)};
    const uint32_t box[4] = {32u, 1u, uint32_t(HT), 1u};
    if (!encode_tmap(&m.cs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, cs2, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B, nullptr) ||
        !encode_tmap(&m.dtT, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dtT, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B, nullptr))
      return cudaErrorInvalidValue;
  }
  switch (p.Q) {
    case 64:
      return launch_tma_q<64, HT>(p, m, A, unit_scale, status, st, sms);
    case 128:
      return launch_tma_q<128, HT>(p, m, A, unit_scale, status, st, sms);
    case 256:
      return launch_tma_q<256, HT>(p, m, A, unit_scale, status, st, sms);
    default:
      return cudaErrorInvalidValue;
  }
}

// Head tile: the widest of 32 / 16 / 8 heads that divides H and still gives two tiles per SM
// (wider tiles read longer runs of each dt row per load); 8 otherwise.
int cumsum_head_tile(const Problem& p, int sms) {
  const int64_t chunks = p.nc * p.b;
  for (int ht : {32, 16}) {
    if (p.H % ht == 0 && chunks * (p.H / ht) >= 2 * int64_t(sms)) return ht;
  }
  return 8;
}

}  // namespace

bool chunk_cumsum_tma_ok(const Problem& p, const float* dt) {
  // TMA needs a 16-byte aligned base and row stride (dt's row stride is 4H bytes)
  return p.H % 4 == 0 && (reinterpret_cast<uintptr_t>(dt) & 15u) == 0;
}

cudaError_t launch_chunk_cumsum(const Problem& p, const float* dt, const float* A, float* cs2,
                                float* dtT, uint32_t* status, cudaStream_t st, bool unit_scale) {
  int sms = num_sms_current_device();
  if (sms <= 0) sms = 1;
  const int ht = cumsum_head_tile(p, sms);
  // the persistent TMA kernel pays off once every CTA has several tiles to pipeline; with a tile
  // or two per SM the one-tile-per-CTA kernel is as fast and has no setup
  const int64_t tiles = p.nc * p.b * ((p.H + ht - 1) / ht);
  if (chunk_cumsum_tma_ok(p, dt) && tiles >= 4 * int64_t(sms)) {
    switch (ht) {
      case 32:
        return launch_tma<32>(p, dt, A, cs2, dtT, unit_scale, status, st, sms);
      case 16:
        return launch_tma<16>(p, dt, A, cs2, dtT, unit_scale, status, st, sms);
      default:
        return launch_tma<8>(p, dt, A, cs2, dtT, unit_scale, status, st, sms);
    }
  }
  switch (ht) {
    case 32:
      return launch_heads<32>(p, dt, A, cs2, dtT, st, unit_scale);
    case 16:
      return launch_heads<16>(p, dt, A, cs2, dtT, st, unit_scale);
    default:
      return launch_heads<8>(p, dt, A, cs2, dtT, st, unit_scale);
  }
}

}  // namespace ssd
