// chunk readout on the 5th-generation tensor cores: the inter-chunk term of chunk_scan for
// large states.
//
// "Mamba-2 cuda-tile forward pass kernels" (devotd.net), section 2: compute_out makes the token
// outputs from the chunk-start states.  Its term through the state entering the chunk is, for
// rows i of chunk c and head h,
//     Z[i, h, p] = 2^{cs2_i} * sum_n C[i, n] hprev[c, h, p, n]
// (the decay from the chunk start to token i times the read-out of the state).  With state sizes
// above 128 the whole C tile of a 128-row m-tile (128 x N) does not fit beside chunk_scan's other
// operands in shared memory, so this kernel computes Z for every (batch, chunk, m-tile, head
// pair) as its own product, the state dimension N being the K loop, and chunk_scan adds it to its
// intra-chunk part.  Z is (b, L, H, P) in bf16.
//
// Persistent CTAs (one per SM) walk the items (head pair fastest, then m-tile, chunk, batch), so
// the CTAs running at one time share C through L2.  Per item: M = 128 rows i, N = 2 heads x P =
// 128, K = N in 64-column steps; operand tiles (C: 128 rows x 64, hprev: both heads' 128 rows
// (h, p) x 64, both K-major, 128-byte swizzled) stream through a ring of stages that runs on
// across items, into one of two TMEM accumulators.
//   warp 0      TMA producer;
//   warp 1      tcgen05.mma issuer (4 MMAs of K = 16 per step);
//   warps 2-5   epilogue: accumulator row i (one TMEM lane) times 2^{cs2_i} of each head, to bf16,
//               swizzled staging, TMA store of the two heads' 64-column blocks of Z.
// Every wait is bounded; after an expiry the roles keep their loop counts but skip their work,
// then drain their own copies and MMAs and release TMEM.
// Requirements (chunk_readout_tc_ok): bf16 I/O, P = 64, Q in {128, 256}, N a multiple of 64.
#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kWarps = 6;
constexpr int kThreads = 32 * kWarps;
constexpr int kEpiWarp0 = 2;
constexpr int kStages = 5;
constexpr uint32_t kTile = 16384;          // one TMA box: 128 rows x 128 bytes
constexpr uint32_t kStage = 2 * kTile;     // C tile + hprev tile
constexpr uint32_t kBarEpi = 1;

struct RoParams {
  int32_t L, H, nc, Q, N, hpg, pairs_per_group, MT;
  int64_t items;
  const float* cs2;
  uint32_t* status;
  uint64_t wait_ns;
};

struct RoSmem {
  static constexpr uint32_t kRing = 0;
  static constexpr uint32_t kOut = kStages * kStage;    // staging: 2 heads x (128 rows x 128 B)
  static constexpr uint32_t kBars = kOut + 2 * kTile;
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kUsed = kAbort + 4;
  static constexpr uint32_t kAlloc = kUsed + 1024;      // slack for 1024-byte alignment
  static_assert(kAlloc <= 232448, "exceeds the per-CTA shared memory limit");
  static constexpr int kFull = 0, kEmpty = kStages, kAccFull = 2 * kStages, kAccEmpty = kAccFull + 2,
                       kDrain = kAccEmpty + 2;
};

struct RoItem {
  int b, c, mt, g, h0, nh;
};
__device__ __forceinline__ RoItem ro_item_at(int64_t i, const RoParams& prm) {
  RoItem it;
  const int64_t pairs = int64_t(prm.H / prm.hpg) * prm.pairs_per_group;
  const int64_t bcm = i / pairs;
  const int pair = static_cast<int>(i - bcm * pairs);
  it.g = pair / prm.pairs_per_group;
  it.h0 = it.g * prm.hpg + 2 * (pair % prm.pairs_per_group);
  it.nh = min(2, (it.g + 1) * prm.hpg - it.h0);
  it.mt = static_cast<int>(bcm % prm.MT);
  const int64_t bc = bcm / prm.MT;
  it.c = static_cast<int>(bc % prm.nc);
  it.b = static_cast<int>(bc / prm.nc);
  return it;
}

__global__ void __launch_bounds__(kThreads, 1)
    chunk_readout_tc_kernel(const __grid_constant__ CUtensorMap tm_C,
                            const __grid_constant__ CUtensorMap tm_h,
                            const __grid_constant__ CUtensorMap tm_z, const RoParams prm) {
  using SM = RoSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ksteps = prm.N / 64;
  auto bar = [&](int i) { return sb + SM::kBars + 8u * i; };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + SM::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kTmemSlot);

  if (threadIdx.x == 0) {
    prefetch_tmap(&tm_C);
    prefetch_tmap(&tm_h);
    prefetch_tmap(&tm_z);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(SM::kFull + i), 1);
      mbar_init(bar(SM::kEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(SM::kAccFull + i), 1);
      mbar_init(bar(SM::kAccEmpty + i), 4);
    }
    mbar_init(bar(SM::kDrain), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{prm.wait_ns, abort_flag, prm.status};
  const int64_t i0 = blockIdx.x, istep = gridDim.x;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool pend[kStages];
      uint32_t ph[kStages];
      for (int s = 0; s < kStages; ++s) pend[s] = false, ph[s] = 0;
      uint32_t gk = 0;
      grid_dep_wait();  // hprev comes from the previous kernel
      for (int64_t i = i0; i < prm.items; i += istep) {
        const RoItem it = ro_item_at(i, prm);
        for (int k = 0; k < ksteps; ++k, ++gk) {
          const int s = static_cast<int>(gk % kStages);
          if (gk >= uint32_t(kStages)) (void)mbar_wait(bar(SM::kEmpty + s), ((gk / kStages) - 1) & 1, ctl);
          if (*abort_flag) continue;
          const uint32_t st = sb + SM::kRing + s * kStage, full = bar(SM::kFull + s);
          mbar_arrive_expect_tx(full, kStage);
          tma_load_3d(st, &tm_C, full, it.g * prm.N + 64 * k, it.c * prm.Q + 128 * it.mt, it.b);
          tma_load_2d(st + kTile, &tm_h, full, 64 * k, ((it.b * prm.nc + it.c) * prm.H + it.h0) * 64);
          pend[s] = true;
          ph[s] = (gk / kStages) & 1;
        }
      }
      for (int s = 0; s < kStages; ++s)
        if (pend[s]) (void)mbar_drain(bar(SM::kFull + s), ph[s], kWaitLimitNs);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------------- MMA issuer
    constexpr uint32_t kIdesc = idesc_bf16_f32(128, 128, 0, 0);
    uint32_t gk = 0, it_local = 0;
    for (int64_t i = i0; i < prm.items; i += istep, ++it_local) {
      const uint32_t a = it_local & 1;
      if (it_local >= 2) (void)mbar_wait(bar(SM::kAccEmpty + a), ((it_local >> 1) - 1) & 1, ctl);
      for (int k = 0; k < ksteps; ++k, ++gk) {
        const int s = static_cast<int>(gk % kStages);
        const bool ok = mbar_wait(bar(SM::kFull + s), (gk / kStages) & 1, ctl) && !*abort_flag;
        if (lane == 0) {
          if (ok) {
            tc_fence_after();
            const uint32_t ca = sb + SM::kRing + s * kStage, ha = ca + kTile;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_f16(tmem + a * 128, sdesc_sw128(ca + kk * 32, 16, 1024), sdesc_sw128(ha + kk * 32, 16, 1024),
                       kIdesc, (k | kk) != 0 ? 1u : 0u);
          }
          umma_commit(bar(SM::kEmpty + s));
        }
        __syncwarp();
      }
      if (lane == 0) umma_commit(bar(SM::kAccFull + a));
      __syncwarp();
    }
    if (lane == 0) {
      umma_commit(bar(SM::kDrain));
      (void)mbar_drain(bar(SM::kDrain), 0, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ------------------ epilogue: Z = 2^{cs2_i} (C hprev^T) -> bf16 -> staging -> TMA store
    const int q4 = warp & 3, r = 32 * q4 + lane;  // TMEM lane quarter; accumulator row = token
    const bool store_thread = warp == kEpiWarp0 && lane == 0;
    uint32_t it_local = 0;
    grid_dep_wait();  // cs2 comes from the earlier kernels; Z overwrites what they read
    for (int64_t i = i0; i < prm.items; i += istep, ++it_local) {
      const RoItem it = ro_item_at(i, prm);
      const uint32_t a = it_local & 1;
      const int row = 128 * it.mt + r;
      float e[2];
#pragma unroll
      for (int k = 0; k < 2; ++k)
        e[k] = k < it.nh ? ex2(__ldg(prm.cs2 + ((int64_t(it.b) * prm.H + it.h0 + k) * prm.nc + it.c) * prm.Q + row))
                         : 0.f;
      const bool ok = mbar_wait(bar(SM::kAccFull + a), (it_local >> 1) & 1, ctl) && !*abort_flag;
      tc_fence_after();
      if (store_thread) bulk_wait_read0();  // the staging buffer is free again
      named_bar_sync(kBarEpi, 128);
      if (ok) {
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {  // 32 columns at a time: head q / 2, p = 32 (q % 2) ..
          uint32_t v[32];
          __syncwarp();
          tmem_ld32(tmem + a * 128 + (uint32_t(32 * q4) << 16) + q * 32, v);
          tmem_ld_wait();
          const float f = e[q >> 1];
          uint8_t* box = smem + SM::kOut + (q >> 1) * kTile + r * 128;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int cc = (q & 1) * 4 + c4;
            uint32_t o[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2)
              o[e2] = pack_bf16x2(f * __uint_as_float(v[8 * c4 + 2 * e2]), f * __uint_as_float(v[8 * c4 + 2 * e2 + 1]));
            *reinterpret_cast<uint4*>(box + ((cc ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(SM::kAccEmpty + a));
      fence_proxy_async_smem();
      named_bar_sync(kBarEpi, 128);
      if (store_thread && ok) {
        for (int k = 0; k < it.nh; ++k)
          tma_store_3d(&tm_z, sb + SM::kOut + k * kTile, (it.h0 + k) * 64, it.c * prm.Q + 128 * it.mt, it.b);
        bulk_commit();
      }
    }
    if (store_thread) bulk_wait_read0();
  }

  grid_dep_launch();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

bool chunk_readout_tc_ok(const Problem& p) {
  return p.io_bf16 && p.P == 64 && (p.Q == 128 || p.Q == 256) && p.N % 64 == 0 && p.N >= 64 &&
         p.L <= (int64_t(1) << 31) - 1 && p.b * p.nc * p.H * p.P < (int64_t(1) << 31) &&
         p.G * p.N < (int64_t(1) << 31);
}

cudaError_t launch_chunk_readout_tc(const Problem& p, const void* C, const float* cs2, const void* hprev,
                                    void* Z, uint32_t* status, cudaStream_t st, const char** why) {
  CUtensorMap tc, th, tz;
  {
    const uint64_t dims[3] = {uint64_t(p.G * p.N), uint64_t(p.L), uint64_t(p.b)};
    const uint64_t strides[2] = {uint64_t(p.G * p.N * 2), uint64_t(p.L * p.G * p.N * 2)};
    const uint32_t box[3] = {64, 128, 1};
    if (!encode_tmap(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, C, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B, why))
      return cudaErrorInvalidValue;
  }
  {
    // hprev (b, nc, H, P, N) as rows (b, c, h, p) of N columns; a box is both heads' 128 rows
    const uint64_t dims[2] = {uint64_t(p.N), uint64_t(p.b * p.nc * p.H * p.P)};
    const uint64_t strides[1] = {uint64_t(p.N * 2)};
    const uint32_t box[2] = {64, 128};
    if (!encode_tmap(&th, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, hprev, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B, why))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {uint64_t(p.H * p.P), uint64_t(p.L), uint64_t(p.b)};
    const uint64_t strides[2] = {uint64_t(p.H * p.P * 2), uint64_t(p.L * p.H * p.P * 2)};
    const uint32_t box[3] = {64, 128, 1};
    if (!encode_tmap(&tz, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, Z, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B, why))
      return cudaErrorInvalidValue;
  }
  RoParams prm;
  prm.L = static_cast<int32_t>(p.L);
  prm.H = static_cast<int32_t>(p.H);
  prm.nc = static_cast<int32_t>(p.nc);
  prm.Q = static_cast<int32_t>(p.Q);
  prm.N = static_cast<int32_t>(p.N);
  prm.hpg = static_cast<int32_t>(p.hpg);
  prm.pairs_per_group = static_cast<int32_t>((p.hpg + 1) / 2);
  prm.MT = static_cast<int32_t>(p.Q / 128);
  prm.items = p.b * p.nc * prm.MT * p.G * prm.pairs_per_group;
  prm.cs2 = cs2;
  prm.status = status;
  prm.wait_ns = kWaitLimitNs;
  auto kern = chunk_readout_tc_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, RoSmem::kAlloc);
  if (e != cudaSuccess) return e;
  int sms = num_sms_current_device();
  if (sms <= 0) sms = 1;
  const int64_t grid = prm.items < sms ? prm.items : sms;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), RoSmem::kAlloc, st, tc, th, tz, prm);
}

}  // namespace ssd
