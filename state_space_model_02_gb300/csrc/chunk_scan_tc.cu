// chunk_scan (compute_out) on the 5th-generation tensor cores -- step 4 of the SSD forward scan.
//
// "Mamba-2 cuda-tile forward pass kernels" (devotd.net), section 2: the third kernel makes the
// token outputs from the chunk-start states, and instead of writing the intermediate matrix to
// global memory it keeps it next to the compute units.  For rows i of a chunk:
//     y[i,p] = sum_{j<=i} 2^{cs2_i - cs2_j} dt_j (C_i . B_j) x[j,p]
//              + 2^{cs2_i} (C_i . hprev[p,:]) + D_h x[i,p]
// Three dense contractions run on tcgen05 with f32 accumulators in tensor memory (TMEM):
//     CB = C_m B^T        (M = 128 rows i, N = j <= 256, K = state N)   once per (b, c, m-tile, group)
//     Y1 = (L o CB) x_h   (M = 128, N = P = 64, K = j)                  per head
//     Y2 = C_m hprev_h^T  (M = 128, N = 64, K = state N)                per head
// CB never leaves TMEM: for every head it is read back into registers, multiplied by the
// decay mask L_ij = 2^{cs2_i - cs2_j} dt_j (j <= i, else 0), rounded to bf16 and written to
// shared memory as Y1's A operand.  The mask is factored per 32-column block j0 as
// 2^{cs2_i - cs2_j0} * (2^{cs2_j0 - cs2_j} dt_j): one exp2 per row per block plus a per-head
// column table, and every factor stays inside float32 range (|cs2| per block <= 32*max(dt|A|)/ln2).
//
// Persistent CTAs (one per SM; 512 TMEM columns and ~210 KB shared memory each) walk a
// contiguous range of (batch, chunk, m-tile, head) units, weighted by the m-tile's causal
// width; CB is recomputed when the range crosses to a new (batch, chunk, m-tile, group).
// Per head, x and hprev arrive by TMA into one of two slots one head ahead, Y1/Y2 alternate
// between two TMEM buffers, and the epilogue of head h-1 overlaps the MMAs of head h.
// Requirements (chunk_scan_tc_ok): bf16 I/O, P = 64, Q in {128, 256}, N in {64, 128}.
#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kThreads = 128;
constexpr uint32_t kBox128 = 16384;  // TMA box: 128 rows x 128 bytes
constexpr uint32_t kBox64 = 8192;    // TMA box: 64 rows x 128 bytes
constexpr uint32_t kTmemCols = 512;  // CB [0,256) | Y1 buf0 | Y2 buf0 | Y1 buf1 | Y2 buf1

struct ScParams {
  int32_t L, H, nc, Q, N, hpg, MT;
  int64_t units, total_weight;
  const float* cs2;
  const float* dtT;
  const float* D;
  const uint16_t* x;
  uint32_t* status;
  uint64_t wait_ns;
};

template <int NB>  // NB = N / 64
struct ScSmem {
  static constexpr uint32_t kC = 0;                          // NB x 16 KB: C rows of the m-tile
  static constexpr uint32_t kP = kC + NB * kBox128;          // 64 KB: L o CB (bf16); B during CB phase
  static constexpr uint32_t kPBytes = 65536;
  static constexpr uint32_t kSlotX = 0;                      // 32 KB: x (up to 256 tokens x 64 p)
  static constexpr uint32_t kSlotH = 32768;                  // NB x 8 KB: hprev (64 p x 64 n)
  static constexpr uint32_t kSlotCs = kSlotH + NB * kBox64;  // 1 KB: cs2 row of the chunk
  static constexpr uint32_t kSlotDt = kSlotCs + 1024;        // 1 KB: dt row of the chunk
  static constexpr uint32_t kSlotBytes = kSlotDt + 1024;
  static constexpr uint32_t kSlot0 = kP + kPBytes;
  static constexpr uint32_t kY = kSlot0 + 2 * kSlotBytes;    // 16 KB: y staging (128 rows x 128 B)
  static constexpr uint32_t kColf = kY + kBox128;            // 1 KB: per-head column factors
  static constexpr uint32_t kBars = kColf + 1024;            // cb_full cb_done slot[2] y[2] drain
  static constexpr uint32_t kTmemSlot = kBars + 8 * 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kUsed = kAbort + 4;
  static constexpr uint32_t kAlloc = kUsed + 1024;           // slack for 1024-byte alignment
  static_assert(kSlotBytes % 1024 == 0, "slots must stay 1024-byte aligned");
  static_assert(kAlloc <= 232448, "exceeds the per-CTA shared memory limit");
};

// First unit whose starting weight is >= w.  Units are ordered (b, c, m-tile, h); a unit of
// m-tile mt has weight mt + 1 (its causal width in 128-column blocks).
__device__ __forceinline__ int64_t unit_at_weight(int64_t w, int32_t H, int32_t MT) {
  if (MT == 1) return w;
  const int64_t wbc = 3 * int64_t(H);
  const int64_t bc = w / wbc, rem = w % wbc;
  if (rem < H) return bc * 2 * H + rem;
  const int64_t h = (rem - H + 1) / 2;
  return h >= H ? (bc + 1) * 2 * H : bc * 2 * H + H + h;
}

template <int NB>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                         const __grid_constant__ CUtensorMap tm_B,
                         const __grid_constant__ CUtensorMap tm_C,
                         const __grid_constant__ CUtensorMap tm_h,
                         const __grid_constant__ CUtensorMap tm_y, const ScParams prm) {
  using SM = ScSmem<NB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int32_t H = prm.H, Q = prm.Q, N = prm.N, MT = prm.MT;

  const uint32_t bar_cb_full = sb + SM::kBars, bar_cb_done = bar_cb_full + 8,
                 bar_slot = bar_cb_full + 16, bar_y = bar_cb_full + 32, bar_drain = bar_cb_full + 48;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + SM::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kTmemSlot);
  float* colf = reinterpret_cast<float*>(smem + SM::kColf);

  if (tid == 0) {
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_B);
    prefetch_tmap(&tm_C);
    prefetch_tmap(&tm_h);
    prefetch_tmap(&tm_y);
    for (int i = 0; i < 7; ++i) mbar_init(bar_cb_full + 8 * i, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_row = tmem + (uint32_t(warp * 32) << 16);
  const WaitCtl ctl{prm.wait_ns, abort_flag, prm.status};

  const int64_t u_begin = unit_at_weight(prm.total_weight * blockIdx.x / gridDim.x, H, MT);
  const int64_t u_end = unit_at_weight(prm.total_weight * (blockIdx.x + 1) / gridDim.x, H, MT);

  // thread-0 bookkeeping of TMA loads in flight, for the drain on abort
  bool pend_cb = false, pend_slot[2] = {false, false};
  uint32_t pend_cb_ph = 0, pend_slot_ph[2] = {0, 0};

  uint32_t gi = 0, cb_phase = 0;
  float e_keep = 0.f;

  for (int64_t u = u_begin; u < u_end;) {
    const int64_t bcm = u / H;
    const int h_begin = static_cast<int>(u % H);
    const int mt = static_cast<int>(bcm % MT);
    const int64_t bc = bcm / MT;
    const int c = static_cast<int>(bc % prm.nc), b = static_cast<int>(bc / prm.nc);
    const int g = h_begin / prm.hpg;
    const int h_end = static_cast<int>(min(int64_t((g + 1) * prm.hpg), h_begin + (u_end - u)));
    const int nh = h_end - h_begin;
    const int i0 = mt * 128, jrows = i0 + 128;
    const int row = i0 + tid;                 // row of the chunk owned by this thread
    const int nblk = jrows / 32, maxblk = i0 / 32 + warp;
    const bool tile_live = int64_t(c) * Q + i0 < prm.L;  // any row of the m-tile inside [0, L)

    auto load_head = [&](int hh, uint32_t k) {  // thread 0: x, hprev, cs2, dt of head hh -> slot
      const uint32_t s = k & 1, ph = (k >> 1) & 1;
      const uint32_t slot = sb + SM::kSlot0 + s * SM::kSlotBytes;
      const uint32_t bar = bar_slot + 8 * s;
      mbar_arrive_expect_tx(bar, jrows * 128 + NB * kBox64 + 2 * jrows * 4);
      for (int jb = 0; jb < jrows / 128; ++jb)
        tma_load_3d(slot + SM::kSlotX + jb * kBox128, &tm_x, bar, hh * 64, c * Q + jb * 128, b);
      for (int nb = 0; nb < NB; ++nb)
        tma_load_2d(slot + SM::kSlotH + nb * kBox64, &tm_h, bar, nb * 64,
                    ((b * prm.nc + c) * H + hh) * 64);
      const int64_t crow = ((int64_t(b) * H + hh) * prm.nc + c) * Q;
      bulk_load(slot + SM::kSlotCs, prm.cs2 + crow, jrows * 4, bar);
      bulk_load(slot + SM::kSlotDt, prm.dtT + crow, jrows * 4, bar);
      pend_slot[s] = true;
      pend_slot_ph[s] = ph;
    };

    // epilogue of head hh whose Y1/Y2 sit in TMEM buffer yb: y = Y1 + e*Y2 + D*x -> TMA store
    auto epilogue = [&](int hh, uint32_t yb, float e) {
      const int64_t t = int64_t(c) * Q + row;
      const float Dh = prm.D ? __ldg(prm.D + hh) : 0.f;
      uint4 xr[8];
      if (t < prm.L) {
        const uint4* xp = reinterpret_cast<const uint4*>(prm.x + ((int64_t(b) * prm.L + t) * H + hh) * 64);
#pragma unroll
        for (int k = 0; k < 8; ++k) xr[k] = __ldg(xp + k);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) xr[k] = make_uint4(0, 0, 0, 0);
      }
      uint8_t* ys = smem + SM::kY + tid * 128;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t a[32], q2[32];
        __syncwarp();
        tmem_ld32(tmem_row + 256 + 128 * yb + 32 * half, a);
        tmem_ld32(tmem_row + 256 + 128 * yb + 64 + 32 * half, q2);
        tmem_ld_wait();
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const uint4 xw = xr[4 * half + qq];
          const uint32_t xs[4] = {xw.x, xw.y, xw.z, xw.w};
          uint32_t o[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const int k0 = 8 * qq + 2 * e2;
            const float lo = __uint_as_float(a[k0]) + e * __uint_as_float(q2[k0]) + Dh * bf16lo_to_f32(xs[e2]);
            const float hi = __uint_as_float(a[k0 + 1]) + e * __uint_as_float(q2[k0 + 1]) +
                             Dh * bf16hi_to_f32(xs[e2]);
            o[e2] = pack_bf16x2(lo, hi);
          }
          *reinterpret_cast<uint4*>(ys + (((4 * half + qq) ^ (tid & 7)) << 4)) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0 && tile_live && !*abort_flag) {
        tma_store_3d(&tm_y, sb + SM::kY, hh * 64, c * Q + i0, b);
        bulk_commit();
      }
    };

    // ---- segment start: operands of CB and the first two heads
    if (tid == 0 && !*abort_flag) {
      mbar_arrive_expect_tx(bar_cb_full, NB * kBox128 + NB * jrows * 128);
      for (int nb = 0; nb < NB; ++nb)
        tma_load_3d(sb + SM::kC + nb * kBox128, &tm_C, bar_cb_full, g * N + nb * 64, c * Q + i0, b);
      for (int nb = 0; nb < NB; ++nb)
        for (int jb = 0; jb < jrows / 128; ++jb)
          tma_load_3d(sb + SM::kP + nb * jrows * 128 + jb * kBox128, &tm_B, bar_cb_full,
                      g * N + nb * 64, c * Q + jb * 128, b);
      pend_cb = true;
      pend_cb_ph = cb_phase;
      for (int k = 0; k < 2 && k < nh; ++k) load_head(h_begin + k, gi + k);
    }
    if (tid == 0) {
      if (mbar_wait(bar_cb_full, cb_phase, ctl)) {
        pend_cb = false;
        if (!*abort_flag) {
          tc_fence_after();
          const uint32_t idesc = idesc_bf16_f32(128, jrows, 0, 0);
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_f16(tmem, sdesc_sw128(sb + SM::kC + nb * kBox128 + k * 32, 16, 1024),
                       sdesc_sw128(sb + SM::kP + nb * jrows * 128 + k * 32, 16, 1024), idesc,
                       (nb | k) != 0 ? 1u : 0u);
        }
      }
      umma_commit(bar_cb_done);
    }
    (void)mbar_wait(bar_cb_done, cb_phase, ctl);
    cb_phase ^= 1u;
    tc_fence_after();
    // blocks of P right of this warp's diagonal block stay zero for the whole segment
    for (int blk = maxblk + 1; blk < nblk; ++blk) {
      const int j0 = 32 * blk;
      uint8_t* pb = smem + SM::kP + (j0 >> 6) * kBox128 + tid * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(pb + (((((j0 & 63) >> 3) + q) ^ (tid & 7)) << 4)) = make_uint4(0, 0, 0, 0);
    }

    for (int hi = 0; hi < nh; ++hi, ++gi) {
      const int h = h_begin + hi;
      const uint32_t s = gi & 1, sph = (gi >> 1) & 1;
      uint8_t* slotp = smem + SM::kSlot0 + s * SM::kSlotBytes;
      const uint32_t slot = sb + SM::kSlot0 + s * SM::kSlotBytes;
      if (hi >= 1) {
        // MMAs of the previous head are done: its slot, the P tile and its TMEM buffer are free
        const uint32_t pg = gi - 1;
        (void)mbar_wait(bar_y + 8 * (pg & 1), (pg >> 1) & 1, ctl);
        tc_fence_after();
        if (tid == 0 && hi + 1 < nh && !*abort_flag) load_head(h + 1, gi + 1);
      }
      const bool have = mbar_wait(bar_slot + 8 * s, sph, ctl);
      if (tid == 0 && have) pend_slot[s] = false;
      const float* cs = reinterpret_cast<const float*>(slotp + SM::kSlotCs);
      const float* dtv = reinterpret_cast<const float*>(slotp + SM::kSlotDt);
      for (int j = tid; j < jrows; j += kThreads) colf[j] = ex2(cs[j & ~31] - cs[j]) * dtv[j];
      const float cs_i = cs[row];
      __syncthreads();
      if (tid == 0 && !*abort_flag) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_f16(tmem + 256 + 128 * s + 64, sdesc_sw128(sb + SM::kC + nb * kBox128 + k * 32, 16, 1024),
                     sdesc_sw128(slot + SM::kSlotH + nb * kBox64 + k * 32, 16, 1024), idesc,
                     (nb | k) != 0 ? 1u : 0u);
      }
      // L o CB for this head -> P (bf16, K-major, 128-byte swizzle)
      for (int blk = 0; blk <= maxblk && blk < nblk; ++blk) {
        uint32_t v[32];
        __syncwarp();
        tmem_ld32(tmem_row + 32 * blk, v);
        tmem_ld_wait();
        const int j0 = 32 * blk;
        const float rowf = ex2(cs_i - cs[j0]);
        const bool diag = blk == maxblk;
        uint8_t* pb = smem + SM::kP + (j0 >> 6) * kBox128 + tid * 128;
        const int cbase = (j0 & 63) >> 3;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t o[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const int k0 = 8 * q + 2 * e2;
            float lo = __uint_as_float(v[k0]) * colf[j0 + k0] * rowf;
            float hi = __uint_as_float(v[k0 + 1]) * colf[j0 + k0 + 1] * rowf;
            if (diag && j0 + k0 > row) lo = 0.f;
            if (diag && j0 + k0 + 1 > row) hi = 0.f;
            o[e2] = pack_bf16x2(lo, hi);
          }
          *reinterpret_cast<uint4*>(pb + (((cbase + q) ^ (tid & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      if (tid == 0) bulk_wait_read0();  // the y staging buffer is free for the epilogue below
      __syncthreads();
      if (tid == 0) {
        if (!*abort_flag) {
          tc_fence_after();
          const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 1);
          for (int k = 0; k < jrows / 16; ++k)
            umma_f16(tmem + 256 + 128 * s, sdesc_sw128(sb + SM::kP + (k >> 2) * kBox128 + (k & 3) * 32, 16, 1024),
                     sdesc_sw128(slot + SM::kSlotX + k * 2048, kBox128, 1024), idesc, k != 0 ? 1u : 0u);
        }
        umma_commit(bar_y + 8 * s);
      }
      const float e_cur = ex2(cs_i);
      if (hi >= 1) epilogue(h - 1, (gi - 1) & 1, e_keep);
      e_keep = e_cur;
    }
    // drain the segment: last head's epilogue
    {
      const uint32_t lg = gi - 1;
      (void)mbar_wait(bar_y + 8 * (lg & 1), (lg >> 1) & 1, ctl);
      tc_fence_after();
      if (tid == 0) bulk_wait_read0();
      __syncthreads();
      epilogue(h_end - 1, lg & 1, e_keep);
    }
    u += nh;
  }

  // teardown: drain whatever is still in flight, then release tensor memory
  if (tid == 0) {
    if (pend_cb) (void)mbar_drain(bar_cb_full, pend_cb_ph, kWaitLimitNs);
    for (int s = 0; s < 2; ++s)
      if (pend_slot[s]) (void)mbar_drain(bar_slot + 8 * s, pend_slot_ph[s], kWaitLimitNs);
    umma_commit(bar_drain);
    (void)mbar_drain(bar_drain, 0, kWaitLimitNs);
    bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NB>
cudaError_t launch_nb(const CUtensorMap* maps, const ScParams& prm, int grid, cudaStream_t st) {
  using SM = ScSmem<NB>;
  auto kern = chunk_scan_tc_kernel<NB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kAlloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, SM::kAlloc, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], prm);
  return cudaGetLastError();
}

}  // namespace

bool chunk_scan_tc_ok(const Problem& p) {
  return p.io_bf16 && p.P == 64 && (p.Q == 128 || p.Q == 256) && (p.N == 64 || p.N == 128) &&
         p.L <= (int64_t(1) << 31) - 1 && p.b * p.nc * p.H * p.P < (int64_t(1) << 31) &&
         p.G * p.N < (int64_t(1) << 31);
}

cudaError_t launch_chunk_scan_tc(const Problem& p, const void* x, const void* B, const void* C,
                                 const float* D, const float* cs2, const float* dtT,
                                 const void* hprev, void* y, uint32_t* status, cudaStream_t st,
                                 const char** why) {
  CUtensorMap maps[5];  // x, B, C, hprev, y
  const uint64_t xdims[3] = {uint64_t(p.H * p.P), uint64_t(p.L), uint64_t(p.b)};
  const uint64_t xstr[2] = {uint64_t(p.H * p.P * 2), uint64_t(p.L * p.H * p.P * 2)};
  const uint64_t bdims[3] = {uint64_t(p.G * p.N), uint64_t(p.L), uint64_t(p.b)};
  const uint64_t bstr[2] = {uint64_t(p.G * p.N * 2), uint64_t(p.L * p.G * p.N * 2)};
  const uint32_t box3[3] = {64, 128, 1};
  const uint64_t hdims[2] = {uint64_t(p.N), uint64_t(p.b * p.nc * p.H * p.P)};
  const uint64_t hstr[1] = {uint64_t(p.N * 2)};
  const uint32_t hbox[2] = {64, 64};
  if (!encode_tmap(&maps[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, xdims, xstr, box3,
                   CU_TENSOR_MAP_SWIZZLE_128B, why) ||
      !encode_tmap(&maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, B, bdims, bstr, box3,
                   CU_TENSOR_MAP_SWIZZLE_128B, why) ||
      !encode_tmap(&maps[2], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, C, bdims, bstr, box3,
                   CU_TENSOR_MAP_SWIZZLE_128B, why) ||
      !encode_tmap(&maps[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, hprev, hdims, hstr, hbox,
                   CU_TENSOR_MAP_SWIZZLE_128B, why) ||
      !encode_tmap(&maps[4], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, y, xdims, xstr, box3,
                   CU_TENSOR_MAP_SWIZZLE_128B, why))
    return cudaErrorInvalidValue;
  ScParams prm;
  prm.L = static_cast<int32_t>(p.L);
  prm.H = static_cast<int32_t>(p.H);
  prm.nc = static_cast<int32_t>(p.nc);
  prm.Q = static_cast<int32_t>(p.Q);
  prm.N = static_cast<int32_t>(p.N);
  prm.hpg = static_cast<int32_t>(p.hpg);
  prm.MT = static_cast<int32_t>(p.Q / 128);
  prm.units = p.b * p.nc * prm.MT * p.H;
  prm.total_weight = p.b * p.nc * p.H * (prm.MT == 2 ? 3 : 1);
  prm.cs2 = cs2;
  prm.dtT = dtT;
  prm.D = D;
  prm.x = static_cast<const uint16_t*>(x);
  prm.status = status;
  prm.wait_ns = kWaitLimitNs;
  int sms = num_sms_current_device();
  if (sms <= 0) sms = 1;
  const int grid = static_cast<int>(prm.units < sms ? prm.units : sms);
  if (p.N == 64) return launch_nb<1>(maps, prm, grid, st);
  return launch_nb<2>(maps, prm, grid, st);
}

}  // namespace ssd
