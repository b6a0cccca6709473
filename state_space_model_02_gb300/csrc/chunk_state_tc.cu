// chunk_state on the 5th-generation tensor cores (tcgen05) -- step 2 of the SSD forward scan.
//
// "Mamba-2 cuda-tile forward pass kernels" (devotd.net), section 1: each chunk's work is
// turned into matrix products for the Tensor Cores; section 2 (fwd_pass_state): the state a
// chunk contributes, before chaining across chunks, is
//     S[b,c,h][p,n] = sum_t x~[t,(h,p)] * B[t,n],   x~[t,(h,p)] = 2^{cs2_last - cs2_t} dt_t x[t,h,p]
// a contraction over the chunk's Q tokens.  Section 3 swaps MMA operands to suit the 5th-gen
// Tensor Core operand layout; here two heads are stacked on the MMA M axis (M = 2 x P = 128,
// x is (token, head, p) so two neighbouring heads are one contiguous 128-wide row) and the
// state dimension is the N axis, so both operands come straight from TMA in MN-major
// 128-byte-swizzled form with no transposition.
//
// Persistent CTAs (one per SM) walk the work items (head pair, n-tile, chunk, batch) with a
// stride of the grid size, so the CTAs running at one time share a chunk's B through L2.  Warp
// roles, synchronised through mbarriers so that one item's epilogue overlaps the next items'
// loads and MMAs:
//   warp 0      TMA producer: per 64-token k-block one box of both heads' x and one of B's NT
//               columns into a ring of kStages stages that runs on across items; per item the
//               two heads' cs2 / dt rows (bulk copies) into one of two weight windows;
//   warp 1      tcgen05.mma issuer: per k-block 4 MMAs (M = 2 x P = 128, N = NT, K = 16) into
//               one of two TMEM accumulators (the item's parity);
//   warps 2-9   the decay weights w_t = 2^{cs2_last - cs2_t} dt_t of each item, then x~ = w x
//               in place in every stage (one weight per 128-byte row, so the swizzle does not
//               matter);
//   warps 10-13 epilogue: accumulator -> bf16 -> swizzled staging -> TMA store of S.
// The scaling of a k-block stands between its load and its MMAs, so eight warps share it (four
// 16-byte chunks a thread): against four warps (eight chunks a thread) that took chunk_state
// from 313 to 284 us at 256K tokens; sixteen warps measured 290 us.
// Every wait is bounded; after an expiry the roles keep their loop counts but skip their work,
// then drain their own copies and MMAs and release TMEM.
// Requirements (checked by chunk_state_tc_ok): bf16 I/O, P = 64, Q in {128, 256},
// N in {64, 128, 256, 512} (512 runs as two 256-wide n-tiles).
#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kWarps = 14;
constexpr int kThreads = 32 * kWarps;
constexpr int kScaleWarp0 = 2, kEpiWarp0 = 10;
constexpr uint32_t kBox = 8192;  // one TMA box: 64 rows x 128 bytes
constexpr uint32_t kBarScale = 1, kBarEpi = 2;  // named barriers of the scale and epilogue groups

struct CsParams {
  int32_t L, H, nc, Q, N, hpg, pairs_per_group, n_tiles;
  int64_t items;
  int64_t chains;            // fused kernel: (batch, head pair, n-tile) chains, each nc items
  const float* cs2;
  const float* dtT;
  const float* init;         // fused kernel: state before the first chunk (b, H, P, N), or null
  float* final_state;        // fused kernel: state after the last chunk (b, H, P, N), or null
  uint32_t* status;
  uint64_t wait_ns;
};

template <int NT>
struct CsSmem {
  static constexpr uint32_t kX = 2 * kBox;                  // x: two heads x (64 tokens x 64 p)
  static constexpr uint32_t kB = (NT / 64) * kBox;          // B: NT/64 boxes of (64 tokens x 64 n)
  static constexpr uint32_t kStage = kX + kB;
  static constexpr int kStages = NT == 256 ? 3 : (NT == 128 ? 5 : 6);
  static constexpr uint32_t kOut = kStages * kStage;        // S staging: NT/64 x 2 boxes
  static constexpr uint32_t kWin = kOut + 2 * (NT / 64) * kBox;  // 2 windows: cs2, dt rows of 2 heads
  static constexpr uint32_t kWinBytes = 4 * 256 * 4;
  static constexpr uint32_t kW = kWin + 2 * kWinBytes;      // 2 x float w[2][256]
  static constexpr uint32_t kBars = kW + 2 * 2048;
  static constexpr int kNumBars = 3 * kStages + 9;
  static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kUsed = kAbort + 4;
  static constexpr uint32_t kAlloc = kUsed + 1024;          // slack for 1024-byte alignment
  static_assert(kAlloc <= 232448, "exceeds the per-CTA shared memory limit");
  // mbarrier indices
  static constexpr int kFull = 0, kScaled = kStages, kEmpty = 2 * kStages, kWinFull = 3 * kStages,
                       kWinEmpty = kWinFull + 2, kAccFull = kWinEmpty + 2, kAccEmpty = kAccFull + 2,
                       kDrain = kAccEmpty + 2;
};

// One work item: (head pair, n-tile) fastest, then chunk, then batch.
struct Item {
  int b, c, g, h0, nh, nt;
};
__device__ __forceinline__ Item item_at(int64_t i, const CsParams& prm) {
  Item it;
  const int64_t per_c = int64_t(prm.H / prm.hpg) * prm.pairs_per_group * prm.n_tiles;
  const int64_t bc = i / per_c;
  const int rem = static_cast<int>(i - bc * per_c);
  it.nt = rem % prm.n_tiles;
  const int pair = rem / prm.n_tiles;
  it.g = pair / prm.pairs_per_group;
  it.h0 = it.g * prm.hpg + 2 * (pair % prm.pairs_per_group);
  it.nh = min(2, (it.g + 1) * prm.hpg - it.h0);  // 1 when the group has an odd head count
  it.c = static_cast<int>(bc % prm.nc);
  it.b = static_cast<int>(bc / prm.nc);
  return it;
}

// Chunk c of chain ch; chains run (n-tile fastest, head pair, batch).
__device__ __forceinline__ Item chain_item(int64_t ch, int c, const CsParams& prm) {
  Item it;
  const int64_t per_b = int64_t(prm.H / prm.hpg) * prm.pairs_per_group * prm.n_tiles;
  const int64_t b = ch / per_b;
  const int rem = static_cast<int>(ch - b * per_b);
  it.nt = rem % prm.n_tiles;
  const int pair = rem / prm.n_tiles;
  it.g = pair / prm.pairs_per_group;
  it.h0 = it.g * prm.hpg + 2 * (pair % prm.pairs_per_group);
  it.nh = min(2, (it.g + 1) * prm.hpg - it.h0);
  it.c = c;
  it.b = static_cast<int>(b);
  return it;
}

// The CTA's j-th work item; false past its last.  Separate kernels: items i = blockIdx.x +
// j * gridDim.x.  Fused: chains ch = blockIdx.x + (j / nc) * gridDim.x, each walked through its
// chunks in order (c = j % nc), so the chain's state can be carried from one item to the next.
template <bool FUSED>
__device__ __forceinline__ bool local_item(uint32_t j, const CsParams& prm, Item& it) {
  if (!FUSED) {
    const int64_t i = blockIdx.x + int64_t(j) * gridDim.x;
    if (i >= prm.items) return false;
    it = item_at(i, prm);
    return true;
  }
  const uint32_t nc = static_cast<uint32_t>(prm.nc);
  const int64_t ch = blockIdx.x + int64_t(j / nc) * gridDim.x;
  if (ch >= prm.chains) return false;
  it = chain_item(ch, static_cast<int>(j % nc), prm);
  return true;
}

// x~ = w x on a packed bf16 pair: w is rounded to bf16 too (one more rounding of the same size
// as the product's), so the pair takes one bf16x2 multiply instead of an unpack, two float
// multiplies and a repack -- the scaling pass sits between every k-block's load and its MMAs.
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t v, uint32_t w2) { return mul_bf16x2(v, w2); }

// FUSED: fwd_pass_state in one kernel -- instead of storing S, the epilogue carries each chain's
// float32 state in tensor memory (h <- 2^{cs2_last} h + S_c, chunk by chunk), stores the state
// entering every chunk as hprev (bf16, through tm_S, which then maps hprev) and the state after
// the last chunk as final_state.
template <int NT, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_state_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                          const __grid_constant__ CUtensorMap tm_B,
                          const __grid_constant__ CUtensorMap tm_S, const CsParams prm) {
  using SM = CsSmem<NT>;
  constexpr int S = SM::kStages;
  // two accumulators, and for the fused kernel the chain's state after them
  constexpr uint32_t kCols = FUSED ? 4 * NT : 2 * NT;
  static_assert(!FUSED || NT <= 128, "the fused kernel keeps three NT-column regions in tensor memory");
  extern __shared__ uint8_t smem_raw[];
  // align by pointer arithmetic on the __shared__ array so accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Q = prm.Q, kblocks = Q / 64;
  auto bar = [&](int i) { return sb + SM::kBars + 8u * i; };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + SM::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kTmemSlot);

  if (threadIdx.x == 0) {
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_B);
    prefetch_tmap(&tm_S);
    for (int i = 0; i < S; ++i) {
      mbar_init(bar(SM::kFull + i), 1);
      mbar_init(bar(SM::kScaled + i), 8);
      mbar_init(bar(SM::kEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(SM::kWinFull + i), 1);
      mbar_init(bar(SM::kWinEmpty + i), 8);
      mbar_init(bar(SM::kAccFull + i), 1);
      mbar_init(bar(SM::kAccEmpty + i), 4);
    }
    mbar_init(bar(SM::kDrain), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{prm.wait_ns, abort_flag, prm.status};

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool pend_full[S], pend_win[2] = {false, false};
      uint32_t ph_full[S], ph_win[2] = {0, 0};
      for (int i = 0; i < S; ++i) pend_full[i] = false, ph_full[i] = 0;
      uint32_t gk = 0, it_local = 0;
      // x and B are inputs of the step: the first item's k-blocks are requested before waiting
      // for the previous kernel (cs2 / dtT come from it)
      Item it0;
      const int pre = local_item<FUSED>(0, prm, it0) ? (kblocks < S ? kblocks : S) : 0;
      auto load_kb = [&](const Item& it, int kb, uint32_t k) {
        const int s = static_cast<int>(k % S);
        const uint32_t st = sb + s * SM::kStage, full = bar(SM::kFull + s);
        const int t0 = it.c * Q + kb * 64;
        mbar_arrive_expect_tx(full, SM::kStage);
        tma_load_4d(st, &tm_x, full, 0, t0, it.h0, it.b);
        tma_load_4d(st + SM::kX, &tm_B, full, 0, t0, (it.g * prm.N + it.nt * NT) / 64, it.b);
        pend_full[s] = true;
        ph_full[s] = (k / S) & 1;
      };
      for (int kb = 0; kb < pre; ++kb) load_kb(it0, kb, uint32_t(kb));
      grid_dep_wait();
      for (;; ++it_local) {
        Item it;
        if (!local_item<FUSED>(it_local, prm, it)) break;
        const uint32_t ws = it_local & 1;
        if (it_local >= 2) (void)mbar_wait(bar(SM::kWinEmpty + ws), ((it_local >> 1) - 1) & 1, ctl);
        if (!*abort_flag) {
          const uint32_t win = sb + SM::kWin + ws * SM::kWinBytes, wf = bar(SM::kWinFull + ws);
          mbar_arrive_expect_tx(wf, it.nh * 2 * Q * 4);
          for (int k = 0; k < it.nh; ++k) {
            const int64_t row = ((int64_t(it.b) * prm.H + it.h0 + k) * prm.nc + it.c) * Q;
            bulk_load(win + k * 1024, prm.cs2 + row, Q * 4, wf);
            bulk_load(win + 2048 + k * 1024, prm.dtT + row, Q * 4, wf);
          }
          pend_win[ws] = true;
          ph_win[ws] = (it_local >> 1) & 1;
        }
        for (int kb = 0; kb < kblocks; ++kb, ++gk) {
          if (it_local == 0 && kb < pre) continue;  // requested before the wait
          const int s = static_cast<int>(gk % S);
          if (gk >= uint32_t(S)) (void)mbar_wait(bar(SM::kEmpty + s), ((gk / S) - 1) & 1, ctl);
          if (!*abort_flag) load_kb(it, kb, gk);
        }
      }
      // drain: every load issued must have landed before the CTA may exit
      for (int s = 0; s < S; ++s)
        if (pend_full[s]) (void)mbar_drain(bar(SM::kFull + s), ph_full[s], kWaitLimitNs);
      for (int w = 0; w < 2; ++w)
        if (pend_win[w]) (void)mbar_drain(bar(SM::kWinFull + w), ph_win[w], kWaitLimitNs);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------------- MMA issuer
    constexpr uint32_t kIdesc = idesc_bf16_f32(128, NT, 1, 1);
    uint32_t gk = 0, it_local = 0;
    for (;; ++it_local) {
      Item it;
      if (!local_item<FUSED>(it_local, prm, it)) break;
      const uint32_t a = it_local & 1;
      if (it_local >= 2) (void)mbar_wait(bar(SM::kAccEmpty + a), ((it_local >> 1) - 1) & 1, ctl);
      for (int kb = 0; kb < kblocks; ++kb, ++gk) {
        const int s = static_cast<int>(gk % S);
        const bool ok = mbar_wait(bar(SM::kScaled + s), (gk / S) & 1, ctl) && !*abort_flag;
        if (lane == 0) {
          if (ok) {
            tc_fence_after();
            const uint32_t xa = sb + s * SM::kStage, ba = xa + SM::kX;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_f16(tmem + a * NT, sdesc_sw128(xa + k * 2048, kBox, 1024),
                       sdesc_sw128(ba + k * 2048, kBox, 1024), kIdesc, (kb | k) != 0 ? 1u : 0u);
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
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------- decay weights, x~ = w x in place
    const int ts = threadIdx.x - 32 * kScaleWarp0;  // 0..255
    uint32_t gk = 0, it_local = 0;
    for (;; ++it_local) {
      Item it;
      if (!local_item<FUSED>(it_local, prm, it)) break;
      const uint32_t ws = it_local & 1;
      const bool have = mbar_wait(bar(SM::kWinFull + ws), (it_local >> 1) & 1, ctl);
      const float* win = reinterpret_cast<const float*>(smem + SM::kWin + ws * SM::kWinBytes);
      float* wsm = reinterpret_cast<float*>(smem + SM::kW + ws * 2048);
      for (int e = ts; e < 2 * Q; e += 256) {
        const int k = e / Q, t = e % Q;
        // w[k][t] = 2^(cs2_last - cs2_t) dt_t; zero for a missing second head
        wsm[k * 256 + t] = have && k < it.nh ? ex2(win[k * 256 + Q - 1] - win[k * 256 + t]) * win[512 + k * 256 + t] : 0.f;
      }
      named_bar_sync(kBarScale, 256);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(SM::kWinEmpty + ws));
      for (int kb = 0; kb < kblocks; ++kb, ++gk) {
        const int s = static_cast<int>(gk % S);
        const bool ok = mbar_wait(bar(SM::kFull + s), (gk / S) & 1, ctl) && !*abort_flag;
        if (ok) {
          // 1024 16-byte chunks (two boxes x 64 rows x 8), 4 per thread
          uint8_t* xs = smem + s * SM::kStage;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int q = ts + 256 * j;
            const int k = q >> 9, r = (q >> 3) & 63;
            const float w = wsm[k * 256 + kb * 64 + r];
            const uint32_t w2 = pack_bf16x2(w, w);
            uint4* pch = reinterpret_cast<uint4*>(xs + q * 16);
            uint4 v = *pch;
            v.x = scale_bf16x2(v.x, w2);
            v.y = scale_bf16x2(v.y, w2);
            v.z = scale_bf16x2(v.z, w2);
            v.w = scale_bf16x2(v.w, w2);
            *pch = v;
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(SM::kScaled + s));
      }
    }
  } else if (FUSED) {
    // ------------- epilogue (fused): hprev = h, then h <- 2^{cs2_last} h + S, chunk by chunk
    const int q4 = warp & 3, r = 32 * q4 + lane;  // TMEM lane quarter; accumulator row = (head, p)
    const int k = r >> 6, pr = r & 63;
    const bool store_thread = warp == kEpiWarp0 && lane == 0;
    const uint32_t hcol = tmem + 2 * NT + (uint32_t(32 * q4) << 16);  // this warp's rows of h
    grid_dep_wait();  // cs2 comes from the previous kernel; hprev may still be read by older ones
    for (uint32_t it_local = 0;; ++it_local) {
      Item it;
      if (!local_item<FUSED>(it_local, prm, it)) break;
      const uint32_t a = it_local & 1;
      const bool row_ok = k < it.nh;
      const int64_t bh = int64_t(it.b) * prm.H + it.h0 + k;  // (batch, head) of this row
      // the chunk's decay, requested before the accumulator wait so that its latency hides
      const float dec = row_ok ? ex2(__ldg(prm.cs2 + (bh * prm.nc + it.c) * Q + Q - 1)) : 0.f;
      const bool ok = mbar_wait(bar(SM::kAccFull + a), (it_local >> 1) & 1, ctl) && !*abort_flag;
      tc_fence_after();
      if (store_thread) bulk_wait_read0();  // the staging buffer is free again
      named_bar_sync(kBarEpi, 128);
      if (ok) {
        const int64_t row = (bh * 64 + pr) * prm.N + it.nt * NT;  // (b, h, p, n-tile) in init / final
        const float* init_row = it.c == 0 && row_ok && prm.init ? prm.init + row : nullptr;
        float* fin_row = it.c == prm.nc - 1 && row_ok && prm.final_state ? prm.final_state + row : nullptr;
#pragma unroll 1
        for (int q = 0; q < NT / 32; ++q) {
          uint32_t sv[32], hv[32];
          __syncwarp();
          tmem_ld32(tmem + a * NT + (uint32_t(32 * q4) << 16) + q * 32, sv);
          if (it.c > 0) tmem_ld32(hcol + q * 32, hv);  // it.c is uniform over the warp
          tmem_ld_wait();
          if (it.c == 0) {  // the chain starts from init (zero without one)
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 f = init_row ? __ldg(reinterpret_cast<const float4*>(init_row + q * 32 + j))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
              hv[j] = __float_as_uint(f.x);
              hv[j + 1] = __float_as_uint(f.y);
              hv[j + 2] = __float_as_uint(f.z);
              hv[j + 3] = __float_as_uint(f.w);
            }
          }
          // hprev of this chunk (the state entering it) in bf16 into the staging box
          uint8_t* box = smem + SM::kOut + ((q >> 1) * 2 + k) * kBox;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int cc = (q & 1) * 4 + c4;
            *reinterpret_cast<uint4*>(box + pr * 128 + ((cc ^ (pr & 7)) << 4)) =
                make_uint4(pack_bf16x2(__uint_as_float(hv[8 * c4]), __uint_as_float(hv[8 * c4 + 1])),
                           pack_bf16x2(__uint_as_float(hv[8 * c4 + 2]), __uint_as_float(hv[8 * c4 + 3])),
                           pack_bf16x2(__uint_as_float(hv[8 * c4 + 4]), __uint_as_float(hv[8 * c4 + 5])),
                           pack_bf16x2(__uint_as_float(hv[8 * c4 + 6]), __uint_as_float(hv[8 * c4 + 7])));
          }
#pragma unroll
          for (int j = 0; j < 32; ++j)
            hv[j] = __float_as_uint(fmaf(dec, __uint_as_float(hv[j]), __uint_as_float(sv[j])));
          tmem_st32(hcol + q * 32, hv);
          if (fin_row) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(fin_row + q * 32 + j) =
                  make_float4(__uint_as_float(hv[j]), __uint_as_float(hv[j + 1]), __uint_as_float(hv[j + 2]),
                              __uint_as_float(hv[j + 3]));
          }
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(SM::kAccEmpty + a));
      fence_proxy_async_smem();
      named_bar_sync(kBarEpi, 128);
      if (store_thread && ok) {
        for (int j = 0; j < NT / 64; ++j)
          for (int kk = 0; kk < it.nh; ++kk)
            tma_store_2d(&tm_S, sb + SM::kOut + (j * 2 + kk) * kBox, it.nt * NT + j * 64,
                         ((it.b * prm.nc + it.c) * prm.H + it.h0 + kk) * 64);
        bulk_commit();
      }
    }
    if (store_thread) bulk_wait_read0();  // the stores have read the staging buffer
  } else {
    // --------------------------------- epilogue: accumulator -> bf16 -> TMA store of S
    const int q4 = warp & 3, r = 32 * q4 + lane;  // TMEM lane quarter; accumulator row = (head, p)
    const int k = r >> 6, pr = r & 63;
    const bool store_thread = warp == kEpiWarp0 && lane == 0;
    grid_dep_wait();  // S may still be read by the kernels before the previous one
    for (uint32_t it_local = 0;; ++it_local) {
      Item it;
      if (!local_item<FUSED>(it_local, prm, it)) break;
      const uint32_t a = it_local & 1;
      const bool ok = mbar_wait(bar(SM::kAccFull + a), (it_local >> 1) & 1, ctl) && !*abort_flag;
      tc_fence_after();
      if (store_thread) bulk_wait_read0();  // the staging buffer is free again
      named_bar_sync(kBarEpi, 128);
      if (ok) {
#pragma unroll 1
        for (int q = 0; q < NT / 32; ++q) {
          uint32_t v[32];
          __syncwarp();
          tmem_ld32(tmem + a * NT + (uint32_t(32 * q4) << 16) + q * 32, v);
          tmem_ld_wait();
          uint8_t* box = smem + SM::kOut + ((q >> 1) * 2 + k) * kBox;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int cc = (q & 1) * 4 + c4;
            *reinterpret_cast<uint4*>(box + pr * 128 + ((cc ^ (pr & 7)) << 4)) =
                make_uint4(pack_bf16x2(__uint_as_float(v[8 * c4]), __uint_as_float(v[8 * c4 + 1])),
                           pack_bf16x2(__uint_as_float(v[8 * c4 + 2]), __uint_as_float(v[8 * c4 + 3])),
                           pack_bf16x2(__uint_as_float(v[8 * c4 + 4]), __uint_as_float(v[8 * c4 + 5])),
                           pack_bf16x2(__uint_as_float(v[8 * c4 + 6]), __uint_as_float(v[8 * c4 + 7])));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(SM::kAccEmpty + a));
      fence_proxy_async_smem();
      named_bar_sync(kBarEpi, 128);
      if (store_thread && ok) {
        for (int j = 0; j < NT / 64; ++j)
          for (int kk = 0; kk < it.nh; ++kk)
            tma_store_2d(&tm_S, sb + SM::kOut + (j * 2 + kk) * kBox, it.nt * NT + j * 64,
                         ((it.b * prm.nc + it.c) * prm.H + it.h0 + kk) * 64);
        bulk_commit();
      }
    }
    if (store_thread) bulk_wait_read0();  // the stores have read the staging buffer
  }

  grid_dep_launch();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

template <int NT, bool FUSED = false>
cudaError_t launch_nt(const CUtensorMap& tx, const CUtensorMap& tb, const CUtensorMap& ts,
                      const CsParams& prm, cudaStream_t st) {
  using SM = CsSmem<NT>;
  auto kern = chunk_state_tc_kernel<NT, FUSED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kAlloc);
  if (e != cudaSuccess) return e;
  int sms = num_sms_current_device();
  if (sms <= 0) sms = 1;
  const int64_t units = FUSED ? prm.chains : prm.items;
  const int64_t grid = units < sms ? units : sms;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), SM::kAlloc, st, tx, tb, ts, prm);
}

// ---- one CTA per work item: the first design, kept for problems with few items per SM ----
//
// One CTA = (head pair, n-tile, chunk, batch), 256 threads, no warp specialisation: thread 0
// issues TMA loads (2-stage ring over 64-token k-blocks) and the MMAs; all threads scale the x
// tile in shared memory by the decay weight, then drain the f32 accumulator from tensor memory
// (two warps per lane quarter, one column half each) and stage it, rounded to bf16, for TMA
// stores of S.  256 threads instead of 128 halve each k-block's scaling pass: 16K-token sweeps
// N = 64 / 128 / 256 29.7 -> 27.3, 37.5 -> 33.4, 53 -> 45 us.  Several CTAs share an SM, so their
// load, MMA and store phases overlap one another; with a few items per SM that beats the
// persistent kernel's single pipeline (130M layer 15.5 against 18.4 us), with many it loses
// (2.7B layer 62 against 58 us, 256K tokens 366 against 316 us).
constexpr int kItemThreads = 256;

template <int NT>
struct ItemSmem {
  static constexpr uint32_t kX = 2 * kBox;            // x: two heads x (64 tokens x 64 p)
  static constexpr uint32_t kB = (NT / 64) * kBox;    // B: NT/64 boxes of (64 tokens x 64 n)
  static constexpr uint32_t kStage = kX + kB;
  static constexpr uint32_t kTiles = 2 * kStage;      // 2-stage ring; reused as epilogue staging
  static constexpr uint32_t kW = kTiles;              // float w[2][256]
  static constexpr uint32_t kBars = kW + 2 * 256 * 4; // full[2], empty[2], done, drain
  static constexpr uint32_t kTmemSlot = kBars + 6 * 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kUsed = kAbort + 4;
  static constexpr uint32_t kAlloc = kUsed + 1024;    // slack for 1024-byte alignment
  static_assert((NT / 64) * 2 * kBox <= kTiles, "epilogue staging must fit in the ring");
};

template <int NT>
__global__ void __launch_bounds__(kItemThreads, 1)
    chunk_state_item_kernel(const __grid_constant__ CUtensorMap tm_x,
                          const __grid_constant__ CUtensorMap tm_B,
                          const __grid_constant__ CUtensorMap tm_S, const CsParams prm) {
  using SM = ItemSmem<NT>;
  extern __shared__ uint8_t smem_raw[];
  // align by pointer arithmetic on the __shared__ array so accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5;

  const int nt = blockIdx.x % prm.n_tiles;
  const int pair = blockIdx.x / prm.n_tiles;
  const int g = pair / prm.pairs_per_group;
  const int h0 = g * prm.hpg + 2 * (pair % prm.pairs_per_group);
  const int nh = min(2, (g + 1) * prm.hpg - h0);  // 1 when the group has an odd head count
  const int c = blockIdx.y, b = blockIdx.z;
  const int Q = prm.Q, kblocks = Q / 64;

  float* wsm = reinterpret_cast<float*>(smem + SM::kW);
  const uint32_t bar_full = sb + SM::kBars, bar_empty = bar_full + 16, bar_done = bar_full + 32,
                 bar_drain = bar_full + 40;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + SM::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kTmemSlot);

  if (tid == 0) {
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_B);
    prefetch_tmap(&tm_S);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_done, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), NT);
    tmem_relinquish();
  }
  // thread-0 bookkeeping of loads in flight (for the drain on abort)
  int issued = 0, consumed = 0;
  auto issue = [&](int kb) {
    const int s = kb & 1;
    const uint32_t st = sb + s * SM::kStage;
    const uint32_t full = bar_full + 8 * s;
    const int t0 = c * Q + kb * 64;
    mbar_arrive_expect_tx(full, SM::kStage);
    // one box each: both heads' x tiles, and all NT / 64 column tiles of B
    tma_load_4d(st, &tm_x, full, 0, t0, h0, b);
    tma_load_4d(st + SM::kX, &tm_B, full, 0, t0, (g * prm.N + nt * NT) / 64, b);
    issued = kb + 1;
  };

  // x and B are inputs of the step, not written by the kernels before this one (and every kernel
  // before the previous one has completed), so the first two k-blocks are requested before
  // waiting for the previous kernel's cs2 / dtT
  if (tid == 0) {
    issue(0);
    if (kblocks > 1) issue(1);
  }
  grid_dep_wait();  // cs2 / dtT come from the previous kernel; S may still be read by older ones
  // decay weights of the (up to) two heads: w[k][t] = 2^(cs2_last - cs2_t) * dt_t
  for (int e = tid; e < 2 * Q; e += kItemThreads) {
    const int k = e / Q, t = e % Q;
    float w = 0.f;
    if (k < nh) {
      const int64_t row = ((int64_t(b) * prm.H + h0 + k) * prm.nc + c) * Q;
      w = ex2(prm.cs2[row + Q - 1] - prm.cs2[row + t]) * prm.dtT[row + t];
    }
    wsm[k * 256 + t] = w;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{prm.wait_ns, abort_flag, prm.status};
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, NT, 1, 1);

  for (int kb = 0; kb < kblocks; ++kb) {
    const int s = kb & 1;
    const uint32_t ph = (kb >> 1) & 1;
    const bool ok = mbar_wait(bar_full + 8 * s, ph, ctl);
    if (tid == 0 && ok) consumed = kb + 1;
    if (ok) {
      // x~ = w * x in place: 1024 16-byte chunks (two boxes x 64 rows x 8), 4 per thread
      uint8_t* xs = smem + s * SM::kStage;
#pragma unroll
      for (int i = 0; i < 1024 / kItemThreads; ++i) {
        const int q = tid + kItemThreads * i;
        const int k = q >> 9, r = (q >> 3) & 63;
        const float w = wsm[k * 256 + kb * 64 + r];
        const uint32_t w2 = pack_bf16x2(w, w);
        uint4* p = reinterpret_cast<uint4*>(xs + q * 16);
        uint4 v = *p;
        v.x = scale_bf16x2(v.x, w2);
        v.y = scale_bf16x2(v.y, w2);
        v.z = scale_bf16x2(v.z, w2);
        v.w = scale_bf16x2(v.w, w2);
        *p = v;
      }
      fence_proxy_async_smem();
    }
    __syncthreads();
    if (tid == 0 && !*abort_flag) {
      tc_fence_after();
      const uint32_t xa = sb + s * SM::kStage, ba = xa + SM::kX;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_f16(tmem, sdesc_sw128(xa + k * 2048, kBox, 1024), sdesc_sw128(ba + k * 2048, kBox, 1024),
                 kIdesc, (kb | k) != 0 ? 1u : 0u);
      umma_commit(bar_empty + 8 * s);
      if (kb + 2 < kblocks) {
        // reuse stage s once the MMAs just issued have read it
        if (mbar_wait(bar_empty + 8 * s, ph, ctl)) issue(kb + 2);
      }
    }
  }

  // all MMAs complete -> accumulator readable
  if (tid == 0) umma_commit(bar_done);
  // uniform across the CTA: the epilogue below contains block-wide barriers
  const bool acc_ok = __syncthreads_and(mbar_wait(bar_done, 0, ctl) && !*abort_flag) != 0;
  tc_fence_after();

  if (acc_ok) {
    // S is stored in bf16: one 64 x 64 box (8 KB, 128-byte rows, swizzled) per (n block, head);
    // warp w reads TMEM lane quarter w % 4 and the column half w / 4
    const int quarter = warp & 3, half = warp >> 2;
    const int rr = 32 * quarter + (tid & 31), k = rr >> 6, r = rr & 63;
#pragma unroll 1
    for (int q = half * (NT / 64); q < (half + 1) * (NT / 64); ++q) {
      uint32_t v[32];
      __syncwarp();
      tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + q * 32, v);
      tmem_ld_wait();
      uint8_t* box = smem + ((q >> 1) * 2 + k) * kBox;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int cc = (q & 1) * 4 + c4;
        *reinterpret_cast<uint4*>(box + r * 128 + ((cc ^ (r & 7)) << 4)) =
            make_uint4(pack_bf16x2(__uint_as_float(v[8 * c4]), __uint_as_float(v[8 * c4 + 1])),
                       pack_bf16x2(__uint_as_float(v[8 * c4 + 2]), __uint_as_float(v[8 * c4 + 3])),
                       pack_bf16x2(__uint_as_float(v[8 * c4 + 4]), __uint_as_float(v[8 * c4 + 5])),
                       pack_bf16x2(__uint_as_float(v[8 * c4 + 6]), __uint_as_float(v[8 * c4 + 7])));
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      for (int j = 0; j < NT / 64; ++j)
        for (int kk = 0; kk < nh; ++kk)
          tma_store_2d(&tm_S, sb + (j * 2 + kk) * kBox, nt * NT + j * 64,
                       ((b * prm.nc + c) * prm.H + h0 + kk) * 64);
      bulk_commit();
    }
  }

  grid_dep_launch();
  // teardown: drain whatever is still in flight, then release tensor memory
  if (tid == 0) {
    for (int kb = consumed; kb < issued; ++kb)
      (void)mbar_drain(bar_full + 8 * (kb & 1), (kb >> 1) & 1, kWaitLimitNs);
    if (!acc_ok) {
      umma_commit(bar_drain);
      (void)mbar_drain(bar_drain, 0, kWaitLimitNs);
    }
    bulk_wait_read0();  // shared memory may be released once the stores have read it
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, NT);
  }
}

template <int NT>
cudaError_t launch_item_nt(const Problem& p, const CUtensorMap& tx, const CUtensorMap& tb,
                      const CUtensorMap& ts, const CsParams& prm, cudaStream_t st) {
  using SM = ItemSmem<NT>;
  auto kern = chunk_state_item_kernel<NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kAlloc);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(p.G * prm.pairs_per_group * prm.n_tiles),
                  static_cast<unsigned>(p.nc), static_cast<unsigned>(p.b));
  return launch_pdl(kern, grid, dim3(kItemThreads), SM::kAlloc, st, tx, tb, ts, prm);
}

}  // namespace

// Items per SM from which the persistent kernel runs (measured: 2.5 and 6.7 per SM favour one
// CTA per item, 13.5 and more the persistent kernel).
constexpr int64_t kPersistentItemsPerSm = 12;

bool chunk_state_tc_ok(const Problem& p) {
  return p.io_bf16 && p.P == 64 && (p.Q == 128 || p.Q == 256) &&
         (p.N == 64 || p.N == 128 || p.N == 256 || p.N == 512) &&
         p.L <= (int64_t(1) << 31) - 1 && p.b * p.nc * p.H * p.P < (int64_t(1) << 31);
}

namespace {

// Tensor maps and parameters shared by the chunk_state launches.  out: S, or hprev for the fused
// kernel (the same (b, nc, H, P, N) bf16 layout).
bool encode_cs_maps(const Problem& p, int NT, const void* x, const void* B, void* out, CUtensorMap* tx,
                    CUtensorMap* tb, CUtensorMap* ts, const char** why) {
  // TMA boxes cost about the same for 8 and 16 KB, so each k-block takes one box for x and one
  // for B: x (b, L, H, P) viewed as (p, token, head, batch) with a box of two heads, and B
  // (b, L, G, N) as (64 columns, token, N / 64 column blocks, batch) with a box of NT / 64 blocks;
  // both land as 64-row x 128-byte swizzled tiles, one after the other.
  {
    const uint64_t dims[4] = {64, uint64_t(p.L), uint64_t(p.H), uint64_t(p.b)};
    const uint64_t strides[3] = {uint64_t(p.H * p.P * 2), uint64_t(p.P * 2), uint64_t(p.L * p.H * p.P * 2)};
    const uint32_t box[4] = {64, 64, 2, 1};
    if (!encode_tmap(tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, x, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B, why))
      return false;
  }
  {
    const uint64_t dims[4] = {64, uint64_t(p.L), uint64_t(p.G * p.N / 64), uint64_t(p.b)};
    const uint64_t strides[3] = {uint64_t(p.G * p.N * 2), 128, uint64_t(p.L * p.G * p.N * 2)};
    const uint32_t box[4] = {64, 64, uint32_t(NT / 64), 1};
    if (!encode_tmap(tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, B, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B, why))
      return false;
  }
  {
    const uint64_t dims[2] = {uint64_t(p.N), uint64_t(p.b * p.nc * p.H * p.P)};
    const uint64_t strides[1] = {uint64_t(p.N * 2)};
    const uint32_t box[2] = {64, 64};
    if (!encode_tmap(ts, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B, why))
      return false;
  }
  return true;
}

CsParams make_cs_params(const Problem& p, int NT, const float* cs2, const float* dtT, uint32_t* status) {
  CsParams prm{};
  prm.L = static_cast<int32_t>(p.L);
  prm.H = static_cast<int32_t>(p.H);
  prm.nc = static_cast<int32_t>(p.nc);
  prm.Q = static_cast<int32_t>(p.Q);
  prm.N = static_cast<int32_t>(p.N);
  prm.hpg = static_cast<int32_t>(p.hpg);
  prm.pairs_per_group = static_cast<int32_t>((p.hpg + 1) / 2);
  prm.n_tiles = static_cast<int32_t>(p.N / NT);
  prm.chains = p.b * p.G * prm.pairs_per_group * prm.n_tiles;
  prm.items = prm.chains * p.nc;
  prm.cs2 = cs2;
  prm.dtT = dtT;
  prm.status = status;
  prm.wait_ns = kWaitLimitNs;
  return prm;
}

}  // namespace

cudaError_t launch_chunk_state_tc(const Problem& p, const void* x, const void* B, const float* cs2,
                                  const float* dtT, void* S, uint32_t* status, cudaStream_t st,
                                  const char** why) {
  const int NT = p.N >= 256 ? 256 : static_cast<int>(p.N);
  CUtensorMap tx, tb, ts;
  if (!encode_cs_maps(p, NT, x, B, S, &tx, &tb, &ts, why)) return cudaErrorInvalidValue;
  const CsParams prm = make_cs_params(p, NT, cs2, dtT, status);
  // the persistent kernel once every SM gets a dozen items or more, one CTA per item below that
  if (chunk_state_tc_persistent(p)) {
    switch (NT) {
      case 64: return launch_nt<64>(tx, tb, ts, prm, st);
      case 128: return launch_nt<128>(tx, tb, ts, prm, st);
      case 256: return launch_nt<256>(tx, tb, ts, prm, st);
    }
  } else {
    switch (NT) {
      case 64: return launch_item_nt<64>(p, tx, tb, ts, prm, st);
      case 128: return launch_item_nt<128>(p, tx, tb, ts, prm, st);
      case 256: return launch_item_nt<256>(p, tx, tb, ts, prm, st);
    }
  }
  return cudaErrorInvalidValue;
}

bool chunk_state_tc_persistent(const Problem& p) {
  const int NT = p.N >= 256 ? 256 : static_cast<int>(p.N);
  const int64_t items = p.b * p.nc * p.G * ((p.hpg + 1) / 2) * (p.N / NT);
  int sms = num_sms_current_device();
  if (sms <= 0) sms = 1;
  return items >= kPersistentItemsPerSm * int64_t(sms);
}

bool chunk_state_fused_ok(const Problem& p) {
  return chunk_state_tc_ok(p) && (p.N == 64 || p.N == 128);
}

cudaError_t launch_chunk_state_fused(const Problem& p, const void* x, const void* B, const float* cs2,
                                     const float* dtT, const float* init, void* hprev, float* final_state,
                                     uint32_t* status, cudaStream_t st, const char** why) {
  if (!chunk_state_fused_ok(p)) return cudaErrorInvalidValue;
  const int NT = static_cast<int>(p.N);
  CUtensorMap tx, tb, th;
  if (!encode_cs_maps(p, NT, x, B, hprev, &tx, &tb, &th, why)) return cudaErrorInvalidValue;
  CsParams prm = make_cs_params(p, NT, cs2, dtT, status);
  prm.init = init;
  prm.final_state = final_state;
  return NT == 64 ? launch_nt<64, true>(tx, tb, th, prm, st) : launch_nt<128, true>(tx, tb, th, prm, st);
}

}  // namespace ssd
