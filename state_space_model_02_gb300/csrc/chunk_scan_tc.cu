// chunk_scan (compute_out) on the 5th-generation tensor cores -- step 4 of the SSD forward scan.
//
// "Mamba-2 cuda-tile forward pass kernels" (devotd.net), section 2: the third kernel makes the
// token outputs from the chunk-start states, and instead of writing the intermediate matrix to
// global memory it keeps it next to the compute units.  For rows i of a chunk:
//     y[i,p] = sum_{j<=i} 2^{cs2_i - cs2_j} dt_j (C_i . B_j) x[j,p]
//              + 2^{cs2_i} (C_i . hprev[p,:]) + D_h x[i,p]
// Three dense contractions run on tcgen05 with f32 accumulators in tensor memory (TMEM):
//     CB = C_m B^T        (M = 128 rows i, N = j <= 256, K = state N)   once per (b, c, m-tile, group)
//     Y1 = P x_h          (M = 128, N = P = 64, K = j)                  per head
//     Y2 = C_m hprev_h^T  (M = 128, N = 64, K = state N)                per head
// with P = L o CB + D_h I: CB never leaves TMEM; for every head it is read back into registers,
// multiplied by the decay mask L_ij = 2^{cs2_i - cs2_j} dt_j (j <= i, else 0), D_h is added on
// the diagonal (so Y1 already holds D_h x_i), and the result is rounded to bf16 into shared
// memory as Y1's A operand.  The mask is factored per 32-column block [j0, j1], j1 = j0 + 31, as
// 2^{cs2_i - cs2_j1} * (2^{cs2_j1 - cs2_j} dt_j): one exp2 per row per block plus a per-head
// column table.  With decaying steps (dt A <= 0, cs2 non-increasing) both factors of a block
// left of the row's own are <= 1, whatever the step sizes, so they can only underflow where the
// weight itself is negligible.  In the row's own (diagonal) block the row factor grows with
// the block's decay span cs2_j0 - cs2_j1; where that span exceeds kMaxFactorSpan (log2 units)
// the block takes every weight as one exp2 per element instead.
//
// Persistent CTAs (one per SM: 512 TMEM columns, ~214 KB shared memory, 23 warps) walk a
// contiguous range of (batch, chunk, m-tile, head) units, weighted 2 : 3 for the two m-tiles
// of a 256-token chunk (their measured cost ratio); CB is recomputed when the range crosses to a new (batch, chunk, m-tile, group).  Warp
// roles, synchronised through mbarriers so the kinds of work overlap across heads:
//   warp 0      TMA producer: C and B per segment; per head hprev (2-slot ring, freed once Y2
//               is done; one box) and x, cs2, dt (2-slot ring, freed once Y1 and the mask are
//               done).  A TMA box costs the SM about the same for 64 or 128 rows, so operands
//               come in few, large boxes; the inputs of the head kPrefetchAhead places ahead
//               are prefetched into L2;
//   warp 1      tcgen05.mma issuer; owns the TMEM allocation.  It touches no shared memory
//               between MMAs (such an access waits for the MMAs already queued): warp 22
//               waits on its mbarriers and hands over through a named barrier
//   warps 2-17  mask: CB (TMEM) -> P (bf16, shared memory) for head h+1 ...
//   warps 18-21 epilogue: ... while these finish head h: y = Y1 + 2^{cs2_i} Y2 -> TMA store
// A warp reads the TMEM lane quarter (warp % 4): four mask warps share each quarter and take
// its 32-column blocks round-robin; the four epilogue warps cover the 128 rows once.  P is handed to
// the MMA issuer in four 64-column groups (one 16 KB swizzle atom each) with their own
// barriers, so Y1's MMAs on group k overlap the mask writing group k+1.
// Every wait is bounded; after an expiry all roles keep their loop trip counts (so named
// barriers stay matched) but skip their work, then drain and release TMEM.
// Requirements (chunk_scan_tc_ok): bf16 I/O, P = 64, Q in {128, 256}, N in {64, 128}, or N a
// multiple of 64 above 128 with N >= Q (WIDE).  A WIDE launch cannot keep the m-tile's C rows
// (128 x N) beside its other operands in shared memory: CB is built by a K loop over the state
// in 64-column steps (C and B tiles through two slots), and the term through hprev, Z =
// 2^{cs2_i} C_m hprev^T, comes from the readout kernel (chunk_readout_tc.cu), which runs first
// and leaves Z in bf16; the producer loads each head's Z rows into the hprev slot and the
// epilogue adds them (y = Y1 + Z), so no per-head C.hprev^T runs here.
#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kMaskWarps = 16, kEpiWarps = 4;  // warps 2-17 mask, 18-21 epilogue, 22 poller
constexpr int kPollWarp = 2 + kMaskWarps + kEpiWarps;
constexpr int kWarps = kPollWarp + 1;
constexpr int kThreads = kWarps * 32;
constexpr uint32_t kBox128 = 16384;  // TMA box: 128 rows x 128 bytes
constexpr uint32_t kBox64 = 8192;    // TMA box: 64 rows x 128 bytes
constexpr uint32_t kTmemCols = 512;  // CB [0,256) | Y1 buf0 | Y2 buf0 | Y1 buf1 | Y2 buf1
// Largest |cs2_j0 - cs2_j1| (log2 units) of a diagonal block for which the factored weights are
// used: each factor then stays within 2^{+-64}, far inside float32's range.
constexpr float kMaxFactorSpan = 64.f;
// named barriers: the mask group, the epilogue group, and the poller -> MMA issuer handoff
constexpr uint32_t kBarMask = 1, kBarEpi = 2, kBarIssue = 3;

// One handoff from the poller warp to the MMA-issuing warp: both warps (64 threads) arrive and
// both get the AND of their flags (the poller's "the awaited barriers completed and the CTA has
// not aborted"; the issuer passes true).  The barrier also orders the poller's acquire of those
// mbarriers before the issuer's following tcgen05 operations (with tcgen05.fence::after_thread_sync).
__device__ __forceinline__ bool issue_handoff(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(ok ? 1u : 0u), "n"(kBarIssue), "n"(64)
      : "memory");
  return r != 0u;
}

struct ScParams {
  int32_t L, H, nc, Q, N, hpg, MT;
  int64_t units, total_weight;
  const float* cs2;
  const float* dtT;
  const float* D;
  uint32_t* status;
  uint64_t wait_ns;
};

template <int NB>  // NB = N / 64
struct ScSmem {
  static constexpr uint32_t kC = 0;                          // NB x 16 KB: C rows of the m-tile
  static constexpr uint32_t kP = kC + NB * kBox128;          // 64 KB: P (bf16); B during CB phase
  static constexpr uint32_t kPBytes = 65536;
  static constexpr uint32_t kHpBytes = NB * kBox64;          // hprev slot: 64 p x N (bf16)
  static constexpr uint32_t kHp0 = kP + kPBytes;
  static constexpr uint32_t kXsX = 0;                        // x slot: 32 KB x (up to 256 tokens x 64 p)
  static constexpr uint32_t kXsCs = 32768;                   //         cs2 row, then dt row (Q floats each)
  static constexpr uint32_t kXsBytes = kXsCs + 2048;
  static constexpr uint32_t kXs0 = kHp0 + 2 * kHpBytes;
  static constexpr uint32_t kY = kXs0 + 2 * kXsBytes;        // 16 KB: y staging (128 rows x 128 B)
  static constexpr uint32_t kColf = kY + kBox128;            // 2 x 1 KB: per-head column factors
  static constexpr uint32_t kBars = kColf + 2048;
  static constexpr int kNumBars = 30;
  static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kWalk = kAbort + 4;              // SegWalk of the CTA's first unit
  static constexpr uint32_t kUsed = kWalk + 32;
  static constexpr uint32_t kAlloc = kUsed + 1024;           // slack for 1024-byte alignment
  static_assert(kXsBytes % 1024 == 0 && kHpBytes % 1024 == 0, "slots must stay 1024-byte aligned");
  static_assert(kAlloc <= 232448, "exceeds the per-CTA shared memory limit");
};

// mbarrier indices
enum : int {
  kCbFull = 0, kCbDone, kCbEmpty, kSegFree, kHpFull0, kHpFull1, kHpEmpty0, kHpEmpty1,
  kXsFull0, kXsFull1, kXsEmpty0, kXsEmpty1, kPFull0, kPEmpty0 = kPFull0 + 4,
  kYFull0 = kPEmpty0 + 4, kYFull1, kYEmpty0, kYEmpty1, kDrain,
  kCbK0, kCbK1, kCbKEmpty0, kCbKEmpty1  // WIDE: the two (C, B) K-step slots of the CB phase
};

// The producer warms L2 with the inputs of the head this many heads ahead in the segment (x rows,
// hprev or Z, cs2 / dt rows).  A head's x and hprev slots free only when the head two places
// earlier has finished its MMAs, and a load issued then takes about as long from HBM as a head
// does on the SM (measured: 1.4-1.8 us for x, 2-2.7 us for hprev at 256K tokens), which left the
// mask waiting for its head's inputs; from L2 the same loads arrive in time.  Measured steps
// (256K tokens / 2.7B layer): no prefetch 1361 / 225 us, 2 heads ahead 1292 / 211 us, 3 ahead
// 1304 / 212, 4 ahead 1326 / 213, 6 ahead 1382 / 222.
constexpr int kPrefetchAhead = 2;

// Work weights of the two 128-row m-tiles of a 256-token chunk (the second one's causal
// width is twice the first's, but its measured cost per head is about 1.5x, since loads and
// handoffs, not the mask and MMA work, dominate a unit).
constexpr int64_t kWeightMt0 = 2, kWeightMt1 = 3;

// First unit whose starting weight is >= w.  Units are ordered (b, c, m-tile, h); with one
// m-tile per chunk every unit weighs 1.
__device__ __forceinline__ int64_t unit_at_weight(int64_t w, int32_t H, int32_t MT) {
  if (MT == 1) return w;
  const int64_t wbc = (kWeightMt0 + kWeightMt1) * H;
  const int64_t bc = w / wbc, rem = w % wbc;
  if (rem <= kWeightMt0 * H) return bc * 2 * H + (rem + kWeightMt0 - 1) / kWeightMt0;
  const int64_t h = (rem - kWeightMt0 * H + kWeightMt1 - 1) / kWeightMt1;
  return h >= H ? (bc + 1) * 2 * H : bc * 2 * H + H + h;
}

// One run of consecutive heads sharing (b, c, m-tile, group): one CB.
struct Segment {
  int b, c, mt, g, h_begin, nh;
};

// Walks the segments of a CTA's unit range with 32-bit counters: the range's first unit is
// decomposed once (by one thread, for the whole CTA), then every role advances by carries, so
// no warp divides 64-bit integers in its loop.  Unit u = ((b * nc + c) * MT + mt) * H + h.
struct SegWalk {
  int32_t b, c, mt, h, u, u_end;

  __device__ __forceinline__ bool more() const { return u < u_end; }
  __device__ __forceinline__ Segment seg(const ScParams& prm) const {
    Segment s;
    s.b = b;
    s.c = c;
    s.mt = mt;
    s.h_begin = h;
    s.g = h / prm.hpg;
    s.nh = min((s.g + 1) * prm.hpg, h + (u_end - u)) - h;
    return s;
  }
  __device__ __forceinline__ void advance(int nh, const ScParams& prm) {
    u += nh;
    h += nh;
    if (h == prm.H) {
      h = 0;
      if (++mt == prm.MT) {
        mt = 0;
        if (++c == prm.nc) {
          c = 0;
          ++b;
        }
      }
    }
  }
};

__device__ __forceinline__ SegWalk walk_from(int64_t u_begin, int64_t u_end, const ScParams& prm) {
  SegWalk w;
  const uint32_t u = static_cast<uint32_t>(u_begin);
  const uint32_t bcm = u / uint32_t(prm.H), bc = bcm / uint32_t(prm.MT);
  w.h = static_cast<int32_t>(u - bcm * uint32_t(prm.H));
  w.mt = static_cast<int32_t>(bcm - bc * uint32_t(prm.MT));
  w.c = static_cast<int32_t>(bc % uint32_t(prm.nc));
  w.b = static_cast<int32_t>(bc / uint32_t(prm.nc));
  w.u = static_cast<int32_t>(u_begin);
  w.u_end = static_cast<int32_t>(u_end);
  return w;
}

// One 32 x 32 block of P for this thread's row: P[row, j0 + e] = CB[row, j0 + e] * colf[e] *
// rowf, rounded to bf16 and stored as four 16-byte chunks of the row's 128-byte swizzled line.
// DIAG: the block holding the diagonal (column dr = row - j0): zero right of it, + D_h on it.
template <bool DIAG>
__device__ __forceinline__ void mask_block(const uint32_t (&v)[32], const float* cf, float rowf, int dr,
                                           float Dh, uint8_t* pb, int cbase, int r) {
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    const float4 fa = reinterpret_cast<const float4*>(cf)[2 * c4];
    const float4 fb = reinterpret_cast<const float4*>(cf)[2 * c4 + 1];
    const float f[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
    uint32_t o[4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const int e = 8 * c4 + 2 * e2;
      // packed pair products (one f32x2 multiply per factor)
      const float2 w = mul_f32x2(mul_f32x2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                                           make_float2(f[2 * e2], f[2 * e2 + 1])),
                                 make_float2(rowf, rowf));
      float w0 = w.x, w1 = w.y;
      if (DIAG) {
        w0 = e > dr ? 0.f : (e == dr ? w0 + Dh : w0);
        w1 = e + 1 > dr ? 0.f : (e + 1 == dr ? w1 + Dh : w1);
      }
      o[e2] = pack_bf16x2(w0, w1);
    }
    *reinterpret_cast<uint4*>(pb + (((cbase + c4) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// The diagonal block of a row whose block decays by more than kMaxFactorSpan: every weight
// 2^{cs2_i - cs2_j} dt_j (j <= i) is one exp2 of its own, so no factor leaves float32's range.
// csb / dtb: the block's cs2 and dt values (shared memory, the same for every lane).
__device__ __forceinline__ void mask_block_exact(const uint32_t (&v)[32], const float* csb, const float* dtb,
                                                 float cs_i, int dr, float Dh, uint8_t* pb, int cbase, int r) {
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    uint32_t o[4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const int e = 8 * c4 + 2 * e2;
      float w[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float wt = e + u > dr ? 0.f : ex2(cs_i - csb[e + u]) * dtb[e + u];
        w[u] = __uint_as_float(v[e + u]) * wt + (e + u == dr ? Dh : 0.f);
      }
      o[e2] = pack_bf16x2(w[0], w[1]);
    }
    *reinterpret_cast<uint4*>(pb + (((cbase + c4) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

template <int NB, bool WIDE>  // WIDE: state above 128 columns (CB by a K loop, Z from the readout)
__global__ void __launch_bounds__(kThreads, 1)
    chunk_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                         const __grid_constant__ CUtensorMap tm_B,
                         const __grid_constant__ CUtensorMap tm_C,
                         const __grid_constant__ CUtensorMap tm_h,  // hprev, or Z when WIDE
                         const __grid_constant__ CUtensorMap tm_y,
                         const __grid_constant__ CUtensorMap tm_x2,  // x in 256-row boxes (Q = 256)
                         const __grid_constant__ CUtensorMap tm_cd,  // (cs2 row, dt row) pairs
                         const ScParams prm) {
  using SM = ScSmem<NB>;
  extern __shared__ uint8_t smem_raw[];
  // align by pointer arithmetic on the __shared__ array so accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t H = prm.H, Q = prm.Q, N = prm.N, MT = prm.MT;
  auto bar = [&](int i) { return sb + SM::kBars + 8u * i; };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + SM::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kTmemSlot);

  if (threadIdx.x == 0) {
    // this CTA's contiguous range of units, balanced by weight
    *reinterpret_cast<SegWalk*>(smem + SM::kWalk) =
        walk_from(unit_at_weight(prm.total_weight * blockIdx.x / gridDim.x, H, MT),
                  unit_at_weight(prm.total_weight * (blockIdx.x + 1) / gridDim.x, H, MT), prm);
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_B);
    prefetch_tmap(&tm_C);
    prefetch_tmap(&tm_h);
    prefetch_tmap(&tm_y);
    prefetch_tmap(&tm_x2);
    prefetch_tmap(&tm_cd);
    const uint32_t counts[SM::kNumBars] = {
        1, 1, kMaskWarps, 1,                                  // cb_full cb_done cb_empty seg_free
        1, 1, WIDE ? kEpiWarps : 1, WIDE ? kEpiWarps : 1,     // hp_full[2] hp_empty[2]
        1, 1, 1 + kMaskWarps, 1 + kMaskWarps,                 // xs_full[2] xs_empty[2]
        kMaskWarps / 2, kMaskWarps / 2, kMaskWarps / 2, kMaskWarps / 2,  // p_full[4]: owners
        1, 1, 1, 1,                                           // p_empty[4]
        1, 1, kEpiWarps, kEpiWarps,                           // y_full[2] y_empty[2]
        1, 1,                                                 // drain, spare
        1, 1, 1, 1};                                          // cbk_full[2] cbk_empty[2]
    for (int i = 0; i < SM::kNumBars; ++i) mbar_init(bar(i), counts[i]);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{prm.wait_ns, abort_flag, prm.status};
  // hprev, cs2 and dtT come from the previous kernels: the producer and the epilogue (the roles
  // that read them from global memory) wait for those in grid_dep_wait; the other roles only
  // see data through the producer's barriers

  const SegWalk walk0 = *reinterpret_cast<const SegWalk*>(smem + SM::kWalk);

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t gi = 0, si = 0, cbk = 0;
      bool pend_cb = false, pend_hp[2] = {false, false}, pend_xs[2] = {false, false};
      bool pend_cbk[2] = {false, false};
      uint32_t ph_cb = 0, ph_hp[2] = {0, 0}, ph_xs[2] = {0, 0}, ph_cbk[2] = {0, 0};
      auto load_cb = [&](const Segment& sg) {
        const int i0 = sg.mt * 128, jrows = i0 + 128;
        mbar_arrive_expect_tx(bar(kCbFull), NB * kBox128 + NB * jrows * 128);
        for (int nb = 0; nb < NB; ++nb)
          tma_load_3d(sb + SM::kC + nb * kBox128, &tm_C, bar(kCbFull), sg.g * N + nb * 64,
                      sg.c * Q + i0, sg.b);
        for (int nb = 0; nb < NB; ++nb)
          for (int jb = 0; jb < jrows / 128; ++jb)
            tma_load_3d(sb + SM::kP + nb * jrows * 128 + jb * kBox128, &tm_B, bar(kCbFull),
                        sg.g * N + nb * 64, sg.c * Q + jb * 128, sg.b);
      };
      // WIDE: the segment's CB operands as N / 64 K steps of 64 state columns, each C tile
      // (128 rows) and B tile (jrows rows) into slot cbk % 2 (C region, P region halves)
      auto load_cb_wide = [&](const Segment& sg) {
        const int i0 = sg.mt * 128, jrows = i0 + 128;
        for (int k = 0; k < N / 64; ++k, ++cbk) {
          const uint32_t slot = cbk & 1;
          if (cbk >= 2) (void)mbar_wait(bar(kCbKEmpty0 + slot), ((cbk >> 1) - 1) & 1, ctl);
          if (*abort_flag) continue;
          const uint32_t fb = bar(kCbK0 + slot);
          mbar_arrive_expect_tx(fb, kBox128 + jrows * 128);
          tma_load_3d(sb + SM::kC + slot * kBox128, &tm_C, fb, sg.g * N + 64 * k, sg.c * Q + i0, sg.b);
          for (int jb = 0; jb < jrows / 128; ++jb)
            tma_load_3d(sb + SM::kP + slot * 32768 + jb * kBox128, &tm_B, fb, sg.g * N + 64 * k,
                        sg.c * Q + jb * 128, sg.b);
          pend_cbk[slot] = true;
          ph_cbk[slot] = (cbk >> 1) & 1;
        }
      };
      // x slot s of a head: its x box(es) now, its cs2 / dt rows (from the previous kernel) later;
      // the slot's barrier expects all three from the start
      auto load_x = [&](const Segment& sg, int hh, uint32_t s) {
        const int jrows = sg.mt * 128 + 128;
        const uint32_t xs = sb + SM::kXs0 + s * SM::kXsBytes;
        const uint32_t xb = bar(kXsFull0 + s);
        mbar_arrive_expect_tx(xb, jrows * 128 + 2 * Q * 4);
        // a 256-row head's x as one box: a TMA operation costs the SM about the same for 128 or
        // 256 rows, and the producer issues several per head
        if (jrows == 256)
          tma_load_3d(xs + SM::kXsX, &tm_x2, xb, hh * 64, sg.c * Q, sg.b);
        else
          tma_load_3d(xs + SM::kXsX, &tm_x, xb, hh * 64, sg.c * Q, sg.b);
      };
      // L2 prefetch of head hh's inputs (no shared memory, no barrier); hprev / Z, cs2 and dt come
      // from the previous kernels, so this runs only after grid_dep_wait
      auto prefetch_head = [&](const Segment& sg, int hh) {
        const int i0 = sg.mt * 128, jrows = i0 + 128;
        if (jrows == 256)
          tma_prefetch_3d(&tm_x2, hh * 64, sg.c * Q, sg.b);
        else
          tma_prefetch_3d(&tm_x, hh * 64, sg.c * Q, sg.b);
        if (WIDE)
          tma_prefetch_3d(&tm_h, hh * 64, sg.c * Q + i0, sg.b);
        else
          tma_prefetch_3d(&tm_h, 0, ((sg.b * prm.nc + sg.c) * H + hh) * 64, 0);
        tma_prefetch_3d(&tm_cd, 0, int32_t((int64_t(sg.b) * H + hh) * prm.nc + sg.c), 0);
      };
      // C, B and x are inputs of the step, not written by the kernels before this one (and every
      // kernel before the previous one has completed): the first segment's C and B and the first
      // two heads' x are requested before waiting for the previous kernels
      int pre_x = 0;
      if (walk0.more()) {
        const Segment sg0 = walk0.seg(prm);
        if (!WIDE) {
          load_cb(sg0);
          pend_cb = true;
        }
        pre_x = sg0.nh < 2 ? sg0.nh : 2;
        for (int hi = 0; hi < pre_x; ++hi) load_x(sg0, sg0.h_begin + hi, uint32_t(hi));
      }
      grid_dep_wait();
      for (SegWalk w = walk0; w.more(); ++si) {
        const Segment sg = w.seg(prm);
        const int i0 = sg.mt * 128;
        // C and B of the new segment overwrite regions the previous segment's MMAs read
        if (si >= 1) (void)mbar_wait(bar(kSegFree), (si - 1) & 1, ctl);
        if (WIDE) {
          load_cb_wide(sg);
        } else if (si >= 1 && !*abort_flag) {
          load_cb(sg);
          pend_cb = true;
          ph_cb = si & 1;
        }
        for (int hi = 0; hi < sg.nh; ++hi, ++gi) {
          const int hh = sg.h_begin + hi;
          const uint32_t s = gi & 1, use = gi >> 1;
          // hprev first: Y2 needs it first, and its slot frees early
          if (gi >= 2) (void)mbar_wait(bar(kHpEmpty0 + s), (use - 1) & 1, ctl);
          if (!*abort_flag) {
            const uint32_t hb = bar(kHpFull0 + s);
            mbar_arrive_expect_tx(hb, SM::kHpBytes);
            if (WIDE)  // the head's Z rows of the m-tile (128 rows x 64 p)
              tma_load_3d(sb + SM::kHp0 + s * SM::kHpBytes, &tm_h, hb, hh * 64, sg.c * Q + i0, sg.b);
            else  // one 3-D box brings both 64-column halves of the head's state (NB 8 KB tiles)
              tma_load_3d(sb + SM::kHp0 + s * SM::kHpBytes, &tm_h, hb, 0,
                          ((sg.b * prm.nc + sg.c) * H + hh) * 64, 0);
            pend_hp[s] = true;
            ph_hp[s] = use & 1;
          }
          if (gi >= 2) (void)mbar_wait(bar(kXsEmpty0 + s), (use - 1) & 1, ctl);
          if (!*abort_flag || gi < uint32_t(pre_x)) {
            // (a slot whose x went out early must still get its cs2 / dt bytes)
            const uint32_t xs = sb + SM::kXs0 + s * SM::kXsBytes;
            const uint32_t xb = bar(kXsFull0 + s);
            if (gi >= uint32_t(pre_x)) load_x(sg, hh, s);
            // the head's cs2 and dt rows as one box of the (Q, row, array) view
            tma_load_3d(xs + SM::kXsCs, &tm_cd, xb, 0, int32_t((int64_t(sg.b) * H + hh) * prm.nc + sg.c), 0);
            pend_xs[s] = true;
            ph_xs[s] = use & 1;
          }
          if (kPrefetchAhead > 0 && hi + kPrefetchAhead < sg.nh && !*abort_flag)
            prefetch_head(sg, hh + kPrefetchAhead);
        }
        w.advance(sg.nh, prm);
      }
      // drain: every load issued must have landed before the CTA may exit
      if (pend_cb) (void)mbar_drain(bar(kCbFull), ph_cb, kWaitLimitNs);
      for (int s = 0; s < 2; ++s) {
        if (pend_cbk[s]) (void)mbar_drain(bar(kCbK0 + s), ph_cbk[s], kWaitLimitNs);
        if (pend_hp[s]) (void)mbar_drain(bar(kHpFull0 + s), ph_hp[s], kWaitLimitNs);
        if (pend_xs[s]) (void)mbar_drain(bar(kXsFull0 + s), ph_xs[s], kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------------- MMA issuer
    // The whole warp walks the schedule and lane 0 issues.  It never waits on an mbarrier or
    // reads the abort flag itself: a shared-memory access by the issuing thread stalls until its
    // queued MMAs have completed, which would serialise the groups.  The poller warp waits and
    // hands each "go" over through kBarIssue, at exactly the same points of the same schedule.
    uint32_t gi = 0, cbk = 0;
    for (SegWalk w = walk0; w.more();) {
      const Segment sg = w.seg(prm);
      const int jrows = sg.mt * 128 + 128;
      const uint32_t idesc_cb = idesc_bf16_f32(128, jrows, 0, 0);
      if (WIDE) {
        // CB = sum over the K steps of C_k B_k^T
        for (int k = 0; k < N / 64; ++k, ++cbk) {
          const uint32_t slot = cbk & 1;
          const bool go = issue_handoff(true);
          if (lane == 0) {
            if (go) {
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_f16(tmem, sdesc_sw128(sb + SM::kC + slot * kBox128 + kk * 32, 16, 1024),
                         sdesc_sw128(sb + SM::kP + slot * 32768 + kk * 32, 16, 1024), idesc_cb,
                         (k | kk) != 0 ? 1u : 0u);
            }
            umma_commit(bar(kCbKEmpty0 + slot));
          }
          __syncwarp();
        }
        if (lane == 0) umma_commit(bar(kCbDone));
        __syncwarp();
      } else {
        const bool go_cb = issue_handoff(true);
        if (lane == 0) {
          if (go_cb) {
            tc_fence_after();
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                umma_f16(tmem, sdesc_sw128(sb + SM::kC + nb * kBox128 + k * 32, 16, 1024),
                         sdesc_sw128(sb + SM::kP + nb * jrows * 128 + k * 32, 16, 1024), idesc_cb,
                         (nb | k) != 0 ? 1u : 0u);
          }
          umma_commit(bar(kCbDone));
        }
        __syncwarp();
      }
      for (int hi = 0; hi < sg.nh; ++hi, ++gi) {
        const uint32_t s = gi & 1;
        const uint32_t xs = sb + SM::kXs0 + s * SM::kXsBytes;
        const uint32_t hp = sb + SM::kHp0 + s * SM::kHpBytes;
        const uint32_t ycol = 256 + 128 * s;
        const bool go_y2 = WIDE || issue_handoff(true);  // WIDE: Z comes from the readout
        if (!WIDE && lane == 0) {
          if (go_y2) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                umma_f16(tmem + ycol + 64, sdesc_sw128(sb + SM::kC + nb * kBox128 + k * 32, 16, 1024),
                         sdesc_sw128(hp + nb * kBox64 + k * 32, 16, 1024), idesc, (nb | k) != 0 ? 1u : 0u);
          }
          umma_commit(bar(kHpEmpty0 + s));
        }
        __syncwarp();
        const uint32_t idesc1 = idesc_bf16_f32(128, 64, 0, 1);
        for (int k = 0; k < jrows / 64; ++k) {
          const bool go = issue_handoff(true);
          if (lane == 0) {
            if (go) {
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_f16(tmem + ycol, sdesc_sw128(sb + SM::kP + k * kBox128 + kk * 32, 16, 1024),
                         sdesc_sw128(xs + SM::kXsX + (4 * k + kk) * 2048, kBox128, 1024), idesc1,
                         (k | kk) != 0 ? 1u : 0u);
            }
            umma_commit(bar(kPEmpty0 + k));
          }
          __syncwarp();
        }
        if (lane == 0) {
          umma_commit(bar(kYFull0 + s));
          umma_commit(bar(kXsEmpty0 + s));
        }
        __syncwarp();
      }
      if (lane == 0) umma_commit(bar(kSegFree));
      __syncwarp();
      w.advance(sg.nh, prm);
    }
    if (lane == 0) {
      umma_commit(bar(kDrain));
      (void)mbar_drain(bar(kDrain), 0, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == kPollWarp) {
    // ----------------------------------------------------- poller for the MMA issuer
    // the issuer's waits, in its order; every wait is bounded, so every handoff is reached
    uint32_t gi = 0, si = 0, gpar = 0, cbk = 0;  // gpar bit k: parity of P group k's uses so far
    for (SegWalk w = walk0; w.more(); ++si) {
      const Segment sg = w.seg(prm);
      const int jrows = sg.mt * 128 + 128;
      const bool e = si == 0 || mbar_wait(bar(kCbEmpty), (si - 1) & 1, ctl);
      if (WIDE) {
        for (int k = 0; k < N / 64; ++k, ++cbk) {
          const bool a = mbar_wait(bar(kCbK0 + (cbk & 1)), (cbk >> 1) & 1, ctl);
          (void)issue_handoff(a && e && !*abort_flag);
        }
      } else {
        const bool a = mbar_wait(bar(kCbFull), si & 1, ctl);
        (void)issue_handoff(a && e && !*abort_flag);
      }
      for (int hi = 0; hi < sg.nh; ++hi, ++gi) {
        const uint32_t s = gi & 1, use = gi >> 1;
        const bool y = gi < 2 || mbar_wait(bar(kYEmpty0 + s), (use - 1) & 1, ctl);
        if (!WIDE) {
          const bool h = mbar_wait(bar(kHpFull0 + s), use & 1, ctl);
          (void)issue_handoff(h && y && !*abort_flag);
        }
        const bool f = mbar_wait(bar(kXsFull0 + s), use & 1, ctl);
        for (int k = 0; k < jrows / 64; ++k) {
          const bool p = mbar_wait(bar(kPFull0 + k), (gpar >> k) & 1u, ctl);
          (void)issue_handoff(f && y && p && !*abort_flag);
          gpar ^= 1u << k;
        }
      }
      w.advance(sg.nh, prm);
    }
  } else if (warp < 2 + kMaskWarps) {
    // ------------------------------------------------------------- mask: CB -> P in smem
    const int q = warp & 3, r = 32 * q + lane;  // TMEM lane quarter and m-tile row
    const int sub = (warp - 2) >> 2;            // which of the quarter's four mask warps
    const int mt_thread = (warp - 2) * 32 + lane;  // 0..511 over the mask group
    const uint32_t trow = tmem + (uint32_t(32 * q) << 16);
    uint32_t gi = 0, si = 0;
    uint32_t gpar = 0, gused = 0;  // per P group: parity of its uses so far, used at least once
    for (SegWalk w = walk0; w.more(); ++si) {
      const Segment sg = w.seg(prm);
      const int i0 = sg.mt * 128, jrows = i0 + 128, row = i0 + r;
      const int nblk = jrows / 32, maxblk = i0 / 32 + q;
      (void)mbar_wait(bar(kCbDone), si & 1, ctl);
      tc_fence_after();
      // blocks right of this quarter's diagonal block stay zero for the whole segment
      for (int blk = maxblk + 1 + sub; blk < nblk; blk += 4) {
        const int j0 = 32 * blk;
        uint8_t* pb = smem + SM::kP + (j0 >> 6) * kBox128 + r * 128;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
          *reinterpret_cast<uint4*>(pb + (((((j0 & 63) >> 3) + c4) ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
      }
      for (int hi = 0; hi < sg.nh; ++hi, ++gi) {
        const uint32_t s = gi & 1;
        const uint8_t* xsp = smem + SM::kXs0 + s * SM::kXsBytes;
        const float* cs = reinterpret_cast<const float*>(xsp + SM::kXsCs);
        const float* dtv = cs + Q;  // the dt row follows the cs2 row
        float* colf = reinterpret_cast<float*>(smem + SM::kColf + (gi & 1) * 1024);
        const bool have = mbar_wait(bar(kXsFull0 + s), (gi >> 1) & 1, ctl);
        if (have && mt_thread < jrows)
          colf[mt_thread] = ex2(cs[mt_thread | 31] - cs[mt_thread]) * dtv[mt_thread];
        const float cs_i = have ? cs[row] : 0.f;
        const float Dh = prm.D ? __ldg(prm.D + sg.h_begin + hi) : 0.f;
        named_bar_sync(kBarMask, 32 * kMaskWarps);
        const bool live = have && !*abort_flag;
        tc_fence_after();
        // group k holds 32-column blocks 2k and 2k+1; a quarter's four warps take its blocks
        // round-robin (warp sub owns block 2k + (sub & 1) of the groups k with k % 2 == sub / 2),
        // so two groups are written at once, and only a group's eight owner warps (two per lane
        // quarter) arrive on its barrier.  The TMEM load of the block is issued before the wait
        // for the group's P buffer (the head-start barrier keeps every warp within one head of
        // the others).
        const int ng = jrows / 64;
#pragma unroll 1
        for (int k = sub >> 1; k < ng; k += 2) {
          const int blk = 2 * k + (sub & 1), j0 = 32 * blk;
          const bool mine = live && blk <= maxblk;
          uint32_t v[32];
          if (mine) {
            __syncwarp();
            tmem_ld32(trow + j0, v);
          }
          const bool pfree = !((gused >> k) & 1u) ||
                             mbar_wait(bar(kPEmpty0 + k), ((gpar >> k) & 1u) ^ 1u, ctl);
          if (mine) tmem_ld_wait();
          if (mine && pfree) {
            // P[row, j] = CB[row, j] colf[j] 2^(cs2_row - cs2_j1), zero right of the diagonal,
            // plus D_h on it
            const float rowf = ex2(cs_i - cs[j0 + 31]);
            const float* cf = colf + j0;
            uint8_t* pb = smem + SM::kP + (j0 >> 6) * kBox128 + r * 128;
            const int cbase = (j0 & 63) >> 3;
            // one branch per block (uniform across the warp): the diagonal block masks j > row and
            // adds D_h on j == row, per element when its decay span is too wide to factor
            if (blk != maxblk)
              mask_block<false>(v, cf, rowf, 0, 0.f, pb, cbase, r);
            else if (fabsf(cs[j0] - cs[j0 + 31]) <= kMaxFactorSpan)
              mask_block<true>(v, cf, rowf, row - j0, Dh, pb, cbase, r);
            else
              mask_block_exact(v, cs + j0, dtv + j0, cs_i, row - j0, Dh, pb, cbase, r);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kPFull0 + k));
          gpar ^= 1u << k;
          gused |= 1u << k;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kXsEmpty0 + s));
      }
      // CB of this segment has been read for the last time
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kCbEmpty));
      w.advance(sg.nh, prm);
    }
  } else if (warp < kPollWarp) {
    // ------------------------ epilogue: y = Y1 + 2^cs2_i Y2 -> staging -> TMA store of y
    // (D x already sits in Y1 through P's diagonal)
    const int q = warp & 3, r = 32 * q + lane;
    const uint32_t trow = tmem + (uint32_t(32 * q) << 16);
    const bool store_thread = warp == 2 + kMaskWarps && lane == 0;
    uint32_t gi = 0;
    grid_dep_wait();  // cs2 comes from the previous kernels
    for (SegWalk w = walk0; w.more();) {
      const Segment sg = w.seg(prm);
      const int i0 = sg.mt * 128, row = i0 + r;
      const bool tile_live = int64_t(sg.c) * Q + i0 < prm.L;
      for (int hi = 0; hi < sg.nh; ++hi, ++gi) {
        const int hh = sg.h_begin + hi;
        const uint32_t s = gi & 1;
        // this row's cs2 (one coalesced L2 read per warp), fetched while the MMAs finish
        const float cs_i = __ldg(prm.cs2 + ((int64_t(sg.b) * H + hh) * prm.nc + sg.c) * Q + row);
        // WIDE: the head's Z rows (2^{cs2_i} C hprev^T, from the readout) in the hprev slot
        const bool zok = !WIDE || mbar_wait(bar(kHpFull0 + s), (gi >> 1) & 1, ctl);
        const bool ok = mbar_wait(bar(kYFull0 + s), (gi >> 1) & 1, ctl) && zok && !*abort_flag;
        tc_fence_after();
        if (store_thread) bulk_wait_read0();  // the staging buffer is free again
        named_bar_sync(kBarEpi, 32 * kEpiWarps);
        if (ok) {
          const float e = ex2(cs_i);
          uint8_t* ys = smem + SM::kY + r * 128;
          const uint8_t* zr = smem + SM::kHp0 + s * SM::kHpBytes + r * 128;
#pragma unroll
          for (int quarter = 0; quarter < 4; ++quarter) {
            uint32_t a[16], q2[16];
            __syncwarp();
            tmem_ld16(trow + 256 + 128 * s + 16 * quarter, a);
            if (!WIDE) tmem_ld16(trow + 256 + 128 * s + 64 + 16 * quarter, q2);
            tmem_ld_wait();
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
              const int cc = 2 * quarter + c2;
              uint32_t o[4];
              if (WIDE) {
                // y = Y1 + Z (Z already carries its decay 2^{cs2_i})
                const uint4 zv = *reinterpret_cast<const uint4*>(zr + ((cc ^ (r & 7)) << 4));
                const uint32_t zw[4] = {zv.x, zv.y, zv.z, zv.w};
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                  const int k0 = 8 * c2 + 2 * e2;
                  o[e2] = pack_bf16x2(__uint_as_float(a[k0]) + bf16lo_to_f32(zw[e2]),
                                      __uint_as_float(a[k0 + 1]) + bf16hi_to_f32(zw[e2]));
                }
              } else {
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                  const int k0 = 8 * c2 + 2 * e2;
                  const float2 v2 = fma_f32x2(make_float2(e, e),
                                              make_float2(__uint_as_float(q2[k0]), __uint_as_float(q2[k0 + 1])),
                                              make_float2(__uint_as_float(a[k0]), __uint_as_float(a[k0 + 1])));
                  o[e2] = pack_bf16x2(v2.x, v2.y);
                }
              }
              *reinterpret_cast<uint4*>(ys + ((cc ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(kYEmpty0 + s));
          if (WIDE) mbar_arrive(bar(kHpEmpty0 + s));  // the Z rows have been read
        }
        fence_proxy_async_smem();
        named_bar_sync(kBarEpi, 32 * kEpiWarps);
        if (store_thread && ok && tile_live) {
          tma_store_3d(&tm_y, sb + SM::kY, hh * 64, sg.c * Q + i0, sg.b);
          bulk_commit();
        }
      }
      w.advance(sg.nh, prm);
    }
    if (store_thread) bulk_wait_read0();  // the stores have read the staging buffer
  }

  grid_dep_launch();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NB, bool WIDE>
cudaError_t launch_nb(const CUtensorMap* maps, const ScParams& prm, int grid, cudaStream_t st) {
  using SM = ScSmem<NB>;
  auto kern = chunk_scan_tc_kernel<NB, WIDE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kAlloc);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), SM::kAlloc, st, maps[0], maps[1], maps[2], maps[3],
                    maps[4], maps[5], maps[6], prm);
}

}  // namespace

bool chunk_scan_wide(const Problem& p) { return p.N > 128 && p.N % 64 == 0 && p.N >= p.Q; }

bool chunk_scan_tc_ok(const Problem& p) {
  return p.io_bf16 && p.P == 64 && (p.Q == 128 || p.Q == 256) &&
         (p.N == 64 || p.N == 128 || chunk_scan_wide(p)) && p.L <= (int64_t(1) << 31) - 1 &&
         p.b * p.nc * p.H * p.P < (int64_t(1) << 31) && p.G * p.N < (int64_t(1) << 31);
}

cudaError_t launch_chunk_scan_tc(const Problem& p, const void* x, const void* B, const void* C,
                                 const float* D, const float* cs2, const float* dtT,
                                 const void* hprev, void* zbuf, void* y, uint32_t* status, cudaStream_t st,
                                 const char** why) {
  const bool wide = chunk_scan_wide(p);
  if (wide) {
    // Z = 2^{cs2_i} C hprev^T first, into zbuf (b, L, H, P) bf16
    const cudaError_t e = launch_chunk_readout_tc(p, C, cs2, hprev, zbuf, status, st, why);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap maps[7];  // x, B, C, hprev or Z, y, x in 256-row boxes, (cs2, dt) row pairs
  const uint64_t xdims[3] = {uint64_t(p.H * p.P), uint64_t(p.L), uint64_t(p.b)};
  const uint64_t xstr[2] = {uint64_t(p.H * p.P * 2), uint64_t(p.L * p.H * p.P * 2)};
  const uint64_t bdims[3] = {uint64_t(p.G * p.N), uint64_t(p.L), uint64_t(p.b)};
  const uint64_t bstr[2] = {uint64_t(p.G * p.N * 2), uint64_t(p.L * p.G * p.N * 2)};
  const uint32_t box3[3] = {64, 128, 1};
  // hprev (rows p of each (b, c, h), N columns) as (64 columns, rows, N / 64 column halves), so
  // that one box {64, 64, N / 64} lands as N / 64 swizzled 8 KB tiles
  const uint64_t hdims[3] = {64, uint64_t(p.b * p.nc * p.H * p.P), uint64_t(wide ? 2 : p.N / 64)};
  const uint64_t hstr[2] = {uint64_t(p.N * 2), 128};
  const uint32_t hbox[3] = {64, 64, uint32_t(wide ? 2 : p.N / 64)};
  if (!encode_tmap(&maps[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, xdims, xstr, box3,
                   CU_TENSOR_MAP_SWIZZLE_128B, why) ||
      !encode_tmap(&maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, B, bdims, bstr, box3,
                   CU_TENSOR_MAP_SWIZZLE_128B, why) ||
      !encode_tmap(&maps[2], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, C, bdims, bstr, box3,
                   CU_TENSOR_MAP_SWIZZLE_128B, why) ||
      !(wide ? encode_tmap(&maps[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, zbuf, xdims, xstr, box3,
                           CU_TENSOR_MAP_SWIZZLE_128B, why)
             : encode_tmap(&maps[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, hprev, hdims, hstr, hbox,
                           CU_TENSOR_MAP_SWIZZLE_128B, why)) ||
      !encode_tmap(&maps[4], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, y, xdims, xstr, box3,
                   CU_TENSOR_MAP_SWIZZLE_128B, why))
    return cudaErrorInvalidValue;
  if (p.Q == 256) {
    const uint32_t box256[3] = {64, 256, 1};
    if (!encode_tmap(&maps[5], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, xdims, xstr, box256,
                     CU_TENSOR_MAP_SWIZZLE_128B, why))
      return cudaErrorInvalidValue;
  } else {
    maps[5] = maps[0];  // never used: every head is 128 rows wide
  }
  {
    // cs2 and dtT (b, H, nc, Q) float32 as one (Q, b H nc, 2) view: the dt array sits at a fixed
    // byte distance after the cs2 array, so one box {Q, 1, 2} brings a head's two rows
    const int64_t gap = reinterpret_cast<const char*>(dtT) - reinterpret_cast<const char*>(cs2);
    const int64_t rows = p.b * p.H * p.nc;
    if (gap < rows * p.Q * 4 || gap % 16 != 0) {
      if (why) *why = "chunk_scan needs the dt array after the cs2 array (the workspace layout)";
      return cudaErrorInvalidValue;
    }
    const uint64_t dims[3] = {uint64_t(p.Q), uint64_t(rows), 2};
    const uint64_t strides[2] = {uint64_t(p.Q * 4), uint64_t(gap)};
    const uint32_t box[3] = {uint32_t(p.Q), 1, 2};
    if (!encode_tmap(&maps[6], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, cs2, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE, why))
      return cudaErrorInvalidValue;
  }
  ScParams prm;
  prm.L = static_cast<int32_t>(p.L);
  prm.H = static_cast<int32_t>(p.H);
  prm.nc = static_cast<int32_t>(p.nc);
  prm.Q = static_cast<int32_t>(p.Q);
  prm.N = static_cast<int32_t>(p.N);
  prm.hpg = static_cast<int32_t>(p.hpg);
  prm.MT = static_cast<int32_t>(p.Q / 128);
  prm.units = p.b * p.nc * prm.MT * p.H;
  prm.total_weight = p.b * p.nc * p.H * (prm.MT == 2 ? kWeightMt0 + kWeightMt1 : 1);
  prm.cs2 = cs2;
  prm.dtT = dtT;
  prm.D = D;
  prm.status = status;
  prm.wait_ns = kWaitLimitNs;
  int sms = num_sms_current_device();
  if (sms <= 0) sms = 1;
  const int grid = static_cast<int>(prm.units < sms ? prm.units : sms);
  if (wide) return launch_nb<2, true>(maps, prm, grid, st);
  if (p.N == 64) return launch_nb<1, false>(maps, prm, grid, st);
  return launch_nb<2, false>(maps, prm, grid, st);
}

}  // namespace ssd
