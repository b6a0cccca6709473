// state_passing -- step 3 of the SSD forward scan.
//
// "Mamba-2 cuda-tile forward pass kernels" (devotd.net), section 2: the second kernel
// produces the hidden state at the start of every chunk and the state after the last chunk,
// keeping chunk order while independent pieces of the state run in parallel.  Per element
// (b, h, p, n) of the P x N state:
//     hprev[c] = h_{c-1},   h_c = 2^{cs2_last(c)} * h_{c-1} + S_c,   h_{-1} = init (or 0),
//     final    = h_{nc-1}
// where cs2_last(c) is the log2-domain decay of the whole chunk (the last entry of the
// chunk_cumsum row; zero padding past the sequence end leaves it unchanged).
//
// The loop over chunks is a dependent FMA chain per element, so the kernel is bound by HBM
// latency x bandwidth: each thread owns consecutive state elements -- 8 (one 16-byte load of S
// per chunk) when S is bf16, 4 when it is float32 -- and loads the chunks in batches of K: all K
// loads of a batch are issued together (with the next batch's issued before this one is
// consumed, where registers allow), then the K chain steps run.  A ring that refills one entry
// per chunk keeps as many loads in flight on paper, but a warp tracks its outstanding loads in a
// handful of dependency counters, so waiting for the oldest entry of the ring also waits for
// loads issued just before it: measured on GB300 at 256K tokens, rings of 8 to 32 chunks all ran
// at 1.9 TB/s, batches of 16 at 6.5 TB/s (a plain copy of the same bytes: 6.5 TB/s).
// The chain itself runs in float32.
#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kVec4Batch = 8;
// bf16x8 kernel: 64-thread CTAs.  Each thread walks all chunks of its column, so the columns
// must fit in one wave of evenly loaded SMs (a second, partial wave would take as long as the
// first); within that, the batch is as large as the registers allow.  Few columns (long
// sequences, small states): batches of 16 with the next batch in flight (<= 4 CTAs per SM);
// layers: batches of 8 (<= 12 CTAs per SM) or 4 (<= 18 CTAs per SM).
constexpr int kBf16x8Threads = 64;

__device__ __forceinline__ void store4(float* dst, float4 v) { *reinterpret_cast<float4*>(dst) = v; }
__device__ __forceinline__ float4 load4(const float* src) { return __ldcs(reinterpret_cast<const float4*>(src)); }
__device__ __forceinline__ float4 load4(const uint16_t* src) {
  const uint2 u = __ldcs(reinterpret_cast<const uint2*>(src));
  return make_float4(bf16lo_to_f32(u.x), bf16hi_to_f32(u.x), bf16lo_to_f32(u.y), bf16hi_to_f32(u.y));
}
__device__ __forceinline__ float load1(const float* src) { return __ldg(src); }
__device__ __forceinline__ float load1(const uint16_t* src) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(src)) << 16);
}
__device__ __forceinline__ void store4(uint16_t* dst, float4 v) {
  uint2 u;
  u.x = pack_bf16x2(v.x, v.y);
  u.y = pack_bf16x2(v.z, v.w);
  *reinterpret_cast<uint2*>(dst) = u;
}

// bf16 S / hprev, 8 elements per thread, chunks in batches of K (PF: the next batch's loads are
// issued before the current batch is consumed).
template <int K, bool PF, int MIN_CTAS>
__global__ void __launch_bounds__(kBf16x8Threads, MIN_CTAS) state_passing_bf16x8_kernel(
    const uint16_t* __restrict__ S, const float* __restrict__ cs2, const float* __restrict__ init,
    uint16_t* __restrict__ hprev, float* __restrict__ final_state, int64_t H, int64_t PN,
    int64_t nc, int64_t Q, int64_t total8) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  grid_dep_wait();  // S and cs2 come from the previous kernels
  if (idx >= total8) {
    grid_dep_launch();
    return;
  }
  const int64_t per_bh = PN / 8;
  const int64_t bh = idx / per_bh, e = (idx % per_bh) * 8;
  const int64_t bi = bh / H, h = bh % H;
  const int64_t cstride = H * PN;  // elements between chunks in S / hprev
  uint16_t* Hp = hprev + (bi * nc * H + h) * PN + e;
  const uint16_t* Sp = S + (bi * nc * H + h) * PN + e;
  const float* dp = cs2 + bh * nc * Q + (Q - 1);
  const int n = static_cast<int>(nc);

  float hv[8];
  if (init) {
    const float4 a0 = __ldg(reinterpret_cast<const float4*>(init + bh * PN + e));
    const float4 a1 = __ldg(reinterpret_cast<const float4*>(init + bh * PN + e + 4));
    hv[0] = a0.x; hv[1] = a0.y; hv[2] = a0.z; hv[3] = a0.w;
    hv[4] = a1.x; hv[5] = a1.y; hv[6] = a1.z; hv[7] = a1.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) hv[i] = 0.f;
  }
  uint4 sb[K], nb[K];
  float db[K], nd[K];
  // Sp / dp always point at the next chunk to load
  auto load_batch = [&](uint4 (&sv)[K], float (&dv)[K], int c0) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (c0 + k < n) {
        sv[k] = __ldcs(reinterpret_cast<const uint4*>(Sp));
        dv[k] = __ldg(dp);
        Sp += cstride;
        dp += Q;
      }
    }
  };
  if (PF) load_batch(nb, nd, 0);
  for (int c0 = 0; c0 < n; c0 += K) {
    if (PF) {
#pragma unroll
      for (int k = 0; k < K; ++k) {
        sb[k] = nb[k];
        db[k] = nd[k];
      }
      if (c0 + K < n) load_batch(nb, nd, c0 + K);
    } else {
      load_batch(sb, db, c0);
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int c = c0 + k;
      if (c < n) {
        uint4 o;
        o.x = pack_bf16x2(hv[0], hv[1]);
        o.y = pack_bf16x2(hv[2], hv[3]);
        o.z = pack_bf16x2(hv[4], hv[5]);
        o.w = pack_bf16x2(hv[6], hv[7]);
        *reinterpret_cast<uint4*>(Hp) = o;
        Hp += cstride;
        const float d = ex2(db[k]);
        hv[0] = fmaf(d, hv[0], bf16lo_to_f32(sb[k].x));
        hv[1] = fmaf(d, hv[1], bf16hi_to_f32(sb[k].x));
        hv[2] = fmaf(d, hv[2], bf16lo_to_f32(sb[k].y));
        hv[3] = fmaf(d, hv[3], bf16hi_to_f32(sb[k].y));
        hv[4] = fmaf(d, hv[4], bf16lo_to_f32(sb[k].z));
        hv[5] = fmaf(d, hv[5], bf16hi_to_f32(sb[k].z));
        hv[6] = fmaf(d, hv[6], bf16lo_to_f32(sb[k].w));
        hv[7] = fmaf(d, hv[7], bf16hi_to_f32(sb[k].w));
      }
    }
  }
  if (final_state) {
    *reinterpret_cast<float4*>(final_state + bh * PN + e) = make_float4(hv[0], hv[1], hv[2], hv[3]);
    *reinterpret_cast<float4*>(final_state + bh * PN + e + 4) = make_float4(hv[4], hv[5], hv[6], hv[7]);
  }
  grid_dep_launch();
}

template <typename HT>
__global__ void __launch_bounds__(256, 4) state_passing_vec4_kernel(
    const HT* __restrict__ S, const float* __restrict__ cs2, const float* __restrict__ init,
    HT* __restrict__ hprev, float* __restrict__ final_state, int64_t H, int64_t PN, int64_t nc,
    int64_t Q, int64_t total4) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  grid_dep_wait();  // S and cs2 come from the previous kernels
  if (idx >= total4) {
    grid_dep_launch();
    return;
  }
  const int64_t per_bh = PN / 4;
  const int64_t bh = idx / per_bh, e = (idx % per_bh) * 4;
  const int64_t bi = bh / H, h = bh % H;
  const int64_t cstride = H * PN;  // elements between chunks in S / hprev
  HT* Hp = hprev + (bi * nc * H + h) * PN + e;
  const int n = static_cast<int>(nc);

  float4 hv = init ? __ldg(reinterpret_cast<const float4*>(init + bh * PN + e))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 sbuf[kVec4Batch];
  float dbuf[kVec4Batch];
  const HT* sp = S + (bi * nc * H + h) * PN + e;
  const float* dp = cs2 + bh * nc * Q + (Q - 1);
  for (int c0 = 0; c0 < n; c0 += kVec4Batch) {
    // one batch of loads in flight together, then its chain steps
#pragma unroll
    for (int k = 0; k < kVec4Batch; ++k) {
      if (c0 + k < n) {
        sbuf[k] = load4(sp);
        dbuf[k] = __ldg(dp);
        sp += cstride;
        dp += Q;
      }
    }
#pragma unroll
    for (int k = 0; k < kVec4Batch; ++k) {
      if (c0 + k < n) {
        store4(Hp, hv);
        Hp += cstride;
        const float d = ex2(dbuf[k]);
        hv.x = fmaf(d, hv.x, sbuf[k].x);
        hv.y = fmaf(d, hv.y, sbuf[k].y);
        hv.z = fmaf(d, hv.z, sbuf[k].z);
        hv.w = fmaf(d, hv.w, sbuf[k].w);
      }
    }
  }
  if (final_state) *reinterpret_cast<float4*>(final_state + bh * PN + e) = hv;
  grid_dep_launch();
}

__device__ __forceinline__ void store1(float* dst, float v) { *dst = v; }
__device__ __forceinline__ void store1(uint16_t* dst, float v) {
  *dst = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu);
}

// Any P*N: one element per thread, no vectorisation.
template <typename HT>
__global__ void __launch_bounds__(256) state_passing_scalar_kernel(
    const HT* __restrict__ S, const float* __restrict__ cs2, const float* __restrict__ init,
    HT* __restrict__ hprev, float* __restrict__ final_state, int64_t H, int64_t PN, int64_t nc,
    int64_t Q, int64_t total) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  grid_dep_wait();
  if (idx >= total) {
    grid_dep_launch();
    return;
  }
  const int64_t bh = idx / PN, e = idx % PN;
  const int64_t bi = bh / H, h = bh % H;
  const int64_t cstride = H * PN;
  const HT* Sp = S + (bi * nc * H + h) * PN + e;
  HT* Hp = hprev + (bi * nc * H + h) * PN + e;
  const float* dec = cs2 + bh * nc * Q + (Q - 1);
  float hv = init ? __ldg(init + bh * PN + e) : 0.f;
  for (int64_t c = 0; c < nc; ++c) {
    store1(Hp + c * cstride, hv);
    hv = fmaf(ex2(__ldg(dec + c * Q)), hv, load1(Sp + c * cstride));
  }
  if (final_state) final_state[bh * PN + e] = hv;
  grid_dep_launch();
}

}  // namespace

cudaError_t launch_state_passing(const Problem& p, const void* S, const float* cs2,
                                 const float* init, void* hprev, float* final_state,
                                 cudaStream_t st, bool pdl) {
  const int64_t PN = p.P * p.N;
  if (p.io_bf16 && PN % 8 == 0) {
    const int64_t total8 = p.b * p.H * (PN / 8);
    const unsigned blocks8 = static_cast<unsigned>((total8 + kBf16x8Threads - 1) / kBf16x8Threads);
    int sms = num_sms_current_device();
    if (sms <= 0) sms = 1;
    const int64_t ctas_per_sm = (int64_t(blocks8) + sms - 1) / sms;
    const auto Sb = static_cast<const uint16_t*>(S);
    const auto hb = static_cast<uint16_t*>(hprev);
    if (ctas_per_sm <= 4)
      return launch_kernel(pdl, state_passing_bf16x8_kernel<16, true, 4>, dim3(blocks8), dim3(kBf16x8Threads), 0, st, Sb,
                        cs2, init, hb, final_state, p.H, PN, p.nc, p.Q, total8);
    if (ctas_per_sm <= 12)
      return launch_kernel(pdl, state_passing_bf16x8_kernel<8, false, 12>, dim3(blocks8), dim3(kBf16x8Threads), 0, st, Sb,
                        cs2, init, hb, final_state, p.H, PN, p.nc, p.Q, total8);
    return launch_kernel(pdl, state_passing_bf16x8_kernel<4, false, 18>, dim3(blocks8), dim3(kBf16x8Threads), 0, st, Sb,
                      cs2, init, hb, final_state, p.H, PN, p.nc, p.Q, total8);
  }
  const bool vec = (PN % 4) == 0;
  const int64_t total = p.b * p.H * (vec ? PN / 4 : PN);
  const unsigned blocks = static_cast<unsigned>((total + 255) / 256);
  if (vec) {
    if (p.io_bf16)
      return launch_kernel(pdl, state_passing_vec4_kernel<uint16_t>, dim3(blocks), dim3(256), 0, st, static_cast<const uint16_t*>(S), cs2,
                        init, static_cast<uint16_t*>(hprev), final_state, p.H, PN, p.nc, p.Q, total);
    else
      return launch_kernel(pdl, state_passing_vec4_kernel<float>, dim3(blocks), dim3(256), 0, st, static_cast<const float*>(S), cs2,
                        init, static_cast<float*>(hprev), final_state, p.H, PN, p.nc, p.Q, total);
  } else {
    if (p.io_bf16)
      return launch_kernel(pdl, state_passing_scalar_kernel<uint16_t>, dim3(blocks), dim3(256), 0, st, static_cast<const uint16_t*>(S), cs2,
                        init, static_cast<uint16_t*>(hprev), final_state, p.H, PN, p.nc, p.Q, total);
    else
      return launch_kernel(pdl, state_passing_scalar_kernel<float>, dim3(blocks), dim3(256), 0, st, static_cast<const float*>(S), cs2,
                        init, static_cast<float*>(hprev), final_state, p.H, PN, p.nc, p.Q, total);
  }
  return cudaGetLastError();
}

}  // namespace ssd
