// ssd_internal.h -- problem description, workspace layout and kernel launchers shared by the
// translation units of libssd.so.  Host-side only declarations; no torch types anywhere.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssd {

// One problem, with every size the kernels need precomputed on the host.
struct Problem {
  int64_t b, L, H, P, N, G, Q;
  int64_t nc;      // number of chunks, ceil(L / Q)
  int64_t hpg;     // heads per group, H / G
  bool io_bf16;    // x, B, C, y are bf16 (else f32); hprev has the same element type
  uint32_t flags;  // SSD_FLAG_*
};

// Mamba-1 selective scan: x, delta, y (b, L, D); B, C (b, L, N); A (D, N).
struct SelProblem {
  int64_t b, L, D, N;
  bool io_bf16;
};

// Byte offsets inside the caller's workspace.  Each region is 1024-byte aligned.
struct Layout {
  size_t status, cs2, dtT, S, hprev, total;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline Layout make_layout(const Problem& p) {
  Layout l{};
  const size_t cs_bytes = static_cast<size_t>(p.b * p.H * p.nc * p.Q) * 4u;
  const size_t st_elems = static_cast<size_t>(p.b * p.nc * p.H * p.P * p.N);
  l.status = 0;
  l.cs2 = 1024;
  l.dtT = align_up(l.cs2 + cs_bytes, 1024);
  l.S = align_up(l.dtT + cs_bytes, 1024);
  l.hprev = align_up(l.S + st_elems * (p.io_bf16 ? 2u : 4u), 1024);
  l.total = align_up(l.hprev + st_elems * (p.io_bf16 ? 2u : 4u), 1024);
  return l;
}

// Launches `kern` on `st`, with programmatic stream serialization when `pdl`: the kernel may
// begin (its prologue: barrier init, tensor-memory allocation, tensor-map prefetch) while the
// previous kernel in the stream is finishing, and waits in grid_dep_wait() before touching
// global memory.  Without it the launch waits for the previous kernel as usual, and the
// kernel's grid_dep_wait / grid_dep_launch do nothing.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  return launch_kernel(true, kern, grid, block, smem, st, args...);
}

// Default limit of one bounded on-chip wait (ns).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// ---- launchers (each returns the launch's cudaError_t; none synchronises) ----

// chunk_cumsum stages dt tiles by TMA when chunk_cumsum_tma_ok (rows 16-byte aligned); its
// bounded waits report SSD_ERR_TIMEOUT in *status.
bool chunk_cumsum_tma_ok(const Problem& p, const float* dt);
cudaError_t launch_chunk_cumsum(const Problem& p, const float* dt, const float* A, float* cs2,
                                float* dtT, uint32_t* status, cudaStream_t st, bool unit_scale = false);

// pdl: launch with programmatic dependent launch (see launch_kernel).
cudaError_t launch_state_passing(const Problem& p, const void* S, const float* cs2,
                                 const float* init, void* hprev, float* final_state,
                                 cudaStream_t st, bool pdl = true);

cudaError_t launch_chunk_state_simt(const Problem& p, const void* x, const void* B, const float* cs2,
                                    const float* dtT, void* S, cudaStream_t st);

cudaError_t launch_chunk_scan_simt(const Problem& p, const void* x, const void* B, const void* C,
                                   const float* D, const float* cs2, const float* dtT,
                                   const void* hprev, void* y, cudaStream_t st);

// Backward pass: the steps between its scans (backward.cu).
cudaError_t launch_flip_expand(const void* src, void* dst, int64_t b, int64_t L, int64_t Hsrc, int64_t Hdst,
                               int64_t src_row_bytes, int64_t col_byte0, int64_t dst_row_bytes, bool flip,
                               cudaStream_t st);
cudaError_t launch_widen_flip_expand(const void* src, float* dst, int64_t b, int64_t L, int64_t Hsrc, int64_t Hdst,
                                     int64_t F, bool flip, bool src_bf16, cudaStream_t st);
cudaError_t launch_reverse_decay(const float* dt, float* out, int64_t b, int64_t L, int64_t H, cudaStream_t st);
cudaError_t launch_transpose_state(const float* src, float* dst, int64_t rows, int64_t P, int64_t N, int64_t n0,
                                   int64_t Nk, cudaStream_t st);
cudaError_t launch_bwd_combine(const Problem& p, const void* dy, const void* x, const float* yssm, const float* gB_rev,
                               const float* dt, const float* D, void* dx, float* dcs, float* xgB, float* dyx,
                               cudaStream_t st);
cudaError_t launch_bwd_scalars(const Problem& p, const float* dfinal, const float* fin, const float* xgB,
                               const float* dyx, const float* dt, const float* A, float* dcs, float* ddt,
                               float* part, float* dA, float* dD, cudaStream_t st);
cudaError_t launch_group_sum(const Problem& p, const void* y, const float* dt, void* out, int64_t n0, int64_t Nk,
                             bool flip, cudaStream_t st);
cudaError_t launch_dinit(const Problem& p, const float* g0, const float* dt, const float* A, float* dinit,
                         cudaStream_t st);

// Mamba-1 selective scan (fused zero-order hold + scan + read-out); applicability by selective_ok.
bool selective_ok(const SelProblem& p);
cudaError_t launch_selective_scan(const SelProblem& p, const void* x, const void* delta, const float* A,
                                  const void* B, const void* C, const float* Dskip, const float* init,
                                  float* final_state, void* y, cudaStream_t st);

// Recurrent form over a short run of tokens (decoding); applicability by decode_ok.
bool decode_ok(const Problem& p);
cudaError_t launch_decode(const Problem& p, const void* x, const float* dt, const float* A,
                          const void* B, const void* C, const float* D, float* state, void* y,
                          cudaStream_t st);

// Tensor-core (tcgen05) kernels.  Applicability is decided by the *_tc_ok predicates.
bool chunk_state_tc_ok(const Problem& p);
// Whether launch_chunk_state_tc runs its persistent kernel for p (many items per SM).
bool chunk_state_tc_persistent(const Problem& p);
bool chunk_scan_tc_ok(const Problem& p);

cudaError_t launch_chunk_state_tc(const Problem& p, const void* x, const void* B, const float* cs2,
                                  const float* dtT, void* S, uint32_t* status, cudaStream_t st,
                                  const char** why);

// fwd_pass_state in one kernel (chunk_state's persistent kernel walking whole chains, each
// chain's float32 state kept in tensor memory): writes hprev and final_state directly, no S and
// no state_passing launch.  Shapes: chunk_state_fused_ok (the tensor-core chunk_state shapes with
// N <= 128); it uses one CTA per (batch, head pair) chain.  Selected only on request
// (SSD_FLAG_FUSED_STATE): with one SM per chain it is slower than the two kernels on the
// workloads measured.
bool chunk_state_fused_ok(const Problem& p);
cudaError_t launch_chunk_state_fused(const Problem& p, const void* x, const void* B, const float* cs2,
                                     const float* dtT, const float* init, void* hprev, float* final_state,
                                     uint32_t* status, cudaStream_t st, const char** why);

// States above 128 columns (chunk_scan_wide): the readout kernel computes the term through
// hprev, Z = 2^{cs2_i} C hprev^T (b, L, H, P) bf16, into zbuf (which needs b * nc * Q * H * P
// bf16 elements: the S region serves, S being dead after state_passing and no smaller when
// N >= Q), then chunk_scan adds it.
bool chunk_scan_wide(const Problem& p);
bool chunk_readout_tc_ok(const Problem& p);
cudaError_t launch_chunk_readout_tc(const Problem& p, const void* C, const float* cs2, const void* hprev,
                                    void* Z, uint32_t* status, cudaStream_t st, const char** why);

cudaError_t launch_chunk_scan_tc(const Problem& p, const void* x, const void* B, const void* C,
                                 const float* D, const float* cs2, const float* dtT,
                                 const void* hprev, void* zbuf, void* y, uint32_t* status,
                                 cudaStream_t st, const char** why);

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t timeout_ns, cudaStream_t st);

// Tensor-map encoder (driver entry point resolved once through the runtime).
// rank 2 or 3; dims/box innermost first; strides in bytes for dims 1..rank-1.
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                 CUtensorMapSwizzle swizzle, const char** why);

int num_sms_current_device();

}  // namespace ssd
