// ssd_api.cu -- the C ABI of include/ssd.h: argument checks, workspace carving, tensor-map
// encoding and kernel dispatch.  Host code only (plus the wait self-test kernel).
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "ssd.h"
#include "ptx.cuh"
#include "ssd_internal.h"

namespace {

thread_local char g_last_error[256] = "";

ssd_status fail(ssd_status s, const char* fmt, const char* arg = nullptr) {
  std::snprintf(g_last_error, sizeof g_last_error, fmt, arg ? arg : "");
  return s;
}

ssd_status cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_last_error, sizeof g_last_error, "%s: %s", where, cudaGetErrorString(e));
  return SSD_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ssd_status make_problem(const ssd_shape* s, ssd::Problem* p) {
  if (!s) return fail(SSD_ERR_INVALID, "shape is null");
  if (s->batch < 1 || s->seqlen < 1 || s->nheads < 1 || s->headdim < 1 || s->dstate < 1 ||
      s->ngroups < 1)
    return fail(SSD_ERR_INVALID, "every dimension must be >= 1");
  if (s->nheads % s->ngroups != 0) return fail(SSD_ERR_INVALID, "nheads must be a multiple of ngroups");
  if (s->chunk != 64 && s->chunk != 128 && s->chunk != 256)
    return fail(SSD_ERR_INVALID, "chunk must be 64, 128 or 256");
  if (s->io_dtype != SSD_F32 && s->io_dtype != SSD_BF16) return fail(SSD_ERR_INVALID, "bad io_dtype");
  // keep every flattened index inside int32 grid limits and int64 element offsets
  const int64_t nc = (s->seqlen + s->chunk - 1) / s->chunk;
  if (s->batch > 65535 || s->nheads > 65535 || nc > (int64_t(1) << 30) ||
      s->headdim > 4096 || s->dstate > 4096)
    return fail(SSD_ERR_UNSUPPORTED, "dimension beyond the supported range");
  const double elems = double(s->batch) * double(nc) * double(s->nheads) * double(s->headdim) *
                       double(s->dstate);
  if (elems > 4.0e11) return fail(SSD_ERR_UNSUPPORTED, "state tensors too large");
  p->b = s->batch;
  p->L = s->seqlen;
  p->H = s->nheads;
  p->P = s->headdim;
  p->N = s->dstate;
  p->G = s->ngroups;
  p->Q = s->chunk;
  p->nc = nc;
  p->hpg = s->nheads / s->ngroups;
  p->io_bf16 = s->io_dtype == SSD_BF16;
  p->flags = s->flags;
  return SSD_OK;
}

struct Views {
  uint32_t* status;
  float* cs2;
  float* dtT;
  void* S;  // per-chunk states, in the I/O dtype
  void* hprev;
};

ssd_status carve(const ssd::Problem& p, void* ws, size_t ws_bytes, Views* v) {
  const ssd::Layout l = ssd::make_layout(p);
  if (!ws) return fail(SSD_ERR_WORKSPACE, "workspace is null");
  if (ws_bytes < l.total) return fail(SSD_ERR_WORKSPACE, "workspace smaller than ssd_workspace_bytes()");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(SSD_ERR_ALIGN, "workspace must be 256-byte aligned");
  char* base = static_cast<char*>(ws);
  v->status = reinterpret_cast<uint32_t*>(base + l.status);
  v->cs2 = reinterpret_cast<float*>(base + l.cs2);
  v->dtT = reinterpret_cast<float*>(base + l.dtT);
  v->S = base + l.S;
  v->hprev = base + l.hprev;
  return SSD_OK;
}

bool use_state_tc(const ssd::Problem& p) {
  return !(p.flags & SSD_FLAG_FORCE_SIMT) && ssd::chunk_state_tc_ok(p);
}
bool use_scan_tc(const ssd::Problem& p) {
  return !(p.flags & SSD_FLAG_FORCE_SIMT) && ssd::chunk_scan_tc_ok(p);
}

// Why a step of p would run on the CUDA-core kernels (null: it runs on the tensor cores).
const char* simt_reason(const ssd::Problem& p, bool scan) {
  if (p.flags & SSD_FLAG_FORCE_SIMT) return "SSD_FLAG_FORCE_SIMT is set";
  if (!p.io_bf16) return "float32 I/O";
  if (p.P != 64) return "headdim is not 64";
  if (p.Q != 128 && p.Q != 256) return "chunk is not 128 or 256";
  if (scan ? !ssd::chunk_scan_tc_ok(p) : !ssd::chunk_state_tc_ok(p))
    return scan ? "dstate is not 64, 128, or a multiple of 64 above 128 and at least chunk"
                : "dstate is not 64, 128, 256 or 512";
  return nullptr;
}

// SSD_FLAG_REQUIRE_TENSOR_CORES: SSD_ERR_UNSUPPORTED when a requested step would fall back.
ssd_status require_tc(const ssd::Problem& p, bool state, bool scan) {
  if (!(p.flags & SSD_FLAG_REQUIRE_TENSOR_CORES)) return SSD_OK;
  const char* why = state ? simt_reason(p, false) : nullptr;
  if (!why && scan) why = simt_reason(p, true);
  return why ? fail(SSD_ERR_UNSUPPORTED, "no tensor-core kernel for this shape: %s", why) : SSD_OK;
}

// ---- the four steps on an already checked problem ----

ssd_status step_cumsum(const ssd::Problem& p, const float* dt, const float* A, const Views& v,
                       cudaStream_t st, bool unit_scale = false) {
  const cudaError_t e = ssd::launch_chunk_cumsum(p, dt, A, v.cs2, v.dtT, v.status, st, unit_scale);
  return e == cudaSuccess ? SSD_OK : cuda_fail(e, "chunk_cumsum launch");
}

ssd_status step_state(const ssd::Problem& p, const void* x, const void* B, const Views& v,
                      cudaStream_t st) {
  cudaError_t e;
  if (use_state_tc(p)) {
    const char* why = nullptr;
    e = ssd::launch_chunk_state_tc(p, x, B, v.cs2, v.dtT, v.S, v.status, st, &why);
    if (why) return fail(SSD_ERR_CUDA, "chunk_state: %s", why);
  } else {
    e = ssd::launch_chunk_state_simt(p, x, B, v.cs2, v.dtT, v.S, st);
  }
  return e == cudaSuccess ? SSD_OK : cuda_fail(e, "chunk_state launch");
}

ssd_status step_passing(const ssd::Problem& p, const float* init, float* final_state,
                        const Views& v, cudaStream_t st) {
  // state_passing starts early (programmatic dependent launch) only behind the one-CTA-per-item
  // chunk_state: behind the persistent chunk_state the early launch measured slower (256K tokens:
  // 1293 against 1224 us a step; 2.7B layer: 211 against 206 us; 130M layer: 47.4 against 48.4
  // with it on)
  const bool pdl = !(use_state_tc(p) && ssd::chunk_state_tc_persistent(p));
  const cudaError_t e = ssd::launch_state_passing(p, v.S, v.cs2, init, v.hprev, final_state, st, pdl);
  return e == cudaSuccess ? SSD_OK : cuda_fail(e, "state_passing launch");
}

// fwd_pass_state as one kernel, on request only.  It runs one CTA per (batch, head pair) chain,
// and a CTA of chunk_state's pipeline moves a chunk's x and B at about the per-SM share of HBM
// bandwidth, so with fewer chains than SMs the separate chunk_state (over every (chunk, head
// pair)) and state_passing finish first on every workload measured.
bool use_fused_state(const ssd::Problem& p) {
  return use_state_tc(p) && ssd::chunk_state_fused_ok(p) && (p.flags & SSD_FLAG_FUSED_STATE) &&
         !(p.flags & SSD_FLAG_SEPARATE_STATE_PASSING);
}

// chunk_state + state_passing, fused where use_fused_state says so.
ssd_status step_state_passing(const ssd::Problem& p, const void* x, const void* B, const float* init,
                              float* final_state, const Views& v, cudaStream_t st) {
  if (!use_fused_state(p)) {
    const ssd_status s1 = step_state(p, x, B, v, st);
    return s1 != SSD_OK ? s1 : step_passing(p, init, final_state, v, st);
  }
  const char* why = nullptr;
  const cudaError_t e = ssd::launch_chunk_state_fused(p, x, B, v.cs2, v.dtT, init, v.hprev, final_state,
                                                      v.status, st, &why);
  if (why) return fail(SSD_ERR_CUDA, "fwd_pass_state: %s", why);
  return e == cudaSuccess ? SSD_OK : cuda_fail(e, "fwd_pass_state launch");
}

ssd_status step_scan(const ssd::Problem& p, const void* x, const void* B, const void* C,
                     const float* D, void* y, const Views& v, cudaStream_t st) {
  cudaError_t e;
  if (use_scan_tc(p)) {
    const char* why = nullptr;
    e = ssd::launch_chunk_scan_tc(p, x, B, C, D, v.cs2, v.dtT, v.hprev, v.S, y, v.status, st, &why);
    if (why) return fail(SSD_ERR_CUDA, "chunk_scan: %s", why);
  } else {
    e = ssd::launch_chunk_scan_simt(p, x, B, C, D, v.cs2, v.dtT, v.hprev, y, st);
  }
  return e == cudaSuccess ? SSD_OK : cuda_fail(e, "chunk_scan launch");
}

#define SSD_TRY(expr)                  \
  do {                                 \
    const ssd_status s_ = (expr);      \
    if (s_ != SSD_OK) return s_;       \
  } while (0)

ssd_status need(const void* p, const char* name) {
  if (!p) return fail(SSD_ERR_INVALID, "%s is null", name);
  if (!aligned16(p)) return fail(SSD_ERR_ALIGN, "%s is not 16-byte aligned", name);
  return SSD_OK;
}

ssd_status maybe(const void* p, const char* name) {
  if (p && !aligned16(p)) return fail(SSD_ERR_ALIGN, "%s is not 16-byte aligned", name);
  return SSD_OK;
}

}  // namespace

namespace ssd {

bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                 CUtensorMapSwizzle swizzle, const char** why) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  if (!fn) {
    if (why) *why = "cuTensorMapEncodeTiled is not available";
    return false;
  }
  if (rank < 1 || rank > 5) {
    if (why) *why = "tensor map rank out of range";
    return false;
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r =
      fn(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base),
         reinterpret_cast<const cuuint64_t*>(dims), reinterpret_cast<const cuuint64_t*>(strides),
         reinterpret_cast<const cuuint32_t*>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (why) *why = "cuTensorMapEncodeTiled rejected a tensor map";
    return false;
  }
  return true;
}

int num_sms_current_device() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Waits on a barrier nothing ever completes; the bounded wait gives up and records the
// timeout status, so the CTA exits normally.
__global__ void wait_selftest_kernel(uint32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  WaitCtl ctl{timeout_ns, &abort_flag, status};
  if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0, ctl);
  __syncthreads();
  // complete the phase so the barrier is left in a finished state before the CTA exits
  if (threadIdx.x == 0) mbar_arrive(smem_u32(&bar));
}

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t timeout_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace ssd

extern "C" {

size_t ssd_workspace_bytes(const ssd_shape* shape) {
  ssd::Problem p;
  if (make_problem(shape, &p) != SSD_OK) return 0;
  return ssd::make_layout(p).total;
}

ssd_status ssd_get_workspace_layout(const ssd_shape* shape, ssd_workspace_layout* out) {
  if (!out) return fail(SSD_ERR_INVALID, "out is null");
  ssd::Problem p;
  SSD_TRY(make_problem(shape, &p));
  const ssd::Layout l = ssd::make_layout(p);
  out->status = l.status;
  out->cs2 = l.cs2;
  out->dtT = l.dtT;
  out->S = l.S;
  out->hprev = l.hprev;
  out->total = l.total;
  out->nchunks = p.nc;
  return SSD_OK;
}

ssd_status ssd_fwd(const ssd_shape* shape, const void* x, const float* dt, const float* A,
                   const void* B, const void* C, const float* D, const float* init_state, void* y,
                   float* final_state, void* workspace, size_t workspace_bytes, void* stream) {
  ssd::Problem p;
  SSD_TRY(make_problem(shape, &p));
  SSD_TRY(need(x, "x"));
  SSD_TRY(need(dt, "dt"));
  SSD_TRY(need(A, "A"));
  SSD_TRY(need(B, "B"));
  SSD_TRY(need(C, "C"));
  SSD_TRY(need(y, "y"));
  SSD_TRY(maybe(D, "D"));
  SSD_TRY(maybe(init_state, "init_state"));
  SSD_TRY(maybe(final_state, "final_state"));
  SSD_TRY(require_tc(p, true, true));
  Views v;
  SSD_TRY(carve(p, workspace, workspace_bytes, &v));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = cudaMemsetAsync(v.status, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return cuda_fail(e, "status reset");
  SSD_TRY(step_cumsum(p, dt, A, v, st));
  SSD_TRY(step_state_passing(p, x, B, init_state, final_state, v, st));
  SSD_TRY(step_scan(p, x, B, C, D, y, v, st));
  g_last_error[0] = '\0';
  return SSD_OK;
}

ssd_status ssd_chunk_cumsum(const ssd_shape* shape, const float* dt, const float* A,
                            void* workspace, size_t workspace_bytes, void* stream) {
  ssd::Problem p;
  SSD_TRY(make_problem(shape, &p));
  SSD_TRY(need(dt, "dt"));
  SSD_TRY(need(A, "A"));
  Views v;
  SSD_TRY(carve(p, workspace, workspace_bytes, &v));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = cudaMemsetAsync(v.status, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return cuda_fail(e, "status reset");
  return step_cumsum(p, dt, A, v, st);
}

ssd_status ssd_chunk_state(const ssd_shape* shape, const void* x, const void* B, void* workspace,
                           size_t workspace_bytes, void* stream) {
  ssd::Problem p;
  SSD_TRY(make_problem(shape, &p));
  SSD_TRY(need(x, "x"));
  SSD_TRY(need(B, "B"));
  SSD_TRY(require_tc(p, true, false));
  Views v;
  SSD_TRY(carve(p, workspace, workspace_bytes, &v));
  return step_state(p, x, B, v, static_cast<cudaStream_t>(stream));
}

ssd_status ssd_state_passing(const ssd_shape* shape, const float* init_state, float* final_state,
                             void* workspace, size_t workspace_bytes, void* stream) {
  ssd::Problem p;
  SSD_TRY(make_problem(shape, &p));
  SSD_TRY(maybe(init_state, "init_state"));
  SSD_TRY(maybe(final_state, "final_state"));
  Views v;
  SSD_TRY(carve(p, workspace, workspace_bytes, &v));
  return step_passing(p, init_state, final_state, v, static_cast<cudaStream_t>(stream));
}

ssd_status ssd_fwd_pass_state(const ssd_shape* shape, const void* x, const void* B,
                              const float* init_state, float* final_state, void* workspace,
                              size_t workspace_bytes, void* stream) {
  ssd::Problem p;
  SSD_TRY(make_problem(shape, &p));
  SSD_TRY(need(x, "x"));
  SSD_TRY(need(B, "B"));
  SSD_TRY(maybe(init_state, "init_state"));
  SSD_TRY(maybe(final_state, "final_state"));
  SSD_TRY(require_tc(p, true, false));
  Views v;
  SSD_TRY(carve(p, workspace, workspace_bytes, &v));
  return step_state_passing(p, x, B, init_state, final_state, v, static_cast<cudaStream_t>(stream));
}

ssd_status ssd_chunk_scan(const ssd_shape* shape, const void* x, const void* B, const void* C,
                          const float* D, void* y, void* workspace, size_t workspace_bytes,
                          void* stream) {
  ssd::Problem p;
  SSD_TRY(make_problem(shape, &p));
  SSD_TRY(need(x, "x"));
  SSD_TRY(need(B, "B"));
  SSD_TRY(need(C, "C"));
  SSD_TRY(need(y, "y"));
  SSD_TRY(maybe(D, "D"));
  SSD_TRY(require_tc(p, false, true));
  Views v;
  SSD_TRY(carve(p, workspace, workspace_bytes, &v));
  return step_scan(p, x, B, C, D, y, v, static_cast<cudaStream_t>(stream));
}

ssd_status ssd_read_status(const void* workspace, void* stream) {
  if (!workspace) return fail(SSD_ERR_WORKSPACE, "workspace is null");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  uint32_t word = 0;
  e = cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (word == 0) return SSD_OK;
  if (word == ssd::kStatusTimeout) return fail(SSD_ERR_TIMEOUT, "a kernel's bounded wait expired");
  return fail(SSD_ERR_CUDA, "unknown status word");
}

ssd_status ssd_selftest_wait_timeout(uint32_t* status_word, uint64_t timeout_ns, void* stream) {
  if (!status_word) return fail(SSD_ERR_INVALID, "status_word is null");
  if (timeout_ns == 0 || timeout_ns > 1000000000ull)
    return fail(SSD_ERR_INVALID, "timeout_ns must be in (0, 1e9]");
  const cudaError_t e = ssd::launch_wait_selftest(status_word, timeout_ns, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSD_OK : cuda_fail(e, "selftest launch");
}

ssd_status ssd_decode(const ssd_shape* shape, const void* x, const float* dt, const float* A,
                      const void* B, const void* C, const float* D, float* state, void* y,
                      void* stream) {
  if (!shape) return fail(SSD_ERR_INVALID, "shape is null");
  ssd_shape s = *shape;
  s.chunk = 64;  // the recurrent form has no chunks
  ssd::Problem p;
  SSD_TRY(make_problem(&s, &p));
  SSD_TRY(need(x, "x"));
  SSD_TRY(need(dt, "dt"));
  SSD_TRY(need(A, "A"));
  SSD_TRY(need(B, "B"));
  SSD_TRY(need(C, "C"));
  SSD_TRY(need(state, "state"));
  SSD_TRY(need(y, "y"));
  SSD_TRY(maybe(D, "D"));
  if (!ssd::decode_ok(p)) return fail(SSD_ERR_UNSUPPORTED, "decode: unsupported headdim / dstate");
  const cudaError_t e = ssd::launch_decode(p, x, dt, A, B, C, D, state, y, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  g_last_error[0] = '\0';
  return SSD_OK;
}

ssd_status ssd_selective_scan(const ssd_sel_shape* shape, const void* x, const void* delta,
                              const float* A, const void* B, const void* C, const float* Dskip,
                              const float* init_state, float* final_state, void* y, void* stream) {
  if (!shape) return fail(SSD_ERR_INVALID, "shape is null");
  const ssd_sel_shape& s = *shape;
  if (s.batch < 1 || s.seqlen < 1 || s.dim < 1 || s.dstate < 1)
    return fail(SSD_ERR_INVALID, "every dimension must be >= 1");
  if (s.io_dtype != SSD_F32 && s.io_dtype != SSD_BF16) return fail(SSD_ERR_INVALID, "bad io_dtype");
  if (s.batch > 65535 || s.dim > (int64_t(1) << 20) || s.seqlen > (int64_t(1) << 31))
    return fail(SSD_ERR_UNSUPPORTED, "dimension beyond the supported range");
  ssd::SelProblem p{s.batch, s.seqlen, s.dim, s.dstate, s.io_dtype == SSD_BF16};
  SSD_TRY(need(x, "x"));
  SSD_TRY(need(delta, "delta"));
  SSD_TRY(need(A, "A"));
  SSD_TRY(need(B, "B"));
  SSD_TRY(need(C, "C"));
  SSD_TRY(need(y, "y"));
  SSD_TRY(maybe(Dskip, "Dskip"));
  SSD_TRY(maybe(init_state, "init_state"));
  SSD_TRY(maybe(final_state, "final_state"));
  if (!ssd::selective_ok(p))
    return fail(SSD_ERR_UNSUPPORTED, "selective scan: dstate must be 8, 16, 32 or 64 and dim a multiple of 64/dstate");
  const cudaError_t e = ssd::launch_selective_scan(p, x, delta, A, B, C, Dskip, init_state, final_state, y,
                                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "selective scan launch");
  g_last_error[0] = '\0';
  return SSD_OK;
}

// ---------------------------------------------------------------------------- backward

namespace {

// Regions of the backward workspace (each 256-byte aligned).
struct BwdLayout {
  size_t scan, y, fin, xin, bin, cin, dtr, init, out, fin1, dcs, xgb, dyx, part, total;
};

// The role-swapped scans (dC, dB) have head dim N and state P with one group per head.  They
// are linear in their x input, so they run as N / kSplit scans of head dim kSplit, a
// tensor-core shape, when P is 64 with bf16 I/O (else as one scan of head dim N).
constexpr int64_t kSplit = 64;
int64_t swapped_width(const ssd_shape& s) {
  return (s.io_dtype == SSD_BF16 && s.headdim == 64 && s.dstate % kSplit == 0) ? kSplit : s.dstate;
}
// The two scans that run in float32 (the forward again and the adjoint scan) take the
// CUDA-core kernels, whose in-chunk (quadratic) work grows with the chunk length: they use
// 64-token chunks whatever the forward's chunk (same arithmetic, a different blocking).
ssd_shape f32_shape(const ssd_shape& s) {
  ssd_shape t = s;
  t.io_dtype = SSD_F32;
  t.chunk = 64;
  return t;
}

ssd_shape swapped_shape(const ssd_shape& s) {
  ssd_shape t = s;
  t.headdim = swapped_width(s);
  t.dstate = s.headdim;
  t.ngroups = s.nheads;
  t.flags = s.flags;
  return t;
}

bool bwd_layout(const ssd_shape* shape, BwdLayout* l) {
  ssd::Problem p, q;
  if (make_problem(shape, &p) != SSD_OK) return false;
  const ssd_shape sw = swapped_shape(*shape);
  if (make_problem(&sw, &q) != SSD_OK) return false;
  ssd::Problem pf;      // the float32 scans
  const ssd_shape fs = f32_shape(*shape);
  if (make_problem(&fs, &pf) != SSD_OK) return false;
  const size_t e = 4;   // every scan buffer is sized for float32
  const size_t BL = size_t(p.b * p.L), PN = size_t(p.P * p.N);
  const size_t F = size_t(p.P > p.N ? p.P : p.N);
  const size_t wide = size_t(p.G * p.N > p.H * p.P ? p.G * p.N : p.H * p.P);
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o = ssd::align_up(o + bytes, 256); return at; };
  const size_t w1 = ssd::make_layout(pf).total, w2 = ssd::make_layout(q).total;
  l->scan = take(w1 > w2 ? w1 : w2);
  l->y = take(BL * p.H * p.P * e);
  l->fin = take(size_t(p.b * p.H) * PN * 4);
  l->xin = take(BL * p.H * F * e);
  l->bin = take(BL * wide * e);
  l->cin = take(BL * wide * e);
  l->dtr = take(BL * p.H * 4);
  l->init = take(size_t(p.b * p.H) * PN * 4);
  l->out = take(BL * p.H * F * e);
  l->fin1 = take(size_t(p.b * p.H) * PN * 4);
  l->dcs = take(BL * p.H * 4);
  l->xgb = take(BL * p.H * 4);
  l->dyx = take(BL * p.H * 4);
  l->part = take(size_t(p.b * p.H) * 8);
  l->total = o;
  return true;
}

// One forward scan (the four steps) of problem p over caller buffers, on workspace ws.
ssd_status run_scan(const ssd::Problem& p, void* ws, const void* x, const float* dt, const float* A,
                    const void* B, const void* C, const float* init, void* y, float* final_state,
                    bool unit_scale, cudaStream_t st) {
  Views v;
  SSD_TRY(carve(p, ws, ssd::make_layout(p).total, &v));
  SSD_TRY(step_cumsum(p, dt, A, v, st, unit_scale));
  SSD_TRY(step_state(p, x, B, v, st));
  SSD_TRY(step_passing(p, init, final_state, v, st));
  return step_scan(p, x, B, C, nullptr, y, v, st);
}

ssd_status cuda_ok(cudaError_t e, const char* where) { return e == cudaSuccess ? SSD_OK : cuda_fail(e, where); }

}  // namespace

size_t ssd_bwd_workspace_bytes(const ssd_shape* shape) {
  BwdLayout l;
  return bwd_layout(shape, &l) ? l.total : 0;
}

ssd_status ssd_bwd(const ssd_shape* shape, const void* x, const float* dt, const float* A, const void* B,
                   const void* C, const float* D, const float* init_state, const void* dy,
                   const float* dfinal, void* dx, float* ddt, float* dA, void* dB, void* dC, float* dD,
                   float* dinit, void* workspace, size_t workspace_bytes, void* stream) {
  ssd::Problem p;
  SSD_TRY(make_problem(shape, &p));
  SSD_TRY(need(x, "x"));
  SSD_TRY(need(dt, "dt"));
  SSD_TRY(need(A, "A"));
  SSD_TRY(need(B, "B"));
  SSD_TRY(need(C, "C"));
  SSD_TRY(need(dy, "dy"));
  SSD_TRY(need(dx, "dx"));
  SSD_TRY(need(ddt, "ddt"));
  SSD_TRY(need(dA, "dA"));
  SSD_TRY(need(dB, "dB"));
  SSD_TRY(need(dC, "dC"));
  SSD_TRY(maybe(D, "D"));
  SSD_TRY(maybe(init_state, "init_state"));
  SSD_TRY(maybe(dfinal, "dfinal"));
  SSD_TRY(maybe(dD, "dD"));
  SSD_TRY(maybe(dinit, "dinit"));
  BwdLayout l;
  if (!bwd_layout(shape, &l)) return fail(SSD_ERR_INVALID, "backward: bad shape");
  if (!workspace) return fail(SSD_ERR_WORKSPACE, "workspace is null");
  if (workspace_bytes < l.total) return fail(SSD_ERR_WORKSPACE, "workspace smaller than ssd_bwd_workspace_bytes()");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return fail(SSD_ERR_ALIGN, "workspace must be 256-byte aligned");
  ssd::Problem q;
  const ssd_shape sw = swapped_shape(*shape);
  SSD_TRY(make_problem(&sw, &q));
  char* w = static_cast<char*>(workspace);
  void* ws_scan = w + l.scan;
  void* t_y = w + l.y;
  float* t_fin = reinterpret_cast<float*>(w + l.fin);
  void* t_x = w + l.xin;
  void* t_b = w + l.bin;
  void* t_c = w + l.cin;
  float* t_dtr = reinterpret_cast<float*>(w + l.dtr);
  float* t_init = reinterpret_cast<float*>(w + l.init);
  void* t_out = w + l.out;
  float* t_fin1 = reinterpret_cast<float*>(w + l.fin1);
  float* t_dcs = reinterpret_cast<float*>(w + l.dcs);
  float* t_xgb = reinterpret_cast<float*>(w + l.xgb);
  float* t_dyx = reinterpret_cast<float*>(w + l.dyx);
  float* t_part = reinterpret_cast<float*>(w + l.part);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t e = p.io_bf16 ? 2 : 4;
  const bool bf = p.io_bf16;
  ssd::Problem pf;
  const ssd_shape fs = f32_shape(*shape);
  SSD_TRY(make_problem(&fs, &pf));
  float* fx = static_cast<float*>(t_x);
  float* fb = static_cast<float*>(t_b);
  float* fc = static_cast<float*>(t_c);
  float* fy = static_cast<float*>(t_y);
  float* fo = static_cast<float*>(t_out);
  SSD_TRY(cuda_ok(cudaMemsetAsync(ws_scan, 0, sizeof(uint32_t), st), "status reset"));

  // 1. the forward again in float32, without the skip term: y - D x and the final state
  SSD_TRY(cuda_ok(ssd::launch_widen_flip_expand(x, fx, p.b, p.L, p.H, p.H, p.P, false, bf, st), "widen"));
  SSD_TRY(cuda_ok(ssd::launch_widen_flip_expand(B, fb, p.b, p.L, p.G, p.G, p.N, false, bf, st), "widen"));
  SSD_TRY(cuda_ok(ssd::launch_widen_flip_expand(C, fc, p.b, p.L, p.G, p.G, p.N, false, bf, st), "widen"));
  SSD_TRY(run_scan(pf, ws_scan, fx, dt, A, fb, fc, init_state, fy, t_fin, false, st));
  // 2. the adjoint scan in reversed time, in float32: x <- dy, B <- C, C <- B, decays shifted
  //    by one token, inputs unscaled, starting from dfinal; its output is g B, its final
  //    state g_0
  SSD_TRY(cuda_ok(ssd::launch_widen_flip_expand(dy, fx, p.b, p.L, p.H, p.H, p.P, true, bf, st), "flip"));
  SSD_TRY(cuda_ok(ssd::launch_widen_flip_expand(C, fb, p.b, p.L, p.G, p.G, p.N, true, bf, st), "flip"));
  SSD_TRY(cuda_ok(ssd::launch_widen_flip_expand(B, fc, p.b, p.L, p.G, p.G, p.N, true, bf, st), "flip"));
  SSD_TRY(cuda_ok(ssd::launch_reverse_decay(dt, t_dtr, p.b, p.L, p.H, st), "reverse decay"));
  SSD_TRY(run_scan(pf, ws_scan, fx, t_dtr, A, fb, fc, dfinal, fo, t_fin1, true, st));
  // 3. dx, dL/dcs, ddt, dA, dD, dinit
  SSD_TRY(cuda_ok(ssd::launch_bwd_combine(p, dy, x, fy, fo, dt, D, dx, t_dcs, t_xgb, t_dyx, st), "combine"));
  SSD_TRY(cuda_ok(ssd::launch_bwd_scalars(p, dfinal, t_fin, t_xgb, t_dyx, dt, A, t_dcs, ddt, t_part, dA, dD, st),
                  "scalars"));
  if (dinit) SSD_TRY(cuda_ok(ssd::launch_dinit(p, t_fin1, dt, A, dinit, st), "dinit"));
  // 4. dC: forward scans with x <- B (per head, kw columns at a time), B <- x, C <- dy, from
  //    init^T; summed per group into those columns of dC
  // 5. dB: reversed scans with x <- C (per head), B <- dy, C <- x, from dfinal^T; times dt,
  //    summed per group
  const int64_t kw = q.P;
  SSD_TRY(cuda_ok(ssd::launch_flip_expand(dy, t_b, p.b, p.L, p.H, p.H, p.P * e, 0, p.P * e, true, st), "flip"));
  SSD_TRY(cuda_ok(ssd::launch_flip_expand(x, t_c, p.b, p.L, p.H, p.H, p.P * e, 0, p.P * e, true, st), "flip"));
  for (int64_t n0 = 0; n0 < p.N; n0 += kw) {
    SSD_TRY(cuda_ok(ssd::launch_flip_expand(B, t_x, p.b, p.L, p.G, p.H, p.N * e, n0 * e, kw * e, false, st), "expand"));
    if (init_state)
      SSD_TRY(cuda_ok(ssd::launch_transpose_state(init_state, t_init, p.b * p.H, p.P, p.N, n0, kw, st), "transpose"));
    SSD_TRY(run_scan(q, ws_scan, t_x, dt, A, x, dy, init_state ? t_init : nullptr, t_out, nullptr, false, st));
    SSD_TRY(cuda_ok(ssd::launch_group_sum(p, t_out, nullptr, dC, n0, kw, false, st), "group sum"));

    SSD_TRY(cuda_ok(ssd::launch_flip_expand(C, t_x, p.b, p.L, p.G, p.H, p.N * e, n0 * e, kw * e, true, st), "flip"));
    if (dfinal)
      SSD_TRY(cuda_ok(ssd::launch_transpose_state(dfinal, t_init, p.b * p.H, p.P, p.N, n0, kw, st), "transpose"));
    SSD_TRY(run_scan(q, ws_scan, t_x, t_dtr, A, t_b, t_c, dfinal ? t_init : nullptr, t_out, nullptr, true, st));
    SSD_TRY(cuda_ok(ssd::launch_group_sum(p, t_out, dt, dB, n0, kw, true, st), "group sum"));
  }
  g_last_error[0] = '\0';
  return SSD_OK;
}

const char* ssd_status_str(ssd_status s) {
  switch (s) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID: return "invalid argument";
    case SSD_ERR_UNSUPPORTED: return "unsupported shape";
    case SSD_ERR_ALIGN: return "misaligned pointer";
    case SSD_ERR_CUDA: return "CUDA error";
    case SSD_ERR_TIMEOUT: return "on-chip wait timed out";
    case SSD_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

const char* ssd_last_error(void) { return g_last_error; }

int ssd_kernel_plan(const ssd_shape* shape) {
  ssd::Problem p;
  if (make_problem(shape, &p) != SSD_OK) return -1;
  return (use_state_tc(p) ? 1 : 0) | (use_scan_tc(p) ? 2 : 0) | (use_fused_state(p) ? 4 : 0);
}

}  // extern "C"
