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

// ---- the four steps on an already checked problem ----

ssd_status step_cumsum(const ssd::Problem& p, const float* dt, const float* A, const Views& v,
                       cudaStream_t st) {
  const cudaError_t e = ssd::launch_chunk_cumsum(p, dt, A, v.cs2, v.dtT, st);
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
  const cudaError_t e = ssd::launch_state_passing(p, v.S, v.cs2, init, v.hprev, final_state, st);
  return e == cudaSuccess ? SSD_OK : cuda_fail(e, "state_passing launch");
}

ssd_status step_scan(const ssd::Problem& p, const void* x, const void* B, const void* C,
                     const float* D, void* y, const Views& v, cudaStream_t st) {
  cudaError_t e;
  if (use_scan_tc(p)) {
    const char* why = nullptr;
    e = ssd::launch_chunk_scan_tc(p, x, B, C, D, v.cs2, v.dtT, v.hprev, y, v.status, st, &why);
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
  Views v;
  SSD_TRY(carve(p, workspace, workspace_bytes, &v));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = cudaMemsetAsync(v.status, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return cuda_fail(e, "status reset");
  SSD_TRY(step_cumsum(p, dt, A, v, st));
  SSD_TRY(step_state(p, x, B, v, st));
  SSD_TRY(step_passing(p, init_state, final_state, v, st));
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
  return (use_state_tc(p) ? 1 : 0) | (use_scan_tc(p) ? 2 : 0);
}

}  // extern "C"
