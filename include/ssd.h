/*
 * ssd.h -- C ABI of the GB300 (sm_103a) Mamba-2 SSD chunked forward scan.
 *
 * The layer (per head h, with B/C group g = h / (H / G)):
 *     h_t = exp(dt_t * A_h) * h_{t-1} + dt_t * outer(x_t, B_t)      (P x N state)
 *     y_t = h_t @ C_t + D_h * x_t
 * computed chunk-wise in the four steps that "Mamba-2 cuda-tile forward pass
 * kernels" (devotd.net) section 2 describes: an in-chunk log2-domain cumsum
 * of A*dt (chunk_cumsum, with its listing), the states at every chunk start
 * and after the last chunk (fwd_pass_state, here split into chunk_state and
 * state_passing), and the token outputs from the chunk-start states with the
 * intermediate C.B^T tile kept on chip (compute_out, here chunk_scan).
 *
 * Conventions for every entry point
 *   - All tensors are dense, row-major, contiguous, in DEVICE memory:
 *       x, y        (batch, seqlen, nheads, headdim)     io dtype
 *       dt          (batch, seqlen, nheads)              float32, the final step size
 *       A, D        (nheads)                             float32
 *       B, C        (batch, seqlen, ngroups, dstate)     io dtype
 *       init_state, final_state (batch, nheads, headdim, dstate)  float32
 *     io dtype is float32 or bfloat16 (ssd_shape.io_dtype).
 *   - Device pointers must be 16-byte aligned (SSD_ERR_ALIGN otherwise).
 *   - The caller owns every buffer, the workspace included.  The library
 *     allocates no device memory, keeps no per-call state, and never
 *     modifies its inputs.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  Outputs are valid once the
 *     stream has been synchronised.  No call synchronises the stream except
 *     ssd_read_status().
 *   - Errors are returned as ssd_status; nothing aborts or throws across the
 *     ABI.  Argument checks happen on the host before any launch; a failed
 *     check launches nothing.  ssd_last_error() gives a one-line detail of the
 *     last failure on the calling thread.
 *   - Step sizes and decay rates: any finite dt >= 0 and A <= 0 (a state that
 *     decays, as in the method), of any magnitude.  The chunked kernels split
 *     each decay weight exp(sum of dt A) into factors that stay inside float32
 *     range for every such input (a chunk's rows whose own 32-token block decays
 *     too steeply for that take per-element exponentials).  Growing states
 *     (dt * A > 0) are computed by the same arithmetic and are exact only while
 *     every weight of a chunk stays inside float32 range.
 *   - Kernels that wait on on-chip barriers give every wait a time limit; on
 *     expiry they record SSD_ERR_TIMEOUT in the workspace status word, drain
 *     their own copies, release tensor memory and return.  ssd_read_status()
 *     reports it.
 */
#ifndef SSD_H_
#define SSD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID = 1,     /* bad shape, null required pointer, bad dtype        */
  SSD_ERR_UNSUPPORTED = 2, /* valid shape that no kernel here handles            */
  SSD_ERR_ALIGN = 3,       /* a device pointer is not 16-byte aligned            */
  SSD_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed               */
  SSD_ERR_TIMEOUT = 5,     /* a kernel's bounded on-chip wait expired            */
  SSD_ERR_WORKSPACE = 6    /* workspace missing or smaller than required         */
} ssd_status;

/* Kernel-selection flags (ssd_shape.flags). */
#define SSD_FLAG_FORCE_SIMT 1u /* use the CUDA-core kernels even where the tensor-core ones apply */
/* Fail instead of falling back: chunk_state and chunk_scan run on the tensor cores for bf16 I/O
 * with headdim 64 and chunk 128 or 256 (chunk_state: dstate 64, 128, 256 or 512; chunk_scan:
 * dstate 64 or 128, or a multiple of 64 above 128 and not below chunk).  Every other shape runs
 * on the float32 CUDA-core kernels, correctly but several times slower (ssd_kernel_plan tells
 * which).  With this flag, ssd_fwd, ssd_chunk_state and ssd_chunk_scan return
 * SSD_ERR_UNSUPPORTED before any launch for such a shape, ssd_last_error() naming the reason. */
#define SSD_FLAG_REQUIRE_TENSOR_CORES 2u
/* fwd_pass_state ("Mamba-2 cuda-tile forward pass kernels", section 2, second kernel): for bf16
 * I/O, headdim 64, chunk 128 or 256 and dstate 64 or 128, one kernel can compute the chunk states
 * and chain them: a CTA walks one (batch, head pair) chain chunk by chunk with the chain's float32
 * state in tensor memory, writing hprev and final_state; S never reaches memory and state_passing
 * does not run.  It keeps one SM per chain and was slower than the two kernels on every workload
 * measured, so ssd_fwd and ssd_fwd_pass_state run it only with SSD_FLAG_FUSED_STATE (where the
 * shape allows it); SSD_FLAG_SEPARATE_STATE_PASSING (the default behaviour) wins if both are set. */
#define SSD_FLAG_SEPARATE_STATE_PASSING 4u
#define SSD_FLAG_FUSED_STATE 8u

typedef struct {
  int64_t batch;   /* b  >= 1                                               */
  int64_t seqlen;  /* L  >= 1 (any length; the last chunk may be ragged)    */
  int64_t nheads;  /* H  >= 1, a multiple of ngroups                        */
  int64_t headdim; /* P  >= 1                                               */
  int64_t dstate;  /* N  >= 1                                               */
  int64_t ngroups; /* G  >= 1                                               */
  int64_t chunk;   /* Q  in {64, 128, 256}                                  */
  int32_t io_dtype;/* ssd_dtype of x, B, C, y                               */
  uint32_t flags;  /* SSD_FLAG_* ; 0 for the default kernel choice          */
} ssd_shape;

/* Byte offsets of the intermediates inside a workspace (for inspection).
 *   cs2   float32 (b, H, nc, Q): log2(e) * in-chunk inclusive cumsum of A*dt,
 *         zero-padded past seqlen (chunk_cumsum output)
 *   dtT   float32 (b, H, nc, Q): dt laid out per head and chunk, zero-padded
 *   S     (b, nc, H, P, N): per-chunk end state started from zero; bfloat16
 *         when io_dtype is SSD_BF16, float32 when SSD_F32
 *   hprev (b, nc, H, P, N): state entering each chunk; bfloat16 when
 *         io_dtype is SSD_BF16, float32 when SSD_F32
 *   status uint32 at offset 0: 0, or an ssd_status recorded by a kernel
 * With bf16 I/O, headdim 64 and dstate above 128 (a multiple of 64, not
 * below chunk), chunk_scan first computes the term through the chunk-start
 * state, 2^{cs2_i} C_i . hprev, as a bf16 (b, L, H, P) tensor in the S
 * region (S is dead by then); S then holds that tensor on return.          */
typedef struct {
  size_t status, cs2, dtT, S, hprev, total;
  int64_t nchunks;
} ssd_workspace_layout;

/* Workspace bytes ssd_fwd needs for `shape`; 0 when the shape is invalid. */
size_t ssd_workspace_bytes(const ssd_shape* shape);

/* Fills *out for `shape`.  SSD_ERR_INVALID on a bad shape or null out. */
ssd_status ssd_get_workspace_layout(const ssd_shape* shape, ssd_workspace_layout* out);

/*
 * Full forward pass: chunk_cumsum -> chunk_state -> state_passing -> chunk_scan.
 *   D           nullable: treated as zeros
 *   init_state  nullable: the scan starts from the zero state
 *   final_state nullable: not written
 *   workspace   device buffer of >= ssd_workspace_bytes(shape) bytes,
 *               256-byte aligned; its contents on entry are ignored and on
 *               return hold the intermediates (see ssd_workspace_layout)
 * y receives the outputs in io dtype (bfloat16 rounded to nearest even).
 */
ssd_status ssd_fwd(const ssd_shape* shape, const void* x, const float* dt, const float* A,
                   const void* B, const void* C, const float* D, const float* init_state,
                   void* y, float* final_state, void* workspace, size_t workspace_bytes,
                   void* stream);

/* The four steps of ssd_fwd, one launch each, for callers that time or
 * inspect them.  They communicate through the workspace and must run in
 * this order on one stream. */

/* Step 1, chunk_cumsum ("Mamba-2 cuda-tile forward pass kernels" section 2,
 * first kernel and its listing): writes cs2 and dtT. */
ssd_status ssd_chunk_cumsum(const ssd_shape* shape, const float* dt, const float* A,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Step 2, chunk_state (same page, section 2, first half of fwd_pass_state):
 * S[b,c,h] = sum_t exp2(cs2_last - cs2_t) * dt_t * outer(x_t, B_t) over the
 * chunk's tokens.  Reads cs2/dtT, writes S. */
ssd_status ssd_chunk_state(const ssd_shape* shape, const void* x, const void* B,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Step 3, state_passing (same page, section 2, second half of fwd_pass_state:
 * chunk order kept, independent state elements in parallel):
 * hprev[c] = h_{c-1}, h_c = exp2(cs2_last,c) * h_{c-1} + S_c, h_{-1} = init.
 * Reads S and cs2, writes hprev and (if non-null) final_state. */
ssd_status ssd_state_passing(const ssd_shape* shape, const float* init_state,
                             float* final_state, void* workspace, size_t workspace_bytes,
                             void* stream);

/* Steps 2 and 3 together, fwd_pass_state (same page, section 2, second kernel): the fused
 * kernel with SSD_FLAG_FUSED_STATE where the shape allows it, else ssd_chunk_state then
 * ssd_state_passing.  Reads cs2/dtT, x, B, init_state (may be null: zero); writes hprev and
 * (if non-null) final_state, float32 (b, H, P, N).  The fused kernel leaves S unwritten. */
ssd_status ssd_fwd_pass_state(const ssd_shape* shape, const void* x, const void* B,
                              const float* init_state, float* final_state, void* workspace,
                              size_t workspace_bytes, void* stream);

/* Step 4, chunk_scan (same page, section 2, compute_out):
 * y_i = sum_{j<=i in chunk} exp2(cs2_i - cs2_j) dt_j (C_i.B_j) x_j
 *       + exp2(cs2_i) C_i . hprev + D x_i.   Reads cs2/dtT/hprev, writes y. */
ssd_status ssd_chunk_scan(const ssd_shape* shape, const void* x, const void* B, const void* C,
                          const float* D, void* y, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Synchronises `stream`, then reads the workspace status word: SSD_OK, or
 * the status a kernel recorded (SSD_ERR_TIMEOUT).  SSD_ERR_CUDA if the
 * synchronisation or the read fails. */
ssd_status ssd_read_status(const void* workspace, void* stream);

/* Diagnostic: launches one block that waits, with the library's bounded
 * wait, on an on-chip barrier that nothing ever completes, limited to
 * `timeout_ns`, and records SSD_ERR_TIMEOUT in the status word at
 * `status_word` (a device uint32).  Exercises the timeout path without any
 * fault.  0 < timeout_ns <= 1e9. */
ssd_status ssd_selftest_wait_timeout(uint32_t* status_word, uint64_t timeout_ns, void* stream);

/*
 * Forward pass without a caller-supplied workspace, for callers that cannot allocate
 * device memory (for example a plugin inside a host application that owns the whole
 * device-memory budget, or a serving loop that must never call the allocator).  The pages
 * this library follows have no counterpart to it.
 *
 * Arguments, layouts and results are those of ssd_fwd; the scratch comes from one fixed
 * array of SSD_NOALLOC_MAX_WORKSPACE_BYTES in the library's device image, which every GPU
 * that loads the library keeps until the process exits.  The call allocates nothing.
 *   - Shapes whose ssd_workspace_bytes() exceeds SSD_NOALLOC_MAX_WORKSPACE_BYTES are
 *     rejected with SSD_ERR_WORKSPACE before anything is launched.
 *   - The first call on a device (with that device current) looks up the array's device
 *     address with cudaGetSymbolAddress and caches it; make that first call before any
 *     stream capture on the device.  The cache is not refreshed: after cudaDeviceReset
 *     the library must be reloaded before this entry point is used again.
 *   - `stream` must belong to the current device; a stream of another device is rejected
 *     with SSD_ERR_INVALID before anything is launched.
 *   - Every call on a device shares the one array, which keeps the previous call's
 *     intermediates: calls whose work overlaps on the GPU (other streams, other threads)
 *     race on it and must be ordered by the caller.
 *   - ssd_read_status() cannot reach the array's status word; use ssd_fwd when a kernel
 *     time-out must be observed.
 */
#define SSD_NOALLOC_MAX_WORKSPACE_BYTES ((size_t)64 << 20)
ssd_status ssd_fwd_noalloc(const ssd_shape* shape, const void* x, const float* dt, const float* A,
                           const void* B, const void* C, const float* D, const float* init_state,
                           void* y, float* final_state, void* stream);

/*
 * Recurrent form over a short run of tokens -- the decoding step ("Compiler-First State Space
 * Duality and Portable O(1) Autoregressive Caching for Inference", technical summary section 2:
 * the fixed-size state is the cache, updated on the device token after token with no host
 * round trip per token).  For every (batch, head), in place, over shape->seqlen tokens t:
 *     state <- exp(dt_t * A_h) * state + dt_t * outer(x_t, B_t),    y_t = state @ C_t + D_h * x_t
 *   - x, y (batch, seqlen, nheads, headdim), dt (batch, seqlen, nheads), B, C (batch, seqlen,
 *     ngroups, dstate), A, D (nheads): as for ssd_fwd (D may be null).
 *   - state: float32 (batch, nheads, headdim, dstate), read at the start and overwritten with the
 *     state after the last token; it must not alias any input.
 *   - shape->chunk and shape->flags are ignored.  One launch reads and writes the state once,
 *     whatever seqlen is; the recurrence runs in float32.
 *   - Needs no workspace.  Supported shapes (else SSD_ERR_UNSUPPORTED): dstate in
 *     {64, 128, 256, 512} with headdim a multiple of 8 and headdim * dstate a multiple of
 *     1024; or dstate = 64 * 2^k <= 2048 with headdim * dstate / 64 a multiple of 32 and at
 *     most 512.
 */
ssd_status ssd_decode(const ssd_shape* shape, const void* x, const float* dt, const float* A,
                      const void* B, const void* C, const float* D, float* state, void* y,
                      void* stream);

/*
 * Mamba-1 selective scan, fused ("3.3 Hardware-aware algorithm and GPU memory hierarchy",
 * booiljung.github.io, section 2.1: zero-order-hold discretisation Abar = exp(delta A),
 * Bbar = (delta A)^-1 (exp(delta A) - I) delta B done on chip, only y written back; section 3:
 * load, discretise, scan and read-out in one kernel; section 4.1: h_t = Abar_t h_{t-1} +
 * Bbar_t x_t).  For every batch b, channel d < dim and state n < dstate, over t < seqlen:
 *     h[d,n] <- exp(delta_t[d] A[d,n]) h[d,n] + (exp(delta_t[d] A[d,n]) - 1) / A[d,n] B_t[n] x_t[d]
 *     y_t[d]  = sum_n C_t[n] h[d,n] + Dskip[d] x_t[d]
 * (the factor is delta_t[d] B_t[n] x_t[d] where A[d,n] = 0).
 *   - x, delta, y: (batch, seqlen, dim); B, C: (batch, seqlen, dstate); all in io_dtype.
 *     A: float32 (dim, dstate); Dskip: float32 (dim), nullable (no skip term).
 *   - init_state: float32 (batch, dim, dstate), nullable (zero state); final_state: float32
 *     (batch, dim, dstate), nullable (not written); neither may alias another argument.
 *   - Every pointer 16-byte aligned (SSD_ERR_ALIGN).  The recurrence runs in float32.
 *   - Supported: dstate in {8, 16, 32, 64} and dim a multiple of 64 / dstate (else
 *     SSD_ERR_UNSUPPORTED).  Needs no workspace; asynchronous on `stream`.
 */
typedef struct {
  int64_t batch;    /* >= 1 */
  int64_t seqlen;   /* >= 1 */
  int64_t dim;      /* D: channels, >= 1 */
  int64_t dstate;   /* N */
  int32_t io_dtype; /* ssd_dtype of x, delta, B, C, y */
  uint32_t flags;   /* reserved, 0 */
} ssd_sel_shape;

ssd_status ssd_selective_scan(const ssd_sel_shape* shape, const void* x, const void* delta,
                              const float* A, const void* B, const void* C, const float* Dskip,
                              const float* init_state, float* final_state, void* y, void* stream);

/*
 * Backward pass of ssd_fwd: the gradients of a loss w.r.t. every input of the forward scan,
 * given dL/dy and dL/dfinal_state.  For the recurrence h_t = a_t h_{t-1} + dt_t x_t (x) B_t,
 * a_t = exp(dt_t A), y_t = h_t C_t + D x_t ("Mamba-2 cuda-tile forward pass kernels" sections
 * 1-2), the adjoint state g_t = dL/dh_t obeys g_t = dy_t (x) C_t + a_{t+1} g_{t+1}: the same
 * kind of scan in reversed time.  The library runs five scans through the forward kernels (the
 * forward again without D; the adjoint scan, read out with B; a role-swapped forward scan for
 * dC and a role-swapped reversed scan for dB, both with head dim dstate and state headdim)
 * and element-wise / reduction kernels between them:
 *     dx = dt (g B) + D dy,  dB = sum_heads dt g^T x,  dC = sum_heads h^T dy,  dD = sum <dy, x>,
 *     dinit = a_0 g_0,  ddt = <x, g B> + A r,  dA = sum dt r,
 * with r_t = sum_{s >= t} (<dy_s, y_s - D x_s> - dt_s <x_s, g_s B_s>) (+ <dfinal, final> at the
 * last token), the derivative along the running sum of A dt that every decay depends on.
 *   - Inputs as for ssd_fwd; dy in the I/O dtype with y's shape; dfinal float32
 *     (batch, nheads, headdim, dstate), nullable (zero).
 *   - Outputs: dx (x's shape, I/O dtype), ddt float32 (batch, seqlen, nheads), dA float32
 *     (nheads), dB and dC (B's shape, I/O dtype), dD float32 (nheads, nullable: not written),
 *     dinit float32 (init's shape, nullable: not written).  No output may alias an input.
 *   - workspace: at least ssd_bwd_workspace_bytes(shape), 256-byte aligned, caller-owned.
 *   - Precision follows the I/O dtype: with bf16 I/O the scans' inputs and outputs are bf16
 *     and their arithmetic float32, as in the forward.
 */
size_t ssd_bwd_workspace_bytes(const ssd_shape* shape);
ssd_status ssd_bwd(const ssd_shape* shape, const void* x, const float* dt, const float* A, const void* B,
                   const void* C, const float* D, const float* init_state, const void* dy,
                   const float* dfinal, void* dx, float* ddt, float* dA, void* dB, void* dC, float* dD,
                   float* dinit, void* workspace, size_t workspace_bytes, void* stream);

/* Static description of a status code. */
const char* ssd_status_str(ssd_status status);

/* Detail of the last failure on the calling thread ("" if none). */
const char* ssd_last_error(void);

/* Which kernel family ssd_fwd would use for each step of `shape`:
 * bit 0 chunk_state on tensor cores, bit 1 chunk_scan on tensor cores, bit 2 chunk_state and
 * state_passing as the one fused fwd_pass_state kernel (SSD_FLAG_FUSED_STATE).  -1 for an
 * invalid shape. */
int ssd_kernel_plan(const ssd_shape* shape);

#ifdef __cplusplus
}
#endif

#endif /* SSD_H_ */
