// ssd_fwd_noalloc -- the forward pass for callers that cannot hand the library a workspace.
//
// Some callers have no way to obtain device memory for scratch: for example a plugin loaded
// into a host application that owns the whole device-memory budget and forbids allocations
// from outside its own pool, or a latency-critical serving loop where a cudaMalloc (which
// can synchronise the device) is not acceptable.  For them this entry point takes its
// scratch from a fixed array that lives in this file's device memory image instead of from
// a caller-supplied workspace.  The pages this project follows describe no such entry point;
// it exists only for those callers.
//
// The array is kNoAllocBytes (64 MiB) long and every GPU that loads this code keeps it until
// the process exits.  Host code cannot use the array's name as a device address (on the host
// it names a stand-in object); the first call on each device, with that device current, asks
// the runtime for the real device address with cudaGetSymbolAddress and caches it.  That first
// call should therefore come before any stream capture on that device.
#include <mutex>

#include "ssd.h"
#include "ssd_internal.h"

namespace {

constexpr size_t kNoAllocBytes = SSD_NOALLOC_MAX_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// Shared by every call on a device: holds the previous call's intermediates.  ssd_fwd resets
// the status word and overwrites every intermediate it reads, so nothing needs clearing.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

ssd_status scratch_for_current_device(cudaStream_t stream, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
  // the cached address belongs to the current device: a stream of another device would run
  // the kernels there with a pointer into this device's array
  int stream_dev = -1;
  if (cudaStreamGetDevice(stream, &stream_dev) != cudaSuccess) return SSD_ERR_CUDA;
  if (stream_dev != dev) return SSD_ERR_INVALID;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return SSD_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SSD_OK;
}

}  // namespace

extern "C" {

ssd_status ssd_fwd_noalloc(const ssd_shape* shape, const void* x, const float* dt, const float* A,
                           const void* B, const void* C, const float* D, const float* init_state,
                           void* y, float* final_state, void* stream) {
  void* scratch = nullptr;
  const ssd_status s = scratch_for_current_device(static_cast<cudaStream_t>(stream), &scratch);
  if (s != SSD_OK) return s;
  // ssd_fwd checks the shape's scratch need against the array's size before it launches
  // anything, and returns SSD_ERR_WORKSPACE when the shape needs more.
  return ssd_fwd(shape, x, dt, A, B, C, D, init_state, y, final_state, scratch, kNoAllocBytes, stream);
}

}  // extern "C"
