// santa_static.cu -- santa_decode_static: santa_decode with its workspace in a
// fixed array of the library's own device memory, for callers that cannot
// allocate device memory (a plug-in that only receives tensors and a stream
// from its host framework; code that must not call cudaMalloc mid-run).
//
// The array is the santa_decode workspace (same layout, same kernels); only
// its first 256 bytes (the device error word) must start at zero for a call,
// and every call clears them on its stream.  Everything else is written by a
// call before the call reads it.  All calls share the array: calls that
// overlap on the GPU race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/santa.h"

// The scratch.  In host code this name is only a handle for the runtime: its
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char santa_static_scratch[SANTA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int MAX_DEVICES = 64;
std::mutex setup_mutex;
void* scratch_on_device[MAX_DEVICES] = {};

// Device address of the scratch on the current device, looked up on the first
// call for that device (with that device current) and kept.
santa_status_t scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return SANTA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(setup_mutex);
  if (!scratch_on_device[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, santa_static_scratch) != cudaSuccess || !ptr) return SANTA_ERR_CUDA;
    scratch_on_device[dev] = ptr;
  }
  *out = scratch_on_device[dev];
  return SANTA_OK;
}

}  // namespace

extern "C" santa_status_t santa_decode_static(const santa_params_t* p, int32_t variant, const void* q,
                                              const void* K, const void* V, float* out, santa_stream_t stream,
                                              int32_t* sample_idx) {
  const size_t need = santa_workspace_size(p);
  if (need == 0)   // invalid or unsupported parameters: santa_decode reports which, before any CUDA call
    return santa_decode(p, variant, q, K, V, out, nullptr, 0, stream, sample_idx);
  if (need > SANTA_STATIC_SCRATCH_BYTES) return SANTA_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  const santa_status_t st = scratch_address(&ws);
  if (st != SANTA_OK) return st;
  const santa_status_t ci = santa_workspace_init(ws, SANTA_STATIC_SCRATCH_BYTES, stream);   // error word to zero
  if (ci != SANTA_OK) return ci;
  return santa_decode(p, variant, q, K, V, out, ws, SANTA_STATIC_SCRATCH_BYTES, stream, sample_idx);
}
