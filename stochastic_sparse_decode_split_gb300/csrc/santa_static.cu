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

#include <cstdint>

#include "../../include/santa.h"

// The scratch.  In host code this name is only a handle for the runtime: its
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char santa_static_scratch[SANTA_STATIC_SCRATCH_BYTES];

namespace {

// Device address of the scratch on the current device.  Looked up on every
// call (a host-side table lookup once the array's module is loaded), so that
// an address never outlives a device reset or a re-created primary context.
santa_status_t scratch_address(void** out) {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, santa_static_scratch) != cudaSuccess || !ptr) {
    (void)cudaGetLastError();
    return SANTA_ERR_CUDA;
  }
  *out = ptr;
  return SANTA_OK;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

extern "C" santa_status_t santa_static_warmup(void) {
  void* ws = nullptr;
  return scratch_address(&ws);
}

extern "C" santa_status_t santa_decode_static(const santa_params_t* p, int32_t variant, const void* q,
                                              const void* K, const void* V, float* out, santa_stream_t stream,
                                              int32_t* sample_idx) {
  const size_t need = santa_workspace_size(p);
  if (need == 0)   // invalid or unsupported parameters: santa_decode reports which, before any CUDA call
    return santa_decode(p, variant, q, K, V, out, nullptr, 0, stream, sample_idx);
  if (need > SANTA_STATIC_SCRATCH_BYTES) return SANTA_ERR_SCRATCH_LIMIT;
  // the rest of santa_decode's argument checks, before any CUDA call
  if (variant < SANTA_IID || variant > SANTA_SYSTEMATIC) return SANTA_ERR_INVALID_ARG;
  if (!q || !K || !V || !out) return SANTA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(out, 16)) return SANTA_ERR_INVALID_ARG;
  if (sample_idx && !aligned(sample_idx, 4)) return SANTA_ERR_INVALID_ARG;
  void* ws = nullptr;
  const santa_status_t st = scratch_address(&ws);
  if (st != SANTA_OK) return st;
  const santa_status_t ci = santa_workspace_init(ws, SANTA_STATIC_SCRATCH_BYTES, stream);   // error word to zero
  if (ci != SANTA_OK) return ci;
  return santa_decode(p, variant, q, K, V, out, ws, SANTA_STATIC_SCRATCH_BYTES, stream, sample_idx);
}
