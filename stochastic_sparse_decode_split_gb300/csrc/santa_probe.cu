// santa_probe.cu -- a read-only streaming microbenchmark: the read ceiling of
// a transfer of a given size on this GPU (launch, ramp and tail included),
// reported beside the decode's roofline.  Not part of the method.
#include "santa_common.cuh"
#include "santa_launch.h"

namespace santa {

constexpr int RP_THREADS = 512;
constexpr int RP_UNROLL = 8;

// CTA i reads its contiguous share of the n16 16-byte words with
// non-allocating loads, RP_UNROLL in flight per thread, and folds them into
// one word per thread so that the loads are kept.
__global__ void __launch_bounds__(RP_THREADS) read_probe_kernel(const uint4* __restrict__ src, size_t n16,
                                                                uint32_t* __restrict__ sink) {
  const size_t per = (n16 + gridDim.x - 1) / gridDim.x;
  const size_t lo = per * blockIdx.x, hi = lo + per < n16 ? lo + per : n16;
  uint32_t acc = 0;
  for (size_t i = lo + threadIdx.x; i < hi; i += (size_t)RP_THREADS * RP_UNROLL) {
    uint4 v[RP_UNROLL];
#pragma unroll
    for (int u = 0; u < RP_UNROLL; ++u) {
      const size_t j = i + (size_t)u * RP_THREADS;
      v[u] = j < hi ? ld_stream(src + j) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < RP_UNROLL; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  sink[(size_t)blockIdx.x * RP_THREADS + threadIdx.x] = acc;
}

cudaError_t launch_read_probe(const void* src, size_t bytes, uint32_t* sink, int ctas, cudaStream_t stream) {
  read_probe_kernel<<<(unsigned)ctas, RP_THREADS, 0, stream>>>(static_cast<const uint4*>(src), bytes / 16, sink);
  return cudaGetLastError();
}

}  // namespace santa
