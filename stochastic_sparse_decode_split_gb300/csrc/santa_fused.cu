// santa_fused.cu -- launch of the single-launch decode step (santa_fused.cuh,
// instantiated per cache dtype in santa_fused_bf16.cu / santa_fused_fp16.cu):
// grid size, the uniform-batch partition, the TMA descriptor of K; and the
// self-test kernel of the bounded grid-barrier wait.
#include <algorithm>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "santa_fused.cuh"

namespace santa {

cudaError_t launch_fused_bf16(const LaunchArgs& a, const CUtensorMap& tm, bool tma, unsigned* bar_count,
                              unsigned* bar_gen, int grid);
cudaError_t launch_fused_fp16(const LaunchArgs& a, const CUtensorMap& tm, bool tma, unsigned* bar_count,
                              unsigned* bar_gen, int grid);

// Self-test of the bounded wait: one CTA waits on a generation word that no
// other CTA advances; the wait must end after limit_ns with ERR_TIMEOUT
// flagged, and the CTA returns normally.
__global__ void wait_timeout_selftest_kernel(const unsigned* gen, int* err, unsigned long long limit_ns) {
  __shared__ unsigned g;
  if (threadIdx.x == 0) g = ld_acquire(gen);
  __syncthreads();
  grid_wait(gen, g, err, limit_ns);
}

cudaError_t launch_wait_timeout_selftest(const unsigned* gen, int* err, unsigned long long limit_ns,
                                         cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(gen, err, limit_ns);
  return cudaGetLastError();
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// K as a (d, KV head, cache row) tensor of 16-bit elements, 64 x 1 x 16 boxes,
// 128-byte swizzle; rows past `rows` read as zero.
bool encode_k_map(CUtensorMap* tm, const void* K, int D, int Hkv, long long rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)BK};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(K), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_fused(const LaunchArgs& a_in, unsigned* bar_count, unsigned* bar_gen) {
  LaunchArgs a = a_in;
  const long long blocks = (long long)a.B * a.Hkv * ((a.nk_max + BK - 1) / BK);
  const int grid = (int)std::min<long long>(std::min<long long>(blocks, (long long)a.num_sms), (long long)MAX_CTAS);
  a.blk_total = a.blk_q = 0;
  a.blk_r = 0;
  if (!a.kv_offsets) {   // uniform batch: the partition is known here
    a.blk_total = blocks;
    a.blk_q = blocks / grid;
    a.blk_r = (int)(blocks % grid);
  }
  const long long nblk = (a.nk_max + BK - 1) / BK;
  a.rdiv_perb = div_reciprocal((unsigned long long)(a.Hkv * nblk));
  a.rdiv_nblk = div_reciprocal((unsigned long long)nblk);
  a.rdiv_grid = div_reciprocal((unsigned long long)grid);
  // TMA boxes address cache rows with 32-bit coordinates; K in host memory is
  // read by cp.async
  const long long rows = (long long)a.B * a.nk_max;
  CUtensorMap tm;
  memset(&tm, 0, sizeof tm);
  const bool tma = !a.k_host && rows < (1ll << 31) && encode_k_map(&tm, a.K, a.D, a.Hkv, rows);
  switch (a.dtype) {
    case 0: return launch_fused_bf16(a, tm, tma, bar_count, bar_gen, grid);
    case 1: return launch_fused_fp16(a, tm, tma, bar_count, bar_gen, grid);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace santa
