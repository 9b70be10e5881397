// santa_flash.cu -- launch of the dense decode attention of santa_flash.cuh:
// grid and partition, the TMA descriptors of K and V.  Shapes it does not
// cover (fp32 caches, more than 8 query heads per KV head, head dims other
// than 64 and 128, K or V outside device memory) return
// cudaErrorNotSupported, and the caller takes the two-kernel path.
#include <algorithm>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "santa_flash.cuh"

namespace santa {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 flash_map_encoder() {
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

// A cache buffer as a (d, KV head, row) tensor of 16-bit elements, 64 x 1 x 16
// boxes, 128-byte swizzle; rows past `rows` read as zero.
bool encode_rows_map(CUtensorMap* tm, const void* base, int D, int Hkv, long long rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = flash_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)BK};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool device_pointer(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice;
}

}  // namespace

size_t flash_part_bytes(int D) { return (size_t)MAX_CTAS * 2 * (FL_MAXG * D + 2 * FL_MAXG) * sizeof(float); }

cudaError_t launch_flash(const LaunchArgs& a_in, unsigned* bar_count, unsigned* bar_gen) {
  LaunchArgs a = a_in;
  if (a.dtype > 1 || (a.D != 64 && a.D != 128) || a.H % a.Hkv != 0 || a.H / a.Hkv > FL_MAXG || !a.fpart)
    return cudaErrorNotSupported;
  const long long rows = a.kv_offsets ? -1 : (long long)a.B * a.nk_max;
  long long nrows = rows;
  if (a.kv_offsets) {   // the rows the offsets can address: at most B * nk_max
    nrows = (long long)a.B * a.nk_max;
  }
  if (nrows >= (1ll << 31) || !device_pointer(a.K) || !device_pointer(a.V)) return cudaErrorNotSupported;
  const long long blocks = (long long)a.B * a.Hkv * ((a.nk_max + BK - 1) / BK);
  const int grid = (int)std::min<long long>(std::min<long long>(blocks, (long long)a.num_sms), (long long)MAX_CTAS);
  a.blk_total = a.blk_q = 0;
  a.blk_r = 0;
  if (!a.kv_offsets) {
    a.blk_total = blocks;
    a.blk_q = blocks / grid;
    a.blk_r = (int)(blocks % grid);
  }
  const long long nblk = (a.nk_max + BK - 1) / BK;
  a.rdiv_perb = div_reciprocal((unsigned long long)(a.Hkv * nblk));
  a.rdiv_nblk = div_reciprocal((unsigned long long)nblk);
  a.rdiv_grid = div_reciprocal((unsigned long long)grid);
  CUtensorMap tk, tv;
  memset(&tk, 0, sizeof tk);
  memset(&tv, 0, sizeof tv);
  if (!encode_rows_map(&tk, a.K, a.D, a.Hkv, nrows) || !encode_rows_map(&tv, a.V, a.D, a.Hkv, nrows))
    return cudaErrorNotSupported;
  if (a.dtype == 0)
    return a.D == 128 ? launch_flash_inst<bf16_t, 128>(a, tk, tv, bar_count, bar_gen, grid)
                      : launch_flash_inst<bf16_t, 64>(a, tk, tv, bar_count, bar_gen, grid);
  return a.D == 128 ? launch_flash_inst<fp16_t, 128>(a, tk, tv, bar_count, bar_gen, grid)
                    : launch_flash_inst<fp16_t, 64>(a, tk, tv, bar_count, bar_gen, grid);
}

}  // namespace santa
