// santa_tma.cuh -- Tensor Memory Accelerator copies and shared-memory
// mbarriers for the single-launch decode (sm_103a).
//
// K is described to the TMA unit as a 3-D tensor (d, KV head, cache row) of
// 16-bit elements, row strides d*2 and H_kv*d*2 bytes.  One box is 64
// elements x 1 KV head x 16 rows = 2 KiB with the 128-byte swizzle: the 16-byte
// chunk j of box row r lands at chunk j ^ (r & 7) of that row, so the eight
// rows one ldmatrix phase reads fall on eight distinct bank groups.
#pragma once

#include <cuda.h>

#include "santa_common.cuh"

namespace santa {

__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Makes the initialised barriers visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// Arrival of the one expected arriver, announcing `bytes` of transactions.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// One plain arrival (the stage was filled by ordinary shared-memory stores).
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Rows [z, z + 16) of a (row, KV head kvh, d) cache into a 16-row stage in
// the TMA's 128-byte swizzled layout by ordinary loads and stores (one warp),
// rows at or past `row_end` as zeros: for the blocks whose box would reach
// past the end of a ragged cache buffer.
template <int D>
__device__ __forceinline__ void fill_stage_plain(uint32_t dst, const uint16_t* base, int64_t z, int kvh, int Hkv,
                                                 int64_t row_end, int lane) {
#pragma unroll
  for (int j = 0; j < 16 * D / 8 / 32; ++j) {
    const int q = lane + 32 * j, r = q / (D / 8), c = q % (D / 8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (z + r < row_end) v = *reinterpret_cast<const uint4*>(base + ((z + r) * Hkv + kvh) * D + c * 8);
    const uint32_t a = (uint32_t)((c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst + a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
  }
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for phase `parity` of a barrier: gives up once `limit_ns` of
// global time have passed (a copy takes microseconds), flags ERR_TIMEOUT and
// returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, unsigned parity, int* err,
                                          unsigned long long limit_ns = 100000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) break;
  }
  flag_error(err, ERR_TIMEOUT);
  return false;
}
// Orders this thread's earlier shared-memory accesses before later
// asynchronous-proxy (TMA) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)tm) : "memory");
}
// One 3-D box to shared memory; completion is counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int x, int y, int z, uint32_t bar,
                                            unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"((uint64_t)tm), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// Byte offset, inside one 16-row stage of 64-element boxes (box b at b*2048),
// of the 16-byte chunk holding elements [8c, 8c + 8) of row r.
__device__ __forceinline__ uint32_t swz128_offset(int r, int c) {
  return (uint32_t)((c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Named barrier over `nthreads` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void group_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace santa
