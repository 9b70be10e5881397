// santa_common.cuh -- device helpers shared by the SANTA / S2ANTA kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace santa {

constexpr unsigned FULL = 0xffffffffu;
constexpr int SUB = 16;             // keys per statistics chunk (one tensor-core m-tile)
constexpr int WIN = 32;             // keys per sampling window (two statistics chunks, one key per lane)
constexpr int TILE = 256;           // keys per stage of the streaming score pass
constexpr int DCHUNK = 256;         // keys per partial of the dense comparator
constexpr int CHUNK = DCHUNK;
constexpr int WARPS = 8;            // warps per CTA
constexpr int THREADS = WARPS * 32;
constexpr int STAGES = 3;           // shared-memory ring depth of the streaming score pass
constexpr int WIN_PER_WARP = 2;     // sampling windows per warp in the sampler
constexpr int SPC = WARPS * WIN_PER_WARP;  // sampling windows per sampler CTA
constexpr int HP = 4;               // query heads handled per pass over a loaded K tile

// Sampling variants (santa_variant_t).
constexpr int VAR_IID = 0;
constexpr int VAR_STRAT = 1;
constexpr int VAR_SYS = 2;

// Device error flags (OR-ed into the workspace error word).
constexpr int ERR_NK_BOUND = 1;     // a ragged nk_b above the stated bound, or negative
constexpr int ERR_S_RANGE = 2;      // a per-sequence budget outside [1, S]
constexpr int ERR_EMPTY = 4;        // a sequence with no keys
constexpr int ERR_TIMEOUT = 8;      // a grid-wide barrier wait ran out of time

struct bf16_t { uint16_t bits; };
struct fp16_t { uint16_t bits; };

// ---------------------------------------------------------------------------
// element traits: how a 16-byte vector of storage elements widens to fp32
// ---------------------------------------------------------------------------
template <typename T> struct Elem;

template <> struct Elem<bf16_t> {
  static constexpr int size = 2;
  // bf16 -> fp32 is a 16-bit left shift of the bit pattern (exact).
  static __device__ __forceinline__ void widen(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

template <> struct Elem<fp16_t> {
  static constexpr int size = 2;
  static __device__ __forceinline__ void widen(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h;
      memcpy(&h, &w[i], 4);
      const float2 p = __half22float2(h);
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
};

template <> struct Elem<float> {
  static constexpr int size = 4;
  static __device__ __forceinline__ void widen(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};

template <typename T> __device__ __forceinline__ float widen_scalar(const T* p);
template <> __device__ __forceinline__ float widen_scalar<bf16_t>(const bf16_t* p) {
  return __uint_as_float(((uint32_t)p->bits) << 16);
}
template <> __device__ __forceinline__ float widen_scalar<fp16_t>(const fp16_t* p) {
  __half h;
  memcpy(&h, &p->bits, 2);
  return __half2float(h);
}
template <> __device__ __forceinline__ float widen_scalar<float>(const float* p) { return *p; }

// Streaming 16-byte load that does not allocate in L1 (each K/V byte is read once).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ---------------------------------------------------------------------------
// Warp geometry of one key tile: a warp covers 32 keys of one KV head.  Each
// key row (D elements) is split over LPK lanes holding NVEC 16-byte vectors
// (EPL elements); KPI keys are read by one warp-wide load instruction.
// ---------------------------------------------------------------------------
template <typename T, int D>
struct Tile {
  static constexpr int ES = Elem<T>::size;
  static constexpr int ROWB = D * ES;
  static constexpr int LPK = ROWB >= 256 ? 16 : ROWB / 16;
  static constexpr int NVEC = ROWB / (16 * LPK);
  static constexpr int EPL = NVEC * 16 / ES;
  static constexpr int KPI = 32 / LPK;
  static constexpr int ITERS = 32 / KPI;  // == LPK
  static_assert(LPK * NVEC * 16 == ROWB, "row must split into 16-byte vectors");
  static_assert(ITERS == LPK, "tile geometry");
};

// ---------------------------------------------------------------------------
// Shared-memory staging of key / value rows.  Rows are copied with cp.async
// (16 bytes per request, no registers held while in flight).  Row r's 16-byte
// chunk s is stored at chunk (s & ~7) | ((s ^ r) & 7) of the row: eight
// consecutive rows read at the same logical chunk then fall on eight distinct
// 16-byte bank groups, so a warp reading one row per lane is conflict-free.
// ---------------------------------------------------------------------------
template <typename T, int D>
struct Rows {
  static constexpr int ES = Elem<T>::size;
  static constexpr int ROWB = D * ES;     // bytes per row (128, 256 or 512)
  static constexpr int NCH = ROWB / 16;   // 16-byte chunks per row
  static constexpr int EPC = 16 / ES;     // elements per chunk
  static_assert(NCH >= 8 && ROWB % 128 == 0, "row layout");
};

__device__ __forceinline__ int swz(int r, int s) { return (s & ~7) | ((s ^ r) & 7); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// cp_async16 whose source lines are marked for early eviction from L2 under
// `policy` (createpolicy): for data read once per step, so that it does not
// displace what the step reads again (scores, statistics).
__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void* src, unsigned long long policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ unsigned long long evict_first_policy() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Brings the 128-byte line holding p into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// Copies rows [0, nrows) (row r starts at src + r * stride elements) into the
// swizzled tile at `base`; NT threads cooperate.  stage_rows_async leaves the
// copies in the current commit group; stage_rows closes it.
template <typename T, int D, int NT>
__device__ __forceinline__ void stage_rows_async(uint32_t base, const T* __restrict__ src, int64_t stride,
                                                 int nrows) {
  using R = Rows<T, D>;
  for (int q = threadIdx.x; q < nrows * R::NCH; q += NT) {
    const int r = q / R::NCH, s = q % R::NCH;
    cp_async16(base + r * R::ROWB + swz(r, s) * 16, src + (int64_t)r * stride + s * R::EPC);
  }
}
template <typename T, int D, int NT>
__device__ __forceinline__ void stage_rows(uint32_t base, const T* __restrict__ src, int64_t stride, int nrows) {
  stage_rows_async<T, D, NT>(base, src, stride, nrows);
  cp_async_commit();
}
// Waits until at most N of this thread's most recent commit groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// Warp-level tensor-core tiles for the score contraction S[keys x heads] =
// K[keys x d] . Q^T[d x heads] with 16-bit inputs and fp32 accumulation
// (mma.m16n8k16: a 16-key x 16-dim A tile, a 16-dim x 8-head B tile).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
template <typename T> struct Mma;
template <> struct Mma<bf16_t> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};
template <> struct Mma<fp16_t> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

// ---------------------------------------------------------------------------
// Packed fp32 pairs (sm_100+ fma.rn.f32x2): one instruction, two lanes of
// fp32 fused multiply-add, each rounded as a scalar fmaf would be.
// ---------------------------------------------------------------------------
typedef unsigned long long f2x;
__device__ __forceinline__ f2x pack2(float x, float y) {
  f2x r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ float2 unpack2(f2x r) {
  float2 a;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
  return a;
}
__device__ __forceinline__ f2x ffma2(f2x a, f2x b, f2x c) {
  f2x d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// A 16-byte chunk of storage elements widened to EPC/2 fp32 pairs.
template <typename T> struct Pairs;
template <> struct Pairs<bf16_t> {
  static __device__ __forceinline__ void get(const uint4& v, f2x* p) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = pack2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  }
};
template <> struct Pairs<fp16_t> {
  static __device__ __forceinline__ void get(const uint4& v, f2x* p) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h;
      memcpy(&h, &w[i], 4);
      const float2 f = __half22float2(h);
      p[i] = pack2(f.x, f.y);
    }
  }
};
template <> struct Pairs<float> {
  static __device__ __forceinline__ void get(const uint4& v, f2x* p) {
    p[0] = pack2(__uint_as_float(v.x), __uint_as_float(v.y));
    p[1] = pack2(__uint_as_float(v.z), __uint_as_float(v.w));
  }
};

// e^x from the hardware base-2 exponential (relative error ~2^-22; e^-inf = 0).
__device__ __forceinline__ float fast_exp(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
  return y;
}

// 2^x from the hardware base-2 exponential (2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(FULL, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(FULL, x, o);
  return x;
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 32x32->64-bit products with the published multipliers, the key advanced by
// the published Weyl increments between rounds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo_a = 0xD2511F53u * c.x, hi_a = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo_b = 0xCD9E8D57u * c.z, hi_b = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi_b ^ c.y ^ k0, lo_b, hi_a ^ c.w ^ k1, lo_a);
  }
  return c;
}

// Uniform in [0, 1): top 24 bits of a Philox word times 2^-24 (exact in fp32 and fp64).
__device__ __forceinline__ double word_to_unit(uint32_t w) { return (double)(w >> 8) * (1.0 / 16777216.0); }

__device__ __forceinline__ void flag_error(int* err, int bits) { atomicOr(err, bits); }

// Nanoseconds of the global timer (for bounded waits).
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor is still running; it must
// wait here before touching anything the predecessor writes.  Without that
// launch attribute both are no-ops.
__device__ __forceinline__ void wait_for_predecessor() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// out[i..i+1] += v with one vectorised fp32 reduction (no return value).
__device__ __forceinline__ void red_add_v2(float* out, float2 v) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(out), "f"(v.x), "f"(v.y) : "memory");
}
// out[i..i+3] += v with one vectorised fp32 reduction (no return value).
__device__ __forceinline__ void red_add_v4(float* out, float4 v) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(out), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

}  // namespace santa
