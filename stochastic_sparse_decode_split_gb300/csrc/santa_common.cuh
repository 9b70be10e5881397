// santa_common.cuh -- device helpers shared by the SANTA / S2ANTA kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace santa {

constexpr unsigned FULL = 0xffffffffu;
constexpr int CHUNK = 256;          // keys per score / sampling chunk
constexpr int WARPS = 8;            // warps per CTA in the chunked kernels
constexpr int THREADS = WARPS * 32;
constexpr int HP = 4;               // query heads handled per pass over a loaded K tile
constexpr int GROUP_CHUNKS = 8;     // chunks per sampling CTA (one warp each)

// Device error flags (OR-ed into the workspace error word).
constexpr int ERR_NK_BOUND = 1;     // a ragged nk_b above the stated bound, or negative
constexpr int ERR_S_RANGE = 2;      // a per-sequence budget outside [1, S]
constexpr int ERR_EMPTY = 4;        // a sequence with no keys

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

// Transpose-reduction over the LPK lanes of a key group.  On entry each lane
// holds N partial sums; at every halving stage a lane keeps one half of its
// values, ships the other half to its partner and adds what it receives.  On
// exit lane `sub` holds the complete sums of original indices
// sub*(N/LPK) + i, i < N/LPK.  Costs N*(1 - 1/LPK) shuffles instead of N*log2(LPK).
template <int O, int N>
struct TransposeReduce {
  static __device__ __forceinline__ void run(float* v, int lane) {
    const bool upper = (lane & O) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const float send = upper ? v[i] : v[i + N / 2];
      const float keep = upper ? v[i + N / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(FULL, send, O);
    }
    TransposeReduce<O / 2, N / 2>::run(v, lane);
  }
};
template <int N>
struct TransposeReduce<0, N> {
  static __device__ __forceinline__ void run(float*, int) {}
};

// Scores of 32 consecutive keys for up to HP heads, one warp.
// Kw points at element 0 of key 0 of this warp's tile for the KV head;
// consecutive keys are row_stride elements apart; keys >= nvalid are not read.
// qreg[g][e] holds this lane's slice of (scale * q_g).  On return the lane owns
// key index my_key() (0..31) and s[g] is its score for head g (garbage when
// the key is not valid).
template <typename T, int D>
struct WarpScores {
  using TL = Tile<T, D>;
  static __device__ __forceinline__ int my_key(int lane) {
    return (lane % TL::LPK) * TL::KPI + lane / TL::LPK;
  }
  static __device__ __forceinline__ void load(const T* __restrict__ Kw, int64_t row_stride, int nvalid,
                                              int lane, uint4 (&kv)[TL::ITERS][TL::NVEC]) {
    const int slot = lane / TL::LPK, sub = lane % TL::LPK;
#pragma unroll
    for (int it = 0; it < TL::ITERS; ++it) {
      const int k = it * TL::KPI + slot;
      const T* src = Kw + (int64_t)k * row_stride + sub * TL::EPL;
#pragma unroll
      for (int v = 0; v < TL::NVEC; ++v) {
        kv[it][v] = (k < nvalid) ? ld_stream(src + v * (16 / TL::ES)) : make_uint4(0, 0, 0, 0);
      }
    }
  }
  static __device__ __forceinline__ void dot(const uint4 (&kv)[TL::ITERS][TL::NVEC],
                                             const float (&qreg)[HP][TL::EPL], int lane, float (&s)[HP]) {
    float v[TL::ITERS * HP];
#pragma unroll
    for (int it = 0; it < TL::ITERS; ++it) {
      float kf[TL::EPL];
#pragma unroll
      for (int w = 0; w < TL::NVEC; ++w) Elem<T>::widen(kv[it][w], kf + w * (16 / TL::ES));
#pragma unroll
      for (int g = 0; g < HP; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < TL::EPL; ++e) acc = fmaf(qreg[g][e], kf[e], acc);
        v[it * HP + g] = acc;
      }
    }
    TransposeReduce<TL::LPK / 2, TL::ITERS * HP>::run(v, lane);
#pragma unroll
    for (int g = 0; g < HP; ++g) s[g] = v[g];
  }
};

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

}  // namespace santa
