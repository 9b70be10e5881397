// santa_flash.cuh -- dense decode attention out = softmax(q K^T * scale) V
// (Eq. 1 of "Stochastic Sparse Attention for Memory-Bound Inference", the
// exact quantity the sampled estimate approximates), split over the keys in
// one cooperative launch on sm_103a, for 16-bit caches.
//
// The partition is the sampler's: blocks of 16 keys of one KV head, ordered
// (sequence, KV head, key block), CTA i taking blocks [lo(i), lo(i + 1)).
// Each warp keeps a ring of NS stages, each stage one block of K and the same
// block of V, filled by TMA (128-byte swizzled 64 x 1 x 16 boxes) and
// completed on an mbarrier.  Per block the warp computes the scores of its KV
// group's query heads on the tensor cores (S[16 keys x 8 heads] = K q^T),
// folds them into a running softmax in base 2, turns the probabilities into
// the B operand of a second tensor-core product with movmatrix, and adds
// P V into its accumulator O^T[d x 8 heads] (A = V^T from ldmatrix.trans).
//
// The range's blocks of one (sequence, KV head) piece form a unit.  At the
// end of a unit every warp leaves its (max, sum, O) in shared memory and the
// CTA merges them; a unit that is a whole piece is normalised into out, the
// (at most two) units of pieces shared with other CTAs go to the workspace as
// partials.  After a grid barrier the CTA holding a shared piece's last block
// merges the piece's partials into out.  Query heads per KV head: at most 8.
#pragma once

#include <climits>
#include <cstring>

#include <cuda_fp16.h>

#include "santa_common.cuh"
#include "santa_grid.cuh"
#include "santa_launch.h"
#include "santa_part.cuh"
#include "santa_seq.cuh"
#include "santa_tma.cuh"

#ifndef SANTA_STAMP
#define SANTA_STAMP(k) ((void)0)
#endif

namespace santa {

constexpr int FL_MAXG = 8;   // query heads per KV head (the MMA's n)

template <int D>
struct FlashGeom {
  static constexpr int NW = D == 128 ? 8 : 16;             // warps per CTA
  static constexpr int NT = NW * 32;
  static constexpr int KB = BK * D * 2;                    // one block of K (or V)
  static constexpr int STAGE = 2 * KB;                     // K, then V
  static constexpr int NS = 3;                             // ring depth per warp
  static constexpr int RING = NW * NS * STAGE;             // 192 KiB
  static constexpr int PART = NW * FL_MAXG * D * 4;        // the warps' unit partials: 32 KiB
  static constexpr size_t SMEM = (size_t)RING + PART + 1024;
};

// 8 x 8 transpose of 16-bit elements across the warp (each thread: one row
// pair of the input fragment in, the same of the transpose out).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// Two fp32 values as one register of the cache's 16-bit type (lo, hi), rounded to nearest.
template <typename T> __device__ __forceinline__ uint32_t pack16x2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack16x2<bf16_t>(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
template <> __device__ __forceinline__ uint32_t pack16x2<fp16_t>(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The two values of such a register back in fp32 (exact).
template <typename T> __device__ __forceinline__ float2 unpack16x2(uint32_t r);
template <> __device__ __forceinline__ float2 unpack16x2<bf16_t>(uint32_t r) {
  return make_float2(__uint_as_float(r << 16), __uint_as_float(r & 0xffff0000u));
}
template <> __device__ __forceinline__ float2 unpack16x2<fp16_t>(uint32_t r) {
  __half2 h;
  memcpy(&h, &r, 4);
  return __half22float2(h);
}

// Workspace partial of CTA j, slot s (0: the first piece of its range, 1: the
// last): O[8][D] unnormalised, then (m, l)[8] in base 2.
template <int D>
__device__ __forceinline__ float* flash_part(float* base, int j, int slot) {
  return base + ((size_t)j * 2 + slot) * (FL_MAXG * D + 2 * FL_MAXG);
}

template <typename T, int D>
__global__ void __launch_bounds__(FlashGeom<D>::NT, 1)
flash_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, LaunchArgs a,
                    unsigned* bar_count, unsigned* bar_gen) {
  using Gm = FlashGeom<D>;
  constexpr int NW = Gm::NW, NS = Gm::NS, STG = Gm::STAGE, NT = Gm::NT;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) unsigned long long s_bar[NW * NS];
  __shared__ float s_pm[NW][FL_MAXG], s_pl[NW][FL_MAXG];
  __shared__ Cur s_cur[2];
  __shared__ long long s_part[2];
  __shared__ unsigned s_gen;

  SANTA_STAMP(0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = gridDim.x, cta = blockIdx.x;
  const int G = a.H / a.Hkv;
  unsigned char* const ring = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t ring_u32 = smem_addr(ring);
  float* const s_po = reinterpret_cast<float*>(ring + Gm::RING);   // [NW][G][D]
  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  Part pt;
  long long lo, hi;
  Cur cA, cB;
  cta_range(a, P, cta, warp, lane, s_part, s_cur, pt, lo, hi, cA, cB);
  const bool has_range = hi > lo;
  SANTA_STAMP(1);

  // ---- rings: warp w streams blocks lo + w + NW k, k < n_mine
  const int n_mine = has_range && hi - lo > warp ? (int)((hi - lo - warp + NW - 1) / NW) : 0;
  const uint32_t wring = ring_u32 + (uint32_t)(warp * NS * STG);
  const uint32_t wbar = smem_addr(&s_bar[warp * NS]);
  const unsigned long long pol = evict_first_policy();   // K and V are read once per step
  if (lane == 0)
    for (int s = 0; s < NS; ++s) mbar_init(wbar + 8 * s, 1);
  mbar_fence_init();
  __syncwarp();
  Cur cur = cA;
  if (n_mine > 0) cur_advance(cur, a, warp);
  Cur prod = cur;
  // the end of the cache buffers: B nk_max rows, or kv_offsets[B] (a box of
  // a ragged batch's last block may not reach past it)
  const int64_t row_end = a.kv_offsets ? a.kv_offsets[a.B] : (int64_t)a.B * a.nk_max;
  auto issue = [&](int k) {
    if (k < n_mine) {
      const int s = k % NS;
      const uint32_t dst = wring + (uint32_t)(s * STG), bar = wbar + 8 * s;
      const int64_t z = prod.row0 + (int64_t)prod.kblk * BK;
      if (z + BK <= row_end) {
        if (lane == 0) {
          fence_proxy_async_smem();
          mbar_expect_tx(bar, STG);
#pragma unroll
          for (int x = 0; x < D / 64; ++x) tma_load_3d(dst + x * 2048, &tmK, x * 64, prod.kvh, (int)z, bar, pol);
#pragma unroll
          for (int x = 0; x < D / 64; ++x)
            tma_load_3d(dst + Gm::KB + x * 2048, &tmV, x * 64, prod.kvh, (int)z, bar, pol);
        }
      } else {
        fill_stage_plain<D>(dst, static_cast<const uint16_t*>(a.K), z, prod.kvh, a.Hkv, row_end, lane);
        fill_stage_plain<D>(dst + Gm::KB, static_cast<const uint16_t*>(a.V), z, prod.kvh, a.Hkv, row_end, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
      }
      cur_advance(prod, a, NW);
    }
  };
#pragma unroll 1
  for (int k = 0; k < NS; ++k) issue(k);
  SANTA_STAMP(2);

  // ---- while the first blocks are in flight: the barrier generation, and
  //      the outputs of sequences the metadata check rejects (zero)
  if (tid == 32) {
    s_gen = ld_acquire(bar_gen);
    if (cta == 0) bar_count[((s_gen & 1u) ^ 1u) * 32] = 0u;
  }
  for (int b = cta; b < a.B; b += P) {
    int S_b;
    const int e = seq_error(a.kv_offsets, a.nk_max, nullptr, 1, b, S_b);
    if (e) {
      if (tid == 0) flag_error(a.err, e);
      float4* o = reinterpret_cast<float4*>(a.out + (int64_t)b * a.H * D);
      for (int i = tid; i < a.H * D / 4; i += NT) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  const int g8 = lane >> 2, t4 = lane & 3;
  const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8, lhalf = lane >> 4;   // K fragments (A = K)
  const int vrow = (lane & 7) + ((lane >> 4) & 1) * 8, vhalf = (lane >> 3) & 1;   // V^T fragments
  const float sl2 = a.scale * LOG2E;

  // The end of a unit (the range's blocks of one piece): the warps' partials
  // merged in shared memory, then out (the piece is inside the range) or the
  // workspace (the piece is shared; slot 0 for the range's first piece).
  Cur uc = cA;          // the unit being closed
  int u_ord = 0;        // its position in the range
  float rm[2], rl[2];
  float oacc[D / 16][4];
  auto reset = [&]() {
    rm[0] = rm[1] = -INFINITY;
    rl[0] = rl[1] = 0.f;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  };
  reset();
  auto close_unit = [&]() {
    // this warp's partial (empty if it had no block of the unit)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float l = rl[hh];
      l += __shfl_xor_sync(FULL, l, 4);
      l += __shfl_xor_sync(FULL, l, 8);
      l += __shfl_xor_sync(FULL, l, 16);
      const int head = 2 * t4 + hh;
      if (g8 == 0 && head < G) {
        s_pm[warp][head] = rm[hh];
        s_pl[warp][head] = l;
      }
      if (head < G) {
        float* po = s_po + (warp * G + head) * D;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
          po[16 * i + g8] = oacc[i][hh];
          po[16 * i + g8 + 8] = oacc[i][2 + hh];
        }
      }
    }
    reset();
    __syncthreads();
    const bool inside = uc.pb_lo >= lo && uc.pb_lo + uc.nblk <= hi;
    const int slot = u_ord == 0 ? 0 : 1;
    const int64_t bh0 = (int64_t)uc.b * a.H + (int64_t)uc.kvh * G;
    float* gp = flash_part<D>(a.fpart, cta, slot);
    for (int i = tid; i < G * D; i += NT) {
      const int g = i / D, d = i - g * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, s_pm[w][g]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = s_pm[w][g] > -INFINITY ? fast_exp2(s_pm[w][g] - M) : 0.f;
        L = fmaf(s_pl[w][g], f, L);
        O = fmaf(s_po[(w * G + g) * D + d], f, O);
      }
      if (inside) {
        a.out[(bh0 + g) * D + d] = L > 0.f ? O / L : 0.f;
      } else {
        gp[g * D + d] = O;
        if (d == 0) {
          gp[FL_MAXG * D + 2 * g] = M;
          gp[FL_MAXG * D + 2 * g + 1] = L;
        }
      }
    }
    __syncthreads();   // the shared partials are free for the next unit
    uc.kblk = uc.nblk;
    cur_norm(uc, a);
    ++u_ord;
  };

  const T* qp = static_cast<const T*>(a.q);
  uint32_t bq[D / 16][2];
  long long bq_piece = -1;
  bool ring_dead = false;
  SANTA_STAMP(3);
  for (int k = 0; k < n_mine; ++k) {
    while (uc.b < a.B && uc.pb_lo < cur.pb_lo) close_unit();   // units before this block's
    const int s = k % NS;
    if (!ring_dead && !mbar_wait(wbar + 8 * s, (unsigned)((k / NS) & 1), a.err)) ring_dead = true;
    __syncwarp();
    if (k == 0) SANTA_STAMP(4);
    const int64_t bh0 = (int64_t)cur.b * a.H + (int64_t)cur.kvh * G;
    if (cur.pb_lo != bq_piece) {   // q fragments of the piece's heads (B = q^T, n = head)
      const T* qg = qp + bh0 * D;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const T* q2 = qg + g8 * D + ks * 16 + t4 * 2;
        bq[ks][0] = (g8 < G) ? *reinterpret_cast<const uint32_t*>(q2) : 0u;
        bq[ks][1] = (g8 < G) ? *reinterpret_cast<const uint32_t*>(q2 + 8) : 0u;
      }
      bq_piece = cur.pb_lo;
    }
    const uint32_t kbase = wring + (uint32_t)(s * STG), vbase = kbase + Gm::KB;
    // S[16 keys x 8 heads]
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < D / 16; ks += 2) {
      uint32_t f0[4], f1[4];
      ldmatrix_x4(kbase + swz128_offset(lrow, ks * 2 + lhalf), f0);
      ldmatrix_x4(kbase + swz128_offset(lrow, ks * 2 + 2 + lhalf), f1);
      Mma<T>::run(acc0, f0, bq[ks][0], bq[ks][1]);
      Mma<T>::run(acc1, f1, bq[ks + 1][0], bq[ks + 1][1]);
    }
    // V^T fragments of the whole block into registers; the stage is then
    // free for the block NS ahead
    uint32_t vf[D / 16][4];
#pragma unroll
    for (int i = 0; i < D / 16; ++i) ldmatrix_x4_trans(vbase + swz128_offset(vrow, 2 * i + vhalf), vf[i]);
    __syncwarp();
    issue(k + NS);
    // running softmax (base 2) of heads 2 t4 + hh over keys g8, g8 + 8
    const int64_t key0 = (int64_t)cur.kblk * BK;
    const bool ok0 = key0 + g8 < cur.nk, ok1 = key0 + g8 + 8 < cur.nk;
    float p0[2], p1[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float s0 = ok0 ? (acc0[hh] + acc1[hh]) * sl2 : -INFINITY;
      const float s1 = ok1 ? (acc0[2 + hh] + acc1[2 + hh]) * sl2 : -INFINITY;
      float m = fmaxf(s0, s1);
      m = fmaxf(m, __shfl_xor_sync(FULL, m, 4));
      m = fmaxf(m, __shfl_xor_sync(FULL, m, 8));
      m = fmaxf(m, __shfl_xor_sync(FULL, m, 16));
      const float mn = fmaxf(rm[hh], m);
      const float alpha = rm[hh] > -INFINITY ? fast_exp2(rm[hh] - mn) : 0.f;
      p0[hh] = ok0 ? fast_exp2(s0 - mn) : 0.f;
      p1[hh] = ok1 ? fast_exp2(s1 - mn) : 0.f;
      rl[hh] = fmaf(rl[hh], alpha, p0[hh] + p1[hh]);
      rm[hh] = mn;
#pragma unroll
      for (int i = 0; i < D / 16; ++i) {
        oacc[i][hh] *= alpha;
        oacc[i][2 + hh] *= alpha;
      }
    }
    // P^T as the B operand (k = key, n = head) of O^T += V^T P^T, P split
    // into a 16-bit head and the 16-bit rounding of the rest (two products:
    // the sum carries about 16 significant bits of P, not 8)
    const uint32_t h0 = pack16x2<T>(p0[0], p0[1]), h1 = pack16x2<T>(p1[0], p1[1]);
    const float2 r0 = unpack16x2<T>(h0), r1 = unpack16x2<T>(h1);
    const uint32_t b01 = movmatrix_trans(h0), b23 = movmatrix_trans(h1);
    const uint32_t c01 = movmatrix_trans(pack16x2<T>(p0[0] - r0.x, p0[1] - r0.y));
    const uint32_t c23 = movmatrix_trans(pack16x2<T>(p1[0] - r1.x, p1[1] - r1.y));
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      Mma<T>::run(oacc[i], vf[i], b01, b23);
      Mma<T>::run(oacc[i], vf[i], c01, c23);
    }
    cur_advance(cur, a, NW);
  }
  SANTA_STAMP(5);
  // the rest of the range's units (every warp closes each unit once)
  while (has_range && uc.b < a.B && uc.pb_lo <= cB.pb_lo) close_unit();
  SANTA_STAMP(6);

  // ---- the shared pieces: every CTA arrives; the CTA holding a piece's last
  //      block (the piece is its range's first, started before it) merges
  //      the covering CTAs' partials into out
  unsigned* const arrivals = bar_count + (s_gen & 1u) * 32;
  __syncthreads();
  if (tid == 0) red_release_add(arrivals, 1u);
  const bool owner = has_range && cA.pb_lo < lo && cA.pb_lo + cA.nblk <= hi;
  SANTA_STAMP(7);
  if (owner || cta == 0) arrivals_wait(arrivals, (unsigned)P, a.err);
  SANTA_STAMP(8);
  if (owner) {
    // the covering CTAs' partials: their O staged 32 CTAs at a time into the
    // ring by asynchronous copies (all in flight at once) while their (m, l)
    // give each head's M and L (one warp per head) and then each partial's
    // weight 2^(m - M) / L
    constexpr int PW = FL_MAXG * D + 2 * FL_MAXG;   // floats per partial (a multiple of 4)
    const int i_first = pt.cta_of(cA.pb_lo), ncov = cta - i_first + 1;
    const int64_t bh0 = (int64_t)cA.b * a.H + (int64_t)cA.kvh * G;
    float* const s_ml = reinterpret_cast<float*>(ring);           // [ncov][G][2]
    float* const s_f = s_ml + ((2 * G * ncov + 3) & ~3);          // [ncov][G]
    float* const s_o = s_f + ((G * ncov + 3) & ~3);               // [32][PW]
    float* const s_hd = s_po;                                     // [G][2]: M, L
    auto part_of = [&](int j) { return flash_part<D>(a.fpart, j, cA.pb_lo <= pt.lo(j) ? 0 : 1); };
    auto stage_o = [&](int j0, int nc) {
      for (int i = tid; i < nc * (FL_MAXG * D / 4); i += NT) {
        const int jj = i / (FL_MAXG * D / 4), q = i - jj * (FL_MAXG * D / 4);
        cp_async16(smem_addr(s_o + jj * PW + 4 * q), part_of(i_first + j0 + jj) + 4 * q);
      }
      cp_async_commit();
    };
    stage_o(0, min(32, ncov));
    for (int i = tid; i < ncov * G; i += NT) {
      const int jj = i / G, g = i - jj * G;
      const float* gp = part_of(i_first + jj) + FL_MAXG * D + 2 * g;
      s_ml[2 * i] = __ldcg(gp);
      s_ml[2 * i + 1] = __ldcg(gp + 1);
    }
    __syncthreads();
    if (warp < G) {
      float M = -INFINITY;
      for (int jj = lane; jj < ncov; jj += 32) M = fmaxf(M, s_ml[2 * (jj * G + warp)]);
      M = warp_max(M);
      float L = 0.f;
      for (int jj = lane; jj < ncov; jj += 32) {
        const float m = s_ml[2 * (jj * G + warp)];
        if (m > -INFINITY) L = fmaf(s_ml[2 * (jj * G + warp) + 1], fast_exp2(m - M), L);
      }
      L = warp_sum(L);
      if (lane == 0) {
        s_hd[2 * warp] = M;
        s_hd[2 * warp + 1] = L;
      }
    }
    __syncthreads();
    for (int i = tid; i < ncov * G; i += NT) {
      const int g = i % G;
      const float m = s_ml[2 * i], M = s_hd[2 * g], L = s_hd[2 * g + 1];
      s_f[i] = (m > -INFINITY && L > 0.f) ? fast_exp2(m - M) / L : 0.f;
    }
    constexpr int RO = (FL_MAXG * D + NT - 1) / NT;   // outputs per thread
    float O[RO];
#pragma unroll
    for (int r = 0; r < RO; ++r) O[r] = 0.f;
    for (int j0 = 0; j0 < ncov; j0 += 32) {
      const int nc = min(32, ncov - j0);
      if (j0 > 0) stage_o(j0, nc);
      cp_async_wait_all();
      __syncthreads();
#pragma unroll
      for (int r = 0; r < RO; ++r) {
        const int i = tid + r * NT, g = min(i / D, G - 1), d = i % D;
#pragma unroll 4
        for (int jj = 0; jj < nc; ++jj) O[r] = fmaf(s_o[jj * PW + g * D + d], s_f[(j0 + jj) * G + g], O[r]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < RO; ++r) {
      const int i = tid + r * NT;
      if (i < G * D) a.out[(bh0 + i / D) * D + i % D] = O[r];
    }
  }
  if (cta == 0 && tid == 0) st_release(bar_gen, s_gen + 1u);
  SANTA_STAMP(9);
}

template <typename T, int D>
inline cudaError_t launch_flash_inst(const LaunchArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                     unsigned* bar_count, unsigned* bar_gen, int grid) {
  using Gm = FlashGeom<D>;
  auto kern = flash_decode_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Gm::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(Gm::NT);
  cfg.dynamicSmemBytes = Gm::SMEM;
  cfg.stream = a.stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, a, bar_count, bar_gen);
}

}  // namespace santa
