// santa_fused.cuh -- one decode step of SANTA / S2ANTA in a single persistent
// launch for 16-bit caches (sm_103a); instantiated per cache dtype in
// santa_fused_bf16.cu and santa_fused_fp16.cu, launched from santa_fused.cu.
//
// "Stochastic Sparse Attention for Memory-Bound Inference":
//   scores and per-chunk statistics   Sec. 2 Eq. (1); App. O, Alg. 3
//   cross-chunk combine               App. O, Alg. 4
//   thresholds                        Sec. 2.1 (i.i.d. Eq. 4; stratified; systematic)
//   inverse CDF, left-closed          App. A.4
//   GQA-deduplicated gather-and-add   Eq. (4), Fig. 1; App. O, Alg. 5
//
// Work is cut into blocks of 16 keys x 1 KV head (one tensor-core m-tile, one
// statistics chunk), enumerated in (sequence, KV head, key block) order; a
// "piece" is the run of blocks of one (sequence, KV head).  One 512-thread CTA
// per SM, launched cooperatively; CTA i takes blocks [iT/P, (i+1)T/P), so the
// K bytes per CTA differ by at most one block.
//
// Phase A (stream): warp w of a CTA scores blocks w, w + 16, ... of its range.
// Each warp owns a ring of shared-memory stages filled by TMA (one 2 KiB box
// per 64 features, 128-byte swizzle) and waits on its own mbarriers only.  It
// scores a block on the tensor cores (16 keys x the G query heads of the KV
// head), writes the fp32 scores (the stash the sampler reads back) and the
// 16-key (max, exp-sum), and keeps running statistics of the pieces its CTA
// shares with neighbours.
//
// Phase B (sample).  Masses are fixed-point integers (units of 2^-40) relative
// to a power of two.  Inside its own range a CTA uses its own power 2^e_own;
// the head's thresholds use 2^E*, the largest of the covering CTAs' powers,
// and a threshold maps into the CTA's units exactly by a shift.  So all that
// needs the other CTAs comes last: a CTA publishes one aggregate per head of
// the (at most two) pieces it shares (max, and the mass in its own units),
// arrives at the one grid barrier, and while it waits stages its scores in
// shared memory and computes its chunk masses in its own units.  After the
// barrier one warp per head reads the covering CTAs' aggregates (about 20 at
// a 32K context), which give E*, the head's total mass Z and the prefix and
// mass of this CTA's range; places the thresholds that fall in the range; and
// resolves them one per lane: the chunk by a halving search over one 32-chunk
// window's prefixes (a warp scan), window after window, or, in a longer range,
// by bisection over prefixes formed in place first; the key by the chunk's 16
// key masses.  The head warps then gather their drawn V rows, each distinct
// row of a head once with its count, at the same time, so a row drawn by
// several heads of the KV group is read from memory once and served to the
// others from L2.  A piece wholly inside one range needs no other CTA and is
// done before the wait by all warps; the two shared pieces of a CTA run on two
// halves of the CTA at once.
//
// Difference from the pages' kernels: Alg. 4 rounds per-tile budgets by
// largest remainder and samples each tile on its own; here the S thresholds of
// a head are placed globally and each CTA resolves the ones in its own mass
// interval, which reproduces the global i.i.d. / stratified / systematic
// estimators.  Thresholds are exact integers, theta_j = floor(t_j * Z), with
// t_j a rational of 24-bit uniforms, so no FP64 arithmetic runs per draw.
#pragma once

#include <climits>

#include "santa_common.cuh"
#include "santa_launch.h"
#include "santa_seq.cuh"
#include "santa_grid.cuh"
#include "santa_part.cuh"
#include "santa_tma.cuh"
#include "santa_window.cuh"

// Phase boundaries of one CTA, for timing builds that define SANTA_STAMP
// (thread 0 records the global timer at boundary k); nothing otherwise.
#ifndef SANTA_STAMP
#define SANTA_STAMP(k) ((void)0)
#endif

namespace santa {

constexpr int FW = 16;              // warps per CTA
constexpr int FT = FW * 32;         // threads per CTA
constexpr int REG = 64 * 1024;      // phase-B shared-memory region
constexpr int BAR_G0 = 1, BAR_G1 = 2, BAR_INT = 3;   // named barriers of the phase-B groups
constexpr int BAR_FIN = 4;                             // the shared pieces' head warps after the grid wait
constexpr int STATS_CAP = 1024;     // (block, head) statistics a CTA keeps in shared memory
constexpr int STG_ROW = 20;         // floats per head row of a warp's score staging (16 keys, padded)

template <int D>
struct FGeom {
  static constexpr int STAGE = BK * D * 2;               // bytes of one block of K
  static constexpr int NSTAGE = D == 128 ? 3 : 6;        // ring depth per warp (same bytes in flight)
  static constexpr int RING = FW * NSTAGE * STAGE;       // 192 KiB
  static constexpr size_t SMEM = (size_t)RING + 1024;    // + alignment of the swizzled stages
  static constexpr int CPL = D / 32;                     // output columns per lane in the gather
  static constexpr int CPB = BK * D / 8 / 32;            // 16-byte copies per lane per block (cp.async path)
  static_assert(RING >= 3 * REG, "phase-B regions fit the ring");
};

// ---------------------------------------------------------------------------
// Exact thresholds.  A threshold is theta = floor(N * Z / (div * 2^24)) for an
// integer numerator N < div * 2^24:
//   systematic  N = j * 2^24 + k          (k: the head's one 24-bit uniform), div = S_b
//   stratified  N = j * 2^24 + k_j        (k_j: uniform j),                  div = S_b
//   i.i.d.      N = k_(j), sorted keys,                                      div = 1
// so theta_j = floor(t_j * Z) with t_j = (j + u_j) / S_b or u_(j), u = k 2^-24.
// ---------------------------------------------------------------------------
struct ThetaCtx {
  unsigned long long Zq, Zr;  // Z / div, Z % div
  unsigned long long rcp;     // ceil(2^64 / div) (div > 1)
  unsigned div;
  long long Z;
};
// rcp = ceil(2^64 / div) when div > 1 (precomputed: a 64-bit division is slow here)
__device__ __forceinline__ ThetaCtx theta_ctx_rcp(long long Z, unsigned div, unsigned long long rcp) {
  ThetaCtx c;
  c.Z = Z;
  c.div = div;
  c.rcp = rcp;
  if (div > 1) {
    // Z < 2^62: mulhi(Z, rcp) is floor(Z / div) or one more
    unsigned long long q = __umul64hi((unsigned long long)Z, c.rcp);
    if (q * div > (unsigned long long)Z) --q;
    c.Zq = q;
    c.Zr = (unsigned long long)Z - q * div;
  } else {
    c.Zq = (unsigned long long)Z;
    c.Zr = 0ull;
  }
  return c;
}
// floor(N Z / (div 2^24)) = floor((N Zq + floor(N Zr / div)) / 2^24), exact in 128 bits.
// N Zr < 2^36 * 2^12 = 2^48 and div <= 2^12, so the quotient by multiply-high
// with rcp is exact: its error is below 2^-16 while the fraction of a
// non-integer quotient is at most 1 - 2^-12.
__device__ __forceinline__ long long theta_of(const ThetaCtx& c, unsigned long long N) {
  unsigned long long lo = N * c.Zq, hi = __umul64hi(N, c.Zq);
  const unsigned long long add = c.div > 1 ? __umul64hi(N * c.Zr, c.rcp) : 0ull;
  lo += add;
  hi += (lo < add) ? 1ull : 0ull;
  return (long long)((hi << 40) | (lo >> 24));
}

template <int V>
struct Draws {
  int S, h, b;
  uint32_t step, k0, k1;
  uint32_t ksys;               // systematic: the head's uniform key
  const uint32_t* sorted;      // i.i.d.: the head's sorted uniform keys
  ThetaCtx tc;

  __device__ __forceinline__ uint32_t key_at(int j) const {
    const uint4 w = philox4x32_10(make_uint4((uint32_t)(j >> 2), (uint32_t)h, (uint32_t)b, step), k0, k1);
    const uint32_t x = (j & 3) == 0 ? w.x : (j & 3) == 1 ? w.y : (j & 3) == 2 ? w.z : w.w;
    return x >> 8;
  }
  __device__ __forceinline__ long long theta(int j) const {
    if constexpr (V == VAR_IID) return theta_of(tc, sorted[j]);
    const uint32_t k = V == VAR_SYS ? ksys : key_at(j);
    return theta_of(tc, ((unsigned long long)j << 24) | k);
  }
  __device__ __forceinline__ int count_serial(long long X, int e) const {
    while (e > 0 && theta(e - 1) >= X) --e;
    while (e < S && theta(e) < X) ++e;
    return e;
  }
  // {#{j < S : theta_j < X1}, #{j < S : theta_j < X2}} (thresholds are
  // non-decreasing in j), computed by the whole warp.
  __device__ __forceinline__ int2 count2(long long X1, long long X2, int lane) const {
    if constexpr (V != VAR_IID) {
      // theta_j lies in [floor(j Z / S), floor((j + 1) Z / S)]: a count is
      // within 2 of e = trunc(X S / Z).  Lanes 0..7 test the window
      // [e1 - 4, e1 + 4) of X1, lanes 8..15 that of X2, in one ballot.
      const long long X = (lane & 8) ? X2 : X1;
      int e = 0;
      if (X >= tc.Z) e = S;
      else if (X > 0) {
        const int sh = max(0, 40 - __clzll(tc.Z));
        e = (int)(__fdividef((float)(uint32_t)(X >> sh), (float)(uint32_t)(tc.Z >> sh)) * (float)S);
        e = min(max(e, 0), S);
      }
      const int j = e - 4 + (lane & 7);
      const bool below = X > 0 && (j < 0 || (j < S && (X >= tc.Z || theta(j) < X)));
      const unsigned bal = __ballot_sync(FULL, below);
      int c[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const unsigned w = (bal >> (8 * q)) & 0xffu;
        const int eq = __shfl_sync(FULL, e, 8 * q);
        const long long Xq = q ? X2 : X1;
        if (Xq <= 0) c[q] = 0;
        else if (Xq >= tc.Z) c[q] = S;
        else if ((w & 1u) && !(w & 0x80u)) c[q] = eq - 4 + __popc(w);
        else c[q] = count_serial(Xq, eq);   // the window missed (never expected)
      }
      return make_int2(c[0], c[1]);
    } else {
      return make_int2(count_sorted(X1, lane), count_sorted(X2, lane));
    }
  }
  // sorted keys: 32-way search, one probe per lane and round
  __device__ __forceinline__ int count_sorted(long long X, int lane) const {
    if (X <= 0) return 0;
    if (X >= tc.Z) return S;
    int lo = 0, n = S;   // the count lies in [lo, lo + n]
    while (n > 0) {
      const int step = (n + 31) >> 5;
      const int p = lo + lane * step;
      const bool below = p < lo + n && theta(p) < X;
      const int c = __popc(__ballot_sync(FULL, below));
      if (c == 0) break;
      const int end = lo + n;
      lo = lo + (c - 1) * step + 1;
      n = min(step - 1, end - lo);
    }
    return lo;
  }
};

// ---------------------------------------------------------------------------
// Per-CTA aggregate of one head over the CTA's keys of a shared piece.
// Masses are taken relative to a power of two so that every reader rescales
// them exactly by a shift:
//   m  max score over the keys
//   e  ceil(m log2(e)), an integer
//   F  sum_n 2^(s_n log2(e) - e) in units of 2^-40 (rounded toward zero)
// With E* the largest e over the CTAs of a head, CTA k's mass relative to
// 2^E* is F_k >> (E* - e_k): the same integer in every CTA that computes it.
// ---------------------------------------------------------------------------
constexpr int AGG_EMPTY = -(1 << 30);   // e of a range with no finite score
struct __align__(16) Agg {
  float m;
  int e;
  long long F;
};
// from the max m and the natural-base sum l = sum_n exp(s_n - m)
__device__ __forceinline__ Agg make_agg(float m, float l) {
  Agg x;
  x.m = m;
  x.e = AGG_EMPTY;
  x.F = 0;
  if (m > -INFINITY) {
    const float t = m * LOG2E;
    x.e = (int)ceilf(t);
    x.F = mass_fixed(l * fast_exp2(t - (float)x.e));
  }
  return x;
}


// The CTA's share of the partition, as phase B reads it (shared memory).
struct CtaRange {
  Part pt;
  long long lo, hi;        // blocks [lo, hi)
  Cur cA, cB;              // blocks lo and hi - 1
  int has_range, first_shared, last_shared, has_interior, use_ss;
};

// One piece as seen by one CTA.
struct Piece {
  int b, kvh, nblk;
  int64_t row0, nk;
  long long pb_lo;
  int c_lo, c_hi;          // this CTA's key blocks (= statistics chunks) of the piece
  int i_first, i_last;     // CTAs covering the piece
};

// Per-head state of phase B (shared memory).  "Own units": relative to the
// CTA's power 2^e_own; "head units": relative to 2^E*.  A threshold theta in
// [pown, pown + town) maps to the own-unit offset (theta - pown) << d, d =
// E* - e_own, exactly.
struct HeadState {
  long long Z, pown, town;  // head units: total mass, prefix and mass of this range
  unsigned long long rcp;   // ceil(2^64 / S_b) (S_b > 1), for the thresholds
  uint32_t ksys;            // systematic: the head's uniform key
  float ref;                // e_own: masses are 2^(s log2(e) - e_own)
  float mstar;              // max score (the piece, when it is this CTA's alone)
  int d;                    // E* - e_own
};

// Shared-memory layout of a piece inside a phase-B region: per head, the
// own-unit masses of the range's chunks when they fit, then the range's
// scores when they fit too.
struct SegLayout {
  long long* w;             // [G][segc] own-unit chunk masses, or NULL (computed when needed)
  float* st;                // [G][capk] the range's scores (staged from the 16-byte boundary below), or NULL
  int segc, capk;
};

// ---------------------------------------------------------------------------
// i.i.d.: sorted 24-bit uniform keys of one head into ukeys (all threads of
// the CTA).  Up to 2048 keys: each key becomes the unique composite
// (key << 12) | index, each warp sorts a run of 32 composites by a bitonic
// network over its lanes, and a composite's rank is its place in its own run
// plus, for every other run, the number of that run's composites below it (a
// bisection of 32 sorted values): the order of the keys with equal keys by
// index, as a stable sort gives.  More keys: a bitonic network over the keys
// in shared memory.  `keys` holds at least 2048 composites.
// ---------------------------------------------------------------------------
static __device__ __noinline__ void sort_head_keys(int b, int h, int S_b, uint32_t step, uint32_t k0, uint32_t k1,
                                                  uint32_t* dst, uint32_t* keys) {
  const int tid = threadIdx.x, lane = tid & 31;
  auto key_of = [&](int i) {
    const uint4 w = philox4x32_10(make_uint4((uint32_t)(i >> 2), (uint32_t)h, (uint32_t)b, step), k0, k1);
    const uint32_t x = (i & 3) == 0 ? w.x : (i & 3) == 1 ? w.y : (i & 3) == 2 ? w.z : w.w;
    return x >> 8;
  };
  if (S_b <= 2048) {
    unsigned long long* ck = reinterpret_cast<unsigned long long*>(keys);
    const int nrun = (S_b + 31) >> 5;
    for (int i = tid; i < nrun * 32; i += FT) {   // whole warps: lane = place in the run
      unsigned long long c = i < S_b ? ((unsigned long long)key_of(i) << 12) | (unsigned)i : ~0ull;
#pragma unroll
      for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
          const unsigned long long o = __shfl_xor_sync(FULL, c, j);
          const bool up = (lane & k) == 0, low = (lane & j) == 0;
          c = (up == low) ? (c < o ? c : o) : (c < o ? o : c);
        }
      ck[i] = c;
    }
    __syncthreads();
    for (int i = tid; i < S_b; i += FT) {
      const unsigned long long c = ck[i];
      if (c == ~0ull) continue;
      const int r = i >> 5;
      int rank = i & 31;
      for (int q = 0; q < nrun; ++q) {
        if (q == r) continue;
        const unsigned long long* run = ck + 32 * q;
        int n = 0;   // composites of run q below c
        if (run[31] < c) {
          n = 32;
        } else {
#pragma unroll
          for (int half = 16; half > 0; half >>= 1)
            if (run[n + half - 1] < c) n += half;
        }
        rank += n;
      }
      dst[rank] = (uint32_t)(c >> 12);
    }
  } else {
    int S2 = 1;
    while (S2 < S_b) S2 <<= 1;
    for (int i = tid; i < S2; i += FT) keys[i] = i < S_b ? key_of(i) : 0xffffffffu;
    __syncthreads();
    for (int kk = 2; kk <= S2; kk <<= 1) {
      for (int jj = kk >> 1; jj > 0; jj >>= 1) {
        for (int i = tid; i < S2; i += FT) {
          const int ixj = i ^ jj;
          if (ixj > i) {
            const uint32_t x = keys[i], y = keys[ixj];
            if ((x > y) == ((i & kk) == 0)) {
              keys[i] = y;
              keys[ixj] = x;
            }
          }
        }
        __syncthreads();
      }
    }
    for (int i = tid; i < S_b; i += FT) dst[i] = keys[i];
  }
  __syncthreads();   // keys is rewritten for the next head
}

// ---------------------------------------------------------------------------
// The kernel.  V: the sampling variant.  TMA_K: K is read by TMA boxes
// through `tmap`; otherwise by per-lane 16-byte cp.async into the same
// swizzled stage layout (K in host memory read in place).
// ---------------------------------------------------------------------------
template <typename T, int D, int V, bool TMA_K>
__global__ void __launch_bounds__(FT, 1)
fused_decode_kernel(const __grid_constant__ CUtensorMap tmap, LaunchArgs a, unsigned* bar_count, unsigned* bar_gen) {
  using Gm = FGeom<D>;
  constexpr int NS = Gm::NSTAGE, STG = Gm::STAGE, CPL = Gm::CPL;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) unsigned long long s_bar[FW * NS];
  __shared__ float s_rm[2][FW][8], s_rl[2][FW][8];   // per-warp running statistics of the first / last piece
  __shared__ int s_eown[2][8];                        // exponent of each published aggregate
  // i.i.d. key sort (prologue), then each warp's score staging for the bulk
  // stores of the stream ([8 heads][STG_ROW] floats per warp)
  constexpr int AUX = (V == VAR_IID && MAX_S * 4 > FW * 8 * STG_ROW * 4) ? MAX_S * 4 : FW * 8 * STG_ROW * 4;
  __shared__ __align__(16) unsigned char s_aux[AUX];
  uint32_t* const s_keys = reinterpret_cast<uint32_t*>(s_aux);
  __shared__ Cur s_cur[2];                            // blocks lo and hi - 1 (ragged batches)
  __shared__ long long s_part[2];                     // T, q (ragged batches)
  __shared__ HeadState s_hs[3][8];                    // per phase-B group and head
  __shared__ float s_pm[FW];                          // pieces inside the range: per-warp partial max,
  __shared__ int s_pe[FW];                            // exponent
  __shared__ long long s_pz[FW];                      // and mass sum
  __shared__ float2 s_stats[STATS_CAP];               // the range's 16-key (max, exp-sum), when they fit
  __shared__ unsigned s_gen;
  __shared__ CtaRange s_rg;
  __shared__ Piece s_psh[2];                          // the range's first / last piece (phase B's shared pieces)
  __shared__ uint32_t s_ksys[2][8];                   // their heads' systematic keys
  __shared__ unsigned long long s_rcp[2];             // their sequences' ceil(2^64 / S_b)

  SANTA_STAMP(0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = gridDim.x, cta = blockIdx.x;
  const int G = a.H / a.Hkv;
  const uint32_t k0 = (uint32_t)a.seed, k1 = (uint32_t)(a.seed >> 32);
  unsigned char* const ring = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t ring_u32 = smem_addr(ring);
  if constexpr (TMA_K)
    if (tid == 0) prefetch_tensormap(&tmap);

  // ---- phase A: per-warp rings.  Warp w scores blocks lo + w + FW k,
  //      k < n_mine; the first NS are requested first, at once for uniform
  //      batches (their partition is closed form), after the scan of the
  //      lengths for ragged ones.
  const uint32_t wring = ring_u32 + (uint32_t)(warp * NS * STG);
  const uint32_t wbar = smem_addr(&s_bar[warp * NS]);
  const unsigned long long pol = evict_first_policy();   // K is read once per step
  if (TMA_K) {
    if (lane == 0)
      for (int s = 0; s < NS; ++s) mbar_init(wbar + 8 * s, 1);
    mbar_fence_init();
    __syncwarp();
  }
  // the end of the K buffer: B nk_max rows, or kv_offsets[B] for a ragged
  // batch (a box of the last sequence's last block may not reach past it)
  const int64_t row_end = a.kv_offsets ? a.kv_offsets[a.B] : (int64_t)a.B * a.nk_max;
  int n_mine = 0;
  Cur cur;    // block being scored
  cur.b = a.B;
  cur.kvh = cur.kblk = cur.nblk = 0;
  cur.row0 = cur.nk = 0;
  cur.pb_lo = LLONG_MAX;
  Cur prod = cur;   // block being requested
  const T* Kp = static_cast<const T*>(a.K);
  auto issue = [&](int k) {
    const int s = k % NS;
    const uint32_t dst = wring + (uint32_t)(s * STG);
    if (k < n_mine) {
      const int z = (int)(prod.row0 + (int64_t)prod.kblk * BK);
      if constexpr (TMA_K) {
        if (z + BK <= row_end) {
          if (lane == 0) {
            fence_proxy_async_smem();
            mbar_expect_tx(wbar + 8 * s, STG);
#pragma unroll
            for (int x = 0; x < D / 64; ++x)
              tma_load_3d(dst + x * 2048, &tmap, x * 64, prod.kvh, z, wbar + 8 * s, pol);
          }
        } else {   // a box would reach past the end of a ragged cache buffer
          fill_stage_plain<D>(dst, static_cast<const uint16_t*>(a.K), z, prod.kvh, a.Hkv, row_end, lane);
          __syncwarp();
          if (lane == 0) mbar_arrive(wbar + 8 * s);
        }
      } else {
        const int rows = (int)min((int64_t)BK, prod.nk - (int64_t)prod.kblk * BK);
        const T* src = Kp + ((int64_t)z * a.Hkv + prod.kvh) * D;
#pragma unroll
        for (int j = 0; j < Gm::CPB; ++j) {
          const int q = lane + 32 * j, r = q / (D / 8), c = q % (D / 8);
          if (r < rows) cp_async16_hint(dst + swz128_offset(r, c), src + (int64_t)r * a.Hkv * D + c * 8, pol);
        }
      }
      cur_advance(prod, a, FW);
    }
    if constexpr (!TMA_K) cp_async_commit();
  };
  if (!a.kv_offsets) {
    Part p0;
    p0.T = a.blk_total;
    p0.q = a.blk_q;
    p0.r = a.blk_r;
    p0.P = P;
    p0.rP = a.rdiv_grid;
    const long long l0 = p0.lo(cta), h0 = p0.lo(cta + 1);
    n_mine = h0 - l0 > warp ? (int)((h0 - l0 - warp + FW - 1) / FW) : 0;
    if (n_mine > 0) cur = locate_uniform(a, l0 + warp);
    prod = cur;
#pragma unroll 1
    for (int k = 0; k < NS; ++k) issue(k);
  }


  // ---- the CTA's block range: closed form for uniform batches (every thread,
  //      no wait), a scan of the lengths by one warp for ragged ones.  Kept in
  //      shared memory (s_rg) and read from there: no register holds it
  //      across the stream.
  {
    Part pt;
    pt.P = P;
    pt.rP = a.rdiv_grid;
    Cur cA, cB;
    if (!a.kv_offsets) {
      pt.T = a.blk_total;
      pt.q = a.blk_q;
      pt.r = a.blk_r;
    } else {
      if (warp == 0) {
        const long long Tb = total_blocks(a, lane);
        if (lane == 0) {
          s_part[0] = Tb;
          s_part[1] = Tb / P;
        }
      }
      __syncthreads();
      pt.T = s_part[0];
      pt.q = s_part[1];
      pt.r = (int)(pt.T - pt.q * P);
    }
    const long long lo = pt.lo(cta), hi = pt.lo(cta + 1);
    const bool has_range = hi > lo;
    if (!a.kv_offsets) {
      if (has_range) {
        cA = locate_uniform(a, lo);
        cB = locate_uniform(a, hi - 1);
      }
    } else {
      if (warp == 0 && has_range) {
        const Cur c0 = locate_block(a, lo, lane), c1 = locate_block(a, hi - 1, lane);
        if (lane == 0) {
          s_cur[0] = c0;
          s_cur[1] = c1;
        }
      }
      __syncthreads();
      cA = s_cur[0];
      cB = s_cur[1];
    }
    if (!has_range) {
      cA.b = cB.b = a.B;
      cA.pb_lo = cB.pb_lo = LLONG_MAX;
      cA.nblk = cB.nblk = INT_MAX;
    }
    // shared pieces: slot 0 = the first piece of the range, slot 1 = the last
    // (when it is another piece); a piece is shared when it crosses the range
    const bool first_shared = has_range && (cA.pb_lo < lo || cA.pb_lo + cA.nblk > hi);
    const bool two_pieces = has_range && cB.pb_lo != cA.pb_lo;
    const bool last_shared = two_pieces && cB.pb_lo + cB.nblk > hi;
    // a piece wholly inside the range: the first or last one unshared, or one between them
    const bool has_interior = has_range && (!first_shared || (two_pieces && !last_shared) ||
                                            cB.pb_lo > cA.pb_lo + cA.nblk);
    const bool use_ss = (hi - lo) * G <= STATS_CAP;   // the range's chunk statistics kept in shared memory
    if (tid == 0) {
      s_rg.pt = pt;
      s_rg.lo = lo;
      s_rg.hi = hi;
      s_rg.cA = cA;
      s_rg.cB = cB;
      s_rg.has_range = has_range;
      s_rg.first_shared = first_shared;
      s_rg.last_shared = last_shared;
      s_rg.has_interior = has_interior;
      s_rg.use_ss = use_ss;
    }
  }
  __syncthreads();
  const Part& pt = s_rg.pt;
  const long long &lo = s_rg.lo, &hi = s_rg.hi;
  const Cur &cA = s_rg.cA, &cB = s_rg.cB;
  const int &has_range = s_rg.has_range, &first_shared = s_rg.first_shared, &last_shared = s_rg.last_shared;
  const int &has_interior = s_rg.has_interior, &use_ss = s_rg.use_ss;
  auto piece_at = [&](const Cur& c) {
    Piece p;
    p.b = c.b;
    p.kvh = c.kvh;
    p.nblk = c.nblk;
    p.row0 = c.row0;
    p.nk = c.nk;
    p.pb_lo = c.pb_lo;
    p.c_lo = (int)(max(lo, c.pb_lo) - c.pb_lo);
    p.c_hi = (int)(min(hi, c.pb_lo + c.nblk) - c.pb_lo);
    p.i_first = pt.cta_of(c.pb_lo);
    p.i_last = pt.cta_of(c.pb_lo + c.nblk - 1);
    return p;
  };
  // the pieces phase B may share with other CTAs, and their threshold
  // constants, while the first blocks are in flight (read after the stream)
  if (has_range && warp == FW - 1) {
    if (lane < 2) {
      const Cur& c = lane == 0 ? cA : cB;
      s_psh[lane] = piece_at(c);
      const int S_b = a.S_per_seq ? a.S_per_seq[c.b] : a.S_max;
      s_rcp[lane] = (V != VAR_IID && S_b > 1) ? ~0ull / (unsigned)S_b + 1ull : 0ull;
    } else if (V == VAR_SYS && lane >= 16) {
      const int slot = (lane >> 3) & 1, g = lane & 7;
      const Cur& c = slot == 0 ? cA : cB;
      if (g < G)
        s_ksys[slot][g] =
            philox4x32_10(make_uint4(0u, (uint32_t)(c.kvh * G + g), (uint32_t)c.b, a.step), k0, k1).x >> 8;
    }
  }
  SANTA_STAMP(1);

  // ragged batches: the ring starts once the partition is known
  if (a.kv_offsets) {
    n_mine = has_range && hi - lo > warp ? (int)((hi - lo - warp + FW - 1) / FW) : 0;
    cur = cA;
    if (n_mine > 0) cur_advance(cur, a, warp);
    prod = cur;
#pragma unroll 1
    for (int k = 0; k < NS; ++k) issue(k);
  }

  // ---- prologue work while the first blocks are in flight
  // the barrier generation before this launch's arrivals (no CTA of this
  // launch can advance it before this one has arrived)
  if (tid == 32) {
    s_gen = ld_acquire(bar_gen);
    // launches alternate between two arrival counters; this launch's first
    // CTA clears the other one for the next launch (the previous launch,
    // which used it, has completed)
    if (cta == 0) bar_count[((s_gen & 1u) ^ 1u) * 32] = 0u;
  }
  if (lane < 16) {   // each warp clears its own running-statistics slots
    s_rm[lane >> 3][warp][lane & 7] = -INFINITY;
    s_rl[lane >> 3][warp][lane & 7] = 0.f;
  }
  // sequence metadata (sequence b checked by CTA b mod P): a sequence the
  // device rejects gets zero outputs and -1 sample slots
  for (int b = cta; b < a.B; b += P) {
    int S_b;
    const int e = seq_error(a, b, S_b);
    if (e) {
      if (tid == 0) flag_error(a.err, e);
      if (a.out) {
        float4* o = reinterpret_cast<float4*>(a.out + (int64_t)b * a.H * D);
        for (int i = tid; i < a.H * D / 4; i += FT) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (a.sample_idx && !a.score_only)
        for (int i = tid; i < a.H * a.S_max; i += FT) a.sample_idx[(int64_t)b * a.H * a.S_max + i] = -1;
    }
  }
  // pieces that start in this range: outputs of shared pieces to zero (their
  // CTAs add into them after the barrier), unused sample slots to -1, and the
  // i.i.d. keys this CTA sorts (head g of a piece: covering CTA i_first + g)
  if (has_range) {
    Cur pc = cA;
    while (pc.b < a.B && pc.pb_lo < hi) {
      int S_b;
      const bool needed = (pc.pb_lo >= lo || V == VAR_IID) && !seq_error(a, pc.b, S_b);
      if (needed) {
        const Piece p = piece_at(pc);
        const int64_t bh0 = (int64_t)p.b * a.H + (int64_t)p.kvh * G;
        if (p.pb_lo >= lo && !a.score_only) {
          if (p.i_first != p.i_last) {
            float4* o = reinterpret_cast<float4*>(a.out + bh0 * D);
            for (int i = tid; i < G * D / 4; i += FT) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
          if (a.sample_idx && S_b < a.S_max)
            for (int i = tid; i < G * (a.S_max - S_b); i += FT)
              a.sample_idx[(bh0 + i / (a.S_max - S_b)) * a.S_max + S_b + i % (a.S_max - S_b)] = -1;
        }
        if constexpr (V == VAR_IID)
          for (int g = 0; g < G && !a.score_only; ++g) {
            int sorter = p.i_first + g;
            if (sorter > p.i_last || !pt.nonempty(sorter)) sorter = p.i_first;
            if (sorter == cta)
              sort_head_keys(p.b, p.kvh * G + g, S_b, a.step, k0, k1, a.ukeys + (bh0 + g) * a.S_max, s_keys);
          }
      }
      pc.kblk = pc.nblk;
      cur_norm(pc, a);
    }
  }

  // ---- phase A: the stream
  SANTA_STAMP(2);
  {
    const int g8 = lane >> 2, t4 = lane & 3;
    const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;   // ldmatrix row of this lane
    const int lhalf = lane >> 4;                           // ldmatrix 8-column half of this lane
    float rm[2] = {-INFINITY, -INFINITY}, rl[2] = {0.f, 0.f};   // running statistics, heads 2*t4 + hh
    long long run_piece = cur.pb_lo;
    auto flush = [&]() {   // running statistics of run_piece into its slot (first / last piece only)
      const int slot = run_piece == cA.pb_lo ? 0 : (run_piece == cB.pb_lo ? 1 : -1);
      if (slot >= 0 && lane < 4) {
        s_rm[slot][warp][2 * lane] = rm[0];
        s_rm[slot][warp][2 * lane + 1] = rm[1];
        s_rl[slot][warp][2 * lane] = rl[0];
        s_rl[slot][warp][2 * lane + 1] = rl[1];
      }
      rm[0] = rm[1] = -INFINITY;
      rl[0] = rl[1] = 0.f;
    };
    const T* qp = static_cast<const T*>(a.q);
    // scores of full blocks go out through this warp's staging rows as one
    // 16-byte store per lane (4 keys of one head; rows start 16-byte aligned
    // when nk_max is a multiple of 4), the rest as plain stores
    float* const stg = reinterpret_cast<float*>(s_aux) + warp * (8 * STG_ROW);
    const bool vec_ok = (a.nk_max & 3) == 0;
    bool ring_dead = false;
    uint32_t bq[D / 16][2];
    int bq_b = -1, bq_kvh = -1;
    for (int k = 0; k < n_mine; ++k) {
      const int s = k % NS;
      if constexpr (TMA_K) {
        // after one expired wait the warp stops waiting (its results are void, the error word says so)
        if (!ring_dead && !mbar_wait(wbar + 8 * s, (unsigned)((k / NS) & 1), a.err)) ring_dead = true;
      } else {
        cp_async_wait<NS - 1>();
      }
      __syncwarp();
      if (cur.pb_lo != run_piece) {
        flush();
        run_piece = cur.pb_lo;
      }
      const int64_t bh0 = (int64_t)cur.b * a.H + (int64_t)cur.kvh * G;
      if (cur.b != bq_b || cur.kvh != bq_kvh) {   // q fragments change only with the piece
        const T* qg = qp + bh0 * D;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const T* q2 = qg + g8 * D + ks * 16 + t4 * 2;
          bq[ks][0] = (g8 < G) ? *reinterpret_cast<const uint32_t*>(q2) : 0u;
          bq[ks][1] = (g8 < G) ? *reinterpret_cast<const uint32_t*>(q2 + 8) : 0u;
        }
        bq_b = cur.b;
        bq_kvh = cur.kvh;
      }
      // 16 keys x 8 heads on the tensor cores, two independent accumulators,
      // the A fragments (16 keys x 16 dims) read from the stage two at a time;
      // then the stage is free for the block NS ahead
      const uint32_t sbase = wring + (uint32_t)(s * STG);
      float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < D / 16; ks += 2) {
        uint32_t f0[4], f1[4];
        ldmatrix_x4(sbase + swz128_offset(lrow, ks * 2 + lhalf), f0);
        ldmatrix_x4(sbase + swz128_offset(lrow, ks * 2 + 2 + lhalf), f1);
        Mma<T>::run(acc0, f0, bq[ks][0], bq[ks][1]);
        Mma<T>::run(acc1, f1, bq[ks + 1][0], bq[ks + 1][1]);
      }
      __syncwarp();
      issue(k + NS);
      // lane holds keys g8 and g8 + 8 of the block for heads 2*t4 and 2*t4 + 1
      const int64_t key0 = (int64_t)cur.kblk * BK;
      const bool ok0 = key0 + g8 < cur.nk, ok1 = key0 + g8 + 8 < cur.nk;
      const bool vec = vec_ok && key0 + BK <= cur.nk;   // warp-uniform
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int head = 2 * t4 + hh;
        const float s0 = (acc0[hh] + acc1[hh]) * a.scale, s1 = (acc0[2 + hh] + acc1[2 + hh]) * a.scale;
        if (head < G) {
          if (vec) {
            stg[head * STG_ROW + g8] = s0;
            stg[head * STG_ROW + g8 + 8] = s1;
          } else {
            float* sp = a.stash + (bh0 + head) * a.nk_max + key0 + g8;
            if (ok0) sp[0] = s0;
            if (ok1) sp[8] = s1;
          }
        }
        float m = fmaxf(ok0 ? s0 : -INFINITY, ok1 ? s1 : -INFINITY);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
        float l = (ok0 ? fast_exp(s0 - m) : 0.f) + (ok1 ? fast_exp(s1 - m) : 0.f);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(FULL, l, o);
        if (g8 == 0 && head < G) {
          if (use_ss) {   // written out after the stream
            s_stats[(warp + FW * k) * G + head] = make_float2(m, l);
          } else {
            a.tile_max[(bh0 + head) * a.chunks_max + cur.kblk] = m;
            a.tile_sum[(bh0 + head) * a.chunks_max + cur.kblk] = l;
          }
        }
        const float nm = fmaxf(rm[hh], m);
        rl[hh] = rl[hh] * fast_exp(rm[hh] - nm) + l * fast_exp(m - nm);
        rm[hh] = nm;
      }
      if (vec) {
        __syncwarp();
        if (lane < 4 * G) {
          const float4 v = *reinterpret_cast<const float4*>(stg + (lane >> 2) * STG_ROW + (lane & 3) * 4);
          *reinterpret_cast<float4*>(a.stash + (bh0 + (lane >> 2)) * a.nk_max + key0 + (lane & 3) * 4) = v;
        }
      }
      cur_advance(cur, a, FW);
    }
    if constexpr (!TMA_K) cp_async_wait_all();
    if (n_mine > 0) flush();
  }
  __syncthreads();   // statistics of the range written; the ring is free
  SANTA_STAMP(3);

  // The range's 16-key statistics, kept in shared memory during the stream,
  // out to the workspace (all threads; while the grid barrier is pending).
  auto write_tile_stats = [&]() {
    if (!use_ss || !has_range) return;
    Cur pc = cA;
    while (pc.b < a.B && pc.pb_lo < hi) {
      const long long x0 = max(lo, pc.pb_lo), x1 = min(hi, pc.pb_lo + pc.nblk);
      const int n = (int)(x1 - x0) * G, kb0 = (int)(x0 - pc.pb_lo), j0 = (int)(x0 - lo);
      const int64_t bh0 = (int64_t)pc.b * a.H + (int64_t)pc.kvh * G;
      for (int i = tid; i < n; i += FT) {
        const int jb = i / G, hd = i - jb * G;
        const float2 st = s_stats[(j0 + jb) * G + hd];
        const int64_t o = (bh0 + hd) * a.chunks_max + kb0 + jb;
        a.tile_max[o] = st.x;
        a.tile_sum[o] = st.y;
      }
      pc.kblk = pc.nblk;
      cur_norm(pc, a);
    }
  };
  if (a.score_only) {   // the score pass alone: the statistics out, no draws
    write_tile_stats();
    return;
  }

  // phase-B regions of the ring: 0 and 1 for the shared pieces (one piece
  // alone takes both), 2 for the pieces inside the range
  const int n_shared = (first_shared ? 1 : 0) + (last_shared ? 1 : 0);
  unsigned char* const regions = ring;
  auto seg_layout = [&](unsigned char* reg, int reg_bytes, int nch_part) {
    SegLayout L;
    // per head: the range's chunk masses in own units (8 bytes each) when
    // they fit, then its scores when they fit too
    L.segc = (nch_part + 3) & ~3;
    L.w = reinterpret_cast<long long*>(reg);
    const int used = G * L.segc * 8;
    const bool w_fit = used + 64 <= reg_bytes;
    if (!w_fit) L.w = nullptr;
    L.capk = BK * nch_part + 8;
    const int off = w_fit ? ((used + 15) & ~15) : 0;
    L.st = off + 16 + G * L.capk * 4 <= reg_bytes ? reinterpret_cast<float*>(reg + off) : nullptr;
    return L;
  };
  // Copies the range's scores of piece p (rows from the 16-byte boundary at
  // or below their first element) into L.st: threads tg of nthr, one commit
  // group per thread.
  auto stage_scores = [&](const Piece& p, const SegLayout& L, int tg, int nthr) {
    const int64_t bh0 = (int64_t)p.b * a.H + (int64_t)p.kvh * G;
    const int64_t key0 = (int64_t)p.c_lo * BK;
    const int nkeys = (int)(min((int64_t)p.c_hi * BK, p.nk) - key0);
    for (int h = 0; h < G; ++h) {
      const int64_t g0 = (bh0 + h) * a.nk_max + key0, a0 = g0 & ~(int64_t)3;
      const int n16 = (int)((g0 + nkeys - a0 + 3) >> 2);
      float* row = L.st + h * L.capk;
      for (int j = tg; j < n16; j += nthr) cp_async16(smem_addr(row + 4 * j), a.stash + a0 + 4 * j);
    }
    cp_async_commit();
  };

  // ---- aggregates of the shared pieces (16 lanes per head combine the 16
  //      warps' running statistics), then arrival at the grid barrier; the
  //      other 8 warps meanwhile copy the shared pieces' scores into their
  //      regions (waited for before the grid wait)
  if (tid >= 256) {
    for (int slot = 0; slot < 2; ++slot) {
      if (!(slot == 0 ? first_shared : last_shared)) continue;
      const Piece p = s_psh[slot];
      const SegLayout L = seg_layout(regions + (n_shared == 2 ? slot * REG : 0), n_shared == 2 ? REG : 2 * REG,
                                     p.c_hi - p.c_lo);
      if (L.st) stage_scores(p, L, tid - 256, FT - 256);
    }
  } else {
    const int slot = tid >> 7, g = (tid >> 4) & 7, w = tid & 15;
    const float m = s_rm[slot][w][g], l = s_rl[slot][w][g];
    float mm = m;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(FULL, mm, o, 16));
    float ll = m > -INFINITY ? l * expf(m - mm) : 0.f;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) ll += __shfl_xor_sync(FULL, ll, o, 16);
    const bool pub = (slot == 0 ? first_shared : last_shared) && g < G;
    if (pub && w == 0) {
      const Cur& c = slot == 0 ? cA : cB;
      const int64_t bh = (int64_t)c.b * a.H + (int64_t)c.kvh * G + g;
      const Agg x = make_agg(mm, ll);
      reinterpret_cast<Agg*>(a.agg)[bh * MAX_CTAS + cta] = x;
      s_eown[slot][g] = x.e;
    }
  }
  __syncthreads();
  SANTA_STAMP(4);
  unsigned* const arrivals = bar_count + (s_gen & 1u) * 32;   // this launch's arrival counter
  // arrival: nothing to wait for, but its release holds the issuing warp for
  // a memory round trip, so it comes from the last warp (no head's warp
  // unless two shared pieces of 8 heads use every warp)
  if (tid == FT - 32) red_release_add(arrivals, 1u);
  SANTA_STAMP(5);

  // =====================================================================
  // phase B
  // =====================================================================
  // Chunk c of head g of piece p (a chunk of this range) as an aggregate:
  // exponent e_c and mass relative to 2^e_c, from its 16-key statistics
  // (kept in shared memory during the stream when the range's chunks fit)
  auto chunk_stats = [&](const Piece& p, int g, int c) {
    if (use_ss) return s_stats[(int)(p.pb_lo + c - lo) * G + g];
    const int64_t gi2 = ((int64_t)p.b * a.H + (int64_t)p.kvh * G + g) * a.chunks_max + c;
    return make_float2(a.tile_max[gi2], a.tile_sum[gi2]);
  };
  auto chunk_agg = [&](const Piece& p, int g, int c) {
    const float2 st = chunk_stats(p, g, c);
    return make_agg(st.x, st.y);
  };
  // Own-unit mass of a chunk with statistics st: its mass relative to 2^e_c
  // shifted to the CTA's power 2^e_own (e_own >= e_c), as T_k of an aggregate.
  auto stats_mass = [&](float2 st, int e_own) {
    const Agg x = make_agg(st.x, st.y);
    const int dd = e_own - x.e;
    return dd < 63 ? (x.F >> dd) : 0ll;
  };
  // the same for chunk c of head g of piece p
  auto chunk_mass = [&](const Piece& p, int g, int c, int e_own) { return stats_mass(chunk_stats(p, g, c), e_own); };

  // Preparation of one piece by one group of nw warps (warps w0 .. w0 + nw -
  // 1; named barrier bar_id) in region reg, needing nothing from other CTAs:
  // per head (warp w0 + g) the own power e_own, the threshold constants
  // (budget reciprocal, systematic key), the own-unit chunk masses when they
  // fit in the region (by the whole group) and, for a piece wholly inside
  // this range, Z; and the range's scores staged when they fit.  Not
  // synchronised at the end.
  auto prep_piece = [&](const Piece& p, const SegLayout& L, bool shared, int slot, int gid, int bar_id, int w0,
                        int nw) {
    const int wl = warp - w0, tg = tid - w0 * 32, nthr = nw * 32;
    int S_b;
    if (seq_error(a, p.b, S_b)) return;
    SANTA_STAMP(16);
    const int nch = p.c_hi - p.c_lo;
    if (shared) {
      // the range's part of a shared piece: its heads' constants, and its
      // chunk masses at the published powers by the whole group (their
      // prefixes are formed while the draws are resolved)
      if (tg < G) {
        HeadState& H = s_hs[gid][tg];
        H.ref = (float)s_eown[slot][tg];
        H.rcp = s_rcp[slot];
        if constexpr (V == VAR_SYS) H.ksys = s_ksys[slot][tg];
      }
      if (L.w) {
        const int cpw = (nch + 31) & ~31;   // chunks per head, rounded to whole warps
        for (int it = tg; it < G * cpw; it += nthr) {
          const int h = it / cpw, c = it - h * cpw;
          if (c < nch) L.w[h * L.segc + c] = chunk_mass(p, h, p.c_lo + c, s_eown[slot][h]);
        }
      }
      SANTA_STAMP(22);
      return;
    }
    // a piece wholly inside the range: its scores, copied while the rest is
    // prepared; per head: the threshold constants (lane 0 of warp w0 + g);
    // by wph = nw / G warps per head, each a stride of the chunks with its
    // loads in flight, combined through shared memory: the max score, e_own
    // the max of the chunks' exponents, then the chunk masses at 2^e_own and
    // Z their exact sum
    if (L.st) stage_scores(p, L, tg, nthr);
    SANTA_STAMP(17);
    if (wl < G && lane == 0) {
      HeadState& H = s_hs[gid][wl];
      H.rcp = (V != VAR_IID && S_b > 1) ? ~0ull / (unsigned)S_b + 1ull : 0ull;
      H.ksys = V == VAR_SYS ? philox4x32_10(make_uint4(0u, (uint32_t)(p.kvh * G + wl), (uint32_t)p.b, a.step), k0,
                                            k1).x >> 8
                            : 0u;
    }
    const int wph = nw / G, hh = wl / wph, sub = wl - hh * wph;
    const bool mine = hh < G;   // warps past G * wph sit the passes out
    float mloc = -INFINITY;
    int eloc = AGG_EMPTY;
    if (mine) {
#pragma unroll 8
      for (int c = sub * 32 + lane; c < nch; c += wph * 32) {
        const float m = chunk_stats(p, hh, c).x;
        mloc = fmaxf(mloc, m);
        eloc = max(eloc, m > -INFINITY ? (int)ceilf(m * LOG2E) : AGG_EMPTY);
      }
    }
    mloc = warp_max(mloc);
    eloc = __reduce_max_sync(FULL, eloc);
    if (lane == 0) {
      s_pm[wl] = mloc;
      s_pe[wl] = eloc;
    }
    group_sync(bar_id, nthr);
    int e_own = AGG_EMPTY;
    if (mine)
      for (int k = 0; k < wph; ++k) e_own = max(e_own, s_pe[hh * wph + k]);
    long long Z = 0;
    if (mine) {
#pragma unroll 8
      for (int c = sub * 32 + lane; c < nch; c += wph * 32) {
        const long long m = stats_mass(chunk_stats(p, hh, c), e_own);
        if (L.w) L.w[hh * L.segc + c] = m;
        Z += m;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(FULL, Z, o);
    if (lane == 0) s_pz[wl] = Z;
    group_sync(bar_id, nthr);
    if (tg < G) {
      HeadState& H = s_hs[gid][tg];
      float mstar = -INFINITY;
      long long Zh = 0;
      int eh = AGG_EMPTY;
      for (int k = 0; k < wph; ++k) {
        mstar = fmaxf(mstar, s_pm[tg * wph + k]);
        Zh += s_pz[tg * wph + k];
        eh = max(eh, s_pe[tg * wph + k]);
      }
      H.ref = (float)eh;
      H.mstar = mstar;
      H.Z = Zh;
      H.pown = 0;
      H.town = Zh;
      H.d = 0;
    }
    SANTA_STAMP(22);
  };

  // The rest of one piece (same group, region and layout as its
  // preparation), one warp per head with no further synchronisation: Z, the
  // range's prefix pown and mass town and d (from the other CTAs' aggregates
  // when shared); the range's thresholds, resolved one per lane (chunk by a
  // search of the prefixes, key by the chunk's 16 key masses); the drawn V
  // rows, each distinct key of the head once with its count, gathered four
  // at a time; the sums, times 1/S_b, into out.  The G head warps of a piece
  // gather at the same time, so a row drawn by several heads of the KV group
  // is fetched from memory once and served to the others from L2.
  auto finish_piece = [&](const Piece& p, const SegLayout& L, bool shared, int gid, int bar_id, int w0, int nw) {
    const int wl = warp - w0, nthr = nw * 32;
    int S_b;
    if (seq_error(a, p.b, S_b)) return;   // the same in every thread of the group
    if (!shared) {   // the preparation's state and staged scores visible (a shared piece: by the grid wait)
      cp_async_wait_all();
      group_sync(bar_id, nthr);
    }
    SANTA_STAMP(20);
    if (wl < G) {
      const int64_t bh0 = (int64_t)p.b * a.H + (int64_t)p.kvh * G, bh = bh0 + wl;
      const HeadState& H = s_hs[gid][wl];
      Draws<V> dr;
      dr.S = S_b;
      dr.b = p.b;
      dr.h = p.kvh * G + wl;
      dr.step = a.step;
      dr.k0 = k0;
      dr.k1 = k1;
      dr.sorted = a.ukeys + bh * a.S_max;
      dr.ksys = H.ksys;
      const float ref = H.ref;
      long long Z, pown, town;
      int d = 0;
      if (shared) {
        // the covering CTAs' aggregates (one per lane): E* by a max, then the
        // masses relative to it, their prefix, this range's prefix and mass
        const Agg* ag = reinterpret_cast<const Agg*>(a.agg) + bh * MAX_CTAS;
        const int ncov = p.i_last - p.i_first + 1;
        Agg x0;
        x0.m = -INFINITY;
        x0.e = AGG_EMPTY;
        x0.F = 0;
        if (lane < ncov && pt.nonempty(p.i_first + lane)) x0 = ag[p.i_first + lane];
        int emax = __reduce_max_sync(FULL, x0.e);
        float mstar = x0.m;
        for (int i = p.i_first + 32 + lane; i - lane <= p.i_last; i += 32) {   // more than 32 covering CTAs
          int e = AGG_EMPTY;
          if (i <= p.i_last && pt.nonempty(i)) {
            e = ag[i].e;
            mstar = fmaxf(mstar, ag[i].m);
          }
          emax = max(emax, __reduce_max_sync(FULL, e));
        }
        SANTA_STAMP(21);
        long long carry = 0;
        pown = town = 0;
        for (int base = 0; base < ncov; base += 32) {
          Agg x = x0;
          if (base > 0) {
            x.e = AGG_EMPTY;
            x.F = 0;
            const int i = p.i_first + base + lane;
            if (base + lane < ncov && pt.nonempty(i)) x = ag[i];
          }
          const int dd = emax - x.e;
          const long long Ti = dd < 63 ? (x.F >> dd) : 0;
          const long long incl = warp_inclusive_scan(Ti, lane) + carry;
          if (p.i_first + base + lane == cta) {
            pown = incl - Ti;
            town = Ti;
          }
          carry = __shfl_sync(FULL, incl, 31);
        }
        Z = carry;
        const int own = (cta - p.i_first) & 31;   // the lane that held this CTA
        pown = __shfl_sync(FULL, pown, own);
        town = __shfl_sync(FULL, town, own);
        d = emax - (int)ref;
        if (cta == p.i_first) {
          mstar = warp_max(mstar);
          if (lane == 0) a.head_max[bh] = mstar;
        }
      } else {
        Z = H.Z;
        pown = H.pown;
        town = H.town;
        if (lane == 0) a.head_max[bh] = H.mstar;
      }
      SANTA_STAMP(19);
      dr.tc = theta_ctx_rcp(Z, V == VAR_IID ? 1u : (unsigned)S_b, H.rcp);
      const bool none = town == 0 || d > 61;   // no threshold falls in this range
      const int2 jr = dr.count2(pown, none ? pown : pown + town, lane);
      SANTA_STAMP(9);
      const T* Vb = static_cast<const T*>(a.V) + (p.row0 * a.Hkv + p.kvh) * (int64_t)D + lane * CPL;
      float acc[CPL];
#pragma unroll
      for (int k = 0; k < CPL; ++k) acc[k] = 0.f;
      // The range's chunks 32 at a time (lane = chunk): their own-unit masses
      // (from the preparation when they fit in shared memory) and, by one
      // 64-bit warp scan carried from window to window, their exact prefixes.
      // Thresholds are non-decreasing, so a window once passed is never needed
      // again; the last window's end is the range's total, past which a
      // threshold (the rounding gap) takes the last chunk with nonzero mass.
      // A range of more than one window whose masses are in shared memory
      // instead turns them into inclusive prefixes in place (four windows at
      // a time, interleaved scans) and each lane bisects them.
      const int nch = p.c_hi - p.c_lo, e_own = (int)ref;
      int wc0 = 0, lastnz = -1;
      long long wcarry = 0, m_l = 0, incl_l = 0;
      bool win = false;
      const bool bis = L.w != nullptr && nch > 32;
      long long* const wrow = L.w ? L.w + wl * L.segc : nullptr;
      if (bis) {
        long long carry = 0;
        for (int c0 = 0; c0 < nch; c0 += 128) {
          long long v4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = c0 + 32 * u + lane;
            v4[u] = c < nch ? wrow[c] : 0ll;
            const unsigned nzb = __ballot_sync(FULL, v4[u] > 0);
            if (nzb) lastnz = c0 + 32 * u + 31 - __clz((int)nzb);
          }
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const long long y = __shfl_up_sync(FULL, v4[u], o);
              if (lane >= o) v4[u] += y;
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = c0 + 32 * u + lane;
            if (c < nch) wrow[c] = v4[u] + carry;
            carry += __shfl_sync(FULL, v4[u], 31);
          }
        }
        __syncwarp();   // the prefixes visible to the warp
      }
      auto load_window = [&]() {
        const int c = wc0 + lane;
        m_l = c < nch ? (L.w ? L.w[wl * L.segc + c] : chunk_mass(p, wl, p.c_lo + c, e_own)) : 0ll;
        incl_l = warp_inclusive_scan(m_l, lane) + wcarry;
        const unsigned nzb = __ballot_sync(FULL, m_l > 0);
        if (nzb) lastnz = wc0 + 31 - __clz((int)nzb);
        win = true;
      };
      SANTA_STAMP(10);
      for (int jb = jr.x; jb < jr.y; jb += 32) {
        // ---- thresholds jb .. jb + 31, one per lane
        const int jj = jb + lane;
        const bool valid = jj < jr.y;
        const long long x = valid ? (dr.theta(jj) - pown) << d : 0ll;   // own-unit offset in this range
        SANTA_STAMP(18);
        int c = -1;
        long long xc = 0;
        bool pending = valid;
        if (bis && valid) {   // the first chunk whose inclusive prefix exceeds x
          int lo2 = 0, hi2 = nch;
          while (lo2 < hi2) {
            const int mid = (lo2 + hi2) >> 1;
            if (wrow[mid] > x) hi2 = mid;
            else lo2 = mid + 1;
          }
          if (lo2 < nch) {
            c = lo2;
            xc = x - (lo2 ? wrow[lo2 - 1] : 0ll);
          } else {   // past the range's total: the rounding gap
            c = lastnz;
            xc = LLONG_MAX;
          }
          pending = false;
        }
        while (!bis && __any_sync(FULL, pending)) {
          if (!win) load_window();
          const long long wend = __shfl_sync(FULL, incl_l, 31);
          const bool here = pending && x < wend;
          if (__any_sync(FULL, here)) {
            // the last lane (chunk) whose exclusive prefix is <= x, by halving
            const long long ex_l = incl_l - m_l;
            int Lc = 0;
#pragma unroll
            for (int sh = 4; sh >= 0; --sh) {
              const int t = Lc + (1 << sh);
              const long long ex_t = __shfl_sync(FULL, ex_l, t & 31);
              if (t < 32 && ex_t <= x) Lc = t;
            }
            const long long ex_c = __shfl_sync(FULL, ex_l, Lc);
            if (here) {
              c = wc0 + Lc;
              xc = x - ex_c;
              pending = false;
            }
          }
          if (__any_sync(FULL, pending)) {
            if (wc0 + 32 >= nch) {   // past the range's total: the rounding gap
              if (pending) {
                c = lastnz;
                xc = LLONG_MAX;
                pending = false;
              }
            } else {
              wcarry = wend;
              wc0 += 32;
              win = false;
            }
          }
        }
        SANTA_STAMP(11);
        int key = -1;
        if (valid) {
          if (c < 0) {
            key = p.c_lo * BK;   // no mass in the range at all (never expected)
          } else {
            // the first key of the chunk whose inclusive key-mass prefix
            // exceeds x - pref[c]; past the chunk's key total, its last
            // nonzero key
            const int64_t kc = (int64_t)(p.c_lo + c) * BK;
            const int64_t kr0 = (int64_t)p.c_lo * BK;   // the range's first key
            const float* sc = L.st ? L.st + wl * L.capk + (int)((bh * a.nk_max + kr0) & 3) + (int)(kc - kr0)
                                   : a.stash + bh * a.nk_max + kc;
            float s[BK];
            if (((reinterpret_cast<uintptr_t>(sc) & 15) == 0) && kc + BK <= p.nk) {   // four 16-byte loads
#pragma unroll
              for (int q4 = 0; q4 < BK / 4; ++q4) {
                const float4 v = reinterpret_cast<const float4*>(sc)[q4];
                s[4 * q4] = v.x;
                s[4 * q4 + 1] = v.y;
                s[4 * q4 + 2] = v.z;
                s[4 * q4 + 3] = v.w;
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < BK; ++kk) s[kk] = kc + kk < p.nk ? sc[kk] : -INFINITY;
            }
            long long F = 0;
            int found = -1, lastk = 0;
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
              const long long w = mass_fixed(fast_exp2(fmaf(s[kk], LOG2E, -ref)));
              F += w;
              lastk = w > 0 ? kk : lastk;
              found = (found < 0 && F > xc) ? kk : found;
            }
            key = (int)(kc + (found >= 0 ? found : lastk));
          }
          if (a.sample_idx) a.sample_idx[bh * a.S_max + jj] = key;
        }
        SANTA_STAMP(12);
        // ---- the distinct keys (keys are non-decreasing along the lanes)
        //      with their counts, gathered four at a time
        const int kprev = __shfl_up_sync(FULL, key, 1);
        const bool start = valid && (lane == 0 || kprev != key);
        if (start) {   // every distinct row of this pass requested at once, into L2
          const char* row = reinterpret_cast<const char*>(Vb - lane * CPL + (int64_t)key * a.Hkv * D);
#pragma unroll
          for (int o = 0; o < D * 2; o += 128) prefetch_l2(row + o);
        }
        unsigned starts = __ballot_sync(FULL, start);
        const int nval = __popc(__ballot_sync(FULL, valid));
        const unsigned later = starts & ~((2u << lane) - 1u);
        const float cnt = (float)((later ? __ffs(later) - 1 : nval) - lane);   // meaningful at run starts
        while (starts) {   // warp-uniform
          int src[4];
          uint2 raw[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            src[u] = starts ? __ffs(starts) - 1 : -1;
            starts &= starts ? starts - 1 : 0u;
            const int kk = __shfl_sync(FULL, key, src[u] < 0 ? 0 : src[u]);
            raw[u] = make_uint2(0u, 0u);
            if (src[u] >= 0) {
              const T* row = Vb + (int64_t)kk * a.Hkv * D;
              if constexpr (CPL == 4) raw[u] = *reinterpret_cast<const uint2*>(row);
              else raw[u].x = *reinterpret_cast<const uint32_t*>(row);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float c = __shfl_sync(FULL, cnt, src[u] < 0 ? 0 : src[u]);
            f2x pr2[4];
            Pairs<T>::get(make_uint4(raw[u].x, raw[u].y, 0u, 0u), pr2);
            const float2 p0 = unpack2(pr2[0]), p1 = unpack2(pr2[1]);
            const float vf[4] = {p0.x, p0.y, p1.x, p1.y};
#pragma unroll
            for (int k = 0; k < CPL; ++k) acc[k] = src[u] >= 0 ? fmaf(c, vf[k], acc[k]) : acc[k];
          }
        }
        SANTA_STAMP(13);
        }
      // ---- the head's sums, times 1/S_b, into out
      const float inv_S = 1.0f / (float)S_b;
      float* o = a.out + bh * D + lane * CPL;
      if constexpr (CPL == 4) {
        const float4 v4 = make_float4(acc[0] * inv_S, acc[1] * inv_S, acc[2] * inv_S, acc[3] * inv_S);
        if (!shared) *reinterpret_cast<float4*>(o) = v4;
        else if (__any_sync(FULL, acc[0] != 0.f || acc[1] != 0.f || acc[2] != 0.f || acc[3] != 0.f)) red_add_v4(o, v4);
      } else {
        const float2 v2 = make_float2(acc[0] * inv_S, acc[1] * inv_S);
        if (!shared) *reinterpret_cast<float2*>(o) = v2;
        else if (__any_sync(FULL, acc[0] != 0.f || acc[1] != 0.f)) red_add_v2(o, v2);
      }
      SANTA_STAMP(14);
    }
    if (!shared) group_sync(bar_id, nthr);   // the region is free for the next piece
  };

  // ---- work items, in order: preparation of the shared pieces (their
  //      groups), the pieces inside the range (all warps), the grid wait, the
  //      rest of the shared pieces.  One call site each.
  const int gi = n_shared == 2 ? warp / (FW / 2) : 0;             // this warp's group for the shared pieces
  const int sh_slot = n_shared == 2 ? gi : (first_shared ? 0 : 1);
  const int sh_bar = gi == 0 ? BAR_G0 : BAR_G1;
  const int sh_w0 = n_shared == 2 ? gi * (FW / 2) : 0, sh_nw = n_shared == 2 ? FW / 2 : FW;
  unsigned char* const sh_reg = regions + gi * REG;
  const int sh_bytes = n_shared == 2 ? REG : 2 * REG;
  Piece psh;
  SegLayout Lsh;
  if (n_shared > 0) {
    psh = s_psh[sh_slot];
    Lsh = seg_layout(sh_reg, sh_bytes, psh.c_hi - psh.c_lo);
  }
  Cur pc = cA;
  int stage = n_shared > 0 ? 0 : 1;
  for (;;) {
    Piece p;
    bool shared = false, do_prep = false, do_finish = false;
    int slot = 0, gid = 2, bar_id = BAR_INT, w0 = 0, nw = FW, reg_bytes = REG;
    unsigned char* reg = regions + 2 * REG;
    if (stage == 0) {            // preparation of this warp's shared piece
      stage = 1;
      p = psh;
      shared = true;
      do_prep = true;
      slot = sh_slot;
      gid = gi;
      bar_id = sh_bar;
      w0 = sh_w0;
      nw = sh_nw;
      reg = sh_reg;
      reg_bytes = sh_bytes;
    } else if (stage == 1) {     // next piece wholly inside the range
      bool found = false;
      while (has_interior && pc.b < a.B && pc.pb_lo < hi) {
        const bool inside = pc.pb_lo >= lo && pc.pb_lo + pc.nblk <= hi;
        if (inside) p = piece_at(pc);
        pc.kblk = pc.nblk;
        cur_norm(pc, a);
        if (inside) {
          found = true;
          break;
        }
      }
      if (!found) {
        SANTA_STAMP(7);
        stage = 2;
        write_tile_stats();
        if (n_shared == 0) break;
        cp_async_wait_all();   // the shared pieces' staged scores and prefixes, visible to all
        __syncthreads();
        // only the shared pieces' head warps go on (warps w0 .. w0 + G - 1 of
        // each group; warp 0 among them, whose thread 0 waits for the grid)
        const int nhead = n_shared * G;
        if (warp - sh_w0 >= G) break;
        if (tid == 0) {
          const unsigned long long t0 = global_ns();
          while (ld_acquire(arrivals) < (unsigned)P) {
            if (global_ns() - t0 > GRID_WAIT_NS) {
              flag_error(a.err, ERR_TIMEOUT);
              break;
            }
          }
        }
        group_sync(BAR_FIN, nhead * 32);
        SANTA_STAMP(8);
        continue;
      }
      do_prep = do_finish = true;
    } else if (stage == 2) {     // the rest of this warp's shared piece
      stage = 3;
      p = psh;
      shared = true;
      do_finish = true;
      gid = gi;
      bar_id = sh_bar;
      w0 = sh_w0;
      nw = sh_nw;
      reg = sh_reg;
      reg_bytes = sh_bytes;
    } else {
      break;
    }
    const SegLayout L = shared ? Lsh : seg_layout(reg, reg_bytes, p.c_hi - p.c_lo);
    if (do_prep) prep_piece(p, L, shared, slot, gid, bar_id, w0, nw);
    if (do_finish) finish_piece(p, L, shared, gid, bar_id, w0, nw);
    if (stage == 1 && shared) SANTA_STAMP(6);
  }
  cp_async_wait_all();   // no copy outlives the CTA
  // the first CTA, once every CTA has arrived (each read the generation
  // before arriving), advances the generation for the next launch
  if (cta == 0) {
    if (n_shared == 0) arrivals_wait(arrivals, (unsigned)P, a.err);
    if (tid == 0) st_release(bar_gen, s_gen + 1u);
  }
  SANTA_STAMP(15);
}

// Launch of one instantiation: one CTA per SM (at most MAX_CTAS), cooperative.
template <typename T, int D, int V, bool TMA_K>
inline cudaError_t launch_fused_inst(const LaunchArgs& a, const CUtensorMap& tm, unsigned* bar_count,
                                     unsigned* bar_gen, int grid) {
  using Gm = FGeom<D>;
  auto kern = fused_decode_kernel<T, D, V, TMA_K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Gm::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(FT);
  cfg.dynamicSmemBytes = Gm::SMEM;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm, a, bar_count, bar_gen);
}

// Every instantiation for one cache dtype: head_dim x variant x K access.
template <typename T>
inline cudaError_t launch_fused_dtype(const LaunchArgs& a, const CUtensorMap& tm, bool tma, unsigned* bar_count,
                                      unsigned* bar_gen, int grid) {
#define SANTA_FUSED_CASE(DD, VV)                                                                 \
  if (a.D == DD && a.variant == VV)                                                              \
    return tma ? launch_fused_inst<T, DD, VV, true>(a, tm, bar_count, bar_gen, grid)           \
               : launch_fused_inst<T, DD, VV, false>(a, tm, bar_count, bar_gen, grid);
  SANTA_FUSED_CASE(128, VAR_SYS)
  SANTA_FUSED_CASE(128, VAR_STRAT)
  SANTA_FUSED_CASE(128, VAR_IID)
  SANTA_FUSED_CASE(64, VAR_SYS)
  SANTA_FUSED_CASE(64, VAR_STRAT)
  SANTA_FUSED_CASE(64, VAR_IID)
#undef SANTA_FUSED_CASE
  return cudaErrorInvalidValue;
}

}  // namespace santa
