// santa_fused.cu -- one decode step of SANTA / S2ANTA in a single persistent
// launch for 16-bit caches (sm_103a).
//
// "Stochastic Sparse Attention for Memory-Bound Inference":
//   scores and per-chunk statistics   Sec. 2 Eq. (1); App. O, Alg. 3
//   cross-chunk combine               App. O, Alg. 4
//   thresholds                        Sec. 2.1 (i.i.d. Eq. 4; stratified; systematic)
//   inverse CDF, left-closed          App. A.4
//   GQA-deduplicated gather-and-add   Eq. (4), Fig. 1; App. O, Alg. 5
//
// Grid: one 512-thread CTA per SM, launched cooperatively (all CTAs
// resident).  Phase A streams the CTA's contiguous range of score-pass units
// (santa_stream.cuh) and reduces, for every head it touched, the range's
// (max, exp-sum) aggregate.  One grid-wide barrier.  Phase B: every CTA reads
// the aggregates of the CTAs that cover the same (sequence, KV-head group),
// which gives the head max m*, the total mass Z and the mass prefix P_i of its
// own key range exactly (fixed-point int64, computed identically in every
// CTA), places the thresholds that fall in [P_i, P_i + T_i), resolves them in
// its own chunks and 32-key windows, and gathers and adds the drawn V rows.
//
// Phase B is latency-bound (little data, dependent steps), so it is laid out
// for parallelism: one round of asynchronous copies stages everything a CTA
// reads (aggregates, its chunk statistics, its scores) in shared memory; the
// per-head work runs in groups of 8-32 lanes, all heads of a KV-head group at
// once; windows go to warps in contiguous blocks.
//
// Difference from the pages' kernels: Alg. 4 rounds per-tile budgets by
// largest remainder and samples each tile on its own; here the S thresholds of
// a head are placed globally and each CTA resolves the ones in its own mass
// interval, which reproduces the global i.i.d. / stratified / systematic
// estimators.  Thresholds are exact integers, theta_j = floor(t_j * Z), with
// t_j a rational of 24-bit uniforms, so no FP64 arithmetic runs per draw.
#include <algorithm>

#include "santa_common.cuh"
#include "santa_launch.h"
#include "santa_stream.cuh"
#include "santa_window.cuh"

namespace santa {

constexpr int POOL_CAP = 4096;   // thresholds of one piece kept in shared memory
constexpr int RCAP = 64;         // drawn rows listed per warp before a gather

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
// rcp = ceil(2^64 / div), precomputed once per sequence.
__device__ __forceinline__ ThetaCtx theta_ctx(long long Z, unsigned div, unsigned long long rcp) {
  ThetaCtx c;
  c.Z = Z;
  c.div = div;
  c.rcp = rcp;
  if (div > 1) {
    // Z < 2^62: mulhi(Z, rcp) is floor(Z / div) or one more
    unsigned long long q = __umul64hi((unsigned long long)Z, rcp);
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

// Lane groups of `lph` lanes (8, 16 or 32) inside a warp.
__device__ __forceinline__ float grp_max(float v, int lph) {
  for (int o = lph >> 1; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o, lph));
  return v;
}
__device__ __forceinline__ float grp_sum(float v, int lph) {
  for (int o = lph >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o, lph);
  return v;
}
__device__ __forceinline__ long long grp_scan(long long v, int r, int lph) {   // inclusive
  for (int o = 1; o < lph; o <<= 1) {
    const long long n = __shfl_up_sync(FULL, v, o, lph);
    if (r >= o) v += n;
  }
  return v;
}

// Mass w (relative to the head max, in [0, 2^22)) in units of 2^-40, rounded
// toward zero: one exact scaling and one conversion (the same value as
// mass_fixed for these w).
__device__ __forceinline__ long long fixed40(float w) { return __float2ll_rz(w * 1099511627776.0f); }

struct Draws {
  int variant, S, h, b;
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
    if (variant == VAR_IID) return theta_of(tc, sorted[j]);
    const uint32_t k = variant == VAR_SYS ? ksys : key_at(j);
    return theta_of(tc, ((unsigned long long)j << 24) | k);
  }
  // #{j < S : theta_j < X} (thresholds are non-decreasing in j), the same in
  // every lane of the head's group.  `rounds` (warp-uniform) bounds the
  // group-parallel search over sorted keys so every lane of the warp takes
  // part in the same number of ballots.
  __device__ __forceinline__ int count_below(long long X, int r, int lph, int lane, int rounds) const {
    if (variant != VAR_IID) {
      if (X <= 0) return 0;
      if (X >= tc.Z) return S;
      // theta_j lies in [floor(j Z / S), floor((j + 1) Z / S)): start next to X S / Z
      long long e = (long long)(__fdividef((float)X, (float)tc.Z) * (float)S);
      e = e < 0 ? 0 : (e > S ? S : e);
      while (e > 0 && theta((int)e - 1) >= X) --e;
      while (e < S && theta((int)e) < X) ++e;
      return (int)e;
    }
    // sorted keys: lph-way search, one probe per lane and round
    int lo = 0, hi = S;
    if (X <= 0) hi = 0;
    else if (X >= tc.Z) lo = S;
    const int gbase = lane - r;
    const unsigned gbits = lph == 32 ? 0xffffffffu : ((1u << lph) - 1u);
    for (int it = 0; it < rounds; ++it) {
      const int step = (hi - lo + lph - 1) / lph;
      const int p = lo + r * step;
      const bool below = lo < hi && p < hi && theta(p) < X;
      const int t = __popc((__ballot_sync(FULL, below) >> gbase) & gbits);
      if (lo < hi) {
        if (t == 0) {
          hi = lo;
        } else {
          const int plast = lo + (t - 1) * step;
          lo = plast + 1;
          hi = min(hi, plast + step);
        }
      }
    }
    return lo;
  }
};

// ---------------------------------------------------------------------------
// Grid-wide barrier (all CTAs are resident: cooperative launch).  A counter
// and a generation word in the workspace; the last CTA to arrive resets the
// counter and advances the generation.  Waits are bounded (WAIT_LIMIT_NS);
// on expiry ERR_TIMEOUT is flagged and the CTA proceeds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void grid_barrier(unsigned* count, unsigned* gen, int* err) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned g = ld_acquire(gen);
    __threadfence();
    const unsigned arrived = atomicAdd(count, 1u);
    if (arrived == gridDim.x - 1) {
      atomicExch(count, 0u);
      __threadfence();
      atomicAdd(gen, 1u);
    } else {
      const unsigned long long t0 = global_ns();
      while (ld_acquire(gen) == g) {
        if (global_ns() - t0 > WAIT_LIMIT_NS) {
          flag_error(err, ERR_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
  }
  __syncthreads();
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// A maximal run of one CTA's units that belong to one (sequence, KV-head group).
struct Piece {
  int b, hg, kb0, nkb;
  int units_b;
  long long ubase;   // global index of unit (b, hg, kb = 0)
  int64_t row0, nk;
};

// Calls fn(piece) for every piece of this CTA's unit range, in order (every
// thread of the CTA walks the same pieces).
template <typename Fn>
__device__ __forceinline__ void for_each_piece(const LaunchArgs& a, int n_hg, int unit_rows, const int* start,
                                               long long u0, Fn fn) {
  UnitCursor c;
  c.kv_offsets = a.kv_offsets;
  c.nk_max = a.nk_max;
  c.B = a.B;
  c.n_hg = n_hg;
  c.unit_rows = unit_rows;
  c.b = start[0];
  c.hg = start[1];
  c.kb = start[2];
  int left = start[3];
  if (left <= 0) return;
  c.load_seq();
  long long u = u0;
  while (left > 0) {
    Piece p;
    p.b = c.b;
    p.hg = c.hg;
    p.kb0 = c.kb;
    p.nkb = min(left, c.units_b - c.kb);
    p.units_b = c.units_b;
    p.ubase = u - c.kb;
    p.row0 = c.row0;
    p.nk = c.nk;
    fn(p);
    left -= p.nkb;
    u += p.nkb;
    c.kb += p.nkb - 1;
    c.advance();
  }
}

// Sequence metadata: length within [1, nk_max] and budget within [1, S_max].
__device__ __forceinline__ int seq_error(const LaunchArgs& a, int b, int& S_b) {
  int err = 0;
  int64_t nk = a.nk_max, row0 = 0;
  if (a.kv_offsets) {
    row0 = a.kv_offsets[b];
    nk = a.kv_offsets[b + 1] - row0;
  }
  if (nk < 1) err |= ERR_EMPTY;
  else if (nk > a.nk_max || row0 < 0) err |= ERR_NK_BOUND;
  S_b = a.S_per_seq ? a.S_per_seq[b] : a.S_max;
  if (S_b < 1 || S_b > a.S_max) err |= ERR_S_RANGE;
  return err;
}

// Per-head state of phase B (shared memory).
struct HeadInfo {
  int jlo, jhi;   // this CTA's threshold range [jlo, jhi)
  int off;        // offset of its thresholds in the shared pool, -1: in the global array
  float mstar;    // the head's max score
};

// Count-weighted gather-and-add of the listed rows keys[0..n) (key indices of
// one sequence and KV head) with counts cnt[r * GM + g] into acc (head g, the
// lane's output columns; partial sums spread over the row slots).
template <typename T, int D, int GM>
__device__ __forceinline__ void gather_list(float (&acc)[GM][Tile<T, D>::EPL], const int* keys, const int* cnt,
                                            int n, const T* __restrict__ Vbase, int Hkv, int G, int lane) {
  using TL = Tile<T, D>;
  const int slot = lane / TL::LPK;
  constexpr int UNR = 4;
  for (int r0 = 0; r0 < n; r0 += UNR * TL::KPI) {
    uint4 vv[UNR][TL::NVEC];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = r0 + u * TL::KPI + slot;
#pragma unroll
      for (int v = 0; v < TL::NVEC; ++v)
        vv[u][v] = r < n ? ld_stream(Vbase + (int64_t)keys[r] * Hkv * D + v * (16 / TL::ES)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = r0 + u * TL::KPI + slot;
      if (r0 + u * TL::KPI < n) {   // warp-uniform
        float vf[TL::EPL];
#pragma unroll
        for (int v = 0; v < TL::NVEC; ++v) Elem<T>::widen(vv[u][v], vf + v * (16 / TL::ES));
#pragma unroll
        for (int g = 0; g < GM; ++g) {
          if (g < G) {
            const float cg = r < n ? (float)cnt[r * GM + g] : 0.f;
#pragma unroll
            for (int e = 0; e < TL::EPL; ++e) acc[g][e] = fmaf(cg, vf[e], acc[g][e]);
          }
        }
      }
    }
  }
}

template <typename T, int D, int GM>
__global__ void __launch_bounds__(SB_THREADS, 1)
fused_decode_kernel(LaunchArgs a, unsigned* bar_count, unsigned* bar_gen) {
  using TL = Tile<T, D>;
  using Gm = StreamGeom<T, D>;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int start[4];
  __shared__ long long range[2];
  __shared__ int pool_used;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int G = a.H / a.Hkv, W = unit_heads(a.Hkv), n_hg = a.Hkv / W;
  const int unit_rows = SB_UNIT_ROWS_X_W / W;
  const int GW = G * W;                       // query heads of one KV-head group
  const int lph = GW > 32 ? 8 : (GW > 16 ? 16 : 32);   // lanes per head in the per-head steps
  const int P = gridDim.x, cta = blockIdx.x;
  const int cm1 = a.chunks_max + 1;
  const int C_of_unit = unit_rows / SUB;      // statistics chunks per unit
  const uint32_t k0 = (uint32_t)a.seed, k1 = (uint32_t)(a.seed >> 32);
  // head group of this thread in the per-head steps (groups fill whole warps)
  const int grp = tid / lph, r = tid % lph;
  const bool warp_on = (warp * 32) / lph < GW;
  const bool hv = grp < GW;
  const int hl = hv ? grp : GW - 1;

  // ======================= phase A =======================
  if (warp == 0) unit_range_start(a.kv_offsets, a.nk_max, a.B, n_hg, unit_rows, cta, P, start, range);
  {
    const int64_t n4 = (int64_t)a.B * a.H * D / 4;   // out is accumulated into in phase B
    for (int64_t i = (int64_t)cta * SB_THREADS + tid; i < n4; i += (int64_t)P * SB_THREADS)
      reinterpret_cast<float4*>(a.out)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // sequence metadata (sequence b checked by CTA b mod P): flags, reciprocal
  // of the budget, unused sample slots
  for (int b = cta; b < a.B; b += P) {
    int S_b;
    const int e = seq_error(a, b, S_b);
    if (tid == 0) {
      if (e) flag_error(a.err, e);
      else a.rcp_S[b] = S_b > 1 ? ~0ull / (unsigned)S_b + 1ull : 0ull;
    }
    if (a.sample_idx) {
      const int from = e ? 0 : S_b;
      for (int i = tid; i < a.H * (a.S_max - from); i += SB_THREADS) {
        const int h = i / (a.S_max - from), j = from + i % (a.S_max - from);
        a.sample_idx[((int64_t)b * a.H + h) * a.S_max + j] = -1;
      }
    }
  }
  __syncthreads();
  {
    StreamArgs sa;
    sa.q = a.q;
    sa.K = a.K;
    sa.kv_offsets = a.kv_offsets;
    sa.nk_max = a.nk_max;
    sa.B = a.B;
    sa.H = a.H;
    sa.Hkv = a.Hkv;
    sa.W = W;
    sa.scale = a.scale;
    sa.stash = a.stash;
    sa.sub_max = a.tile_max;
    sa.sub_sum = a.tile_sum;
    sa.subs_max = a.chunks_max;
    stream_scores<T, D>(sa, smem_addr(smem), start);
  }
  __syncthreads();   // statistics of the whole range written; the ring is free

  // i.i.d.: sorted 24-bit uniform keys of the heads bh = cta (mod P)
  if (a.variant == VAR_IID) {
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
    for (int64_t bh = cta; bh < (int64_t)a.B * a.H; bh += P) {
      const int b = (int)(bh / a.H), h = (int)(bh % a.H);
      int S_b;
      if (seq_error(a, b, S_b)) continue;
      int S2 = 1;
      while (S2 < S_b) S2 <<= 1;
      for (int i = tid; i < S2; i += SB_THREADS) {
        uint32_t k = 0xffffffffu;
        if (i < S_b) {
          const uint4 w = philox4x32_10(make_uint4((uint32_t)(i >> 2), (uint32_t)h, (uint32_t)b, a.step), k0, k1);
          const uint32_t x = (i & 3) == 0 ? w.x : (i & 3) == 1 ? w.y : (i & 3) == 2 ? w.z : w.w;
          k = x >> 8;
        }
        keys[i] = k;
      }
      __syncthreads();
      for (int kk = 2; kk <= S2; kk <<= 1) {
        for (int jj = kk >> 1; jj > 0; jj >>= 1) {
          for (int i = tid; i < S2; i += SB_THREADS) {
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
      for (int i = tid; i < S_b; i += SB_THREADS) a.ukeys[bh * a.S_max + i] = keys[i];
      __syncthreads();
    }
  }

  // aggregates (max, sum exp(s - max)) of every head over this CTA's keys
  for_each_piece(a, n_hg, unit_rows, start, range[1], [&](const Piece& p) {
    if (!warp_on) return;
    const int c_lo = p.kb0 * C_of_unit;
    const int c_hi = (int)min((int64_t)(p.kb0 + p.nkb) * C_of_unit, (p.nk + SUB - 1) / SUB);
    const int64_t bh = (int64_t)p.b * a.H + (int64_t)p.hg * GW + hl;
    const float* mx = a.tile_max + bh * a.chunks_max;
    const float* sm = a.tile_sum + bh * a.chunks_max;
    float m = -INFINITY;
    for (int c = c_lo + r; c < c_hi; c += lph) m = fmaxf(m, mx[c]);
    m = grp_max(m, lph);
    float l = 0.f;
    for (int c = c_lo + r; c < c_hi; c += lph) l += expf(mx[c] - m) * sm[c];
    l = grp_sum(l, lph);
    if (hv && r == 0) {
      a.agg_m[bh * MAX_CTAS + cta] = m;
      a.agg_l[bh * MAX_CTAS + cta] = l;
    }
  });

  grid_barrier(bar_count, bar_gen, a.err);

  // ======================= phase B =======================
  const long long n_units = range[0];
  auto nonempty = [&](int i) {   // CTA i owns at least one unit
    return n_units >= P || n_units * i / P < n_units * (i + 1) / P;
  };
  // fixed shared-memory regions (inside the ring, free by now)
  float* obuf = reinterpret_cast<float*>(smem);                                   // [GW][D] this CTA's sums
  int* cnt_all = reinterpret_cast<int*>(obuf + GM * 8 * D);                      // [warps][RCAP][GM]
  int* rows_all = cnt_all + SB_WARPS * RCAP * GM;                                 // [warps][RCAP]
  HeadInfo* hinfo = reinterpret_cast<HeadInfo*>(rows_all + SB_WARPS * RCAP);      // [GW]
  long long* pool = reinterpret_cast<long long*>(hinfo + GM * 8);                // [POOL_CAP]
  unsigned char* var0 = reinterpret_cast<unsigned char*>(pool + POOL_CAP);       // per-piece staging
  int* cnt_s = cnt_all + warp * RCAP * GM;
  int* rows = rows_all + warp * RCAP;
  const size_t var_cap = Gm::SMEM - (size_t)(var0 - smem);

  for_each_piece(a, n_hg, unit_rows, start, range[1], [&](const Piece& p) {
    int S_b;
    if (seq_error(a, p.b, S_b)) return;   // uniform over the CTA
    const long long ufirst = p.ubase, ulast = p.ubase + p.units_b - 1;   // units of (b, hg)
    const int i_first = (int)(((ufirst + 1) * P - 1) / n_units), i_last = (int)(((ulast + 1) * P - 1) / n_units);
    const int ncov = i_last - i_first + 1;
    const int c_lo = p.kb0 * C_of_unit;
    const int c_hi = (int)min((int64_t)(p.kb0 + p.nkb) * C_of_unit, (p.nk + SUB - 1) / SUB);
    const int nch = c_hi - c_lo;
    const int64_t key_lo = (int64_t)c_lo * SUB, key_hi = min((int64_t)c_hi * SUB, p.nk);
    const int nkeys = (int)(key_hi - key_lo);
    const int64_t bh0 = (int64_t)p.b * a.H + (int64_t)p.hg * GW;   // first head of the group

    // ---- staging plan: aggregates always; chunk statistics + chunk tables
    //      and scores when they fit.  Rows are copied in 16-byte pieces from
    //      the 16-byte boundary at or below their first element (reading up
    //      to 12 bytes either side of a row stays inside the workspace).
    size_t off = 0;
    auto take = [&](size_t bytes) {
      const size_t o = (off + 15) & ~(size_t)15;
      off = o + bytes;
      return var0 + o;
    };
    auto row_cap = [](int len) { return (len + 7) & ~3; };   // floats per staged row
    const int cap_agg = row_cap(ncov), cap_ch = row_cap(nch), cap_st = row_cap(nkeys);
    float* s_am = reinterpret_cast<float*>(take((size_t)GW * cap_agg * 4));
    float* s_al = reinterpret_cast<float*>(take((size_t)GW * cap_agg * 4));
    const size_t off_after_agg = off;
    float* s_mx = reinterpret_cast<float*>(take((size_t)GW * cap_ch * 4));
    float* s_sm = reinterpret_cast<float*>(take((size_t)GW * cap_ch * 4));
    long long* s_pref = reinterpret_cast<long long*>(take((size_t)GW * nch * 8));
    int* s_js = reinterpret_cast<int*>(take((size_t)GW * nch * 4));
    const bool ch_smem = off <= var_cap;
    if (!ch_smem) off = off_after_agg;
    float* s_st = reinterpret_cast<float*>(take((size_t)GW * cap_st * 4));
    const bool st_smem = off <= var_cap;
    // row h of length len starting at global float index g0 -> s_row + h * cap (+ (g0 & 3))
    auto stage_row = [&](float* s_row, const float* base, int64_t g0, int len) {
      const int64_t a0 = g0 & ~(int64_t)3;
      const int n16 = (int)((g0 + len - a0 + 3) >> 2);
      for (int j = lane; j < n16; j += 32) cp_async16(smem_addr(s_row + 4 * j), base + a0 + 4 * j);
    };
    for (int h = warp; h < GW; h += SB_WARPS) {
      const int64_t bh = bh0 + h;
      stage_row(s_am + h * cap_agg, a.agg_m, bh * MAX_CTAS + i_first, ncov);
      stage_row(s_al + h * cap_agg, a.agg_l, bh * MAX_CTAS + i_first, ncov);
      if (ch_smem) {
        stage_row(s_mx + h * cap_ch, a.tile_max, bh * a.chunks_max + c_lo, nch);
        stage_row(s_sm + h * cap_ch, a.tile_sum, bh * a.chunks_max + c_lo, nch);
      }
      if (st_smem) stage_row(s_st + h * cap_st, a.stash, bh * a.nk_max + key_lo, nkeys);
    }
    cp_async_commit();
    for (int i = tid; i < GW * D; i += SB_THREADS) obuf[i] = 0.f;
    if (tid == 0) pool_used = 0;
    const unsigned long long rcp = a.rcp_S[p.b];
    cp_async_wait_all();
    __syncthreads();

    // ---- per head (a group of lph lanes each, all heads at once): m*, Z,
    //      this CTA's interval, its thresholds, and the prefix / first
    //      threshold of each of its chunks
    if (warp_on) {
      const int h = p.hg * GW + hl;
      const int64_t bh = bh0 + hl;
      const int oa = (int)((bh * MAX_CTAS + i_first) & 3);
      const float* am = s_am + hl * cap_agg + oa;
      const float* al = s_al + hl * cap_agg + oa;
      float m = -INFINITY;
      for (int i = r; i < ncov; i += lph)
        if (nonempty(i_first + i)) m = fmaxf(m, am[i]);
      const float mstar = grp_max(m, lph);
      const int kseg = (ncov + lph - 1) / lph;   // lane r sums the CTAs [r kseg, (r + 1) kseg)
      long long seg = 0, before = 0, Tc = 0;
      for (int t = 0; t < kseg; ++t) {
        const int i = r * kseg + t;
        if (i < ncov && nonempty(i_first + i)) {
          const long long Ti = fixed40(fast_exp(am[i] - mstar) * al[i]);
          seg += Ti;
          if (i_first + i < cta) before += Ti;
          if (i_first + i == cta) Tc = Ti;
        }
      }
      const long long incl = grp_scan(seg, r, lph);
      const int own = min((cta - i_first) / kseg, lph - 1);
      const long long P_own = __shfl_sync(FULL, incl - seg + before, own, lph);
      const long long T_own = __shfl_sync(FULL, Tc, own, lph);
      const long long Z = __shfl_sync(FULL, incl, lph - 1, lph);
      Draws dr;
      dr.variant = a.variant;
      dr.S = S_b;
      dr.h = h;
      dr.b = p.b;
      dr.step = a.step;
      dr.k0 = k0;
      dr.k1 = k1;
      dr.ksys = a.variant == VAR_SYS
                    ? philox4x32_10(make_uint4(0u, (uint32_t)h, (uint32_t)p.b, a.step), k0, k1).x >> 8
                    : 0u;
      dr.sorted = a.ukeys + bh * a.S_max;
      dr.tc = a.variant == VAR_IID ? theta_ctx(Z, 1u, 0ull) : theta_ctx(Z, (unsigned)S_b, rcp);
      int rounds = 1;
      if (a.variant == VAR_IID)
        for (int span = S_b; span > 1; span = (span + lph - 1) / lph) ++rounds;
      const int jlo = dr.count_below(P_own, r, lph, lane, rounds);
      const int jhi = dr.count_below(P_own + T_own, r, lph, lane, rounds);
      const int nt = jhi - jlo;
      int toff = -1;
      if (r == 0 && hv && nt > 0) {
        const int o = atomicAdd(&pool_used, nt);
        toff = (o + nt <= POOL_CAP) ? o : -1;
      }
      toff = __shfl_sync(FULL, toff, 0, lph);
      long long* thp = toff >= 0 ? pool + toff : a.thresh + bh * a.S_max + jlo;
      if (hv)
        for (int j = jlo + r; j < jhi; j += lph) thp[j - jlo] = dr.theta(j);
      if (r == 0 && hv) {
        hinfo[hl].jlo = jlo;
        hinfo[hl].jhi = jhi;
        hinfo[hl].off = toff;
        hinfo[hl].mstar = mstar;
        a.head_max[bh] = mstar;
      }
      __syncwarp();
      // chunk masses of this CTA's chunks, exclusive prefix from P_own
      const int oc = (int)((bh * a.chunks_max + c_lo) & 3);
      const float* mx = ch_smem ? s_mx + hl * cap_ch + oc : a.tile_max + bh * a.chunks_max + c_lo;
      const float* sm = ch_smem ? s_sm + hl * cap_ch + oc : a.tile_sum + bh * a.chunks_max + c_lo;
      long long* pr = ch_smem ? s_pref + hl * nch : a.prefix + bh * cm1 + c_lo;
      int* jsr = ch_smem ? s_js + hl * nch : a.jstart + bh * cm1 + c_lo;
      long long run = P_own;
      for (int c0 = 0; c0 < nch; c0 += lph) {
        const int c = c0 + r;
        const long long Wc = c < nch ? fixed40(fast_exp(mx[c] - mstar) * sm[c]) : 0;
        const long long ci = grp_scan(Wc, r, lph);
        const long long pref = run + ci - Wc;
        if (c < nch && hv) {
          int lo = 0, hi = nt;   // first threshold >= pref among [jlo, jhi)
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (thp[mid] < pref) lo = mid + 1;
            else hi = mid;
          }
          pr[c] = pref;
          jsr[c] = jlo + lo;
        }
        run += __shfl_sync(FULL, ci, lph - 1, lph);
      }
    }
    __syncthreads();   // per-head intervals, chunk tables and thresholds visible

    // ---- per (KV head, 32-key window) with thresholds: draws, the union of
    //      the drawn rows listed per warp, count-weighted gather into obuf.
    //      Warp w takes a contiguous block of the (KV head, window) list, so
    //      it gathers and flushes when the KV head changes or its list is full.
    const int w_lo = c_lo / 2, nwin = (nch + 1) / 2;
    const int ntask = W * nwin;
    const int t_begin = (int)((long long)ntask * warp / SB_WARPS);
    const int t_end = (int)((long long)ntask * (warp + 1) / SB_WARPS);
    int nrows = 0, cur_wk = -1;
    auto flush = [&]() {   // warp-uniform
      if (nrows > 0) {
        const int sub = lane % TL::LPK;
        float acc[GM][TL::EPL];
#pragma unroll
        for (int g = 0; g < GM; ++g)
#pragma unroll
          for (int e = 0; e < TL::EPL; ++e) acc[g][e] = 0.f;
        const T* Vb = reinterpret_cast<const T*>(a.V) + (p.row0 * a.Hkv + (int64_t)(p.hg * W + cur_wk)) * (int64_t)D +
                      sub * TL::EPL;
        gather_list<T, D, GM>(acc, rows, cnt_s, nrows, Vb, a.Hkv, G, lane);
        reduce_slots<T, D, GM>(acc);
        if (lane < TL::LPK) {
#pragma unroll
          for (int g = 0; g < GM; ++g)
            if (g < G)
#pragma unroll
              for (int e = 0; e < TL::EPL; ++e) atomicAdd(&obuf[(cur_wk * G + g) * D + sub * TL::EPL + e], acc[g][e]);
        }
      }
      nrows = 0;
      __syncwarp();
    };
    for (int task = t_begin; task < t_end; ++task) {
      const int wk = task / nwin, wi = task % nwin;
      if (wk != cur_wk) {
        flush();
        cur_wk = wk;
      }
      const int w = w_lo + wi;
      int js[GM], nt[GM];
      long long pb[GM];
      bool any = false;
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        js[g] = 0;
        nt[g] = 0;
        pb[g] = 0;
        if (g < G) {
          const int h2 = wk * G + g;
          const int64_t bh = bh0 + h2;
          const int* jsr = ch_smem ? s_js + h2 * nch : a.jstart + bh * cm1 + c_lo;
          js[g] = jsr[2 * wi];
          const int je = (2 * wi + 2 < nch) ? jsr[2 * wi + 2] : hinfo[h2].jhi;
          nt[g] = je - js[g];
          if (nt[g] > 0) pb[g] = ch_smem ? s_pref[h2 * nch + 2 * wi] : a.prefix[bh * cm1 + c_lo + 2 * wi];
          any |= nt[g] > 0;
        }
      }
      if (!any) continue;   // warp-uniform
      const int64_t key = (int64_t)w * WIN + lane;
      // all heads of the window at once: key masses, exact prefixes, thresholds
      long long F[GM], th0[GM];
      float mst[GM];
      int lastnz[GM], cnt[GM];
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        const int h2 = g < G ? wk * G + g : 0;
        const int64_t bh = bh0 + h2;
        const HeadInfo hi = hinfo[h2];
        mst[g] = hi.mstar;
        float sv = -INFINITY;
        if (nt[g] > 0 && key < p.nk)
          sv = st_smem ? s_st[h2 * cap_st + (int)((bh * a.nk_max + key_lo) & 3) + (int)(key - key_lo)]
                       : a.stash[bh * a.nk_max + key];
        F[g] = fixed40(fast_exp(sv - mst[g]));   // e^{-inf} = 0 past the sequence end
        th0[g] = LLONG_MAX;
        if (lane < nt[g])
          th0[g] = hi.off >= 0 ? pool[hi.off + js[g] - hi.jlo + lane] : a.thresh[bh * a.S_max + js[g] + lane];
        cnt[g] = 0;
      }
#pragma unroll
      for (int g = 0; g < GM; ++g) lastnz[g] = __ballot_sync(FULL, F[g] > 0);
#pragma unroll
      for (int g = 0; g < GM; ++g) lastnz[g] = lastnz[g] ? 31 - __clz(lastnz[g]) : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int g = 0; g < GM; ++g) {
          const long long n = __shfl_up_sync(FULL, F[g], o);
          if (lane >= o) F[g] += n;
        }
      }
      int ntmax = 0;
#pragma unroll
      for (int g = 0; g < GM; ++g) ntmax = max(ntmax, nt[g]);
      if (ntmax <= 8) {
        // one ballot per threshold: the key is the first lane with F > x (the
        // last nonzero key for x beyond the window's total)
        for (int t = 0; t < ntmax; ++t) {
#pragma unroll
          for (int g = 0; g < GM; ++g) {
            if (t < nt[g]) {   // warp-uniform
              const long long x = __shfl_sync(FULL, th0[g], t) - pb[g];
              const unsigned above = __ballot_sync(FULL, F[g] > x);
              const int k = above ? __ffs(above) - 1 : lastnz[g];
              if (lane == k) {
                ++cnt[g];
                if (a.sample_idx) a.sample_idx[(bh0 + wk * G + g) * a.S_max + js[g] + t] = (int)key;
              }
            }
          }
        }
      } else {
#pragma unroll
        for (int g = 0; g < GM; ++g) {
          if (nt[g] > 0) {   // warp-uniform
            const int h2 = wk * G + g;
            const int64_t bh = bh0 + h2;
            const HeadInfo hi = hinfo[h2];
            const long long* th = hi.off >= 0 ? pool + hi.off + (js[g] - hi.jlo) : a.thresh + bh * a.S_max + js[g];
            float sv = -INFINITY;
            if (key < p.nk)
              sv = st_smem ? s_st[h2 * cap_st + (int)((bh * a.nk_max + key_lo) & 3) + (int)(key - key_lo)]
                           : a.stash[bh * a.nk_max + key];
            cnt[g] = window_draws(sv, hi.mstar, th0[g], nt[g], pb[g], th,
                                  a.sample_idx ? a.sample_idx + bh * a.S_max + js[g] : nullptr, (int)key, lane);
          }
        }
      }
      bool mine = false;
#pragma unroll
      for (int g = 0; g < GM; ++g) mine |= cnt[g] > 0;
      const unsigned drawn = __ballot_sync(FULL, mine);
      if (nrows + __popc(drawn) > RCAP) flush();   // warp-uniform
      if (mine) {
        const int rr = nrows + __popc(drawn & ((1u << lane) - 1u));
        rows[rr] = (int)key;
#pragma unroll
        for (int g = 0; g < GM; ++g) cnt_s[rr * GM + g] = cnt[g];
      }
      nrows += __popc(drawn);
      __syncwarp();
    }
    flush();
    __syncthreads();
    // this CTA's sums, times 1/S_b, into out (vectorised fp32 reductions;
    // the order of the additions across CTAs is not fixed)
    const float inv_S = 1.0f / (float)S_b;
    float* outp = a.out + bh0 * D;
    for (int i4 = tid; i4 < GW * D / 4; i4 += SB_THREADS) {
      const float4 v = reinterpret_cast<const float4*>(obuf)[i4];
      if (v.x != 0.f || v.y != 0.f || v.z != 0.f || v.w != 0.f)
        red_add_v4(outp + 4 * i4, make_float4(v.x * inv_S, v.y * inv_S, v.z * inv_S, v.w * inv_S));
    }
    __syncthreads();
  });
}

// ---------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------
template <typename T, int D, int GM>
static cudaError_t launch_fused_g(const LaunchArgs& a, unsigned* bar_count, unsigned* bar_gen) {
  using Gm = StreamGeom<T, D>;
  static_assert((size_t)GM * 8 * D * 4 + (size_t)SB_WARPS * RCAP * (GM + 1) * 4 + (size_t)GM * 8 * sizeof(HeadInfo) +
                        (size_t)POOL_CAP * 8 + (size_t)64 * MAX_CTAS * 8 + 64 <=
                    Gm::SMEM,
                "phase B fixed regions and the aggregates fit the ring");
  const int W = unit_heads(a.Hkv);
  const int unit_rows = SB_UNIT_ROWS_X_W / W;
  const long long units = (long long)a.B * ((a.nk_max + unit_rows - 1) / unit_rows) * (a.Hkv / W);
  const int grid = (int)std::min<long long>(std::min<long long>(units, (long long)a.num_sms), (long long)MAX_CTAS);
  cudaError_t e = cudaFuncSetAttribute(fused_decode_kernel<T, D, GM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Gm::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(SB_THREADS);
  cfg.dynamicSmemBytes = Gm::SMEM;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_decode_kernel<T, D, GM>, a, bar_count, bar_gen);
}

template <typename T, int D>
static cudaError_t launch_fused_t(const LaunchArgs& a, unsigned* bar_count, unsigned* bar_gen) {
  return (a.H / a.Hkv <= 4) ? launch_fused_g<T, D, 4>(a, bar_count, bar_gen)
                            : launch_fused_g<T, D, 8>(a, bar_count, bar_gen);
}

cudaError_t launch_fused(const LaunchArgs& a, unsigned* bar_count, unsigned* bar_gen) {
  switch (a.dtype * 2 + (a.D == 128)) {
    case 0: return launch_fused_t<bf16_t, 64>(a, bar_count, bar_gen);
    case 1: return launch_fused_t<bf16_t, 128>(a, bar_count, bar_gen);
    case 2: return launch_fused_t<fp16_t, 64>(a, bar_count, bar_gen);
    case 3: return launch_fused_t<fp16_t, 128>(a, bar_count, bar_gen);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace santa
