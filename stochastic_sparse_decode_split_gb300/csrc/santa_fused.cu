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
// Arrival half of the barrier (thread 0 acts; call after __syncthreads):
// returns the generation seen before arriving, for grid_wait.
__device__ __forceinline__ unsigned grid_arrive(unsigned* count, unsigned* gen) {
  unsigned g = 0;
  if (threadIdx.x == 0) {
    g = ld_acquire(gen);
    __threadfence();
    const unsigned arrived = atomicAdd(count, 1u);
    if (arrived == gridDim.x - 1) {
      atomicExch(count, 0u);
      __threadfence();
      atomicAdd(gen, 1u);
    }
  }
  return g;
}
// Waiting half: thread 0 spins until the generation moves past g (bounded),
// then the CTA proceeds together.
__device__ __forceinline__ void grid_wait(const unsigned* gen, unsigned g, int* err) {
  if (threadIdx.x == 0) {
    const unsigned long long t0 = global_ns();
    while (ld_acquire(gen) == g) {
      if (global_ns() - t0 > WAIT_LIMIT_NS) {
        flag_error(err, ERR_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  __syncthreads();
}
__device__ __forceinline__ void grid_barrier(unsigned* count, unsigned* gen, int* err) {
  __syncthreads();
  const unsigned g = grid_arrive(count, gen);
  grid_wait(gen, g, err);
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

// Geometry of head bh (global index b * H + h) for the owner step: its
// sequence's validity and budget, the covering CTAs [i_first, i_last] of its
// (sequence, KV-head group), the budget reciprocal and the systematic uniform.
// Warp-uniform (the ragged unit count is a warp reduction).
struct HeadGeom {
  int b, h, S_b, i_first, i_last;
  unsigned long long rcp;   // ceil(2^64 / S_b)
  uint32_t ksys;            // systematic: the head's uniform key
  bool ok;
};
__device__ __forceinline__ HeadGeom head_geom(const LaunchArgs& a, long long bh, int unit_rows, int n_hg, int GW, int P,
                                           long long n_units, uint32_t k0, uint32_t k1) {
  const int lane = threadIdx.x % 32;
  HeadGeom q;
  q.b = (int)(bh / a.H);
  q.h = (int)(bh % a.H);
  q.ok = seq_error(a, q.b, q.S_b) == 0;
  int64_t r0_, nk_;
  const int units_b = UnitCursor::seq_units(a.kv_offsets, a.nk_max, unit_rows, q.b, r0_, nk_);
  long long base = (long long)q.b * units_b;
  if (a.kv_offsets) {
    base = 0;
    for (int b0 = 0; b0 < q.b; b0 += 32) {
      int64_t r1, n1;
      long long u = (b0 + lane < q.b) ? UnitCursor::seq_units(a.kv_offsets, a.nk_max, unit_rows, b0 + lane, r1, n1) : 0;
      for (int o = 16; o > 0; o >>= 1) u += __shfl_xor_sync(FULL, u, o);
      base += u;
    }
  }
  const long long U = base * n_hg + (long long)(q.h / GW) * units_b;   // unit (b, hg, kb = 0)
  q.i_first = (int)(((U + 1) * P - 1) / n_units);
  q.i_last = (int)(((U + units_b) * P - 1) / n_units);
  q.ok = q.ok && units_b > 0;
  q.rcp = (q.ok && q.S_b > 1) ? ~0ull / (unsigned)q.S_b + 1ull : 0ull;
  q.ksys = a.variant == VAR_SYS ? philox4x32_10(make_uint4(0u, (uint32_t)q.h, (uint32_t)q.b, a.step), k0, k1).x >> 8
                                : 0u;
  return q;
}

// Per-head state of phase B (shared memory).
struct HeadInfo {
  long long pown;   // mass prefix of this CTA's key range
  int jlo, jhi;     // this CTA's threshold range [jlo, jhi)
  int off;          // offset of its thresholds in the shared pool, -1: in the global array
  float mstar;      // the head's max score
};

template <typename T, int D, int GM>
__global__ void __launch_bounds__(SB_THREADS, 1)
fused_decode_kernel(LaunchArgs a, unsigned* bar_count, unsigned* bar_gen) {
  using TL = Tile<T, D>;
  using Gm = StreamGeom<T, D>;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int start[4];
  __shared__ long long range[2];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int G = a.H / a.Hkv, W = unit_heads(a.Hkv), n_hg = a.Hkv / W;
  const int unit_rows = SB_UNIT_ROWS_X_W / W;
  const int GW = G * W;                       // query heads of one KV-head group
  const int lph = GW > 32 ? 8 : (GW > 16 ? 16 : 32);   // lanes per head in the per-head steps
  const int P = gridDim.x, cta = blockIdx.x;
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
  __shared__ float run_m[SB_WARPS * 8], run_l[SB_WARPS * 8];   // per-warp running statistics
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
    stream_scores<T, D>(sa, smem_addr(smem), start, run_m, run_l);
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

  // aggregates (max, sum exp(s - max)) of every head over this CTA's keys:
  // from the warps' running statistics when the range is one (sequence,
  // KV-head group), else from the range's chunk statistics
  bool one_piece = false;
  if (start[3] > 0) {
    int64_t r0_, nk_;
    const int ub = UnitCursor::seq_units(a.kv_offsets, a.nk_max, unit_rows, start[0], r0_, nk_);
    one_piece = start[2] + start[3] <= ub;
  }
  if (one_piece) {
    if (tid < GW) {
      const int wl = tid / G, g = tid % G;   // KV head within the group, head within its query group
      float m = -INFINITY;
      for (int w = 0; w < SB_WARPS; ++w)
        if (((w >> 1) % W) == wl) m = fmaxf(m, run_m[w * 8 + g]);
      float l = 0.f;
      for (int w = 0; w < SB_WARPS; ++w)
        if (((w >> 1) % W) == wl && run_m[w * 8 + g] > -INFINITY) l += run_l[w * 8 + g] * expf(run_m[w * 8 + g] - m);
      const int64_t bh = (int64_t)start[0] * a.H + (int64_t)start[1] * GW + tid;
      a.agg_m[bh * MAX_CTAS + cta] = m;
      a.agg_l[bh * MAX_CTAS + cta] = l;
    }
  } else
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

  // ---------------------------------------------------------------------------
  // shared-memory plan of phase B (inside the ring, free by now)
  // ---------------------------------------------------------------------------
  const long long n_units = range[0];
  HeadInfo* hinfo = reinterpret_cast<HeadInfo*>(smem);                           // [GW]
  long long* pool = reinterpret_cast<long long*>(hinfo + GM * 8);                // [POOL_CAP]
  unsigned char* var0 = reinterpret_cast<unsigned char*>(pool + POOL_CAP);       // per-segment staging
  const size_t var_cap = Gm::SMEM - (size_t)(var0 - smem);
  __shared__ int pool_used, n_items;
  __shared__ float red_f[SB_WARPS];
  __shared__ long long red_ll[SB_WARPS];
  // A piece's key range is processed in segments of SEG statistics chunks, so
  // that a segment's chunk statistics, scores, chunk tables, item list and
  // (KV head, key) count table all fit in shared memory.
  const int SEG = [&] {
    const size_t per_chunk = (size_t)GW * (8 + 16 + 4 * SUB) + (size_t)W * SUB * GM * 4;
    const size_t fixed = (size_t)GW * (2 * 7 * 4 + 7 * 4) + 8 * 16;   // row caps and alignment of 7 buffers
    const int n = (int)((var_cap - fixed) / per_chunk);
    return max(2, n & ~1);
  }();
  struct Seg {
    int c_lo, nch, nkeys, cap_ch, cap_st;   // first statistics chunk (in the sequence), chunks, keys
    int64_t key_lo;
    float *mx, *sm, *st;
    long long* pref;
    int *js, *items, *table;
  };
  // segment k of piece p: chunks [c_lo + k SEG, ...) of the piece's range
  auto seg_of = [&](const Piece& p, int k) {
    Seg g;
    const int pc_lo = p.kb0 * C_of_unit;
    const int pc_hi = (int)min((int64_t)(p.kb0 + p.nkb) * C_of_unit, (p.nk + SUB - 1) / SUB);
    g.c_lo = pc_lo + k * SEG;
    g.nch = max(0, min(SEG, pc_hi - g.c_lo));
    g.key_lo = (int64_t)g.c_lo * SUB;
    g.nkeys = (int)max((int64_t)0, min((int64_t)(g.c_lo + g.nch) * SUB, p.nk) - g.key_lo);
    g.cap_ch = (g.nch + 7) & ~3;   // floats per staged row (16-byte pieces from the boundary below)
    g.cap_st = (g.nkeys + 7) & ~3;
    size_t off = 0;
    auto take = [&](size_t bytes) {
      const size_t o = (off + 15) & ~(size_t)15;
      off = o + bytes;
      return var0 + o;
    };
    g.mx = reinterpret_cast<float*>(take((size_t)GW * g.cap_ch * 4));
    g.sm = reinterpret_cast<float*>(take((size_t)GW * g.cap_ch * 4));
    g.pref = reinterpret_cast<long long*>(take((size_t)GW * g.nch * 8));
    g.js = reinterpret_cast<int*>(take((size_t)GW * g.nch * 4));
    g.items = reinterpret_cast<int*>(take((size_t)GW * g.nch * 4));
    g.st = reinterpret_cast<float*>(take((size_t)GW * g.cap_st * 4));
    g.table = reinterpret_cast<int*>(take((size_t)W * g.nkeys * GM * 4));
    return g;
  };
  auto seg_count = [&](const Piece& p) {
    const int pc_lo = p.kb0 * C_of_unit;
    const int pc_hi = (int)min((int64_t)(p.kb0 + p.nkb) * C_of_unit, (p.nk + SUB - 1) / SUB);
    return (pc_hi - pc_lo + SEG - 1) / SEG;
  };
  // rows are copied in 16-byte pieces from the 16-byte boundary at or below
  // their first element (reading up to 12 bytes either side of a row stays
  // inside the workspace); row h lands at s_row + h * cap + (g0 & 3)
  auto stage_row = [&](float* s_row, const float* base, int64_t g0, int len) {
    const int64_t a0 = g0 & ~(int64_t)3;
    const int n16 = (int)((g0 + len - a0 + 3) >> 2);
    for (int j = lane; j < n16; j += 32) cp_async16(smem_addr(s_row + 4 * j), base + a0 + 4 * j);
  };
  // copies of a segment's statistics and scores (one commit group), count table cleared
  auto stage = [&](const Piece& p, const Seg& g) {
    const int64_t bh0 = (int64_t)p.b * a.H + (int64_t)p.hg * GW;
    for (int h = warp; h < GW; h += SB_WARPS) {
      const int64_t bh = bh0 + h;
      stage_row(g.mx + h * g.cap_ch, a.tile_max, bh * a.chunks_max + g.c_lo, g.nch);
      stage_row(g.sm + h * g.cap_ch, a.tile_sum, bh * a.chunks_max + g.c_lo, g.nch);
      stage_row(g.st + h * g.cap_st, a.stash, bh * a.nk_max + g.key_lo, g.nkeys);
    }
    cp_async_commit();
    for (int i = tid; i < W * g.nkeys * GM; i += SB_THREADS) g.table[i] = 0;
  };

  auto nonempty = [&](int i) {   // CTA i owns at least one unit
    return n_units >= P || n_units * i / P < n_units * (i + 1) / P;
  };
  auto geom = [&](long long bh) {   // the same in every lane of a warp
    return head_geom(a, bh, unit_rows, n_hg, GW, P, n_units, k0, k1);
  };
  auto make_draws = [&](const HeadGeom& q, long long bh, long long Z) {
    Draws dr;
    dr.variant = a.variant;
    dr.S = q.S_b;
    dr.h = q.h;
    dr.b = q.b;
    dr.step = a.step;
    dr.k0 = k0;
    dr.k1 = k1;
    dr.ksys = q.ksys;
    dr.sorted = a.ukeys + bh * a.S_max;
    dr.tc = a.variant == VAR_IID ? theta_ctx(Z, 1u, 0ull) : theta_ctx(Z, (unsigned)q.S_b, q.rcp);
    return dr;
  };
  // boundary i of a head: prefix, mass and the first threshold of the range
  // (counts of the i.i.d. sorted thresholds are taken in the CTA that owns the
  // range); the range ends where the next one starts
  // first barrier; while waiting, this CTA stages its first piece's chunk
  // statistics and scores (its own data, already written)
  __syncthreads();
  const unsigned gen1 = grid_arrive(bar_count, bar_gen);
  bool prestaged = false;
  __shared__ int pre_S0;
  __shared__ bool pre_bad0;
  if (start[3] > 0) {
    UnitCursor c0;
    c0.kv_offsets = a.kv_offsets;
    c0.nk_max = a.nk_max;
    c0.B = a.B;
    c0.n_hg = n_hg;
    c0.unit_rows = unit_rows;
    c0.b = start[0];
    c0.hg = start[1];
    c0.kb = start[2];
    c0.load_seq();
    Piece p0;
    p0.b = c0.b;
    p0.hg = c0.hg;
    p0.kb0 = c0.kb;
    p0.nkb = min(start[3], c0.units_b - c0.kb);
    p0.nk = c0.nk;
    stage(p0, seg_of(p0, 0));
    prestaged = true;
    if (tid == 0) pre_bad0 = seq_error(a, p0.b, pre_S0) != 0;
  }
  // ... and the geometry of the heads it will own in the next step (metadata
  // loads, budget reciprocal, systematic uniform), one warp per head
  constexpr int PRE_MAX = SB_WARPS;
  __shared__ HeadGeom pre_geom[PRE_MAX];
  {
    const long long bh = cta + (long long)warp * P;
    if (bh < (long long)a.B * a.H) {
      const HeadGeom q = geom(bh);
      if (lane == 0) pre_geom[warp] = q;
    }
  }
  grid_wait(bar_gen, gen1, a.err);   // its __syncthreads also publishes pre_geom
  // the k-th head owned by this CTA
  auto owned_geom = [&](long long bh) {
    const long long k = (bh - cta) / P;
    return k < PRE_MAX ? pre_geom[k] : geom(bh);
  };

  // ======================= phase B0: per-head globals =======================
  // From the aggregates of the CTAs covering a head's (sequence, KV-head
  // group): the head max m*, the total mass Z, and for each covering CTA i its
  // mass prefix P_i, mass T_i and threshold range [count(P_i), count(P_i + T_i)).
  // Heads covered by more than 32 CTAs take a whole CTA (one covering CTA per
  // thread); the others a warp (one per lane).
  auto write_bnd = [&](const Draws& dr, long long bh, int i, long long Pi, long long Ti) {
    const int64_t o = bh * MAX_CTAS + i;
    a.bnd_P[o] = Pi;
    a.bnd_T[o] = Ti;
    const int jlo = a.variant == VAR_IID ? -1 : dr.count_below(Pi, 0, 32, lane, 0);
    a.bnd_jlo[o] = jlo;
    return jlo;
  };
  __shared__ int s_jlo[MAX_CTAS + 1];
  // (1) wide heads: one CTA each
  for (long long bh = cta; bh < (long long)a.B * a.H; bh += P) {
    const HeadGeom q = owned_geom(bh);
    const int ncov = q.i_last - q.i_first + 1;
    const int i = q.i_first + tid;
    // loaded before the validity test so that these loads overlap the metadata loads
    const bool ok = tid < ncov && i < MAX_CTAS && nonempty(i);
    const float mi = ok ? a.agg_m[bh * MAX_CTAS + i] : -INFINITY;
    const float li = ok ? a.agg_l[bh * MAX_CTAS + i] : 0.f;
    if (!q.ok || ncov <= 32) continue;   // uniform over the CTA
    float m = warp_max(mi);
    if (lane == 0) red_f[warp] = m;
    __syncthreads();
    m = red_f[0];
#pragma unroll
    for (int w = 1; w < SB_WARPS; ++w) m = fmaxf(m, red_f[w]);
    const long long Ti = ok ? fixed40(fast_exp(mi - m) * li) : 0;
    const long long incl = warp_inclusive_scan(Ti, lane);
    if (lane == 31) red_ll[warp] = incl;
    __syncthreads();
    long long before = 0, Z = 0;
#pragma unroll
    for (int w = 0; w < SB_WARPS; ++w) {
      before += w < warp ? red_ll[w] : 0;
      Z += red_ll[w];
    }
    const Draws dr = make_draws(q, bh, Z);
    if (tid < ncov) s_jlo[tid] = write_bnd(dr, bh, i, before + incl - Ti, Ti);
    if (tid == 0) {
      a.head_max[bh] = m;
      a.head_Z[bh] = Z;
    }
    __syncthreads();
    if (tid < ncov)
      a.bnd_jhi[bh * MAX_CTAS + i] = a.variant == VAR_IID ? -1 : (tid + 1 < ncov ? s_jlo[tid + 1] : q.S_b);
    __syncthreads();
  }
  // (2) narrow heads: one warp each
  for (long long bh = (long long)warp * P + cta; bh < (long long)a.B * a.H; bh += (long long)SB_WARPS * P) {
    const HeadGeom q = owned_geom(bh);
    const int ncov = q.i_last - q.i_first + 1;
    const int i = q.i_first + lane;
    const bool ok = lane < ncov && i < MAX_CTAS && nonempty(i);
    const float mi = ok ? a.agg_m[bh * MAX_CTAS + i] : -INFINITY;
    const float li = ok ? a.agg_l[bh * MAX_CTAS + i] : 0.f;
    if (!q.ok || ncov > 32) continue;   // warp-uniform
    const float m = warp_max(mi);
    const long long Ti = ok ? fixed40(fast_exp(mi - m) * li) : 0;
    const long long incl = warp_inclusive_scan(Ti, lane);
    const long long Z = __shfl_sync(FULL, incl, 31);
    const Draws dr = make_draws(q, bh, Z);
    const int jlo = lane < ncov ? write_bnd(dr, bh, i, incl - Ti, Ti) : 0;
    const int jnext = __shfl_down_sync(FULL, jlo, 1);
    if (lane < ncov)
      a.bnd_jhi[bh * MAX_CTAS + i] = a.variant == VAR_IID ? -1 : (lane + 1 < ncov ? jnext : q.S_b);
    if (lane == 0) {
      a.head_max[bh] = m;
      a.head_Z[bh] = Z;
    }
  }

  grid_barrier(bar_count, bar_gen, a.err);

  // ======================= phase B1: this CTA's draws =======================
  __shared__ long long carry_s[GM * 8];   // per head: mass prefix at the current segment's start
  __shared__ int jend_s[GM * 8];          // per head: end of the current segment's thresholds
  int piece_no = 0;
  for_each_piece(a, n_hg, unit_rows, start, range[1], [&](const Piece& p) {
    int S_b;
    bool bad;
    if (piece_no == 0 && prestaged) {   // checked while waiting at the first barrier
      bad = pre_bad0;
      S_b = pre_S0;
    } else {
      bad = seq_error(a, p.b, S_b) != 0;
    }
    const bool first = piece_no == 0 && prestaged;
    ++piece_no;
    if (bad) return;   // uniform over the CTA
    const int64_t bh0 = (int64_t)p.b * a.H + (int64_t)p.hg * GW;   // first head of the group
    if (tid == 0) pool_used = 0;
    __syncthreads();

    // ---- per head (groups of lph lanes, all heads at once): this CTA's
    //      interval and its thresholds
    if (warp_on) {
      const int h = p.hg * GW + hl;
      const int64_t bh = bh0 + hl;
      const int64_t o = bh * MAX_CTAS + cta;
      const long long P_own = a.bnd_P[o], T_own = a.bnd_T[o], Z = a.head_Z[bh];
      int jlo = a.bnd_jlo[o], jhi = a.bnd_jhi[o];
      const float mstar = a.head_max[bh];
      HeadGeom q;
      q.b = p.b;
      q.h = h;
      q.S_b = S_b;
      q.rcp = a.rcp_S[p.b];
      q.ksys = a.variant == VAR_SYS ? philox4x32_10(make_uint4(0u, (uint32_t)h, (uint32_t)p.b, a.step), k0, k1).x >> 8
                                    : 0u;
      const Draws dr = make_draws(q, bh, Z);
      if (a.variant == VAR_IID) {
        int rounds = 1;
        for (int span = S_b; span > 1; span = (span + lph - 1) / lph) ++rounds;
        jlo = dr.count_below(P_own, r, lph, lane, rounds);
        jhi = dr.count_below(P_own + T_own, r, lph, lane, rounds);
      }
      const int nt = jhi - jlo;
      int toff = -1;
      if (r == 0 && hv && nt > 0) {
        const int qq = atomicAdd(&pool_used, nt);
        toff = (qq + nt <= POOL_CAP) ? qq : -1;
      }
      toff = __shfl_sync(FULL, toff, 0, lph);
      long long* thp = toff >= 0 ? pool + toff : a.thresh + bh * a.S_max + jlo;
      if (hv)
        for (int j = jlo + r; j < jhi; j += lph) thp[j - jlo] = dr.theta(j);
      if (r == 0 && hv) {
        hinfo[hl].pown = P_own;
        hinfo[hl].jlo = jlo;
        hinfo[hl].jhi = jhi;
        hinfo[hl].off = toff;
        hinfo[hl].mstar = mstar;
        carry_s[hl] = P_own;
      }
    }
    const int nseg = seg_count(p);
    for (int sg_i = 0; sg_i < nseg; ++sg_i) {
      const Seg g = seg_of(p, sg_i);
      if (!(first && sg_i == 0)) stage(p, g);   // the first piece's first segment was staged at the first barrier
      if (tid == 0) n_items = 0;
      cp_async_wait_all();
      __syncthreads();   // staged data, cleared table, thresholds and head state visible

      // ---- per head: the segment's chunk prefixes (from the running carry),
      //      first threshold of each chunk, and the chunks that hold thresholds
      if (warp_on) {
        const int64_t bh = bh0 + hl;
        const HeadInfo hi = hinfo[hl];
        const int nt = hi.jhi - hi.jlo;
        const long long* thp = hi.off >= 0 ? pool + hi.off : a.thresh + bh * a.S_max + hi.jlo;
        const int oc = (int)((bh * a.chunks_max + g.c_lo) & 3);
        const float* mx = g.mx + hl * g.cap_ch + oc;
        const float* sm = g.sm + hl * g.cap_ch + oc;
        long long* pr = g.pref + hl * g.nch;
        int* jsr = g.js + hl * g.nch;
        auto first_at_or_above = [&](long long v) {   // index of the first threshold >= v among [jlo, jhi)
          int lo = 0, hi2 = nt;
          while (lo < hi2) {
            const int mid = (lo + hi2) >> 1;
            if (thp[mid] < v) lo = mid + 1;
            else hi2 = mid;
          }
          return hi.jlo + lo;
        };
        long long run = carry_s[hl];
        for (int c0 = 0; c0 < g.nch; c0 += lph) {
          const int c = c0 + r;
          const long long Wc = c < g.nch ? fixed40(fast_exp(mx[c] - hi.mstar) * sm[c]) : 0;
          const long long ci = grp_scan(Wc, r, lph);
          const long long pref = run + ci - Wc;
          if (c < g.nch && hv) {
            pr[c] = pref;
            jsr[c] = first_at_or_above(pref);
          }
          run += __shfl_sync(FULL, ci, lph - 1, lph);
        }
        // end of this segment's thresholds: the next segment's first, or the
        // range's end for the last segment (thresholds in the rounding gap
        // between the chunk sums and the range mass go to its last chunk)
        const int jend = sg_i + 1 < nseg ? first_at_or_above(run) : hi.jhi;
        __syncwarp();
        if (hv) {
          for (int c = r; c < g.nch; c += lph) {
            const int je = c + 1 < g.nch ? jsr[c + 1] : jend;
            if (je > jsr[c]) g.items[atomicAdd(&n_items, 1)] = hl * 65536 + c;
          }
          if (r == 0) {
            jend_s[hl] = jend;
            carry_s[hl] = run;
          }
        }
      }
      __syncthreads();   // chunk tables and items visible

      // ---- per (head, 16-key chunk) holding thresholds, one half-warp each:
      //      exact key-mass prefix over the chunk, one ballot per threshold
      //      (the key is the first with F > x; a threshold at or beyond the
      //      chunk's key total goes to its last nonzero key); counts into the
      //      (KV head, key) table, the union of the group's draws.
      const int h16 = lane >> 4, l16 = lane & 15, hb = h16 * 16;
      const int nwork = n_items;
      for (int q0 = warp * 2; q0 < nwork; q0 += SB_WARPS * 2) {
        const int q = q0 + h16;
        const bool qv = q < nwork;
        const int qh = qv ? g.items[q] >> 16 : 0, qc = qv ? g.items[q] & 0xffff : 0;
        const int* jsr = g.js + qh * g.nch;
        const HeadInfo hi = hinfo[qh];
        const int j0 = qv ? jsr[qc] : 0;
        const int j1 = qv ? (qc + 1 < g.nch ? jsr[qc + 1] : jend_s[qh]) : 0;
        const int nthr = j1 - j0;
        const int tmax = max(nthr, __shfl_xor_sync(FULL, nthr, 16));
        const int64_t bh = bh0 + qh;
        const int64_t key = (int64_t)(g.c_lo + qc) * SUB + l16;
        float sv = -INFINITY;
        if (nthr > 0 && key < p.nk)
          sv = g.st[qh * g.cap_st + (int)((bh * a.nk_max + g.key_lo) & 3) + (int)(key - g.key_lo)];
        long long F = fixed40(fast_exp(sv - hi.mstar));   // e^{-inf} = 0 past the sequence end
        const unsigned nzb = (__ballot_sync(FULL, F > 0) >> hb) & 0xffffu;
        const int lastnz = nzb ? 31 - __clz(nzb) : 0;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
          const long long n = __shfl_up_sync(FULL, F, o, 16);
          if (l16 >= o) F += n;
        }
        const long long pref = nthr > 0 ? g.pref[qh * g.nch + qc] : 0;
        int cnt = 0;
        for (int t = 0; t < tmax; ++t) {
          const bool ok = t < nthr;
          long long x = 0;
          if (ok) x = (hi.off >= 0 ? pool[hi.off + (j0 - hi.jlo) + t] : a.thresh[bh * a.S_max + j0 + t]) - pref;
          const unsigned above = (__ballot_sync(FULL, ok && F > x) >> hb) & 0xffffu;
          const int k = above ? __ffs(above) - 1 : lastnz;
          if (ok && l16 == k) {
            ++cnt;
            if (a.sample_idx) a.sample_idx[bh * a.S_max + j0 + t] = (int)key;
          }
        }
        if (cnt > 0) {
          atomicAdd(&g.table[((qh / G) * g.nkeys + (int)(key - g.key_lo)) * GM + qh % G], cnt);
          // the gather reads this row once the table is complete: start it towards L2 now
          const T* vrow = reinterpret_cast<const T*>(a.V) + ((p.row0 + key) * a.Hkv + p.hg * W + qh / G) * (int64_t)D;
#pragma unroll
          for (int ln = 0; ln < (D * 2 + 127) / 128; ++ln)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(vrow + ln * 64));
        }
      }
      __syncthreads();   // the count table is complete

      // ---- gather by KV head: warp w takes KV head w % W and every
      //      (16 / W)-th 32-key block of the segment; each drawn V row is read
      //      once for all heads of its group, lane l owns output columns
      //      [l CPL, (l + 1) CPL) of every head, and the warp's sums, times
      //      1/S_b, go into out with vectorised fp32 reductions (their order
      //      across warps and CTAs is not fixed).
      {
        const int wk = warp % W, part = warp / W, nparts = SB_WARPS / W;
        constexpr int CPL = D / 32;   // output columns per lane
        float acc[GM][CPL];
#pragma unroll
        for (int gg = 0; gg < GM; ++gg)
#pragma unroll
          for (int c = 0; c < CPL; ++c) acc[gg][c] = 0.f;
        const int* tab = g.table + (size_t)wk * g.nkeys * GM;
        const T* Vk = reinterpret_cast<const T*>(a.V) + (p.row0 * a.Hkv + p.hg * W + wk) * (int64_t)D + lane * CPL;
        bool any_rows = false;
        int nmine = 0;
        int rk_l = -1;   // lane l holds the l-th listed row of this warp
        int rc_l[GM];
#pragma unroll
        for (int gg = 0; gg < GM; ++gg) rc_l[gg] = 0;
        auto gather_batch = [&](int n) {   // rows held by lanes 0..n-1, four loads in flight
          for (int r0 = 0; r0 < n; r0 += 4) {
            uint2 raw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int kr = __shfl_sync(FULL, rk_l, (r0 + u) & 31);
              raw[u] = make_uint2(0u, 0u);
              if (r0 + u < n) {
                const T* src = Vk + (g.key_lo + kr) * a.Hkv * D;
                if constexpr (CPL == 4) raw[u] = *reinterpret_cast<const uint2*>(src);
                else raw[u].x = *reinterpret_cast<const uint32_t*>(src);
              }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (r0 + u < n) {   // warp-uniform
                f2x pr[4];
                Pairs<T>::get(make_uint4(raw[u].x, raw[u].y, 0u, 0u), pr);
                const float2 p0 = unpack2(pr[0]), p1 = unpack2(pr[1]);
                const float vf[4] = {p0.x, p0.y, p1.x, p1.y};
#pragma unroll
                for (int gg = 0; gg < GM; ++gg) {
                  const float cw = (float)__shfl_sync(FULL, rc_l[gg], (r0 + u) & 31);
#pragma unroll
                  for (int c = 0; c < CPL; ++c) acc[gg][c] = fmaf(cw, vf[c], acc[gg][c]);
                }
              }
            }
          }
        };
        for (int k0b = part * 32; k0b < g.nkeys; k0b += 32 * nparts) {
          const int kr = k0b + lane;
          int cg[GM];
          bool drawn_here = false;
#pragma unroll
          for (int gg = 0; gg < GM; ++gg) {
            cg[gg] = (kr < g.nkeys && gg < G) ? tab[kr * GM + gg] : 0;
            drawn_here |= cg[gg] != 0;
          }
          const unsigned mine = __ballot_sync(FULL, drawn_here);
          const int add = __popc(mine);
          if (nmine + add > 32) {
            gather_batch(nmine);
            any_rows = any_rows || nmine > 0;
            nmine = 0;
          }
          for (int t = 0; t < add; ++t) {   // lane nmine + t receives the t-th row of this block
            const int src_lane = (int)__fns(mine, 0, t + 1);
            const int krow = __shfl_sync(FULL, kr, src_lane);
            int cgs[GM];
#pragma unroll
            for (int gg = 0; gg < GM; ++gg) cgs[gg] = __shfl_sync(FULL, cg[gg], src_lane);
            if (lane == nmine + t) {
              rk_l = krow;
#pragma unroll
              for (int gg = 0; gg < GM; ++gg) rc_l[gg] = cgs[gg];
            }
          }
          nmine += add;
        }
        if (nmine > 0) {
          gather_batch(nmine);
          any_rows = true;
        }
        if (any_rows) {   // warp-uniform
          const float inv_S = 1.0f / (float)S_b;
          float* outp = a.out + (bh0 + (int64_t)wk * G) * D + lane * CPL;
#pragma unroll
          for (int gg = 0; gg < GM; ++gg) {
            if (gg < G) {
              if constexpr (CPL == 4)
                red_add_v4(outp + (int64_t)gg * D,
                           make_float4(acc[gg][0] * inv_S, acc[gg][1] * inv_S, acc[gg][2] * inv_S, acc[gg][3] * inv_S));
              else
                red_add_v2(outp + (int64_t)gg * D, make_float2(acc[gg][0] * inv_S, acc[gg][1] * inv_S));
            }
          }
        }
      }
      __syncthreads();   // the segment's buffers are free for the next one
    }
  });
  cp_async_wait_all();   // no copy outlives the CTA (a staged piece that was skipped)
}

// ---------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------
template <typename T, int D, int GM>
static cudaError_t launch_fused_g(const LaunchArgs& a, unsigned* bar_count, unsigned* bar_gen) {
  using Gm = StreamGeom<T, D>;
  static_assert((size_t)GM * 8 * sizeof(HeadInfo) + (size_t)POOL_CAP * 8 +
                        (size_t)64 * (8 + 16 + 4 * SUB) * 2 + (size_t)8 * SUB * GM * 4 * 2 + 64 * 84 + 96 <=
                    Gm::SMEM,
                "phase B fixed regions and a two-chunk segment fit the ring");
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
