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
// aggregate (max, and the mass relative to a power of two).  One grid-wide
// barrier.  Phase B: every CTA reads the aggregates of the CTAs that cover the
// same (sequence, KV-head group), which gives the head's reference 2^E*, the
// total mass Z and the mass prefix P_i of its own key range exactly
// (fixed-point int64, the same integers in every CTA), places the thresholds
// that fall in [P_i, P_i + T_i), resolves them in its own chunks, and gathers
// and adds the drawn V rows.
//
// Phase B is latency-bound (little data, dependent steps), so it is laid out
// for parallelism and few waits: the first segment of chunk statistics and
// scores is staged in shared memory while the CTA waits at the barrier; the
// per-head work runs in groups of 8-32 lanes, all heads of a KV-head group at
// once; each (head, chunk) holding draws takes a half-warp; drawn (head, key)
// pairs go to a list, and warp w sums the V rows of its heads (w, w + 16, ...)
// in registers until the end of the piece.
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
#include "santa_seq.cuh"
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

// Mass w (relative to the head's reference, in [0, 2^22)) in units of 2^-40,
// rounded toward zero, by integer operations (mass_fixed).
__device__ __forceinline__ long long fixed40(float w) { return mass_fixed(w); }

// Aggregate of one head over one CTA's keys.  Masses are taken relative to a
// power of two so that every reader rescales them exactly by a shift:
//   m  max score over the keys
//   e  ceil(m log2(e)), an integer
//   F  sum_n 2^(s_n log2(e) - e) in units of 2^-40 (rounded toward zero)
// With E* the largest e over the CTAs of a head, CTA k's mass relative to
// 2^E* is F_k >> (E* - e_k): the same integer in every CTA that computes it.
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
    x.F = fixed40(l * fast_exp2(t - (float)x.e));
  }
  return x;
}

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
      // (24 leading bits of X and Z: 32-bit conversions, not the FP64-pipe int64 ones)
      const int sh = max(0, 40 - __clzll(tc.Z));
      int e = (int)(__fdividef((float)(uint32_t)(X >> sh), (float)(uint32_t)(tc.Z >> sh)) * (float)S);
      e = e < 0 ? 0 : (e > S ? S : e);
      while (e > 0 && theta(e - 1) >= X) --e;
      while (e < S && theta(e) < X) ++e;
      return e;
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
__device__ __forceinline__ void grid_wait(const unsigned* gen, unsigned g, int* err,
                                          unsigned long long limit_ns = WAIT_LIMIT_NS) {
  if (threadIdx.x == 0) {
    const unsigned long long t0 = global_ns();
    while (ld_acquire(gen) == g) {
      if (global_ns() - t0 > limit_ns) {
        flag_error(err, ERR_TIMEOUT);
        break;
      }
      __nanosleep(64);
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


// Per-head constants of the thresholds.
struct HeadGeom {
  int b, h, S_b;
  unsigned long long rcp;   // ceil(2^64 / S_b)
  uint32_t ksys;            // systematic: the head's uniform key
};

// Per-head state of phase B (shared memory).
struct HeadInfo {
  long long pown;   // mass prefix of this CTA's key range
  int jlo, jhi;     // this CTA's threshold range [jlo, jhi)
  int off;          // offset of its thresholds in the shared pool, -1: in the global array
  float ref;        // masses are 2^(s log2(e) - ref): ref = E*, the head's largest aggregate exponent
};

// i.i.d.: sorted 24-bit uniform keys of every head (out of line: the other
// variants never run it).  When the Tu units do not divide evenly over the P
// CTAs, the CTAs with one unit fewer (done streaming about a unit earlier)
// sort, head j going to the (j mod n)-th of them; else CTA bh mod P.  Up to
// 1024 keys a head are placed by rank (each thread counts the keys below its
// own: one barrier), more by a bitonic network in `keys` (shared memory).
static __device__ __noinline__ void sort_iid_keys(int B, int H, int S_max, uint32_t step, const int64_t* kv_offsets,
                                                 int64_t nk_max, const int32_t* S_per_seq, uint32_t* ukeys,
                                                 uint32_t* keys, long long Tu, int P, int cta, uint32_t k0,
                                                 uint32_t k1) {
  const int tid = threadIdx.x;
  const long long qu = Tu / P, rem = Tu % P;
  int srank = cta, nsort = P;
  if (rem != 0) {
    const long long mine = Tu * (cta + 1) / P - Tu * cta / P;
    const long long large_before = Tu * cta / P - (long long)cta * qu;
    nsort = (int)(P - rem);
    srank = mine == qu ? (int)(cta - large_before) : -1;
  }
  for (int64_t bh = srank; srank >= 0 && bh < (int64_t)B * H; bh += nsort) {
    const int b = (int)(bh / H), h = (int)(bh % H);
    int S_b;
    if (seq_error(kv_offsets, nk_max, S_per_seq, S_max, b, S_b)) continue;
    uint32_t* dst = ukeys + bh * S_max;
    int S2 = 1;
    while (S2 < S_b) S2 <<= 1;
    for (int i = tid; i < S2; i += SB_THREADS) {
      uint32_t k = 0xffffffffu;
      if (i < S_b) {
        const uint4 w = philox4x32_10(make_uint4((uint32_t)(i >> 2), (uint32_t)h, (uint32_t)b, step), k0, k1);
        const uint32_t x = (i & 3) == 0 ? w.x : (i & 3) == 1 ? w.y : (i & 3) == 2 ? w.z : w.w;
        k = x >> 8;
      }
      keys[i] = k;
    }
    __syncthreads();
    if (S_b <= 1024) {
      for (int i = tid; i < S_b; i += SB_THREADS) {
        const uint32_t ki = keys[i];
        int rank = 0;
        for (int u = 0; u < S_b; ++u) {
          const uint32_t ku = keys[u];
          rank += (ku < ki || (ku == ki && u < i)) ? 1 : 0;
        }
        dst[rank] = ki;
      }
    } else {
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
      for (int i = tid; i < S_b; i += SB_THREADS) dst[i] = keys[i];
    }
    __syncthreads();   // keys is rewritten for the next head
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
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int G = a.H / a.Hkv, W = a.W, n_hg = a.Hkv / W;
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
  if (a.variant == VAR_IID)
  sort_iid_keys(a.B, a.H, a.S_max, a.step, a.kv_offsets, a.nk_max, a.S_per_seq, a.ukeys,
                reinterpret_cast<uint32_t*>(smem), range[0], P, cta, k0, k1);
  // aggregates (max, sum exp(s - max)) of every head over this CTA's keys:
  // from the warps' running statistics when the range is one (sequence,
  // KV-head group), else from the range's chunk statistics
  bool one_piece = false;
  if (start[3] > 0) {
  int64_t r0_, nk_;
  const int ub = UnitCursor::seq_units(a.kv_offsets, a.nk_max, unit_rows, start[0], r0_, nk_);
  one_piece = start[2] + start[3] <= ub;
  }
  Agg* const agg = reinterpret_cast<Agg*>(a.agg);
  if (one_piece) {
  if (tid < GW) {
    // warps 2x and 2x + 1 stream KV head x mod W of the group
    const int wl = tid / G, g = tid % G;   // KV head within the group, head within its query group
    float m = -INFINITY;
    for (int x = wl; x < SB_WARPS / 2; x += W) m = fmaxf(m, fmaxf(run_m[2 * x * 8 + g], run_m[(2 * x + 1) * 8 + g]));
    float l = 0.f;
    for (int x = wl; x < SB_WARPS / 2; x += W)
      for (int w = 2 * x; w < 2 * x + 2; ++w)
        if (run_m[w * 8 + g] > -INFINITY) l += run_l[w * 8 + g] * expf(run_m[w * 8 + g] - m);
    const int64_t bh = (int64_t)start[0] * a.H + (int64_t)start[1] * GW + tid;
    agg[bh * MAX_CTAS + cta] = make_agg(m, l);
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
  if (hv && r == 0) agg[bh * MAX_CTAS + cta] = make_agg(m, l);
  });
  // ---------------------------------------------------------------------------
  // shared-memory plan of phase B (inside the ring, free by now)
  // ---------------------------------------------------------------------------
  const long long n_units = range[0];
  HeadInfo* hinfo = reinterpret_cast<HeadInfo*>(smem);                           // [GW]
  long long* pool = reinterpret_cast<long long*>(hinfo + GM * 8);                // [POOL_CAP]
  unsigned char* var0 = reinterpret_cast<unsigned char*>(pool + POOL_CAP);       // per-segment staging
  const size_t var_cap = Gm::SMEM - (size_t)(var0 - smem);
  __shared__ int pool_used, n_items, n_ent;
  constexpr int HPW = GM / 2;    // heads per warp in the gather: head h goes to warp h mod 16 (GW <= 8 GM)
  constexpr int CPL = D / 32;    // output columns per lane
  // A piece's key range is processed in segments of SEG statistics chunks, so
  // that a segment's chunk statistics, scores, chunk tables, item list and
  // list of drawn (head, key) pairs all fit in shared memory.
  const int SEG = [&] {
  const size_t per_chunk = (size_t)GW * (8 + 16 + 4 * SUB) + (size_t)GW * SUB * 4;
  const size_t fixed = (size_t)GW * (2 * 7 * 4 + 7 * 4) + 8 * 16;   // row caps and alignment of 7 buffers
  const int n = (int)((var_cap - fixed) / per_chunk);
  return min(512, max(2, n & ~1));   // keys of a segment fit the 13-bit key field of a list entry
  }();
  struct Seg {
  int c_lo, nch, nkeys, cap_ch, cap_st;   // first statistics chunk (in the sequence), chunks, keys
  int64_t key_lo;
  float *mx, *sm, *st;
  long long* pref;
  int *js, *items;
  uint32_t* ent;   // drawn (head, key) pairs: key << 19 | head << 13 | count
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
  g.ent = reinterpret_cast<uint32_t*>(take((size_t)GW * g.nkeys * 4));
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
  // copies of a segment's statistics and scores (one commit group)
  auto stage = [&](const Piece& p, const Seg& g) {
  const int64_t bh0 = (int64_t)p.b * a.H + (int64_t)p.hg * GW;
  for (int h = warp; h < GW; h += SB_WARPS) {
    const int64_t bh = bh0 + h;
    stage_row(g.mx + h * g.cap_ch, a.tile_max, bh * a.chunks_max + g.c_lo, g.nch);
    stage_row(g.sm + h * g.cap_ch, a.tile_sum, bh * a.chunks_max + g.c_lo, g.nch);
    stage_row(g.st + h * g.cap_st, a.stash, bh * a.nk_max + g.key_lo, g.nkeys);
  }
  cp_async_commit();
  };
  auto nonempty = [&](int i) {   // CTA i owns at least one unit
  return n_units >= P || n_units * i / P < n_units * (i + 1) / P;
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
  // first barrier; while waiting, this CTA stages its first piece's chunk
  // statistics and scores (its own data, already written) and sets up what
  // its first piece needs that does not depend on other CTAs
  __syncthreads();
  const unsigned gen1 = grid_arrive(bar_count, bar_gen);
  bool prestaged = false;
  __shared__ int pre_S0;
  __shared__ bool pre_bad0;
  __shared__ int cov_s[2];                    // the CTAs covering the piece's (sequence, KV-head group)
  __shared__ unsigned long long pre_rcp;     // first piece: ceil(2^64 / S_b)
  __shared__ uint32_t pre_ksys[GM * 8];      // first piece, systematic: each head's uniform key
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
  if (tid == 0) {
    int S0;
    pre_bad0 = seq_error(a, p0.b, S0) != 0;
    pre_S0 = S0;
    pre_rcp = (!pre_bad0 && S0 > 1) ? ~0ull / (unsigned)S0 + 1ull : 0ull;
    const long long ubase = range[1] - c0.kb;   // unit (b, hg, kb = 0)
    cov_s[0] = (int)(((ubase + 1) * P - 1) / range[0]);
    cov_s[1] = (int)(((ubase + c0.units_b) * P - 1) / range[0]);
  }
  if (a.variant == VAR_SYS && tid < GW)
    pre_ksys[tid] = philox4x32_10(make_uint4(0u, (uint32_t)(p0.hg * GW + tid), (uint32_t)p0.b, a.step), k0, k1).x >> 8;
  }
  grid_wait(bar_gen, gen1, a.err);
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
  if (tid == 0) {
    pool_used = 0;
    if (!first) {
      cov_s[0] = (int)(((p.ubase + 1) * P - 1) / n_units);
      cov_s[1] = (int)(((p.ubase + p.units_b) * P - 1) / n_units);
    }
  }
  __syncthreads();
  // ---- per head (groups of lph lanes, all heads at once): from the
  //      aggregates of the CTAs covering the piece's (sequence, KV-head
  //      group), the reference exponent E*, the head max m*, the total mass Z, this CTA's mass prefix
  //      P_own and mass T_own, and its threshold range [count(P_own),
  //      count(P_own + T_own)).  Every covering CTA computes the same
  //      integers in the same way, so the intervals tile [0, Z) exactly.
  if (warp_on) {
    const int h = p.hg * GW + hl;
    const int64_t bh = bh0 + hl;
    HeadGeom q;   // first: independent of the aggregates, overlaps their loads
    q.b = p.b;
    q.h = h;
    q.S_b = S_b;
    q.rcp = first ? pre_rcp : a.rcp_S[p.b];
    q.ksys = a.variant != VAR_SYS ? 0u
             : first ? pre_ksys[hl]
                     : philox4x32_10(make_uint4(0u, (uint32_t)h, (uint32_t)p.b, a.step), k0, k1).x >> 8;
    const int i_first = cov_s[0], i_last = cov_s[1];
    const Agg* ag = agg + bh * MAX_CTAS;
    constexpr int KR = 10;   // aggregates a lane keeps in registers (10 x 16 lanes covers every grid)
    int ek[KR];
    long long Fk[KR];
    int emax = AGG_EMPTY;
    float mloc = -INFINITY;
#pragma unroll
    for (int k = 0; k < KR; ++k) {
      const int i = i_first + r + k * lph;
      Agg x;
      x.m = -INFINITY;
      x.e = AGG_EMPTY;
      x.F = 0;
      if (i <= i_last && nonempty(i)) x = ag[i];
      ek[k] = x.e;
      Fk[k] = x.F;
      emax = max(emax, x.e);
      mloc = fmaxf(mloc, x.m);
    }
    for (int i = i_first + r + KR * lph; i <= i_last; i += lph)
      if (nonempty(i)) {
        emax = max(emax, ag[i].e);
        mloc = fmaxf(mloc, ag[i].m);
      }
    for (int o = lph >> 1; o > 0; o >>= 1) emax = max(emax, __shfl_xor_sync(FULL, emax, o, lph));
    const float mstar = grp_max(mloc, lph);
    long long before = 0, Z = 0, T_own = 0;
    auto add = [&](int i, int e, long long F) {
      const int d = emax - e;
      const long long Ti = d < 63 ? (F >> d) : 0;
      Z += Ti;
      before += i < cta ? Ti : 0;
      T_own += i == cta ? Ti : 0;
    };
#pragma unroll
    for (int k = 0; k < KR; ++k) add(i_first + r + k * lph, ek[k], Fk[k]);
    for (int i = i_first + r + KR * lph; i <= i_last; i += lph)
      if (nonempty(i)) add(i, ag[i].e, ag[i].F);
    for (int o = lph >> 1; o > 0; o >>= 1) {
      Z += __shfl_xor_sync(FULL, Z, o, lph);
      before += __shfl_xor_sync(FULL, before, o, lph);
      T_own += __shfl_xor_sync(FULL, T_own, o, lph);
    }
    const long long P_own = before;
    if (cta == i_first && r == 0 && hv) a.head_max[bh] = mstar;
    const Draws dr = make_draws(q, bh, Z);
    int jlo, jhi;
    if (a.variant == VAR_IID) {
      int rounds = 1;
      for (int span = S_b; span > 1; span = (span + lph - 1) / lph) ++rounds;
      jlo = dr.count_below(P_own, r, lph, lane, rounds);
      jhi = dr.count_below(P_own + T_own, r, lph, lane, rounds);
    } else {
      // even lanes of the group count the thresholds below P_own, odd
      // lanes those below P_own + T_own.  theta_j lies in
      // [floor(j Z / S), floor((j + 1) Z / S)], so the count is within 2 of
      // e = trunc(X S / Z): the lanes test the window [e - w, e + w) at once
      // (w = lph / 4 >= 2); the serial search covers a missed window.
      const long long X = (r & 1) ? P_own + T_own : P_own;
      const int w = lph >> 2;
      int e = 0;
      if (X >= Z) e = S_b;
      else if (X > 0) {
        const int sh = max(0, 40 - __clzll(Z));
        e = (int)(__fdividef((float)(uint32_t)(X >> sh), (float)(uint32_t)(Z >> sh)) * (float)S_b);
        e = min(max(e, 0), S_b);
      }
      const int j = e - w + (r >> 1);
      const bool below = X > 0 && (X >= Z ? j < S_b : (j < 0 || (j < S_b && dr.theta(j) < X)));
      const unsigned gbits = lph == 32 ? 0xffffffffu : ((1u << lph) - 1u);
      const unsigned par = (r & 1) ? 0xaaaaaaaau : 0x55555555u;
      const unsigned bal = (__ballot_sync(FULL, below) >> (lane - r)) & gbits & par;
      int c = X <= 0 ? 0 : X >= Z ? S_b : e - w + __popc(bal);
      const int last = lph - 2 + (r & 1);   // the lane testing j = e + w - 1
      const bool miss = X > 0 && X < Z && (!((bal >> (r & 1)) & 1u) && e - w >= 0 || ((bal >> last) & 1u));
      if (miss) c = dr.count_below(X, 0, lph, lane, 0);
      jlo = __shfl_sync(FULL, c, 0, lph);
      jhi = __shfl_sync(FULL, c, 1, lph);
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
      hinfo[hl].ref = (float)emax;
      carry_s[hl] = P_own;
    }
  }
  float acc[HPW][CPL];   // this warp's heads' sums of count x V (output columns of the lane)
#pragma unroll
  for (int j = 0; j < HPW; ++j)
#pragma unroll
    for (int k = 0; k < CPL; ++k) acc[j][k] = 0.f;
  const int nseg = seg_count(p);
  for (int sg_i = 0; sg_i < nseg; ++sg_i) {
    const Seg g = seg_of(p, sg_i);
    if (!(first && sg_i == 0)) stage(p, g);   // the first piece's first segment was staged at the first barrier
    if (tid == 0) {
      n_items = 0;
      n_ent = 0;
    }
    cp_async_wait_all();
    __syncthreads();   // staged data, thresholds and head state visible
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
        const long long Wc = c < g.nch ? fixed40(fast_exp2(fmaf(mx[c], LOG2E, -hi.ref)) * sm[c]) : 0;
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
    //      chunk's key total goes to its last nonzero key); each drawn
    //      (head, key) pair and its count go to the segment's list, and its
    //      V row is started towards L2.
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
      long long F = fixed40(fast_exp2(fmaf(sv, LOG2E, -hi.ref)));   // 2^-inf = 0 past the sequence end
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
      const unsigned dm = __ballot_sync(FULL, cnt > 0);
      if (dm) {   // warp-uniform: one list slot per drawn (head, key)
        int base = 0;
        if (lane == __ffs(dm) - 1) base = atomicAdd(&n_ent, __popc(dm));
        base = __shfl_sync(FULL, base, __ffs(dm) - 1);
        if (cnt > 0) {
          g.ent[base + __popc(dm & ((1u << lane) - 1u))] =
              ((uint32_t)(key - g.key_lo) << 19) | ((uint32_t)qh << 13) | (uint32_t)cnt;
          const T* vrow = reinterpret_cast<const T*>(a.V) + ((p.row0 + key) * a.Hkv + p.hg * W + qh / G) * (int64_t)D;
#pragma unroll
          for (int ln = 0; ln < (D * 2 + 127) / 128; ++ln)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(vrow + ln * 64));
        }
      }
    }
    __syncthreads();   // the list is complete
    // ---- gather: warp w sums the listed pairs of its heads (w, w + 16,
    //      ...), four V rows in flight; lane l owns output columns
    //      [l CPL, (l + 1) CPL), the sums stay in registers for the piece
    {
      const int ne = n_ent;
      const T* Vb = reinterpret_cast<const T*>(a.V) + (p.row0 + g.key_lo) * a.Hkv * D + (int64_t)p.hg * W * D +
                    lane * CPL;
      for (int e0 = 0; e0 < ne; e0 += 32) {
        const uint32_t ev = e0 + lane < ne ? g.ent[e0 + lane] : 0u;
        unsigned mine = __ballot_sync(FULL, e0 + lane < ne && (int)((ev >> 13) & 63u) % SB_WARPS == warp);
        while (mine) {   // warp-uniform
          uint32_t eu[4];
          uint2 raw[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int src = mine ? __ffs(mine) - 1 : 0;
            eu[u] = mine ? __shfl_sync(FULL, ev, src) : 0u;
            mine &= mine - 1;
            raw[u] = make_uint2(0u, 0u);
            if (eu[u] & 8191u) {   // a count of zero marks an empty slot
              const T* srow = Vb + ((int64_t)(eu[u] >> 19) * a.Hkv + (int)((eu[u] >> 13) & 63u) / G) * D;
              if constexpr (CPL == 4) raw[u] = *reinterpret_cast<const uint2*>(srow);
              else raw[u].x = *reinterpret_cast<const uint32_t*>(srow);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (eu[u] & 8191u) {   // warp-uniform
              const int jj = (int)((eu[u] >> 13) & 63u) / SB_WARPS;
              const float c = (float)(eu[u] & 8191u);
              f2x pr[4];
              Pairs<T>::get(make_uint4(raw[u].x, raw[u].y, 0u, 0u), pr);
              const float2 p0 = unpack2(pr[0]), p1 = unpack2(pr[1]);
              const float vf[4] = {p0.x, p0.y, p1.x, p1.y};
#pragma unroll
              for (int j = 0; j < HPW; ++j)
                if (j == jj)
#pragma unroll
                  for (int k = 0; k < CPL; ++k) acc[j][k] = fmaf(c, vf[k], acc[j][k]);
            }
          }
        }
      }
    }
    __syncthreads();   // the segment's buffers are free for the next one
  }
  // ---- the piece's sums, times 1/S_b, into out (vectorised fp32
  //      reductions, their order across CTAs not fixed)
  {
    const float inv_S = 1.0f / (float)S_b;
#pragma unroll
    for (int j = 0; j < HPW; ++j) {
      const int hl2 = warp + j * SB_WARPS;
      bool nz = false;
#pragma unroll
      for (int k = 0; k < CPL; ++k) nz |= acc[j][k] != 0.f;
      if (hl2 < GW && nz) {
        float* o = a.out + (bh0 + hl2) * D + lane * CPL;
        if constexpr (CPL == 4)
          red_add_v4(o, make_float4(acc[j][0] * inv_S, acc[j][1] * inv_S, acc[j][2] * inv_S, acc[j][3] * inv_S));
        else
          red_add_v2(o, make_float2(acc[j][0] * inv_S, acc[j][1] * inv_S));
      }
    }
  }
  });
  cp_async_wait_all();   // no copy outlives the CTA (a staged piece that was skipped)
}
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

// ---------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------
template <typename T, int D, int GM>
static cudaError_t launch_fused_g(const LaunchArgs& a, unsigned* bar_count, unsigned* bar_gen) {
  using Gm = StreamGeom<T, D>;
  static_assert((size_t)GM * 8 * sizeof(HeadInfo) + (size_t)POOL_CAP * 8 +
                        (size_t)64 * (8 + 16 + 4 * SUB) * 2 + (size_t)64 * SUB * 4 * 2 + 64 * 84 + 128 <=
                    Gm::SMEM,
                "phase B fixed regions and a two-chunk segment fit the ring");
  const int W = a.W;
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

cudaError_t launch_fused(const LaunchArgs& a_in, unsigned* bar_count, unsigned* bar_gen) {
  LaunchArgs a = a_in;
  // W = the largest power of two <= 8 dividing H_kv: units of 32 keys x W KV
  // heads (measured against W = 1, 2, 4 on 8K-128K contexts and batched
  // workloads, this was the fastest or within 1% except at 8K)
  a.W = unit_heads(a.Hkv);
  switch (a.dtype * 2 + (a.D == 128)) {
    case 0: return launch_fused_t<bf16_t, 64>(a, bar_count, bar_gen);
    case 1: return launch_fused_t<bf16_t, 128>(a, bar_count, bar_gen);
    case 2: return launch_fused_t<fp16_t, 64>(a, bar_count, bar_gen);
    case 3: return launch_fused_t<fp16_t, 128>(a, bar_count, bar_gen);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace santa
