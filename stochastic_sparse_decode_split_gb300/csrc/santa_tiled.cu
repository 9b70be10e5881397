// santa_tiled.cu -- the pages' tile samplers, S2ANTA-prop and S2ANTA-flash
// ("Stochastic Sparse Attention for Memory-Bound Inference", App. O,
// Alg. 2-5; App. P, Alg. 6-8), for bf16 / fp16 / fp32 caches.
//
// Both run after the score pass (santa_score.cu), which leaves the scaled
// scores and the 16-key chunk statistics (max, exp-sum) in the workspace:
//   prop   tiled_budget_kernel   Alg. 4: largest-remainder tile budgets    (one CTA per head)
//          tiled_sample_kernel   Alg. 5: per-tile systematic counts, gather (one CTA per tile and KV head)
//          tiled_merge_kernel    sum of the tiles' partial outputs, x 1/S  (one CTA per head)
//   flash  tiled_sample_kernel   Alg. 7: the same counts with the uniform budget S_tile
//          tiled_merge_kernel    Alg. 8: partials weighted by W_t / (Z S_tile)
// The pages' flash kernel 1 also computes the scores; here the score pass
// does that for both samplers, and both sum the tiles' partials in a fixed
// order in the merge (no atomics: the result does not depend on timing).
//
// Counts.  Inside tile t of a head with budget S_t, Alg. 5 gives key n the
// integers k in (a0 + P_n, a0 + P_n + x_n], x_n = S_t u_n / l_t and P_n the
// running sum of x.  So key n takes threshold k (k = 1..S_t) when
// U_n < (k - a0) l_t / S_t <= U_n+1, U the running sum of u_n = exp(s_n - m_t).
// Masses are fixed-point integers relative to the tile max (units of 2^-40:
// every prefix is exact) and a0 = a24 2^-24 is a 24-bit uniform, so each
// threshold theta_k = ceil((k 2^24 - a24) L / (S_t 2^24)) is an exact integer
// in [1, L] and key n takes the thetas with F_n-1 < theta <= F_n, F the
// inclusive prefix of the masses.  The intervals are open on the left, as
// the pages' floor rule makes them.
#include "santa_common.cuh"
#include "santa_launch.h"
#include "santa_seq.cuh"
#include "santa_window.cuh"

namespace santa {

constexpr int TB_THREADS = 256;   // budget and merge kernels
constexpr int TB_SMEM_T = 4096;   // tiles whose fractional parts the budget kernel keeps in shared memory
constexpr int TB_RANK_T = 256;    // up to this many tiles the leftover samples are placed by ranking
constexpr int TF_THREADS = 1024;  // budget and merge kernels, fast path
constexpr int TF_KC = 8;          // statistics chunks per thread on the fast path
constexpr int TF_T = TF_THREADS;  // tiles per head on the fast path

__device__ __forceinline__ int64_t seq_rows(const LaunchArgs& a, int b, int64_t& row0) {
  if (a.kv_offsets) {
    row0 = a.kv_offsets[b];
    return a.kv_offsets[b + 1] - row0;
  }
  row0 = (int64_t)b * a.nk_max;
  return a.nk_max;
}

// mass_fixed's integer for w in [0, 2^23) by one conversion: the scale by 2^40
// is exact in fp32 and the conversion toward zero is the floor; anything else
// (negative, not finite, not a number, 2^23 and above) gives 0.  Equal to
// mass_fixed on [0, 2^23) and on negative and non-finite inputs (checked on
// every float below 2^23); measured faster in the tile sampler and slower in
// the single-launch decode's key step, which keeps mass_fixed.
__device__ __forceinline__ long long mass_fixed_cvt(float w) {
  return (w >= 0.f && w < 8388608.f) ? (long long)__float2ull_rz(w * 1099511627776.0f) : 0ll;
}

// S_tile of S2ANTA-flash: S / T rounded half up, at least 1 (App. P, Alg. 6).
__device__ __forceinline__ int flash_tile_budget(int S_b, int T) { return max(1, (2 * S_b + T) / (2 * T)); }

struct OpMax {
  __device__ __forceinline__ double operator()(double x, double y) const { return fmax(x, y); }
  __device__ __forceinline__ float operator()(float x, float y) const { return fmaxf(x, y); }
};
struct OpAdd {
  template <typename V_>
  __device__ __forceinline__ V_ operator()(V_ x, V_ y) const { return x + y; }
};
// Reduction over the CTA (every thread gets the result); red holds N / 32 values.
template <int N, typename V_, typename Op>
__device__ __forceinline__ V_ block_reduce(V_ v, Op op, V_* red) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(FULL, v, o));
  __syncthreads();   // red is free
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
#pragma unroll
  for (int w = 1; w < N / 32; ++w) v = op(v, red[w]);
  return v;
}

// Tile masses of one head (App. O, Alg. 4; App. P, Alg. 8) from the chunk
// statistics: m_t = max of the tile's chunk maxima, l_t = sum_c sum_c-chunk *
// exp(max_c - m_t), W_t = exp(m_t - m*) l_t into w[0..T); returns
// Z = sum_t W_t (float64 sums of fp32 terms, the same in every call).
__device__ double tile_masses(const LaunchArgs& a, int64_t bh, int64_t nk, int T, double* w, double* red) {
  const int C = a.tl_len / SUB;
  const int nch = (int)((nk + SUB - 1) / SUB);
  const float* mx = a.tile_max + bh * a.chunks_max;
  const float* sm = a.tile_sum + bh * a.chunks_max;
  double* mt = w + a.tl_T;   // second half of the scratch row: m_t
  // fp32 per chunk (the FP64 pipe is narrow on this part), float64 sums
  double mloc = -INFINITY;
  for (int t = threadIdx.x; t < T; t += TB_THREADS) {
    const int c0 = t * C, c1 = min(c0 + C, nch);
    float m = -INFINITY;
#pragma unroll 8
    for (int c = c0; c < c1; ++c) m = fmaxf(m, mx[c]);
    float l = 0.f;
#pragma unroll 8
    for (int c = c0; c < c1; ++c) l += sm[c] * expf(mx[c] - m);
    w[t] = (double)l;
    mt[t] = (double)m;
    mloc = fmax(mloc, (double)m);
  }
  const double mstar = block_reduce<TB_THREADS>(mloc, OpMax(), red);
  double zloc = 0.0;
  for (int t = threadIdx.x; t < T; t += TB_THREADS) {
    w[t] = (double)expf((float)(mt[t] - mstar)) * w[t];
    zloc += w[t];
  }
  return block_reduce<TB_THREADS>(zloc, OpAdd(), red);
}

// Reduction over a CTA of TF_THREADS threads (every thread gets the result,
// the same in each: a fixed butterfly order); red holds 32 values.
template <typename V_, typename Op>
__device__ __forceinline__ V_ block_reduce_1k(V_ v, Op op, V_* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(FULL, v, o));
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(FULL, v, o));
  return v;
}

// The fast path's tile statistics (TF_THREADS threads, every load in flight
// at once): tiles of C chunks, C a power of two <= 32, at most TF_KC *
// TF_THREADS chunks and TF_T tiles.  Thread i takes chunks i + TF_THREADS k,
// so a tile's C chunks sit on C neighbouring lanes and combine by shuffles:
// m_t the max of the chunk maxima, l_t = sum_c sum_c-chunk * exp(max_c - m_t),
// into sm_m[t], sm_l[t].
__device__ __forceinline__ void tile_stats_fast(const LaunchArgs& a, int64_t bh, int nch, int C, int T, float* sm_m,
                                                float* sm_l) {
  const int tid = threadIdx.x, lane = tid & 31;
  const float* mx = a.tile_max + bh * a.chunks_max;
  const float* sm = a.tile_sum + bh * a.chunks_max;
  float vm[TF_KC], vs[TF_KC];
#pragma unroll
  for (int k = 0; k < TF_KC; ++k) {
    const int c = k * TF_THREADS + tid;
    vm[k] = c < nch ? mx[c] : -INFINITY;
    vs[k] = c < nch ? sm[c] : 0.f;
  }
#pragma unroll
  for (int k = 0; k < TF_KC; ++k) {
    if (k * TF_THREADS >= nch) break;   // uniform over the CTA
    float m = vm[k];
    for (int o = 1; o < C; o <<= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
    float l = vm[k] > -INFINITY ? vs[k] * expf(vm[k] - m) : 0.f;
    for (int o = 1; o < C; o <<= 1) l += __shfl_xor_sync(FULL, l, o);
    const int c = k * TF_THREADS + tid;
    if ((lane & (C - 1)) == 0 && c / C < T) {
      sm_m[c / C] = m;
      sm_l[c / C] = l;
    }
  }
}

// W = e * l (e in [0, 1], l in [1, 2^10]: an exp factor and a tile's sum) as
// an integer in units of 2^-40, exactly (the 48-bit product of the two
// mantissas, shifted; truncated below 2^-40).
__device__ __forceinline__ unsigned long long weight_fixed(float e, float l) {
  const uint32_t be = __float_as_uint(e), bl = __float_as_uint(l);
  const int xe = (int)((be >> 23) & 0xffu), xl = (int)((bl >> 23) & 0xffu);
  if (xe == 0 || xl == 0 || xe == 0xff || xl == 0xff || ((be | bl) >> 31)) return 0ull;
  const unsigned long long prod =
      (unsigned long long)((be & 0x7fffffu) | 0x800000u) * (unsigned long long)((bl & 0x7fffffu) | 0x800000u);
  const int sh = (xe - 150) + (xl - 150) + 40;   // e l 2^40 = prod 2^sh
  return sh >= 0 ? prod << min(sh, 15) : (sh > -64 ? prod >> -sh : 0ull);
}

// ---------------------------------------------------------------------------
// S2ANTA-prop budgets (App. O, Alg. 4): S_t = floor(q_t), q_t = S W_t / Z,
// and the S - sum floor(q_t) samples left go to the largest fractional
// parts (equal parts: the lower tile first).  Output: the exclusive prefix of
// the budgets, tl_pre[bh][0..T], which also places each tile's draws in the
// head's row of sample_idx.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(TB_THREADS) tiled_budget_kernel(LaunchArgs a) {
  const int64_t bh = blockIdx.x;
  const int b = (int)(bh / a.H);
  const int tid = threadIdx.x;
  __shared__ double red[TB_THREADS / 32];
  __shared__ int redi[TB_THREADS / 32];
  __shared__ unsigned long long fr_s[TB_SMEM_T];
  int S_b;
  if (seq_error(a, b, S_b)) return;   // flagged by the merge kernel
  int64_t row0;
  const int64_t nk = seq_rows(a, b, row0);
  const int T = (int)((nk + a.tl_len - 1) / a.tl_len);
  double* w = a.tl_w + bh * 2 * a.tl_T;
  int32_t* pre = a.tl_pre + bh * (a.tl_T + 1);
  const double Z = tile_masses(a, bh, nk, T, w, red);
  // floors and fractional parts; a non-negative double orders as its bit
  // pattern read as an unsigned integer, so the ranking below compares
  // integers (comparisons on the FP64 pipe, narrow on this part, made the
  // quadratic ranking the slowest step)
  unsigned long long* frg = reinterpret_cast<unsigned long long*>(w);
  int floc = 0;
  for (int t = tid; t < T; t += TB_THREADS) {
    const double q = (double)S_b * w[t] / Z;
    const double f = floor(q);
    pre[t] = (int)f;
    floc += (int)f;
    const unsigned long long key = (unsigned long long)__double_as_longlong(q - f);
    if (T <= TB_SMEM_T) fr_s[t] = key;
    else frg[t] = key;
  }
  const int R = S_b - block_reduce<TB_THREADS>(floc, OpAdd(), redi);
  __syncthreads();   // every fractional part written
  // tile t gets one more sample when fewer than R tiles rank above it
  auto rank_pass = [&](const unsigned long long* fr) {
    for (int t = tid; t < T; t += TB_THREADS) {
      const unsigned long long ft = fr[t];
      int above = 0;
      for (int u = 0; u < T && above < R; ++u) above += (fr[u] > ft || (fr[u] == ft && u < t)) ? 1 : 0;
      if (above < R) pre[t] += 1;
    }
  };
  if (T <= TB_RANK_T) {
    rank_pass(fr_s);
  } else if (T <= TB_SMEM_T) {
    // more tiles: sort instead of ranking.  Each key keeps the fractional
    // part's bits above the lowest 12 of its mantissa and takes 4095 - t in
    // those 12 (a fraction equal to another's to 2^-40 goes to the lower
    // tile, as exact equality does); a bitonic network sorts the keys in
    // decreasing order (zeros pad to a power of two) and the first R tiles
    // get one more sample
    int T2 = 1;
    while (T2 < T) T2 <<= 1;
    for (int t = tid; t < T2; t += TB_THREADS)
      fr_s[t] = t < T ? ((fr_s[t] & ~0xFFFull) | (unsigned long long)(4095 - t)) : 0ull;
    __syncthreads();
    for (int k = 2; k <= T2; k <<= 1)
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = tid; i < T2; i += TB_THREADS) {
          const int l = i ^ j;
          if (l > i) {
            const unsigned long long x = fr_s[i], y = fr_s[l];
            const bool desc = (i & k) == 0;   // this run sorts in decreasing order
            if (desc ? x < y : x > y) {
              fr_s[i] = y;
              fr_s[l] = x;
            }
          }
        }
        __syncthreads();
      }
    for (int r = tid; r < R; r += TB_THREADS) pre[4095 - (int)(fr_s[r] & 0xFFFull)] += 1;
  } else {
    rank_pass(frg);
  }
  __syncthreads();
  // exclusive prefix in place, TB_THREADS tiles at a time
  int run = 0;
  for (int base = 0; base < T; base += TB_THREADS) {
    const int t = base + tid;
    const int v = t < T ? pre[t] : 0;
    int x = v;
    const int lane = tid % 32, warp = tid / 32;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(FULL, x, o);
      if (lane >= o) x += n;
    }
    __syncthreads();   // redi is free, every thread has read its budget
    if (lane == 31) redi[warp] = x;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int u = 0; u < TB_THREADS / 32; ++u) {
      before += u < warp ? redi[u] : 0;
      total += redi[u];
    }
    if (t < T) pre[t] = run + before + x - v;
    run += total;
  }
  if (tid == 0) pre[T] = run;
}

// The same budgets on the fast path (one CTA of TF_THREADS threads per head,
// thread t = tile t), with no float64 (its pipe is narrow on this part): the
// statistics with every load in flight; W_t = exp(m_t - m*) l_t as an exact
// 2^-40 integer and Z their integer sum, so that S W_t = S_t Z + r_t by one
// integer division gives the floor S_t and the fractional part r_t / Z, and
// the fractional parts rank as the remainders r_t (one denominator); the
// leftover samples by a parallel ranking (several threads per tile, up to
// TB_RANK_T tiles) or a bitonic sort of the remainders.
__global__ void __launch_bounds__(TF_THREADS) tiled_budget_fast_kernel(LaunchArgs a) {
  const int64_t bh = blockIdx.x;
  const int b = (int)(bh / a.H);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ float s_m[TF_T], s_l[TF_T];
  __shared__ unsigned long long s_key[TF_T];
  __shared__ int s_bud[TF_T];
  __shared__ unsigned long long s_redz[32];
  __shared__ float s_redf[32];
  __shared__ int s_redi[32], s_wsum[32];
  int S_b;
  if (seq_error(a, b, S_b)) return;   // flagged by the merge kernel
  int64_t row0;
  const int64_t nk = seq_rows(a, b, row0);
  const int T = (int)((nk + a.tl_len - 1) / a.tl_len);
  const int nch = (int)((nk + SUB - 1) / SUB);
  int32_t* pre = a.tl_pre + bh * (a.tl_T + 1);
  tile_stats_fast(a, bh, nch, a.tl_len / SUB, T, s_m, s_l);
  __syncthreads();
  const float mt = tid < T ? s_m[tid] : -INFINITY;
  const float mstar = block_reduce_1k(mt, OpMax(), s_redf);
  const unsigned long long W = (tid < T && mt > -INFINITY) ? weight_fixed(expf(mt - mstar), s_l[tid]) : 0ull;
  const unsigned long long Z = block_reduce_1k(W, OpAdd(), s_redz);
  int fl = 0;
  if (tid < T) {
    const unsigned long long SW = (unsigned long long)S_b * W;   // < 2^62: W < 2^50, S_b < 2^12
    const unsigned long long f = Z ? SW / Z : 0ull;
    fl = (int)f;
    s_bud[tid] = fl;
    s_key[tid] = SW - f * Z;   // the fractional part's numerator over Z
  }
  const int R = S_b - block_reduce_1k(fl, OpAdd(), s_redi);
  __syncthreads();   // every key and floor written
  if (T <= TB_RANK_T) {
    // tile tt gets one more sample when fewer than R tiles rank above it;
    // tpt threads per tile each compare every tpt-th key
    int T2 = 1;
    while (T2 < T) T2 <<= 1;
    const int tpt = min(32, TF_THREADS / T2);
    const int tt = tid / tpt, j = tid & (tpt - 1);
    int above = 0;
    if (tt < T) {
      const unsigned long long kt = s_key[tt];
      for (int u = j; u < T; u += tpt) {
        const unsigned long long ku = s_key[u];
        above += (ku > kt || (ku == kt && u < tt)) ? 1 : 0;
      }
    }
    for (int o = 1; o < tpt; o <<= 1) above += __shfl_xor_sync(FULL, above, o);
    if (j == 0 && tt < T && above < R) s_bud[tt] += 1;
  } else {
    // as the general kernel: keys keep the remainder's bits above the lowest
    // 12 and take 4095 - t in those 12 (remainders equal to 2^-48 of Z go to
    // the lower tile); a bitonic network sorts them in decreasing order and
    // the first R tiles get one more sample
    int T2 = 1;
    while (T2 < T) T2 <<= 1;
    if (tid < T2) s_key[tid] = tid < T ? ((s_key[tid] & ~0xFFFull) | (unsigned long long)(4095 - tid)) : 0ull;
    __syncthreads();
    for (int k = 2; k <= T2; k <<= 1)
      for (int j = k >> 1; j > 0; j >>= 1) {
        const int l = tid ^ j;
        if (tid < T2 && l > tid) {
          const unsigned long long x = s_key[tid], y = s_key[l];
          const bool desc = (tid & k) == 0;
          if (desc ? x < y : x > y) {
            s_key[tid] = y;
            s_key[l] = x;
          }
        }
        __syncthreads();
      }
    if (tid < R) s_bud[4095 - (int)(s_key[tid] & 0xFFFull)] += 1;
  }
  __syncthreads();
  // exclusive prefix of the budgets (one per thread), then the total
  const int v = tid < T ? s_bud[tid] : 0;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(FULL, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) s_wsum[warp] = x;
  __syncthreads();
  const int y = s_wsum[lane];
  int yi = y;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(FULL, yi, o);
    if (lane >= o) yi += n;
  }
  const int before = __shfl_sync(FULL, yi - y, warp), total = __shfl_sync(FULL, yi, 31);
  if (tid < T) pre[tid] = before + x - v;
  if (tid == 0) pre[T] = total;
}

// ---------------------------------------------------------------------------
// Per-tile systematic counts and the count-weighted gather (App. O, Alg. 5;
// App. P, Alg. 7).  One CTA per (tile, sequence, KV head): each head
// of the group takes its S_t thresholds; then every row drawn by any head is
// read once and added, times its per-head counts, into the tile's partial
// sums tl_o[bh][t] (zero for a head with no draws in the tile).
// ---------------------------------------------------------------------------
// Loads the CPL elements of a V row that lane `lane` owns, widened to fp32.
template <typename T, int CPL>
__device__ __forceinline__ void load_cols(const T* src, float (&v)[CPL]) {
  if constexpr (sizeof(T) == 2 && CPL == 4) {
    const uint2 r = *reinterpret_cast<const uint2*>(src);
    float f[8];
    Elem<T>::widen(make_uint4(r.x, r.y, 0u, 0u), f);
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = f[c];
  } else if constexpr (sizeof(T) == 2 && CPL == 2) {
    const uint32_t r = *reinterpret_cast<const uint32_t*>(src);
    float f[8];
    Elem<T>::widen(make_uint4(r, 0u, 0u, 0u), f);
    v[0] = f[0];
    v[1] = f[1];
  } else if constexpr (CPL == 4) {
    const float4 r = *reinterpret_cast<const float4*>(src);
    v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
  } else {
    const float2 r = *reinterpret_cast<const float2*>(src);
    v[0] = r.x; v[1] = r.y;
  }
}

// Dynamic shared memory of tiled_sample_kernel for tiles of `len` keys (GM
// warps: one per head of the group).
template <int D, int GM>
__host__ __device__ constexpr size_t tiled_sample_smem(int len) {
  return (size_t)GM * len * 8 + (size_t)GM * len * 4 + (size_t)GM * GM * D * 4;
}

template <typename T, int D, int GM>
__global__ void __launch_bounds__(32 * GM, 32 / GM) tiled_sample_kernel(LaunchArgs a) {
  constexpr int TS_WARPS = GM, TS_THREADS = 32 * GM;
  extern __shared__ __align__(16) unsigned char smem[];
  const int Lt = a.tl_len;
  long long* Fall = reinterpret_cast<long long*>(smem);             // [GM][Lt] inclusive mass prefix per head
  int* cnt = reinterpret_cast<int*>(Fall + (size_t)GM * Lt);          // [GM][Lt] counts
  float* part = reinterpret_cast<float*>(cnt + (size_t)GM * Lt);     // [TS_WARPS][GM][D] per-warp sums
  __shared__ int rows[TL_MAX_LEN];
  __shared__ int red_i[TS_WARPS];
  constexpr int CPL = D / 32;   // output columns per lane

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int64_t blk = blockIdx.x;
  const int t = (int)(blk % a.tl_T);
  const int bk = (int)(blk / a.tl_T);
  const int b = bk / a.Hkv, kvh = bk % a.Hkv;
  const int G = a.H / a.Hkv;
  int S_b;
  if (seq_error(a, b, S_b)) return;   // flagged by the merge kernel
  int64_t row0;
  const int64_t nk = seq_rows(a, b, row0);
  const int Tb = (int)((nk + Lt - 1) / Lt);
  if (t >= Tb) return;
  const int64_t k0 = (int64_t)t * Lt;   // first key of the tile
  const int len = (int)min((int64_t)Lt, nk - k0);
  const int S_tile = flash_tile_budget(S_b, Tb);
  const uint32_t s0 = (uint32_t)a.seed, s1 = (uint32_t)(a.seed >> 32);

  for (int i = tid; i < G * Lt; i += TS_THREADS) cnt[i] = 0;
  __syncthreads();

  // one warp per head of the group: tile max, fixed-point masses
  // 2^((s_n - m_t) log2 e) with their inclusive prefix, then the head's S_t
  // thresholds.  Keys n = lane + 32 i, eight rounds i at a time in
  // registers: their loads at once (with the budget's), eight interleaved
  // warp scans, the rounds' sums carried in order
  constexpr int RG = 8;
  for (int g = warp; g < G; g += TS_WARPS) {
    const int h = kvh * G + g;
    const int64_t bh = (int64_t)b * a.H + h;
    const int32_t* pre = a.tl_pre + bh * (a.tl_T + 1);
    const float* st = a.stash + bh * a.nk_max + k0;
    const int St = a.tl_sampler == 0 ? pre[t + 1] - pre[t] : S_tile;
    float v[RG];
#pragma unroll
    for (int i = 0; i < RG; ++i) v[i] = lane + 32 * i < len ? st[lane + 32 * i] : -INFINITY;
    if (St <= 0) continue;   // uniform over the warp
    long long* F = Fall + (size_t)g * Lt;
    float m = -INFINITY;
    for (int n = lane + 32 * RG; n < len; n += 32) m = fmaxf(m, st[n]);   // tiles past 32 RG keys
#pragma unroll
    for (int i = 0; i < RG; ++i) m = fmaxf(m, v[i]);
    m = warp_max(m);
    long long carry = 0;
    for (int r0 = 0; r0 < len; r0 += 32 * RG) {
      long long x[RG];
#pragma unroll
      for (int i = 0; i < RG; ++i) {
        const int n = r0 + lane + 32 * i;
        if (r0 > 0) v[i] = n < len ? st[n] : -INFINITY;
        x[i] = n < len ? mass_fixed_cvt(fast_exp2((v[i] - m) * LOG2E)) : 0ll;
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int i = 0; i < RG; ++i) {
          const long long y = __shfl_up_sync(FULL, x[i], o);
          if (lane >= o) x[i] += y;
        }
      }
#pragma unroll
      for (int i = 0; i < RG; ++i) {
        const int n = r0 + lane + 32 * i;
        if (n < len) F[n] = carry + x[i];
        carry += __shfl_sync(FULL, x[i], 31);
      }
    }
    __syncwarp();   // F visible to the warp
    const long long L = carry;
    // the tile's offset a0: uniform number t of head (b, h)
    const uint4 r4 = philox4x32_10(make_uint4((uint32_t)(t >> 2), (uint32_t)h, (uint32_t)b, a.step), s0, s1);
    const uint32_t a24 = ((t & 3) == 0 ? r4.x : (t & 3) == 1 ? r4.y : (t & 3) == 2 ? r4.z : r4.w) >> 8;
    const int pos0 = a.tl_sampler == 0 ? pre[t] : t * S_tile;
    // ceil(2^64 / St), once per head: top < 2^62 (N <= 2^36, L <= 2^50), so
    // the multiply-high below is floor(top / St) or one more
    const unsigned long long rcpSt = St > 1 ? ~0ull / (unsigned)St + 1ull : 0ull;
    for (int k = 1 + lane; k <= St; k += 32) {
      // theta = ceil(N L / (St 2^24)), N = k 2^24 - a24 <= St 2^24, in 128 bits
      const unsigned long long N = ((unsigned long long)k << 24) - a24;
      const unsigned long long lo = N * (unsigned long long)L, hi = __umul64hi(N, (unsigned long long)L);
      const unsigned long long top = (hi << 40) | (lo >> 24);   // floor(N L / 2^24) < 2^64
      unsigned long long Q = top;
      if (St > 1) {
        Q = __umul64hi(top, rcpSt);
        if (Q * (unsigned)St > top) --Q;
      }
      const unsigned long long Rm = top - Q * (unsigned)St;
      const long long theta = (long long)(Q + ((Rm | (lo & 0xffffffull)) ? 1ull : 0ull));
      int l0 = 0, l1 = len - 1;   // the first key with F >= theta (F[len - 1] = L >= theta)
      while (l0 < l1) {
        const int mid = (l0 + l1) >> 1;
        if (F[mid] >= theta) l1 = mid;
        else l0 = mid + 1;
      }
      atomicAdd(&cnt[g * Lt + l0], 1);
      if (a.sample_idx) a.sample_idx[bh * a.tl_draws + pos0 + k - 1] = (int32_t)(k0 + l0);
    }
  }
  __syncthreads();   // counts complete

  // rows drawn by any head of the group, in key order
  int nrow = 0;
  for (int base = 0; base < len; base += TS_THREADS) {
    const int n = base + tid;
    bool any = false;
    if (n < len)
      for (int g = 0; g < G; ++g) any |= cnt[g * Lt + n] != 0;
    const unsigned bal = __ballot_sync(FULL, any);
    if (lane == 0) red_i[warp] = __popc(bal);
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int u = 0; u < TS_WARPS; ++u) {
      before += u < warp ? red_i[u] : 0;
      total += red_i[u];
    }
    if (any) rows[nrow + before + __popc(bal & ((1u << lane) - 1u))] = n;
    nrow += total;
    __syncthreads();   // red_i is rewritten next round
  }

  // each drawn row once for all heads of the group; lane owns CPL columns
  float acc[GM][CPL];
#pragma unroll
  for (int g = 0; g < GM; ++g)
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[g][c] = 0.f;
  const T* Vb = reinterpret_cast<const T*>(a.V) + ((row0 + k0) * a.Hkv + kvh) * (int64_t)D + lane * CPL;
  for (int i0 = warp; i0 < nrow; i0 += 2 * TS_WARPS) {   // two rows in flight per warp
    const int i1 = i0 + TS_WARPS;
    const int n0 = rows[i0], n1 = i1 < nrow ? rows[i1] : n0;
    float v0[CPL], v1[CPL];
    load_cols<T, CPL>(Vb + (int64_t)n0 * a.Hkv * D, v0);
    load_cols<T, CPL>(Vb + (int64_t)n1 * a.Hkv * D, v1);
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      if (g < G) {
        const float c0 = (float)cnt[g * Lt + n0], c1 = i1 < nrow ? (float)cnt[g * Lt + n1] : 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[g][c] = fmaf(c1, v1[c], fmaf(c0, v0[c], acc[g][c]));
      }
    }
  }
#pragma unroll
  for (int g = 0; g < GM; ++g)
#pragma unroll
    for (int c = 0; c < CPL; ++c) part[(warp * GM + g) * D + lane * CPL + c] = acc[g][c];
  __syncthreads();
  for (int i = tid; i < G * D; i += TS_THREADS) {
    const int g = i / D, col = i % D;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < TS_WARPS; ++w) sum += part[(w * GM + g) * D + col];
    const int64_t bh = (int64_t)b * a.H + kvh * G + g;
    a.tl_o[(bh * a.tl_T + t) * D + col] = sum;
  }
}

// ---------------------------------------------------------------------------
// Merge (one CTA per head, thread per output column): out = sum_t w_t O_t
// with w_t = 1 / S for prop (tiles with a budget) and W_t / (Z S_tile) for
// flash (App. P, Alg. 8).  Also flags bad sequence metadata and marks
// the unused entries of the head's sample_idx row with -1.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(TB_THREADS) tiled_merge_kernel(LaunchArgs a) {
  const int64_t bh = blockIdx.x;
  const int b = (int)(bh / a.H), h = (int)(bh % a.H);
  const int tid = threadIdx.x;
  __shared__ double red[TB_THREADS / 32];
  int S_b;
  const int e = seq_error(a, b, S_b);
  if (e) {
    if (tid == 0 && h == 0) flag_error(a.err, e);
    for (int c = tid; c < D; c += TB_THREADS) a.out[bh * D + c] = 0.f;
    if (a.sample_idx)
      for (int j = tid; j < a.tl_draws; j += TB_THREADS) a.sample_idx[bh * a.tl_draws + j] = -1;
    return;
  }
  int64_t row0;
  const int64_t nk = seq_rows(a, b, row0);
  const int T = (int)((nk + a.tl_len - 1) / a.tl_len);
  const int S_tile = flash_tile_budget(S_b, T);
  double* w = a.tl_w + bh * 2 * a.tl_T;
  float* wf = reinterpret_cast<float*>(w + a.tl_T);   // the tiles' weights in fp32
  const int32_t* pre = a.tl_pre + bh * (a.tl_T + 1);
  if (a.tl_sampler == 1) {
    const double Z = tile_masses(a, bh, nk, T, w, red);
    const float inv = (float)(1.0 / (Z * (double)S_tile));
    __syncthreads();   // tile_masses used the second half of the row
    for (int t = tid; t < T; t += TB_THREADS) wf[t] = (float)w[t] * inv;
  } else {
    const float inv = 1.f / (float)S_b;
    for (int t = tid; t < T; t += TB_THREADS) wf[t] = pre[t + 1] > pre[t] ? inv : 0.f;
  }
  __syncthreads();
  // thread (c, j): column c, tiles j, j + NJ, ... (NJ = TB_THREADS / D), eight
  // loads in flight; the NJ partial sums are added in a fixed order
  constexpr int NJ = TB_THREADS / D;
  __shared__ float part[TB_THREADS];
  const float* o = a.tl_o + bh * a.tl_T * D;
  {
    const int c = tid % D, j = tid / D;
    float sum = 0.f;
    for (int t0 = j; t0 < T; t0 += 8 * NJ) {
      float v[8], wt[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int t = t0 + u * NJ;
        wt[u] = t < T ? wf[t] : 0.f;
        v[u] = (t < T && wt[u] != 0.f) ? o[(int64_t)t * D + c] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) sum = fmaf(wt[u], v[u], sum);
    }
    part[tid] = sum;
  }
  __syncthreads();
  if (tid < D) {
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) sum += part[j * D + tid];
    a.out[bh * D + tid] = sum;
  }
  if (a.sample_idx) {
    const int used = a.tl_sampler == 0 ? S_b : T * S_tile;
    for (int j = used + tid; j < a.tl_draws; j += TB_THREADS) a.sample_idx[bh * a.tl_draws + j] = -1;
  }
}

// The merge on the fast path (one CTA of TF_THREADS threads per head): the
// tiles' weights as above (flash: from the fast tile statistics), then thread
// (c, j) sums column c over tiles j, j + NJ, ... with all its loads in flight
// (NJ = TF_THREADS / D), and the NJ partial sums are added in a fixed order.
template <int D>
__global__ void __launch_bounds__(TF_THREADS) tiled_merge_fast_kernel(LaunchArgs a) {
  const int64_t bh = blockIdx.x;
  const int b = (int)(bh / a.H), h = (int)(bh % a.H);
  const int tid = threadIdx.x;
  __shared__ float s_m[TF_T], s_w[TF_T];
  __shared__ float s_part[TF_THREADS];
  __shared__ unsigned long long s_redz[32];
  __shared__ float s_redf[32];
  int S_b;
  const int e = seq_error(a, b, S_b);
  if (e) {
    if (tid == 0 && h == 0) flag_error(a.err, e);
    for (int c = tid; c < D; c += TF_THREADS) a.out[bh * D + c] = 0.f;
    if (a.sample_idx)
      for (int j = tid; j < a.tl_draws; j += TF_THREADS) a.sample_idx[bh * a.tl_draws + j] = -1;
    return;
  }
  int64_t row0;
  const int64_t nk = seq_rows(a, b, row0);
  const int T = (int)((nk + a.tl_len - 1) / a.tl_len);
  const int S_tile = flash_tile_budget(S_b, T);
  // thread (c, j): column c, tiles j, j + NJ, ...; its first U partials are
  // requested now, in flight while the weights are formed (a tile without a
  // budget holds zeros)
  constexpr int NJ = TF_THREADS / D, U = 16;
  const float* o = a.tl_o + bh * a.tl_T * D;
  const int c = tid % D, j = tid / D;
  float v0[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int t = j + u * NJ;
    v0[u] = t < T ? o[(int64_t)t * D + c] : 0.f;
  }
  if (a.tl_sampler == 1) {
    tile_stats_fast(a, bh, (int)((nk + SUB - 1) / SUB), a.tl_len / SUB, T, s_m, s_w);
    __syncthreads();
    const float mt = tid < T ? s_m[tid] : -INFINITY;
    const float mstar = block_reduce_1k(mt, OpMax(), s_redf);
    const unsigned long long W = (tid < T && mt > -INFINITY) ? weight_fixed(expf(mt - mstar), s_w[tid]) : 0ull;
    const unsigned long long Z = block_reduce_1k(W, OpAdd(), s_redz);
    // W_t / (Z S_tile) in fp32 (both in units of 2^-40)
    const float inv = 1.f / ((float)Z * (float)S_tile);
    __syncthreads();   // every s_w read
    if (tid < T) s_w[tid] = (float)W * inv;
  } else if (tid < T) {
    const int32_t* pre = a.tl_pre + bh * (a.tl_T + 1);
    s_w[tid] = pre[tid + 1] > pre[tid] ? 1.f / (float)S_b : 0.f;
  }
  __syncthreads();
  {
    float sum = 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = j + u * NJ;
      sum = fmaf(t < T ? s_w[t] : 0.f, v0[u], sum);
    }
    for (int t0 = j + U * NJ; t0 < T; t0 += U * NJ) {   // more than U NJ tiles
      float v[U], wt[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int t = t0 + u * NJ;
        wt[u] = t < T ? s_w[t] : 0.f;
        v[u] = (t < T && wt[u] != 0.f) ? o[(int64_t)t * D + c] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) sum = fmaf(wt[u], v[u], sum);
    }
    s_part[tid] = sum;
  }
  __syncthreads();
  if (tid < D) {
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) sum += s_part[j * D + tid];
    a.out[bh * D + tid] = sum;
  }
  if (a.sample_idx) {
    const int used = a.tl_sampler == 0 ? S_b : T * S_tile;
    for (int j = used + tid; j < a.tl_draws; j += TF_THREADS) a.sample_idx[bh * a.tl_draws + j] = -1;
  }
}

// ---------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------
template <typename T, int D, int GM>
static cudaError_t launch_tiled_g(const LaunchArgs& a) {
  const size_t smem = tiled_sample_smem<D, GM>(a.tl_len);
  cudaError_t e = cudaFuncSetAttribute(tiled_sample_kernel<T, D, GM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tiled_sample_smem<D, GM>(TL_MAX_LEN));
  if (e != cudaSuccess) return e;
  // one wave of samplers needs about seven CTAs per SM: all of its shared memory
  e = cudaFuncSetAttribute(tiled_sample_kernel<T, D, GM>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  const unsigned heads = (unsigned)((int64_t)a.B * a.H);
  // the fast budget and merge kernels: tiles of a power-of-two number of
  // chunks (at most 32), at most TF_T tiles and TF_KC * TF_THREADS chunks
  const int C = a.tl_len / SUB;
  const bool fast = (C & (C - 1)) == 0 && C <= 32 && a.tl_T <= TF_T && a.chunks_max <= TF_KC * TF_THREADS;
  // plain stream order (launching the next kernel early with programmatic
  // dependent launch was measured slower: its waiting CTAs hold SM slots)
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(fast ? TF_THREADS : TB_THREADS);
  cfg.stream = a.stream;
  if (a.tl_sampler == 0) {
    cfg.gridDim = dim3(heads);
    cfg.dynamicSmemBytes = 0;
    if ((e = fast ? cudaLaunchKernelEx(&cfg, tiled_budget_fast_kernel, a)
                  : cudaLaunchKernelEx(&cfg, tiled_budget_kernel, a)) != cudaSuccess)
      return e;
  }
  cfg.gridDim = dim3((unsigned)((unsigned long long)a.tl_T * a.B * a.Hkv));
  cfg.blockDim = dim3(32 * GM);
  cfg.dynamicSmemBytes = smem;
  if ((e = cudaLaunchKernelEx(&cfg, tiled_sample_kernel<T, D, GM>, a)) != cudaSuccess) return e;
  cfg.gridDim = dim3(heads);
  cfg.blockDim = dim3(fast ? TF_THREADS : TB_THREADS);
  cfg.dynamicSmemBytes = 0;
  return fast ? cudaLaunchKernelEx(&cfg, tiled_merge_fast_kernel<D>, a)
              : cudaLaunchKernelEx(&cfg, tiled_merge_kernel<D>, a);
}

template <typename T, int D>
static cudaError_t launch_tiled_t(const LaunchArgs& a) {
  return (a.H / a.Hkv <= 4) ? launch_tiled_g<T, D, 4>(a) : launch_tiled_g<T, D, 8>(a);
}

cudaError_t launch_tiled(const LaunchArgs& a) {
  switch (a.dtype * 2 + (a.D == 128)) {
    case 0: return launch_tiled_t<bf16_t, 64>(a);
    case 1: return launch_tiled_t<bf16_t, 128>(a);
    case 2: return launch_tiled_t<fp16_t, 64>(a);
    case 3: return launch_tiled_t<fp16_t, 128>(a);
    case 4: return launch_tiled_t<float, 64>(a);
    case 5: return launch_tiled_t<float, 128>(a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace santa
