// santa_sample.cu -- cross-chunk combine, Philox thresholds, inverse-CDF
// sampling and the GQA-deduplicated V gather-add, for sm_103a.
//
// "Stochastic Sparse Attention for Memory-Bound Inference":
//   combine   m* = max_t m_t, W_t = e^{m_t - m*} l_t, Z = sum_t W_t   (App. O, Alg. 4)
//   samplers  i.i.d. / stratified / systematic thresholds            (Sec. 2.1; Eq. 4)
//   inverse CDF, left-closed: F(n-1) <= t < F(n)                     (App. A.4)
//   gather    O_h = (1/S) sum_n c_{h,n} V_n over the union of rows
//             drawn by the heads of a KV group                        (Eq. 4, Fig. 1; App. O, Alg. 5)
//
// Difference from the pages' kernels: Alg. 4 rounds per-tile budgets by
// largest remainder and then samples each tile systematically on its own.
// Here every head's S thresholds are placed globally (prefix of chunk masses)
// and resolved inside the 32-key window that holds them, which reproduces the
// global i.i.d. / stratified / systematic estimators exactly.
#include <climits>

#include "santa_common.cuh"
#include "santa_launch.h"
#include "santa_window.cuh"

namespace santa {

struct HeadCtx {
  int64_t row0, nk;
  int S;
  int err;  // 0 when the head is usable
};

__device__ __forceinline__ HeadCtx head_ctx(const LaunchArgs& a, int b) {
  HeadCtx c;
  if (a.kv_offsets) {
    c.row0 = a.kv_offsets[b];
    c.nk = a.kv_offsets[b + 1] - c.row0;
  } else {
    c.row0 = (int64_t)b * a.nk_max;
    c.nk = a.nk_max;
  }
  c.S = a.S_per_seq ? a.S_per_seq[b] : a.S_max;
  c.err = 0;
  if (c.nk < 1) c.err |= ERR_EMPTY;
  else if (c.nk > a.nk_max || c.row0 < 0) c.err |= ERR_NK_BOUND;
  if (c.S < 1 || c.S > a.S_max) c.err |= ERR_S_RANGE;
  return c;
}

// Inclusive block-wide scan of one int64 per thread (NT threads).
template <int NT>
__device__ __forceinline__ long long block_inclusive_scan(long long v, long long* warp_tot) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(FULL, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  long long off = 0;
  for (int w = 0; w < warp; ++w) off += warp_tot[w];
  __syncthreads();
  return v + off;
}

// ---------------------------------------------------------------------------
// Combine + thresholds.  grid = (H, B), block = 256.  Three passes over the
// head's chunk statistics (max; per-thread run sums and a block scan; the
// prefix and first-threshold index of every chunk).
// dynamic smem: theta int64[S_max] | ukey uint32[S_pow2]
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(THREADS)
combine_kernel(LaunchArgs a, int S_pow2) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  long long* theta = reinterpret_cast<long long*>(smem_raw);
  uint32_t* ukey = reinterpret_cast<uint32_t*>(theta + a.S_max);
  __shared__ float red[WARPS];
  __shared__ long long warp_tot[WARPS];
  __shared__ long long s_Z;
  __shared__ double s_invS;

  const int h = blockIdx.x, b = blockIdx.y;
  const int64_t bh = (int64_t)b * a.H + h;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  wait_for_predecessor();   // the score pass has completed and its writes are visible
  allow_dependents();
  const HeadCtx hc = head_ctx(a, b);
  if (hc.err) {
    if (tid == 0 && h == 0) flag_error(a.err, hc.err);
    if (a.sample_idx)
      for (int j = tid; j < a.S_max; j += THREADS) a.sample_idx[bh * a.S_max + j] = -1;
    return;
  }
  const int C = (int)((hc.nk + SUB - 1) / SUB);
  const int S = hc.S;
  const float* tmax = a.tile_max + bh * a.chunks_max;
  const float* tsum = a.tile_sum + bh * a.chunks_max;

  // each thread owns a contiguous run of chunks; its statistics are loaded once
  // (kept in registers for runs of up to PMAX chunks)
  constexpr int PMAX = 16;
  const int per = (C + THREADS - 1) / THREADS;
  const int c_lo = min(C, tid * per), c_hi = min(C, c_lo + per);
  const bool in_regs = per <= PMAX;
  float lm[PMAX], ll[PMAX];
  float m = -INFINITY;
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < PMAX; ++i) {
      const int c = c_lo + i;
      lm[i] = (c < c_hi) ? tmax[c] : -INFINITY;
      ll[i] = (c < c_hi) ? tsum[c] : 0.f;
      m = fmaxf(m, lm[i]);
    }
  } else {
    for (int c = c_lo; c < c_hi; ++c) m = fmaxf(m, tmax[c]);
  }
  m = warp_max(m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float mstar = red[0];
#pragma unroll
  for (int w = 1; w < WARPS; ++w) mstar = fmaxf(mstar, red[w]);

  // chunk masses W_c = e^{m_c - m*} l_c over the run, block scan
  auto mass = [&](int i, int c) -> long long {
    return in_regs ? ((c < c_hi) ? mass_fixed(expf(lm[i] - mstar) * ll[i]) : 0)
                   : mass_fixed(expf(tmax[c] - mstar) * tsum[c]);
  };
  long long local = 0;
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < PMAX; ++i) local += mass(i, c_lo + i);
  } else {
    for (int c = c_lo; c < c_hi; ++c) local += mass(0, c);
  }
  const long long incl = block_inclusive_scan<THREADS>(local, warp_tot);
  if (tid == THREADS - 1) s_Z = incl;
  if (tid == 0) s_invS = 1.0 / (double)S;  // one fp64 division per head
  __syncthreads();
  const double Z = (double)s_Z;
  const double invS = s_invS;

  // thresholds t_j (Sec. 2.1) in mass units: theta_j = t_j * Z.  Uniforms are
  // 24-bit integers k (u = k * 2^-24); t_j = (j + u) / S is formed in fp64
  // once per threshold (the only fp64 arithmetic, S operations per head).
  const uint32_t k0 = (uint32_t)a.seed, k1 = (uint32_t)(a.seed >> 32);
  if (a.variant == 2) {  // systematic: one offset
    double u;
    if (a.uniforms) u = a.uniforms[bh * a.S_max];
    else u = word_to_unit(philox4x32_10(make_uint4(0u, (uint32_t)h, (uint32_t)b, a.step), k0, k1).x);
    for (int j = tid; j < S; j += THREADS) theta[j] = (long long)(((double)j + u) * invS * Z);
  } else {
    for (int i = tid; i < (S + 3) / 4; i += THREADS) {
      double u4[4];
      if (a.uniforms) {
#pragma unroll
        for (int r = 0; r < 4; ++r) u4[r] = (4 * i + r < S) ? a.uniforms[bh * a.S_max + 4 * i + r] : 0.0;
      } else {
        const uint4 w = philox4x32_10(make_uint4((uint32_t)i, (uint32_t)h, (uint32_t)b, a.step), k0, k1);
        u4[0] = word_to_unit(w.x);
        u4[1] = word_to_unit(w.y);
        u4[2] = word_to_unit(w.z);
        u4[3] = word_to_unit(w.w);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int j = 4 * i + r;
        if (j >= S) break;
        if (a.variant == 1) theta[j] = (long long)(((double)j + u4[r]) * invS * Z);
        else ukey[j] = (uint32_t)(u4[r] * 16777216.0);   // exact: u has 24 fraction bits
      }
    }
  }
  if (a.variant == 0) {  // i.i.d. draws are unordered: sort the 24-bit keys (bitonic, integer compares)
    for (int j = S + tid; j < S_pow2; j += THREADS) ukey[j] = 0xffffffffu;
    __syncthreads();
    for (int k = 2; k <= S_pow2; k <<= 1) {
      for (int jj = k >> 1; jj > 0; jj >>= 1) {
        for (int i = tid; i < S_pow2; i += THREADS) {
          const int ixj = i ^ jj;
          if (ixj > i) {
            const uint32_t x = ukey[i], y = ukey[ixj];
            const bool up = (i & k) == 0;
            if ((x > y) == up) {
              ukey[i] = y;
              ukey[ixj] = x;
            }
          }
        }
        __syncthreads();
      }
    }
    for (int j = tid; j < S; j += THREADS) theta[j] = (long long)((double)ukey[j] * (1.0 / 16777216.0) * Z);
  }
  __syncthreads();

  // prefix P_c and first threshold jstart[c] = #{j : theta_j < P_c} of every chunk
  long long run = incl - local;
  long long* pref = a.prefix + bh * (a.chunks_max + 1);
  int32_t* js = a.jstart + bh * (a.chunks_max + 1);
  auto emit = [&](int c, long long w) {
    int lo = 0, hi = S;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (theta[mid] < run) lo = mid + 1;
      else hi = mid;
    }
    pref[c] = run;
    js[c] = lo;
    run += w;
  };
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < PMAX; ++i)
      if (c_lo + i < c_hi) emit(c_lo + i, mass(i, c_lo + i));
  } else {
    for (int c = c_lo; c < c_hi; ++c) emit(c, mass(0, c));
  }
  if (tid == THREADS - 1) {
    pref[C] = s_Z;
    js[C] = S;  // every threshold lies below the total mass
  }
  for (int j = tid; j < S; j += THREADS) a.thresh[bh * a.S_max + j] = theta[j];
  if (a.sample_idx)
    for (int j = S + tid; j < a.S_max; j += THREADS) a.sample_idx[bh * a.S_max + j] = -1;
  if (tid == 0) a.head_max[bh] = mstar;
}

// ---------------------------------------------------------------------------
// Sample + gather.  grid = (H_kv, groups_max, B), block = 256 (8 warps);
// warp w owns sampling windows blockIdx.y * SPC + w * 2 + {0, 1} (32 keys
// each, one key per lane, i.e. two 16-key statistics chunks) for all heads of
// the KV group.
//
// Per (window, head) with thresholds: the lane's key mass e^{s - m*} in fixed
// point, an exact warp scan gives each key's inclusive prefix F_lane, and the
// thresholds x_j = theta_j - P_w (sorted, one per lane, batches of 32) are
// searched by shuffles: key `lane` is drawn by the thresholds with
// F_{lane-1} <= x_j < F_lane.  Windows without thresholds read nothing but
// their threshold range.  The rows drawn by any head form the union (each V
// row read once per KV head); the gather adds count * V in fp32.
//
// dynamic smem: counts int[8 warps][2][GM][32] | rows int[8 warps][64] | wbuf float[8 warps][G][D]
// ---------------------------------------------------------------------------
constexpr int SG_WARPS = WARPS;
constexpr int SG_THREADS = SG_WARPS * 32;
constexpr int SG_NSW = WIN_PER_WARP;   // sampling windows per warp
static_assert(SG_NSW * SG_WARPS == SPC, "windows per CTA");
static_assert(WIN == 32 && WIN == 2 * SUB, "a window is one key per lane, two statistics chunks");

template <int GM>
__host__ __device__ constexpr size_t sample_gather_smem(int G, int D) {
  return (size_t)SG_WARPS * SG_NSW * GM * 32 * sizeof(int) + (size_t)SG_WARPS * SG_NSW * 32 * sizeof(int) +
         (size_t)SG_WARPS * G * D * sizeof(float);
}

template <typename T, int D, int GM>
__global__ void __launch_bounds__(SG_THREADS)
sample_gather_kernel(LaunchArgs a) {
  using TL = Tile<T, D>;   // V row split: LPK lanes per row, KPI rows per load instruction
  constexpr int NSW = SG_NSW;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int has_rows[SG_WARPS];
  const int G = a.H / a.Hkv;
  const int kvh = blockIdx.x, grp = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  int* cnt_s = reinterpret_cast<int*>(smem_raw) + warp * (NSW * GM * 32);                 // [NSW][GM][32]
  int* rows = reinterpret_cast<int*>(smem_raw) + SG_WARPS * NSW * GM * 32 + warp * (NSW * 32);
  float* wbuf = reinterpret_cast<float*>(smem_raw + (size_t)SG_WARPS * NSW * (GM + 1) * 32 * sizeof(int));
  wait_for_predecessor();   // the combine has completed and its writes are visible
  const HeadCtx hc = head_ctx(a, b);
  const int64_t bh0 = (int64_t)b * a.H + kvh * G;
  if (hc.err) return;       // out was cleared by the score pass
  const int C = (int)((hc.nk + SUB - 1) / SUB);
  const int NW = (int)((hc.nk + WIN - 1) / WIN);
  const int NG = (NW + SPC - 1) / SPC;
  if (grp >= NG) return;
  const int w0 = grp * SPC + warp * NSW;   // first window of this warp
  const int cm1 = a.chunks_max + 1;

  // first pass: threshold range [js, je) and mass prefix of every (head, window)
  int js[GM][NSW], je[GM][NSW];
  long long pb[GM][NSW];
  float mst[GM];
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    mst[g] = (g < G) ? a.head_max[bh0 + g] : 0.f;
#pragma unroll
    for (int i = 0; i < NSW; ++i) {
      const int w = w0 + i;
      const bool act = g < G && w < NW;
      const int64_t base = (bh0 + g) * cm1;
      js[g][i] = act ? a.jstart[base + 2 * w] : 0;
      je[g][i] = act ? a.jstart[base + min(2 * w + 2, C)] : 0;
      pb[g][i] = act ? a.prefix[base + 2 * w] : 0;
    }
  }
  // second pass: scores and first 32 thresholds of the (head, window) pairs that draw
  float sv[GM][NSW];
  long long th[GM][NSW];
#pragma unroll
  for (int g = 0; g < GM; ++g)
#pragma unroll
    for (int i = 0; i < NSW; ++i) {
      const int64_t bh = bh0 + g;
      const int64_t key = (int64_t)(w0 + i) * WIN + lane;
      const bool draws = je[g][i] > js[g][i];
      sv[g][i] = (draws && key < hc.nk) ? a.stash[bh * a.nk_max + key] : -INFINITY;
      th[g][i] = (js[g][i] + lane < je[g][i]) ? a.thresh[bh * a.S_max + js[g][i] + lane] : LLONG_MAX;
    }

  // sampling: counts per (window, head, key) into shared memory
  unsigned drawn[NSW];
#pragma unroll
  for (int i = 0; i < NSW; ++i) {
    drawn[i] = 0u;
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      int cnt = 0;
      if (je[g][i] > js[g][i]) {  // warp-uniform
        const int64_t bh = bh0 + g;
        cnt = window_draws(sv[g][i], mst[g], th[g][i], je[g][i] - js[g][i], pb[g][i],
                           a.thresh + bh * a.S_max + js[g][i],
                           a.sample_idx ? a.sample_idx + bh * a.S_max + js[g][i] : nullptr, (w0 + i) * WIN + lane,
                           lane);
      }
      cnt_s[(i * GM + g) * 32 + lane] = cnt;
      drawn[i] |= __ballot_sync(FULL, cnt > 0);
    }
  }

  // union of the rows drawn by any head: compact list of (window, key) per warp
  int nrows = 0;
#pragma unroll
  for (int i = 0; i < NSW; ++i) {
    if (drawn[i] & (1u << lane)) rows[nrows + __popc(drawn[i] & ((1u << lane) - 1u))] = i * 32 + lane;
    nrows += __popc(drawn[i]);
  }
  if (lane == 0) has_rows[warp] = nrows > 0;
  __syncwarp();

  // count-weighted gather-and-add (each drawn V row read once, fp32 accumulation)
  if (nrows > 0) {
    const int slot = lane / TL::LPK, sub = lane % TL::LPK;
    float acc[GM][TL::EPL];
#pragma unroll
    for (int g = 0; g < GM; ++g)
#pragma unroll
      for (int e = 0; e < TL::EPL; ++e) acc[g][e] = 0.f;
    const T* Vbase = reinterpret_cast<const T*>(a.V) + (hc.row0 * a.Hkv + kvh) * (int64_t)D + sub * TL::EPL;
    gather_rows<T, D, GM>(acc, rows, nrows, cnt_s, Vbase, w0, a.Hkv, G, lane);
    reduce_slots<T, D, GM>(acc);
    if (slot == 0) {
#pragma unroll
      for (int g = 0; g < GM; ++g)
        if (g < G)
#pragma unroll
          for (int e = 0; e < TL::EPL; ++e) wbuf[(warp * G + g) * D + sub * TL::EPL + e] = acc[g][e];
    }
  }
  __syncthreads();

  // this CTA's sum per head, times 1/S, added into out (cleared by the score
  // pass) with vectorised fp32 reductions; warps that drew nothing are
  // skipped.  The order of the additions across CTAs is not fixed, so the last
  // bits of out may differ between runs; the drawn indices never do.
  unsigned warps_with_rows = 0u;
#pragma unroll
  for (int w = 0; w < SG_WARPS; ++w) warps_with_rows |= has_rows[w] ? (1u << w) : 0u;
  if (!warps_with_rows) return;
  const float inv_S = 1.0f / (float)hc.S;
  for (int i4 = tid; i4 < G * D / 4; i4 += SG_THREADS) {
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < SG_WARPS; ++w) {
      if (warps_with_rows & (1u << w)) {
        const float4 v = reinterpret_cast<const float4*>(wbuf)[w * G * D / 4 + i4];
        sum.x += v.x;
        sum.y += v.y;
        sum.z += v.z;
        sum.w += v.w;
      }
    }
    if (sum.x != 0.f || sum.y != 0.f || sum.z != 0.f || sum.w != 0.f)
      red_add_v4(a.out + bh0 * D + 4 * i4,
                 make_float4(sum.x * inv_S, sum.y * inv_S, sum.z * inv_S, sum.w * inv_S));
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Launch with programmatic stream serialization: the kernel may be scheduled
// while its predecessor finishes and waits in wait_for_predecessor().
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t launch_combine(const LaunchArgs& a) {
  const int S_pow2 = next_pow2(a.S_max);
  const size_t smem = sizeof(long long) * (size_t)a.S_max + sizeof(uint32_t) * S_pow2;
  if (smem + 1024 > 48 * 1024) {  // plus a little static shared memory
    cudaError_t e = cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(combine_kernel, dim3((unsigned)a.H, (unsigned)a.B), dim3(THREADS), smem, a.stream, a, S_pow2);
}

template <typename T, int D, int GM>
static cudaError_t launch_sample_gather_g(const LaunchArgs& a) {
  const int G = a.H / a.Hkv;
  const size_t smem = sample_gather_smem<GM>(G, D);
  cudaError_t e = cudaFuncSetAttribute(sample_gather_kernel<T, D, GM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(sample_gather_kernel<T, D, GM>, dim3((unsigned)a.Hkv, (unsigned)a.groups_max, (unsigned)a.B),
                    dim3(SG_THREADS), smem, a.stream, a);
}

template <typename T, int D>
static cudaError_t launch_sample_gather_t(const LaunchArgs& a) {
  return (a.H / a.Hkv <= 4) ? launch_sample_gather_g<T, D, 4>(a) : launch_sample_gather_g<T, D, 8>(a);
}

cudaError_t launch_sample_gather(const LaunchArgs& a) {
  switch (a.dtype * 2 + (a.D == 128)) {
    case 0: return launch_sample_gather_t<bf16_t, 64>(a);
    case 1: return launch_sample_gather_t<bf16_t, 128>(a);
    case 2: return launch_sample_gather_t<fp16_t, 64>(a);
    case 3: return launch_sample_gather_t<fp16_t, 128>(a);
    case 4: return launch_sample_gather_t<float, 64>(a);
    case 5: return launch_sample_gather_t<float, 128>(a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace santa
