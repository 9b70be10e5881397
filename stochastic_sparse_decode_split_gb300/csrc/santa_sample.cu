// santa_sample.cu -- cross-chunk combine, Philox thresholds, inverse-CDF
// sampling and the GQA-deduplicated V gather-add, for sm_103a.
//
// "Stochastic Sparse Attention for Memory-Bound Inference":
//   combine   m* = max_t m_t, W_t = e^{m_t - m*} l_t, Z = sum_t W_t   (App. O, Alg. 4, lines 2-3)
//   samplers  i.i.d. / stratified / systematic thresholds            (Sec. 2.1; Eq. 4)
//   inverse CDF, left-closed: F(n-1) <= t < F(n)                     (App. A.4)
//   gather    O_h = (1/S) sum_n c_{h,n} V_n over the union of rows
//             drawn by the heads of a KV group                        (Eq. 4, Fig. 1; App. O, Alg. 5)
//
// Difference from the pages' kernels: Alg. 4 rounds per-tile budgets by
// largest remainder and then samples each tile systematically on its own.
// Here every head's S thresholds are placed globally (prefix of chunk masses)
// and resolved inside the chunk that holds them, which reproduces the global
// i.i.d. / stratified / systematic estimators exactly.
#include "santa_common.cuh"
#include "santa_launch.h"

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

// Chunk masses are summed as fixed-point integers (units of 2^-40 of the head
// max's own mass): integer prefix sums are exact in any association, so the
// chunk prefix is monotone however the block scan groups the additions.
constexpr double MASS_ONE = 1099511627776.0;  // 2^40
__device__ __forceinline__ long long mass_fixed(float w) { return __double2ll_rn((double)w * MASS_ONE); }

// Inclusive block-wide scan of one int64 per thread (THREADS threads).
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
// Combine + thresholds.  grid = (H, B), block = 256.
// dynamic smem: prefix double[chunks_max + 1] | theta double[S_pow2]
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(THREADS)
combine_kernel(LaunchArgs a, int S_pow2) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  double* P = reinterpret_cast<double*>(smem_raw);
  double* theta = P + (a.chunks_max + 1);
  __shared__ float red[WARPS];
  __shared__ long long warp_tot[WARPS];

  const int h = blockIdx.x, b = blockIdx.y;
  const int G = a.H / a.Hkv;
  const int64_t bh = (int64_t)b * a.H + h;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const HeadCtx hc = head_ctx(a, b);

  if (h % G == 0 && tid == 0) a.counters[b * a.Hkv + h / G] = 0u;  // hand-off counter of the gather
  if (hc.err) {
    if (tid == 0 && h == 0) flag_error(a.err, hc.err);
    if (a.sample_idx)
      for (int j = tid; j < a.S_max; j += THREADS) a.sample_idx[bh * a.S_max + j] = -1;
    return;
  }
  const int C = (int)((hc.nk + CHUNK - 1) / CHUNK);
  const int S = hc.S;
  const float* tmax = a.tile_max + bh * a.chunks_max;
  const float* tsum = a.tile_sum + bh * a.chunks_max;

  // m* = max over chunks
  float m = -INFINITY;
  for (int c = tid; c < C; c += THREADS) m = fmaxf(m, tmax[c]);
  m = warp_max(m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float mstar = red[0];
#pragma unroll
  for (int w = 1; w < WARPS; ++w) mstar = fmaxf(mstar, red[w]);

  // exclusive prefix of chunk masses W_c = e^{m_c - m*} l_c, each thread a contiguous run
  const int per = (C + THREADS - 1) / THREADS;
  const int c_lo = min(C, tid * per), c_hi = min(C, c_lo + per);
  long long local = 0;
  for (int c = c_lo; c < c_hi; ++c) local += mass_fixed(expf(tmax[c] - mstar) * tsum[c]);
  const long long incl = block_inclusive_scan(local, warp_tot);
  long long run = incl - local;
  for (int c = c_lo; c < c_hi; ++c) {
    P[c] = (double)run * (1.0 / MASS_ONE);
    run += mass_fixed(expf(tmax[c] - mstar) * tsum[c]);
  }
  if (tid == THREADS - 1) P[C] = (double)incl * (1.0 / MASS_ONE);
  __syncthreads();
  const double Z = P[C];

  // thresholds t_j (Sec. 2.1) scaled to mass units: theta_j = t_j * Z
  const uint32_t k0 = (uint32_t)a.seed, k1 = (uint32_t)(a.seed >> 32);
  if (a.variant == 2) {  // systematic: one offset
    double u;
    if (a.uniforms) u = a.uniforms[bh * a.S_max];
    else u = word_to_unit(philox4x32_10(make_uint4(0u, (uint32_t)h, (uint32_t)b, a.step), k0, k1).x);
    for (int j = tid; j < S; j += THREADS) theta[j] = (((double)j + u) / (double)S) * Z;
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
        const double t = (a.variant == 1) ? ((double)j + u4[r]) / (double)S : u4[r];
        theta[j] = t * Z;
      }
    }
  }
  if (a.variant == 0) {  // i.i.d. draws are unordered: sort them (bitonic, +inf padding)
    for (int j = S + tid; j < S_pow2; j += THREADS) theta[j] = INFINITY;
    __syncthreads();
    for (int k = 2; k <= S_pow2; k <<= 1) {
      for (int jj = k >> 1; jj > 0; jj >>= 1) {
        for (int i = tid; i < S_pow2; i += THREADS) {
          const int ixj = i ^ jj;
          if (ixj > i) {
            const double x = theta[i], y = theta[ixj];
            const bool up = (i & k) == 0;
            if ((x > y) == up) {
              theta[i] = y;
              theta[ixj] = x;
            }
          }
        }
        __syncthreads();
      }
    }
  }
  __syncthreads();

  // first threshold of every chunk: jstart[c] = #{j : theta_j < P_c}
  for (int c = tid; c <= C; c += THREADS) {
    const double pc = P[c];
    int lo = 0, hi = S;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (theta[mid] < pc) lo = mid + 1;
      else hi = mid;
    }
    a.jstart[bh * (a.chunks_max + 1) + c] = lo;
    a.prefix[bh * (a.chunks_max + 1) + c] = pc;
  }
  for (int j = tid; j < S; j += THREADS) a.thresh[bh * a.S_max + j] = theta[j];
  if (a.sample_idx)
    for (int j = S + tid; j < a.S_max; j += THREADS) a.sample_idx[bh * a.S_max + j] = -1;
  if (tid == 0) a.head_max[bh] = mstar;
}

// ---------------------------------------------------------------------------
// Sample + gather.  grid = (groups_max, H_kv, B), block = 256; warp w owns
// chunk blockIdx.x * 8 + w.  dynamic smem per warp:
//   pref double[CHUNK] | cnt uint32[G][CHUNK] | rows int32[CHUNK];
// then wbuf float[WARPS][G][D].
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(THREADS)
sample_gather_kernel(LaunchArgs a) {
  using TL = Tile<T, D>;
  constexpr int GM = SANTA_MAX_GROUP_DEV;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int G = a.H / a.Hkv;
  const int grp = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const size_t warp_bytes = (size_t)CHUNK * (8 + 4 * G + 4);
  unsigned char* wbase = smem_raw + warp * warp_bytes;
  double* pref = reinterpret_cast<double*>(wbase);
  unsigned* cnt = reinterpret_cast<unsigned*>(wbase + CHUNK * 8);
  int* rows = reinterpret_cast<int*>(wbase + CHUNK * (8 + 4 * G));
  float* wbuf = reinterpret_cast<float*>(smem_raw + WARPS * warp_bytes);
  __shared__ double lane_tot[WARPS][32];
  __shared__ int s_last;

  const HeadCtx hc = head_ctx(a, b);
  if (hc.err) {
    if (grp == 0)
      for (int i = tid; i < G * D; i += THREADS) a.out[((int64_t)b * a.H + kvh * G) * D + i] = 0.f;
    return;
  }
  const int C = (int)((hc.nk + CHUNK - 1) / CHUNK);
  const int NG = (C + GROUP_CHUNKS - 1) / GROUP_CHUNKS;
  if (grp >= NG) return;
  const int c = grp * GROUP_CHUNKS + warp;
  const bool active = c < C;
  const int len = active ? (int)min((int64_t)CHUNK, hc.nk - (int64_t)c * CHUNK) : 0;

  for (int i = lane; i < G * CHUNK; i += 32) cnt[i] = 0u;

  // thresholds of every head that fall in this chunk, and the stash rows they need
  int j0[GM], j1[GM];
  float sv[GM][8];
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    j0[g] = j1[g] = 0;
    if (g < G && active) {
      const int64_t bh = (int64_t)b * a.H + kvh * G + g;
      const int32_t* js = a.jstart + bh * (a.chunks_max + 1) + c;
      j0[g] = js[0];
      j1[g] = js[1];
      if (j1[g] > j0[g]) {
        const float* st = a.stash + bh * a.nk_max + (int64_t)c * CHUNK;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int k = lane * 8 + r;
          sv[g][r] = (k < len) ? st[k] : -INFINITY;
        }
      }
    }
  }
  __syncwarp();

#pragma unroll
  for (int g = 0; g < GM; ++g) {
    if (g >= G || j1[g] <= j0[g]) continue;  // warp-uniform
    const int64_t bh = (int64_t)b * a.H + kvh * G + g;
    const float mstar = a.head_max[bh];
    // in-chunk masses relative to the head max and their inclusive prefix (fp64)
    double loc[8];
    double run = 0.0;
    int lastpos = -1;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float w = (lane * 8 + r < len) ? expf(sv[g][r] - mstar) : 0.f;
      run += (double)w;
      loc[r] = run;
      if (w > 0.f) lastpos = lane * 8 + r;
    }
    lane_tot[warp][lane] = run;
    __syncwarp();
    double excl = 0.0;
    for (int l = 0; l < lane; ++l) excl += lane_tot[warp][l];  // serial: keeps the prefix monotone
#pragma unroll
    for (int r = 0; r < 8; ++r) pref[lane * 8 + r] = excl + loc[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lastpos = max(lastpos, __shfl_xor_sync(FULL, lastpos, o));
    __syncwarp();
    const double base = a.prefix[bh * (a.chunks_max + 1) + c];
    for (int j = j0[g] + lane; j < j1[g]; j += 32) {
      const double x = a.thresh[bh * a.S_max + j] - base;
      int lo = 0, hi = len;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (pref[mid] <= x) lo = mid + 1;
        else hi = mid;
      }
      const int idx = (lo < len) ? lo : max(lastpos, 0);  // rounding past the chunk mass
      atomicAdd(&cnt[g * CHUNK + idx], 1u);
      if (a.sample_idx) a.sample_idx[bh * a.S_max + j] = c * CHUNK + idx;
    }
    __syncwarp();
  }

  // union of the rows drawn by any head of the group (each V row read once)
  int nrows = 0;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int k = r * 32 + lane;
    bool any = false;
    for (int g = 0; g < G; ++g) any |= cnt[g * CHUNK + k] != 0u;
    const unsigned bal = __ballot_sync(FULL, any);
    if (any) rows[nrows + __popc(bal & ((1u << lane) - 1u))] = k;
    nrows += __popc(bal);
  }
  __syncwarp();

  // count-weighted gather-and-add, fp32 accumulation
  const int slot = lane / TL::LPK, sub = lane % TL::LPK;
  float acc[GM][TL::EPL];
#pragma unroll
  for (int g = 0; g < GM; ++g)
#pragma unroll
    for (int e = 0; e < TL::EPL; ++e) acc[g][e] = 0.f;
  const T* Vbase = reinterpret_cast<const T*>(a.V) + ((hc.row0 + (int64_t)c * CHUNK) * a.Hkv + kvh) * (int64_t)D;
  constexpr int UNR = 4;
  for (int i0 = slot; i0 < nrows; i0 += UNR * TL::KPI) {
    uint4 vv[UNR][TL::NVEC];
    int key[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int i = i0 + u * TL::KPI;
      key[u] = (i < nrows) ? rows[i] : -1;
#pragma unroll
      for (int v = 0; v < TL::NVEC; ++v)
        vv[u][v] = (key[u] >= 0)
                       ? ld_stream(Vbase + (int64_t)key[u] * a.Hkv * D + sub * TL::EPL + v * (16 / TL::ES))
                       : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      if (key[u] < 0) continue;
      float vf[TL::EPL];
#pragma unroll
      for (int v = 0; v < TL::NVEC; ++v) Elem<T>::widen(vv[u][v], vf + v * (16 / TL::ES));
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        if (g >= G) break;
        const float cg = (float)cnt[g * CHUNK + key[u]];
#pragma unroll
        for (int e = 0; e < TL::EPL; ++e) acc[g][e] = fmaf(cg, vf[e], acc[g][e]);
      }
    }
  }
#pragma unroll
  for (int o = TL::LPK; o < 32; o <<= 1)
#pragma unroll
    for (int g = 0; g < GM; ++g)
#pragma unroll
      for (int e = 0; e < TL::EPL; ++e) acc[g][e] += __shfl_xor_sync(FULL, acc[g][e], o);
  if (slot == 0) {
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      if (g >= G) break;
#pragma unroll
      for (int e = 0; e < TL::EPL; ++e) wbuf[(warp * G + g) * D + sub * TL::EPL + e] = acc[g][e];
    }
  }
  __syncthreads();

  // this CTA's partial sum per head, then the last CTA of the group reduces
  // all partials in a fixed order (deterministic) and applies 1/S.
  const int64_t bh0 = (int64_t)b * a.H + kvh * G;
  for (int i = tid; i < G * D; i += THREADS) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) s += wbuf[w * G * D + i];
    const int g = i / D, col = i % D;
    a.part_o[((bh0 + g) * a.groups_max + grp) * D + col] = s;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&a.counters[b * a.Hkv + kvh], 1u) == (unsigned)(NG - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float inv_S = 1.0f / (float)hc.S;
  for (int i = tid; i < G * D; i += THREADS) {
    const int g = i / D, col = i % D;
    const float* src = a.part_o + (bh0 + g) * a.groups_max * D + col;
    float s = 0.f;
    for (int q = 0; q < NG; ++q) s += __ldcg(src + (int64_t)q * D);
    a.out[(bh0 + g) * D + col] = s * inv_S;
  }
  if (tid == 0) a.counters[b * a.Hkv + kvh] = 0u;
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

cudaError_t launch_combine(const LaunchArgs& a) {
  const int S_pow2 = next_pow2(a.S_max);
  const size_t smem = sizeof(double) * ((size_t)a.chunks_max + 1 + (size_t)S_pow2);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  combine_kernel<<<dim3((unsigned)a.H, (unsigned)a.B), THREADS, smem, a.stream>>>(a, S_pow2);
  return cudaGetLastError();
}

size_t sample_gather_smem(int G, int D) {
  return (size_t)WARPS * CHUNK * (8 + 4 * G + 4) + (size_t)WARPS * G * D * sizeof(float);
}

template <typename T, int D>
static cudaError_t launch_sample_gather_t(const LaunchArgs& a) {
  const int G = a.H / a.Hkv;
  const size_t smem = sample_gather_smem(G, D);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(sample_gather_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  sample_gather_kernel<T, D><<<dim3((unsigned)a.groups_max, (unsigned)a.Hkv, (unsigned)a.B), THREADS, smem,
                               a.stream>>>(a);
  return cudaGetLastError();
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
