// santa_score.cu -- score pass (per-chunk max / exp-sum + score stash) and the
// dense split-KV comparator, for sm_103a.
//
// Score pass: "Stochastic Sparse Attention for Memory-Bound Inference",
// Sec. 2 Eq. (1) for s_n and App. O, Alg. 3 for the per-tile statistics.  One
// CTA owns a 256-key chunk of one KV head and reads each K row once for the
// whole query group; 16-byte streaming loads, fp32 dot products and a warp
// transpose-reduction put every score in one lane.  Tensor cores are not used:
// each K element feeds only G <= 8 multiply-adds, far below the tensor-core
// ridge, so the pass is bound by HBM bandwidth.
#include "santa_common.cuh"
#include "santa_launch.h"

namespace santa {

struct ChunkCtx {
  int64_t row0, nk;
  bool ok;
};

// Rows of sequence b and whether its length is within the stated bound.
__device__ __forceinline__ ChunkCtx chunk_ctx(const int64_t* kv_offsets, int64_t nk_max, int b) {
  ChunkCtx c;
  if (kv_offsets) {
    c.row0 = kv_offsets[b];
    c.nk = kv_offsets[b + 1] - c.row0;
  } else {
    c.row0 = (int64_t)b * nk_max;
    c.nk = nk_max;
  }
  c.ok = c.nk >= 1 && c.nk <= nk_max && c.row0 >= 0;
  return c;
}

template <typename T, int D>
__device__ __forceinline__ void load_scaled_q(float* qs, const T* __restrict__ q, int b, int H, int G, int kvh,
                                              float scale) {
  for (int i = threadIdx.x; i < G * D; i += THREADS) {
    const int g = i / D, e = i % D;
    qs[i] = widen_scalar<T>(q + ((int64_t)b * H + kvh * G + g) * D + e) * scale;
  }
}

template <typename T, int D>
__device__ __forceinline__ void lane_q(float (&qreg)[HP][Tile<T, D>::EPL], const float* qs, int g0, int G,
                                       int lane) {
  using TL = Tile<T, D>;
  const int sub = lane % TL::LPK;
#pragma unroll
  for (int g = 0; g < HP; ++g)
#pragma unroll
    for (int e = 0; e < TL::EPL; ++e) qreg[g][e] = (g0 + g < G) ? qs[(g0 + g) * D + sub * TL::EPL + e] : 0.f;
}

// ---------------------------------------------------------------------------
// Score pass.  grid = (chunks_max, H_kv, B), block = 256.
// ---------------------------------------------------------------------------
template <typename T, int D, int NP>
__global__ void __launch_bounds__(THREADS, 2)
score_chunks_kernel(const T* __restrict__ q, const T* __restrict__ K, const int64_t* __restrict__ kv_offsets,
                    int64_t nk_max, int H, int Hkv, float scale, float* __restrict__ stash,
                    float* __restrict__ tile_max, float* __restrict__ tile_sum, int chunks_max) {
  using TL = Tile<T, D>;
  using WS = WarpScores<T, D>;
  const int c = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = H / Hkv;
  const ChunkCtx cx = chunk_ctx(kv_offsets, nk_max, b);
  const int64_t key0 = (int64_t)c * CHUNK;
  if (!cx.ok || key0 >= cx.nk) return;   // bad metadata is flagged by the combine kernel
  const int chunk_len = (int)min((int64_t)CHUNK, cx.nk - key0);

  __shared__ float qs[SANTA_MAX_GROUP_DEV * D];
  __shared__ float red[WARPS][HP];
  __shared__ float cmax[HP];

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int wkey0 = warp * 32;
  const int nvalid = max(0, min(32, chunk_len - wkey0));
  uint4 kv[TL::ITERS][TL::NVEC];
  WS::load(K + ((cx.row0 + key0 + wkey0) * Hkv + kvh) * (int64_t)D, (int64_t)Hkv * D, nvalid, lane, kv);

  load_scaled_q<T, D>(qs, q, b, H, G, kvh, scale);
  __syncthreads();

  const int mk = WS::my_key(lane);
  const bool valid = mk < nvalid;
  const int64_t n = key0 + wkey0 + mk;

  // NP passes of HP heads over the tile; a second pass re-reads the tile (L2)
  // rather than keeping it in registers across passes.
#pragma unroll 1
  for (int pass = 0; pass < NP; ++pass) {
    const int g0 = pass * HP;
    float qreg[HP][TL::EPL];
    lane_q<T, D>(qreg, qs, g0, G, lane);
    float s[HP];
    WS::dot(kv, qreg, lane, s);
    if (pass + 1 < NP) WS::load(K + ((cx.row0 + key0 + wkey0) * Hkv + kvh) * (int64_t)D, (int64_t)Hkv * D, nvalid, lane, kv);
#pragma unroll
    for (int g = 0; g < HP; ++g) {
      if (g0 + g < G && valid) stash[((int64_t)b * H + kvh * G + g0 + g) * nk_max + n] = s[g];
      const float m = warp_max(valid ? s[g] : -INFINITY);
      if (lane == 0) red[warp][g] = m;
    }
    __syncthreads();
    if (threadIdx.x < HP) {
      float m = red[0][threadIdx.x];
#pragma unroll
      for (int w = 1; w < WARPS; ++w) m = fmaxf(m, red[w][threadIdx.x]);
      cmax[threadIdx.x] = m;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < HP; ++g) {
      const float e = warp_sum(valid ? expf(s[g] - cmax[g]) : 0.f);
      if (lane == 0) red[warp][g] = e;
    }
    __syncthreads();
    if (threadIdx.x < HP && g0 + (int)threadIdx.x < G) {
      float l = 0.f;
#pragma unroll
      for (int w = 0; w < WARPS; ++w) l += red[w][threadIdx.x];
      const int64_t idx = ((int64_t)b * H + kvh * G + g0 + threadIdx.x) * chunks_max + c;
      tile_max[idx] = cmax[threadIdx.x];
      tile_sum[idx] = l;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Dense comparator, stage 1: per chunk (m_c, l_c, O_c = sum exp(s_n - m_c) V_n).
// grid = (chunks_max, H_kv, B), block = 256.
// ---------------------------------------------------------------------------
template <typename T, int D, int NP>
__global__ void __launch_bounds__(THREADS, 2)
dense_chunks_kernel(const T* __restrict__ q, const T* __restrict__ K, const T* __restrict__ V,
                    const int64_t* __restrict__ kv_offsets, int64_t nk_max, int H, int Hkv, float scale,
                    float* __restrict__ part_m, float* __restrict__ part_l, float* __restrict__ part_o,
                    int chunks_max) {
  using TL = Tile<T, D>;
  using WS = WarpScores<T, D>;
  const int c = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = H / Hkv;
  const ChunkCtx cx = chunk_ctx(kv_offsets, nk_max, b);
  const int64_t key0 = (int64_t)c * CHUNK;
  if (!cx.ok || key0 >= cx.nk) return;
  const int chunk_len = (int)min((int64_t)CHUNK, cx.nk - key0);

  __shared__ float qs[SANTA_MAX_GROUP_DEV * D];
  __shared__ float red[WARPS][HP];
  __shared__ float cmax[HP];
  __shared__ float obuf[WARPS][HP][D];

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int slot = lane / TL::LPK, sub = lane % TL::LPK;
  const int wkey0 = warp * 32;
  const int nvalid = max(0, min(32, chunk_len - wkey0));
  const int64_t tile_off = ((cx.row0 + key0 + wkey0) * Hkv + kvh) * (int64_t)D;
  uint4 kv[TL::ITERS][TL::NVEC];
  WS::load(K + tile_off, (int64_t)Hkv * D, nvalid, lane, kv);

  load_scaled_q<T, D>(qs, q, b, H, G, kvh, scale);
  __syncthreads();

  const int mk = WS::my_key(lane);
  const bool valid = mk < nvalid;

#pragma unroll 1
  for (int pass = 0; pass < NP; ++pass) {
    const int g0 = pass * HP;
    float qreg[HP][TL::EPL];
    lane_q<T, D>(qreg, qs, g0, G, lane);
    float s[HP];
    WS::dot(kv, qreg, lane, s);
    if (pass + 1 < NP) WS::load(K + tile_off, (int64_t)Hkv * D, nvalid, lane, kv);
#pragma unroll
    for (int g = 0; g < HP; ++g) {
      const float m = warp_max(valid ? s[g] : -INFINITY);
      if (lane == 0) red[warp][g] = m;
    }
    __syncthreads();
    if (threadIdx.x < HP) {
      float m = red[0][threadIdx.x];
#pragma unroll
      for (int w = 1; w < WARPS; ++w) m = fmaxf(m, red[w][threadIdx.x]);
      cmax[threadIdx.x] = m;
    }
    __syncthreads();
    float p[HP];
#pragma unroll
    for (int g = 0; g < HP; ++g) {
      p[g] = valid ? expf(s[g] - cmax[g]) : 0.f;
      const float e = warp_sum(p[g]);
      if (lane == 0) red[warp][g] = e;
    }
    // weighted V rows of this warp's keys
    uint4 vv[TL::ITERS][TL::NVEC];
    WS::load(V + tile_off, (int64_t)Hkv * D, nvalid, lane, vv);
    float acc[HP][TL::EPL];
#pragma unroll
    for (int g = 0; g < HP; ++g)
#pragma unroll
      for (int e = 0; e < TL::EPL; ++e) acc[g][e] = 0.f;
#pragma unroll
    for (int it = 0; it < TL::ITERS; ++it) {
      float vf[TL::EPL];
#pragma unroll
      for (int w = 0; w < TL::NVEC; ++w) Elem<T>::widen(vv[it][w], vf + w * (16 / TL::ES));
      const int owner = slot * TL::LPK + it;   // lane whose key is it*KPI + slot
#pragma unroll
      for (int g = 0; g < HP; ++g) {
        const float wgt = __shfl_sync(FULL, p[g], owner);
#pragma unroll
        for (int e = 0; e < TL::EPL; ++e) acc[g][e] = fmaf(wgt, vf[e], acc[g][e]);
      }
    }
#pragma unroll
    for (int o = TL::LPK; o < 32; o <<= 1)
#pragma unroll
      for (int g = 0; g < HP; ++g)
#pragma unroll
        for (int e = 0; e < TL::EPL; ++e) acc[g][e] += __shfl_xor_sync(FULL, acc[g][e], o);
    if (slot == 0) {
#pragma unroll
      for (int g = 0; g < HP; ++g)
#pragma unroll
        for (int e = 0; e < TL::EPL; ++e) obuf[warp][g][sub * TL::EPL + e] = acc[g][e];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < HP * D; i += THREADS) {
      const int g = i / D, col = i % D;
      if (g0 + g >= G) continue;
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < WARPS; ++w) o += obuf[w][g][col];
      const int64_t bh = (int64_t)b * H + kvh * G + g0 + g;
      part_o[(bh * chunks_max + c) * D + col] = o;
    }
    if (threadIdx.x < HP && g0 + (int)threadIdx.x < G) {
      float l = 0.f;
#pragma unroll
      for (int w = 0; w < WARPS; ++w) l += red[w][threadIdx.x];
      const int64_t idx = ((int64_t)b * H + kvh * G + g0 + threadIdx.x) * chunks_max + c;
      part_m[idx] = cmax[threadIdx.x];
      part_l[idx] = l;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Dense comparator, stage 2: merge the chunk partials of one head,
// O = sum_c e^{m_c - m*} O_c / sum_c e^{m_c - m*} l_c.  grid = (H, B).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(THREADS)
dense_merge_kernel(const int64_t* __restrict__ kv_offsets, int64_t nk_max, int H, const float* __restrict__ part_m,
                   const float* __restrict__ part_l, const float* __restrict__ part_o, int chunks_max,
                   float* __restrict__ out, int* err) {
  constexpr int CPL = D / 32;  // columns per lane
  const int h = blockIdx.x, b = blockIdx.y;
  const int64_t bh = (int64_t)b * H + h;
  const ChunkCtx cx = chunk_ctx(kv_offsets, nk_max, b);
  if (!cx.ok) {
    for (int i = threadIdx.x; i < D; i += THREADS) out[bh * D + i] = 0.f;
    if (threadIdx.x == 0) flag_error(err, cx.nk < 1 ? ERR_EMPTY : ERR_NK_BOUND);
    return;
  }
  const int C = (int)((cx.nk + CHUNK - 1) / CHUNK);
  const float* pm = part_m + bh * chunks_max;
  const float* pl = part_l + bh * chunks_max;
  const float* po = part_o + bh * chunks_max * D;
  __shared__ float red[WARPS];
  __shared__ float acc_s[WARPS][D];
  __shared__ float lsum_s[WARPS];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  float m = -INFINITY;
  for (int c = threadIdx.x; c < C; c += THREADS) m = fmaxf(m, pm[c]);
  m = warp_max(m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float mstar = red[0];
#pragma unroll
  for (int w = 1; w < WARPS; ++w) mstar = fmaxf(mstar, red[w]);

  float acc[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) acc[i] = 0.f;
  float lsum = 0.f;
  for (int c = warp; c < C; c += WARPS) {
    const float f = expf(pm[c] - mstar);
    lsum += f * pl[c];
#pragma unroll
    for (int i = 0; i < CPL; ++i) acc[i] = fmaf(f, po[(int64_t)c * D + lane * CPL + i], acc[i]);
  }
#pragma unroll
  for (int i = 0; i < CPL; ++i) acc_s[warp][lane * CPL + i] = acc[i];
  if (lane == 0) lsum_s[warp] = lsum;
  __syncthreads();
  if (threadIdx.x < D) {
    float o = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      o += acc_s[w][threadIdx.x];
      l += lsum_s[w];
    }
    out[bh * D + threadIdx.x] = o / l;
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
template <typename T, int D>
static cudaError_t launch_score_t(const LaunchArgs& a) {
  dim3 grid((unsigned)a.chunks_max, (unsigned)a.Hkv, (unsigned)a.B);
  auto kern = (a.H / a.Hkv <= HP) ? score_chunks_kernel<T, D, 1> : score_chunks_kernel<T, D, 2>;
  kern<<<grid, THREADS, 0, a.stream>>>((const T*)a.q, (const T*)a.K, a.kv_offsets, a.nk_max, a.H, a.Hkv,
                                       a.scale, a.stash, a.tile_max, a.tile_sum, a.chunks_max);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch_dense_t(const LaunchArgs& a) {
  dim3 grid((unsigned)a.chunks_max, (unsigned)a.Hkv, (unsigned)a.B);
  auto kern = (a.H / a.Hkv <= HP) ? dense_chunks_kernel<T, D, 1> : dense_chunks_kernel<T, D, 2>;
  kern<<<grid, THREADS, 0, a.stream>>>((const T*)a.q, (const T*)a.K, (const T*)a.V, a.kv_offsets, a.nk_max,
                                       a.H, a.Hkv, a.scale, a.tile_max, a.tile_sum, a.part_o, a.chunks_max);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dense_merge_kernel<D><<<dim3((unsigned)a.H, (unsigned)a.B), THREADS, 0, a.stream>>>(
      a.kv_offsets, a.nk_max, a.H, a.tile_max, a.tile_sum, a.part_o, a.chunks_max, a.out, a.err);
  return cudaGetLastError();
}

#define SANTA_DISPATCH(FN, a)                                                     \
  switch ((a).dtype * 2 + ((a).D == 128)) {                                       \
    case 0: return FN<bf16_t, 64>(a);                                             \
    case 1: return FN<bf16_t, 128>(a);                                            \
    case 2: return FN<fp16_t, 64>(a);                                             \
    case 3: return FN<fp16_t, 128>(a);                                            \
    case 4: return FN<float, 64>(a);                                              \
    case 5: return FN<float, 128>(a);                                             \
    default: return cudaErrorInvalidValue;                                        \
  }

cudaError_t launch_score(const LaunchArgs& a) { SANTA_DISPATCH(launch_score_t, a) }
cudaError_t launch_dense(const LaunchArgs& a) { SANTA_DISPATCH(launch_dense_t, a) }

}  // namespace santa
