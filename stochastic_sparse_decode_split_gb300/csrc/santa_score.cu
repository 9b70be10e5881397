// santa_score.cu -- score pass (per-chunk max / exp-sum + score stash) and the
// dense split-KV comparator, for sm_103a.
//
// Score pass: "Stochastic Sparse Attention for Memory-Bound Inference",
// Sec. 2 Eq. (1) for s_n and App. O, Alg. 3 for the per-tile statistics.
#include <algorithm>

#include "santa_common.cuh"
#include "santa_launch.h"
#include "santa_stream.cuh"

namespace santa {

constexpr int SC_WARPS = 4;                   // warps per dense chunk CTA
constexpr int SC_THREADS = SC_WARPS * 32;

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

// q of the KV head's query group, widened (unscaled; bf16/fp16 values are exact in fp32).
template <typename T, int D>
__device__ __forceinline__ void load_group_q(float* qs, const T* __restrict__ q, int b, int H, int G, int kvh) {
  for (int i = threadIdx.x; i < G * D; i += SC_THREADS)
    qs[i] = widen_scalar<T>(q + ((int64_t)b * H + kvh * G) * D + i);
}

// Scores of the lane's two keys (tile rows r and r + 32) for heads g0..g0+HP-1,
// CUDA cores (dense comparator).
template <typename T, int D>
__device__ __forceinline__ void lane_scores(uint32_t kbase, const float* qs, int g0, int G, int r, float scale,
                                            float (&s)[2][HP]) {
  using R = Rows<T, D>;
  constexpr int NP2 = R::EPC / 2;  // fp32 pairs per chunk
  f2x acc[2][HP][2];
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int g = 0; g < HP; ++g) acc[k][g][0] = acc[k][g][1] = 0ull;
  const uint32_t rowA = kbase + r * R::ROWB, rowB = kbase + (r + 32) * R::ROWB;
#pragma unroll
  for (int c = 0; c < R::NCH; ++c) {
    f2x pa[NP2], pb[NP2];
    Pairs<T>::get(lds128(rowA + swz(r, c) * 16), pa);
    Pairs<T>::get(lds128(rowB + swz(r + 32, c) * 16), pb);
#pragma unroll
    for (int g = 0; g < HP; ++g) {
      if (g0 + g < G) {
        const f2x* qp = reinterpret_cast<const f2x*>(qs + (g0 + g) * D + c * R::EPC);
#pragma unroll
        for (int p = 0; p < NP2; ++p) {
          const f2x qq = qp[p];
          acc[0][g][c & 1] = ffma2(qq, pa[p], acc[0][g][c & 1]);
          acc[1][g][c & 1] = ffma2(qq, pb[p], acc[1][g][c & 1]);
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int g = 0; g < HP; ++g) {
      const float2 a0 = unpack2(acc[k][g][0]), a1 = unpack2(acc[k][g][1]);
      s[k][g] = ((a0.x + a1.x) + (a0.y + a1.y)) * scale;
    }
}

// Max over the CTA's keys of one value per lane, for HP heads at once.
__device__ __forceinline__ void cta_max(float (&v)[HP], float (*red)[HP], float* out) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
#pragma unroll
  for (int g = 0; g < HP; ++g) {
    const float m = warp_max(v[g]);
    if (lane == 0) red[warp][g] = m;
  }
  __syncthreads();
  if (threadIdx.x < HP) {
    float m = red[0][threadIdx.x];
#pragma unroll
    for (int w = 1; w < SC_WARPS; ++w) m = fmaxf(m, red[w][threadIdx.x]);
    out[threadIdx.x] = m;
  }
  __syncthreads();
}

template <typename T, int D>
constexpr size_t score_smem_bytes() {
  return (size_t)CHUNK * Rows<T, D>::ROWB + (size_t)SANTA_MAX_GROUP_DEV * D * sizeof(float);
}

// Scores of one key (tile row r, at row_addr) for heads g0..g0+HP-1, two fp32
// pair accumulators per head (even / odd 16-byte chunks); q read through L1.
template <typename T, int D>
__device__ __forceinline__ void key_scores(uint32_t row_addr, int r, const float* qs, int g0, int G, float scale,
                                           float (&s)[HP]) {
  using R = Rows<T, D>;
  constexpr int NP2 = R::EPC / 2;  // fp32 pairs per 16-byte chunk
  f2x acc[HP][2];
#pragma unroll
  for (int g = 0; g < HP; ++g) acc[g][0] = acc[g][1] = 0ull;
#pragma unroll
  for (int c = 0; c < R::NCH; ++c) {
    f2x pk[NP2];
    Pairs<T>::get(lds128(row_addr + swz(r, c) * 16), pk);
#pragma unroll
    for (int g = 0; g < HP; ++g) {
      if (g0 + g < G) {
        const ulonglong2* qp = reinterpret_cast<const ulonglong2*>(qs + (g0 + g) * D + c * R::EPC);
#pragma unroll
        for (int p = 0; p < NP2 / 2; ++p) {
          const ulonglong2 qq = qp[p];
          acc[g][c & 1] = ffma2(qq.x, pk[2 * p], acc[g][c & 1]);
          acc[g][c & 1] = ffma2(qq.y, pk[2 * p + 1], acc[g][c & 1]);
        }
      }
    }
  }
#pragma unroll
  for (int g = 0; g < HP; ++g) {
    const float2 a0 = unpack2(acc[g][0]), a1 = unpack2(acc[g][1]);
    s[g] = ((a0.x + a1.x) + (a0.y + a1.y)) * scale;
  }
}

// ---------------------------------------------------------------------------
// Score pass, streaming.  One 512-thread CTA per SM walks work units
// u = blockIdx.x, blockIdx.x + gridDim.x, ...  A unit is a block of R*32 key
// rows x W KV heads of one sequence, with W = min(H_kv, 8) (a power of two
// dividing H_kv) and R = 8 / W, i.e. eight (32 keys, one KV head) tasks; two
// warps share a task, one 16-key half each.  When W = H_kv a unit is one
// contiguous span of the cache (64 KiB for 8 KV heads x 128 dims x bf16), so
// the HBM stream is sequential.  A 3-stage cp.async ring keeps two units in
// flight while the third is scored.  Each warp writes the statistics of its
// 16-key chunk (max, sum of exp(s - max)) directly: no block reduction.  One
// __syncthreads per unit.
//
// 16-bit inputs: a warp's scores are a [16 keys x d] . [d x 8 heads] product,
// computed with mma.m16n8k16 (bf16 / fp16 products are exact in fp32; fp32
// accumulation): K fragments by ldmatrix from the swizzled tile, q fragments
// from the raw query bits (L1-resident), heads beyond the group are zero.  A
// CUDA-core formulation needs one widen and G fused multiply-adds per K
// element, which at HBM rate would take most of the SMs' issue capacity; the
// tensor-core tile needs ~2 instructions per 16 keys x 16 dimensions.  fp32
// inputs use the CUDA-core path (one key per lane).
// ---------------------------------------------------------------------------
constexpr int UNIT_TASKS = 8;                // (32 keys x 1 KV head) tasks per unit
constexpr int ST_WARPS = 2 * UNIT_TASKS;     // one warp per 16-key half of a task
constexpr int ST_THREADS = ST_WARPS * 32;

template <typename T, int D>
constexpr uint32_t unit_bytes() { return (uint32_t)UNIT_TASKS * 32 * Rows<T, D>::ROWB; }
// Ring depth: three 64 KiB stages for 16-bit rows of 128 elements; a single
// stage when a unit is 128 KiB (fp32 rows of 128 elements).
template <typename T, int D>
constexpr int stream_stages() {
  return (size_t)unit_bytes<T, D>() * STAGES <= 200 * 1024 ? STAGES : 1;
}
template <typename T, int D>
constexpr size_t stream_smem_bytes() {
  return (size_t)stream_stages<T, D>() * unit_bytes<T, D>();
}

__device__ __forceinline__ uint32_t ldg32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

template <typename T, int D, int NP>
__global__ void __launch_bounds__(ST_THREADS, 1)
score_stream_kernel(const T* __restrict__ q, const T* __restrict__ K, const int64_t* __restrict__ kv_offsets,
                    int64_t nk_max, int B, int H, int Hkv, int W, float scale, float* __restrict__ stash,
                    float* __restrict__ sub_max, float* __restrict__ sub_sum, int subs_max,
                    float* __restrict__ out) {
  using R = Rows<T, D>;
  constexpr bool TC = sizeof(T) == 2;
  constexpr int NS = stream_stages<T, D>();
  constexpr uint32_t UB = unit_bytes<T, D>();
  constexpr int HCH = R::NCH;                    // 16-byte chunks of one head's row slice
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t sbase = smem_addr(smem);
  const int G = H / Hkv;
  const int RB = UNIT_TASKS / W;                 // 32-key blocks per unit
  const int unit_rows = 32 * RB;
  const uint32_t urow_bytes = (uint32_t)W * R::ROWB;
  const int n_hg = Hkv / W;
  const int n_kb = (int)((nk_max + unit_rows - 1) / unit_rows);
  const int n_units = B * n_kb * n_hg;
  const int n_mine = (int)blockIdx.x < n_units ? (n_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int task = warp >> 1, half = warp & 1;
  const int wkb = task / W, wkv = task % W;      // this warp's key block and KV head within the unit
  const int kr0 = wkb * 32 + half * 16;          // first unit row of this warp's 16 keys

  struct Unit {
    int b, hg, kb, len;
    int64_t row0;
  };
  __shared__ Unit meta[NS];                       // decoded units of the ring stages
  auto decode = [&](int k) {
    Unit U;
    const int u = (int)blockIdx.x + k * (int)gridDim.x;
    U.hg = u % n_hg;
    const int t = u / n_hg;
    U.kb = t % n_kb;
    U.b = t / n_kb;
    const ChunkCtx cx = chunk_ctx(kv_offsets, nk_max, U.b);
    const int64_t key0 = (int64_t)U.kb * unit_rows;
    U.row0 = cx.row0;
    U.len = (cx.ok && key0 < cx.nk) ? (int)min((int64_t)unit_rows, cx.nk - key0) : 0;
    return U;
  };
  // Copy pattern: thread t always copies 16-byte column cc of unit rows
  // rr0, rr0 + RS, ...; addresses advance by constant strides.
  const int uch = W * HCH;                        // 16-byte chunks per unit row
  const int RS = ST_THREADS / uch > 0 ? ST_THREADS / uch : 1;
  const int cc = threadIdx.x % uch, rr0 = threadIdx.x / uch;
  const bool copier = rr0 < RS;
  const int64_t gstride = (int64_t)RS * Hkv * D;  // elements between this thread's rows
  // one commit group per unit (empty when there is nothing to copy)
  auto issue = [&](int k) {
    if (k < n_mine) {
      const Unit U = decode(k);
      if (threadIdx.x == 0) meta[k % NS] = U;
      if (U.len > 0 && copier) {
        const T* src = K + ((U.row0 + (int64_t)U.kb * unit_rows + rr0) * Hkv + U.hg * W) * (int64_t)D + cc * R::EPC;
        uint32_t dst = sbase + (uint32_t)(k % NS) * UB + rr0 * urow_bytes + (uint32_t)(cc & ~7) * 16;
        if (U.len == unit_rows) {
          for (int r = rr0; r < unit_rows; r += RS, src += gstride, dst += RS * urow_bytes)
            cp_async16(dst + (uint32_t)((cc ^ r) & 7) * 16, src);
        } else {
          for (int r = rr0; r < U.len; r += RS, src += gstride, dst += RS * urow_bytes)
            cp_async16(dst + (uint32_t)((cc ^ r) & 7) * 16, src);
        }
      }
    }
    cp_async_commit();
  };

  for (int s = 0; s + 1 < NS; ++s) issue(s);  // NS - 1 units ahead
  allow_dependents();  // the next stage may launch now; it waits for this grid before reading
  if (out) {           // the sampler accumulates into out: clear it
    const int64_t n4 = (int64_t)B * H * D / 4;
    for (int64_t i = (int64_t)blockIdx.x * ST_THREADS + threadIdx.x; i < n4; i += (int64_t)gridDim.x * ST_THREADS)
      reinterpret_cast<float4*>(out)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  uint32_t bq[D / 16][2];                         // q fragments (16-bit path) of the current sequence
  int bq_b = -1, bq_kvh = -1;
  for (int k = 0; k < n_mine; ++k) {
    if constexpr (NS == 1) issue(k);
    if constexpr (NS >= 3) cp_async_wait<1>();   // unit k has landed (unit k+1 may be in flight)
    else cp_async_wait<0>();
    __syncthreads();                      // every thread's copies visible; unit k-1 fully consumed
    const Unit U = meta[k % NS];
    if constexpr (NS >= 2) issue(k + NS - 1);  // refill the stage unit k-1 used
    const int kvh = U.hg * W + wkv;
    const int64_t bh0 = (int64_t)U.b * H + kvh * G;
    const T* qg = q + bh0 * D;                  // this warp's query group
    if (U.len > kr0) {                          // this warp's 16-key statistics chunk has keys
      const int sc = U.kb * (unit_rows / SUB) + kr0 / SUB;
      const int64_t key_base = (int64_t)U.kb * unit_rows + kr0;
      const uint32_t tile = sbase + (uint32_t)(k % NS) * UB;
      if constexpr (TC) {
        const int g8 = lane >> 2, t4 = lane & 3;
        if (U.b != bq_b || kvh != bq_kvh) {     // q fragments change only with the sequence / head group
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const T* qp = qg + g8 * D + ks * 16 + t4 * 2;
            bq[ks][0] = (g8 < G) ? ldg32(qp) : 0u;
            bq[ks][1] = (g8 < G) ? ldg32(qp + 8) : 0u;
          }
          bq_b = U.b;
          bq_kvh = kvh;
        }
        // ---- tensor-core tile: 16 keys x 8 heads ----
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int row = kr0 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const uint32_t rbase = tile + row * urow_bytes;
        const int cbase = wkv * HCH + (lane >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t a[4];
          ldmatrix_x4(rbase + swz(row, cbase + ks * 2) * 16, a);
          Mma<T>::run(acc, a, bq[ks][0], bq[ks][1]);
        }
        // lane holds keys g8 and g8 + 8 of the 16 for heads 2*t4 and 2*t4 + 1
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int head = 2 * t4 + hh;
          const float s0 = acc[hh] * scale, s1 = acc[2 + hh] * scale;
          const bool ok0 = kr0 + g8 < U.len, ok1 = kr0 + g8 + 8 < U.len;
          if (head < G) {
            float* sp = stash + (bh0 + head) * nk_max + key_base + g8;
            if (ok0) sp[0] = s0;
            if (ok1) sp[8] = s1;
          }
          float m = fmaxf(ok0 ? s0 : -INFINITY, ok1 ? s1 : -INFINITY);
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
          float l = (ok0 ? fast_exp(s0 - m) : 0.f) + (ok1 ? fast_exp(s1 - m) : 0.f);
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(FULL, l, o);
          if (g8 == 0 && head < G) {
            sub_max[(bh0 + head) * subs_max + sc] = m;
            sub_sum[(bh0 + head) * subs_max + sc] = l;
          }
        }
      } else {
        // ---- CUDA-core path (fp32 inputs): one key per lane, lanes 0..15 ----
        const int r = kr0 + (lane & 15);
        const bool valid = lane < 16 && r < U.len;
        const float* qk = reinterpret_cast<const float*>(qg);
        const uint32_t row_addr = tile + r * urow_bytes + (uint32_t)wkv * HCH * 16;
#pragma unroll 1
        for (int pass = 0; pass < NP; ++pass) {
          const int g0 = pass * HP;
          float s[HP];
          key_scores<T, D>(row_addr, r, qk, g0, G, scale, s);
#pragma unroll
          for (int g = 0; g < HP; ++g) {
            if (g0 + g < G) {
              const int64_t bh = bh0 + g0 + g;
              if (valid) stash[bh * nk_max + key_base + lane] = s[g];
              const float m = warp_max(valid ? s[g] : -INFINITY);
              const float l = warp_sum(valid ? fast_exp(s[g] - m) : 0.f);
              if (lane == 0) {
                sub_max[bh * subs_max + sc] = m;
                sub_sum[bh * subs_max + sc] = l;
              }
            }
          }
        }
      }
    }
    if constexpr (NS == 1) __syncthreads();  // the single stage is refilled next iteration
  }
}

// ---------------------------------------------------------------------------
// Dense comparator, stage 1: per chunk (m_c, l_c, O_c = sum exp(s_n - m_c) V_n).
// Scores as in the score pass; then the V rows of the chunk are staged into the
// same shared memory and every lane accumulates D/32 output columns for all
// heads.  grid = (H_kv, chunks_max, B), block = 128.
// ---------------------------------------------------------------------------
template <typename T, int D>
constexpr size_t dense_smem_bytes() {
  return score_smem_bytes<T, D>() + (size_t)CHUNK * SANTA_MAX_GROUP_DEV * sizeof(float) +
         (size_t)SC_WARPS * SANTA_MAX_GROUP_DEV * D * sizeof(float);
}

template <typename T, int D, int NP>
__global__ void __launch_bounds__(SC_THREADS, 2)
dense_chunks_kernel(const T* __restrict__ q, const T* __restrict__ K, const T* __restrict__ V,
                    const int64_t* __restrict__ kv_offsets, int64_t nk_max, int H, int Hkv, float scale,
                    float* __restrict__ part_m, float* __restrict__ part_l, float* __restrict__ part_o,
                    int chunks_max) {
  using R = Rows<T, D>;
  constexpr int GM = SANTA_MAX_GROUP_DEV;
  constexpr int CPL = D / 32;                  // output columns per lane
  extern __shared__ __align__(128) unsigned char smem[];
  const int kvh = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
  const int G = H / Hkv;
  const ChunkCtx cx = chunk_ctx(kv_offsets, nk_max, b);
  const int64_t key0 = (int64_t)c * CHUNK;
  if (!cx.ok || key0 >= cx.nk) return;
  const int len = (int)min((int64_t)CHUNK, cx.nk - key0);

  const uint32_t kbase = smem_addr(smem);
  float* qs = reinterpret_cast<float*>(smem + CHUNK * R::ROWB);
  float* pS = qs + GM * D;                     // [CHUNK][GM] softmax numerators
  float* obuf = pS + CHUNK * GM;               // [SC_WARPS][GM][D]
  __shared__ float red[SC_WARPS][HP];
  __shared__ float cmax[HP];

  const int64_t tile_off = ((cx.row0 + key0) * Hkv + kvh) * (int64_t)D;
  stage_rows<T, D, SC_THREADS>(kbase, K + tile_off, (int64_t)Hkv * D, len);
  // start the chunk's V rows towards L2 while its K rows are scored, so that
  // their staging below waits for L2 rather than HBM
  {
    constexpr int LINES = (R::ROWB + 127) / 128;   // 128-byte lines per row
    const unsigned char* vt = reinterpret_cast<const unsigned char*>(V + tile_off);
    for (int i = threadIdx.x; i < len * LINES; i += SC_THREADS)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(vt + (int64_t)(i / LINES) * Hkv * R::ROWB + (i % LINES) * 128));
  }
  load_group_q<T, D>(qs, q, b, H, G, kvh);
  cp_async_wait_all();
  __syncthreads();

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int r = warp * 64 + lane;
  const bool va = r < len, vb = r + 32 < len;

#pragma unroll 1
  for (int pass = 0; pass < NP; ++pass) {
    const int g0 = pass * HP;
    float s[2][HP];
    lane_scores<T, D>(kbase, qs, g0, G, r, scale, s);
    float m[HP];
#pragma unroll
    for (int g = 0; g < HP; ++g) m[g] = fmaxf(va ? s[0][g] : -INFINITY, vb ? s[1][g] : -INFINITY);
    cta_max(m, red, cmax);
    float e[HP];
#pragma unroll
    for (int g = 0; g < HP; ++g) {
      const float pa = va ? expf(s[0][g] - cmax[g]) : 0.f, pb = vb ? expf(s[1][g] - cmax[g]) : 0.f;
      if (g0 + g < GM) {
        pS[r * GM + g0 + g] = pa;
        pS[(r + 32) * GM + g0 + g] = pb;
      }
      e[g] = warp_sum(pa + pb);
    }
    if (lane == 0)
#pragma unroll
      for (int g = 0; g < HP; ++g) red[warp][g] = e[g];
    __syncthreads();
    if (threadIdx.x < HP && g0 + (int)threadIdx.x < G) {
      float l = 0.f;
#pragma unroll
      for (int w = 0; w < SC_WARPS; ++w) l += red[w][threadIdx.x];
      const int64_t idx = ((int64_t)b * H + kvh * G + g0 + threadIdx.x) * chunks_max + c;
      part_m[idx] = cmax[threadIdx.x];
      part_l[idx] = l;
    }
    __syncthreads();
  }

  // V rows of the chunk replace the K rows in shared memory
  stage_rows<T, D, SC_THREADS>(kbase, V + tile_off, (int64_t)Hkv * D, len);
  cp_async_wait_all();
  __syncthreads();

  // lane owns columns [lane * CPL, lane * CPL + CPL): 16-byte chunk cc, byte offset within it
  constexpr int LANE_BYTES = CPL * R::ES;      // 4, 8 or 16
  const int cc = (lane * LANE_BYTES) / 16, within = (lane * LANE_BYTES) % 16;
  f2x acc[GM][CPL / 2];
#pragma unroll
  for (int g = 0; g < GM; ++g)
#pragma unroll
    for (int i = 0; i < CPL / 2; ++i) acc[g][i] = 0ull;
  for (int n = warp; n < len; n += SC_WARPS) {
    const uint32_t addr = kbase + n * R::ROWB + swz(n, cc) * 16 + within;
    f2x v[CPL / 2];
    if constexpr (LANE_BYTES == 16) {
      f2x tmp[R::EPC / 2];
      Pairs<T>::get(lds128(addr), tmp);
#pragma unroll
      for (int i = 0; i < CPL / 2; ++i) v[i] = tmp[i];
    } else if constexpr (LANE_BYTES == 8) {
      uint2 w;
      asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(w.x), "=r"(w.y) : "r"(addr));
      f2x tmp[4];
      Pairs<T>::get(make_uint4(w.x, w.y, 0u, 0u), tmp);
#pragma unroll
      for (int i = 0; i < CPL / 2; ++i) v[i] = tmp[i];
    } else {
      uint32_t w;
      asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(addr));
      f2x tmp[4];
      Pairs<T>::get(make_uint4(w, 0u, 0u, 0u), tmp);
      v[0] = tmp[0];
    }
    const float4 p0 = *reinterpret_cast<const float4*>(pS + n * GM);
    const float4 p1 = *reinterpret_cast<const float4*>(pS + n * GM + 4);
    const float pw[GM] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      if (g < G) {
        const f2x pp = pack2(pw[g], pw[g]);
#pragma unroll
        for (int i = 0; i < CPL / 2; ++i) acc[g][i] = ffma2(pp, v[i], acc[g][i]);
      }
    }
  }
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    if (g < G) {
#pragma unroll
      for (int i = 0; i < CPL / 2; ++i) {
        const float2 a = unpack2(acc[g][i]);
        obuf[(warp * GM + g) * D + lane * CPL + 2 * i] = a.x;
        obuf[(warp * GM + g) * D + lane * CPL + 2 * i + 1] = a.y;
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += SC_THREADS) {
    const int g = i / D, col = i % D;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < SC_WARPS; ++w) o += obuf[(w * GM + g) * D + col];
    const int64_t bh = (int64_t)b * H + kvh * G + g;
    part_o[(bh * chunks_max + c) * D + col] = o;
  }
}

// ---------------------------------------------------------------------------
// Dense comparator, stage 2: merge the chunk partials of one head,
// O = sum_c e^{m_c - m*} O_c / sum_c e^{m_c - m*} l_c.  grid = (H, B), block =
// 256; each warp takes every 8th chunk, with four chunks' loads in flight.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(THREADS)
dense_merge_kernel(const int64_t* __restrict__ kv_offsets, int64_t nk_max, int H, const float* __restrict__ part_m,
                   const float* __restrict__ part_l, const float* __restrict__ part_o, int chunks_max,
                   float* __restrict__ out, int* err) {
  constexpr int CPL = D / 32;  // columns per lane
  constexpr int U = 4;         // chunks per batch per warp
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
  for (int c0 = warp; c0 < C; c0 += WARPS * U) {
    float mm[U], ll[U], oo[U][CPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * WARPS;
      const bool ok = c < C;
      mm[u] = ok ? pm[c] : -INFINITY;
      ll[u] = ok ? pl[c] : 0.f;
#pragma unroll
      for (int i = 0; i < CPL; ++i) oo[u][i] = ok ? po[(int64_t)c * D + lane * CPL + i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float f = expf(mm[u] - mstar);
      lsum += f * ll[u];
#pragma unroll
      for (int i = 0; i < CPL; ++i) acc[i] = fmaf(f, oo[u][i], acc[i]);
    }
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
template <typename KernelT>
static cudaError_t allow_smem(KernelT kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Score pass for 16-bit caches: the per-warp streaming pipelines of
// santa_stream.cuh; the CTA also clears `out` (the sampler accumulates into it).
template <typename T, int D>
__global__ void __launch_bounds__(SB_THREADS, 1)
score_warp_kernel(StreamArgs a, float* __restrict__ out, int64_t out_n4) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int start[4];
  if (threadIdx.x < 32)
    unit_range_start(a.kv_offsets, a.nk_max, a.B, a.Hkv / a.W, SB_UNIT_ROWS_X_W / a.W, blockIdx.x, gridDim.x, start);
  __syncthreads();
  allow_dependents();  // the next stage may launch now; it waits for this grid before reading
  if (out)
    for (int64_t i = (int64_t)blockIdx.x * SB_THREADS + threadIdx.x; i < out_n4; i += (int64_t)gridDim.x * SB_THREADS)
      reinterpret_cast<float4*>(out)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  stream_scores<T, D>(a, smem_addr(smem), start);
}

template <typename T, int D>
static cudaError_t launch_score_warp(const LaunchArgs& a) {
  using Gm = StreamGeom<T, D>;
  StreamArgs s;
  s.q = a.q;
  s.K = a.K;
  s.kv_offsets = a.kv_offsets;
  s.nk_max = a.nk_max;
  s.B = a.B;
  s.H = a.H;
  s.Hkv = a.Hkv;
  s.W = unit_heads(a.Hkv);
  s.scale = a.scale;
  s.stash = a.stash;
  s.sub_max = a.tile_max;
  s.sub_sum = a.tile_sum;
  s.subs_max = a.chunks_max;
  const int unit_rows = SB_UNIT_ROWS_X_W / s.W;
  const long long units = (long long)a.B * ((a.nk_max + unit_rows - 1) / unit_rows) * (a.Hkv / s.W);
  const unsigned grid = (unsigned)std::min<long long>(units, (long long)a.num_sms);
  cudaError_t e = allow_smem(score_warp_kernel<T, D>, Gm::SMEM);
  if (e != cudaSuccess) return e;
  score_warp_kernel<T, D><<<grid, SB_THREADS, Gm::SMEM, a.stream>>>(s, a.out, a.out ? (int64_t)a.B * a.H * D / 4 : 0);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch_score_t(const LaunchArgs& a) {
  if constexpr (sizeof(T) == 2) {
    return launch_score_warp<T, D>(a);
  } else {
    const int W = unit_heads(a.Hkv);
    const int unit_rows = 32 * (UNIT_TASKS / W);
    const long long units = (long long)a.B * ((a.nk_max + unit_rows - 1) / unit_rows) * (a.Hkv / W);
    const unsigned grid = (unsigned)std::min<long long>(units, (long long)a.num_sms);
    auto kern = (a.H / a.Hkv <= HP) ? score_stream_kernel<T, D, 1> : score_stream_kernel<T, D, 2>;
    const size_t smem = stream_smem_bytes<T, D>();
    cudaError_t e = allow_smem(kern, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, ST_THREADS, smem, a.stream>>>((const T*)a.q, (const T*)a.K, a.kv_offsets, a.nk_max, a.B, a.H,
                                               a.Hkv, W, a.scale, a.stash, a.tile_max, a.tile_sum, a.chunks_max,
                                               a.out);
    return cudaGetLastError();
  }
}

template <typename T, int D>
static cudaError_t launch_dense_t(const LaunchArgs& a) {
  dim3 grid((unsigned)a.Hkv, (unsigned)a.chunks_max, (unsigned)a.B);
  auto kern = (a.H / a.Hkv <= HP) ? dense_chunks_kernel<T, D, 1> : dense_chunks_kernel<T, D, 2>;
  const size_t smem = dense_smem_bytes<T, D>();
  cudaError_t e = allow_smem(kern, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, SC_THREADS, smem, a.stream>>>((const T*)a.q, (const T*)a.K, (const T*)a.V, a.kv_offsets, a.nk_max,
                                             a.H, a.Hkv, a.scale, a.tile_max, a.tile_sum, a.part_o, a.chunks_max);
  e = cudaGetLastError();
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
