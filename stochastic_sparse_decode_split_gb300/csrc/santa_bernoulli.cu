// santa_bernoulli.cu -- Bernoulli qK^T with the mean group query ("Stochastic
// Sparse Attention for Memory-Bound Inference", Sec. 5.1, App. C.2,
// Eq. 10-13), in front of the decode step.
//
// For the query group of each (sequence, KV head), with m_i = (1/G) sum_g
// |q_g,i| (Eq. 10) and norm = max_i m_i, feature i keeps c_i of B Bernoulli
// draws with probability m_i / norm (Eq. 11; stratified: draw n is one when
// (n + u)/B < m_i / norm, one uniform per stratum), m^_i = norm c_i / B
// (Eq. 12), and every head of the group takes the effective query
// q~_g,i = m^_i q_g,i / m_i, so that q~_g . K_n is Eq. 13's (m^ o q_g / m) K_n.
// Features with c_i = 0 are zero in every q~ of the group: the keys' feature
// i is not needed by any head.  The decode then runs on q~ unchanged.
//
// The arithmetic is fp32 in a fixed order, each operation IEEE-rounded (no
// contraction: no product feeds an addition): m_i summed over g in order,
// then / G; p_i = m_i / norm; m^_i = (norm c_i) / B; q~ = (m^_i q) / m_i,
// rounded to nearest even into the cache dtype.  The Bernoulli tests compare
// 24-bit uniforms exactly (a24 < p_i 2^24; stratified n 2^24 + a24 <
// B p_i 2^24, both exact in float64).  Uniform r = n d + i of the group is
// word r % 4 of the Philox block at counter (r / 4, H + kvh, b, step): a
// stream of its own beside the query heads' 0..H-1.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "santa_common.cuh"
#include "santa_launch.h"

namespace santa {

template <typename T> __device__ __forceinline__ T round_store(float x);
template <> __device__ __forceinline__ bf16_t round_store<bf16_t>(float x) {
  bf16_t r;
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  memcpy(&r, &h, 2);
  return r;
}
template <> __device__ __forceinline__ fp16_t round_store<fp16_t>(float x) {
  fp16_t r;
  const __half h = __float2half_rn(x);
  memcpy(&r, &h, 2);
  return r;
}
template <> __device__ __forceinline__ float round_store<float>(float x) { return x; }

// One CTA per (sequence, KV head), one thread per feature (blockDim = D).
template <typename T, int D>
__global__ void __launch_bounds__(D) bernoulli_query_kernel(const T* __restrict__ q, T* __restrict__ qt,
                                                            int32_t* __restrict__ counts, int H, int Hkv, int nsamp,
                                                            int stratified, uint64_t seed, uint32_t step) {
  const int bk = blockIdx.x, b = bk / Hkv, kvh = bk % Hkv, G = H / Hkv, i = threadIdx.x;
  const int64_t base = ((int64_t)b * H + (int64_t)kvh * G) * D + i;   // q[b, kvh G + g, i] at base + g D
  float acc = 0.f;
  for (int g = 0; g < G; ++g) acc += fabsf(widen_scalar<T>(q + base + (int64_t)g * D));
  const float m = acc / (float)G;
  __shared__ float red[D / 32];
  const float wm = warp_max(m);
  if (i % 32 == 0) red[i / 32] = wm;
  __syncthreads();
  float norm = red[0];
#pragma unroll
  for (int w = 1; w < D / 32; ++w) norm = fmaxf(norm, red[w]);
  int c = 0;
  if (norm > 0.f && m > 0.f) {
    const float pr = m / norm;
    const double lim = stratified ? ((double)nsamp * (double)pr) * 16777216.0 : (double)pr * 16777216.0;
    const uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
    for (int n = 0; n < nsamp; ++n) {
      const uint32_t r = (uint32_t)(n * D + i);
      const uint4 w4 = philox4x32_10(make_uint4(r >> 2, (uint32_t)(H + kvh), (uint32_t)b, step), k0, k1);
      const uint32_t word = (r & 3) == 0 ? w4.x : (r & 3) == 1 ? w4.y : (r & 3) == 2 ? w4.z : w4.w;
      const double a24 = (double)(word >> 8);
      c += (stratified ? (double)n * 16777216.0 + a24 : a24) < lim ? 1 : 0;
    }
  }
  if (counts) counts[(int64_t)bk * D + i] = c;
  const float mh = (norm * (float)c) / (float)nsamp;
  for (int g = 0; g < G; ++g) {
    const float qv = widen_scalar<T>(q + base + (int64_t)g * D);
    qt[base + (int64_t)g * D] = round_store<T>(m > 0.f ? (mh * qv) / m : 0.f);
  }
}

template <typename T, int D>
static cudaError_t launch_bq(const LaunchArgs& a, void* qt, int32_t* counts, int nsamp, int stratified) {
  bernoulli_query_kernel<T, D><<<(unsigned)((int64_t)a.B * a.Hkv), D, 0, a.stream>>>(
      (const T*)a.q, (T*)qt, counts, a.H, a.Hkv, nsamp, stratified, a.seed, a.step);
  return cudaGetLastError();
}

cudaError_t launch_bernoulli_query(const LaunchArgs& a, void* qt, int32_t* counts, int nsamp, int stratified) {
  switch (a.dtype * 2 + (a.D == 128)) {
    case 0: return launch_bq<bf16_t, 64>(a, qt, counts, nsamp, stratified);
    case 1: return launch_bq<bf16_t, 128>(a, qt, counts, nsamp, stratified);
    case 2: return launch_bq<fp16_t, 64>(a, qt, counts, nsamp, stratified);
    case 3: return launch_bq<fp16_t, 128>(a, qt, counts, nsamp, stratified);
    case 4: return launch_bq<float, 64>(a, qt, counts, nsamp, stratified);
    case 5: return launch_bq<float, 128>(a, qt, counts, nsamp, stratified);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace santa
