// santa_window.cuh -- inverse-CDF resolution inside one 32-key window and the
// count-weighted V gather, shared by the staged sampler and the single-launch
// decode ("Stochastic Sparse Attention for Memory-Bound Inference": inverse
// CDF App. A.4; gather-and-add Eq. (4), Fig. 1).
#pragma once

#include <climits>

#include "santa_common.cuh"

namespace santa {

// Probability masses are handled as fixed-point integers in units of 2^-40 of
// the head-max key's mass (a key's mass relative to the max is <= 1).  Integer
// sums are exact in any association, so every prefix is exactly monotone and
// no FP64 arithmetic (slow on this part) is needed in any loop.  Conversion
// truncates; masses below 2^-40 of the max key count as zero.
constexpr int MASS_SHIFT = 40;

// w * 2^40 rounded toward zero, for finite w in [0, 2^22), by integer
// operations without branches (both shifts computed, one selected): zero,
// subnormal, non-finite and negative w give 0.
__device__ __forceinline__ long long mass_fixed(float w) {
  const uint32_t bits = __float_as_uint(w);
  const int e = (int)((bits >> 23) & 0xffu);
  const unsigned long long m = (unsigned long long)((bits & 0x7fffffu) | 0x800000u);
  const int sh = e - 127 - 23 + MASS_SHIFT;                  // w * 2^40 = m * 2^sh
  const unsigned long long up = m << (unsigned)min(max(sh, 0), 39);
  const unsigned long long dn = m >> (unsigned)min(max(-sh, 0), 63);
  const bool ok = e != 0 && e != 0xff && !(bits >> 31);
  return ok ? (long long)(sh >= 0 ? up : dn) : 0ll;
}

// Inclusive warp scan of one int64 per lane.
__device__ __forceinline__ long long warp_inclusive_scan(long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(FULL, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// lower_bound of v among the sorted values x held one per lane (lanes >= n hold +inf)
__device__ __forceinline__ int lane_lower_bound(long long x, int n, long long v) {
  int lo = 0, hi = n;
#pragma unroll
  for (int it = 0; it < 6; ++it) {
    const int mid = (lo + hi) >> 1;
    const long long xm = __shfl_sync(FULL, x, mid & 31);
    if (lo < hi) {
      if (xm < v) lo = mid + 1;
      else hi = mid;
    }
  }
  return lo;
}

// Draws of the lane's key among the nt thresholds of one head that fall in
// this 32-key window (warp-uniform arguments except sv, th0, key).
//   sv        the lane's key score (-inf past the sequence end)
//   mst       the head's max score m*
//   th0       the window's threshold number `lane` (absolute mass units), LLONG_MAX past nt
//   pb        mass prefix at the window start
//   th        the window's sorted thresholds (read for batches beyond the first 32)
//   idx       the head's sample_idx entry of the window's first threshold, or NULL
// A key n is drawn by threshold x with F(n-1) <= x < F(n) (window-relative
// exact prefixes); thresholds at or beyond the window's total (rounding of the
// chunk masses against the key masses) go to the window's last nonzero key.
// Not inlined (the staged sampler calls it from many unrolled sites).
static __device__ __noinline__ int window_draws(float sv, float mst, long long th0, int nt, long long pb,
                                            const long long* th, int32_t* idx, int key, int lane) {
  const long long w = mass_fixed(expf(sv - mst));   // e^{-inf} = 0 past the sequence end
  const long long F = warp_inclusive_scan(w, lane);
  const unsigned nz = __ballot_sync(FULL, w > 0);
  const int last_nz = nz ? 31 - __clz(nz) : 0;
  if (nt <= 8) {   // few thresholds: one ballot each, the key is the first lane with F > x
    int cnt = 0;
    for (int t = 0; t < nt; ++t) {
      const long long x = __shfl_sync(FULL, th0, t) - pb;
      const unsigned above = __ballot_sync(FULL, F > x);
      const int k = above ? __ffs(above) - 1 : last_nz;
      cnt += (lane == k) ? 1 : 0;
      if (idx && lane == k) idx[t] = key;
    }
    return cnt;
  }
  const long long total = __shfl_sync(FULL, F, 31);
  int lb = 0, lb_total = 0;
  for (int base = 0; base < nt; base += 32) {
    const int n = min(32, nt - base);
    long long x = (base == 0) ? th0 : ((lane < n) ? th[base + lane] : LLONG_MAX);
    x = (lane < n) ? x - pb : LLONG_MAX;
    lb += lane_lower_bound(x, n, F);
    lb_total += lane_lower_bound(x, n, total);
  }
  const int lb_up = __shfl_up_sync(FULL, lb, 1);
  const int lb_prev = (lane == 0) ? 0 : lb_up;
  int cnt = lb - lb_prev;                                    // F_{lane-1} <= x < F_lane
  if (lane == last_nz) cnt += nt - lb_total;                 // x >= the window's total
  if (idx) {
    for (int j = lb_prev; j < lb; ++j) idx[j] = key;
    if (lane == last_nz)
      for (int j = lb_total; j < nt; ++j) idx[j] = key;
  }
  return cnt;
}

// Count-weighted gather-and-add of the rows `rows[0..nrows)` (entries i*32 +
// lane: key lane of window w0 + i) of one KV head into acc[g][e] (head g, the
// lane's EPL output columns); cnt holds the per-(window, head, key) counts,
// [window][GM][32].  Each drawn row is read once for all heads of the group.
// Partial sums stay spread over the warp's row slots: reduce_slots adds them.
template <typename T, int D, int GM>
__device__ __forceinline__ void gather_rows(float (&acc)[GM][Tile<T, D>::EPL], const int* rows, int nrows,
                                            const int* cnt, const T* __restrict__ Vbase, int64_t w0, int Hkv, int G,
                                            int lane) {
  using TL = Tile<T, D>;
  const int slot = lane / TL::LPK;
  constexpr int UNR = 8;
  for (int i0 = slot; i0 < nrows; i0 += UNR * TL::KPI) {
    uint4 vv[UNR][TL::NVEC];
    int rk[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int i = i0 + u * TL::KPI;
      rk[u] = (i < nrows) ? rows[i] : -1;
      const int64_t key = (w0 + (rk[u] >> 5)) * 32 + (rk[u] & 31);
#pragma unroll
      for (int v = 0; v < TL::NVEC; ++v)
        vv[u][v] = (rk[u] >= 0) ? ld_stream(Vbase + key * Hkv * D + v * (16 / TL::ES)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      if (rk[u] < 0) continue;
      float vf[TL::EPL];
#pragma unroll
      for (int v = 0; v < TL::NVEC; ++v) Elem<T>::widen(vv[u][v], vf + v * (16 / TL::ES));
      const int* cr = cnt + (rk[u] >> 5) * GM * 32 + (rk[u] & 31);
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        if (g < G) {
          const float cg = (float)cr[g * 32];
#pragma unroll
          for (int e = 0; e < TL::EPL; ++e) acc[g][e] = fmaf(cg, vf[e], acc[g][e]);
        }
      }
    }
  }
}

// Sums acc over the lanes that hold the same output columns (the KPI row
// slots of a warp); afterwards every lane holds the warp's total.
template <typename T, int D, int GM>
__device__ __forceinline__ void reduce_slots(float (&acc)[GM][Tile<T, D>::EPL]) {
  using TL = Tile<T, D>;
#pragma unroll
  for (int o = TL::LPK; o < 32; o <<= 1)
#pragma unroll
    for (int g = 0; g < GM; ++g)
#pragma unroll
      for (int e = 0; e < TL::EPL; ++e) acc[g][e] += __shfl_xor_sync(FULL, acc[g][e], o);
}

}  // namespace santa
