// santa_part.cuh -- the key-block partition shared by the single-launch
// decode kernels (sm_103a): blocks of 16 keys of one KV head, ordered
// (sequence, KV head, key block); CTA i of P takes the blocks
// [floor(T i / P), floor(T (i + 1) / P)) of the T blocks of the batch, so a
// (sequence, KV head) "piece" may span several CTAs.  Sequence geometry of
// uniform and ragged batches, cursors over blocks, and the multiply-high
// divisions the partition uses.
#pragma once

#include <climits>

#include "santa_common.cuh"
#include "santa_launch.h"

namespace santa {

constexpr int BK = SUB;   // keys per block (== statistics chunk)

// x / d for 32-bit x by a precomputed reciprocal r = floor(2^64 / d) + 1
// (r = 0 stands for d = 1): the 64-bit multiply-high is exact for x < 2^32.
__host__ __device__ inline unsigned long long div_reciprocal(unsigned long long d) {
  return d <= 1 ? 0ull : ~0ull / d + 1ull;
}
__device__ __forceinline__ uint32_t div_by(uint32_t x, unsigned long long r) {
  return r ? (uint32_t)__umul64hi((unsigned long long)x, r) : x;
}

// ---------------------------------------------------------------------------
// Block enumeration over the actual sequence lengths
// ---------------------------------------------------------------------------
struct SeqGeo {
  int64_t row0, nk;
  int nblk;
};
// Rows of sequence b; lengths outside [1, nk_max] are clamped here (the
// metadata check reports them).
__device__ __forceinline__ SeqGeo seq_geo(const LaunchArgs& a, int b) {
  SeqGeo g;
  if (a.kv_offsets) {
    g.row0 = a.kv_offsets[b];
    g.nk = a.kv_offsets[b + 1] - g.row0;
  } else {
    g.row0 = (int64_t)b * a.nk_max;
    g.nk = a.nk_max;
  }
  if (g.nk < 1 || g.row0 < 0) g.nk = 0;
  if (g.nk > a.nk_max) g.nk = a.nk_max;
  g.nblk = (int)((g.nk + BK - 1) / BK);
  return g;
}

// Position of one block: sequence b, KV head kvh, key block kblk of the
// sequence; pb_lo is the global index of block 0 of piece (b, kvh).
struct Cur {
  int b, kvh, kblk, nblk;
  int64_t row0, nk;
  long long pb_lo;
};
// Moves kblk past the end of its piece into the following pieces (b = B: end).
__device__ __forceinline__ void cur_norm(Cur& c, const LaunchArgs& a) {
  while (c.kblk >= c.nblk) {
    c.kblk -= c.nblk;
    c.pb_lo += c.nblk;
    if (++c.kvh == a.Hkv) {
      c.kvh = 0;
      if (++c.b >= a.B) {
        c.b = a.B;
        c.nblk = INT_MAX;
        return;
      }
      const SeqGeo g = seq_geo(a, c.b);
      c.row0 = g.row0;
      c.nk = g.nk;
      c.nblk = g.nblk;
    }
  }
}
__device__ __forceinline__ void cur_advance(Cur& c, const LaunchArgs& a, int n) {
  c.kblk += n;
  cur_norm(c, a);
}

// The cursors of blocks x0 and x1 (x0 <= x1 < T) and the total T, computed by
// one warp.  Uniform batches are closed form; ragged ones scan the lengths.
__device__ __forceinline__ long long total_blocks(const LaunchArgs& a, int lane) {
  if (!a.kv_offsets) return (long long)a.B * a.Hkv * ((a.nk_max + BK - 1) / BK);
  long long total = 0;
  for (int b0 = 0; b0 < a.B; b0 += 32) {
    long long s = (b0 + lane < a.B) ? (long long)seq_geo(a, b0 + lane).nblk : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
    total += s;
  }
  return total * a.Hkv;
}
__device__ __forceinline__ Cur locate_block(const LaunchArgs& a, long long x, int lane) {
  Cur c;
  if (!a.kv_offsets) {
    const int nblk = (int)((a.nk_max + BK - 1) / BK);
    const long long per_b = (long long)a.Hkv * nblk;
    c.b = (int)(x / per_b);
    const long long r = x - (long long)c.b * per_b;
    c.kvh = (int)(r / nblk);
    c.kblk = (int)(r - (long long)c.kvh * nblk);
    c.nblk = nblk;
    c.row0 = (int64_t)c.b * a.nk_max;
    c.nk = a.nk_max;
    c.pb_lo = x - c.kblk;
    return c;
  }
  long long base = 0;
  c.b = a.B;
  for (int b0 = 0; b0 < a.B; b0 += 32) {
    const int nb = (b0 + lane < a.B) ? seq_geo(a, b0 + lane).nblk : 0;
    long long incl = (long long)nb * a.Hkv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(FULL, base + incl > x);
    if (hit) {
      const int l = __ffs(hit) - 1;
      const int nbl = __shfl_sync(FULL, nb, l);
      const long long excl = base + __shfl_sync(FULL, incl, l) - (long long)nbl * a.Hkv;
      c.b = b0 + l;
      const long long r = x - excl;
      c.kvh = (int)(r / nbl);
      c.kblk = (int)(r - (long long)c.kvh * nbl);
      c.nblk = nbl;
      const SeqGeo g = seq_geo(a, c.b);
      c.row0 = g.row0;
      c.nk = g.nk;
      c.pb_lo = x - c.kblk;
      break;
    }
    base += __shfl_sync(FULL, incl, 31);
  }
  return c;
}

// The single-launch partition: CTA i of P takes blocks [lo(i), lo(i + 1)),
// lo(i) = floor(T i / P) = q i + floor(r i / P) with T = q P + r.
struct Part {
  long long T, q;
  int r, P;
  unsigned long long rP;   // reciprocal of P (div_reciprocal)
  __device__ __forceinline__ long long lo(int i) const { return q * i + div_by((uint32_t)(r * i), rP); }
  // the CTA whose range holds block x (0 <= x < T): the largest i with lo(i) <= x
  __device__ __forceinline__ int cta_of(long long x) const {
    int c = (int)(((float)x + 0.5f) / (float)T * (float)P);
    c = min(max(c, 0), P - 1);
    while (c + 1 < P && lo(c + 1) <= x) ++c;
    while (c > 0 && lo(c) > x) --c;
    return c;
  }
  __device__ __forceinline__ bool nonempty(int i) const { return T >= P || lo(i) < lo(i + 1); }
};

// Cursor of block x of a uniform batch (every sequence nk_max keys).
__device__ __forceinline__ Cur locate_uniform(const LaunchArgs& a, long long x) {
  Cur c;
  const int nblk = (int)((a.nk_max + BK - 1) / BK);
  const long long per_b = (long long)a.Hkv * nblk;
  long long r;
  if (x < (1ll << 32) && per_b < (1ll << 32)) {   // 32-bit dividends: multiply-high reciprocals
    c.b = (int)div_by((uint32_t)x, a.rdiv_perb);
    r = (long long)((uint32_t)x - (uint32_t)c.b * (uint32_t)per_b);
  } else {
    c.b = (int)(x / per_b);
    r = x - (long long)c.b * per_b;
  }
  c.kvh = (int)div_by((uint32_t)r, a.rdiv_nblk);
  c.kblk = (int)(r - (long long)c.kvh * nblk);
  c.nblk = nblk;
  c.row0 = (int64_t)c.b * a.nk_max;
  c.nk = a.nk_max;
  c.pb_lo = x - c.kblk;
  return c;
}

// The range [lo, hi) of CTA `cta` of P and the cursors of blocks lo and
// hi - 1 (b = B when the range is empty), for uniform batches in closed form,
// for ragged ones by a scan of the lengths in warp 0.  Called by every thread
// of the CTA (ragged batches synchronise it through s_part and s_cur).
__device__ __forceinline__ void cta_range(const LaunchArgs& a, int P, int cta, int warp, int lane,
                                          long long* s_part, Cur* s_cur, Part& pt, long long& lo, long long& hi,
                                          Cur& cA, Cur& cB) {
  pt.P = P;
  pt.rP = a.rdiv_grid;
  if (!a.kv_offsets) {
    pt.T = a.blk_total;
    pt.q = a.blk_q;
    pt.r = a.blk_r;
  } else {
    if (warp == 0) {
      const long long Tb = total_blocks(a, lane);
      if (lane == 0) {
        s_part[0] = Tb;
        s_part[1] = Tb / P;
      }
    }
    __syncthreads();
    pt.T = s_part[0];
    pt.q = s_part[1];
    pt.r = (int)(pt.T - pt.q * P);
  }
  lo = pt.lo(cta);
  hi = pt.lo(cta + 1);
  const bool has_range = hi > lo;
  if (!a.kv_offsets) {
    if (has_range) {
      cA = locate_uniform(a, lo);
      cB = locate_uniform(a, hi - 1);
    }
  } else {
    if (warp == 0 && has_range) {
      const Cur c0 = locate_block(a, lo, lane), c1 = locate_block(a, hi - 1, lane);
      if (lane == 0) {
        s_cur[0] = c0;
        s_cur[1] = c1;
      }
    }
    __syncthreads();
    cA = s_cur[0];
    cB = s_cur[1];
  }
  if (!has_range) {
    cA.b = cB.b = a.B;
    cA.pb_lo = cB.pb_lo = LLONG_MAX;
    cA.nblk = cB.nblk = INT_MAX;
  }
}

}  // namespace santa
