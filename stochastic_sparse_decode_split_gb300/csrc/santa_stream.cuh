// santa_stream.cuh -- the streaming score pass for 16-bit caches (sm_103a):
// exact scores s_n = scale * q . K_n of every query head over the whole cache
// and per-16-key (max, exp-sum) statistics ("Stochastic Sparse Attention for
// Memory-Bound Inference", Sec. 2 Eq. (1); App. O, Alg. 3).
//
// One persistent 512-thread CTA per SM.  Each of its 16 warps is an
// independent pipeline: it copies exactly the 16 K rows (16 keys x 1 KV head)
// it will score from HBM into its own ring of shared-memory stages with
// cp.async (16 bytes per request, NS - 1 units in flight), waits for its own
// copies only, and scores the rows on the tensor cores.  No barrier couples
// the warps.  Rows are stored with a 16-byte pad (pitch = 16 mod 128 bytes),
// so the eight rows an ldmatrix phase reads fall on distinct bank groups.
//
// Work units: W KV heads (W = largest power of two <= 8 dividing H_kv) x
// 8 / W blocks of 32 keys of one sequence (two warps per 32-key block and KV
// head), enumerated in (sequence, KV-head group, key block) order over the
// actual sequence lengths; CTA i takes the contiguous unit range
// [i T / P, (i + 1) T / P) of the T units.
#pragma once

#include "santa_common.cuh"

namespace santa {

constexpr int SB_WARPS = 16;                    // warps per CTA: one 16-key x 1 KV head m-tile each
constexpr int SB_THREADS = SB_WARPS * 32;
constexpr int SB_TASKS = 8;                     // (32 keys x 1 KV head) tasks per unit
constexpr int SB_UNIT_ROWS_X_W = SB_TASKS * 32; // K rows (key, KV head) per unit: 256

// Bound on any single wait of a grid-wide barrier.  Expected waits are
// microseconds; on expiry the kernel flags ERR_TIMEOUT and stops waiting.
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;


// Width of a score-pass unit in KV heads: the largest power of two <= 8 dividing H_kv.
__host__ __device__ inline int unit_heads(int Hkv) {
  int w = 8;
  while (w > 1 && Hkv % w) w >>= 1;
  return w;
}

// ---------------------------------------------------------------------------
// Unit enumeration over the actual sequence lengths
// ---------------------------------------------------------------------------
struct UnitCursor {
  const int64_t* kv_offsets;
  int64_t nk_max;
  int B, n_hg, unit_rows;
  int b, hg, kb, units_b;
  int64_t row0, nk;

  // Rows of sequence b; lengths outside [1, nk_max] are clamped here (they
  // are reported by the stage that checks the metadata).
  __device__ __forceinline__ static int seq_units(const int64_t* kv_offsets, int64_t nk_max, int unit_rows, int b,
                                                  int64_t& row0, int64_t& nk) {
    if (kv_offsets) {
      row0 = kv_offsets[b];
      nk = kv_offsets[b + 1] - row0;
    } else {
      row0 = (int64_t)b * nk_max;
      nk = nk_max;
    }
    if (nk < 1 || row0 < 0) nk = 0;
    nk = nk < nk_max ? nk : nk_max;
    return (int)((nk + unit_rows - 1) / unit_rows);
  }
  __device__ __forceinline__ void load_seq() { units_b = seq_units(kv_offsets, nk_max, unit_rows, b, row0, nk); }
  __device__ __forceinline__ void advance() {
    if (++kb < units_b) return;
    kb = 0;
    if (++hg < n_hg) return;
    hg = 0;
    for (;;) {
      if (++b >= B) {
        units_b = 0;
        return;
      }
      load_seq();
      if (units_b) return;
    }
  }
};

// Start of CTA `cta`'s unit range (of `ctas`), computed by one warp:
// out = {b, hg, kb, n_units}; range = {T, u0} (total units, first unit) when not NULL.
__device__ __forceinline__ void unit_range_start(const int64_t* kv_offsets, int64_t nk_max, int B, int n_hg,
                                                 int unit_rows, int cta, int ctas, int* out,
                                                 long long* range = nullptr) {
  const int lane = threadIdx.x % 32;
  long long total = 0;
  if (!kv_offsets) {
    total = (long long)B * n_hg * ((nk_max + unit_rows - 1) / unit_rows);
  } else {
    for (int b0 = 0; b0 < B; b0 += 32) {
      int64_t r0, n;
      const int u = (b0 + lane < B) ? UnitCursor::seq_units(kv_offsets, nk_max, unit_rows, b0 + lane, r0, n) : 0;
      long long s = u;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
      total += s;
    }
    total *= n_hg;
  }
  const long long u0 = total * cta / ctas, u1 = total * (cta + 1) / ctas;
  // locate u0: first sequence whose cumulative unit count exceeds it
  int b = 0, hg = 0, kb = 0;
  if (u1 > u0) {
    if (!kv_offsets) {
      const long long per_b = total / B, ub = per_b / n_hg;
      b = (int)(u0 / per_b);
      const long long r = u0 - (long long)b * per_b;
      hg = (int)(r / ub);
      kb = (int)(r % ub);
    } else {
      long long base = 0;
      for (int b0 = 0; b0 < B; b0 += 32) {
        int64_t r0, n;
        const int u = (b0 + lane < B) ? UnitCursor::seq_units(kv_offsets, nk_max, unit_rows, b0 + lane, r0, n) : 0;
        long long incl = (long long)u * n_hg;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long t = __shfl_up_sync(FULL, incl, o);
          if (lane >= o) incl += t;
        }
        const unsigned hit = __ballot_sync(FULL, base + incl > u0);
        if (hit) {
          const int l = __ffs(hit) - 1;
          const int ul = __shfl_sync(FULL, u, l);
          const long long excl = base + __shfl_sync(FULL, incl, l) - (long long)ul * n_hg;
          b = b0 + l;
          hg = (int)((u0 - excl) / ul);
          kb = (int)((u0 - excl) % ul);
          break;
        }
        base += __shfl_sync(FULL, incl, 31);
      }
    }
  }
  if (lane == 0) {
    out[0] = b;
    out[1] = hg;
    out[2] = kb;
    out[3] = (int)(u1 - u0);
    if (range) {
      range[0] = total;
      range[1] = u0;
    }
  }
}

// ---------------------------------------------------------------------------
// Stage geometry
// ---------------------------------------------------------------------------
template <typename T, int D>
struct StreamGeom {
  static constexpr int ROWB = D * 2;             // bytes of one K row (16-bit elements)
  static constexpr int NCH = ROWB / 16;          // 16-byte chunks per row
  static constexpr int RSTR = ROWB + 16;         // padded row pitch in shared memory
  static constexpr int WSTAGE = 16 * RSTR;       // one warp's stage: 16 rows
  // ring depth: as many stages as fit the 227 KiB opt-in limit less static use, at most 6
  static constexpr int NS = (225 * 1024) / (SB_WARPS * WSTAGE) < 6 ? (225 * 1024) / (SB_WARPS * WSTAGE) : 6;
  static constexpr size_t SMEM = (size_t)SB_WARPS * NS * WSTAGE;
  static_assert(sizeof(T) == 2, "16-bit caches only");
  static_assert(NS >= 3, "ring of at least three stages");
  static_assert((16 * NCH) % 32 == 0, "copy split");
};

// Parameters of one streaming pass.
struct StreamArgs {
  const void* q;
  const void* K;
  const int64_t* kv_offsets;
  int64_t nk_max;
  int B, H, Hkv, W;
  float scale;
  float* stash;       // [B, H, nk_max]
  float* sub_max;     // [B, H, subs_max]
  float* sub_sum;
  int subs_max;
};

// The streaming loop of one CTA over its unit range.  `ring` is the dynamic
// shared memory (SMEM bytes, 16-byte aligned), `start` the range start
// broadcast by unit_range_start.  Called by all SB_THREADS threads.
//
// run_m / run_l (shared memory, [16 warps][8 heads], may be NULL): each warp's
// running (max, sum exp(s - max)) over every key it scored, per head of its
// KV head's query group; meaningful when the range is one (sequence, KV-head
// group), which the caller checks.
template <typename T, int D>
__device__ __forceinline__ void stream_scores(const StreamArgs& a, uint32_t ring, const int* start,
                                              float* run_m = nullptr, float* run_l = nullptr) {
  using Gm = StreamGeom<T, D>;
  constexpr int NS = Gm::NS;
  constexpr int CPL = 16 * Gm::NCH / 32;      // 16-byte copies per lane per unit
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int W = a.W, G = a.H / a.Hkv;
  const int unit_rows = SB_UNIT_ROWS_X_W / W;
  const int n_mine = start[3];
  if (n_mine <= 0) return;
  UnitCursor cur;                              // unit being scored
  cur.kv_offsets = a.kv_offsets;
  cur.nk_max = a.nk_max;
  cur.B = a.B;
  cur.n_hg = a.Hkv / W;
  cur.unit_rows = unit_rows;
  cur.b = start[0];
  cur.hg = start[1];
  cur.kb = start[2];
  cur.load_seq();
  UnitCursor nxt = cur;                        // unit being copied

  const int task = warp >> 1, half = warp & 1;
  const int wkb = task / W, wkv = task % W;    // this warp's key block and KV head within a unit
  const int kr0 = wkb * 32 + half * 16;        // first unit row of this warp's 16 keys
  const uint32_t wring = ring + (uint32_t)warp * NS * Gm::WSTAGE;
  const T* K = static_cast<const T*>(a.K);
  const unsigned long long pol = evict_first_policy();   // K is read once per step

  // copies of this warp's 16 rows of unit `u` into stage `s` (one commit group)
  auto issue = [&](const UnitCursor& u, int s, bool live) {
    if (live) {
      const int64_t key0 = (int64_t)u.kb * unit_rows + kr0;
      const int rows = (int)min((int64_t)16, u.nk - key0);
      const T* src = K + ((u.row0 + key0) * a.Hkv + (int64_t)u.hg * W + wkv) * D;
      const uint32_t dst = wring + (uint32_t)s * Gm::WSTAGE;
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int i = lane + 32 * j, r = i / Gm::NCH, c = i % Gm::NCH;
        if (r < rows) cp_async16_hint(dst + r * Gm::RSTR + c * 16, src + (int64_t)r * a.Hkv * D + c * 8, pol);
      }
    }
    cp_async_commit();
  };
  for (int s = 0; s + 1 < NS; ++s) {
    issue(nxt, s, s < n_mine);
    if (s < n_mine) nxt.advance();
  }

  const int g8 = lane >> 2, t4 = lane & 3;
  float rm[2] = {-INFINITY, -INFINITY}, rl[2] = {0.f, 0.f};   // running statistics, heads 2*t4 + hh
  const T* q = static_cast<const T*>(a.q);
  uint32_t bq[D / 16][2];
  int bq_b = -1, bq_kvh = -1;
  const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row of this lane
  const uint32_t lane_off = (uint32_t)lrow * Gm::RSTR + (uint32_t)(lane >> 4) * 16;
  for (int k = 0; k < n_mine; ++k) {
    cp_async_wait<NS - 2>();  // this lane's copies of unit k have landed
    __syncwarp();             // ... and every lane's; stage (k - 1) % NS is free
    {
      const int kn = k + NS - 1;
      issue(nxt, kn % NS, kn < n_mine);
      if (kn < n_mine) nxt.advance();
    }
    const int64_t key0 = (int64_t)cur.kb * unit_rows;
    const int len = (int)min((int64_t)unit_rows, cur.nk - key0);
    if (len > kr0) {
      const int kvh = cur.hg * W + wkv;
      const int64_t bh0 = (int64_t)cur.b * a.H + (int64_t)kvh * G;
      if (cur.b != bq_b || kvh != bq_kvh) {  // q fragments change only with the sequence / KV head
        const T* qg = q + bh0 * D;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const T* qp = qg + g8 * D + ks * 16 + t4 * 2;
          bq[ks][0] = (g8 < G) ? *reinterpret_cast<const uint32_t*>(qp) : 0u;
          bq[ks][1] = (g8 < G) ? *reinterpret_cast<const uint32_t*>(qp + 8) : 0u;
        }
        bq_b = cur.b;
        bq_kvh = kvh;
      }
      // 16 keys x 8 heads on the tensor cores, two independent accumulators
      float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t abase = wring + (uint32_t)(k % NS) * Gm::WSTAGE + lane_off;
#pragma unroll
      for (int ks = 0; ks < D / 16; ks += 2) {
        uint32_t x0[4], x1[4];
        ldmatrix_x4(abase + ks * 32, x0);
        ldmatrix_x4(abase + ks * 32 + 32, x1);
        Mma<T>::run(acc0, x0, bq[ks][0], bq[ks][1]);
        Mma<T>::run(acc1, x1, bq[ks + 1][0], bq[ks + 1][1]);
      }
      // lane holds keys g8 and g8 + 8 of the 16 for heads 2*t4 and 2*t4 + 1
      const int64_t key_base = key0 + kr0;
      const int sc = (int)(key_base / SUB);
      const bool ok0 = kr0 + g8 < len, ok1 = kr0 + g8 + 8 < len;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int head = 2 * t4 + hh;
        const float s0 = (acc0[hh] + acc1[hh]) * a.scale, s1 = (acc0[2 + hh] + acc1[2 + hh]) * a.scale;
        if (head < G) {
          float* sp = a.stash + (bh0 + head) * a.nk_max + key_base + g8;
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
          a.sub_max[(bh0 + head) * a.subs_max + sc] = m;
          a.sub_sum[(bh0 + head) * a.subs_max + sc] = l;
        }
        const float nm = fmaxf(rm[hh], m);
        rl[hh] = rl[hh] * fast_exp(rm[hh] - nm) + l * fast_exp(m - nm);
        rm[hh] = nm;
      }
    }
    cur.advance();
  }
  cp_async_wait<0>();
  if (run_m && (lane & ~3) == 0) {   // lanes 0..3: this warp's running statistics of heads 2*lane, 2*lane + 1
    run_m[warp * 8 + 2 * lane] = rm[0];
    run_m[warp * 8 + 2 * lane + 1] = rm[1];
    run_l[warp * 8 + 2 * lane] = rl[0];
    run_l[warp * 8 + 2 * lane + 1] = rl[1];
  }
}

}  // namespace santa
