/*
 * santa_oracle.c -- plain float64 CPU reference for SANTA / S2ANTA decode-step
 * attention.  TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU-baseline
 * timing); it shares no code with the CUDA library.
 *
 * Each head is processed on its own, straight from the definitions in
 * "Stochastic Sparse Attention for Memory-Bound Inference":
 *   1. s_n = scale * q . K_n, A = softmax(s)                     (Sec. 2, Eq. 1)
 *   2. F(n) = p_0 + ... + p_n, keys in index order              (App. A.4)
 *   3. thresholds t_j per sampling scheme                       (Sec. 2.1; Eq. 4)
 *   4. J_j = the unique n with F(n-1) <= t_j < F(n)              (App. A.4)
 *   5. estimate = (1/S) * sum_n c_n V_n, c_n = #{j : J_j = n}    (Eq. 4, Fig. 1)
 * No blocking, fusion or reordering beyond these steps.
 */
#include "santa_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* storage widening (exact)                                            */
/* ------------------------------------------------------------------ */

static double bf16_to_double(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

static double fp16_to_double(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int expo = (bits >> 10) & 0x1f;
  int mant = bits & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)mant, -24);                 /* subnormal: mant * 2^-24 */
  } else if (expo == 31) {
    v = mant ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + mant), expo - 25);  /* (1.mant) * 2^(expo-15) */
  }
  return sign ? -v : v;
}

static double load_elem(int dtype, const void* base, int64_t idx) {
  if (dtype == ORACLE_BF16) return bf16_to_double(((const uint16_t*)base)[idx]);
  if (dtype == ORACLE_FP16) return fp16_to_double(((const uint16_t*)base)[idx]);
  return (double)((const float*)base)[idx];
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11)                                */
/* ------------------------------------------------------------------ */

/* One Philox S-box round: two 32x32->64 products of counter words 0 and 2
 * with the published multipliers, outputs permuted and keyed by XOR. */
static void philox_round(uint32_t c[4], uint32_t k0, uint32_t k1) {
  const uint64_t prod_a = (uint64_t)0xD2511F53u * (uint64_t)c[0];
  const uint64_t prod_b = (uint64_t)0xCD9E8D57u * (uint64_t)c[2];
  const uint32_t a_hi = (uint32_t)(prod_a >> 32), a_lo = (uint32_t)prod_a;
  const uint32_t b_hi = (uint32_t)(prod_b >> 32), b_lo = (uint32_t)prod_b;
  const uint32_t x0 = b_hi ^ c[1] ^ k0;
  const uint32_t x2 = a_hi ^ c[3] ^ k1;
  c[0] = x0;
  c[1] = b_lo;
  c[2] = x2;
  c[3] = a_lo;
}

void santa_oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {          /* key schedule: add the Weyl constants between rounds */
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    philox_round(c, k0, k1);
  }
  memcpy(out, c, sizeof c);
}

double santa_oracle_uniform(uint64_t seed, uint32_t b, uint32_t h, uint32_t step, uint32_t r) {
  const uint32_t ctr[4] = {r / 4u, h, b, step};
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t words[4];
  santa_oracle_philox4x32_10(ctr, key, words);
  return (double)(words[r % 4u] >> 8) * (1.0 / 16777216.0);
}

static int cmp_double(const void* a, const void* b) {
  const double x = *(const double*)a, y = *(const double*)b;
  return (x > y) - (x < y);
}

/* Sec. 2.1: iid draws t_j = u_j (with replacement, unordered, so sorted here);
 * independent stratified t_j = (j + u_j) / S with u_j independent;
 * systematic t_j = (j + u) / S with one u for all strata. */
void santa_oracle_thresholds(int32_t variant, int32_t S, uint64_t seed, uint32_t b, uint32_t h,
                             uint32_t step, double* t) {
  if (variant == ORACLE_SYSTEMATIC) {
    const double u = santa_oracle_uniform(seed, b, h, step, 0);
    for (int32_t j = 0; j < S; ++j) t[j] = ((double)j + u) / (double)S;
  } else if (variant == ORACLE_STRATIFIED) {
    for (int32_t j = 0; j < S; ++j)
      t[j] = ((double)j + santa_oracle_uniform(seed, b, h, step, (uint32_t)j)) / (double)S;
  } else {
    for (int32_t j = 0; j < S; ++j) t[j] = santa_oracle_uniform(seed, b, h, step, (uint32_t)j);
    qsort(t, (size_t)S, sizeof(double), cmp_double);
  }
}

/* ------------------------------------------------------------------ */
/* scores and softmax (Eq. 1)                                          */
/* ------------------------------------------------------------------ */

static int check_head(const oracle_problem* P, int32_t b, int32_t h) {
  if (!P || b < 0 || b >= P->batch || h < 0 || h >= P->n_q_heads) return -1;
  if (P->n_kv_heads <= 0 || P->n_q_heads % P->n_kv_heads) return -1;
  if (P->kv_offsets[b + 1] < P->kv_offsets[b]) return -1;
  return 0;
}

static int64_t nk_of(const oracle_problem* P, int32_t b) {
  return P->kv_offsets[b + 1] - P->kv_offsets[b];
}

int santa_oracle_scores(const oracle_problem* P, int32_t b, int32_t h, double* s, double* p) {
  if (check_head(P, b, h)) return -1;
  const int32_t d = P->head_dim, Hkv = P->n_kv_heads;
  const int32_t kvh = h / (P->n_q_heads / Hkv);
  const int64_t nk = nk_of(P, b), row0 = P->kv_offsets[b];
  const double scale = P->scale > 0.0 ? P->scale : 1.0 / sqrt((double)d);
  double* sc = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
  if (!sc) return -2;
  double qv[1024];
  if (d > 1024) { free(sc); return -1; }
  for (int32_t k = 0; k < d; ++k)
    qv[k] = load_elem(P->dtype, P->q, ((int64_t)b * P->n_q_heads + h) * d + k);
  for (int64_t n = 0; n < nk; ++n) {
    double dot = 0.0;
    const int64_t base = ((row0 + n) * Hkv + kvh) * (int64_t)d;
    for (int32_t k = 0; k < d; ++k) dot += qv[k] * load_elem(P->dtype, P->K, base + k);
    sc[n] = scale * dot;
  }
  if (s) memcpy(s, sc, sizeof(double) * (size_t)nk);
  if (p && nk > 0) {
    double m = sc[0];
    for (int64_t n = 1; n < nk; ++n) if (sc[n] > m) m = sc[n];
    double Z = 0.0;
    for (int64_t n = 0; n < nk; ++n) { p[n] = exp(sc[n] - m); Z += p[n]; }
    for (int64_t n = 0; n < nk; ++n) p[n] /= Z;
  }
  free(sc);
  return 0;
}

/* App. O, Alg. 3: per tile T_t, m_t = max s_n and l_t = sum exp(s_n - m_t). */
int santa_oracle_tile_stats(const oracle_problem* P, int32_t b, int32_t h, int32_t tile_len,
                            double* m, double* l) {
  if (check_head(P, b, h) || tile_len <= 0) return -1;
  const int64_t nk = nk_of(P, b);
  double* s = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
  if (!s) return -2;
  santa_oracle_scores(P, b, h, s, NULL);
  const int64_t T = (nk + tile_len - 1) / tile_len;
  for (int64_t t = 0; t < T; ++t) {
    const int64_t lo = t * tile_len, hi = (lo + tile_len < nk) ? lo + tile_len : nk;
    double mx = s[lo];
    for (int64_t n = lo + 1; n < hi; ++n) if (s[n] > mx) mx = s[n];
    double sum = 0.0;
    for (int64_t n = lo; n < hi; ++n) sum += exp(s[n] - mx);
    m[t] = mx;
    l[t] = sum;
  }
  free(s);
  return 0;
}

/* ------------------------------------------------------------------ */
/* inverse-CDF sampling and count-weighted gather (App. A.4, Eq. 4)    */
/* ------------------------------------------------------------------ */

int santa_oracle_sample_head(const oracle_problem* P, int32_t b, int32_t h, int32_t S,
                             const double* t, double* est, int32_t* J, double* delta) {
  if (check_head(P, b, h) || S <= 0) return -1;
  const int64_t nk = nk_of(P, b);
  if (nk <= 0) return -1;
  const int32_t d = P->head_dim, Hkv = P->n_kv_heads;
  const int32_t kvh = h / (P->n_q_heads / Hkv);
  const int64_t row0 = P->kv_offsets[b];
  double* p = (double*)malloc(sizeof(double) * (size_t)nk);
  double* F = (double*)malloc(sizeof(double) * (size_t)nk);
  int32_t* counts = (int32_t*)calloc((size_t)nk, sizeof(int32_t));
  if (!p || !F || !counts) { free(p); free(F); free(counts); return -2; }
  santa_oracle_scores(P, b, h, NULL, p);

  /* CDF over keys in index order */
  double run = 0.0;
  int64_t last_pos = 0;                       /* last key with nonzero mass */
  for (int64_t n = 0; n < nk; ++n) {
    run += p[n];
    F[n] = run;
    if (p[n] > 0.0) last_pos = n;
  }

  for (int32_t j = 0; j < S; ++j) {
    const double tj = t[j];
    /* J = #{n : F(n) <= t}: the first n with F(n) > t, so F(n-1) <= t < F(n) */
    int64_t lo = 0, hi = nk;
    while (lo < hi) {
      const int64_t mid = lo + (hi - lo) / 2;
      if (F[mid] <= tj) lo = mid + 1; else hi = mid;
    }
    int64_t n = lo;
    double dist;
    if (n >= nk) {                 /* t at or beyond the rounded total mass */
      n = last_pos;
      dist = 0.0;
    } else {
      const double left = n > 0 ? F[n - 1] : 0.0;
      const double a = tj - left, c = F[n] - tj;
      dist = a < c ? a : c;
    }
    counts[n] += 1;
    if (J) J[j] = (int32_t)n;
    if (delta) delta[j] = dist;
  }

  if (est) {
    for (int32_t k = 0; k < d; ++k) est[k] = 0.0;
    for (int64_t n = 0; n < nk; ++n) {
      if (!counts[n]) continue;
      const int64_t base = ((row0 + n) * Hkv + kvh) * (int64_t)d;
      for (int32_t k = 0; k < d; ++k) est[k] += (double)counts[n] * load_elem(P->dtype, P->V, base + k);
    }
    for (int32_t k = 0; k < d; ++k) est[k] *= 1.0 / (double)S;
  }
  free(p);
  free(F);
  free(counts);
  return 0;
}

/* Eq. (4) for a given index multiset: est = (1/S) * sum_j V[J_j]. */
int santa_oracle_gather(const oracle_problem* P, int32_t b, int32_t h, int32_t S, const int32_t* J,
                        double* est) {
  if (check_head(P, b, h) || S <= 0) return -1;
  const int64_t nk = nk_of(P, b);
  const int32_t d = P->head_dim, Hkv = P->n_kv_heads;
  const int32_t kvh = h / (P->n_q_heads / Hkv);
  const int64_t row0 = P->kv_offsets[b];
  for (int32_t k = 0; k < d; ++k) est[k] = 0.0;
  for (int32_t j = 0; j < S; ++j) {
    if (J[j] < 0 || J[j] >= nk) return -1;
    const int64_t base = ((row0 + J[j]) * Hkv + kvh) * (int64_t)d;
    for (int32_t k = 0; k < d; ++k) est[k] += load_elem(P->dtype, P->V, base + k);
  }
  for (int32_t k = 0; k < d; ++k) est[k] *= 1.0 / (double)S;
  return 0;
}

int santa_oracle_dense_head(const oracle_problem* P, int32_t b, int32_t h, double* out) {
  if (check_head(P, b, h)) return -1;
  const int64_t nk = nk_of(P, b);
  const int32_t d = P->head_dim, Hkv = P->n_kv_heads;
  const int32_t kvh = h / (P->n_q_heads / Hkv);
  const int64_t row0 = P->kv_offsets[b];
  for (int32_t k = 0; k < d; ++k) out[k] = 0.0;
  if (nk <= 0) return 0;
  double* p = (double*)malloc(sizeof(double) * (size_t)nk);
  if (!p) return -2;
  santa_oracle_scores(P, b, h, NULL, p);
  for (int64_t n = 0; n < nk; ++n) {
    const int64_t base = ((row0 + n) * Hkv + kvh) * (int64_t)d;
    for (int32_t k = 0; k < d; ++k) out[k] += p[n] * load_elem(P->dtype, P->V, base + k);
  }
  free(p);
  return 0;
}

/* ------------------------------------------------------------------ */
/* tile samplers: S2ANTA-prop (App. O, Alg. 2-5) and S2ANTA-flash       */
/* (App. P, Alg. 6-8)                                                   */
/* ------------------------------------------------------------------ */

/* App. O, Alg. 4: q_t = S W_t / Z, S_t = floor(q_t), and the
 * S - sum_t S_t samples left over go one each to the tiles with the largest
 * fractional parts q_t - S_t (largest remainder).  The pages do not say how
 * equal fractional parts are ordered: the lower tile index goes first. */
int santa_oracle_prop_budgets(int32_t T, const double* W, int32_t S, int32_t* St) {
  if (T <= 0 || S < 0 || !W || !St) return -1;
  double Z = 0.0;
  for (int32_t t = 0; t < T; ++t) {
    if (!(W[t] >= 0.0)) return -1;
    Z += W[t];
  }
  if (!(Z > 0.0)) return -1;
  double* frac = (double*)malloc(sizeof(double) * (size_t)T);
  if (!frac) return -2;
  int64_t given = 0;
  for (int32_t t = 0; t < T; ++t) {
    const double q = (double)S * W[t] / Z;
    St[t] = (int32_t)floor(q);
    frac[t] = q - (double)St[t];
    given += St[t];
  }
  for (int64_t left = (int64_t)S - given; left > 0; --left) {
    int32_t best = -1;
    for (int32_t t = 0; t < T; ++t)
      if (frac[t] >= 0.0 && (best < 0 || frac[t] > frac[best])) best = t;
    if (best < 0) break;
    St[best] += 1;
    frac[best] = -1.0;   /* one extra sample per tile at most */
  }
  free(frac);
  return 0;
}

/* Systematic counts inside one tile, App. O, Alg. 5 (and App. P,
 * Alg. 7): for the tile's keys in increasing order, x = inv_delta u_n,
 * c_n = floor(a0 + p + x) - floor(a0 + p), p <- p + x.  delta_n (if not NULL)
 * is the distance, in units of x, of the integers the key crossed to the
 * nearer end of its interval (a0 + p, a0 + p + x]; -1 where it crossed none. */
static void tile_counts(int64_t len, const double* u, double inv_delta, double a0, int32_t* c, double* dx) {
  double pacc = 0.0;
  for (int64_t n = 0; n < len; ++n) {
    const double x = inv_delta * u[n];
    const double lo = a0 + pacc, hi = a0 + pacc + x;
    c[n] = (int32_t)(floor(hi) - floor(lo));
    if (dx) {
      dx[n] = -1.0;
      if (c[n] > 0) {
        const double k_first = floor(lo) + 1.0, k_last = floor(hi);
        const double d1 = k_first - lo, d2 = hi - k_last;
        dx[n] = d1 < d2 ? d1 : d2;
      }
    }
    pacc += x;
  }
}

/* One head through a tile sampler.
 *   sampler 0, S2ANTA-prop: integer tile budgets S_t (Alg. 4), then the
 *     systematic counts of Alg. 5 with inv_delta_t = S_t / l_t; est =
 *     (1/S) sum_n c_n V_n (Alg. 2).
 *   sampler 1, S2ANTA-flash: the same budget S_tile in every tile (Alg. 6),
 *     per-tile counts with inv_delta_t = S_tile / l_t and partial
 *     O_t = sum_n c_n V_n (Alg. 7), merged as est = (1/Z) sum_t W_t O_t /
 *     S_tile, W_t = exp(m_t - m*) l_t, Z = sum_t W_t (Alg. 8).
 * Tiles are [t L, min((t + 1) L, nk)) for L = tile_len (Alg. 3); u_n =
 * exp(s_n - m_t).  a0_t is a0[t] when a0 is not NULL, else uniform number t
 * of head (b, h) (the pages draw a0 ~ U[0, 1) per head and tile and name no
 * generator).  Outputs (any may be NULL): est [d]; counts [nk_b]; delta
 * [nk_b], the counts' distance to an interval end in probability units
 * (x units times W_t / (Z budget_t)), -1 for keys with no draw; St [T] the
 * budgets. */
int santa_oracle_tiled_head(const oracle_problem* P, int32_t b, int32_t h, int32_t sampler, int32_t S,
                            int32_t tile_len, uint64_t seed, uint32_t step, const double* a0, double* est,
                            int32_t* counts, double* delta, int32_t* St) {
  if (check_head(P, b, h) || S <= 0 || tile_len <= 0 || (sampler != 0 && sampler != 1)) return -1;
  const int64_t nk = nk_of(P, b);
  if (nk <= 0) return -1;
  const int32_t d = P->head_dim, Hkv = P->n_kv_heads;
  const int32_t kvh = h / (P->n_q_heads / Hkv);
  const int64_t row0 = P->kv_offsets[b];
  const int64_t T = (nk + tile_len - 1) / tile_len;
  double* s = (double*)malloc(sizeof(double) * (size_t)nk);
  double* u = (double*)malloc(sizeof(double) * (size_t)nk);
  double* dx = (double*)malloc(sizeof(double) * (size_t)nk);
  int32_t* c = (int32_t*)malloc(sizeof(int32_t) * (size_t)nk);
  double* m = (double*)malloc(sizeof(double) * (size_t)T);
  double* l = (double*)malloc(sizeof(double) * (size_t)T);
  double* W = (double*)malloc(sizeof(double) * (size_t)T);
  int32_t* bud = (int32_t*)malloc(sizeof(int32_t) * (size_t)T);
  double* acc = (double*)calloc((size_t)d, sizeof(double));
  int rc = 0;
  if (!s || !u || !dx || !c || !m || !l || !W || !bud || !acc) { rc = -2; goto done; }
  santa_oracle_scores(P, b, h, s, NULL);
  /* Alg. 3: tile max, exp-sum, and the stash u */
  for (int64_t t = 0; t < T; ++t) {
    const int64_t lo = t * tile_len, hi = (lo + tile_len < nk) ? lo + tile_len : nk;
    double mx = s[lo];
    for (int64_t n = lo + 1; n < hi; ++n) if (s[n] > mx) mx = s[n];
    double sum = 0.0;
    for (int64_t n = lo; n < hi; ++n) { u[n] = exp(s[n] - mx); sum += u[n]; }
    m[t] = mx;
    l[t] = sum;
  }
  /* global max, tile masses W_t and Z (Alg. 4; Alg. 8) */
  double mstar = m[0];
  for (int64_t t = 1; t < T; ++t) if (m[t] > mstar) mstar = m[t];
  double Z = 0.0;
  for (int64_t t = 0; t < T; ++t) { W[t] = exp(m[t] - mstar) * l[t]; Z += W[t]; }
  if (sampler == 0) {
    if (santa_oracle_prop_budgets((int32_t)T, W, S, bud)) { rc = -1; goto done; }
  } else {
    /* S_tile ~ S / T, rounded half up, at least one sample per tile */
    int32_t st = (int32_t)floor((double)S / (double)T + 0.5);
    if (st < 1) st = 1;
    for (int64_t t = 0; t < T; ++t) bud[t] = st;
  }
  for (int64_t t = 0; t < T; ++t) {
    const int64_t lo = t * tile_len, hi = (lo + tile_len < nk) ? lo + tile_len : nk;
    const double inv_delta = bud[t] > 0 ? (double)bud[t] / l[t] : 0.0;
    const double a = a0 ? a0[t] : santa_oracle_uniform(seed, (uint32_t)b, (uint32_t)h, step, (uint32_t)t);
    tile_counts(hi - lo, u + lo, inv_delta, a, c + lo, dx + lo);
    /* this tile's sum_n c_n V_n, weighted for the estimate */
    const double wgt = sampler == 0 ? 1.0 / (double)S : (W[t] / Z) / (double)bud[t];
    for (int64_t n = lo; n < hi; ++n) {
      if (!c[n]) continue;
      const int64_t base = ((row0 + n) * Hkv + kvh) * (int64_t)d;
      for (int32_t k = 0; k < d; ++k) acc[k] += wgt * (double)c[n] * load_elem(P->dtype, P->V, base + k);
    }
    for (int64_t n = lo; n < hi; ++n)
      if (dx[n] >= 0.0) dx[n] *= W[t] / (Z * (double)bud[t]);
  }
  if (est) memcpy(est, acc, sizeof(double) * (size_t)d);
  if (counts) memcpy(counts, c, sizeof(int32_t) * (size_t)nk);
  if (delta) memcpy(delta, dx, sizeof(double) * (size_t)nk);
  if (St) memcpy(St, bud, sizeof(int32_t) * (size_t)T);
done:
  free(s); free(u); free(dx); free(c); free(m); free(l); free(W); free(bud); free(acc);
  return rc;
}

/* Whole step of a tile sampler over all (b, h): est [batch, H, d].  S_per_seq
 * (host, may be NULL) overrides S. */
int santa_oracle_tiled_decode(const oracle_problem* P, int32_t sampler, int32_t S, const int32_t* S_per_seq,
                              int32_t tile_len, uint64_t seed, uint32_t step, double* est, int32_t n_threads) {
  if (!P) return -1;
  const int32_t B = P->batch, H = P->n_q_heads, d = P->head_dim;
  int status = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
  for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
    const int32_t b = (int32_t)(bh / H), h = (int32_t)(bh % H);
    const int32_t Sb = S_per_seq ? S_per_seq[b] : S;
    if (santa_oracle_tiled_head(P, b, h, sampler, Sb, tile_len, seed, step, NULL, est + bh * d, NULL, NULL, NULL))
      status |= 1;
  }
  return status ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* Bernoulli qK^T with the mean group query (App. C, Eq. 8-13)          */
/* ------------------------------------------------------------------ */

/* fp32 -> bf16 bits, round to nearest even. */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);   /* NaN stays NaN */
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* fp32 -> IEEE binary16 bits, round to nearest even, with subnormals and
 * overflow to infinity. */
static uint16_t f32_to_fp16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  const uint32_t sign = (u >> 16) & 0x8000u, a = u & 0x7fffffffu;
  if (a > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);
  if (a >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u);   /* >= 65520 rounds to infinity */
  if (a < 0x33000000u) return (uint16_t)sign;                 /* < 2^-25 rounds to zero */
  const int e = (int)(a >> 23);
  uint32_t q, r, half;
  if (e < 113) {   /* below 2^-14: subnormal, value = m 2^(e-150) = h 2^-24 */
    const uint32_t m = (a & 0x7fffffu) | 0x800000u;
    const int s = 126 - e;   /* 14..24 */
    q = m >> s;
    r = m & ((1u << s) - 1u);
    half = 1u << (s - 1);
  } else {         /* normal: exponent e - 112, 10 mantissa bits */
    q = ((uint32_t)(e - 112) << 10) | ((a & 0x7fffffu) >> 13);
    r = a & 0x1fffu;
    half = 0x1000u;
  }
  if (r > half || (r == half && (q & 1u))) ++q;   /* a mantissa carry moves into the exponent */
  return (uint16_t)(sign | q);
}

void santa_oracle_store_elem(int32_t dtype, float x, void* out) {
  if (dtype == ORACLE_BF16) *(uint16_t*)out = f32_to_bf16_rne(x);
  else if (dtype == ORACLE_FP16) *(uint16_t*)out = f32_to_fp16_rne(x);
  else *(float*)out = x;
}

/* The effective queries of one GQA group under Bernoulli qK^T with the mean
 * group query (App. C.2):
 *   m_i = (1/G) sum_g |q_g,i|                                   (Eq. 10)
 *   b_i^(n) ~ Bernoulli(m_i / norm), norm = max_i m_i            (Eq. 11)
 *   m^_i = (norm / B) sum_n b_i^(n)                              (Eq. 12)
 *   q~_g,i = m^_i q_g,i / m_i, so that q~_g . K_n = (m^ o q_g / m) . K_n   (Eq. 13)
 * Stratified (App. C.1, Fig. 6): sample n of feature i is 1 when
 * (n + u)/B < m_i / norm, i.e. one uniform per stratum of [0, 1).
 * Arithmetic is fp32 in this fixed order (the pages fix no precision; the
 * decode consumes the queries in the cache dtype): m_i summed over g in
 * order then divided by G, p_i = m_i / norm, m^_i = (norm c_i) / B,
 * q~ = (m^_i q_g,i) / m_i rounded to the storage dtype; the Bernoulli tests
 * compare 24-bit uniforms exactly, a24 < p_i 2^24 (stratified:
 * n 2^24 + a24 < B p_i 2^24, exact in float64).  Uniform r = n d + i of the
 * group is word r % 4 of the Philox block at counter (r / 4, H + kvh, b,
 * step), a stream of its own beside the query heads' (0..H-1).
 * qt: storage dtype [G, d]; counts (may be NULL): [d] ones per feature. */
int santa_oracle_bernoulli_group(const oracle_problem* P, int32_t b, int32_t kvh, int32_t nsamp, int32_t stratified,
                                 uint64_t seed, uint32_t step, void* qt, int32_t* counts) {
  if (!P || b < 0 || b >= P->batch || kvh < 0 || kvh >= P->n_kv_heads || nsamp < 1 || nsamp > 1024) return -1;
  if (P->n_q_heads % P->n_kv_heads) return -1;
  const int32_t G = P->n_q_heads / P->n_kv_heads, d = P->head_dim, H = P->n_q_heads;
  const size_t es = P->dtype == ORACLE_FP32 ? 4 : 2;
  float* q = (float*)malloc(sizeof(float) * (size_t)G * d);
  float* m = (float*)malloc(sizeof(float) * (size_t)d);
  if (!q || !m) { free(q); free(m); return -2; }
  for (int32_t g = 0; g < G; ++g)
    for (int32_t i = 0; i < d; ++i)
      q[g * d + i] = (float)load_elem(P->dtype, P->q, ((int64_t)b * H + (int64_t)kvh * G + g) * d + i);
  float norm = 0.f;
  for (int32_t i = 0; i < d; ++i) {
    float acc = 0.f;
    for (int32_t g = 0; g < G; ++g) acc += fabsf(q[g * d + i]);
    m[i] = acc / (float)G;
    if (m[i] > norm) norm = m[i];
  }
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  for (int32_t i = 0; i < d; ++i) {
    int32_t c = 0;
    if (norm > 0.f && m[i] > 0.f) {
      const float pr = m[i] / norm;
      for (int32_t n = 0; n < nsamp; ++n) {
        const uint32_t r = (uint32_t)(n * d + i);
        const uint32_t ctr[4] = {r / 4, (uint32_t)(H + kvh), (uint32_t)b, step};
        uint32_t w[4];
        santa_oracle_philox4x32_10(ctr, key, w);
        const double a24 = (double)(w[r % 4] >> 8);
        const int hit = stratified ? ((double)n * 16777216.0 + a24 < (double)nsamp * (double)pr * 16777216.0)
                                   : (a24 < (double)pr * 16777216.0);
        c += hit;
      }
    }
    if (counts) counts[i] = c;
    const float mh = (norm * (float)c) / (float)nsamp;
    for (int32_t g = 0; g < G; ++g) {
      const float v = m[i] > 0.f ? (mh * q[g * d + i]) / m[i] : 0.f;
      santa_oracle_store_elem(P->dtype, v, (unsigned char*)qt + ((size_t)g * d + i) * es);
    }
  }
  free(q);
  free(m);
  return 0;
}

/* ------------------------------------------------------------------ */
/* whole decode step                                                    */
/* ------------------------------------------------------------------ */

int santa_oracle_decode(const oracle_problem* P, int32_t variant, int32_t S,
                        const int32_t* S_per_seq, int32_t S_stride, uint64_t seed, uint32_t step,
                        double* est, int32_t* J, double* delta, int32_t n_threads) {
  if (!P || variant < 0 || variant > 2) return -1;
  const int32_t B = P->batch, H = P->n_q_heads, d = P->head_dim;
  int status = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
  for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
    const int32_t b = (int32_t)(bh / H), h = (int32_t)(bh % H);
    const int32_t Sb = S_per_seq ? S_per_seq[b] : S;
    if (Sb <= 0 || Sb > S_stride) { status |= 1; continue; }
    double* t = (double*)malloc(sizeof(double) * (size_t)Sb);
    if (!t) { status |= 2; continue; }
    santa_oracle_thresholds(variant, Sb, seed, (uint32_t)b, (uint32_t)h, step, t);
    int32_t* Jrow = J ? J + bh * S_stride : NULL;
    double* drow = delta ? delta + bh * S_stride : NULL;
    if (santa_oracle_sample_head(P, b, h, Sb, t, est ? est + bh * d : NULL, Jrow, drow)) status |= 4;
    for (int32_t j = Sb; j < S_stride; ++j) {
      if (Jrow) Jrow[j] = -1;
      if (drow) drow[j] = -1.0;
    }
    free(t);
  }
  return status ? -1 : 0;
}

int santa_oracle_dense(const oracle_problem* P, double* out, int32_t n_threads) {
  if (!P) return -1;
  const int32_t B = P->batch, H = P->n_q_heads, d = P->head_dim;
  int status = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
  for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
    if (santa_oracle_dense_head(P, (int32_t)(bh / H), (int32_t)(bh % H), out + bh * d)) status |= 1;
  }
  return status ? -1 : 0;
}
