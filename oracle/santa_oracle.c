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
