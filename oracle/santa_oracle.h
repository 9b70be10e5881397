/*
 * santa_oracle.h -- CPU reference ("oracle") for SANTA / S2ANTA decode-step
 * attention.  TEST INFRASTRUCTURE: only the tests, the smoke check and the
 * benchmark's CPU-baseline leg use this library.  It shares no code with the
 * CUDA library and is not part of the product path.
 *
 * Everything is computed in float64 from the same storage bytes the GPU reads
 * (bf16 / fp16 / fp32 widened exactly).  Sources, all from "Stochastic Sparse
 * Attention for Memory-Bound Inference" (arXiv:2605.01910):
 *   scores + softmax ........ Sec. 2, Eq. (1)
 *   i.i.d. estimator ........ Sec. 2, Eq. (4); App. A, Def. A.1
 *   stratified / systematic . Sec. 2.1 ("Construction")
 *   inverse CDF ............. App. A.4, the indicator 1{F(j-1) <= t < F(j)}
 *   tile statistics ......... App. O, Algorithm 3 (per-tile max and exp-sum)
 *   S2ANTA-prop ............. App. O, Algorithms 2, 4, 5 (largest-remainder
 *                             tile budgets, per-tile systematic counts)
 *   S2ANTA-flash ............ App. P, Algorithms 6-8 (uniform tile budgets,
 *                             merge weighted by the tile masses)
 *   Bernoulli qK^T .......... App. C, Eq. (8)-(13) (mean group query)
 * The Philox4x32-10 generator follows Salmon, Moraes, Dror, Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3" (SC'11); the pages name no generator.
 */
#ifndef SANTA_ORACLE_H
#define SANTA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_BF16 = 0, ORACLE_FP16 = 1, ORACLE_FP32 = 2 };
enum { ORACLE_IID = 0, ORACLE_STRATIFIED = 1, ORACLE_SYSTEMATIC = 2 };

typedef struct {
  int32_t dtype;            /* ORACLE_BF16 / ORACLE_FP16 / ORACLE_FP32 */
  int32_t batch;
  int32_t n_q_heads;
  int32_t n_kv_heads;       /* n_q_heads % n_kv_heads == 0 */
  int32_t head_dim;
  const int64_t* kv_offsets;/* host [batch + 1]: rows of sequence b are [off[b], off[b+1]) */
  const void* q;            /* [batch, n_q_heads, head_dim] */
  const void* K;            /* [off[batch], n_kv_heads, head_dim] */
  const void* V;            /* same layout as K */
  double scale;             /* <= 0 selects 1/sqrt(head_dim) */
} oracle_problem;

/* Philox4x32-10: one 128-bit block for counter ctr and key. */
void santa_oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* Uniform number r of head (b, h): word r%4 of block r/4 at counter
 * (r/4, h, b, step), key (seed_lo, seed_hi), mapped as (x >> 8) * 2^-24. */
double santa_oracle_uniform(uint64_t seed, uint32_t b, uint32_t h, uint32_t step, uint32_t r);

/* The S sorted thresholds t_j in [0,1) of one head for a variant. */
void santa_oracle_thresholds(int32_t variant, int32_t S, uint64_t seed, uint32_t b, uint32_t h,
                             uint32_t step, double* t);

/* Scaled scores s_n and softmax probabilities p_n of one head (nk_b each; either may be NULL). */
int santa_oracle_scores(const oracle_problem* P, int32_t b, int32_t h, double* s, double* p);

/* Per-tile max m_t and exp-sum l_t over tiles of length tile_len (ceil(nk_b/tile_len) each). */
int santa_oracle_tile_stats(const oracle_problem* P, int32_t b, int32_t h, int32_t tile_len,
                            double* m, double* l);

/* Inverse-CDF sampling of one head for S given thresholds t (in [0,1), any order):
 * J[j] = F^-1(t[j]); est = (1/S) sum_j V[J[j]]; delta[j] = distance of t[j] to the nearer
 * edge of its CDF interval (0 when the draw had to be clamped).  Any output may be NULL. */
int santa_oracle_sample_head(const oracle_problem* P, int32_t b, int32_t h, int32_t S,
                             const double* t, double* est, int32_t* J, double* delta);

/* Eq. (4) for a given index multiset J[0..S): est = (1/S) sum_j V[J_j]. */
int santa_oracle_gather(const oracle_problem* P, int32_t b, int32_t h, int32_t S, const int32_t* J,
                        double* est);

/* Exact attention of one head: sum_n p_n V_n. */
int santa_oracle_dense_head(const oracle_problem* P, int32_t b, int32_t h, double* out);

/* Largest-remainder integer budgets (App. O, Alg. 4): St[t] in {floor, ceil}
 * of S W_t / Z with sum S; equal fractional parts favour the lower index. */
int santa_oracle_prop_budgets(int32_t T, const double* W, int32_t S, int32_t* St);

/* One head through a tile sampler: sampler 0 = S2ANTA-prop (App. O, Alg. 2-5),
 * 1 = S2ANTA-flash (App. P, Alg. 6-8), tiles of tile_len keys.  a0 [T] (may be
 * NULL: uniform number t of the head) are the per-tile offsets.  Outputs (any
 * may be NULL): est [d]; counts [nk_b]; delta [nk_b] (probability-unit
 * distance of a key's draws to its interval ends, -1 if none); St [T]. */
int santa_oracle_tiled_head(const oracle_problem* P, int32_t b, int32_t h, int32_t sampler, int32_t S,
                            int32_t tile_len, uint64_t seed, uint32_t step, const double* a0, double* est,
                            int32_t* counts, double* delta, int32_t* St);

/* Whole step of a tile sampler: est [batch, H, d]. */
int santa_oracle_tiled_decode(const oracle_problem* P, int32_t sampler, int32_t S, const int32_t* S_per_seq,
                              int32_t tile_len, uint64_t seed, uint32_t step, double* est, int32_t n_threads);

/* Storage rounding: fp32 x to the dtype (bf16 / fp16 round to nearest even). */
void santa_oracle_store_elem(int32_t dtype, float x, void* out);

/* Bernoulli qK^T with the mean group query (App. C.2, Eq. 10-13): the
 * effective queries q~ [G, d] (storage dtype) of the group of KV head kvh,
 * from nsamp Bernoulli samples per feature (stratified != 0: one uniform per
 * stratum, App. C.1).  counts [d] (may be NULL) gets the ones per feature. */
int santa_oracle_bernoulli_group(const oracle_problem* P, int32_t b, int32_t kvh, int32_t nsamp, int32_t stratified,
                                 uint64_t seed, uint32_t step, void* qt, int32_t* counts);

/* Full decode step over all (b, h).  S_per_seq (host, may be NULL) overrides S.
 * est: [batch, H, d]; J / delta: [batch, H, S_stride] (entries j >= S_b get -1).
 * n_threads <= 0 uses the OpenMP default. */
int santa_oracle_decode(const oracle_problem* P, int32_t variant, int32_t S,
                        const int32_t* S_per_seq, int32_t S_stride, uint64_t seed, uint32_t step,
                        double* est, int32_t* J, double* delta, int32_t n_threads);

/* Exact attention for all (b, h): out [batch, H, d]. */
int santa_oracle_dense(const oracle_problem* P, double* out, int32_t n_threads);

#ifdef __cplusplus
}
#endif
#endif
