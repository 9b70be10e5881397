/*
 * santa.h -- C ABI of the GB300 (sm_103a) SANTA / S2ANTA decode-step attention
 * library (libsanta.so).
 *
 * The operator, per query head h of sequence b ("Stochastic Sparse Attention
 * for Memory-Bound Inference", arXiv:2605.01910):
 *   s_n = scale * q[b,h] . K[b,n,kvh]       scores over the whole key cache (Sec. 2, Eq. 1)
 *   A   = softmax(s)                         post-softmax distribution     (Sec. 2, Eq. 1)
 *   J_j = F^-1(t_j), j = 0..S-1              inverse-CDF draws              (App. A.4)
 *         t_j = u_j          (SANTA, i.i.d.; Eq. 4, Def. A.1)
 *         t_j = (j + u_j)/S  (S2ANTA-strat; Sec. 2.1)
 *         t_j = (j + u)/S    (S2ANTA-sys;   Sec. 2.1)
 *   out = (1/S) * sum_n c_n V[b,n,kvh]       count-weighted gather-and-add (Eq. 4, Fig. 1)
 * with kvh = h / (n_q_heads / n_kv_heads) (grouped-query attention).  The
 * uniforms u come from Philox4x32-10 (Salmon et al., SC'11): number r of head
 * (b, h) is word r%4 of the block at counter (r/4, h, b, step) under key
 * (seed_lo, seed_hi), mapped to [0,1) as (word >> 8) * 2^-24.  The pages name
 * no generator; this keying by (seed, batch, head, step) is this library's.
 *
 * Layouts (row-major, sequence-major caches as in App. Q of the paper):
 *   q    [batch, n_q_heads, head_dim]               dtype
 *   K, V [total_rows, n_kv_heads, head_dim]         dtype; rows of sequence b are
 *        [kv_offsets[b], kv_offsets[b+1]) (or [b*nk, (b+1)*nk) when kv_offsets is NULL)
 *   out  [batch, n_q_heads, head_dim]               float32
 *
 * Ownership and threading: the caller owns every buffer (device memory unless
 * stated) including the workspace; the library allocates nothing and keeps no
 * state outside the workspace.  All work is enqueued asynchronously on the
 * caller's stream; calls that share a workspace must be ordered on one stream.
 *
 * Errors: arguments are validated on the host before any launch and reported
 * as a status.  Conditions only visible on the device (a ragged length above
 * the stated bound or empty, a per-sequence budget out of range) set an error
 * word in the workspace (SANTA_DEVERR_* bits) and leave the heads of that
 * sequence zero; santa_get_error reports it.
 * Kernels never trap.
 */
#ifndef SANTA_H
#define SANTA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* santa_stream_t; /* identical to cudaStream_t */

typedef enum {
  SANTA_IID = 0,        /* SANTA: S i.i.d. draws from Categorical(A) (Eq. 4) */
  SANTA_STRATIFIED = 1, /* S2ANTA-strat: one independent draw per equal-mass stratum (Sec. 2.1) */
  SANTA_SYSTEMATIC = 2  /* S2ANTA-sys: one offset shared by all strata (Sec. 2.1) */
} santa_variant_t;

typedef enum { SANTA_BF16 = 0, SANTA_FP16 = 1, SANTA_FP32 = 2 } santa_dtype_t;

typedef enum {
  SANTA_OK = 0,
  SANTA_ERR_INVALID_ARG = 1, /* NULL pointer, bad shape, misalignment, S or nk out of range */
  SANTA_ERR_UNSUPPORTED = 2, /* head_dim / dtype / group size the library does not provide */
  SANTA_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned or smaller than *_workspace_size */
  SANTA_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, copy, sync) */
  SANTA_ERR_DEVICE = 5,      /* the device flagged bad ragged metadata (see santa_get_error) */
  SANTA_ERR_SCRATCH_LIMIT = 6 /* santa_decode_static: the problem needs more than SANTA_STATIC_SCRATCH_BYTES */
} santa_status_t;

typedef struct {
  int32_t batch;             /* >= 1 */
  int32_t n_q_heads;         /* H >= 1 */
  int32_t n_kv_heads;        /* H_kv >= 1, H % H_kv == 0, group H/H_kv <= 8 */
  int32_t head_dim;          /* 64 or 128 */
  int32_t dtype;             /* santa_dtype_t, shared by q, K and V */
  const int64_t* kv_offsets; /* device [batch+1] row offsets, non-decreasing from 0; NULL = uniform */
  int64_t nk;                /* keys per sequence; with kv_offsets, an upper bound on every nk_b */
  int32_t S;                 /* sample budget >= 1; with S_per_seq, an upper bound on every S_b */
  const int32_t* S_per_seq;  /* device [batch] budgets S_b in [1, S], or NULL */
  float scale;               /* score scale; <= 0 selects 1/sqrt(head_dim) (Eq. 1) */
  uint64_t seed;             /* Philox key */
  uint32_t step;             /* decode step, part of the Philox counter */
} santa_params_t;

/* Limits of the library. */
#define SANTA_MAX_S 4096        /* S (and every S_b) */
#define SANTA_MAX_NK (1 << 21)  /* keys per sequence */
#define SANTA_MAX_GROUP 8       /* n_q_heads / n_kv_heads */
#define SANTA_CHUNK 16          /* keys per statistics chunk */

/* Byte size of the workspace santa_decode needs for these parameters
 * (0 when the parameters are invalid).  The variant does not change it. */
size_t santa_workspace_size(const santa_params_t* p);

/* Clears the workspace's control word (the device error word).
 * Call once after allocating a workspace, before its first use. */
santa_status_t santa_workspace_init(void* workspace, size_t ws_bytes, santa_stream_t stream);

/* One S2ANTA / SANTA decode step (all of Sec. 2 / 2.1 above) on `stream`.
 *   q, K, V    device, 16-byte aligned, layouts above.
 *   out        device float32 [batch, n_q_heads, head_dim], overwritten.
 *   workspace  device, 256-byte aligned, >= santa_workspace_size(p) bytes.
 *   sample_idx optional device int32 [batch, n_q_heads, S]: the drawn key index
 *              (within its sequence) of every sorted threshold j; entries
 *              j >= S_b are -1.  NULL skips it.
 * Stages: score pass with per-chunk (max, exp-sum) and a score stash; per-head
 * combine into chunk mass prefixes and Philox thresholds; per-chunk inverse
 * CDF, GQA row union and V gather-add.  The drawn indices are a deterministic
 * function of (inputs, seed, step); the fp32 partial sums of the gather are
 * added into out in an unspecified order, so its last bits may vary between
 * runs. */
santa_status_t santa_decode(const santa_params_t* p, int32_t variant, const void* q, const void* K,
                            const void* V, float* out, void* workspace, size_t ws_bytes,
                            santa_stream_t stream, int32_t* sample_idx);

/* santa_decode with the K/V cache wholly or partly in host memory.  K and V
 * are each device memory or page-locked host memory (cudaHostAlloc /
 * cudaMallocHost, or host memory registered with cudaHostRegister), in the
 * K/V layout above and covering every row the offsets name; the GPU reads host
 * buffers in place through their mapped device addresses.  A step reads K in
 * full but, of V, only the drawn rows (Sec. 2.2, Eq. 4), so V can stay in
 * host memory at the cost of a few hundred row reads across the host link
 * while K stays in (or is copied to) device memory; both in host memory also
 * works.  q, out, workspace, sample_idx, kv_offsets and S_per_seq are device
 * memory as in santa_decode, and the drawn keys equal santa_decode's on the
 * same data.  Returns SANTA_ERR_INVALID_ARG, before any launch, when K or V is
 * neither memory of the current device nor page-locked host memory that the
 * device can address (pageable memory, for one). */
santa_status_t santa_decode_host_kv(const santa_params_t* p, int32_t variant, const void* q, const void* K,
                                    const void* V, float* out, void* workspace, size_t ws_bytes,
                                    santa_stream_t stream, int32_t* sample_idx);

/* santa_decode that also records stage_events[i] (cudaEvent_t, created by the
 * caller) on `stream` before stage i (0 score pass, 1 combine, 2 sample and
 * gather) and stage_events[3] after the last stage, so a caller can time each
 * stage on the launching stream.  stage_events may be NULL (then identical to
 * santa_decode). */
santa_status_t santa_decode_profiled(const santa_params_t* p, int32_t variant, const void* q, const void* K,
                                     const void* V, float* out, void* workspace, size_t ws_bytes,
                                     santa_stream_t stream, int32_t* sample_idx, void* const* stage_events);

/* Only the first stage of santa_decode: scores over the whole cache (Sec. 2,
 * Eq. 1) and the per-chunk statistics of App. O, Alg. 3, written to the
 * workspace (stash and tile statistics, see santa_workspace_layout).  Same
 * argument rules as santa_decode.  For timing or inspecting that stage. */
santa_status_t santa_score_pass(const santa_params_t* p, const void* q, const void* K, void* workspace,
                                size_t ws_bytes, santa_stream_t stream);

/* santa_decode with caller-supplied uniforms in place of Philox: device float64
 * u[batch, n_q_heads, S] in [0,1) (only u[...,0] is read for SANTA_SYSTEMATIC;
 * SANTA_IID sorts them at the 2^-24 resolution of the Philox uniforms).
 * For checking the sampler against hand-made cases such as the nk = 3 worked
 * example of Sec. 1 (Eq. 2-3). */
santa_status_t santa_decode_with_uniforms(const santa_params_t* p, int32_t variant, const void* q,
                                          const void* K, const void* V, const double* uniforms,
                                          float* out, void* workspace, size_t ws_bytes,
                                          santa_stream_t stream, int32_t* sample_idx);

/* Exact decode attention softmax(q K^T * scale) V (Eq. 1) by split-KV partials
 * (max, exp-sum, partial output) per 256-key chunk and a per-head merge.  This
 * library's own dense comparator.  Same argument rules as santa_decode;
 * S, S_per_seq, seed and step are ignored. */
size_t santa_dense_workspace_size(const santa_params_t* p);
santa_status_t santa_dense_decode(const santa_params_t* p, const void* q, const void* K, const void* V,
                                  float* out, void* workspace, size_t ws_bytes, santa_stream_t stream);

/* The pages' tile samplers ("Stochastic Sparse Attention for Memory-Bound
 * Inference", Sec. 3.2-3.3): the keys of each sequence are cut into tiles of
 * tile_len keys, [t L, min((t + 1) L, nk_b)).
 *   SANTA_TILE_PROP   S2ANTA-prop (App. O, Alg. 2-5): integer tile budgets
 *                     S_t ~ S W_t / Z by largest remainder (equal fractional
 *                     parts: the lower tile first), systematic counts inside
 *                     each tile, out = (1/S_b) sum_n c_n V_n.
 *   SANTA_TILE_FLASH  S2ANTA-flash (App. P, Alg. 6-8): every tile draws
 *                     S_tile = max(1, round(S_b / T_b)) samples as if it held
 *                     all the mass; out = (1/Z) sum_t W_t O_t / S_tile with O_t
 *                     the tile's sum_n c_n V_n and W_t its mass.
 * Inside tile t the count rule is the pages' c_n = floor(a0 + p + x_n) -
 * floor(a0 + p), x_n = S_t exp(s_n - m_t) / l_t: key n takes the integers in
 * (a0 + p, a0 + p + x_n].  a0 of tile t is uniform number t of the head in
 * the Philox layout above (the pages name no generator).  Both run the
 * score pass of santa_decode first.
 *   tile_len   a multiple of SANTA_CHUNK in [SANTA_CHUNK, SANTA_MAX_TILE].
 *   sample_idx optional device int32 [batch, n_q_heads, santa_tiled_max_draws]:
 *              the drawn key index of every draw, tiles in order and keys
 *              increasing inside a tile (prop: S_b draws; flash: T_b S_tile),
 *              the rest -1.
 * Other arguments and rules as santa_decode; the workspace must hold
 * santa_tiled_workspace_size bytes (0 for invalid arguments).  The output is
 * summed in a fixed order: equal inputs give equal bits. */
#define SANTA_TILE_PROP 0
#define SANTA_TILE_FLASH 1
#define SANTA_MAX_TILE 1024
size_t santa_tiled_workspace_size(const santa_params_t* p, int32_t sampler, int32_t tile_len);
int32_t santa_tiled_max_draws(const santa_params_t* p, int32_t sampler, int32_t tile_len);
santa_status_t santa_decode_tiled(const santa_params_t* p, int32_t sampler, int32_t tile_len, const void* q,
                                  const void* K, const void* V, float* out, void* workspace, size_t ws_bytes,
                                  santa_stream_t stream, int32_t* sample_idx);

/* santa_decode on Bernoulli qK^T scores with the mean group query ("Stochastic
 * Sparse Attention for Memory-Bound Inference", Sec. 5.1, App. C.2, Eq. 10-13).
 * For each (sequence, KV head) group: m_i = mean_g |q_g,i|, norm = max_i m_i,
 * c_i of n_samples Bernoulli(m_i / norm) draws are one (stratified != 0: draw
 * n is one when (n + u)/n_samples < m_i / norm, one uniform per stratum,
 * App. C.1), m^_i = norm c_i / n_samples, and each head's query becomes
 * q~_g,i = m^_i q_g,i / m_i (fp32, rounded to nearest even into the cache
 * dtype); the step then runs as santa_decode on q~ (features with c_i = 0
 * multiply zero in every head of the group).  Uniform r = n d + i of a group
 * is word r % 4 of the Philox block at counter (r / 4, n_q_heads + kvh, b, step).
 *   n_samples       1..1024
 *   feature_counts  optional device int32 [batch, n_kv_heads, head_dim]: c_i.
 * The workspace must hold santa_bernoulli_workspace_size(p) bytes; the
 * effective queries are left in it, [batch, n_q_heads, head_dim] in the cache
 * dtype, starting at byte santa_workspace_size(p) rounded up to 256.  Other
 * arguments, results and errors as santa_decode. */
size_t santa_bernoulli_workspace_size(const santa_params_t* p);
santa_status_t santa_decode_bernoulli(const santa_params_t* p, int32_t variant, int32_t n_samples, int32_t stratified,
                                      const void* q, const void* K, const void* V, float* out, void* workspace,
                                      size_t ws_bytes, santa_stream_t stream, int32_t* sample_idx,
                                      int32_t* feature_counts);

/* Byte offsets of the intermediate arrays inside a santa_decode workspace, for
 * inspection by tests and tools after the stream has synchronised:
 *   stash     float32 [batch, n_q_heads, nk]        scaled scores s_n
 *   tile_max  float32 [batch, n_q_heads, chunks]    per-chunk max of s_n
 *   tile_sum  float32 [batch, n_q_heads, chunks]    per-chunk sum of exp(s_n - tile_max)
 *   prefix    int64   [batch, n_q_heads, chunks+1]  chunk mass prefix in units of 2^-40 of the
 *                                                   head-max key's mass (exact integer sums)
 *   thresh    int64   [batch, n_q_heads, S]         sorted thresholds t_j * Z, same units
 *   head_max  float32 [batch, n_q_heads]            max_n s_n
 * with chunks = ceil(nk / SANTA_CHUNK).  Returns 0 on success. */
typedef struct {
  size_t stash, tile_max, tile_sum, prefix, thresh, head_max;
  int64_t chunks;
} santa_ws_layout_t;
int32_t santa_workspace_layout(const santa_params_t* p, santa_ws_layout_t* layout);

/* Bits of the device error word (the *code of santa_get_error).  A flagged
 * sequence's heads come out zero; the other sequences are computed as usual. */
#define SANTA_DEVERR_NK_BOUND 1 /* nk_b = kv_offsets[b+1] - kv_offsets[b] above p->nk, or kv_offsets[b] < 0 */
#define SANTA_DEVERR_S_RANGE 2  /* S_per_seq[b] outside [1, S] */
#define SANTA_DEVERR_EMPTY 4    /* a sequence with no keys (nk_b < 1): its softmax is undefined */
#define SANTA_DEVERR_TIMEOUT 8  /* a bounded grid-wide wait ran out (the single-launch paths) */

/* Synchronises `stream`, reads and clears the workspace error word.
 * Returns SANTA_OK, SANTA_ERR_DEVICE (device flagged bad metadata; *code gets
 * the SANTA_DEVERR_* bits when code != NULL) or SANTA_ERR_CUDA. */
santa_status_t santa_get_error(void* workspace, santa_stream_t stream, int32_t* code);

/* santa_decode without a caller-supplied workspace, for callers that cannot
 * allocate device memory: for example a plug-in that its host framework hands
 * only tensors and a stream (all device memory belongs to the framework's own
 * pool), or code that must not call cudaMalloc in the middle of a run because
 * the call synchronises the device and may fail once the pool holds the rest
 * of the GPU.  The paper has no counterpart; this entry point is a property of
 * this library's interface, not of the method.
 *
 * Arguments, layouts and results are those of santa_decode.  The workspace is
 * a fixed array of SANTA_STATIC_SCRATCH_BYTES bytes in the library's own
 * device memory, held by each device from the moment the array's module is
 * loaded there until the process exits.  Under CUDA's default lazy module
 * loading (CUDA_MODULE_LOADING=LAZY) that happens at the first lookup of the
 * array's address on the device: the one implicit device allocation (8 MiB)
 * this entry point makes.  Call santa_static_warmup() once per device at
 * startup (before the framework's pool takes the device, and before any
 * stream capture), or run with CUDA_MODULE_LOADING=EAGER; after that no call
 * allocates.  Problems whose santa_workspace_size exceeds the array are
 * rejected with SANTA_ERR_SCRATCH_LIMIT, invalid parameters, variants and
 * buffers with santa_decode's statuses, all before any CUDA call.  Every call
 * looks up the array's address on the current device again (host-side), so
 * nothing stale survives a device reset.  Each call clears the array's error word on `stream` first;
 * ragged metadata the device rejects leaves those heads' outputs zero (and
 * their sample_idx entries -1), as in santa_decode, but the flag itself is not
 * reported here (use santa_decode with a workspace and santa_get_error).
 * All calls share the one array, which keeps the last call's contents: calls
 * whose work overlaps on the GPU (different streams, or several host threads
 * without ordering) race on it and give wrong results. */
#define SANTA_STATIC_SCRATCH_BYTES ((size_t)8 << 20)
santa_status_t santa_decode_static(const santa_params_t* p, int32_t variant, const void* q, const void* K,
                                   const void* V, float* out, santa_stream_t stream, int32_t* sample_idx);
/* Loads santa_decode_static's array on the current device (the lookup of its
 * address: under lazy module loading, an 8 MiB device allocation the first
 * time on each device) and returns SANTA_OK, or SANTA_ERR_CUDA when the
 * device cannot hold it.  Launches nothing; safe to call again. */
santa_status_t santa_static_warmup(void);

/* Measurement helper, not part of the method: reads `bytes` bytes at `src`
 * (device, 16-byte aligned, a multiple of 16) once with 16-byte
 * non-allocating loads, 2 CTAs of 512 threads per SM, on `stream`, and writes
 * one word per thread to `sink` (device, santa_read_probe_sink_words()
 * uint32 words).  Timed by the caller, it gives the read ceiling of a transfer
 * of that size (launch, ramp and tail included) beside a kernel's roofline. */
int32_t santa_read_probe_sink_words(void);
santa_status_t santa_read_probe(const void* src, size_t bytes, uint32_t* sink, santa_stream_t stream);

/* Self-test of the bounded grid-barrier wait (no counterpart in the paper):
 * one CTA waits on the workspace's barrier generation word, which nothing
 * advances, for limit_ns nanoseconds (1 ms .. 2 s) of %globaltimer time; the
 * wait must then end with SANTA_DEVERR_TIMEOUT in the workspace error word, read
 * by santa_get_error, and the GPU context stays usable.  The workspace (at
 * least 256 bytes, initialised) must not be in use by a decode meanwhile. */
santa_status_t santa_selftest_wait_timeout(void* workspace, size_t ws_bytes, uint64_t limit_ns,
                                           santa_stream_t stream);

/* Static description of a status code. */
const char* santa_status_string(santa_status_t status);

/* Library version, major*10000 + minor*100 + patch. */
int32_t santa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SANTA_H */
