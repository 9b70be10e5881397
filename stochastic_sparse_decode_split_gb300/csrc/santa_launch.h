// santa_launch.h -- internal interface between the C ABI (santa_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#define SANTA_MAX_GROUP_DEV 8

namespace santa {

constexpr int MAX_CTAS = 160;   // bound on the single-launch grid (aggregate slots per head)
constexpr int MAX_S = 4096;     // largest sample budget (SANTA_MAX_S)

// Everything one decode call needs, already validated and carved out of the workspace.
struct LaunchArgs {
  int dtype;       // 0 bf16, 1 fp16, 2 fp32
  int D;           // head_dim (64 or 128)
  int B, H, Hkv;
  int W;           // single-launch decode: KV heads per work unit (chosen by launch_fused)
  int64_t nk_max;
  int chunks_max;  // santa: ceil(nk_max / SUB) statistics chunks; dense: ceil(nk_max / DCHUNK)
  int groups_max;  // santa: ceil(ceil(nk_max / WIN) / SPC) sampler CTAs per (b, kv head)
  int tiles_max;   // ceil(nk_max / TILE) score-pass tiles per (b, kv head)
  int num_sms;     // streaming multiprocessors of the device (persistent grid size)
  int k_host;      // K is page-locked host memory read in place (no TMA on it)
  int score_only;  // single launch: the score pass alone (stash and 16-key statistics), then exit
  // single-launch partition of uniform batches, computed by the launcher
  // (blk_total = 0: ragged, the kernel computes it): total 16-key blocks and
  // blk_total = blk_q * grid + blk_r
  long long blk_total, blk_q;
  int blk_r;
  // uniform batch: multiply-high reciprocals of H_kv * blocks per sequence,
  // blocks per sequence and the grid (division by invariant integers, for
  // 32-bit dividends; 0 for a divisor of 1)
  unsigned long long rdiv_perb, rdiv_nblk, rdiv_grid;
  int S_max;
  int variant;
  float scale;
  uint64_t seed;
  uint32_t step;
  const void* q;
  const void* K;
  const void* V;
  const int64_t* kv_offsets;
  const int32_t* S_per_seq;
  const double* uniforms;  // optional debug uniforms [B, H, S_max]
  float* out;
  int32_t* sample_idx;     // optional [B, H, S_max]
  // workspace views
  int* err;
  float* stash;            // [B, H, nk_max]
  float* tile_max;         // [B, H, chunks_max]
  float* tile_sum;         // [B, H, chunks_max]
  long long* prefix;       // [B, H, chunks_max + 1] chunk-mass prefix, units of 2^-40 of the head max
  long long* thresh;       // [B, H, S_max] sorted thresholds, same units
  int32_t* jstart;         // [B, H, chunks_max + 1]
  float* head_max;         // [B, H]
  float* part_o;           // dense: [B, H, chunks_max, D] chunk partial outputs
  float* fpart;            // dense, one launch: [MAX_CTAS][2] partials of shared pieces (santa_flash.cuh)
  // single-launch decode
  void* agg;               // [B, H, MAX_CTAS] per-CTA aggregates (16 bytes each, see santa_fused.cu)
  uint32_t* ukeys;         // [B, H, S_max] sorted 24-bit uniform keys (i.i.d.)
  unsigned long long* rcp_S;  // [B] ceil(2^64 / S_b)
  // tile samplers (S2ANTA-prop / S2ANTA-flash)
  int tl_sampler;          // 0 prop, 1 flash
  int tl_len;              // keys per tile (a multiple of SUB, <= TL_MAX_LEN)
  int tl_T;                // tiles of the longest sequence
  int tl_draws;            // row length of sample_idx
  int32_t* tl_pre;         // [B, H, tl_T + 1] prop: exclusive prefix of the tile budgets
  double* tl_w;            // [B, H, tl_T] scratch: tile masses
  float* tl_o;             // [B, H, tl_T, D] flash: per-tile sums of count x V
  cudaStream_t stream;
};

cudaError_t launch_score(const LaunchArgs& a);
cudaError_t launch_combine(const LaunchArgs& a);
cudaError_t launch_sample_gather(const LaunchArgs& a);
cudaError_t launch_dense(const LaunchArgs& a);
// Dense decode in one cooperative launch (16-bit caches, group <= 8);
// cudaErrorNotSupported for the shapes it does not cover.
cudaError_t launch_flash(const LaunchArgs& a, unsigned* bar_count, unsigned* bar_gen);
size_t flash_part_bytes(int D);   // workspace bytes of its shared-piece partials
// The whole decode step in one cooperative launch (16-bit caches, Philox uniforms).
cudaError_t launch_fused(const LaunchArgs& a, unsigned* bar_count, unsigned* bar_gen);
constexpr int TL_MAX_LEN = 1024;   // longest tile of the tile samplers
cudaError_t launch_tiled(const LaunchArgs& a);   // after launch_score
// Bernoulli qK^T effective queries qt [B, H, D] (cache dtype) from a.q; counts [B, Hkv, D] may be NULL.
cudaError_t launch_wait_timeout_selftest(const unsigned* gen, int* err, unsigned long long limit_ns,
                                         cudaStream_t stream);
cudaError_t launch_read_probe(const void* src, size_t bytes, uint32_t* sink, int ctas, cudaStream_t stream);
cudaError_t launch_bernoulli_query(const LaunchArgs& a, void* qt, int32_t* counts, int nsamp, int stratified);

}  // namespace santa
