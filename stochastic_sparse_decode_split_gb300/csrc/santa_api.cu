// santa_api.cu -- C ABI of libsanta.so: host-side validation, workspace
// layout and the launch sequence of one decode step.  Every check here runs
// before any CUDA call, so argument errors never reach the device.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "../../include/santa.h"
#include "santa_common.cuh"
#include "santa_launch.h"

static_assert(SANTA_MAX_GROUP == SANTA_MAX_GROUP_DEV, "group limit");
static_assert(SANTA_MAX_S == santa::MAX_S, "sample budget limit");
static_assert(SANTA_CHUNK == santa::SUB, "chunk length");
static_assert(SANTA_MAX_TILE == santa::TL_MAX_LEN, "tile length");
static_assert(SANTA_DEVERR_NK_BOUND == santa::ERR_NK_BOUND && SANTA_DEVERR_S_RANGE == santa::ERR_S_RANGE &&
                  SANTA_DEVERR_EMPTY == santa::ERR_EMPTY && SANTA_DEVERR_TIMEOUT == santa::ERR_TIMEOUT,
              "device error bits");

namespace {

constexpr size_t ALIGN = 256;
constexpr size_t HEADER = 256;  // error word, grid-barrier arrival counters and generation, padding
// header offsets of the grid-barrier words: arrival counters at 64 and 192
// (the second at the first + 32 words), generation at 128
constexpr size_t BAR_COUNT = 64, BAR_GEN = 128;

size_t up(size_t x) { return (x + ALIGN - 1) / ALIGN * ALIGN; }

struct Layout {
  size_t stash, tile_max, tile_sum, prefix, thresh, jstart, head_max, part_o, fpart, agg, ukeys, rcp_S, total;
  size_t tl_pre, tl_w, tl_o;
  int64_t tl_T;
  int64_t chunks, groups;
};

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Multiprocessor count of the current device, cached per device.
int device_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cached[dev] = n;
  return n;
}

santa_status_t check_params(const santa_params_t* p, bool need_S) {
  if (!p) return SANTA_ERR_INVALID_ARG;
  if (p->batch < 1 || p->n_q_heads < 1 || p->n_kv_heads < 1) return SANTA_ERR_INVALID_ARG;
  if (p->n_q_heads % p->n_kv_heads) return SANTA_ERR_INVALID_ARG;
  if (p->batch > 65535 || p->n_kv_heads > 65535 || p->n_q_heads > 65535) return SANTA_ERR_INVALID_ARG;
  if (p->nk < 1 || p->nk > SANTA_MAX_NK) return SANTA_ERR_INVALID_ARG;
  if (p->dtype < SANTA_BF16 || p->dtype > SANTA_FP32) return SANTA_ERR_UNSUPPORTED;
  if (p->head_dim != 64 && p->head_dim != 128) return SANTA_ERR_UNSUPPORTED;
  if (p->n_q_heads / p->n_kv_heads > SANTA_MAX_GROUP) return SANTA_ERR_UNSUPPORTED;
  if (need_S && (p->S < 1 || p->S > SANTA_MAX_S)) return SANTA_ERR_INVALID_ARG;
  if (!(p->scale == p->scale) || isinf(p->scale)) return SANTA_ERR_INVALID_ARG;
  return SANTA_OK;
}

Layout santa_layout(const santa_params_t* p) {
  Layout L;
  const size_t B = (size_t)p->batch, H = (size_t)p->n_q_heads;
  const size_t nk = (size_t)p->nk, S = (size_t)p->S;
  L.chunks = (p->nk + SANTA_CHUNK - 1) / SANTA_CHUNK;
  L.groups = ((p->nk + santa::WIN - 1) / santa::WIN + santa::SPC - 1) / santa::SPC;
  size_t off = HEADER;
  L.stash = off;    off += up(B * H * nk * sizeof(float));
  L.tile_max = off; off += up(B * H * (size_t)L.chunks * sizeof(float));
  L.tile_sum = off; off += up(B * H * (size_t)L.chunks * sizeof(float));
  L.prefix = off;   off += up(B * H * ((size_t)L.chunks + 1) * sizeof(long long));
  L.thresh = off;   off += up(B * H * S * sizeof(long long));
  L.jstart = off;   off += up(B * H * ((size_t)L.chunks + 1) * sizeof(int32_t));
  L.head_max = off; off += up(B * H * sizeof(float));
  L.agg = off;      off += up(B * H * santa::MAX_CTAS * 16);
  L.ukeys = off;    off += up(B * H * S * sizeof(uint32_t));
  L.rcp_S = off;    off += up(B * sizeof(unsigned long long));
  L.part_o = 0;
  L.total = off;
  return L;
}

// santa_layout followed by the tile samplers' arrays (tl_T = tiles of the longest sequence).
Layout tiled_layout(const santa_params_t* p, int32_t tile_len) {
  Layout L = santa_layout(p);
  const size_t B = (size_t)p->batch, H = (size_t)p->n_q_heads, D = (size_t)p->head_dim;
  L.tl_T = (p->nk + tile_len - 1) / tile_len;
  const size_t T = (size_t)L.tl_T;
  size_t off = L.total;
  L.tl_pre = off; off += up(B * H * (T + 1) * sizeof(int32_t));
  L.tl_w = off;   off += up(B * H * 2 * T * sizeof(double));
  L.tl_o = off;   off += up(B * H * T * D * sizeof(float));
  L.total = off;
  return L;
}

santa_status_t check_tiled(const santa_params_t* p, int32_t sampler, int32_t tile_len) {
  santa_status_t st = check_params(p, true);
  if (st != SANTA_OK) return st;
  if (sampler != SANTA_TILE_PROP && sampler != SANTA_TILE_FLASH) return SANTA_ERR_INVALID_ARG;
  if (tile_len < SANTA_CHUNK || tile_len > SANTA_MAX_TILE || tile_len % SANTA_CHUNK) return SANTA_ERR_INVALID_ARG;
  const int64_t T = (p->nk + tile_len - 1) / tile_len;
  if (T * (int64_t)p->batch * p->n_kv_heads > INT32_MAX) return SANTA_ERR_UNSUPPORTED;   // one CTA per tile
  return SANTA_OK;
}

int32_t tiled_draws(const santa_params_t* p, int32_t sampler, int32_t tile_len) {
  const int64_t T = (p->nk + tile_len - 1) / tile_len;
  // flash: T_b round(S_b / T_b) <= S + T_b / 2, and T_b when S_b / T_b < 1/2
  return sampler == SANTA_TILE_PROP ? p->S : (int32_t)(p->S + T);
}

Layout dense_layout(const santa_params_t* p) {
  Layout L;
  memset(&L, 0, sizeof L);
  const size_t B = (size_t)p->batch, H = (size_t)p->n_q_heads, D = (size_t)p->head_dim;
  L.chunks = (p->nk + santa::DCHUNK - 1) / santa::DCHUNK;
  size_t off = HEADER;
  L.tile_max = off; off += up(B * H * (size_t)L.chunks * sizeof(float));
  L.tile_sum = off; off += up(B * H * (size_t)L.chunks * sizeof(float));
  L.part_o = off;   off += up(B * H * (size_t)L.chunks * D * sizeof(float));
  L.fpart = off;    off += up(santa::flash_part_bytes((int)D));
  L.total = off;
  return L;
}

santa_status_t check_buffers(const void* q, const void* K, const void* V, const void* out, const void* ws,
                             size_t ws_bytes, size_t need) {
  if (!q || !K || !V || !out) return SANTA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(out, 16)) return SANTA_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, ALIGN) || ws_bytes < need) return SANTA_ERR_WORKSPACE;
  return SANTA_OK;
}

santa::LaunchArgs base_args(const santa_params_t* p, const Layout& L, const void* q, const void* K, const void* V,
                            float* out, void* ws, cudaStream_t stream) {
  santa::LaunchArgs a;
  memset(&a, 0, sizeof a);
  unsigned char* w = static_cast<unsigned char*>(ws);
  a.dtype = p->dtype;
  a.D = p->head_dim;
  a.B = p->batch;
  a.H = p->n_q_heads;
  a.Hkv = p->n_kv_heads;
  a.nk_max = p->nk;
  a.chunks_max = (int)L.chunks;
  a.groups_max = (int)L.groups;
  a.tiles_max = (int)((p->nk + santa::TILE - 1) / santa::TILE);
  a.num_sms = device_sms();
  a.S_max = p->S;
  a.scale = p->scale > 0.f ? p->scale : (float)(1.0 / sqrt((double)p->head_dim));
  a.seed = p->seed;
  a.step = p->step;
  a.q = q;
  a.K = K;
  a.V = V;
  a.kv_offsets = p->kv_offsets;
  a.S_per_seq = p->S_per_seq;
  a.out = out;
  a.err = reinterpret_cast<int*>(w);
  a.tile_max = reinterpret_cast<float*>(w + L.tile_max);
  a.tile_sum = reinterpret_cast<float*>(w + L.tile_sum);
  a.part_o = reinterpret_cast<float*>(w + L.part_o);
  a.stream = stream;
  return a;
}

santa_status_t decode_impl(const santa_params_t* p, int32_t variant, const void* q, const void* K, const void* V,
                           const double* uniforms, float* out, void* ws, size_t ws_bytes, santa_stream_t stream,
                           int32_t* sample_idx, void* const* events = nullptr, bool score_only = false,
                           bool k_host = false) {
  santa_status_t st = check_params(p, true);
  if (st != SANTA_OK) return st;
  if (variant < SANTA_IID || variant > SANTA_SYSTEMATIC) return SANTA_ERR_INVALID_ARG;
  const Layout L = santa_layout(p);
  st = score_only ? check_buffers(q, K, K, K, ws, ws_bytes, L.total)
                  : check_buffers(q, K, V, out, ws, ws_bytes, L.total);
  if (st != SANTA_OK) return st;
  if (sample_idx && !aligned(sample_idx, 4)) return SANTA_ERR_INVALID_ARG;
  if (uniforms && !aligned(uniforms, 8)) return SANTA_ERR_INVALID_ARG;

  santa::LaunchArgs a = base_args(p, L, q, K, V, out, ws, (cudaStream_t)stream);
  unsigned char* w = static_cast<unsigned char*>(ws);
  a.variant = variant;
  a.k_host = k_host ? 1 : 0;
  a.uniforms = uniforms;
  a.sample_idx = sample_idx;
  a.stash = reinterpret_cast<float*>(w + L.stash);
  a.prefix = reinterpret_cast<long long*>(w + L.prefix);
  a.thresh = reinterpret_cast<long long*>(w + L.thresh);
  a.jstart = reinterpret_cast<int32_t*>(w + L.jstart);
  a.head_max = reinterpret_cast<float*>(w + L.head_max);
  a.agg = w + L.agg;
  a.ukeys = reinterpret_cast<uint32_t*>(w + L.ukeys);
  a.rcp_S = reinterpret_cast<unsigned long long*>(w + L.rcp_S);

  // 16-bit caches with Philox uniforms: the whole step in one cooperative
  // launch; otherwise (fp32, caller uniforms, per-stage events) three stages.
  if (!score_only && !events && !uniforms && p->dtype != SANTA_FP32)
    return santa::launch_fused(a, reinterpret_cast<unsigned*>(w + BAR_COUNT),
                               reinterpret_cast<unsigned*>(w + BAR_GEN)) == cudaSuccess
               ? SANTA_OK
               : SANTA_ERR_CUDA;

  auto mark = [&](int i) {
    return !events || cudaEventRecord((cudaEvent_t)events[i], (cudaStream_t)stream) == cudaSuccess;
  };
  if (score_only) return santa::launch_score(a) == cudaSuccess ? SANTA_OK : SANTA_ERR_CUDA;
  if (!mark(0) || santa::launch_score(a) != cudaSuccess) return SANTA_ERR_CUDA;
  if (!mark(1) || santa::launch_combine(a) != cudaSuccess) return SANTA_ERR_CUDA;
  if (!mark(2) || santa::launch_sample_gather(a) != cudaSuccess) return SANTA_ERR_CUDA;
  if (!mark(3)) return SANTA_ERR_CUDA;
  return SANTA_OK;
}

}  // namespace

extern "C" {

size_t santa_workspace_size(const santa_params_t* p) {
  if (check_params(p, true) != SANTA_OK) return 0;
  return santa_layout(p).total;
}

santa_status_t santa_workspace_init(void* workspace, size_t ws_bytes, santa_stream_t stream) {
  if (!workspace || !aligned(workspace, ALIGN) || ws_bytes < HEADER) return SANTA_ERR_WORKSPACE;
  return cudaMemsetAsync(workspace, 0, HEADER, (cudaStream_t)stream) == cudaSuccess ? SANTA_OK : SANTA_ERR_CUDA;
}

santa_status_t santa_decode(const santa_params_t* p, int32_t variant, const void* q, const void* K, const void* V,
                            float* out, void* workspace, size_t ws_bytes, santa_stream_t stream,
                            int32_t* sample_idx) {
  return decode_impl(p, variant, q, K, V, nullptr, out, workspace, ws_bytes, stream, sample_idx);
}

// The address the device reads a K or V buffer through: device memory of the
// current device (or managed memory) as it is, page-locked host memory
// (cudaHostAlloc'd or cudaHostRegister'ed) through its mapped device address;
// INVALID_ARG for anything else (pageable memory, another GPU's memory, a
// pointer CUDA does not know).  Nothing is launched.
static santa_status_t kv_address(const void* h, const void** d, bool* host = nullptr) {
  if (!h) return SANTA_ERR_INVALID_ARG;
  cudaPointerAttributes at;
  int cur = -1;
  if (cudaPointerGetAttributes(&at, h) != cudaSuccess || cudaGetDevice(&cur) != cudaSuccess) {
    (void)cudaGetLastError();
    return SANTA_ERR_INVALID_ARG;
  }
  if (at.type == cudaMemoryTypeDevice && at.device != cur) return SANTA_ERR_INVALID_ARG;
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
    *d = h;
    return SANTA_OK;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return SANTA_ERR_INVALID_ARG;
  *d = at.devicePointer;
  if (host) *host = true;
  return SANTA_OK;
}

santa_status_t santa_decode_host_kv(const santa_params_t* p, int32_t variant, const void* q, const void* K,
                                    const void* V, float* out, void* workspace, size_t ws_bytes,
                                    santa_stream_t stream, int32_t* sample_idx) {
  santa_status_t st = check_params(p, true);
  if (st != SANTA_OK) return st;
  if (!K || !V) return SANTA_ERR_INVALID_ARG;
  const void *Kd = nullptr, *Vd = nullptr;
  bool k_host = false;
  if ((st = kv_address(K, &Kd, &k_host)) != SANTA_OK || (st = kv_address(V, &Vd)) != SANTA_OK) return st;
  return decode_impl(p, variant, q, Kd, Vd, nullptr, out, workspace, ws_bytes, stream, sample_idx, nullptr, false,
                     k_host);
}

santa_status_t santa_score_pass(const santa_params_t* p, const void* q, const void* K, void* workspace,
                                size_t ws_bytes, santa_stream_t stream) {
  return decode_impl(p, SANTA_SYSTEMATIC, q, K, K, nullptr, nullptr, workspace, ws_bytes, stream, nullptr, nullptr,
                     true);
}

santa_status_t santa_decode_profiled(const santa_params_t* p, int32_t variant, const void* q, const void* K,
                                     const void* V, float* out, void* workspace, size_t ws_bytes,
                                     santa_stream_t stream, int32_t* sample_idx, void* const* stage_events) {
  return decode_impl(p, variant, q, K, V, nullptr, out, workspace, ws_bytes, stream, sample_idx, stage_events);
}

santa_status_t santa_decode_with_uniforms(const santa_params_t* p, int32_t variant, const void* q, const void* K,
                                          const void* V, const double* uniforms, float* out, void* workspace,
                                          size_t ws_bytes, santa_stream_t stream, int32_t* sample_idx) {
  if (!uniforms) return SANTA_ERR_INVALID_ARG;
  return decode_impl(p, variant, q, K, V, uniforms, out, workspace, ws_bytes, stream, sample_idx);
}

size_t santa_tiled_workspace_size(const santa_params_t* p, int32_t sampler, int32_t tile_len) {
  if (check_tiled(p, sampler, tile_len) != SANTA_OK) return 0;
  return tiled_layout(p, tile_len).total;
}

int32_t santa_tiled_max_draws(const santa_params_t* p, int32_t sampler, int32_t tile_len) {
  if (check_tiled(p, sampler, tile_len) != SANTA_OK) return 0;
  return tiled_draws(p, sampler, tile_len);
}

santa_status_t santa_decode_tiled(const santa_params_t* p, int32_t sampler, int32_t tile_len, const void* q,
                                  const void* K, const void* V, float* out, void* workspace, size_t ws_bytes,
                                  santa_stream_t stream, int32_t* sample_idx) {
  santa_status_t st = check_tiled(p, sampler, tile_len);
  if (st != SANTA_OK) return st;
  const Layout L = tiled_layout(p, tile_len);
  st = check_buffers(q, K, V, out, workspace, ws_bytes, L.total);
  if (st != SANTA_OK) return st;
  if (sample_idx && !aligned(sample_idx, 4)) return SANTA_ERR_INVALID_ARG;
  santa::LaunchArgs a = base_args(p, L, q, K, V, nullptr, workspace, (cudaStream_t)stream);
  unsigned char* w = static_cast<unsigned char*>(workspace);
  a.stash = reinterpret_cast<float*>(w + L.stash);
  a.head_max = reinterpret_cast<float*>(w + L.head_max);
  a.sample_idx = sample_idx;
  a.tl_sampler = sampler;
  a.tl_len = tile_len;
  a.tl_T = (int)L.tl_T;
  a.tl_draws = tiled_draws(p, sampler, tile_len);
  a.tl_pre = reinterpret_cast<int32_t*>(w + L.tl_pre);
  a.tl_w = reinterpret_cast<double*>(w + L.tl_w);
  a.tl_o = reinterpret_cast<float*>(w + L.tl_o);
  // the score pass (out is not touched here): for 16-bit caches the single
  // launch's stream alone, else the staged score kernel
  if (p->dtype != SANTA_FP32) {
    a.score_only = 1;
    a.variant = SANTA_SYSTEMATIC;
    if (santa::launch_fused(a, reinterpret_cast<unsigned*>(w + BAR_COUNT), reinterpret_cast<unsigned*>(w + BAR_GEN)) !=
        cudaSuccess)
      return SANTA_ERR_CUDA;
    a.score_only = 0;
  } else if (santa::launch_score(a) != cudaSuccess) {
    return SANTA_ERR_CUDA;
  }
  a.out = out;
  return santa::launch_tiled(a) == cudaSuccess ? SANTA_OK : SANTA_ERR_CUDA;
}

size_t santa_bernoulli_workspace_size(const santa_params_t* p) {
  if (check_params(p, true) != SANTA_OK) return 0;
  const size_t es = p->dtype == SANTA_FP32 ? 4 : 2;
  return up(santa_layout(p).total) + up((size_t)p->batch * p->n_q_heads * p->head_dim * es);
}

santa_status_t santa_decode_bernoulli(const santa_params_t* p, int32_t variant, int32_t n_samples, int32_t stratified,
                                      const void* q, const void* K, const void* V, float* out, void* workspace,
                                      size_t ws_bytes, santa_stream_t stream, int32_t* sample_idx,
                                      int32_t* feature_counts) {
  santa_status_t st = check_params(p, true);
  if (st != SANTA_OK) return st;
  if (n_samples < 1 || n_samples > 1024) return SANTA_ERR_INVALID_ARG;
  if (variant < SANTA_IID || variant > SANTA_SYSTEMATIC) return SANTA_ERR_INVALID_ARG;
  if (feature_counts && !aligned(feature_counts, 4)) return SANTA_ERR_INVALID_ARG;
  if (sample_idx && !aligned(sample_idx, 4)) return SANTA_ERR_INVALID_ARG;
  const size_t need = santa_bernoulli_workspace_size(p);
  st = check_buffers(q, K, V, out, workspace, ws_bytes, need);
  if (st != SANTA_OK) return st;
  const Layout L = santa_layout(p);
  void* qt = static_cast<unsigned char*>(workspace) + up(L.total);
  santa::LaunchArgs a = base_args(p, L, q, K, V, out, workspace, (cudaStream_t)stream);
  if (santa::launch_bernoulli_query(a, qt, feature_counts, n_samples, stratified ? 1 : 0) != cudaSuccess)
    return SANTA_ERR_CUDA;
  return santa_decode(p, variant, qt, K, V, out, workspace, ws_bytes, stream, sample_idx);
}

santa_status_t santa_selftest_wait_timeout(void* workspace, size_t ws_bytes, uint64_t limit_ns,
                                           santa_stream_t stream) {
  if (!workspace || !aligned(workspace, ALIGN) || ws_bytes < HEADER) return SANTA_ERR_WORKSPACE;
  if (limit_ns < 1000000ull || limit_ns > 2000000000ull) return SANTA_ERR_INVALID_ARG;
  unsigned char* w = static_cast<unsigned char*>(workspace);
  return santa::launch_wait_timeout_selftest(reinterpret_cast<const unsigned*>(w + BAR_GEN),
                                             reinterpret_cast<int*>(w), limit_ns,
                                             (cudaStream_t)stream) == cudaSuccess
             ? SANTA_OK
             : SANTA_ERR_CUDA;
}

int32_t santa_read_probe_sink_words(void) { return 2 * 512 * device_sms(); }

santa_status_t santa_read_probe(const void* src, size_t bytes, uint32_t* sink, santa_stream_t stream) {
  if (!src || !sink || !aligned(src, 16) || !aligned(sink, 4) || bytes == 0 || bytes % 16) return SANTA_ERR_INVALID_ARG;
  return santa::launch_read_probe(src, bytes, sink, 2 * device_sms(), (cudaStream_t)stream) == cudaSuccess
             ? SANTA_OK
             : SANTA_ERR_CUDA;
}

size_t santa_dense_workspace_size(const santa_params_t* p) {
  if (check_params(p, false) != SANTA_OK) return 0;
  return dense_layout(p).total;
}

santa_status_t santa_dense_decode(const santa_params_t* p, const void* q, const void* K, const void* V, float* out,
                                  void* workspace, size_t ws_bytes, santa_stream_t stream) {
  santa_status_t st = check_params(p, false);
  if (st != SANTA_OK) return st;
  const Layout L = dense_layout(p);
  st = check_buffers(q, K, V, out, workspace, ws_bytes, L.total);
  if (st != SANTA_OK) return st;
  santa::LaunchArgs a = base_args(p, L, q, K, V, out, workspace, (cudaStream_t)stream);
  a.fpart = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + L.fpart);
  // 16-bit caches: one cooperative launch (santa_flash.cuh); the rest, or a
  // shape it does not cover, the two-kernel split (santa_score.cu)
  unsigned char* w = static_cast<unsigned char*>(workspace);
  const cudaError_t e =
      santa::launch_flash(a, reinterpret_cast<unsigned*>(w + BAR_COUNT), reinterpret_cast<unsigned*>(w + BAR_GEN));
  if (e == cudaErrorNotSupported) {
    (void)cudaGetLastError();
    return santa::launch_dense(a) == cudaSuccess ? SANTA_OK : SANTA_ERR_CUDA;
  }
  return e == cudaSuccess ? SANTA_OK : SANTA_ERR_CUDA;
}

int32_t santa_workspace_layout(const santa_params_t* p, santa_ws_layout_t* layout) {
  if (!layout || check_params(p, true) != SANTA_OK) return -1;
  const Layout L = santa_layout(p);
  layout->stash = L.stash;
  layout->tile_max = L.tile_max;
  layout->tile_sum = L.tile_sum;
  layout->prefix = L.prefix;
  layout->thresh = L.thresh;
  layout->head_max = L.head_max;
  layout->chunks = L.chunks;
  return 0;
}

santa_status_t santa_get_error(void* workspace, santa_stream_t stream, int32_t* code) {
  if (!workspace || !aligned(workspace, ALIGN)) return SANTA_ERR_WORKSPACE;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SANTA_ERR_CUDA;
  int32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return SANTA_ERR_CUDA;
  if (word && cudaMemset(workspace, 0, sizeof word) != cudaSuccess) return SANTA_ERR_CUDA;
  if (code) *code = word;
  return word ? SANTA_ERR_DEVICE : SANTA_OK;
}

const char* santa_status_string(santa_status_t status) {
  switch (status) {
    case SANTA_OK: return "ok";
    case SANTA_ERR_INVALID_ARG: return "invalid argument";
    case SANTA_ERR_UNSUPPORTED: return "unsupported head_dim, dtype or group size";
    case SANTA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SANTA_ERR_CUDA: return "CUDA runtime error";
    case SANTA_ERR_DEVICE: return "device flagged bad ragged metadata";
    case SANTA_ERR_SCRATCH_LIMIT: return "problem needs more than the SANTA_STATIC_SCRATCH_BYTES of santa_decode_static";
    default: return "unknown status";
  }
}

int32_t santa_version(void) { return 100; }

}  // extern "C"
