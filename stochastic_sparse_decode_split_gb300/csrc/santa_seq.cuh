// santa_seq.cuh -- per-sequence metadata checks shared by the device paths.
#pragma once

#include "santa_common.cuh"
#include "santa_launch.h"

namespace santa {

// Sequence metadata: length within [1, nk_max] and budget within [1, S_max].
__device__ __forceinline__ int seq_error(const int64_t* kv_offsets, int64_t nk_max, const int32_t* S_per_seq,
                                         int S_max, int b, int& S_b) {
  int err = 0;
  int64_t nk = nk_max, row0 = 0;
  if (kv_offsets) {
    row0 = kv_offsets[b];
    nk = kv_offsets[b + 1] - row0;
  }
  if (nk < 1) err |= ERR_EMPTY;
  else if (nk > nk_max || row0 < 0) err |= ERR_NK_BOUND;
  S_b = S_per_seq ? S_per_seq[b] : S_max;
  if (S_b < 1 || S_b > S_max) err |= ERR_S_RANGE;
  return err;
}
__device__ __forceinline__ int seq_error(const LaunchArgs& a, int b, int& S_b) {
  return seq_error(a.kv_offsets, a.nk_max, a.S_per_seq, a.S_max, b, S_b);
}

}  // namespace santa
