// santa_seq.cuh -- per-sequence metadata checks shared by the device paths.
#pragma once

#include "santa_common.cuh"
#include "santa_launch.h"

namespace santa {

// Sequence metadata: length within [1, nk_max] and budget within [1, S_max].
__device__ __forceinline__ int seq_error(const LaunchArgs& a, int b, int& S_b) {
  int err = 0;
  int64_t nk = a.nk_max, row0 = 0;
  if (a.kv_offsets) {
    row0 = a.kv_offsets[b];
    nk = a.kv_offsets[b + 1] - row0;
  }
  if (nk < 1) err |= ERR_EMPTY;
  else if (nk > a.nk_max || row0 < 0) err |= ERR_NK_BOUND;
  S_b = a.S_per_seq ? a.S_per_seq[b] : a.S_max;
  if (S_b < 1 || S_b > a.S_max) err |= ERR_S_RANGE;
  return err;
}

}  // namespace santa
