// Test helper: exposes PyTorch's header-only Philox4x32-10 engine
// (ATen/core/PhiloxRNGEngine.h) through a C symbol so the oracle's own
// Philox can be checked against an independent implementation.
#include <ATen/core/PhiloxRNGEngine.h>
#include <cstdint>

extern "C" void torch_philox_block(uint64_t seed, uint64_t subsequence, uint64_t offset,
                                   uint32_t* out4) {
  at::philox_engine engine(seed, subsequence, offset);
  for (int i = 0; i < 4; ++i) out4[i] = engine();
}
