// santa_fused_bf16.cu -- the single-launch decode step (santa_fused.cuh) for
// bf16 caches: every head_dim x sampling variant x K access instantiation.
#include "santa_fused.cuh"

namespace santa {

cudaError_t launch_fused_bf16(const LaunchArgs& a, const CUtensorMap& tm, bool tma, unsigned* bar_count,
                              unsigned* bar_gen, int grid) {
  return launch_fused_dtype<bf16_t>(a, tm, tma, bar_count, bar_gen, grid);
}

}  // namespace santa
