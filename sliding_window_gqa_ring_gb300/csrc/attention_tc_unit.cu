// attention_tc_unit.cu -- the instantiations whose row sums the softmax
// threads keep per lane (LP), used by unit-mode calls with 16-row tiles at
// head_dim 256 (the sliding layers of a large batch, bf16 or FP8 rings).
// Compiled apart from attention_tc.cu so the two builds run side by side.
#include "attention_tc.cuh"

namespace carat {

cudaError_t launch_tc_lane_sums(const AttnParams &p, const TcPlan &plan, const TcMaps &maps,
                                int grid, int rows_per_tile, bool fp8, cudaStream_t stream) {
    if (p.head_dim != 256 || rows_per_tile != 16) return cudaErrorNotSupported;
    if (fp8) return launch_tc<256, 16, 5, 1, 3, true>(p, plan, maps, grid, stream);
    return launch_tc<256, 16, 3, 2, 0, true>(p, plan, maps, grid, stream);
}

}  // namespace carat
