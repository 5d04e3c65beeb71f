// Grouped-GEMM arm: not built yet.
#include "common.cuh"
#include "gemm.h"

namespace moe {

bool gemm_supported(const moe_config&) { return false; }
int gemm_max_tiles(int, int, int, int) { return 0; }
int gemm_prepare_weights(const moe_config&, const moe_expert_weights*, const moe_expert_weights*, GemmWeights* out) {
    out->ready = false;
    return MOE_OK;
}
int gemm_plan(const GemmWeights&, const GemmCall&, GemmLaunch*) { return MOE_ERR_UNSUPPORTED; }
cudaError_t launch_gemm_gateup(const GemmLaunch&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_gemm_down(const GemmLaunch&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace moe
