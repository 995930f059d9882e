// Tensor-core (tcgen05) path for bf16 prefill. Placeholder until the kernels land.
#include "lla_internal.cuh"

namespace lla {

bool tc_supported(int, int, int, int) { return false; }
bool make_tc_plan(int, int, int, int, int, TcPlan*) { return false; }
cudaError_t tc_forward(const TcPlan&, const void*, const void*, const void*, const float*, const float*, void*, void*,
                       int*, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace lla
