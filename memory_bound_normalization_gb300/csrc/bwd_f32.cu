// Backward kernel instantiations for fp32 activations and weight.
#include "bwd_kernels.cuh"

namespace rmsn {

const void* bwd_main_kernel_f32(const rmsnorm_plan_t& p, bool pipelined) {
    return main_kernel<float, float, false>(p, pipelined);
}

}  // namespace rmsn
