// Backward kernel instantiations with the residual gradient (dres) for fp32 activations and weight.
#include "bwd_kernels.cuh"

namespace rmsn {

const void* bwd_res_kernel_f32(const rmsnorm_plan_t& p, bool pipelined) {
    return main_kernel<float, float, true>(p, pipelined);
}

}  // namespace rmsn
