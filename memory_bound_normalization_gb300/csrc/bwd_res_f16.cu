// Backward kernel instantiations with the residual gradient (dres) for fp16 activations with an fp16 or an fp32 weight.
#include "bwd_kernels.cuh"

namespace rmsn {

const void* bwd_res_kernel_f16(const rmsnorm_plan_t& p, bool pipelined) {
    return main_kernel<__half, __half, true>(p, pipelined);
}

const void* bwd_res_kernel_f16_w_f32(const rmsnorm_plan_t& p, bool pipelined) {
    return main_kernel<__half, float, true>(p, pipelined);
}

}  // namespace rmsn
