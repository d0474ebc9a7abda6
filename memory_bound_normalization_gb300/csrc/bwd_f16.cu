// Backward kernel instantiations for fp16 activations with an fp16 or an fp32 weight.
#include "bwd_kernels.cuh"

namespace rmsn {

const void* bwd_main_kernel_f16(const rmsnorm_plan_t& p, bool pipelined) {
    return main_kernel<__half, __half, false>(p, pipelined);
}

const void* bwd_main_kernel_f16_w_f32(const rmsnorm_plan_t& p, bool pipelined) {
    return main_kernel<__half, float, false>(p, pipelined);
}

}  // namespace rmsn
