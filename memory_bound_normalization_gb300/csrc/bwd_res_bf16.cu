// Backward kernel instantiations with the residual gradient (dres) for bf16 activations with a bf16 or an fp32 weight.
#include "bwd_kernels.cuh"

namespace rmsn {

const void* bwd_res_kernel_bf16(const rmsnorm_plan_t& p, bool pipelined) {
    return main_kernel<__nv_bfloat16, __nv_bfloat16, true>(p, pipelined);
}

const void* bwd_res_kernel_bf16_w_f32(const rmsnorm_plan_t& p, bool pipelined) {
    return main_kernel<__nv_bfloat16, float, true>(p, pipelined);
}

}  // namespace rmsn
