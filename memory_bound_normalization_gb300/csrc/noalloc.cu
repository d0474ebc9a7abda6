// rmsnorm_bwd_noalloc: the backward for callers that cannot allocate device
// memory -- code that runs where cudaMalloc / cudaMallocAsync are off limits
// or unsafe (a custom allocator that owns all device memory, a real-time loop
// that must not allocate after start-up, an embedding runtime that forbids
// allocator calls from library code). It runs exactly the kernels of
// rmsnorm_bwd, but the per-block dw partial rows go to a fixed scratch array
// that lives in this file, so the call allocates nothing.
#include <mutex>

#include "kernels.h"

namespace rmsn {
namespace {

// The scratch: one array per device that loads the library, held until the
// process exits. Its contents persist from call to call; every partial row a
// call reads back is first written by that same call, so nothing has to be
// cleared between calls.
constexpr size_t kScratchBytes = RMSNORM_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's scratch array. In host code the name
// g_bwd_scratch is only a host-side stand-in, so the address comes from the
// runtime, once per device, with that device current.
int scratch_address(int device, void** out) {
    if (device < 0 || device >= kMaxDevices) return RMSNORM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_addr[device] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return RMSNORM_ERR_CUDA;
        }
        g_scratch_addr[device] = p;
    }
    *out = g_scratch_addr[device];
    return RMSNORM_OK;
}

bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace rmsn

using namespace rmsn;

extern "C" int rmsnorm_bwd_noalloc(const void* x, const void* w, const void* dy,
                                   const float* rstd, void* dx, float* dw, int64_t M, int64_t N,
                                   int dtype, cudaStream_t stream) {
    if (M < 0 || N <= 0 || N > INT32_MAX) return RMSNORM_ERR_INVALID_ARG;
    if (dtype != RMSNORM_F32 && dtype != RMSNORM_BF16) return RMSNORM_ERR_INVALID_ARG;
    if (M == 0) {
        if (dw == nullptr) return RMSNORM_OK;
        if (!is_aligned(dw, 4)) return RMSNORM_ERR_MISALIGNED;
        if (cudaMemsetAsync(dw, 0, static_cast<size_t>(N) * 4, stream) != cudaSuccess) {
            cudaGetLastError();
            return RMSNORM_ERR_CUDA;
        }
        return RMSNORM_OK;
    }
    if (!x || !w || !dy || !rstd || !dx || !dw) return RMSNORM_ERR_INVALID_ARG;
    const int sz = dtype_size(dtype);
    if (!is_aligned(x, sz) || !is_aligned(w, sz) || !is_aligned(dy, sz) || !is_aligned(dx, sz) ||
        !is_aligned(rstd, 4) || !is_aligned(dw, 4))
        return RMSNORM_ERR_MISALIGNED;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) {
        cudaGetLastError();
        return RMSNORM_ERR_CUDA;
    }
    const DeviceInfo* dev = device_info(device);
    if (dev == nullptr) return RMSNORM_ERR_CUDA;
    const bool vec = is_aligned(x, 16) && is_aligned(w, 16) && is_aligned(dy, 16) &&
                     is_aligned(dx, 16) && (N * sz) % 16 == 0;
    rmsnorm_plan_t plan;
    bwd_choose(N, dtype, vec, &plan);
    if (bwd_finish_plan(*dev, dtype, M, N, &plan) != cudaSuccess) {
        cudaGetLastError();
        return RMSNORM_ERR_CUDA;
    }
    // the partial rows must fit in the scratch; nothing is launched otherwise
    if (plan.workspace_bytes < 0 || static_cast<size_t>(plan.workspace_bytes) > kScratchBytes)
        return RMSNORM_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const int st = scratch_address(device, &scratch);
    if (st != RMSNORM_OK) return st;

    BwdArgs a{};
    a.x = x;
    a.w = w;
    a.dy = dy;
    a.rstd = rstd;
    a.dx = dx;
    a.partial = static_cast<float*>(scratch);
    a.dw = dw;
    a.M = M;
    a.N = static_cast<int>(N);
    a.status = dev->status_word;
    a.sm_count = dev->sm_count;
    a.wait_limit_ns = 1000000000ull;  // one second, as for the other entry points by default
    a.drop_unit = -1;
    if (bwd_launch(plan, dtype, a, stream) != cudaSuccess) {
        cudaGetLastError();
        return RMSNORM_ERR_CUDA;
    }
    return RMSNORM_OK;
}

extern "C" size_t rmsnorm_noalloc_scratch_bytes(void) { return kScratchBytes; }
