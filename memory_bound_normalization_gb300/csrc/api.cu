// C ABI of librmsnorm.so (declared in include/rmsnorm.h): argument checks,
// per-device properties, the device status word, workspace handling and
// dispatch to the kernel translation units.
#include <atomic>
#include <cstdlib>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "kernels.h"

namespace rmsn {

// One status word per device (a module-scope variable lives once in every
// device context that loads the library). Kernels receive its address.
__device__ int g_status_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitLimitNs = 1000000000ull;  // one second

std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices] = {};

std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int64_t> g_drop_unit{-1};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Maps a CUDA result to a status. A failure is also cleared from the
// runtime's last-error slot, so it does not surface in the caller's next,
// unrelated CUDA call.
int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return RMSNORM_OK;
    cudaGetLastError();
    return RMSNORM_ERR_CUDA;
}

int shape_status(int64_t M, int64_t N, int dtype) {
    if (M < 0 || N <= 0 || N > INT32_MAX) return RMSNORM_ERR_INVALID_ARG;
    if (!dtype_known(dtype)) return RMSNORM_ERR_INVALID_ARG;
    return RMSNORM_OK;
}

int current_device(const DeviceInfo** out) {
    int dev = -1;
    if (cuda_status(cudaGetDevice(&dev)) != RMSNORM_OK) return RMSNORM_ERR_CUDA;
    *out = device_info(dev);
    return *out ? RMSNORM_OK : RMSNORM_ERR_CUDA;
}

// Backward checks shared by rmsnorm_bwd and rmsnorm_bwd_ws. On success fills
// the plan (with M > 0) or reports that there is nothing to do besides
// clearing dw (M == 0).
int bwd_prepare(const void* x, const void* w, const void* dy, const float* rstd, void* dx,
                float* dw, int64_t M, int64_t N, int dtype, const DeviceInfo** dev,
                rmsnorm_plan_t* plan, const void* dres = nullptr) {
    int st = shape_status(M, N, dtype);
    if (st != RMSNORM_OK) return st;
    if (M == 0) {
        if (dw != nullptr && !aligned(dw, 4)) return RMSNORM_ERR_MISALIGNED;
        *plan = rmsnorm_plan_t{};
        return RMSNORM_OK;
    }
    if (!x || !w || !dy || !rstd || !dx || !dw) return RMSNORM_ERR_INVALID_ARG;
    const int sz = dtype_size(dtype), wsz = weight_size(dtype);
    if (!aligned(x, sz) || !aligned(w, wsz) || !aligned(dy, sz) || !aligned(dx, sz) ||
        !aligned(rstd, 4) || !aligned(dw, 4) || (dres && !aligned(dres, sz)))
        return RMSNORM_ERR_MISALIGNED;
    const bool vec = aligned(x, 16) && aligned(w, 16) && aligned(dy, 16) && aligned(dx, 16) &&
                     (!dres || aligned(dres, 16)) && (N * sz) % 16 == 0 && (N * wsz) % 16 == 0;
    bwd_choose(N, dtype, vec, plan, dres != nullptr);
    st = current_device(dev);
    if (st != RMSNORM_OK) return st;
    return cuda_status(bwd_finish_plan(**dev, dtype, M, N, plan, dres != nullptr));
}

int bwd_run(const void* x, const void* w, const void* dy, const float* rstd, void* dx, float* dw,
            int64_t M, int64_t N, int dtype, const DeviceInfo& dev, const rmsnorm_plan_t& plan,
            void* workspace, cudaStream_t stream, const void* dres = nullptr) {
    BwdArgs a{};
    a.x = x;
    a.w = w;
    a.dy = dy;
    a.rstd = rstd;
    a.dx = dx;
    a.partial = static_cast<float*>(workspace);
    a.dw = dw;
    a.M = M;
    a.N = static_cast<int>(N);
    a.status = dev.status_word;
    a.sm_count = dev.sm_count;
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.drop_unit = plan.variant != RMSNORM_VARIANT_SCALAR ? g_drop_unit.exchange(-1) : -1;
    a.dres = dres;
    return cuda_status(bwd_launch(plan, dtype, a, stream));
}

// Forward checks, plan and launch shared by rmsnorm_fwd and rmsnorm_add_fwd
// (res and h are both NULL for the plain forward).
int fwd_run(const void* x, const void* res, const void* w, void* h, void* y, float* rstd,
            int64_t M, int64_t N, float eps, int dtype, cudaStream_t stream) {
    int st = shape_status(M, N, dtype);
    if (st != RMSNORM_OK) return st;
    if (!(eps >= 0.f)) return RMSNORM_ERR_INVALID_ARG;  // negative or NaN
    if (M == 0) return RMSNORM_OK;
    const bool add = res != nullptr || h != nullptr;
    if (!x || !w || !y || !rstd || (add && (!res || !h))) return RMSNORM_ERR_INVALID_ARG;
    const int sz = dtype_size(dtype), wsz = weight_size(dtype);
    if (!aligned(x, sz) || !aligned(w, wsz) || !aligned(y, sz) || !aligned(rstd, 4) ||
        (add && (!aligned(res, sz) || !aligned(h, sz))))
        return RMSNORM_ERR_MISALIGNED;
    const bool vec = aligned(x, 16) && aligned(w, 16) && aligned(y, 16) && (N * sz) % 16 == 0 &&
                     (N * wsz) % 16 == 0 && (!add || (aligned(res, 16) && aligned(h, 16)));
    rmsnorm_plan_t plan;
    fwd_choose(N, dtype, vec, &plan, add);
    const DeviceInfo* dev = nullptr;
    st = current_device(&dev);
    if (st != RMSNORM_OK) return st;
    st = cuda_status(fwd_finish_plan(*dev, dtype, M, N, &plan, add));
    if (st != RMSNORM_OK) return st;
    if (static_cast<int64_t>(plan.grid) <= 0 ||
        ((plan.variant == RMSNORM_VARIANT_ROWGROUP || plan.variant == RMSNORM_VARIANT_CTA_ROW ||
          plan.variant == RMSNORM_VARIANT_CLUSTER_ROW) &&
         cdiv(M, plan.variant == RMSNORM_VARIANT_ROWGROUP ? plan.rows_per_unit : 1) * plan.cluster >
             INT32_MAX))
        return RMSNORM_ERR_UNSUPPORTED;
    FwdArgs a{x, w, y, rstd, M, static_cast<int>(N), eps, dev->status_word, g_wait_limit_ns.load(),
              res, h};
    a.drop_unit = plan.variant == RMSNORM_VARIANT_RING ? g_drop_unit.exchange(-1) : -1;
    return cuda_status(fwd_launch(plan, dtype, a, stream));
}

// rmsnorm_bwd and rmsnorm_add_bwd: workspace from the stream-ordered pool.
int bwd_alloc_run(const void* x, const void* w, const void* dy, const float* rstd,
                  const void* dres, void* dx, float* dw, int64_t M, int64_t N, int dtype,
                  cudaStream_t stream) {
    const DeviceInfo* dev = nullptr;
    rmsnorm_plan_t plan;
    int st = bwd_prepare(x, w, dy, rstd, dx, dw, M, N, dtype, &dev, &plan, dres);
    if (st != RMSNORM_OK) return st;
    if (M == 0) {
        if (dw == nullptr) return RMSNORM_OK;
        return cuda_status(cudaMemsetAsync(dw, 0, static_cast<size_t>(N) * 4, stream));
    }
    if (plan.workspace_bytes == 0)  // one partial row: written straight to dw
        return bwd_run(x, w, dy, rstd, dx, dw, M, N, dtype, *dev, plan, nullptr, stream, dres);
    void* ws = nullptr;
    if (cuda_status(cudaMallocAsync(&ws, static_cast<size_t>(plan.workspace_bytes), stream)) !=
        RMSNORM_OK)
        return RMSNORM_ERR_NOMEM;
    st = bwd_run(x, w, dy, rstd, dx, dw, M, N, dtype, *dev, plan, ws, stream, dres);
    const int freed = cuda_status(cudaFreeAsync(ws, stream));
    if (st == RMSNORM_OK) st = freed;
    return st;
}

}  // namespace

int pdl_mode() {
    static const int mode = [] {
        const char* v = getenv("RMSNORM_PDL");
        return (v == nullptr || *v == 0) ? 1 : (atoi(v) != 0 ? 1 : 0);
    }();
    return mode;
}

const DeviceInfo* device_info(int device) {
    if (device < 0 || device >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_dev_ready[device]) return &g_dev[device];
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess || (prev != device && cudaSetDevice(device) != cudaSuccess)) {
        cudaGetLastError();
        return nullptr;
    }
    DeviceInfo d;
    d.device = device;
    bool ok = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device) == cudaSuccess &&
              cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) == cudaSuccess &&
              cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, device) == cudaSuccess &&
              cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status_word), g_status_word) == cudaSuccess;
    if (prev != device) cudaSetDevice(prev);
    if (!ok || d.sm_count <= 0) {
        cudaGetLastError();
        return nullptr;
    }
    g_dev[device] = d;
    g_dev_ready[device] = true;
    return &g_dev[device];
}

}  // namespace rmsn

using namespace rmsn;

extern "C" {

int rmsnorm_fwd(const void* x, const void* w, void* y, float* rstd, int64_t M, int64_t N,
                float eps, int dtype, cudaStream_t stream) {
    return fwd_run(x, nullptr, w, nullptr, y, rstd, M, N, eps, dtype, stream);
}

int rmsnorm_add_fwd(const void* x, const void* residual, const void* w, void* h, void* y,
                    float* rstd, int64_t M, int64_t N, float eps, int dtype,
                    cudaStream_t stream) {
    if (M > 0 && (residual == nullptr || h == nullptr)) return RMSNORM_ERR_INVALID_ARG;
    return fwd_run(x, residual, w, h, y, rstd, M, N, eps, dtype, stream);
}

size_t rmsnorm_bwd_workspace_size(int64_t M, int64_t N, int dtype, int device) {
    if (shape_status(M, N, dtype) != RMSNORM_OK || M == 0) return 0;
    const DeviceInfo* dev = device_info(device);
    if (!dev) return 0;
    rmsnorm_plan_t plan;
    // the workspace only depends on the partial-row count; take the largest
    // of the vector and scalar plans so either alignment class fits
    size_t need = 0;
    for (int vec = 0; vec < 2; ++vec) {
        if (vec && (N * dtype_size(dtype)) % 16 != 0) continue;
        bwd_choose(N, dtype, vec != 0, &plan);
        if (cuda_status(bwd_finish_plan(*dev, dtype, M, N, &plan)) != RMSNORM_OK) return 0;
        if (static_cast<size_t>(plan.workspace_bytes) > need) need = static_cast<size_t>(plan.workspace_bytes);
    }
    return need;
}

int rmsnorm_bwd_ws(const void* x, const void* w, const void* dy, const float* rstd, void* dx,
                   float* dw, int64_t M, int64_t N, int dtype, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
    const DeviceInfo* dev = nullptr;
    rmsnorm_plan_t plan;
    int st = bwd_prepare(x, w, dy, rstd, dx, dw, M, N, dtype, &dev, &plan);
    if (st != RMSNORM_OK) return st;
    if (M == 0) {
        if (dw == nullptr) return RMSNORM_OK;
        return cuda_status(cudaMemsetAsync(dw, 0, static_cast<size_t>(N) * 4, stream));
    }
    if (plan.workspace_bytes > 0 &&
        (workspace == nullptr || workspace_bytes < static_cast<size_t>(plan.workspace_bytes)))
        return RMSNORM_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return RMSNORM_ERR_MISALIGNED;
    return bwd_run(x, w, dy, rstd, dx, dw, M, N, dtype, *dev, plan, workspace, stream);
}

int rmsnorm_bwd(const void* x, const void* w, const void* dy, const float* rstd, void* dx,
                float* dw, int64_t M, int64_t N, int dtype, cudaStream_t stream) {
    return bwd_alloc_run(x, w, dy, rstd, nullptr, dx, dw, M, N, dtype, stream);
}

int rmsnorm_add_bwd(const void* h, const void* w, const void* dy, const float* rstd,
                    const void* dres, void* dx, float* dw, int64_t M, int64_t N, int dtype,
                    cudaStream_t stream) {
    return bwd_alloc_run(h, w, dy, rstd, dres, dx, dw, M, N, dtype, stream);
}

int rmsnorm_bwd_naive(const void* x, const void* w, const void* dy, void* dx, float* dw,
                      int64_t M, int64_t N, float eps, int dtype, cudaStream_t stream) {
    int st = shape_status(M, N, dtype);
    if (st != RMSNORM_OK) return st;
    if (!(eps >= 0.f)) return RMSNORM_ERR_INVALID_ARG;
    if (dw != nullptr && !aligned(dw, 4)) return RMSNORM_ERR_MISALIGNED;
    if (M == 0) {
        if (dw == nullptr) return RMSNORM_OK;
        return cuda_status(cudaMemsetAsync(dw, 0, static_cast<size_t>(N) * 4, stream));
    }
    if (!x || !w || !dy || !dx || !dw) return RMSNORM_ERR_INVALID_ARG;
    const int sz = dtype_size(dtype), wsz = weight_size(dtype);
    if (!aligned(x, sz) || !aligned(w, wsz) || !aligned(dy, sz) || !aligned(dx, sz))
        return RMSNORM_ERR_MISALIGNED;
    const bool vec = aligned(x, 16) && aligned(w, 16) && aligned(dy, 16) && aligned(dx, 16) &&
                     (N * sz) % 16 == 0 && (N * wsz) % 16 == 0;
    if (!vec || N / dtype_vec(dtype) > kNaiveMaxVectors || M > INT32_MAX)
        return RMSNORM_ERR_UNSUPPORTED;
    const DeviceInfo* dev = nullptr;
    st = current_device(&dev);
    if (st != RMSNORM_OK) return st;
    void* ws = nullptr;
    if (cuda_status(cudaMallocAsync(&ws, naive_workspace_bytes(M, N, dtype), stream)) != RMSNORM_OK)
        return RMSNORM_ERR_NOMEM;
    st = cuda_status(naive_launch(dtype, x, w, dy, dx, dw, M, static_cast<int>(N), eps, ws, stream));
    const int freed = cuda_status(cudaFreeAsync(ws, stream));
    if (st == RMSNORM_OK) st = freed;
    return st;
}

int rmsnorm_get_last_device_error(cudaStream_t stream) {
    if (cuda_status(cudaStreamSynchronize(stream)) != RMSNORM_OK) return RMSNORM_ERR_CUDA;
    const DeviceInfo* dev = nullptr;
    if (current_device(&dev) != RMSNORM_OK) return RMSNORM_ERR_CUDA;
    int v = 0;
    if (cuda_status(cudaMemcpy(&v, dev->status_word, sizeof v, cudaMemcpyDeviceToHost)) != RMSNORM_OK)
        return RMSNORM_ERR_CUDA;
    if (v != 0 && cuda_status(cudaMemset(dev->status_word, 0, sizeof v)) != RMSNORM_OK)
        return RMSNORM_ERR_CUDA;
    return v;
}

const char* rmsnorm_status_string(int status) {
    switch (status) {
        case RMSNORM_OK: return "RMSNORM_OK";
        case RMSNORM_ERR_INVALID_ARG: return "RMSNORM_ERR_INVALID_ARG";
        case RMSNORM_ERR_UNSUPPORTED: return "RMSNORM_ERR_UNSUPPORTED";
        case RMSNORM_ERR_MISALIGNED: return "RMSNORM_ERR_MISALIGNED";
        case RMSNORM_ERR_CUDA: return "RMSNORM_ERR_CUDA";
        case RMSNORM_ERR_NOMEM: return "RMSNORM_ERR_NOMEM";
        case RMSNORM_ERR_DEVICE_TIMEOUT: return "RMSNORM_ERR_DEVICE_TIMEOUT";
        case RMSNORM_ERR_OUT_OF_BOUNDS: return "RMSNORM_ERR_OUT_OF_BOUNDS";
        default: return "RMSNORM_STATUS_UNKNOWN";
    }
}

void rmsnorm_set_wait_limit_ns(uint64_t ns) {
    g_wait_limit_ns.store(ns == 0 ? kDefaultWaitLimitNs : ns);
}

void rmsnorm_test_drop_copy(int64_t unit) { g_drop_unit.store(unit < 0 ? -1 : unit); }

int rmsnorm_probe(int kind, void* dst, const void* a, const void* b, size_t bytes,
                  int blocks_per_sm, cudaStream_t stream) {
    if (kind < RMSNORM_PROBE_COPY || kind > RMSNORM_PROBE_2R1W) return RMSNORM_ERR_INVALID_ARG;
    if (bytes % 16 != 0 || blocks_per_sm < 1) return RMSNORM_ERR_INVALID_ARG;
    if (bytes == 0) return RMSNORM_OK;
    if (dst == nullptr) return RMSNORM_ERR_INVALID_ARG;
    if (kind != RMSNORM_PROBE_WRITE && a == nullptr) return RMSNORM_ERR_INVALID_ARG;
    if (kind == RMSNORM_PROBE_2R1W && b == nullptr) return RMSNORM_ERR_INVALID_ARG;
    if (!aligned(dst, 16) || (a && !aligned(a, 16)) || (b && !aligned(b, 16)))
        return RMSNORM_ERR_MISALIGNED;
    const DeviceInfo* dev = nullptr;
    int st = current_device(&dev);
    if (st != RMSNORM_OK) return st;
    const int grid = dev->sm_count * blocks_per_sm;
    return cuda_status(probe_launch(kind, dst, a, b, bytes, grid, stream));
}

int rmsnorm_plan(int64_t M, int64_t N, int dtype, int pass, int device, rmsnorm_plan_t* out) {
    if (out == nullptr) return RMSNORM_ERR_INVALID_ARG;
    int st = shape_status(M, N, dtype);
    if (st != RMSNORM_OK) return st;
    if (pass < RMSNORM_PASS_FWD || pass > RMSNORM_PASS_FWD_ADD) return RMSNORM_ERR_INVALID_ARG;
    const bool fwd = pass == RMSNORM_PASS_FWD || pass == RMSNORM_PASS_FWD_ADD;
    if (M == 0) {
        *out = rmsnorm_plan_t{};
        return RMSNORM_OK;
    }
    const bool vec = (N * dtype_size(dtype)) % 16 == 0;
    if (fwd)
        fwd_choose(N, dtype, vec, out, pass == RMSNORM_PASS_FWD_ADD);
    else
        bwd_choose(N, dtype, vec, out, pass == RMSNORM_PASS_BWD_RES);
    if (device < 0) return RMSNORM_OK;
    const DeviceInfo* dev = device_info(device);
    if (!dev) return RMSNORM_ERR_CUDA;
    cudaError_t e = fwd ? fwd_finish_plan(*dev, dtype, M, N, out, pass == RMSNORM_PASS_FWD_ADD)
                                             : bwd_finish_plan(*dev, dtype, M, N, out,
                                                               pass == RMSNORM_PASS_BWD_RES);
    return cuda_status(e);
}

#ifdef RMSNORM_CHECKS
const char* rmsnorm_version(void) { return "0.2.0+checks"; }
#else
const char* rmsnorm_version(void) { return "0.2.0"; }
#endif

}  // extern "C"
