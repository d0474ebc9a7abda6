// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units (fwd.cu, bwd.cu, probe.cu). Host code only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "rmsnorm.h"

namespace rmsn {

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int max_smem_optin = 0;  // bytes of dynamic shared memory a block may opt into
    int l2_bytes = 0;
    int* status_word = nullptr;  // device address of this device's status word
};

// Cached properties of `device` (nullptr if the query fails).
const DeviceInfo* device_info(int device);

struct FwdArgs {
    const void* x;
    const void* w;
    void* y;
    float* rstd;
    int64_t M;
    int N;
    float eps;
    int* status;             // device status word (bounded waits)
    uint64_t wait_limit_ns;
    const void* res;         // residual added to x first (nullptr: plain forward)
    void* h;                 // x + res as stored (written when res is set)
    int64_t drop_unit = -1;  // failure-injection hook (ring kernel), -1 = off
};

struct BwdArgs {
    const void* x;
    const void* w;
    const void* dy;
    const float* rstd;
    void* dx;
    float* partial;  // [partial_rows, N] fp32 workspace
    float* dw;
    int64_t M;
    int N;
    int* status;
    uint64_t wait_limit_ns;
    int64_t drop_unit;  // failure-injection hook, -1 = off
    const void* dres;   // gradient added to dx (residual path), nullptr = none
    int sm_count;       // the device's SMs (sizes the column sum)
    int early_refill;   // refill a ring stage right after pass 2 of its row
    int cluster_dw;     // the grid is one cluster that sums dw on chip (no workspace)
};

constexpr int kMaxCluster = 8;

// Programmatic stream serialization of library launches: on, except where
// a launch asks for plain stream order; RMSNORM_PDL=0 turns it off for every
// launch (read once; a sweep knob).
int pdl_mode();
inline int pdl_allowed(bool want = true) { return want && pdl_mode() != 0 ? 1 : 0; }

// Launches a library kernel with programmatic stream serialization (it may
// start while the previous kernel of the stream finishes; the kernel waits
// for it before touching memory) unless `pdl` is false, and, for
// cluster > 1, a cluster shape.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*fn)(KArgs...), int grid, int threads, size_t smem, int cluster,
                      cudaStream_t s, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_allowed(pdl);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, fn, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*fn)(KArgs...), int grid, int threads, size_t smem, int cluster,
                       cudaStream_t s, Args... args) {
    return launch_ex(fn, grid, threads, smem, cluster, s, true, args...);
}

// Width-dependent choices (host only, no device queries). `vector_ok` says
// whether the pointers and N allow 16-byte vector access.
// `add`: plan the residual forward (the ring kernel then carries the residual).
void fwd_choose(int64_t N, int dtype, bool vector_ok, rmsnorm_plan_t* p, bool add = false);
// `res`: plan the residual backward (dres rides in the rings as well).
void bwd_choose(int64_t N, int dtype, bool vector_ok, rmsnorm_plan_t* p, bool res = false);

// Device-dependent completion of a plan (grid size, shared-memory opt-in).
cudaError_t fwd_finish_plan(const DeviceInfo& dev, int dtype, int64_t M, int64_t N,
                            rmsnorm_plan_t* p, bool add = false);
// `res`: the plan is for the backward with a residual gradient (its kernels
// differ, and so may the number of resident blocks).
cudaError_t bwd_finish_plan(const DeviceInfo& dev, int dtype, int64_t M, int64_t N,
                            rmsnorm_plan_t* p, bool res = false);

cudaError_t fwd_launch(const rmsnorm_plan_t& p, int dtype, const FwdArgs& a, cudaStream_t s);
cudaError_t bwd_launch(const rmsnorm_plan_t& p, int dtype, const BwdArgs& a, cudaStream_t s);

// The naive three-kernel backward (naive.cu), an ablation: workspace bytes
// (the M x N intermediate, then the fp32 partial rows) and the launch chain.
size_t naive_contrib_bytes(int64_t M, int64_t N, int elem);
size_t naive_workspace_bytes(int64_t M, int64_t N, int dtype);
constexpr int kNaiveMaxVectors = 1024;  // one 16-byte vector per thread of one block
cudaError_t naive_launch(int dtype, const void* x, const void* w, const void* dy, void* dx,
                         float* dw, int64_t M, int N, float eps, void* workspace, cudaStream_t s);
// Fixed-order column sum of P fp32 partial rows into dw (bwd.cu), launched
// in plain stream order.
cudaError_t colsum_launch(const float* partial, float* dw, int P, int N, cudaStream_t s);

cudaError_t probe_launch(int kind, void* dst, const void* a, const void* b, size_t bytes,
                         int grid, cudaStream_t s);

// Row-group geometry of the short-row kernels: G lanes per row, V 16-byte
// vectors per lane, R rows per group per pass, block size.
struct GroupShape {
    int G, V, R, threads;
};
// Forward: each lane holds 8-64 elements of R rows in registers. Two rows
// per lane (one where a lane holds 4 vectors) measured best on GB300: 1-3%
// above four (two) for the plain forward and 7-24% for the residual forward,
// whose lanes hold the residual as well; the narrowest rows keep four.
inline bool fwd_group_shape(int64_t nvec, GroupShape* g) {
    if (nvec <= 4) *g = {4, 1, 4, 256};
    else if (nvec <= 8) *g = {4, 2, 2, 128};
    else if (nvec <= 16) *g = {8, 2, 2, 128};
    else if (nvec <= 32) *g = {8, 4, 1, 128};
    else if (nvec <= 64) *g = {16, 4, 1, 128};
    else if (nvec <= 128) *g = {32, 4, 1, 256};
    else if (nvec <= 256) *g = {32, 8, 1, 128};
    else return false;
    return true;
}
// Backward: 128-thread blocks whose tile of rows is about 8 KB per tensor, so
// a three-stage ring of x and dy fits in about 48 KB and four blocks (16
// warps) share an SM. Wider rows take the grouped row kernel.
inline bool bwd_group_shape(int64_t nvec, GroupShape* g) {
    if (nvec <= 4) *g = {4, 1, 4, 128};
    else if (nvec <= 8) *g = {4, 2, 2, 128};
    else if (nvec <= 16) *g = {8, 2, 2, 128};
    else if (nvec <= 32) *g = {8, 4, 1, 128};
    else if (nvec <= 64) *g = {16, 4, 1, 128};
    else if (nvec <= 128) *g = {32, 4, 1, 128};
    else if (nvec <= 256) *g = {32, 8, 1, 128};
    else return false;
    return true;
}

inline bool dtype_known(int dtype) { return dtype >= RMSNORM_F32 && dtype <= RMSNORM_F16_W_F32; }
// bytes of one activation element (x, y, dy, dx)
inline int dtype_size(int dtype) { return dtype == RMSNORM_F32 ? 4 : 2; }
// bytes of one weight element
inline int weight_size(int dtype) { return dtype == RMSNORM_BF16 || dtype == RMSNORM_F16 ? 2 : 4; }
inline int dtype_vec(int dtype) { return 16 / dtype_size(dtype); }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int round_up(int a, int b) { return (a + b - 1) / b * b; }

}  // namespace rmsn
