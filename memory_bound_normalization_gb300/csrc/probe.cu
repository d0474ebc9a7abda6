// HBM roofline probes: the measured denominator of every throughput ratio.
// "What a tuned RMSNorm kernel actually costs on Hopper", section 02: the
// achievable bandwidth is the best of a copy, a pure write and a
// two-reads-one-write pattern, measured on the machine in the same run.
// Grid-stride loops over 16-byte vectors, four vectors in flight per thread.
#include "common.cuh"
#include "kernels.h"

namespace rmsn {
namespace {

__global__ void __launch_bounds__(512) probe_copy_kernel(uint4* __restrict__ dst,
                                                         const uint4* __restrict__ src,
                                                         int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = ld_global_16_stream(src + i + u * stride);
#pragma unroll
        for (int u = 0; u < 4; ++u) dst[i + u * stride] = v[u];
    }
    for (; i < n; i += stride) dst[i] = ld_global_16_stream(src + i);
}

__global__ void __launch_bounds__(512) probe_write_kernel(uint4* __restrict__ dst, int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = z;
}

__global__ void __launch_bounds__(512) probe_2r1w_kernel(float4* __restrict__ dst,
                                                         const uint4* __restrict__ a,
                                                         const uint4* __restrict__ b, int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + stride < n; i += 2 * stride) {
        uint4 va[2], vb[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            va[u] = ld_global_16_stream(a + i + u * stride);
            vb[u] = ld_global_16_stream(b + i + u * stride);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
            dst[i + u * stride] = make_float4(
                __uint_as_float(va[u].x) + __uint_as_float(vb[u].x),
                __uint_as_float(va[u].y) + __uint_as_float(vb[u].y),
                __uint_as_float(va[u].z) + __uint_as_float(vb[u].z),
                __uint_as_float(va[u].w) + __uint_as_float(vb[u].w));
    }
    for (; i < n; i += stride) {
        const uint4 va = ld_global_16_stream(a + i), vb = ld_global_16_stream(b + i);
        dst[i] = make_float4(__uint_as_float(va.x) + __uint_as_float(vb.x),
                             __uint_as_float(va.y) + __uint_as_float(vb.y),
                             __uint_as_float(va.z) + __uint_as_float(vb.z),
                             __uint_as_float(va.w) + __uint_as_float(vb.w));
    }
}

}  // namespace

cudaError_t probe_launch(int kind, void* dst, const void* a, const void* b, size_t bytes, int grid,
                         cudaStream_t s) {
    const int64_t n = static_cast<int64_t>(bytes / 16);
    if (n == 0) return cudaSuccess;
    switch (kind) {
        case RMSNORM_PROBE_COPY:
            probe_copy_kernel<<<grid, 512, 0, s>>>(static_cast<uint4*>(dst),
                                                   static_cast<const uint4*>(a), n);
            break;
        case RMSNORM_PROBE_WRITE:
            probe_write_kernel<<<grid, 512, 0, s>>>(static_cast<uint4*>(dst), n);
            break;
        case RMSNORM_PROBE_2R1W:
            probe_2r1w_kernel<<<grid, 512, 0, s>>>(static_cast<float4*>(dst),
                                                   static_cast<const uint4*>(a),
                                                   static_cast<const uint4*>(b), n);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace rmsn
