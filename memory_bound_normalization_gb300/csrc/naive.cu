// The naive three-kernel backward, kept as an ablation: it shows on the same
// GPU what the persistent backward saves. Structure of "RMSNorm backward
// (almost) without the column reduction", section "The naive kernel":
//
//   1. naive_row_kernel: one block per row, one 16-byte vector per thread;
//      recomputes rstd from x (sum of squares and sum of dy*w*x in one block
//      reduction), writes dx, and writes every row's weight-gradient
//      contribution dy*x*rstd, rounded into the activation type, to an M x N
//      intermediate;
//   2. naive_colsum_kernel: splits the rows into kSplit contiguous chunks and
//      sums each chunk's column in fp32, M x N -> kSplit partial rows;
//   3. the fixed-order column sum of the persistent backward (colsum_kernel
//      in bwd.cu), kSplit partial rows -> dw.
//
// The chain moves about five passes over the tensor (x, dy read; dx and the
// intermediate written; the intermediate read again) against three for the
// persistent backward, and it rounds each dw contribution to the activation
// type before summing, so its dw is less accurate than the persistent one.
// Deterministic: every sum has a fixed order. Rows are limited to one
// 16-byte vector per thread of one block (N * element size <= 16 KiB).
#include "common.cuh"
#include "kernels.h"

namespace rmsn {
namespace {

constexpr int kSplit = 64;          // partial rows after the first column pass
constexpr int kColsumThreads = 128; // vectors of columns per column-pass block

template <typename T, typename TW>
__global__ void __launch_bounds__(1024) naive_row_kernel(const T* __restrict__ x,
                                                         const TW* __restrict__ w,
                                                         const T* __restrict__ dy,
                                                         T* __restrict__ dx,
                                                         T* __restrict__ contrib, int64_t M,
                                                         int N, float eps, int* status) {
    using P = Pack<T>;
    using WP = WPack<T, TW>;
    constexpr int VEC = P::VEC, PR = P::PAIRS;
    __shared__ float2 red[32];
    const int64_t row = blockIdx.x;
    const int k = threadIdx.x;  // this thread's vector; whole warps, N / VEC of them used
    const bool ok = k < N / VEC;
    const int64_t off = row * N + static_cast<int64_t>(k) * VEC;
    float2 fx[PR], fd[PR], fw[PR];
    uint4 wq[WP::WORDS];
    if (ok) {
        P::unpack2(ld_global_16_stream(x + off), fx);
        P::unpack2(ld_global_16_stream(dy + off), fd);
        WP::load(w, k, wq);
    } else {
        P::unpack2(make_uint4(0, 0, 0, 0), fx);
        P::unpack2(make_uint4(0, 0, 0, 0), fd);
        WP::zero(wq);
    }
    WP::unpack2(wq, fw);
    // (sum of dy*w*x, sum of x^2) over the row
    float2 s = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < PR; ++e) {
        const float2 gw = __fmul2_rn(fd[e], fw[e]);
        s.x = fmaf(gw.x, fx[e].x, fmaf(gw.y, fx[e].y, s.x));
        s.y = fmaf(fx[e].x, fx[e].x, fmaf(fx[e].y, fx[e].y, s.y));
    }
    s.x = group_allreduce<32>(s.x);
    s.y = group_allreduce<32>(s.y);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = s;
    __syncthreads();
    float2 t = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : make_float2(0.f, 0.f);
    t.x = group_allreduce<32>(t.x);
    t.y = group_allreduce<32>(t.y);
    const float r = rsqrtf(t.y / static_cast<float>(N) + eps);
    const float c = r * (t.x / static_cast<float>(N));  // mean(g * xhat)
    const float2 r2 = f2_splat(r), nc2 = f2_splat(-c);
    float2 o[PR], q[PR];
#pragma unroll
    for (int e = 0; e < PR; ++e) {
        const float2 xh = __fmul2_rn(fx[e], r2);
        o[e] = __fmul2_rn(r2, __ffma2_rn(xh, nc2, __fmul2_rn(fd[e], fw[e])));
        q[e] = __fmul2_rn(fd[e], xh);
    }
    // extent of dx and of the intermediate, for the checked build
    [[maybe_unused]] const int64_t tbytes =
        M * static_cast<int64_t>(N) * static_cast<int64_t>(sizeof(T));
    if (ok && RMSN_OK(span_in(dx + off, 16, dx, tbytes) &&
                          span_in(contrib + off, 16, contrib, tbytes),
                      status)) {
        st_global_16(dx + off, P::pack2(o));
        st_global_16(contrib + off, P::pack2(q));
    }
}

// Block (c, s) sums rows [s*chunk, (s+1)*chunk) of the vectors of columns
// c*128 + t in ascending row order, in fp32, into partial row s.
template <typename T>
__global__ void __launch_bounds__(kColsumThreads) naive_colsum_kernel(const T* __restrict__ contrib,
                                                                      float* __restrict__ partial,
                                                                      int64_t M, int N,
                                                                      int64_t chunk, int* status) {
    using P = Pack<T>;
    constexpr int VEC = P::VEC, PR = P::PAIRS;
    const int nvec = N / VEC;
    const int k = blockIdx.x * kColsumThreads + threadIdx.x;
    if (k >= nvec) return;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * chunk;
    const int64_t r1 = M < r0 + chunk ? M : r0 + chunk;
    float2 acc[PR];
#pragma unroll
    for (int e = 0; e < PR; ++e) acc[e] = make_float2(0.f, 0.f);
    for (int64_t i = r0; i < r1; ++i) {
        float2 f[PR];
        P::unpack2(ld_global_16_stream(contrib + i * N + static_cast<int64_t>(k) * VEC), f);
#pragma unroll
        for (int e = 0; e < PR; ++e) acc[e] = __fadd2_rn(acc[e], f[e]);
    }
    float* prow = partial + static_cast<int64_t>(blockIdx.y) * N + static_cast<int64_t>(k) * VEC;
    [[maybe_unused]] const int64_t pbytes = static_cast<int64_t>(gridDim.y) * N * 4;
#pragma unroll
    for (int e = 0; e < PR; e += 2)
        if (RMSN_OK(span_in(prow + 2 * e, 16, partial, pbytes), status))
            *reinterpret_cast<float4*>(prow + 2 * e) =
                make_float4(acc[e].x, acc[e].y, acc[e + 1].x, acc[e + 1].y);
}

template <typename T, typename TW>
cudaError_t launch_chain(const void* x, const void* w, const void* dy, void* dx, float* dw,
                         int64_t M, int N, float eps, void* workspace, cudaStream_t s) {
    constexpr int VEC = Pack<T>::VEC;
    const int nvec = N / VEC;
    T* contrib = static_cast<T*>(workspace);
    float* partial = reinterpret_cast<float*>(
        static_cast<unsigned char*>(workspace) + naive_contrib_bytes(M, N, sizeof(T)));
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    const DeviceInfo* dev = device_info(device);
    int* status = dev ? dev->status_word : nullptr;
    naive_row_kernel<T, TW><<<static_cast<unsigned>(M), round_up(nvec, 32), 0, s>>>(
        static_cast<const T*>(x), static_cast<const TW*>(w), static_cast<const T*>(dy),
        static_cast<T*>(dx), contrib, M, N, eps, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t chunk = (M + kSplit - 1) / kSplit;
    const int parts = static_cast<int>((M + chunk - 1) / chunk);
    naive_colsum_kernel<T><<<dim3(static_cast<unsigned>((nvec + kColsumThreads - 1) / kColsumThreads),
                                  static_cast<unsigned>(parts)),
                             kColsumThreads, 0, s>>>(contrib, partial, M, N, chunk, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return colsum_launch(partial, dw, parts, N, s);
}

}  // namespace

size_t naive_contrib_bytes(int64_t M, int64_t N, int elem) {
    return (static_cast<size_t>(M) * static_cast<size_t>(N) * elem + 255) / 256 * 256;
}

size_t naive_workspace_bytes(int64_t M, int64_t N, int dtype) {
    return naive_contrib_bytes(M, N, dtype_size(dtype)) +
           static_cast<size_t>(kSplit) * static_cast<size_t>(N) * 4;
}

cudaError_t naive_launch(int dtype, const void* x, const void* w, const void* dy, void* dx,
                         float* dw, int64_t M, int N, float eps, void* workspace, cudaStream_t s) {
    switch (dtype) {
        case RMSNORM_F32: return launch_chain<float, float>(x, w, dy, dx, dw, M, N, eps, workspace, s);
        case RMSNORM_BF16:
            return launch_chain<__nv_bfloat16, __nv_bfloat16>(x, w, dy, dx, dw, M, N, eps, workspace, s);
        case RMSNORM_F16: return launch_chain<__half, __half>(x, w, dy, dx, dw, M, N, eps, workspace, s);
        case RMSNORM_BF16_W_F32:
            return launch_chain<__nv_bfloat16, float>(x, w, dy, dx, dw, M, N, eps, workspace, s);
        case RMSNORM_F16_W_F32:
            return launch_chain<__half, float>(x, w, dy, dx, dw, M, N, eps, workspace, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rmsn
