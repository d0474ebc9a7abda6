// RMSNorm forward kernels: y = x * rstd * w, rstd = 1/sqrt(mean(x^2) + eps).
//
// Definition: "Chapter 13: Fused RMSNorm" (hello-gpu), section 13.1 (eps
// inside the square root; the mean divides by the true column count N, not a
// padded width -- same chapter, the masking note under the Triton route).
// Layout of the work follows the width of a row:
//   * short rows (at most 256 16-byte vectors): a group of G <= 32 lanes per
//     row, several rows per lane in flight, shuffle-only reduction;
//   * mid rows: one thread block per row, row held in registers (x is read
//     once from HBM), warp shuffles then one shared-memory hop -- the block
//     per row shape of "RMSNorm backward (almost) without the column
//     reduction", section "The forward pass", and the block kernel of the
//     hello-gpu chapter;
//   * wide rows: a persistent ring kernel (each block's slice of the coming
//     rows arrives by bulk copies into a shared-memory ring; with a cluster
//     the row sum is exchanged through distributed shared memory), or a
//     thread-block cluster per row with the slices in registers, or, for rows
//     the ring cannot hold, two passes over the row with the second served
//     by L2.
// Any input that is not 16-byte aligned, or whose row is not a whole number
// of 16-byte vectors, takes the scalar kernel.
//
// With ADD every kernel first forms h = x + res, rounded once into T, stores
// h and normalises it ("Profiling, GPU utilisation and writing a fused
// kernel", Problem 15: the kernel takes a residual, writes the sum back and
// normalises the sum). h may share memory with x or res: each element of h
// is written by the thread that read it, and h is read back only through
// coherent loads.
#include <algorithm>
#include <cstdlib>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "common.cuh"
#include "kernels.h"

namespace rmsn {
namespace {

// ---------------------------------------------------------------- short rows
// Block = threads/G groups; group g handles rows tile + r*groups + g for
// r < R, so at each r the block touches consecutive rows.
template <typename T, typename TW, int G, int V, int R, bool ADD>
__global__ void __launch_bounds__(256) fwd_rowgroup_kernel(const T* x, const TW* __restrict__ w,
                                                           T* __restrict__ y,
                                                           float* __restrict__ rstd, int64_t M,
                                                           int N, float eps, const T* res,
                                                           T* hout, int* status) {
    using P = Pack<T>;
    // extents for the checked build: x, res, h, y; rstd
    [[maybe_unused]] const int64_t tbytes =
        M * static_cast<int64_t>(N) * static_cast<int64_t>(sizeof(T));
    [[maybe_unused]] const int64_t rbytes = M * 4;
    constexpr int VEC = P::VEC;
    const int nvec = N / VEC;
    const int lane = threadIdx.x % G;
    const int group = threadIdx.x / G;
    const int groups = blockDim.x / G;
    const int64_t tile = static_cast<int64_t>(blockIdx.x) * groups * R;
    wait_for_prerequisite_grid();  // no global access before this

    uint4 xv[R][V];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = tile + static_cast<int64_t>(r) * groups + group;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = j * G + lane;
            xv[r][j] = (row < M && k < nvec)
                           ? ld_global_16_stream(x + row * N + static_cast<int64_t>(k) * VEC)
                           : make_uint4(0, 0, 0, 0);
        }
    }
    if constexpr (ADD) {
        // every residual load is issued before the first add, so they are in
        // flight together (the loads cannot be moved past the stores of h)
        uint4 rv[R][V];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = tile + static_cast<int64_t>(r) * groups + group;
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int k = j * G + lane;
                rv[r][j] = (row < M && k < nvec)
                               ? ld_global_16_stream(res + row * N + static_cast<int64_t>(k) * VEC)
                               : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = tile + static_cast<int64_t>(r) * groups + group;
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int k = j * G + lane;
                if (row < M && k < nvec) {
                    xv[r][j] = add_vec<T>(xv[r][j], rv[r][j]);
                    T* hd = hout + row * N + static_cast<int64_t>(k) * VEC;
                    if (RMSN_OK(span_in(hd, 16, hout, tbytes), status)) st_global_16(hd, xv[r][j]);
                }
            }
        }
    }
    using WP = WPack<T, TW>;
    uint4 wv[V][WP::WORDS];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int k = j * G + lane;
        if (k < nvec) WP::load(w, k, wv[j]);
        else WP::zero(wv[j]);
    }

    constexpr int PR = P::PAIRS;
    float ss[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            float2 f[PR];
            P::unpack2(xv[r][j], f);
#pragma unroll
            for (int e = 0; e < PR; ++e) acc = __ffma2_rn(f[e], f[e], acc);
        }
        ss[r] = acc.x + acc.y;
    }
#pragma unroll
    for (int off = G / 2; off >= 1; off /= 2)
#pragma unroll
        for (int r = 0; r < R; ++r) ss[r] += __shfl_xor_sync(0xffffffffu, ss[r], off);

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = tile + static_cast<int64_t>(r) * groups + group;
        if (row >= M) continue;
        const float rs = rsqrtf(ss[r] / static_cast<float>(N) + eps);
        const float2 rs2 = f2_splat(rs);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = j * G + lane;
            if (k >= nvec) continue;
            float2 fx[PR], fw[PR], fy[PR];
            P::unpack2(xv[r][j], fx);
            WP::unpack2(wv[j], fw);
#pragma unroll
            for (int e = 0; e < PR; ++e) fy[e] = __fmul2_rn(__fmul2_rn(fx[e], rs2), fw[e]);
            T* yd = y + row * N + static_cast<int64_t>(k) * VEC;
            if (RMSN_OK(span_in(yd, 16, y, tbytes), status)) st_global_16(yd, P::pack2(fy));
        }
        if (lane == 0 && RMSN_OK(span_in(rstd + row, 4, rstd, rbytes), status)) rstd[row] = rs;
    }
    allow_dependent_launch();
}

// ------------------------------------------------------- block/cluster per row
// Cluster c (a single block when launched without clusters) owns row c; block
// rank q of the cluster owns vector slots [q*S, (q+1)*S), S = V*blockDim.x,
// thread t holding slots q*S + j*blockDim.x + t. In a cluster the blocks'
// sums of squares are exchanged by asynchronous stores into every block's
// shared memory (thread q writes to block q), counted as transaction bytes on
// that block's mbarrier, and added in rank order (the same bits everywhere).
// An fp32 weight with 16-bit activations doubles the weight registers: that
// instantiation is bounded to 512 threads (the ladder never gives it more),
// which leaves it 128 registers a thread instead of 64.
template <typename T, typename TW>
constexpr int row_kernel_max_threads() { return std::is_same<T, TW>::value ? 1024 : 512; }

template <typename T, typename TW, int V, bool ADD>
__global__ void __launch_bounds__(row_kernel_max_threads<T, TW>())
    fwd_row_kernel(const T* x, const TW* __restrict__ w, T* __restrict__ y,
                   float* __restrict__ rstd, int64_t M, int N, float eps, int* status,
                   uint64_t wait_limit_ns, const T* res, T* hout) {
    using P = Pack<T>;
    // extents for the checked build: x, res, h, y; rstd
    [[maybe_unused]] const int64_t tbytes =
        M * static_cast<int64_t>(N) * static_cast<int64_t>(sizeof(T));
    [[maybe_unused]] const int64_t rbytes = M * 4;
    constexpr int VEC = P::VEC;
    __shared__ float red[32];
    __shared__ float xslot[kMaxCluster];
    __shared__ __align__(8) uint64_t xbar;

    const uint32_t csize = cluster_size();
    const uint32_t crank = csize > 1 ? cluster_rank() : 0u;
    const int64_t row = csize > 1 ? static_cast<int64_t>(cluster_index()) : blockIdx.x;
    const int nthr = blockDim.x;
    const int nvec = N / VEC;
    const int base = static_cast<int>(crank) * V * nthr;
    const T* xr = x + row * N;
    bool xok = true;  // the cluster exchange completed in time

    if (csize > 1) {
        if (threadIdx.x == 0) {
            mbar_init(&xbar, 1);
            fence_mbarrier_init();
        }
        cluster_arrive_relaxed();  // waited for below, after the loads
    }
    wait_for_prerequisite_grid();  // no global access before this
    using WP = WPack<T, TW>;
    // fp32 rows load their weights only for the scaling, after the row's sum:
    // holding them through the reduction took the kernel to 62 registers, so
    // that a block of 384 threads fitted only twice on an SM
    constexpr bool kLateW = sizeof(T) == 4;  // (16-bit rows stay at 64 registers either way)
    uint4 xv[V], wv[V][WP::WORDS];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int k = base + j * nthr + threadIdx.x;
        const bool ok = k < nvec;
        xv[j] = ok ? ld_global_16_stream(xr + static_cast<int64_t>(k) * VEC) : make_uint4(0, 0, 0, 0);
        if (!kLateW && ok) WP::load(w, k, wv[j]);
        else WP::zero(wv[j]);
    }
    if constexpr (ADD) {
        // all residual loads first, then the adds and the stores of h
        uint4 rv[V];
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = base + j * nthr + threadIdx.x;
            rv[j] = k < nvec ? ld_global_16_stream(res + row * N + static_cast<int64_t>(k) * VEC)
                             : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = base + j * nthr + threadIdx.x;
            if (k < nvec) {
                xv[j] = add_vec<T>(xv[j], rv[j]);
                T* hd = hout + row * N + static_cast<int64_t>(k) * VEC;
                if (RMSN_OK(span_in(hd, 16, hout, tbytes), status)) st_global_16(hd, xv[j]);
            }
        }
    }
    constexpr int PR = P::PAIRS;
    float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < V; ++j) {
        float2 f[PR];
        P::unpack2(xv[j], f);
#pragma unroll
        for (int e = 0; e < PR; ++e) ss2 = __ffma2_rn(f[e], f[e], ss2);
    }
    // block: butterfly per warp, then one shared-memory hop
    float ss = group_allreduce<32>(ss2.x + ss2.y);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float total = lane < (nthr >> 5) ? red[lane] : 0.f;
    total = group_allreduce<32>(total);
    if (csize > 1) {
        cluster_wait();  // every block's barrier is initialised
        if (threadIdx.x == 0) mbar_arrive_expect_tx(&xbar, 4u * csize);
        if (threadIdx.x < csize)
            st_async_cluster_f32(cluster_map(&xslot[crank], threadIdx.x), total,
                                 cluster_map(&xbar, threadIdx.x));
        xok = mbar_wait_cluster_bounded(&xbar, 0u, wait_limit_ns);
        if (!xok) report_status(status, kStatusTimeout);
        total = 0.f;
        for (uint32_t q = 0; q < csize; ++q) total += xslot[q];
        // this block is done with its slots and its barrier; it leaves only
        // after every block of the cluster has arrived here too (below)
        cluster_arrive_relaxed();
    }
    const float rs = rsqrtf(total / static_cast<float>(N) + eps);
    const float2 rs2 = f2_splat(rs);
    T* yr = y + row * N;
    if constexpr (kLateW) {
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = base + j * nthr + threadIdx.x;
            if (k < nvec) WP::load(w, k, wv[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int k = base + j * nthr + threadIdx.x;
        if (k >= nvec) continue;
        float2 fx[PR], fw[PR], fy[PR];
        P::unpack2(xv[j], fx);
        WP::unpack2(wv[j], fw);
#pragma unroll
        for (int e = 0; e < PR; ++e) fy[e] = __fmul2_rn(__fmul2_rn(fx[e], rs2), fw[e]);
        T* yd = yr + static_cast<int64_t>(k) * VEC;
        if (RMSN_OK(span_in(yd, 16, y, tbytes), status)) st_global_16(yd, P::pack2(fy));
    }
    if (crank == 0 && threadIdx.x == 0 && RMSN_OK(span_in(rstd + row, 4, rstd, rbytes), status))
        rstd[row] = rs;
    allow_dependent_launch();
    if (csize > 1) {
        // No block may leave while a peer can still store into its shared
        // memory: every block has sent its sum before it arrives. After a
        // wait that ran out, a late sum may still be in flight to this
        // block: let it land (bounded) before leaving.
        cluster_wait();
        if (!xok) mbar_wait_cluster_bounded(&xbar, 0u, wait_limit_ns);
    }
}

// ---------------------------------------------------------------- wide rows
// Rows too wide for one block's registers: a block per row (grid-strided over
// a small persistent grid), the row streamed in chunks of blockDim.x*U
// vectors twice. Pass 1 sums x^2 and asks L2 to keep x (evict_last); pass 2
// reads x back from L2 (evict_first: last use), scales and stores y. HBM reads
// x once; with one or two blocks per SM the rows in flight take a few tens
// of MB of L2, far below its size.
template <typename T, typename TW, int U, bool ADD>
__global__ void __launch_bounds__(1024) fwd_wide_kernel(const T* x, const TW* __restrict__ w,
                                                       T* __restrict__ y, float* __restrict__ rstd,
                                                       int64_t M, int N, float eps, const T* res,
                                                       T* hout, int* status) {
    using P = Pack<T>;
    // extents for the checked build: x, res, h, y; rstd
    [[maybe_unused]] const int64_t tbytes =
        M * static_cast<int64_t>(N) * static_cast<int64_t>(sizeof(T));
    [[maybe_unused]] const int64_t rbytes = M * 4;
    using WP = WPack<T, TW>;
    constexpr int VEC = P::VEC;
    constexpr int PR = P::PAIRS;
    __shared__ float red[2][32];
    const int nthr = blockDim.x, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31, nw = nthr >> 5;
    const int nvec = N / VEC;
    const uint64_t keep = l2_policy_evict_last();
    const uint64_t last = l2_policy_evict_first();
    wait_for_prerequisite_grid();  // no global access before this
    int it = 0;
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x, ++it) {
        const T* xr = x + row * N;
        float2 ss2 = make_float2(0.f, 0.f);
        // pass 1 of a plain fp32 row keeps 16 vectors a thread in flight: with
        // 4 (or 8) the 1024-thread block streamed too little to fill HBM
        // (fp32 N = 196608 and 262144: 62% and 60% of the copy roofline
        // against 52% and 49%; 16-bit rows did not move)
        constexpr int U1 = (sizeof(T) == 4 && !ADD) ? 16 : U;
        for (int base = 0; base < nvec; base += nthr * U1) {
            uint4 v[U1];
#pragma unroll
            for (int u = 0; u < U1; ++u) {
                const int k = base + u * nthr + tid;
                v[u] = k < nvec ? ld_global_16_hint(xr + static_cast<int64_t>(k) * VEC, keep)
                                : make_uint4(0, 0, 0, 0);
            }
            if constexpr (ADD) {
                // h = x + res goes to L2 (evict_last) for pass 2 and on to
                // HBM; all residual loads are issued before the first store
                uint4 rv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = base + u * nthr + tid;
                    rv[u] = k < nvec ? ld_global_16_stream(res + row * N + static_cast<int64_t>(k) * VEC)
                                     : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = base + u * nthr + tid;
                    if (k < nvec) {
                        v[u] = add_vec<T>(v[u], rv[u]);
                        T* hd = hout + row * N + static_cast<int64_t>(k) * VEC;
                        if (RMSN_OK(span_in(hd, 16, hout, tbytes), status))
                            st_global_16_hint(hd, v[u], keep);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U1; ++u) {
                float2 f[PR];
                P::unpack2(v[u], f);
#pragma unroll
                for (int e = 0; e < PR; ++e) ss2 = __ffma2_rn(f[e], f[e], ss2);
            }
        }
        float ss = group_allreduce<32>(ss2.x + ss2.y);
        if (lane == 0) red[it & 1][warp] = ss;
        __syncthreads();
        float total = lane < nw ? red[it & 1][lane] : 0.f;
        total = group_allreduce<32>(total);
        const float rs = rsqrtf(total / static_cast<float>(N) + eps);
        const float2 rs2 = f2_splat(rs);
        T* yr = y + row * N;
        for (int base = 0; base < nvec; base += nthr * U) {
            uint4 v[U], wv[U][WP::WORDS];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = base + u * nthr + tid;
                const bool ok = k < nvec;
                if constexpr (ADD)  // h was written by this kernel: coherent loads
                    v[u] = ok ? ld_global_16_coherent_hint(hout + row * N + static_cast<int64_t>(k) * VEC, last)
                              : make_uint4(0, 0, 0, 0);
                else
                    v[u] = ok ? ld_global_16_hint(xr + static_cast<int64_t>(k) * VEC, last)
                              : make_uint4(0, 0, 0, 0);
                if (ok) WP::load(w, k, wv[u]);
                else WP::zero(wv[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = base + u * nthr + tid;
                if (k >= nvec) continue;
                float2 fx[PR], fw[PR], fy[PR];
                P::unpack2(v[u], fx);
                WP::unpack2(wv[u], fw);
#pragma unroll
                for (int e = 0; e < PR; ++e) fy[e] = __fmul2_rn(__fmul2_rn(fx[e], rs2), fw[e]);
                T* yd = yr + static_cast<int64_t>(k) * VEC;
                if (RMSN_OK(span_in(yd, 16, y, tbytes), status)) st_global_16(yd, P::pack2(fy));
            }
        }
        if (tid == 0 && RMSN_OK(span_in(rstd + row, 4, rstd, rbytes), status)) rstd[row] = rs;
    }
    allow_dependent_launch();
}

// ------------------------------------------------- wide rows, persistent ring
// Shared memory of the ring kernel: [S][unit] x | ([S][unit] residual) |
// mbarrier[S] (copies) | mbarrier[4] (cluster exchange) | reduction slots
// [2][32] | exchange slots [4][kMaxCluster] | failure flag.
__host__ __device__ inline int fwd_ring_smem_bytes(int stages, int unit, int nt) {
    return nt * stages * unit + stages * 8 + 4 * 8 + 64 * 4 + 4 * kMaxCluster * 4 + 16;
}

// Rows too wide for one block's registers, persistent: cluster cid (a single
// block when launched without clusters) walks rows cid, cid + ncl, ...; block
// rank q of the cluster owns vector slots [q*V*T, (q+1)*V*T) of every row.
// The slices of the coming rows arrive by 1-D bulk copies into an S-stage
// shared-memory ring, completion counted on an mbarrier. Per row: the slice
// moves from shared memory into registers (with ADD, h = x + res is formed
// and stored there), the sum of squares is reduced over the block, the block
// barrier frees the stage, which is refilled with row t + S at once, the
// blocks of a cluster exchange their sums by st.async into a 4-slot ring of
// exchange slots (as in the wide backward: a block sends row t + 1 only after
// receiving every sum of row t, so a writer is at most three rows ahead of a
// reader), and y is scaled from registers. A 16-bit slice of 8 vectors a
// thread does not fit in registers: it is read from its stage once for the
// sum of squares and again for the scaling, and its stage is refilled after
// the next row's block barrier (S - 1 rows ahead). Every wait is bounded.
template <typename T, typename TW, int V, bool ADD>
__global__ void __launch_bounds__(512) fwd_ring_kernel(const T* x, const TW* __restrict__ w,
                                                      T* __restrict__ y, float* __restrict__ rstd,
                                                      int64_t M, int N, float eps, int stages,
                                                      int* status, uint64_t wait_limit_ns,
                                                      const T* res, T* hout, int64_t drop_unit) {
    using P = Pack<T>;
    // extents for the checked build: x, res, h, y; rstd
    [[maybe_unused]] const int64_t tbytes =
        M * static_cast<int64_t>(N) * static_cast<int64_t>(sizeof(T));
    [[maybe_unused]] const int64_t rbytes = M * 4;
    using WP = WPack<T, TW>;
    constexpr int VEC = P::VEC;
    constexpr int PR = P::PAIRS;
    constexpr int NT = ADD ? 2 : 1;
    extern __shared__ __align__(128) unsigned char smem[];

    const int nthr = blockDim.x, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31, nw = nthr >> 5;
    const uint32_t csize = cluster_size();
    const uint32_t crank = csize > 1 ? cluster_rank() : 0u;
    const int64_t cid = csize > 1 ? static_cast<int64_t>(cluster_index()) : blockIdx.x;
    const int64_t ncl = csize > 1 ? static_cast<int64_t>(cluster_count()) : gridDim.x;
    const float inv_n = 1.f / static_cast<float>(N);
    const int nvec = N / VEC;
    const int slots = V * nthr;
    const int vbeg = static_cast<int>(crank) * slots;
    const int vcnt = max(0, min(slots, nvec - vbeg));
    const uint32_t bytes = static_cast<uint32_t>(vcnt) * 16u;
    const int S = stages;
    const int unit = slots * 16;
    // 16-bit slices of 8 vectors a thread are read from the stage twice (for
    // the sum of squares, then for the scaling) instead of being held in
    // registers, and their stage is refilled one row later
    constexpr bool HOLD = !(V == 8 && sizeof(T) == 2);

    unsigned char* sx = smem;
    unsigned char* sr = smem + S * unit;  // residual (ADD only)
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + NT * S * unit);
    uint64_t* xbar = bar + S;                          // [4]
    float* red = reinterpret_cast<float*>(xbar + 4);  // [2][32]
    float* xslot = red + 64;                           // [4][kMaxCluster]
    volatile int* fail = reinterpret_cast<volatile int*>(xslot + 4 * kMaxCluster);

    const int64_t nrows = cid < M ? (M - 1 - cid) / ncl + 1 : 0;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
        for (int b = 0; b < 4; ++b) mbar_init(&xbar[b], 1);
        *fail = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    // every block's barriers must exist before any peer arrives on them
    if (csize > 1) cluster_sync_all();
    wait_for_prerequisite_grid();  // no global access before this

    uint32_t pending = 0, pending_parity = 0;  // producer state (thread 0)
    int ps = 0;
    uint32_t ppar = 0;  // ring position of the next row to issue (issued in order)
    auto issue = [&](int64_t t) {
        const int s = ps;
        const uint32_t par = ppar;
        if (++ps == S) {
            ps = 0;
            ppar ^= 1u;
        }
        if (bytes == 0) {
            mbar_arrive(&bar[s]);
            return;
        }
        mbar_arrive_expect_tx(&bar[s], static_cast<uint32_t>(NT) * bytes);
        if (cid + t * ncl == drop_unit) return;  // failure injection: this wait runs out
        const int64_t off = (cid + t * ncl) * N + static_cast<int64_t>(vbeg) * VEC;
        if (!RMSN_OK(span_in(x + off, bytes, x, tbytes) && smem_span_in(sx + s * unit, bytes) &&
                         (!ADD || (span_in(res + off, bytes, res, tbytes) &&
                                   smem_span_in(sr + s * unit, bytes))),
                     status))
            return;  // checked build: the wait for this stage runs out instead
        bulk_copy_g2s(sx + s * unit, x + off, bytes, &bar[s]);
        if constexpr (ADD) bulk_copy_g2s(sr + s * unit, res + off, bytes, &bar[s]);
        pending |= 1u << s;
        pending_parity = (pending_parity & ~(1u << s)) | (par << s);
    };
    if (tid == 0)
        for (int64_t t = 0; t < S && t < nrows; ++t) issue(t);

    uint4 wv[V][WP::WORDS];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int k = j * nthr + tid;
        if (k < vcnt) WP::load(w, vbeg + k, wv[j]);
        else WP::zero(wv[j]);
    }

    bool failed = false, xfailed = false;
    int cs = 0;
    uint32_t cpar = 0;  // ring position of row t
    for (int64_t t = 0; t < nrows; ++t) {
        const int64_t row = cid + t * ncl;
        const int s = cs;
        const uint32_t parity = cpar;
        if (++cs == S) {
            cs = 0;
            cpar ^= 1u;
        }
        if (!failed) {
            if (mbar_wait_bounded(&bar[s], parity, wait_limit_ns)) {
                if (tid == 0) pending &= ~(1u << s);
            } else {
                *fail = 1;
                report_status(status, kStatusTimeout);
            }
        }
        // the slice (h = x + res with ADD, stored to global), into registers
        // when held
        uint4 xv[HOLD ? V : 1];
        float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = j * nthr + tid;
            uint4 v = k < vcnt ? ld_ring_16(sx + s * unit + k * 16, status) : make_uint4(0, 0, 0, 0);
            if constexpr (ADD) {
                if (k < vcnt) {
                    v = add_vec<T>(v, ld_ring_16(sr + s * unit + k * 16, status));
                    T* hd = hout + row * N + static_cast<int64_t>(vbeg + k) * VEC;
                    if (RMSN_OK(span_in(hd, 16, hout, tbytes), status)) st_global_16(hd, v);
                }
            }
            if constexpr (HOLD) xv[j] = v;
            float2 f[PR];
            P::unpack2(v, f);
#pragma unroll
            for (int e = 0; e < PR; ++e) ss2 = __ffma2_rn(f[e], f[e], ss2);
        }
        const float part = group_allreduce<32>(ss2.x + ss2.y);
        if (lane == 0) red[(t & 1) * 32 + warp] = part;
        // a held slice's stage is read; a re-read slice's stage of row t - 1 is
        // (its scaling came before this barrier); the warp sums of row t are
        // published
        __syncthreads();
        failed = *fail != 0;
        if constexpr (HOLD) {
            if (tid == 0 && !failed && t + S < nrows) {
                fence_proxy_async_shared();
                issue(t + S);
            }
        } else {
            if (tid == 0 && !failed && t >= 1 && t + S - 1 < nrows) {
                fence_proxy_async_shared();
                issue(t + S - 1);
            }
        }
        float tot = lane < nw ? red[(t & 1) * 32 + lane] : 0.f;
        tot = group_allreduce<32>(tot);
        if (csize > 1) {
            const int b = static_cast<int>(t & 3);
            // this block expects the C sums of row t as 4*C transaction bytes
            if (tid == 0) mbar_arrive_expect_tx(&xbar[b], 4u * csize);
            if (static_cast<uint32_t>(tid) < csize) {
                const uint32_t q = static_cast<uint32_t>(tid);  // thread q sends to block q
                st_async_cluster_f32(cluster_map(&xslot[b * kMaxCluster + crank], q), tot,
                                     cluster_map(&xbar[b], q));
            }
            if (!xfailed &&
                !mbar_wait_cluster_bounded(&xbar[b], static_cast<uint32_t>((t >> 2) & 1), wait_limit_ns)) {
                xfailed = true;  // later exchanges are not waited for again
                *fail = 1;
                report_status(status, kStatusTimeout);
            }
            tot = 0.f;
            for (uint32_t q = 0; q < csize; ++q) tot += xslot[b * kMaxCluster + q];
        }
        const float rs = rsqrtf(tot * inv_n + eps);
        const float2 rs2 = f2_splat(rs);
        T* yr = y + row * N;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = j * nthr + tid;
            if (k >= vcnt) continue;
            uint4 v;
            if constexpr (HOLD) {
                v = xv[j];
            } else {
                v = ld_ring_16(sx + s * unit + k * 16, status);
                if constexpr (ADD) v = add_vec<T>(v, ld_ring_16(sr + s * unit + k * 16, status));
            }
            float2 fx[PR], fw[PR], fy[PR];
            P::unpack2(v, fx);
            WP::unpack2(wv[j], fw);
#pragma unroll
            for (int e = 0; e < PR; ++e) fy[e] = __fmul2_rn(__fmul2_rn(fx[e], rs2), fw[e]);
            T* yd = yr + static_cast<int64_t>(vbeg + k) * VEC;
            if (RMSN_OK(span_in(yd, 16, y, tbytes), status)) st_global_16(yd, P::pack2(fy));
        }
        if (crank == 0 && tid == 0 && RMSN_OK(span_in(rstd + row, 4, rstd, rbytes), status))
            rstd[row] = rs;
    }
    allow_dependent_launch();
    // after a failure, let copies already in flight land before going on
    if (tid == 0 && failed)
        for (int s = 0; s < S; ++s)
            if ((pending >> s) & 1u) mbar_wait_bounded(&bar[s], (pending_parity >> s) & 1u, wait_limit_ns);
    // no block may leave while a peer can still reach its shared memory
    if (csize > 1) cluster_sync_all();
}

// -------------------------------------------------------------------- scalar
// Any alignment, any N: one block per row (grid-strided over rows), two
// passes over the row with scalar loads.
template <typename T, typename TW, bool ADD>
__global__ void __launch_bounds__(256) fwd_scalar_kernel(const T* x, const TW* __restrict__ w,
                                                         T* __restrict__ y,
                                                         float* __restrict__ rstd, int64_t M,
                                                         int N, float eps, const T* res,
                                                         T* hout, int* status) {
    using P = Pack<T>;
    // extents for the checked build: x, res, h, y; rstd
    [[maybe_unused]] const int64_t tbytes =
        M * static_cast<int64_t>(N) * static_cast<int64_t>(sizeof(T));
    [[maybe_unused]] const int64_t rbytes = M * 4;
    __shared__ float red[2][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    wait_for_prerequisite_grid();  // no global access before this
    int it = 0;
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x, ++it) {
        const T* xr = x + row * N;
        float ss = 0.f;
        for (int j = threadIdx.x; j < N; j += blockDim.x) {
            float v = to_f32(xr[j]);
            if constexpr (ADD) {
                const T hv = P::from_float(v + to_f32(res[row * N + j]));
                if (RMSN_OK(span_in(hout + row * N + j, sizeof(T), hout, tbytes), status))
                    hout[row * N + j] = hv;
                v = to_f32(hv);
            }
            ss = fmaf(v, v, ss);
        }
        ss = group_allreduce<32>(ss);
        if (lane == 0) red[it & 1][warp] = ss;
        __syncthreads();
        float total = lane < nw ? red[it & 1][lane] : 0.f;
        total = group_allreduce<32>(total);
        const float rs = rsqrtf(total / static_cast<float>(N) + eps);
        T* yr = y + row * N;
        // with ADD, h is read back from the elements this thread stored
        const T* src = ADD ? hout + row * N : xr;
        for (int j = threadIdx.x; j < N; j += blockDim.x)
            if (RMSN_OK(span_in(yr + j, sizeof(T), y, tbytes), status))
                yr[j] = P::from_float(to_f32(src[j]) * rs * to_f32(w[j]));
        if (threadIdx.x == 0 && RMSN_OK(span_in(rstd + row, 4, rstd, rbytes), status))
            rstd[row] = rs;
    }
}

template <typename T, typename TW, int G, int V, int R>
cudaError_t launch_rowgroup(const rmsnorm_plan_t& p, const FwdArgs& a, cudaStream_t s) {
    auto fn = a.res != nullptr ? fwd_rowgroup_kernel<T, TW, G, V, R, true>
                               : fwd_rowgroup_kernel<T, TW, G, V, R, false>;
    return launch_pdl(fn, p.grid, p.threads, 0, 1, s, static_cast<const T*>(a.x),
                      static_cast<const TW*>(a.w), static_cast<T*>(a.y), a.rstd, a.M, a.N, a.eps,
                      static_cast<const T*>(a.res), static_cast<T*>(a.h), a.status);
}

template <typename T, typename TW>
cudaError_t dispatch_rowgroup(const rmsnorm_plan_t& p, const FwdArgs& a, cudaStream_t s) {
    const int G = p.threads_per_row, V = p.vectors_per_thread;
    const int R = p.rows_per_unit / (p.threads / G);
    if (G == 4 && V == 1 && R == 4) return launch_rowgroup<T, TW, 4, 1, 4>(p, a, s);
    if (G == 4 && V == 2 && R == 2) return launch_rowgroup<T, TW, 4, 2, 2>(p, a, s);
    if (G == 8 && V == 2 && R == 2) return launch_rowgroup<T, TW, 8, 2, 2>(p, a, s);
    if (G == 8 && V == 4 && R == 1) return launch_rowgroup<T, TW, 8, 4, 1>(p, a, s);
    if (G == 16 && V == 4 && R == 1) return launch_rowgroup<T, TW, 16, 4, 1>(p, a, s);
    if (G == 32 && V == 4 && R == 1) return launch_rowgroup<T, TW, 32, 4, 1>(p, a, s);
    if (G == 32 && V == 8 && R == 1) return launch_rowgroup<T, TW, 32, 8, 1>(p, a, s);
    return cudaErrorInvalidValue;
}

template <typename T, typename TW, int V>
cudaError_t launch_row(const rmsnorm_plan_t& p, const FwdArgs& a, cudaStream_t s) {
    auto fn = a.res != nullptr ? fwd_row_kernel<T, TW, V, true> : fwd_row_kernel<T, TW, V, false>;
    return launch_pdl(fn, p.grid, p.threads, 0, p.cluster, s, static_cast<const T*>(a.x),
                      static_cast<const TW*>(a.w), static_cast<T*>(a.y), a.rstd, a.M, a.N, a.eps,
                      a.status, a.wait_limit_ns, static_cast<const T*>(a.res),
                      static_cast<T*>(a.h));
}

template <typename T, typename TW>
cudaError_t dispatch_row(const rmsnorm_plan_t& p, const FwdArgs& a, cudaStream_t s) {
    return p.vectors_per_thread == 4 ? launch_row<T, TW, 4>(p, a, s) : cudaErrorInvalidValue;
}

template <typename T, typename TW>
const void* ring_kernel(int V, bool add) {
    if (V == 4) return add ? reinterpret_cast<const void*>(&fwd_ring_kernel<T, TW, 4, true>)
                           : reinterpret_cast<const void*>(&fwd_ring_kernel<T, TW, 4, false>);
    if (V == 8) return add ? reinterpret_cast<const void*>(&fwd_ring_kernel<T, TW, 8, true>)
                           : reinterpret_cast<const void*>(&fwd_ring_kernel<T, TW, 8, false>);
    return nullptr;
}

const void* ring_kernel_for(int dtype, int V, bool add) {
    switch (dtype) {
        case RMSNORM_BF16: return ring_kernel<__nv_bfloat16, __nv_bfloat16>(V, add);
        case RMSNORM_F16: return ring_kernel<__half, __half>(V, add);
        case RMSNORM_BF16_W_F32: return ring_kernel<__nv_bfloat16, float>(V, add);
        case RMSNORM_F16_W_F32: return ring_kernel<__half, float>(V, add);
        case RMSNORM_F32: return ring_kernel<float, float>(V, add);
        default: return nullptr;
    }
}

// A ring grid of clusters is launched in plain stream order. Launched early
// (programmatic serialization) while the previous kernel still held SMs, its
// persistent clusters ran the steady forward + backward step of 2048 x 65536
// rows at 74% (bf16) and 82% (fp32) of the copy roofline against 92% in
// stream order; single-block ring grids and every other kernel gain from the
// early launch.
template <typename T, typename TW, int V, bool ADD>
cudaError_t launch_ring(const rmsnorm_plan_t& p, const FwdArgs& a, cudaStream_t s) {
    return launch_ex(fwd_ring_kernel<T, TW, V, ADD>, p.grid, p.threads,
                     static_cast<size_t>(p.smem_bytes), p.cluster, s, p.cluster <= 1,
                     static_cast<const T*>(a.x),
                     static_cast<const TW*>(a.w), static_cast<T*>(a.y), a.rstd, a.M, a.N, a.eps,
                     p.stages, a.status, a.wait_limit_ns, static_cast<const T*>(a.res),
                     static_cast<T*>(a.h), a.drop_unit);
}

template <typename T, typename TW>
cudaError_t dispatch_ring(const rmsnorm_plan_t& p, const FwdArgs& a, cudaStream_t s) {
    const bool add = a.res != nullptr;
    if (p.vectors_per_thread == 4)
        return add ? launch_ring<T, TW, 4, true>(p, a, s) : launch_ring<T, TW, 4, false>(p, a, s);
    if (p.vectors_per_thread == 8)
        return add ? launch_ring<T, TW, 8, true>(p, a, s) : launch_ring<T, TW, 8, false>(p, a, s);
    return cudaErrorInvalidValue;
}

template <typename T, typename TW>
cudaError_t dispatch(const rmsnorm_plan_t& p, const FwdArgs& a, cudaStream_t s) {
    if (p.variant == RMSNORM_VARIANT_RING) return dispatch_ring<T, TW>(p, a, s);
    if (p.variant == RMSNORM_VARIANT_TWO_PASS) {
        auto fn = a.res != nullptr ? fwd_wide_kernel<T, TW, 4, true> : fwd_wide_kernel<T, TW, 4, false>;
        return launch_pdl(fn, p.grid, p.threads, 0, 1, s, static_cast<const T*>(a.x),
                          static_cast<const TW*>(a.w), static_cast<T*>(a.y), a.rstd, a.M, a.N,
                          a.eps, static_cast<const T*>(a.res), static_cast<T*>(a.h), a.status);
    }
    switch (p.variant) {
        case RMSNORM_VARIANT_ROWGROUP: return dispatch_rowgroup<T, TW>(p, a, s);
        case RMSNORM_VARIANT_CTA_ROW:
        case RMSNORM_VARIANT_CLUSTER_ROW: return dispatch_row<T, TW>(p, a, s);
        case RMSNORM_VARIANT_SCALAR:
        {
            auto fn = a.res != nullptr ? fwd_scalar_kernel<T, TW, true> : fwd_scalar_kernel<T, TW, false>;
            return launch_pdl(fn, p.grid, p.threads, 0, 1, s, static_cast<const T*>(a.x),
                              static_cast<const TW*>(a.w), static_cast<T*>(a.y), a.rstd, a.M, a.N,
                              a.eps, static_cast<const T*>(a.res), static_cast<T*>(a.h),
                              a.status);
        }
        default: return cudaErrorInvalidValue;
    }
}

// Resident blocks (or clusters) of a ring kernel configuration, cached per
// (device, kernel, shape) so every call sees the same persistent grid; the
// kernel is opted into the device's largest dynamic shared memory once.
std::mutex g_ring_mu;
std::map<std::tuple<int, const void*, int, int, int>, int> g_ring_units;
std::map<std::pair<int, const void*>, bool> g_ring_optin;

cudaError_t ring_resident_units(const DeviceInfo& dev, const void* fn, int threads, int smem,
                                int cluster, int* out) {
    std::lock_guard<std::mutex> lk(g_ring_mu);
    const auto key = std::make_tuple(dev.device, fn, threads, smem, cluster);
    auto it = g_ring_units.find(key);
    if (it != g_ring_units.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    cudaError_t err = cudaSuccess;
    if (!g_ring_optin[std::make_pair(dev.device, fn)]) {
        cudaFuncAttributes fa;
        err = cudaFuncGetAttributes(&fa, fn);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       dev.max_smem_optin - static_cast<int>(fa.sharedSizeBytes));
        if (err != cudaSuccess) return err;
        g_ring_optin[std::make_pair(dev.device, fn)] = true;
    }
    int units = 0;
    if (cluster <= 1) {
        int per_sm = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
        units = per_sm * dev.sm_count;
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(cluster * dev.sm_count));
        cfg.blockDim = dim3(static_cast<unsigned>(threads));
        cfg.dynamicSmemBytes = static_cast<size_t>(smem);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        err = cudaOccupancyMaxActiveClusters(&units, fn, &cfg);
    }
    if (err != cudaSuccess) return err;
    if (units < 1) return cudaErrorInvalidConfiguration;
    g_ring_units[key] = units;
    *out = units;
    return cudaSuccess;
}

}  // namespace

// Mid rows: a block holds the row in registers (4 vectors per thread). Wider
// rows: the persistent ring kernel, a cluster of up to 8 blocks holding the
// row in registers, or the two-pass kernel. RMSNORM_FWD_WIDE (cluster |
// two_pass | ring), RMSNORM_FWD_ROW_THREADS and RMSNORM_FWD_CLUSTER_THREADS
// override the choices below for sweeps.
// Measured on GB300: bf16 rows do best in one block of up to 256 threads and,
// wider, in the ring kernel (N = 12288: 94% against 82% for a block of 384
// threads; N = 16384: 95% against 92%; N = 32768: 94% against 91% two-pass;
// N = 65536: 92% against 86%; N = 196608 and 262144, 16-bit slices of 8
// vectors: 94% and 91% against 74% and 70%); fp16 rows, the same bytes per
// element, follow bf16. fp32 rows do best in blocks of at most 256 threads,
// then in clusters of 2, then in the ring kernel (N = 16384: 96% against 90%
// for a cluster of 4; N = 65536: 96% against 72% for a cluster of 8; wider,
// up to 32768 vectors); with the residual, fp32 rows stay in clusters, and
// every row the ring cannot hold takes the two-pass kernel.
struct FwdTuning {
    int wide = -1;             // -1: per dtype; 0: two passes; 1: clusters; 2: ring
    int row_threads = 0;       // largest block holding a row (0: per dtype)
    int cluster_threads = 256; // block size aimed at in a cluster
    int ring_min_vec = 0;      // rows of at least this many vectors take the ring (0: ladder)
    int ring_cluster = 0;      // blocks of the ring kernel's cluster (0: ladder)
    int ring_smem = 200 * 1024;  // shared memory the ring's stages aim at per block
    int wide_select = 2;       // ring clusters shaped on the device: 0 never, 1 without the
                               // residual, 2 always
    int rowgroup_max_vec = -1; // widest row (16-byte vectors) for the short-row kernel
                               // (-1: 256, or 128 with the residual)
    // largest stage budget the device choice tries: with 200 KB rings as
    // well, the deeper ring won the ties and bf16 rows of 32768 and 98304 ran
    // their forward at 94.6% and 84.8% of the copy roofline, against 96.2%
    // and 85.9% with 100 KB (other widths unchanged)
    int ring_max_budget = 100 * 1024;
    // most vectors a thread of a 16-bit ring slice: 0 by width (below), 4, or
    // 8 (the slice re-read from its stage, up to 4096 vectors a block)
    int ring16_max_v = 0;
};

const FwdTuning& fwd_tuning() {
    static const FwdTuning t = [] {
        FwdTuning u;
        const char* wide = getenv("RMSNORM_FWD_WIDE");
        if (wide != nullptr && std::string(wide) == "cluster") u.wide = 1;
        if (wide != nullptr && std::string(wide) == "two_pass") u.wide = 0;
        if (wide != nullptr && std::string(wide) == "ring") u.wide = 2;
        const char* rt = getenv("RMSNORM_FWD_ROW_THREADS");
        if (rt && *rt) u.row_threads = std::max(64, std::min(1024, atoi(rt) / 32 * 32));
        const char* ct = getenv("RMSNORM_FWD_CLUSTER_THREADS");
        if (ct && *ct) u.cluster_threads = std::max(64, std::min(1024, atoi(ct) / 32 * 32));
        const char* rm = getenv("RMSNORM_FWD_RING_MIN_VEC");
        if (rm && *rm) u.ring_min_vec = std::max(0, atoi(rm));
        const char* rc = getenv("RMSNORM_FWD_RING_CLUSTER");
        if (rc && *rc) u.ring_cluster = std::max(0, std::min(kMaxCluster, atoi(rc)));
        const char* rs = getenv("RMSNORM_FWD_RING_SMEM");
        if (rs && *rs) u.ring_smem = std::max(16 * 1024, std::min(227 * 1024, atoi(rs)));
        const char* ws = getenv("RMSNORM_WIDE_SELECT");
        if (ws && *ws) u.wide_select = std::max(0, std::min(2, atoi(ws)));
        const char* rb = getenv("RMSNORM_FWD_RING_MAX_BUDGET");
        if (rb && *rb) u.ring_max_budget = std::max(16 * 1024, std::min(227 * 1024, atoi(rb)));
        const char* r16 = getenv("RMSNORM_FWD_RING16_V");
        if (r16 && *r16) u.ring16_max_v = atoi(r16) >= 8 ? 8 : 4;
        const char* gm = getenv("RMSNORM_FWD_ROWGROUP_MAX_VEC");
        if (gm && *gm) u.rowgroup_max_vec = std::max(0, std::min(256, atoi(gm)));
        return u;
    }();
    return t;
}

// Most vectors a thread of a ring slice: 8 for 32-bit elements. A 16-bit
// slice of 8 vectors is read from its stage twice (its unpacked pairs would
// not fit in registers), which pays in one block of 256-384 threads
// (fwd_ring_plan) and where 4 vectors a thread would need clusters of more
// than 4 blocks, rows wider than 8192 vectors. There, clusters of 4 blocks
// of 8 vectors (up to 144 SMs busy) ran the forward at
// 91-92% of the copy roofline for bf16 and fp16 N = 131072, against 76% for
// 8 blocks of 4 vectors (15 clusters, 120 SMs), and bf16 N = 98304 at 94%
// against 83%; at N = 65536 (91% against 94%) and 32768 (one block: cold
// 95% against 92%, back to back 87% against 92%) 4 vectors stay.
constexpr int64_t kRing16WideVec = 8192;
// 16-bit rows one block takes at 8 vectors a thread (below)
constexpr int64_t kRing16OneBlockMin = 2048;
constexpr int64_t kRing16OneBlockMax = 3072;

int ring_max_v(int elem, int64_t nvec) {
    if (elem == 4) return 8;
    const int knob = fwd_tuning().ring16_max_v;
    if (knob > 0) return knob;
    return nvec > kRing16WideVec ? 8 : 4;
}

// The ring plan for rows of nvec vectors over c blocks: 4 vectors a thread,
// or 8 where max_v allows it and 4 would need more than 512 threads (or
// where want_v8 asks for it), and as many stages, 3 to 6, as `budget` bytes
// of shared memory hold.
bool ring_plan_c(int64_t nvec, int nt, int elem, int c, int max_v, int budget,
                 rmsnorm_plan_t* p, bool want_v8 = false) {
    constexpr int kSmemMax = 227 * 1024;
    const int64_t slots = cdiv(nvec, c);
    if (slots > (max_v >= 8 ? 4096 : 2048)) return false;
    const int v = (slots > 2048 || (want_v8 && max_v >= 8)) ? 8 : 4;
    const int t = std::max(32, round_up(static_cast<int>(cdiv(slots, v)), 32));
    const int unit = v * t * 16;
    int stages = std::min(6, budget / (nt * unit));
    while (stages > 3 && fwd_ring_smem_bytes(stages, unit, nt) > kSmemMax) --stages;
    if (stages < 3 || fwd_ring_smem_bytes(stages, unit, nt) > kSmemMax) return false;
    p->variant = RMSNORM_VARIANT_RING;
    p->cluster = c;
    p->vectors_per_thread = v;
    p->threads = t;
    p->threads_per_row = t * c;
    p->stages = stages;
    p->smem_bytes = fwd_ring_smem_bytes(stages, unit, nt);
    return true;
}

// The persistent ring kernel for a row of nvec vectors: the smallest cluster
// (1, 2, 4, then 8 blocks) whose blocks hold a slice of at most 4096 vectors
// (512 threads x 8; 2048 for 16-bit elements) with room for at least three
// ring stages in about 200 KB of shared memory. nt tensors ride in the ring
// (2 with the residual).
bool fwd_ring_plan(int64_t nvec, int nt, int elem, rmsnorm_plan_t* p) {
    const FwdTuning& tu = fwd_tuning();
    const int max_v = ring_max_v(elem, nvec);
    // 16-bit rows of 2048-3072 vectors (N = 16384-24576), no residual: one
    // block of 256-384 threads at 8 vectors a thread, the slice read twice
    // from a ring at least four stages deep. Against 512 threads at 4 vectors
    // (N = 16384) or clusters of 2 (wider) it ran the forward at 97 / 97%
    // (cold / back to back) against 96 / 85% for bf16 N = 16384, 97 / 99%
    // against 94 / 91% at 18432, and 93-95 / 85-86% against 93 / 83-85% at
    // 20480 and 24576; fp16 N = 16384 lost 2.6 points cold (94%) and gained
    // 1.3 on the forward + backward step. Three stages (wider rows) lost back
    // to back, and fewer than 256 threads (narrower rows) lost both ways.
    if (tu.ring_cluster == 0 && tu.ring16_max_v != 4 && elem == 2 && nt == 1 &&
        nvec >= kRing16OneBlockMin && nvec <= kRing16OneBlockMax) {
        rmsnorm_plan_t q = *p;
        if (ring_plan_c(nvec, nt, elem, 1, 8, tu.ring_smem, &q, true) && q.stages >= 4) {
            *p = q;
            return true;
        }
    }
    if (tu.ring_cluster > 0) return ring_plan_c(nvec, nt, elem, tu.ring_cluster, max_v, tu.ring_smem, p);
    for (int c = 1; c <= kMaxCluster; c *= 2)
        if (ring_plan_c(nvec, nt, elem, c, max_v, tu.ring_smem, p)) return true;
    return false;
}

void fwd_choose(int64_t N, int dtype, bool vector_ok, rmsnorm_plan_t* p, bool add) {
    *p = rmsnorm_plan_t{};
    p->stages = 0;
    p->cluster = 1;
    p->row_groups = 1;
    p->rows_per_unit = 1;
    const int64_t nvec = N / dtype_vec(dtype);
    const FwdTuning& tu = fwd_tuning();
    // With the residual, a lane of the short-row kernel holds 8 vectors of x
    // and 8 of the residual at 129..256 vectors a row; a block per row (4
    // vectors of each a thread) ran 8..20 points of the copy roofline faster
    // there. Without it the short-row kernel stays ahead.
    const int64_t rowgroup_max_vec = tu.rowgroup_max_vec >= 0 ? tu.rowgroup_max_vec
                                     : add ? 128 : 256;
    GroupShape g;
    if (vector_ok && nvec <= rowgroup_max_vec && fwd_group_shape(nvec, &g)) {
        p->variant = RMSNORM_VARIANT_ROWGROUP;
        p->threads = g.threads;
        p->threads_per_row = g.G;
        p->vectors_per_thread = g.V;
        p->rows_per_unit = (g.threads / g.G) * g.R;
        return;
    }
    const bool half = dtype_size(dtype) == 2;  // 16-bit activations
    // the ring kernel from this many vectors on: 16-bit rows wider than 256
    // threads x 4 vectors, and, with an fp32 weight and no residual, every
    // row past the short-row kernel (its block per row holds twice the weight
    // registers: 75-92% against 88-95% in the ring; with the residual the
    // block per row stays ahead). RMSNORM_FWD_RING_MIN_VEC overrides.
    const bool wide_weight = weight_size(dtype) > dtype_size(dtype);
    const int64_t ring_from = tu.ring_min_vec > 0 ? tu.ring_min_vec
                              : (wide_weight && !add) ? 257
                              : half ? 1025 : INT64_MAX;
    if (vector_ok && tu.wide < 0 && nvec >= ring_from &&
        fwd_ring_plan(nvec, add ? 2 : 1, dtype_size(dtype), p))
        return;
    const bool clusters = tu.wide >= 0 ? tu.wide == 1 : !half;
    const int row_cap = dtype_size(dtype) == weight_size(dtype) ? 1024 : 512;
    // one block per row up to this many threads, clusters beyond: fp32 rows in
    // one block of up to 384 threads ran their forward at 103% of the copy
    // roofline (N = 4352 to 6144) against 92-97% as pairs of blocks, while at
    // 448 and 512 threads (N = 7168, 8192) the pairs ran 1-1.5 points ahead
    // (the row kernel holds fp32 weights only for the scaling, 46 registers)
    const int row_threads = std::min(row_cap, tu.row_threads > 0 ? tu.row_threads
                                              : half ? 512 : add ? 256 : 384);
    if (vector_ok && nvec <= static_cast<int64_t>(row_threads) * 4) {
        p->variant = RMSNORM_VARIANT_CTA_ROW;
        p->vectors_per_thread = 4;
        p->threads = round_up(static_cast<int>(cdiv(nvec, 4)), 32);
        p->threads_per_row = p->threads;
        return;
    }
    const bool ladder = tu.wide < 0;  // no override
    // 16-bit rows too wide for one block (and any such row under
    // RMSNORM_FWD_WIDE=ring): the persistent ring kernel
    if (vector_ok && (tu.wide == 2 || (ladder && half)) &&
        fwd_ring_plan(nvec, add ? 2 : 1, dtype_size(dtype), p))
        return;
    if (vector_ok && clusters) {
        int c = 1, v = 4;
        while (cdiv(nvec, c) > static_cast<int64_t>(tu.cluster_threads) * v && c < kMaxCluster) c *= 2;
        if (cdiv(nvec, c) <= 512 * v) {
            // fp32 rows that need four or more blocks: the ring kernel
            // (measured faster there, though not with the residual)
            if (ladder && !add && c >= 4 && fwd_ring_plan(nvec, 1, dtype_size(dtype), p)) return;
            const int64_t slots = cdiv(nvec, c);
            p->variant = c > 1 ? RMSNORM_VARIANT_CLUSTER_ROW : RMSNORM_VARIANT_CTA_ROW;
            p->cluster = c;
            p->vectors_per_thread = v;
            p->threads = round_up(static_cast<int>(cdiv(slots, v)), 32);
            p->threads_per_row = p->threads * c;
            return;
        }
        // fp32 rows too wide for a cluster of blocks that hold them: the
        // ring kernel, 8 vectors a thread over up to 8 blocks (N = 98304 and
        // 131072: 100% and 93% of the copy roofline against 60% and 57% for
        // the two-pass kernel)
        if (ladder && !add && fwd_ring_plan(nvec, 1, dtype_size(dtype), p)) return;
    }
    if (vector_ok) {
        p->variant = RMSNORM_VARIANT_TWO_PASS;
        p->vectors_per_thread = 4;
        // blocks per SM: rows in flight must stay far below L2; one block of
        // 1024 threads for rows over 128 KB, else two of 512
        p->rows_per_unit = N * dtype_size(dtype) > 128 * 1024 ? 1 : 2;
        p->threads = p->rows_per_unit == 1 ? 1024 : 512;
        p->threads_per_row = p->threads;
        return;
    }
    p->variant = RMSNORM_VARIANT_SCALAR;
    p->threads = 256;
    p->threads_per_row = 256;
    p->vectors_per_thread = 0;
}

namespace {

// Ring plans chosen on a device, per (device, dtype, N).
std::mutex g_ring_sel_mu;
std::map<std::tuple<int, int, int64_t, bool>, rmsnorm_plan_t> g_ring_sel;

// A row split over a ring cluster runs best where the clusters resident at
// once times the threads resident with them is largest; ties go to more
// resident blocks (two to an SM hide each other's per-row exchanges), then to
// the deeper ring. The occupancy API counts them for cluster sizes 2, 4, 5, 6
// and 8, four vectors a thread (also eight for fp32 rows) and stage budgets
// of 100 and 200 KB (the residual rides in the ring too when there is one).
// On GB300 this took bf16 N = 40960..57344 from 73..85% of the copy roofline
// to 94..95% and N = 98304 from 69% to 85% (with the residual: 93% to 100%).
cudaError_t ring_select(const DeviceInfo& dev, int dtype, int64_t N, bool add, rmsnorm_plan_t* p) {
    const auto key = std::make_tuple(dev.device, dtype, N, add);
    {
        std::lock_guard<std::mutex> lk(g_ring_sel_mu);
        auto it = g_ring_sel.find(key);
        if (it != g_ring_sel.end()) {
            *p = it->second;
            return cudaSuccess;
        }
    }
    const int elem = dtype_size(dtype);
    const int64_t nvec = N / dtype_vec(dtype);
    rmsnorm_plan_t best = *p;
    int64_t best_score[3] = {-1, -1, -1};
    for (int c : {2, 4, 5, 6, 8}) {
        for (int max_v : {4, 8}) {
            if (max_v > ring_max_v(elem, nvec)) continue;
            for (int budget : {100 * 1024, 200 * 1024}) {
                rmsnorm_plan_t q = *p;
                if (!ring_plan_c(nvec, add ? 2 : 1, elem, c, max_v, budget, &q)) continue;
                // past the budget cap only 16-bit slices of 8 vectors, whose
                // three stages at 512 threads take 192 KB
                if (budget > fwd_tuning().ring_max_budget &&
                    !(elem == 2 && q.vectors_per_thread == 8))
                    continue;
                if (q.smem_bytes > dev.max_smem_optin) continue;
                const void* fn = ring_kernel_for(dtype, q.vectors_per_thread, add);
                if (fn == nullptr) continue;
                int units = 0;
                if (ring_resident_units(dev, fn, q.threads, q.smem_bytes, c, &units) != cudaSuccess ||
                    units < 1) {
                    cudaGetLastError();  // an occupancy query that fails rules the shape out
                    continue;
                }
                // rows in flight times resident threads, then resident blocks
                const int64_t blocks = static_cast<int64_t>(units) * c;
                const int64_t score[3] = {units * blocks * q.threads, blocks, q.stages};
                if (std::lexicographical_compare(best_score, best_score + 3, score, score + 3)) {
                    best = q;
                    std::copy(score, score + 3, best_score);
                }
            }
        }
    }
    std::lock_guard<std::mutex> lk(g_ring_sel_mu);
    g_ring_sel[key] = best;
    *p = best;
    return cudaSuccess;
}

}  // namespace

cudaError_t fwd_finish_plan(const DeviceInfo& dev, int dtype, int64_t M, int64_t N,
                            rmsnorm_plan_t* p, bool add) {
    const FwdTuning& tu = fwd_tuning();
    if (p->variant == RMSNORM_VARIANT_RING && p->cluster >= 2 && tu.ring_cluster == 0 &&
        tu.ring_smem == 200 * 1024 && tu.wide_select >= (add ? 2 : 1)) {
        cudaError_t e = ring_select(dev, dtype, N, add, p);
        if (e != cudaSuccess) return e;
    }
    switch (p->variant) {
        case RMSNORM_VARIANT_RING: {
            const void* fn = ring_kernel_for(dtype, p->vectors_per_thread, add);
            if (fn == nullptr) return cudaErrorInvalidValue;
            int units = 0;
            cudaError_t e = ring_resident_units(dev, fn, p->threads, p->smem_bytes, p->cluster, &units);
            if (e != cudaSuccess) return e;
            p->grid = static_cast<int>(std::min<int64_t>(M, units) * p->cluster);
            break;
        }
        case RMSNORM_VARIANT_ROWGROUP:
            p->grid = static_cast<int>(cdiv(M, p->rows_per_unit));
            break;
        case RMSNORM_VARIANT_CTA_ROW:
        case RMSNORM_VARIANT_CLUSTER_ROW:
            p->grid = static_cast<int>(M * p->cluster);
            break;
        case RMSNORM_VARIANT_TWO_PASS:
            // rows_per_unit blocks per SM walk all rows (a smaller grid, to keep
            // fewer rows in L2, ran slower in proportion at N = 196608..1048576)
            p->grid = static_cast<int>(
                std::min<int64_t>(M, static_cast<int64_t>(p->rows_per_unit) * dev.sm_count));
            break;
        case RMSNORM_VARIANT_SCALAR:
            p->grid = static_cast<int>(std::min<int64_t>(M, static_cast<int64_t>(dev.sm_count) * 64));
            break;
        default:
            p->grid = 0;
    }
    return cudaSuccess;
}

cudaError_t fwd_launch(const rmsnorm_plan_t& p, int dtype, const FwdArgs& a, cudaStream_t s) {
    if (p.grid <= 0) return cudaSuccess;
    switch (dtype) {
        case RMSNORM_BF16: return dispatch<__nv_bfloat16, __nv_bfloat16>(p, a, s);
        case RMSNORM_F16: return dispatch<__half, __half>(p, a, s);
        case RMSNORM_BF16_W_F32: return dispatch<__nv_bfloat16, float>(p, a, s);
        case RMSNORM_F16_W_F32: return dispatch<__half, float>(p, a, s);
        case RMSNORM_F32: return dispatch<float, float>(p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rmsn
