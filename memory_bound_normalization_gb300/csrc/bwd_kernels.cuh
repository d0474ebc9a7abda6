// RMSNorm backward kernels (device side; bwd.cu plans and launches them,
// bwd_f32.cu / bwd_bf16.cu / bwd_f16.cu instantiate them per element type).
//
//   xhat = x * rstd, g = dy * w
//   dx   = rstd * (g - xhat * mean_j(g * xhat))
//   dw   = sum over rows of dy * xhat
//
// Definitions: "RMSNorm backward (almost) without the column reduction",
// sections "The backward pass" (the gradients) and "The problem: summing
// across rows" (no float atomics: their order changes the bits run to run).
// Structure follows that page's section "The persistent kernel": the grid is
// sized by the machine (resident blocks per SM times SMs, at most one block
// per row), block b walks rows b, b+P, b+2P, ..., keeps its dw contribution
// in registers across those rows and writes one partial row at the end; a
// second kernel sums the P partial rows in a fixed order. The next rows are
// prefetched into a shared-memory ring while the current row is computed.
//
// What differs from that page's kernel: rows land through 1-D bulk copies
// (cp.async.bulk, completion counted on an mbarrier) instead of per-thread
// cp.async; the ring depth is a parameter (2-4 stages) rather than 2; rstd is
// read from the forward (as the Quack backward does, "What a tuned RMSNorm
// kernel actually costs on Hopper", section 05) rather than recomputed, so a
// row needs one reduction, not two; rows may be split over a thread-block
// cluster with the row sum exchanged through distributed shared memory; and
// short rows move as tiles of whole rows. Every wait on a copy is bounded in
// time and reports a status instead of hanging.
//
// Types: T is the activation type (x, dy, dx), TW the weight type (T, or
// fp32 with 16-bit activations). rstd, the dw partial rows and dw are fp32.
//
// RES (residual path): x is the stored sum h = x + res of the forward, and
// dx = rstd*(g - xhat*c) + dres, where dres is the gradient reaching h from
// its other uses; that dx is the gradient of both summands ("Profiling, GPU
// utilisation and writing a fused kernel", Problem 15, the residual step).
// dres travels through the bulk-copy ring as a third tensor beside x and dy,
// so pass 2 reads it from shared memory; the copy of a row lands before that
// row's dx is written, so dx may be the dres buffer.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace rmsn {

// The rings hold nt tensors per stage: x and dy, plus dres on the residual
// path (nt = 3).
//
// Shared memory of the short-row kernel: [S][unit] x | [S][unit] dy |
// ([S][unit] dres) | mbarrier[S] | 66 floats of reduction slots | failure flag.
__host__ __device__ inline int bwd_smem_bytes(int stages, int unit, int nt = 2) {
    return nt * stages * unit + stages * 8 + 64 * 4 + 2 * 4 + 16;
}

// Shared memory of the grouped row kernel, per group: [S][unit] x |
// [S][unit] dy | ([S][unit] dres) | mbarrier[S] | reduction slots [2][32] |
// failure flag, padded to a multiple of 128 bytes so that every group's ring
// starts 16-byte aligned (bulk copies and 16-byte shared loads need it).
__host__ __device__ inline int bwd_row_group_stride(int stages, int unit, int nt = 2) {
    return (nt * stages * unit + stages * 8 + 64 * 4 + 16 + 127) / 128 * 128;
}

// Shared memory of the wide-row kernel: [S][unit] x | [S][unit] dy |
// ([S][unit] dres) | mbarrier[S] (copies) | mbarrier[4] (cluster exchange) |
// reduction slots [2][32] | exchange slots [4][kMaxClusterSize] | failure flag.
constexpr int kMaxClusterSize = 16;
__host__ __device__ inline int bwd_wide_smem_bytes(int stages, int unit, int nt = 2) {
    return nt * stages * unit + stages * 8 + 4 * 8 + 64 * 4 + 4 * kMaxClusterSize * 4 + 16;
}
__host__ __device__ inline int bwd_row_smem_bytes(int groups, int stages, int unit, int nt = 2) {
    return groups * bwd_row_group_stride(stages, unit, nt);
}

// Main (row) kernel of a backward plan for each element-type code, without
// (bwd_main_kernel_*) and with (bwd_res_kernel_*) the residual gradient. Each
// is defined in its own translation unit, so the instantiations compile in
// parallel; nullptr when the plan names no instantiated kernel.
const void* bwd_main_kernel_f32(const rmsnorm_plan_t& p, bool pipelined);
const void* bwd_main_kernel_bf16(const rmsnorm_plan_t& p, bool pipelined);
const void* bwd_main_kernel_bf16_w_f32(const rmsnorm_plan_t& p, bool pipelined);
const void* bwd_main_kernel_f16(const rmsnorm_plan_t& p, bool pipelined);
const void* bwd_main_kernel_f16_w_f32(const rmsnorm_plan_t& p, bool pipelined);
const void* bwd_res_kernel_f32(const rmsnorm_plan_t& p, bool pipelined);
const void* bwd_res_kernel_bf16(const rmsnorm_plan_t& p, bool pipelined);
const void* bwd_res_kernel_bf16_w_f32(const rmsnorm_plan_t& p, bool pipelined);
const void* bwd_res_kernel_f16(const rmsnorm_plan_t& p, bool pipelined);
const void* bwd_res_kernel_f16_w_f32(const rmsnorm_plan_t& p, bool pipelined);

namespace {

// Stage of consecutive rows (or tiles) in an S-stage ring, and the parity of
// the mbarrier phase that completes it, advanced one row at a time: no
// division by the run-time S in the loops.
struct RingPos {
    int s = 0;
    uint32_t parity = 0;
    __device__ __forceinline__ void next(int S) {
        if (++s == S) {
            s = 0;
            parity ^= 1u;
        }
    }
};

__device__ __forceinline__ void group_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}


// Few rows: the grid is a single cluster, and dw is summed on chip instead of
// through partial rows in global memory and a second kernel. Every block has
// its dw contribution in its shared memory at `row` (W floats, W a multiple of
// 4, 16-byte aligned); block rank r adds the C blocks' values of its share of
// the columns in rank order and writes them to dw. The same bits on every run
// for a given cluster size. Called by every thread of every block.
__device__ __forceinline__ void cluster_rows_to_dw(const float* row, int W, float* dw,
                                                   int* status) {
    cluster_sync_all();  // every block's row is complete and visible to the cluster
    const uint32_t C = cluster_size(), r = cluster_rank();
    const int n4 = W / 4;
    const int per = (n4 + static_cast<int>(C) - 1) / static_cast<int>(C);
    const int beg = static_cast<int>(r) * per, end = min(n4, beg + per);
    for (int k = beg + static_cast<int>(threadIdx.x); k < end; k += blockDim.x) {
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (uint32_t q = 0; q < C; ++q) {
            const float4 v = ld_cluster_f32x4(row + 4 * k, q);
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
        float* d = dw + 4 * k;
        if (RMSN_OK(span_in(d, 16, dw, static_cast<int64_t>(W) * 4), status)) {
            d[0] = s.x;
            d[1] = s.y;
            d[2] = s.z;
            d[3] = s.w;
        }
    }
    cluster_sync_all();  // no block leaves while a peer still reads its row
}

// ------------------------------------------------------ row groups per block
// A block holds `groups` independent row groups of TG = blockDim.x / groups
// threads. Group g of block b works as a virtual block v = b*groups + g of
// P*groups: it owns rows v, v + P*groups, ..., has its own bulk-copy ring and
// named barrier, and keeps its dw contribution in registers. At the end the
// groups' dw are added in group order, so every block writes one partial row.
template <typename T, typename TW, int V, bool RES>
__global__ void __launch_bounds__(512) bwd_row_kernel(BwdArgs a, int stages, int groups) {
    using P = Pack<T>;
    constexpr int VEC = P::VEC;
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x;
    const int TG = blockDim.x / groups;
    const int g = tid / TG, gt = tid % TG;
    const int gwarp = gt >> 5, lane = tid & 31, gnw = TG >> 5;
    const int64_t cid = blockIdx.x;
    const int64_t ncl = gridDim.x;
    const int64_t vid = cid * groups + g;       // virtual block of this group
    const int64_t nvirt = ncl * groups;
    const int N = a.N;
    const float inv_n = 1.f / static_cast<float>(N);  // mean = sum * inv_n, one multiply a row
    const int nvec = N / VEC;
    const int slots = V * TG;
    const int vbeg = 0;
    const int vcnt = min(slots, nvec);
    const uint32_t bytes = static_cast<uint32_t>(vcnt) * 16u;
    const int S = stages;
    const int unit = slots * 16;

    constexpr int NT = RES ? 3 : 2;  // tensors in the ring
    const int gstride = bwd_row_group_stride(S, unit, NT);
    unsigned char* gbase = smem + g * gstride;
    unsigned char* sx = gbase;
    unsigned char* sdy = gbase + S * unit;
    unsigned char* sdr = gbase + 2 * S * unit;  // dres (RES only)
    uint64_t* bar = reinterpret_cast<uint64_t*>(gbase + NT * S * unit);
    float* red = reinterpret_cast<float*>(bar + S);
    volatile int* fail = reinterpret_cast<volatile int*>(red + 64);

    const T* X = static_cast<const T*>(a.x);
    const T* DY = static_cast<const T*>(a.dy);
    const TW* W = static_cast<const TW*>(a.w);
    T* DX = static_cast<T*>(a.dx);
    const T* DRES = static_cast<const T*>(a.dres);
    // extents for the checked build: x, dy, dx, dres; the partial rows
    [[maybe_unused]] const int64_t tbytes =
        a.M * static_cast<int64_t>(N) * static_cast<int64_t>(sizeof(T));
    [[maybe_unused]] const int64_t pbytes = ncl * static_cast<int64_t>(N) * 4;
    const int bar_id = 1 + g;  // named barrier of this group (0 is __syncthreads)

    // rows of this group: vid, vid + nvirt, ...
    const int64_t nrows = vid < a.M ? (a.M - 1 - vid) / nvirt + 1 : 0;

    if (gt == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
        *fail = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    wait_for_prerequisite_grid();  // no global access before this

    // Producer state, meaningful in the group's thread 0 only: stages with a
    // copy in flight and the parity of the phase that copy completes.
    uint32_t pending = 0, pending_parity = 0;
    RingPos prod;  // ring position of the next row to issue (issued in order)
    auto issue = [&](int64_t t) {
        const int s = prod.s;
        const uint32_t par = prod.parity;
        prod.next(S);
        const int64_t row = vid + t * nvirt;
        if (bytes == 0) {
            mbar_arrive(&bar[s]);
            return;
        }
        mbar_arrive_expect_tx(&bar[s], static_cast<uint32_t>(NT) * bytes);
        if (row == a.drop_unit) return;  // failure injection: this wait runs out
        const int64_t off = row * N + static_cast<int64_t>(vbeg) * VEC;
        if (!RMSN_OK(span_in(X + off, bytes, X, tbytes) && span_in(DY + off, bytes, DY, tbytes) &&
                         smem_span_in(sx + s * unit, bytes) && smem_span_in(sdy + s * unit, bytes) &&
                         (!RES || (span_in(DRES + off, bytes, DRES, tbytes) &&
                                   smem_span_in(sdr + s * unit, bytes))),
                     a.status))
            return;  // checked build: the wait for this stage runs out instead
        bulk_copy_g2s(sx + s * unit, X + off, bytes, &bar[s]);
        bulk_copy_g2s(sdy + s * unit, DY + off, bytes, &bar[s]);
        if constexpr (RES) bulk_copy_g2s(sdr + s * unit, DRES + off, bytes, &bar[s]);
        pending |= 1u << s;
        pending_parity = (pending_parity & ~(1u << s)) | (par << s);
    };
    if (gt == 0)
        for (int64_t t = 0; t < S && t < nrows; ++t) issue(t);

    // The weights of the thread's slots stay in registers across rows when
    // they take at most 8 16-byte words; more (an fp32 weight with 8 vectors
    // a thread) would spill, so those are re-read from cache at each use.
    using WP = WPack<T, TW>;
    constexpr bool kWReg = WP::WORDS * V <= 8;
    uint4 wv[kWReg ? V : 1][WP::WORDS];
    if constexpr (kWReg) {
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = j * TG + gt;
            if (k < vcnt) WP::load(W, vbeg + k, wv[j]);
            else WP::zero(wv[j]);
        }
    }
    auto weights = [&](int j, int k, float2 (&fw)[WP::PAIRS]) {
        if constexpr (kWReg) {
            WP::unpack2(wv[j], fw);
        } else {
            uint4 wq[WP::WORDS];
            WP::load(W, vbeg + k, wq);
            WP::unpack2(wq, fw);
        }
    };
    constexpr int PR = P::PAIRS;
    float2 acc[V][PR];
#pragma unroll
    for (int j = 0; j < V; ++j)
#pragma unroll
        for (int e = 0; e < PR; ++e) acc[j][e] = make_float2(0.f, 0.f);

    // rstd is read two rows ahead so its latency hides behind the rows before
    float r1 = nrows > 0 ? __ldg(a.rstd + vid) : 0.f;
    float r2 = nrows > 1 ? __ldg(a.rstd + vid + nvirt) : 0.f;
    bool failed = false;  // a copy wait ran out in this group

    const bool early = a.early_refill != 0;  // refill a stage after pass 2 of its row
    RingPos cons;  // ring position of row t
    for (int64_t t = 0; t < nrows; ++t) {
        const int64_t row = vid + t * nvirt;
        const int s = cons.s;
        const uint32_t parity = cons.parity;
        cons.next(S);
        const float r = r1;
        r1 = r2;
        if (t + 2 < nrows) r2 = __ldg(a.rstd + row + 2 * nvirt);

        if (!failed) {
            if (mbar_wait_bounded(&bar[s], parity, a.wait_limit_ns)) {
                if (gt == 0) pending &= ~(1u << s);
            } else {
                *fail = 1;
                report_status(a.status, kStatusTimeout);
            }
        }
        // pass 1: dot = sum_j (dy*w)*x over this thread's slots
        const unsigned char* xs = sx + s * unit;
        const unsigned char* ds = sdy + s * unit;
        float2 dot2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = j * TG + gt;
            if (k >= vcnt) continue;
            float2 fx[PR], fd[PR], fw[PR];
            P::unpack2(ld_ring_16(xs + k * 16, a.status), fx);
            P::unpack2(ld_ring_16(ds + k * 16, a.status), fd);
            weights(j, k, fw);
#pragma unroll
            for (int e = 0; e < PR; ++e) dot2 = __ffma2_rn(__fmul2_rn(fd[e], fw[e]), fx[e], dot2);
        }
        float dot = group_allreduce<32>(dot2.x + dot2.y);
        float* rslot = red + (t & 1) * 32;
        if (lane == 0) rslot[gwarp] = dot;
        group_barrier(bar_id, TG);  // sums published; the group is done with row t-1
        failed = *fail != 0;
        float tot = lane < gnw ? rslot[lane] : 0.f;
        tot = group_allreduce<32>(tot);
        // the stage of row t-1 is free now: refill it with row t-1+S
        if (!early && gt == 0 && !failed && t >= 1 && t - 1 + S < nrows) {
            fence_proxy_async_shared();
            issue(t - 1 + S);
        }
        // mean_j(g * xhat) = rstd * mean_j(g * x)
        const float c = r * (tot * inv_n);
        const float2 r2 = f2_splat(r), nc2 = f2_splat(-c);
        T* dxr = DX + row * N;
        // pass 2: dx = r*(g - xhat*c) and dw += dy*xhat, re-reading the row
        // from shared memory
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = j * TG + gt;
            if (k >= vcnt) continue;
            float2 fx[PR], fd[PR], fw[PR], o[PR], fr[PR];
            if constexpr (RES) P::unpack2(ld_ring_16(sdr + s * unit + k * 16, a.status), fr);
            P::unpack2(ld_ring_16(xs + k * 16, a.status), fx);
            P::unpack2(ld_ring_16(ds + k * 16, a.status), fd);
            weights(j, k, fw);
#pragma unroll
            for (int e = 0; e < PR; ++e) {
                const float2 xh = __fmul2_rn(fx[e], r2);
                const float2 gg = __fmul2_rn(fd[e], fw[e]);
                if constexpr (RES)
                    o[e] = __ffma2_rn(r2, __ffma2_rn(xh, nc2, gg), fr[e]);
                else
                    o[e] = __fmul2_rn(r2, __ffma2_rn(xh, nc2, gg));
                acc[j][e] = __ffma2_rn(fd[e], xh, acc[j][e]);
            }
            T* dst = dxr + static_cast<int64_t>(vbeg + k) * VEC;
            if (RMSN_OK(span_in(dst, 16, DX, tbytes), a.status)) st_global_16(dst, P::pack2(o));
        }
        if (early) {
            // refill row t's stage as soon as the group is done with it
            group_barrier(bar_id, TG);
            if (gt == 0 && !failed && t + S < nrows) {
                fence_proxy_async_shared();
                issue(t + S);
            }
        }
    }
    allow_dependent_launch();

    // after a failure, let copies already in flight land before going on
    if (gt == 0 && failed)
        for (int s = 0; s < S; ++s)
            if ((pending >> s) & 1u)
                mbar_wait_bounded(&bar[s], (pending_parity >> s) & 1u, a.wait_limit_ns);

    // one partial row per cluster (or block); each block writes its column slice
    float* prow = a.partial + cid * N + static_cast<int64_t>(vbeg) * VEC;
    if (a.cluster_dw) {
        // the grid is one cluster: the groups' dw meet in shared memory (group
        // order), then the blocks' rows in dw (rank order)
        __syncthreads();
        float* comb = reinterpret_cast<float*>(smem);
        const int W = vcnt * VEC;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = j * TG + gt;
            if (k >= vcnt) continue;
#pragma unroll
            for (int q = 0; q < PR / 2; ++q)
                if (float* cd = comb + g * W + k * VEC + 4 * q;
                    RMSN_OK(smem_span_in(cd, 16), a.status))
                *reinterpret_cast<float4*>(cd) =
                    make_float4(acc[j][2 * q].x, acc[j][2 * q].y, acc[j][2 * q + 1].x,
                                acc[j][2 * q + 1].y);
        }
        __syncthreads();
        if (groups > 1)
            for (int col = tid; col < W; col += blockDim.x) {
                float sum = 0.f;
                for (int gi = 0; gi < groups; ++gi)
                    sum += RMSN_OK(smem_span_in(comb + gi * W + col, 4), a.status)
                               ? comb[gi * W + col] : 0.f;
                comb[col] = sum;  // group 0's value of this column was read above
            }
        cluster_rows_to_dw(comb, W, a.dw, a.status);
    } else if (groups == 1) {
        // one partial row per cluster; each block writes its column slice
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = j * TG + gt;
            if (k >= vcnt) continue;
#pragma unroll
            for (int q = 0; q < PR / 2; ++q)
                if (float* pd = prow + static_cast<int64_t>(k) * VEC + 4 * q;
                    RMSN_OK(span_in(pd, 16, a.partial, pbytes), a.status))
                *reinterpret_cast<float4*>(pd) =
                    make_float4(acc[j][2 * q].x, acc[j][2 * q].y, acc[j][2 * q + 1].x,
                                acc[j][2 * q + 1].y);
        }
    } else {
        // add the groups' dw in group order through shared memory; the rings
        // are idle and the slice's groups*W*4 bytes (W = this block's
        // columns) fit in the groups*2*S*unit bytes of the rings
        __syncthreads();
        float* comb = reinterpret_cast<float*>(smem);
        const int W = vcnt * VEC;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = j * TG + gt;
            if (k >= vcnt) continue;
#pragma unroll
            for (int q = 0; q < PR / 2; ++q)
                if (float* cd = comb + g * W + k * VEC + 4 * q;
                    RMSN_OK(smem_span_in(cd, 16), a.status))
                *reinterpret_cast<float4*>(cd) =
                    make_float4(acc[j][2 * q].x, acc[j][2 * q].y, acc[j][2 * q + 1].x,
                                acc[j][2 * q + 1].y);
        }
        __syncthreads();
        for (int col = tid; col < W; col += blockDim.x) {
            float sum = 0.f;
            for (int gi = 0; gi < groups; ++gi)
                sum += RMSN_OK(smem_span_in(comb + gi * W + col, 4), a.status) ? comb[gi * W + col]
                                                                               : 0.f;
            if (RMSN_OK(span_in(prow + col, 4, a.partial, pbytes), a.status)) prow[col] = sum;
        }
    }
}

// ----------------------------------------------- wide rows, software-pipelined
// One row pipeline per block. A row too wide for one block is split over a
// cluster of C blocks (block rank q holds vector slots [q*V*T, (q+1)*V*T));
// otherwise C = 1. Each row goes through: wait for its bulk copy, pass 1 (the
// block's part of sum_j dy*w*x), block reduction, exchange of the C block
// sums through distributed shared memory, pass 2 (dx and the dw partial).
// The loop does pass 1 and the reduction of row t+1 before pass 2 of row t,
// so the exchange of row t is in flight while row t+1 is read.
//
// Exchange: the block's sum of row t goes to slot [t&3][q] of every block q
// of the cluster (itself included; thread q does the sending) by an
// asynchronous store whose completion counts 4 transaction bytes on that
// block's barrier [t&3]; each block arms its barrier for 4*C bytes once per
// row, waits (acquire), and adds the C slots in rank order, the same bits in
// every block. A store may land before the arming: the barrier's transaction
// count goes below zero, but the phase cannot end before the local arrival
// that comes with the arming. Four slots suffice: a
// peer sends row r+1 only after receiving row r-1, which needs this block's
// send of row r-1, made before this block reads the slots of row r-2; so a
// writer is at most three rows ahead of a reader.
template <typename T, typename TW, int V, bool PIPE, bool RES>
__global__ void __launch_bounds__(512) bwd_wide_kernel(BwdArgs a, int stages, int /*groups*/) {
    using P = Pack<T>;
    constexpr int VEC = P::VEC;
    constexpr int PR = P::PAIRS;
    extern __shared__ __align__(128) unsigned char smem[];

    const int nthr = blockDim.x, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31, nw = nthr >> 5;
    const uint32_t csize = cluster_size();
    const uint32_t crank = csize > 1 ? cluster_rank() : 0u;
    const int64_t cid = csize > 1 ? static_cast<int64_t>(cluster_index()) : blockIdx.x;
    const int64_t ncl = csize > 1 ? static_cast<int64_t>(cluster_count()) : gridDim.x;
    const int N = a.N;
    const float inv_n = 1.f / static_cast<float>(N);  // mean = sum * inv_n, one multiply a row
    const int nvec = N / VEC;
    const int slots = V * nthr;
    const int vbeg = static_cast<int>(crank) * slots;
    const int vcnt = max(0, min(slots, nvec - vbeg));
    const uint32_t bytes = static_cast<uint32_t>(vcnt) * 16u;
    const int S = stages;
    const int unit = slots * 16;

    constexpr int NT = RES ? 3 : 2;  // tensors in the ring
    unsigned char* sx = smem;
    unsigned char* sdy = smem + S * unit;
    unsigned char* sdr = smem + 2 * S * unit;  // dres (RES only)
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + NT * S * unit);
    uint64_t* xbar = bar + S;                          // [4]
    float* red = reinterpret_cast<float*>(xbar + 4);  // [2][32]
    float* xslot = red + 64;                           // [4][kMaxClusterSize]
    volatile int* fail = reinterpret_cast<volatile int*>(xslot + 4 * kMaxClusterSize);

    const T* X = static_cast<const T*>(a.x);
    const T* DY = static_cast<const T*>(a.dy);
    const TW* W = static_cast<const TW*>(a.w);
    T* DX = static_cast<T*>(a.dx);
    const T* DRES = static_cast<const T*>(a.dres);
    // extents for the checked build: x, dy, dx, dres; the partial rows
    [[maybe_unused]] const int64_t tbytes =
        a.M * static_cast<int64_t>(N) * static_cast<int64_t>(sizeof(T));
    [[maybe_unused]] const int64_t pbytes = ncl * static_cast<int64_t>(N) * 4;

    // rows of this cluster: cid, cid+ncl, ...
    const int64_t nrows = cid < a.M ? (a.M - 1 - cid) / ncl + 1 : 0;

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
    RingPos prod;  // ring position of the next row to issue (issued in order)
    auto issue = [&](int64_t t) {
        const int s = prod.s;
        const uint32_t par = prod.parity;
        prod.next(S);
        const int64_t row = cid + t * ncl;
        if (bytes == 0) {
            mbar_arrive(&bar[s]);
            return;
        }
        mbar_arrive_expect_tx(&bar[s], static_cast<uint32_t>(NT) * bytes);
        if (row == a.drop_unit) return;  // failure injection: this wait runs out
        const int64_t off = row * N + static_cast<int64_t>(vbeg) * VEC;
        if (!RMSN_OK(span_in(X + off, bytes, X, tbytes) && span_in(DY + off, bytes, DY, tbytes) &&
                         smem_span_in(sx + s * unit, bytes) && smem_span_in(sdy + s * unit, bytes) &&
                         (!RES || (span_in(DRES + off, bytes, DRES, tbytes) &&
                                   smem_span_in(sdr + s * unit, bytes))),
                     a.status))
            return;  // checked build: the wait for this stage runs out instead
        bulk_copy_g2s(sx + s * unit, X + off, bytes, &bar[s]);
        bulk_copy_g2s(sdy + s * unit, DY + off, bytes, &bar[s]);
        if constexpr (RES) bulk_copy_g2s(sdr + s * unit, DRES + off, bytes, &bar[s]);
        pending |= 1u << s;
        pending_parity = (pending_parity & ~(1u << s)) | (par << s);
    };
    if (tid == 0)
        for (int64_t t = 0; t < S && t < nrows; ++t) issue(t);

    // The weights of the thread's slots stay in registers across rows when
    // they take at most 8 16-byte words and the thread holds at most 4
    // vectors of 16-bit elements; otherwise (an fp32 weight with 8 vectors a
    // thread, or 8 vectors of 16-bit elements, whose 64 dw accumulators
    // leave no room) they would spill, so they are re-read from cache at
    // each use.
    using WP = WPack<T, TW>;
    constexpr bool kWReg = WP::WORDS * V <= 8 && !(sizeof(T) == 2 && V > 4);
    uint4 wv[kWReg ? V : 1][WP::WORDS];
    if constexpr (kWReg) {
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = j * nthr + tid;
            if (k < vcnt) WP::load(W, vbeg + k, wv[j]);
            else WP::zero(wv[j]);
        }
    }
    auto weights = [&](int j, int k, float2 (&fw)[WP::PAIRS]) {
        if constexpr (kWReg) {
            WP::unpack2(wv[j], fw);
        } else {
            uint4 wq[WP::WORDS];
            WP::load(W, vbeg + k, wq);
            WP::unpack2(wq, fw);
        }
    };
    float2 acc[V][PR];
#pragma unroll
    for (int j = 0; j < V; ++j)
#pragma unroll
        for (int e = 0; e < PR; ++e) acc[j][e] = make_float2(0.f, 0.f);

    bool failed = false;   // a copy wait ran out in this block
    bool xfailed = false;  // an exchange wait ran out in this thread

    // pass 1 of row t: wait for its copy, partial dot, warp sums to red[t&1]
    RingPos pos1, pos2;  // ring positions of the rows of pass 1 and pass 2 (each in order)
    auto pass1 = [&](int64_t t) {
        const int s = pos1.s;
        const uint32_t parity = pos1.parity;
        pos1.next(S);
        if (!failed) {
            if (mbar_wait_bounded(&bar[s], parity, a.wait_limit_ns)) {
                if (tid == 0) pending &= ~(1u << s);
            } else {
                *fail = 1;
                report_status(a.status, kStatusTimeout);
            }
        }
        const unsigned char* xs = sx + s * unit;
        const unsigned char* ds = sdy + s * unit;
        float2 dot2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = j * nthr + tid;
            if (k >= vcnt) continue;
            float2 fx[PR], fd[PR], fw[PR];
            P::unpack2(ld_ring_16(xs + k * 16, a.status), fx);
            P::unpack2(ld_ring_16(ds + k * 16, a.status), fd);
            weights(j, k, fw);
#pragma unroll
            for (int e = 0; e < PR; ++e) dot2 = __ffma2_rn(__fmul2_rn(fd[e], fw[e]), fx[e], dot2);
        }
        const float dot = group_allreduce<32>(dot2.x + dot2.y);
        if (lane == 0) red[(t & 1) * 32 + warp] = dot;
    };
    // after the block barrier: the block's sum of row t, sent to the cluster
    auto reduce_send = [&](int64_t t) -> float {
        float tot = lane < nw ? red[(t & 1) * 32 + lane] : 0.f;
        tot = group_allreduce<32>(tot);
        if (csize > 1) {
            const int b = static_cast<int>(t & 3);
            // this block expects the C sums of row t as 4*C transaction bytes
            if (tid == 0) mbar_arrive_expect_tx(&xbar[b], 4u * csize);
            // thread q sends to block q (every thread holds the same sum)
            if (static_cast<uint32_t>(tid) < csize) {
                const uint32_t q = static_cast<uint32_t>(tid);
                st_async_cluster_f32(cluster_map(&xslot[b * kMaxClusterSize + crank], q), tot,
                                     cluster_map(&xbar[b], q));
            }
        }
        return tot;
    };
    // the row sum of row t: the block's own, or the C blocks' in rank order
    auto receive = [&](int64_t t, float own) -> float {
        if (csize == 1) return own;
        const int b = static_cast<int>(t & 3);
        if (!xfailed &&
            !mbar_wait_cluster_bounded(&xbar[b], static_cast<uint32_t>((t >> 2) & 1), a.wait_limit_ns)) {
            xfailed = true;  // later exchanges are not waited for again
            *fail = 1;
            report_status(a.status, kStatusTimeout);
        }
        float tot = 0.f;
        for (uint32_t q = 0; q < csize; ++q) tot += xslot[b * kMaxClusterSize + q];
        return tot;
    };
    // pass 2 of row t: dx = r*(g - xhat*c), dw += dy*xhat
    auto pass2 = [&](int64_t t, float r, float tot) {
        const int s = pos2.s;
        pos2.next(S);
        const unsigned char* xs = sx + s * unit;
        const unsigned char* ds = sdy + s * unit;
        const float c = r * (tot * inv_n);
        const float2 r2 = f2_splat(r), nc2 = f2_splat(-c);
        T* dxr = DX + (cid + t * ncl) * N;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k = j * nthr + tid;
            if (k >= vcnt) continue;
            float2 fx[PR], fd[PR], fw[PR], o[PR], fr[PR];
            if constexpr (RES) P::unpack2(ld_ring_16(sdr + s * unit + k * 16, a.status), fr);
            P::unpack2(ld_ring_16(xs + k * 16, a.status), fx);
            P::unpack2(ld_ring_16(ds + k * 16, a.status), fd);
            weights(j, k, fw);
#pragma unroll
            for (int e = 0; e < PR; ++e) {
                const float2 xh = __fmul2_rn(fx[e], r2);
                const float2 gg = __fmul2_rn(fd[e], fw[e]);
                if constexpr (RES)
                    o[e] = __ffma2_rn(r2, __ffma2_rn(xh, nc2, gg), fr[e]);
                else
                    o[e] = __fmul2_rn(r2, __ffma2_rn(xh, nc2, gg));
                acc[j][e] = __ffma2_rn(fd[e], xh, acc[j][e]);
            }
            T* dst = dxr + static_cast<int64_t>(vbeg + k) * VEC;
            if (RMSN_OK(span_in(dst, 16, DX, tbytes), a.status)) st_global_16(dst, P::pack2(o));
        }
    };

    float r_cur = nrows > 0 ? __ldg(a.rstd + cid) : 0.f;
    float r_next = nrows > 1 ? __ldg(a.rstd + cid + ncl) : 0.f;
    if (PIPE) {
        // pass 1 of row t+1 runs before pass 2 of row t; the ring keeps two
        // rows resident, so S-2 rows are in flight
        float tot_cur = 0.f;
        if (nrows > 0) {
            pass1(0);
            __syncthreads();
            failed = *fail != 0;
            tot_cur = reduce_send(0);
        }
        for (int64_t t = 0; t < nrows; ++t) {
            const float r_after = t + 2 < nrows ? __ldg(a.rstd + cid + (t + 2) * ncl) : 0.f;
            if (t + 1 < nrows) pass1(t + 1);
            __syncthreads();  // sums of row t+1 published; every thread is done with row t-1
            failed = *fail != 0;
            const float tot_next = t + 1 < nrows ? reduce_send(t + 1) : 0.f;
            // the stage of row t-1 is free now: refill it with row t-1+S
            if (tid == 0 && !failed && t >= 1 && t - 1 + S < nrows) {
                fence_proxy_async_shared();
                issue(t - 1 + S);
            }
            pass2(t, r_cur, receive(t, tot_cur));
            tot_cur = tot_next;
            r_cur = r_next;
            r_next = r_after;
        }
    } else {
        // one row at a time: S-1 rows in flight, the exchange waited for in place
        const bool early = a.early_refill != 0;
        for (int64_t t = 0; t < nrows; ++t) {
            const float r_after = t + 2 < nrows ? __ldg(a.rstd + cid + (t + 2) * ncl) : 0.f;
            pass1(t);
            __syncthreads();  // sums of row t published; every thread is done with row t-1
            failed = *fail != 0;
            const float own = reduce_send(t);
            if (!early && tid == 0 && !failed && t >= 1 && t - 1 + S < nrows) {
                fence_proxy_async_shared();
                issue(t - 1 + S);
            }
            pass2(t, r_cur, receive(t, own));
            if (early) {
                // refill row t's stage as soon as every thread is done with it
                __syncthreads();
                if (tid == 0 && !failed && t + S < nrows) {
                    fence_proxy_async_shared();
                    issue(t + S);
                }
            }
            r_cur = r_next;
            r_next = r_after;
        }
    }
    allow_dependent_launch();

    if (tid == 0 && failed)
        for (int s = 0; s < S; ++s)
            if ((pending >> s) & 1u)
                mbar_wait_bounded(&bar[s], (pending_parity >> s) & 1u, a.wait_limit_ns);

    // one partial row per cluster; each block writes its column slice
    float* prow = a.partial + cid * N + static_cast<int64_t>(vbeg) * VEC;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int k = j * nthr + tid;
        if (k >= vcnt) continue;
#pragma unroll
        for (int q = 0; q < PR / 2; ++q)
            if (float* pd = prow + static_cast<int64_t>(k) * VEC + 4 * q;
                    RMSN_OK(span_in(pd, 16, a.partial, pbytes), a.status))
                *reinterpret_cast<float4*>(pd) =
                make_float4(acc[j][2 * q].x, acc[j][2 * q].y, acc[j][2 * q + 1].x, acc[j][2 * q + 1].y);
    }
    // no block may leave while a peer can still reach its shared memory
    if (csize > 1) cluster_sync_all();
}

// ---------------------------------------------------------- short rows
// A unit is a tile of RT = (threads/G)*R consecutive rows, moved by one bulk
// copy per tensor. Group g (G lanes) handles tile rows r*groups + g.
template <typename T, typename TW, int G, int V, int R, bool RES>
__global__ void __launch_bounds__(256) bwd_rowgroup_kernel(BwdArgs a, int stages, int /*groups*/) {
    using P = Pack<T>;
    constexpr int VEC = P::VEC;
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x;
    const int lane = tid % G, group = tid / G, groups = blockDim.x / G;
    const int RT = groups * R;
    const int N = a.N;
    const float inv_n = 1.f / static_cast<float>(N);  // mean = sum * inv_n, one multiply a row
    const int nvec = N / VEC;
    const int64_t ntiles = (a.M + RT - 1) / RT;
    const int64_t b = blockIdx.x, nb = gridDim.x;
    const int64_t count = b < ntiles ? (ntiles - 1 - b) / nb + 1 : 0;
    const int S = stages;
    const int unit = RT * N * static_cast<int>(sizeof(T));

    constexpr int NT = RES ? 3 : 2;  // tensors in the ring
    unsigned char* sx = smem;
    unsigned char* sdy = smem + S * unit;
    unsigned char* sdr = smem + 2 * S * unit;  // dres (RES only)
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + NT * S * unit);
    volatile int* fail = reinterpret_cast<volatile int*>(reinterpret_cast<float*>(bar + S) + 66);

    const T* X = static_cast<const T*>(a.x);
    const T* DY = static_cast<const T*>(a.dy);
    const TW* W = static_cast<const TW*>(a.w);
    T* DX = static_cast<T*>(a.dx);
    const T* DRES = static_cast<const T*>(a.dres);
    // extents for the checked build: x, dy, dx, dres; the partial rows
    [[maybe_unused]] const int64_t tbytes =
        a.M * static_cast<int64_t>(N) * static_cast<int64_t>(sizeof(T));
    [[maybe_unused]] const int64_t pbytes = nb * static_cast<int64_t>(N) * 4;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
        *fail = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    wait_for_prerequisite_grid();  // no global access before this

    uint32_t pending = 0, pending_parity = 0;
    RingPos prod;  // ring position of the next tile to issue (issued in order)
    auto issue = [&](int64_t t) {
        const int s = prod.s;
        const uint32_t par = prod.parity;
        prod.next(S);
        const int64_t tile = b + t * nb;
        const int64_t rows = min(static_cast<int64_t>(RT), a.M - tile * RT);
        const uint32_t bytes = static_cast<uint32_t>(rows * N * static_cast<int64_t>(sizeof(T)));
        mbar_arrive_expect_tx(&bar[s], static_cast<uint32_t>(NT) * bytes);
        if (tile == a.drop_unit) return;  // failure injection
        const int64_t off = tile * RT * N;
        if (!RMSN_OK(span_in(X + off, bytes, X, tbytes) && span_in(DY + off, bytes, DY, tbytes) &&
                         smem_span_in(sx + s * unit, bytes) && smem_span_in(sdy + s * unit, bytes) &&
                         (!RES || (span_in(DRES + off, bytes, DRES, tbytes) &&
                                   smem_span_in(sdr + s * unit, bytes))),
                     a.status))
            return;  // checked build: the wait for this tile runs out instead
        bulk_copy_g2s(sx + s * unit, X + off, bytes, &bar[s]);
        bulk_copy_g2s(sdy + s * unit, DY + off, bytes, &bar[s]);
        if constexpr (RES) bulk_copy_g2s(sdr + s * unit, DRES + off, bytes, &bar[s]);
        pending |= 1u << s;
        pending_parity = (pending_parity & ~(1u << s)) | (par << s);
    };
    if (tid == 0)
        for (int64_t t = 0; t < S && t < count; ++t) issue(t);

    using WP = WPack<T, TW>;
    uint4 wv[V][WP::WORDS];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int k = j * G + lane;
        if (k < nvec) WP::load(W, k, wv[j]);
        else WP::zero(wv[j]);
    }
    constexpr int PR = P::PAIRS;
    float2 acc[V][PR];
#pragma unroll
    for (int j = 0; j < V; ++j)
#pragma unroll
        for (int e = 0; e < PR; ++e) acc[j][e] = make_float2(0.f, 0.f);

    float rnext[R];
    auto load_rstd = [&](int64_t t, float (&dst)[R]) {
        const int64_t tile = b + t * nb;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = tile * RT + r * groups + group;
            dst[r] = (t < count && row < a.M) ? __ldg(a.rstd + row) : 0.f;
        }
    };
    load_rstd(0, rnext);
    bool failed = false;

    RingPos cons;  // ring position of tile t
    for (int64_t t = 0; t < count; ++t) {
        const int64_t tile = b + t * nb;
        const int s = cons.s;
        const uint32_t parity = cons.parity;
        cons.next(S);
        float rcur[R];
#pragma unroll
        for (int r = 0; r < R; ++r) rcur[r] = rnext[r];
        load_rstd(t + 1, rnext);

        if (!failed) {
            if (mbar_wait_bounded(&bar[s], parity, a.wait_limit_ns)) {
                if (tid == 0) pending &= ~(1u << s);
            } else {
                *fail = 1;
                report_status(a.status, kStatusTimeout);
            }
        }
        // pass 1: per-row dot = sum_j (dy*w)*x over this lane's slots
        float dot[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int lr = r * groups + group;
            const bool row_ok = tile * RT + lr < a.M;
            float2 dot2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int k = j * G + lane;
                if (!row_ok || k >= nvec) continue;
                const int off = (lr * N + k * VEC) * static_cast<int>(sizeof(T));
                float2 fx[PR], fd[PR], fw[PR];
                P::unpack2(ld_ring_16(sx + s * unit + off, a.status), fx);
                P::unpack2(ld_ring_16(sdy + s * unit + off, a.status), fd);
                WP::unpack2(wv[j], fw);
#pragma unroll
                for (int e = 0; e < PR; ++e) dot2 = __ffma2_rn(__fmul2_rn(fd[e], fw[e]), fx[e], dot2);
            }
            dot[r] = dot2.x + dot2.y;
        }
        __syncthreads();  // every thread is done with tile t-1
        failed = *fail != 0;
        if (tid == 0 && !failed && t >= 1 && t - 1 + S < count) {
            fence_proxy_async_shared();
            issue(t - 1 + S);
        }
#pragma unroll
        for (int off = G / 2; off >= 1; off /= 2)
#pragma unroll
            for (int r = 0; r < R; ++r) dot[r] += __shfl_xor_sync(0xffffffffu, dot[r], off);

        // pass 2: dx and the dw contribution, re-reading the tile from shared memory
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int lr = r * groups + group;
            const int64_t row = tile * RT + lr;
            if (row >= a.M) continue;
            const float rs = rcur[r];
            const float c = rs * (dot[r] * inv_n);
            const float2 r2 = f2_splat(rs), nc2 = f2_splat(-c);
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int k = j * G + lane;
                if (k >= nvec) continue;
                const int off = (lr * N + k * VEC) * static_cast<int>(sizeof(T));
                float2 fx[PR], fd[PR], fw[PR], o[PR], fr[PR];
                if constexpr (RES) P::unpack2(ld_ring_16(sdr + s * unit + off, a.status), fr);
                P::unpack2(ld_ring_16(sx + s * unit + off, a.status), fx);
                P::unpack2(ld_ring_16(sdy + s * unit + off, a.status), fd);
                WP::unpack2(wv[j], fw);
#pragma unroll
                for (int e = 0; e < PR; ++e) {
                    const float2 xh = __fmul2_rn(fx[e], r2);
                    const float2 g = __fmul2_rn(fd[e], fw[e]);
                    if constexpr (RES)
                        o[e] = __ffma2_rn(r2, __ffma2_rn(xh, nc2, g), fr[e]);
                    else
                        o[e] = __fmul2_rn(r2, __ffma2_rn(xh, nc2, g));
                    acc[j][e] = __ffma2_rn(fd[e], xh, acc[j][e]);
                }
                T* dst = DX + row * N + static_cast<int64_t>(k) * VEC;
                if (RMSN_OK(span_in(dst, 16, DX, tbytes), a.status)) st_global_16(dst, P::pack2(o));
            }
        }
    }

    allow_dependent_launch();
    if (tid == 0 && failed)
        for (int s = 0; s < S; ++s)
            if ((pending >> s) & 1u) mbar_wait_bounded(&bar[s], (pending_parity >> s) & 1u, a.wait_limit_ns);
    __syncthreads();  // all lanes done with the last tile; the ring is idle
    // combine the groups' dw in group order through shared memory
    // (groups*N*4 bytes always fit in the 2*S*unit bytes of the ring)
    float* comb = reinterpret_cast<float*>(smem);
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int k = j * G + lane;
        if (k >= nvec) continue;
#pragma unroll
        for (int q = 0; q < PR / 2; ++q)
            if (float* cd = comb + group * N + k * VEC + 4 * q;
                    RMSN_OK(smem_span_in(cd, 16), a.status))
                *reinterpret_cast<float4*>(cd) =
                make_float4(acc[j][2 * q].x, acc[j][2 * q].y, acc[j][2 * q + 1].x,
                            acc[j][2 * q + 1].y);
    }
    __syncthreads();
    if (a.cluster_dw) {
        // the grid is one cluster: the groups' dw meet in shared memory (group
        // order), then the blocks' rows in dw (rank order)
        for (int col = tid; col < N; col += blockDim.x) {
            float sum = 0.f;
            for (int gi = 0; gi < groups; ++gi)
                sum += RMSN_OK(smem_span_in(comb + gi * N + col, 4), a.status)
                           ? comb[gi * N + col] : 0.f;
            comb[col] = sum;  // group 0's value of this column was read above
        }
        cluster_rows_to_dw(comb, N, a.dw, a.status);
        return;
    }
    float* prow = a.partial + b * N;
    for (int col = tid; col < N; col += blockDim.x) {
        float sum = 0.f;
        for (int gi = 0; gi < groups; ++gi)
            sum += RMSN_OK(smem_span_in(comb + gi * N + col, 4), a.status) ? comb[gi * N + col]
                                                                           : 0.f;
        if (RMSN_OK(span_in(prow + col, 4, a.partial, pbytes), a.status)) prow[col] = sum;
    }
}

// ------------------------------------------------------------------ scalar
// Any alignment, any N. Persistent: block b owns rows b, b+P, ... and its
// partial row, which thread t updates at columns t, t+blockDim, ... only.
template <typename T, typename TW, bool RES>
__global__ void __launch_bounds__(256) bwd_scalar_kernel(BwdArgs a, int /*stages*/, int /*groups*/) {
    using P = Pack<T>;
    __shared__ float red[2][32];
    const int N = a.N;
    const float inv_n = 1.f / static_cast<float>(N);  // mean = sum * inv_n, one multiply a row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const T* X = static_cast<const T*>(a.x);
    const T* DY = static_cast<const T*>(a.dy);
    const TW* W = static_cast<const TW*>(a.w);
    T* DX = static_cast<T*>(a.dx);
    const T* DRES = static_cast<const T*>(a.dres);
    // extents for the checked build: x, dy, dx, dres; the partial rows
    [[maybe_unused]] const int64_t tbytes =
        a.M * static_cast<int64_t>(N) * static_cast<int64_t>(sizeof(T));
    [[maybe_unused]] const int64_t pbytes =
        static_cast<int64_t>(gridDim.x) * static_cast<int64_t>(N) * 4;
    float* prow = a.partial + static_cast<int64_t>(blockIdx.x) * N;
    wait_for_prerequisite_grid();  // no global access before this
    for (int col = threadIdx.x; col < N; col += blockDim.x)
        if (RMSN_OK(span_in(prow + col, 4, a.partial, pbytes), a.status)) prow[col] = 0.f;
    int it = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x, ++it) {
        const T* xr = X + row * N;
        const T* dyr = DY + row * N;
        const float r = a.rstd[row];
        float dot = 0.f;
        for (int col = threadIdx.x; col < N; col += blockDim.x)
            dot = fmaf(to_f32(dyr[col]) * to_f32(W[col]), to_f32(xr[col]), dot);
        dot = group_allreduce<32>(dot);
        if (lane == 0) red[it & 1][warp] = dot;
        __syncthreads();
        float tot = lane < nw ? red[it & 1][lane] : 0.f;
        tot = group_allreduce<32>(tot);
        const float c = r * (tot * inv_n);
        T* dxr = DX + row * N;
        for (int col = threadIdx.x; col < N; col += blockDim.x) {
            const float d = to_f32(dyr[col]);
            const float xh = to_f32(xr[col]) * r;
            const float g = d * to_f32(W[col]);
            if (RMSN_OK(span_in(dxr + col, sizeof(T), DX, tbytes), a.status)) {
                if constexpr (RES)
                    dxr[col] = P::from_float(fmaf(r, g - xh * c, to_f32(DRES[row * N + col])));
                else
                    dxr[col] = P::from_float(r * (g - xh * c));
            }
            if (RMSN_OK(span_in(prow + col, 4, a.partial, pbytes), a.status))
                prow[col] = fmaf(d, xh, prow[col]);
        }
    }
}

// ------------------------------------------------------ kernel selection
template <typename T, typename TW, bool RES>
const void* row_kernel(int V) {
    switch (V) {
        case 1: return reinterpret_cast<const void*>(&bwd_row_kernel<T, TW, 1, RES>);
        case 2: return reinterpret_cast<const void*>(&bwd_row_kernel<T, TW, 2, RES>);
        case 4: return reinterpret_cast<const void*>(&bwd_row_kernel<T, TW, 4, RES>);
        case 8: return reinterpret_cast<const void*>(&bwd_row_kernel<T, TW, 8, RES>);
        default: return nullptr;
    }
}

template <typename T, typename TW, bool RES>
const void* wide_kernel(int V, bool pipelined) {
    if (V == 4) return pipelined ? reinterpret_cast<const void*>(&bwd_wide_kernel<T, TW, 4, true, RES>)
                                 : reinterpret_cast<const void*>(&bwd_wide_kernel<T, TW, 4, false, RES>);
    if (V == 8) return pipelined ? reinterpret_cast<const void*>(&bwd_wide_kernel<T, TW, 8, true, RES>)
                                 : reinterpret_cast<const void*>(&bwd_wide_kernel<T, TW, 8, false, RES>);
    return nullptr;
}

template <typename T, typename TW, bool RES>
const void* rowgroup_kernel(int G, int V) {
    if (G == 4 && V == 1) return reinterpret_cast<const void*>(&bwd_rowgroup_kernel<T, TW, 4, 1, 4, RES>);
    if (G == 4 && V == 2) return reinterpret_cast<const void*>(&bwd_rowgroup_kernel<T, TW, 4, 2, 2, RES>);
    if (G == 8 && V == 2) return reinterpret_cast<const void*>(&bwd_rowgroup_kernel<T, TW, 8, 2, 2, RES>);
    if (G == 8 && V == 4) return reinterpret_cast<const void*>(&bwd_rowgroup_kernel<T, TW, 8, 4, 1, RES>);
    if (G == 16 && V == 4) return reinterpret_cast<const void*>(&bwd_rowgroup_kernel<T, TW, 16, 4, 1, RES>);
    if (G == 32 && V == 4) return reinterpret_cast<const void*>(&bwd_rowgroup_kernel<T, TW, 32, 4, 1, RES>);
    if (G == 32 && V == 8) return reinterpret_cast<const void*>(&bwd_rowgroup_kernel<T, TW, 32, 8, 1, RES>);
    return nullptr;
}

template <typename T, typename TW, bool RES>
const void* main_kernel(const rmsnorm_plan_t& p, bool pipelined) {
    switch (p.variant) {
        case RMSNORM_VARIANT_ROWGROUP: return rowgroup_kernel<T, TW, RES>(p.threads_per_row, p.vectors_per_thread);
        case RMSNORM_VARIANT_CTA_ROW:  // a row per group of a block (in a cluster for few rows)
            return row_kernel<T, TW, RES>(p.vectors_per_thread);
        case RMSNORM_VARIANT_CLUSTER_ROW:  // a row split over a cluster
            return p.cluster == 1 ? row_kernel<T, TW, RES>(p.vectors_per_thread)
                                  : wide_kernel<T, TW, RES>(p.vectors_per_thread, pipelined);
        case RMSNORM_VARIANT_SCALAR: return reinterpret_cast<const void*>(&bwd_scalar_kernel<T, TW, RES>);
        default: return nullptr;
    }
}

}  // namespace
}  // namespace rmsn
