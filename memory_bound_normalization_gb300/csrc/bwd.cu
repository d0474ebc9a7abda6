// RMSNorm backward, host side: the plan (kernel family, block shape, ring
// depth, persistent grid size), the fixed-order column sum that turns the
// per-block dw partial rows into dw, and the two launches. The row kernels
// and their design are in bwd_kernels.cuh.
#include <algorithm>
#include <cstdlib>
#include <map>
#include <mutex>
#include <set>
#include <utility>
#include <tuple>

#include "bwd_kernels.cuh"

namespace rmsn {

static_assert(kStatusTimeout == RMSNORM_ERR_DEVICE_TIMEOUT, "device status codes follow the C ABI");
static_assert(kStatusOutOfBounds == RMSNORM_ERR_OUT_OF_BOUNDS,
              "device status codes follow the C ABI");

namespace {

constexpr int kStageBudget = 48 * 1024;   // ring bytes aimed at per short-row block
constexpr int kSliceBudget = 64 * 1024;   // x+dy bytes of one row slice per stage
constexpr int kSmemMax = 227 * 1024;      // dynamic shared memory a block may opt into
constexpr int kMaxRowGroups = 8;          // named barriers 1..8 (0 is __syncthreads)
constexpr int kClusterDwMax = 16;         // blocks of the one cluster that sums dw on chip
constexpr int kClusterWideMax = 16;       // blocks of a cluster for rows 8 blocks cannot hold

// Tuning overrides for sweeps (read once; unset = built-in ladder). They
// change the persistent grid, hence the order of the dw sum: results stay
// deterministic for a fixed setting.
struct BwdTuning {
    int vectors = 4;        // 16-byte vectors per thread in a row group
    int groups = 0;         // row groups per block (0 = as many as 512 threads hold)
    int stages = 0;         // ring depth (0 = from the shared-memory budget)
    int smem_multi = 200 * 1024;   // shared memory aimed at, several groups
    int smem_single = 100 * 1024;  // shared memory aimed at, one group
    int slice = kSliceBudget;      // x+dy bytes of a block's row slice per stage
    bool pipelined = false;        // cluster rows: pass 1 of the next row first
    int cluster = 0;               // blocks a wide row is split over (0 = from the ladder)
    int wide_select = 2;           // cluster rows shaped on the device: 0 never, 1 without
                                   // dres, 2 always
    int rowgroup_max_vec = -1;     // widest row (16-byte vectors) for the short-row kernel
                                   // (-1 = by type: 256 for fp32 rows, 128 for 16-bit rows)
    int early_refill = -1;         // refill a ring stage after pass 2 of its row (1) or
                                   // after pass 1 of the next row (0); -1 = by plan
    int cluster_dw_units = 16;     // rows (or tiles, or row-group units) up to which one
                                   // cluster sums dw on chip (0 = never)
    int pdl_wide = -1;             // programmatic launch of rows split over a cluster:
                                   // 1 always, 0 never, -1 by plan
};

int env_int(const char* name, int dflt) {
    const char* v = getenv(name);
    if (v == nullptr || *v == 0) return dflt;
    return atoi(v);
}

const BwdTuning& tuning() {
    static const BwdTuning t = [] {
        BwdTuning u;
        u.vectors = env_int("RMSNORM_BWD_VECTORS", u.vectors);
        if (u.vectors != 1 && u.vectors != 2 && u.vectors != 4 && u.vectors != 8) u.vectors = 4;
        u.groups = std::max(0, std::min(kMaxRowGroups, env_int("RMSNORM_BWD_GROUPS", 0)));
        u.stages = std::max(0, std::min(8, env_int("RMSNORM_BWD_STAGES", 0)));
        u.smem_multi = std::max(32 * 1024, std::min(kSmemMax, env_int("RMSNORM_BWD_SMEM", u.smem_multi)));
        u.slice = std::max(8 * 1024, std::min(kSmemMax, env_int("RMSNORM_BWD_SLICE", u.slice)));
        u.pipelined = env_int("RMSNORM_BWD_PIPE", 0) != 0;
        u.cluster = std::max(0, std::min(kMaxCluster, env_int("RMSNORM_BWD_CLUSTER", 0)));
        u.wide_select = std::max(0, std::min(2, env_int("RMSNORM_WIDE_SELECT", 2)));
        u.rowgroup_max_vec = std::max(-1, std::min(256, env_int("RMSNORM_BWD_ROWGROUP_MAX_VEC", -1)));
        u.early_refill = std::max(-1, std::min(1, env_int("RMSNORM_BWD_EARLY_REFILL", -1)));
        u.cluster_dw_units = std::max(0, env_int("RMSNORM_BWD_CLUSTER_DW_UNITS", u.cluster_dw_units));
        u.pdl_wide = std::max(-1, std::min(1, env_int("RMSNORM_BWD_PDL_WIDE", u.pdl_wide)));
        return u;
    }();
    return t;
}

// ---------------------------------------------------------- column sum
// dw[j] = sum over p of partial[p][j] in a fixed tree: thread row q of the
// block (Q rows of 32 threads, 32 columns) sums p = q, q+Q, q+2Q, ... in
// ascending order; then warp c adds the Q sums of column c (and of c+Q,
// c+2Q, ... when Q < 32) by a fixed xor-butterfly of shuffles. Same bits on
// every run for a given P and Q. (Adding the Q sums one after another in a
// single thread made a chain of 32 dependent shared-memory reads and adds
// at the end of every backward call.)
template <int Q>
__global__ void __launch_bounds__(32 * Q) colsum_kernel(const float* __restrict__ partial,
                                                        float* __restrict__ dw, int P, int N,
                                                        int* status) {
    __shared__ float part[Q][33];
    wait_for_prerequisite_grid();  // partial rows complete and visible
    allow_dependent_launch();
    const int cx = threadIdx.x, q = threadIdx.y;
    const int64_t col0 = static_cast<int64_t>(blockIdx.x) * 32;
    const int64_t col = col0 + cx;
    [[maybe_unused]] const int64_t pbytes = static_cast<int64_t>(P) * N * 4;
    float s = 0.f;
    if (col < N) {
#pragma unroll 4
        for (int p = q; p < P; p += Q) {
            const float* src = partial + static_cast<int64_t>(p) * N + col;
            if (RMSN_OK(span_in(src, 4, partial, pbytes), status)) s += *src;
        }
    }
    part[q][cx] = s;
    __syncthreads();
    for (int c = q; c < 32; c += Q) {
        // lane l holds thread row l's sum of column c (zero past Q rows)
        float v = cx < Q ? part[cx][c] : 0.f;
        v = group_allreduce<32>(v);
        if (cx == 0 && col0 + c < N &&
            RMSN_OK(span_in(dw + col0 + c, 4, dw, static_cast<int64_t>(N) * 4), status))
            dw[col0 + c] = v;
    }
}

// Narrow rows (N < 2048): C columns by R = 1024/C thread rows a block, C
// chosen so that at least 64 blocks share the sum. Thread row q adds
// p = q, q+R, q+2R, ... in ascending order, then the R sums of a column are
// added by a fixed pairwise tree (halving strides), the same bits on every
// run for a given P, N and C. With 32 columns a block, QK-norm's 608 partial
// rows of 128 columns went to 4 blocks whose threads read 19 values each, one
// after another.
template <int C>
__global__ void __launch_bounds__(1024) colsum_narrow_kernel(const float* __restrict__ partial,
                                                             float* __restrict__ dw, int P,
                                                             int N, int* status) {
    constexpr int R = 1024 / C;
    __shared__ float part[R][C + 1];
    wait_for_prerequisite_grid();  // partial rows complete and visible
    allow_dependent_launch();
    const int cx = threadIdx.x, q = threadIdx.y;
    const int64_t col = static_cast<int64_t>(blockIdx.x) * C + cx;
    float s = 0.f;
    if (col < N) {
#pragma unroll 2
        for (int p = q; p < P; p += R) {
            const float* src = partial + static_cast<int64_t>(p) * N + col;
            if (RMSN_OK(span_in(src, 4, partial, static_cast<int64_t>(P) * N * 4), status)) s += *src;
        }
    }
    part[q][cx] = s;
    __syncthreads();
#pragma unroll
    for (int h = R / 2; h > 0; h >>= 1) {
        if (q < h) part[q][cx] += part[q + h][cx];
        __syncthreads();
    }
    if (q == 0 && col < N && RMSN_OK(span_in(dw + col, 4, dw, static_cast<int64_t>(N) * 4), status))
        dw[col] = part[0][cx];
}

// Columns a block of the narrow column sum takes: at least 64 blocks.
int colsum_narrow_cols(int N) {
    int c = 16;
    while (c > 1 && N < 64 * c) c >>= 1;
    return c;
}

const void* colsum_narrow_for(int c) {
    switch (c) {
        case 16: return reinterpret_cast<const void*>(&colsum_narrow_kernel<16>);
        case 8: return reinterpret_cast<const void*>(&colsum_narrow_kernel<8>);
        case 4: return reinterpret_cast<const void*>(&colsum_narrow_kernel<4>);
        case 2: return reinterpret_cast<const void*>(&colsum_narrow_kernel<2>);
        default: return reinterpret_cast<const void*>(&colsum_narrow_kernel<1>);
    }
}

// The column-sum kernel with q thread rows (a power of two up to 32).
const void* colsum_kernel_for(int q) {
    switch (q) {
        case 1: return reinterpret_cast<const void*>(&colsum_kernel<1>);
        case 2: return reinterpret_cast<const void*>(&colsum_kernel<2>);
        case 4: return reinterpret_cast<const void*>(&colsum_kernel<4>);
        case 8: return reinterpret_cast<const void*>(&colsum_kernel<8>);
        case 16: return reinterpret_cast<const void*>(&colsum_kernel<16>);
        default: return reinterpret_cast<const void*>(&colsum_kernel<32>);
    }
}

// Rows narrower than this take the narrow column sum.
constexpr int kColsumNarrowBelow = 2048;

// Thread rows of the column sum: 32 while one wave of blocks (32 columns
// each) covers every column, halved for wider rows until it does. With 32
// rows at N = 65536 the sum ran as about seven waves of blocks that each
// read one or two values a thread.
int colsum_phases(int N, int sm_count) {
    const int64_t resident = static_cast<int64_t>(std::max(1, sm_count)) * 2048;
    int q = 32;
    while (q > 1 && static_cast<int64_t>(N) * q > resident) q >>= 1;
    return q;
}
// ------------------------------------------------------------ host side
const void* main_kernel_for(int dtype, const rmsnorm_plan_t& p, bool res) {
    const bool pipe = tuning().pipelined;
    if (res) {
        switch (dtype) {
            case RMSNORM_F32: return bwd_res_kernel_f32(p, pipe);
            case RMSNORM_BF16: return bwd_res_kernel_bf16(p, pipe);
            case RMSNORM_F16: return bwd_res_kernel_f16(p, pipe);
            case RMSNORM_BF16_W_F32: return bwd_res_kernel_bf16_w_f32(p, pipe);
            case RMSNORM_F16_W_F32: return bwd_res_kernel_f16_w_f32(p, pipe);
            default: return nullptr;
        }
    }
    switch (dtype) {
        case RMSNORM_F32: return bwd_main_kernel_f32(p, pipe);
        case RMSNORM_BF16: return bwd_main_kernel_bf16(p, pipe);
        case RMSNORM_F16: return bwd_main_kernel_f16(p, pipe);
        case RMSNORM_BF16_W_F32: return bwd_main_kernel_bf16_w_f32(p, pipe);
        case RMSNORM_F16_W_F32: return bwd_main_kernel_f16_w_f32(p, pipe);
        default: return nullptr;
    }
}

// Resident blocks (or clusters) per GPU for one kernel configuration, cached
// so that every call on a device sees the same persistent grid.
struct OccKey {
    int device;
    const void* fn;
    int threads, smem, cluster;
    bool operator<(const OccKey& o) const {
        return std::tie(device, fn, threads, smem, cluster) <
               std::tie(o.device, o.fn, o.threads, o.smem, o.cluster);
    }
};
std::mutex g_occ_mu;
std::map<OccKey, int> g_occ;
std::set<std::pair<int, const void*>> g_optin;

cudaError_t resident_units(const DeviceInfo& dev, const void* fn, int threads, int smem,
                           int cluster, int* out) {
    const OccKey key{dev.device, fn, threads, smem, cluster};
    {
        std::lock_guard<std::mutex> lk(g_occ_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) {
            *out = it->second;
            return cudaSuccess;
        }
    }
    // Opt the kernel into the device's largest dynamic shared memory once,
    // so plans of different sizes for the same kernel never lower the limit.
    cudaError_t err = cudaSuccess;
    {
        std::lock_guard<std::mutex> lk(g_occ_mu);
        if (g_optin.insert(std::make_pair(dev.device, fn)).second) {
            // the opt-in covers dynamic memory only: leave room for static
            cudaFuncAttributes fa;
            err = cudaFuncGetAttributes(&fa, fn);
            if (err == cudaSuccess)
                err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           dev.max_smem_optin - static_cast<int>(fa.sharedSizeBytes));
            if (err != cudaSuccess) {
                g_optin.erase(std::make_pair(dev.device, fn));
                return err;
            }
        }
    }
    int units = 0;
    if (cluster <= 1) {
        int per_sm = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
        if (err != cudaSuccess) return err;
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
        if (err != cudaSuccess) return err;
    }
    if (units < 1) return cudaErrorInvalidConfiguration;
    std::lock_guard<std::mutex> lk(g_occ_mu);
    g_occ[key] = units;
    *out = units;
    return cudaSuccess;
}



// A cluster-row plan for rows of nvec 16-byte vectors split over c blocks:
// 4 vectors a thread, else up to max_v, so that a block has at most 512
// threads; a ring of `stages` stages (0: as many as `budget` bytes of shared
// memory hold, at most 6), lowered to st_min while it does not fit. False
// when the block or its ring cannot fit.
bool wide_plan(int64_t nvec, int nt, int c, int max_v, int st_min, int stages, int budget,
               rmsnorm_plan_t* p) {
    const int64_t slots = cdiv(nvec, c);
    int v = 4;
    while (cdiv(slots, v) > 512 && v < max_v) v *= 2;
    const int t = std::max(32, round_up(static_cast<int>(cdiv(slots, v)), 32));
    const int unit = v * t * 16;
    if (stages <= 0) stages = std::max(st_min, std::min(6, budget / (nt * unit)));
    while (stages > st_min && bwd_wide_smem_bytes(stages, unit, nt) > kSmemMax) --stages;
    if (t > 512 || bwd_wide_smem_bytes(stages, unit, nt) > kSmemMax) return false;
    p->variant = c > 1 ? RMSNORM_VARIANT_CLUSTER_ROW : RMSNORM_VARIANT_CTA_ROW;
    p->cluster = c;
    p->row_groups = 1;
    p->vectors_per_thread = v;
    p->threads = t;
    p->threads_per_row = t * c;
    p->rows_per_unit = 1;
    p->stages = stages;
    p->smem_bytes = bwd_wide_smem_bytes(stages, unit, nt);
    return true;
}

}  // namespace

// Any alignment, any N: one block per row, scalar loads.
static void scalar_plan(rmsnorm_plan_t* p) {
    p->variant = RMSNORM_VARIANT_SCALAR;
    p->cluster = 1;
    p->row_groups = 1;
    p->rows_per_unit = 1;
    p->threads = 256;
    p->threads_per_row = 256;
    p->vectors_per_thread = 0;
    p->stages = 0;
    p->smem_bytes = 0;
}

// With res (the residual backward) the rings carry dres as a third tensor:
// stages may drop to two before a row group or a ring is given up, and wide
// rows may take a larger cluster. Plans without res are unchanged by it.
void bwd_choose(int64_t N, int dtype, bool vector_ok, rmsnorm_plan_t* p, bool res) {
    *p = rmsnorm_plan_t{};
    p->cluster = 1;
    p->row_groups = 1;
    p->rows_per_unit = 1;
    const int sz = dtype_size(dtype);
    const int64_t nvec = N / dtype_vec(dtype);
    const BwdTuning& tu = tuning();
    const int nt = res ? 3 : 2;          // tensors in a ring stage
    const int min_stages = res ? 2 : 3;
    // 16-bit rows of 129..256 vectors ran 7..15 points of the copy roofline
    // faster as one row per 64-thread group (8 groups a block) than as one
    // row per 32-thread group; fp32 rows of 256 vectors ran 1 point slower
    const int rowgroup_max_vec = tu.rowgroup_max_vec >= 0 ? tu.rowgroup_max_vec
                                                          : (sz == 4 ? 256 : 128);
    GroupShape g;
    if (vector_ok && nvec <= rowgroup_max_vec && bwd_group_shape(nvec, &g)) {
        p->variant = RMSNORM_VARIANT_ROWGROUP;
        p->threads = g.threads;
        p->threads_per_row = g.G;
        p->vectors_per_thread = g.V;
        p->rows_per_unit = (g.threads / g.G) * g.R;
        const int unit = static_cast<int>(p->rows_per_unit * N * sz);
        p->stages = tu.stages > 0 ? tu.stages
                                  : std::max(min_stages, std::min(6, kStageBudget / (nt * unit)));
        p->smem_bytes = bwd_smem_bytes(p->stages, unit, nt);
        return;
    }
    if (vector_ok) {
        // rows one block covers with 4 vectors per thread: as many row groups
        // as 512 threads hold (one for the widest rows, five at 96 threads)
        const int tg = std::max(32, round_up(static_cast<int>(cdiv(nvec, tu.vectors)), 32));
        int groups = tu.groups > 0 ? tu.groups : std::max(1, std::min(kMaxRowGroups, 512 / tg));
        while (groups > 1 && groups * tg > 512) --groups;
        if (tg <= 512) {
            const int unit = tu.vectors * tg * 16;
            int stages = tu.stages > 0 ? tu.stages
                                       : std::max(min_stages,
                                                  std::min(6, tu.smem_multi / (groups * nt * unit)));
            auto bytes = [&] { return bwd_row_smem_bytes(groups, stages, unit, nt); };
            if (res) {
                while (stages > min_stages && bytes() > kSmemMax) --stages;
                while (groups > 1 && bytes() > kSmemMax) --groups;
            } else {
                while (groups > 1 && bytes() > kSmemMax) --groups;
                while (stages > min_stages && bytes() > kSmemMax) --stages;
            }
            if (bytes() <= kSmemMax) {
                p->variant = RMSNORM_VARIANT_CTA_ROW;
                p->row_groups = groups;
                p->vectors_per_thread = tu.vectors;
                p->threads = tg * groups;
                p->threads_per_row = tg;
                p->rows_per_unit = groups;
                p->stages = stages;
                p->smem_bytes = bytes();
                return;
            }
        }
        // wider rows: split over a cluster, one row at a time per block
        auto try_wide = [&](int c, int st_min, int max_v = 8) {
            return wide_plan(nvec, nt, c, max_v, st_min, tu.stages, tu.smem_multi, p);
        };
        // a forced cluster size may run a two-deep ring; the ladder's own
        // sizes keep three stages (two with dres in the ring)
        if (tu.cluster > 0 && try_wide(tu.cluster, 2)) return;
        int c = 1;
        while (2 * cdiv(nvec, c) * 16 > tu.slice && c < kMaxCluster) c *= 2;
        // Clusters of 8 leave SMs idle: 15 fit at once on a 152-SM GB300 (120
        // SMs), against 28 of 5 (140) and 23 of 6 (138). A row that would take
        // 8 blocks takes 5 or 6 where 4 vectors a thread and a three-deep ring
        // fit (fp32 N = 40960: 89% against 63%; N = 49152: 87% against 69%;
        // bf16 N = 98304: 86% against 70%); an fp32 row also takes 5 blocks of
        // 8 vectors a thread with a two-deep ring (N = 65536: 89% against 79%),
        // which 16-bit rows do not (their 8-vector threads ran at 35-50%).
        if (c == kMaxCluster && !res) {
            if (try_wide(5, 3, 4) || try_wide(6, 3, 4)) return;
            if (sz == 4 && try_wide(5, 2)) return;
        }
        for (;; c *= 2) {
            if (try_wide(c, min_stages)) return;
            if (!res || c >= kMaxCluster) break;
        }
        // rows no cluster of 8 holds (past 256 KiB a row): a cluster of 16
        // blocks, a size the device must allow (bwd_finish_plan falls back to
        // the scalar kernel where it does not). On GB300 seven such clusters
        // fit (112 SMs): bf16 N = 196608 and 262144 ran at 63% and 71% of the
        // copy roofline, fp32 N = 131072 at 86%, against 6-21% for the scalar
        // kernel (fp32 N = 98304 takes 8 blocks of 8 vectors with a two-deep
        // ring in the device's choice: 101%)
        if (tu.cluster == 0 &&
            (try_wide(kClusterWideMax, min_stages) || (sz == 4 && !res && try_wide(kClusterWideMax, 2))))
            return;
    }
    scalar_plan(p);
}

namespace {

// Cluster-row plans chosen on a device, per (device, dtype, N).
std::mutex g_wide_mu;
std::map<std::tuple<int, int, int64_t, bool>, rmsnorm_plan_t> g_wide;

// A row split over a cluster runs best where the clusters resident at once
// (rows in flight) times the threads resident with them is largest; ties go
// to fewer, larger blocks (at N = 65536, 4 blocks of 512 threads against 8 of
// 256: fp16 81% against 77%, bf16 90% against 89%), then to the deeper ring. How
// many fit depends on registers, shared memory and the device's GPC layout,
// so the occupancy API counts them for cluster sizes 2, 4, 5, 6 and 8, four
// vectors a thread (also eight for fp32 rows) and rings two to six deep
// (three to six for 16-bit rows without dres, whose two-deep rings never
// gained there; with dres, a third tensor in the ring, two to six). On
// GB300 this took fp32 rows of N = 16384..49152 from 83..97% of the copy
// roofline to 93..101% (blocks of 128..448 threads, two-deep rings, two or
// more blocks to an SM) and bf16 N = 40960 from 72% to 91%.
cudaError_t wide_select(const DeviceInfo& dev, int dtype, int64_t N, bool res, rmsnorm_plan_t* p) {
    const auto key = std::make_tuple(dev.device, dtype, N, res);
    {
        std::lock_guard<std::mutex> lk(g_wide_mu);
        auto it = g_wide.find(key);
        if (it != g_wide.end()) {
            *p = it->second;
            return cudaSuccess;
        }
    }
    const int sz = dtype_size(dtype);
    const int64_t nvec = N / dtype_vec(dtype);
    const BwdTuning& tu = tuning();
    rmsnorm_plan_t best = *p;
    int64_t best_score[3] = {-1, -1, -1};
    for (int c : {2, 4, 5, 6, 8}) {
        for (int max_v : {4, 8}) {
            if (max_v == 8 && sz != 4) continue;
            for (int st = (sz == 4 || res) ? 2 : 3; st <= 6; ++st) {
                rmsnorm_plan_t q = *p;
                if (!wide_plan(nvec, res ? 3 : 2, c, max_v, st, st, tu.smem_multi, &q)) continue;
                if (q.cluster != c || q.stages != st || q.smem_bytes > dev.max_smem_optin) continue;
                const void* fn = main_kernel_for(dtype, q, res);
                if (fn == nullptr) continue;
                int units = 0;
                if (resident_units(dev, fn, q.threads, q.smem_bytes, c, &units) != cudaSuccess) {
                    cudaGetLastError();  // an occupancy query that fails rules the shape out
                    continue;
                }
                // rows in flight times resident threads, then fewer (larger)
                // blocks, then the deeper ring
                const int64_t blocks = static_cast<int64_t>(units) * c;
                const int64_t score[3] = {units * blocks * q.threads, -blocks, st};
                if (std::lexicographical_compare(best_score, best_score + 3, score, score + 3)) {
                    best = q;
                    std::copy(score, score + 3, best_score);
                }
            }
        }
    }
    std::lock_guard<std::mutex> lk(g_wide_mu);
    g_wide[key] = best;
    *p = best;
    return cudaSuccess;
}

}  // namespace

cudaError_t bwd_finish_plan(const DeviceInfo& dev, int dtype, int64_t M, int64_t N,
                            rmsnorm_plan_t* p, bool res) {
    const BwdTuning& tu = tuning();
    const bool wide_overridden = tu.cluster > 0 || tu.stages > 0 || tu.pipelined ||
                                 tu.smem_multi != 200 * 1024 || tu.slice != kSliceBudget;
    if (p->variant == RMSNORM_VARIANT_CLUSTER_ROW && !wide_overridden &&
        tu.wide_select >= (res ? 2 : 1)) {
        cudaError_t e = wide_select(dev, dtype, N, res, p);
        if (e != cudaSuccess) return e;
    }
    if (p->smem_bytes > dev.max_smem_optin) return cudaErrorInvalidConfiguration;
    const void* fn = main_kernel_for(dtype, *p, res);
    if (fn == nullptr) return cudaErrorInvalidValue;
    int units = 0;
    if (p->cluster > kMaxCluster) {
        // a non-portable cluster size: the scalar kernel where the device
        // refuses it or cannot hold one such cluster
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                cudaSuccess ||
            resident_units(dev, fn, p->threads, p->smem_bytes, p->cluster, &units) != cudaSuccess) {
            cudaGetLastError();
            scalar_plan(p);
            fn = main_kernel_for(dtype, *p, res);
            if (fn == nullptr) return cudaErrorInvalidValue;
        }
    }
    cudaError_t err = resident_units(dev, fn, p->threads, p->smem_bytes, p->cluster, &units);
    if (err != cudaSuccess) return err;
    int64_t work = M;  // rows, tiles of rows, or rows per block's row groups
    if (p->variant == RMSNORM_VARIANT_ROWGROUP || p->variant == RMSNORM_VARIANT_CTA_ROW)
        work = cdiv(M, p->rows_per_unit);
    const int64_t n = std::min<int64_t>(units, work);
    // Few rows for several blocks: one cluster of up to 16 blocks takes them
    // all and sums dw on chip (no partial rows in memory, no second kernel).
    // Eager forward + backward steps of 16 x 4096 bf16 went from 12.1 to
    // 9.5 us. Up to 16 units every block still takes one; with 64 (256 x 1024,
    // 256 x 4096) a block walked four and the steps took 2-3 us longer than
    // with the column sum.
    if ((p->variant == RMSNORM_VARIANT_ROWGROUP || p->variant == RMSNORM_VARIANT_CTA_ROW) &&
        p->cluster == 1 && n > 1 && work <= tu.cluster_dw_units) {
        int c = static_cast<int>(std::min<int64_t>(work, kClusterDwMax));
        for (; c >= 2; --c) {
            if (c > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                              cudaSuccess) {
                cudaGetLastError();
                continue;
            }
            int clusters = 0;
            if (resident_units(dev, fn, p->threads, p->smem_bytes, c, &clusters) == cudaSuccess &&
                clusters >= 1)
                break;
            cudaGetLastError();
        }
        if (c >= 2) {
            p->cluster = c;
            p->partial_rows = 1;
            p->grid = c;
            p->workspace_bytes = 0;
            return cudaSuccess;
        }
    }
    p->partial_rows = static_cast<int>(n);
    p->grid = static_cast<int>(n * p->cluster);
    // one partial row is dw itself: no workspace and no column sum
    p->workspace_bytes = n == 1 ? 0 : (n * N * 4 + 255) / 256 * 256;
    return cudaSuccess;
}

cudaError_t colsum_launch(const float* partial, float* dw, int P, int N, cudaStream_t s) {
    int device = 0;
    cudaError_t err = cudaGetDevice(&device);
    if (err != cudaSuccess) return err;
    const DeviceInfo* dev = device_info(device);
    int* status = dev ? dev->status_word : nullptr;
    void* args[5] = {&partial, &dw, &P, &N, &status};
    if (N < kColsumNarrowBelow) {
        const int c = colsum_narrow_cols(N);
        return cudaLaunchKernel(colsum_narrow_for(c), dim3(static_cast<unsigned>(cdiv(N, c))),
                                dim3(c, 1024 / c), args, 0, s);
    }
    const int q = colsum_phases(N, dev ? dev->sm_count : 1);
    const void* fn = colsum_kernel_for(q);
    return cudaLaunchKernel(fn, dim3(static_cast<unsigned>(cdiv(N, 32))), dim3(32, q), args, 0, s);
}

// Whether a backward launch may start early behind the previous kernel of
// the stream. Rows split over a cluster with a two-deep ring and two blocks
// to an SM go in plain stream order: launched early, the steady forward +
// backward step of fp32 rows of 32768 and 49152 ran at 85% and 83% of the
// copy roofline, in stream order at 95% and 97%. Every other wide plan
// measured (fp32 16384 and 65536, 16-bit 32768 to 98304) lost 1 point there.
static bool wide_pdl(const rmsnorm_plan_t& p, const void* fn) {
    if (p.variant != RMSNORM_VARIANT_CLUSTER_ROW) return true;
    const int mode = tuning().pdl_wide;
    if (mode >= 0) return mode == 1;
    if (p.stages != 2) return true;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    const DeviceInfo* dev = device_info(device);
    int units = 0;
    if (dev == nullptr || resident_units(*dev, fn, p.threads, p.smem_bytes, 1, &units) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return units / dev->sm_count != 2;
}

cudaError_t bwd_launch(const rmsnorm_plan_t& p, int dtype, const BwdArgs& a, cudaStream_t s) {
    if (p.grid <= 0) return cudaSuccess;
    const void* fn = main_kernel_for(dtype, p, a.dres != nullptr);
    if (fn == nullptr) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(p.threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(p.smem_bytes);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_allowed(wide_pdl(p, fn));
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(p.cluster);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    BwdArgs args = a;
    args.cluster_dw = p.cluster > 1 && p.variant != RMSNORM_VARIANT_CLUSTER_ROW;
    // A stage is refilled once pass 2 of its row is done (one more block
    // barrier a row) where a thread holds 8 vectors of a wide row: its row
    // takes twice as long, and refilling only after the next row's pass 1
    // left the two-deep ring of the fp32 2048 x 65536 backward at 90% of the
    // copy roofline (99% with the early refill). Everywhere else the extra
    // barrier cost 1-4 points and the later refill stays.
    args.early_refill = tuning().early_refill >= 0
                            ? tuning().early_refill
                            : (p.cluster > 1 && p.vectors_per_thread >= 8 ? 1 : 0);
    if (p.partial_rows == 1) args.partial = a.dw;  // the one partial row is dw
    int stages = p.stages, groups = p.row_groups;
    void* kargs[3] = {&args, &stages, &groups};
    cudaError_t err = cudaLaunchKernelExC(&cfg, fn, kargs);
    if (err != cudaSuccess) return err;
    if (p.partial_rows == 1) return cudaSuccess;
    // the column sum may launch early and waits on the grid above
    // (programmatic dependent launch) instead of a full stream boundary
    cudaLaunchConfig_t cs = {};
    const bool narrow = a.N < kColsumNarrowBelow;
    const int q = colsum_phases(a.N, a.sm_count);
    const int c = colsum_narrow_cols(a.N);
    cs.gridDim = dim3(static_cast<unsigned>(narrow ? cdiv(a.N, c) : cdiv(a.N, 32)));
    cs.blockDim = narrow ? dim3(static_cast<unsigned>(c), static_cast<unsigned>(1024 / c))
                         : dim3(32, static_cast<unsigned>(q));
    cs.stream = s;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = pdl_allowed();
    cs.attrs = pdl;
    cs.numAttrs = 1;
    const float* part = a.partial;
    float* dw = a.dw;
    int P = p.partial_rows, N = a.N;
    int* status = a.status;
    void* cargs[5] = {&part, &dw, &P, &N, &status};
    return cudaLaunchKernelExC(&cs, narrow ? colsum_narrow_for(c) : colsum_kernel_for(q), cargs);
}

}  // namespace rmsn
