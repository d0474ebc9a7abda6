// Device helpers shared by the RMSNorm kernels: 16-byte packing of
// fp32/bf16/fp16 rows and of weights stored in their own type, warp
// reductions, inline-PTX wrappers for mbarriers, 1-D bulk copies
// (cp.async.bulk, no tensor map), thread-block clusters and the global timer
// used by the bounded waits, and the range tests of the checked build.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace rmsn {

// Status codes written to the device status word (match rmsnorm_status_t).
constexpr int kStatusTimeout = 6;

// ---------------------------------------------------------------- packing
// A 16-byte vector holds VEC elements; arithmetic is always fp32.
template <typename T>
struct Pack;

// Pairs: a 16-byte vector seen as PAIRS float2 values, element 2e in .x and
// 2e+1 in .y, so that the element math runs on packed fp32x2 instructions
// (__ffma2_rn / __fmul2_rn: two IEEE round-to-nearest operations each).
template <>
struct Pack<float> {
    static constexpr int VEC = 4;
    static constexpr int PAIRS = 2;
    __device__ __forceinline__ static void unpack2(const uint4& v, float2 (&f)[PAIRS]) {
        f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
        f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
    }
    __device__ __forceinline__ static uint4 pack2(const float2 (&f)[PAIRS]) {
        return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y),
                          __float_as_uint(f[1].x), __float_as_uint(f[1].y));
    }
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[VEC]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[VEC]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                          __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
    __device__ __forceinline__ static float to_float(float v) { return v; }
    __device__ __forceinline__ static float from_float(float v) { return v; }
};

template <>
struct Pack<__nv_bfloat16> {
    static constexpr int VEC = 8;
    static constexpr int PAIRS = 4;
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
        return *reinterpret_cast<uint32_t*>(&h);
    }
    // one bf16x2 word -> one float2 (low half is the lower-addressed element):
    // a shift and a mask (the mixed-precision add that fp16 uses ran the
    // bf16 backward at 2048 x 65536 at 89.4% of the copy roofline, against
    // 92.9% this way)
    __device__ __forceinline__ static float2 word_to_f2(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    __device__ __forceinline__ static void unpack2(const uint4& v, float2 (&f)[PAIRS]) {
        f[0] = word_to_f2(v.x);
        f[1] = word_to_f2(v.y);
        f[2] = word_to_f2(v.z);
        f[3] = word_to_f2(v.w);
    }
    __device__ __forceinline__ static uint4 pack2(const float2 (&f)[PAIRS]) {
        return make_uint4(pack2(f[0].x, f[0].y), pack2(f[1].x, f[1].y), pack2(f[2].x, f[2].y),
                          pack2(f[3].x, f[3].y));
    }
    // bf16 is the high half of an fp32 bit pattern, so widening is a shift.
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[VEC]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            f[2 * k] = __uint_as_float(w[k] << 16);
            f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[VEC]) {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
    __device__ __forceinline__ static float to_float(__nv_bfloat16 v) {
        return __bfloat162float(v);
    }
    __device__ __forceinline__ static __nv_bfloat16 from_float(float v) {
        return __float2bfloat16_rn(v);
    }
};

template <>
struct Pack<__half> {
    static constexpr int VEC = 8;
    static constexpr int PAIRS = 4;
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);  // round to nearest even
        return *reinterpret_cast<uint32_t*>(&h);
    }
    // one f16x2 word -> one float2 (low half is the lower-addressed element).
    // Each half is widened by a mixed-precision add of -0.0, which is exact
    // (every binary16 value is an fp32 value, and x + (-0) = x for signed
    // zeros, infinities and NaN as well). Widening with conversions instead
    // held the fp16 backward at 16384 x 4096 to 89.6% of the copy roofline
    // (92.4% this way) and at 2048 x 65536 to 83.4% (89.2%).
    __device__ __forceinline__ static float2 word_to_f2(uint32_t w) {
        float lo, hi;
        asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "add.rn.f32.f16 %0, l, %3;\n\tadd.rn.f32.f16 %1, h, %3;\n\t}"
            : "=f"(lo), "=f"(hi)
            : "r"(w), "f"(-0.0f));
        return make_float2(lo, hi);
    }
    __device__ __forceinline__ static void unpack2(const uint4& v, float2 (&f)[PAIRS]) {
        f[0] = word_to_f2(v.x);
        f[1] = word_to_f2(v.y);
        f[2] = word_to_f2(v.z);
        f[3] = word_to_f2(v.w);
    }
    __device__ __forceinline__ static uint4 pack2(const float2 (&f)[PAIRS]) {
        return make_uint4(pack2(f[0].x, f[0].y), pack2(f[1].x, f[1].y), pack2(f[2].x, f[2].y),
                          pack2(f[3].x, f[3].y));
    }
    __device__ __forceinline__ static float to_float(__half v) { return __half2float(v); }
    __device__ __forceinline__ static __half from_float(float v) { return __float2half_rn(v); }
};

// Scalar widening of any stored element type.
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }

// The weights that go with one 16-byte activation vector of T, stored as TW:
// WORDS 16-byte words (one when TW is T; two for an fp32 weight with 16-bit
// activations), unpacked into the same float2 pairs as the activations.
template <typename T, typename TW>
struct WPack {
    static constexpr int VEC = Pack<T>::VEC;
    static constexpr int PAIRS = Pack<T>::PAIRS;
    static constexpr int WORDS = VEC * static_cast<int>(sizeof(TW)) / 16;
    static_assert(std::is_same<T, TW>::value || std::is_same<TW, float>::value,
                  "the weight has the activation type or fp32");
    // weights of activation vector k (elements k*VEC .. k*VEC+VEC-1)
    __device__ __forceinline__ static void load(const TW* w, int64_t k, uint4 (&o)[WORDS]) {
        const uint4* p = reinterpret_cast<const uint4*>(w + k * VEC);
#pragma unroll
        for (int q = 0; q < WORDS; ++q) o[q] = __ldg(p + q);
    }
    __device__ __forceinline__ static void zero(uint4 (&o)[WORDS]) {
#pragma unroll
        for (int q = 0; q < WORDS; ++q) o[q] = make_uint4(0, 0, 0, 0);
    }
    __device__ __forceinline__ static void unpack2(const uint4 (&o)[WORDS], float2 (&f)[PAIRS]) {
        if constexpr (std::is_same<T, TW>::value) {
            Pack<T>::unpack2(o[0], f);
        } else {
#pragma unroll
            for (int q = 0; q < WORDS; ++q) {
                f[2 * q] = make_float2(__uint_as_float(o[q].x), __uint_as_float(o[q].y));
                f[2 * q + 1] = make_float2(__uint_as_float(o[q].z), __uint_as_float(o[q].w));
            }
        }
    }
};

__device__ __forceinline__ float2 f2_splat(float v) { return make_float2(v, v); }

// a + b element by element, each sum computed in fp32 and rounded once into
// T (for 16-bit T the fp32 sum of two T values is exact unless the two
// exponents are far apart, and then the smaller one is below half an ulp of
// the larger, so the result is the correctly rounded sum either way).
template <typename T>
__device__ __forceinline__ uint4 add_vec(const uint4& a, const uint4& b) {
    using P = Pack<T>;
    float2 fa[P::PAIRS], fb[P::PAIRS];
    P::unpack2(a, fa);
    P::unpack2(b, fb);
#pragma unroll
    for (int e = 0; e < P::PAIRS; ++e) fa[e] = __fadd2_rn(fa[e], fb[e]);
    return P::pack2(fa);
}

// ------------------------------------------------------------ global memory
// Streaming read: the row is used once, do not keep it in L1.
__device__ __forceinline__ uint4 ld_global_16_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void st_global_16(void* p, const uint4& v) {
    *reinterpret_cast<uint4*>(p) = v;
}

// L2 eviction-priority policies (createpolicy): evict_last keeps lines that
// will be read again soon, evict_first marks lines used for the last time.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint4 ld_global_16_hint(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
// Coherent read with an L2 policy, ordered after this thread's earlier
// memory accesses (it reads back what the same thread stored).
__device__ __forceinline__ uint4 ld_global_16_coherent_hint(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol)
                 : "memory");
    return v;
}
__device__ __forceinline__ void st_global_16_hint(void* p, const uint4& v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

// ------------------------------------------------------------ reductions
// xor butterfly: every lane ends with the same bits (each step adds the
// same two operands in both partner lanes, and fp32 addition commutes).
template <int WIDTH>
__device__ __forceinline__ float group_allreduce(float v) {
#pragma unroll
    for (int off = WIDTH / 2; off >= 1; off /= 2) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// -------------------------------------------------------------- shared memory
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint4 ld_shared_16(const void* p) {
    return *reinterpret_cast<const uint4*>(p);
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
// Makes the initialised barriers visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase with the given parity to complete, for at most
// limit_ns nanoseconds. Returns false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
#pragma unroll 1
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// ------------------------------------------------------------ bulk copies
// 1-D global -> shared copy completed on an mbarrier (complete_tx). Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst_smem, const void* src_gmem,
                                              uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses to the same buffers.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ clusters
// Without a cluster launch every block is its own cluster of one.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// Full cluster barrier: release this thread's prior shared-memory writes,
// acquire the other blocks' ones. Every thread of every block calls it.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::
            : "memory");
}
// Split cluster barrier: arrive without ordering (after initialising
// barriers that peers will use), wait with acquire before using theirs.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Reads 16 bytes (16-byte aligned) from the same shared-memory location in
// block `rank` of this cluster.
__device__ __forceinline__ float4 ld_cluster_f32x4(const float* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(remote)
                 : "memory");
    return v;
}

// Address of the same shared-memory location in block `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    return remote;
}
// Asynchronous store of 4 bytes into another block's shared memory whose
// completion is counted (4 transaction bytes) on that block's mbarrier.
__device__ __forceinline__ void st_async_cluster_f32(uint32_t remote, float v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                     remote),
                 "r"(__float_as_uint(v)), "r"(remote_bar)
                 : "memory");
}
// try_wait with acquire at cluster scope: makes the writes released by
// remote arrivals on this barrier visible to the waiting thread.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity,
                                                          uint64_t limit_ns) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
        if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
#pragma unroll 1
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// ------------------------------------------ programmatic dependent launch
// Every library kernel is launched with programmatic stream serialization:
// it may start while the previous kernel of the stream finishes, does only
// work that touches no global memory (index math, shared-memory and
// mbarrier set-up), then waits for the prerequisite grid -- its completion
// and the visibility of its memory -- before the first global load or store.
// Without a programmatic edge the wait returns at once.
__device__ __forceinline__ void wait_for_prerequisite_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel of the stream launch while this grid finishes; that
// kernel still waits for this grid's completion before touching memory.
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Records the first failure on the device status word.
__device__ __forceinline__ void report_status(int* status, int code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------ checked build
// A debug build of the library (compiled with -DRMSNORM_CHECKS) checks every
// global access of the kernels against the extent of the tensor it belongs
// to (M*N elements for the activations, N for w and dw, M for rstd, the
// partial rows for the workspace) and every ring access against the block's
// dynamic shared memory, before it happens. A failed check records
// kStatusOutOfBounds on the device status word and skips the access: it
// never traps. In the normal build RMSN_OK(...) is the constant true and the
// checks are not compiled at all, so the kernels are unchanged.
constexpr int kStatusOutOfBounds = 7;

// [p, p + n) lies inside [base, base + extent); n and extent in bytes.
__host__ __device__ __forceinline__ bool span_in(const void* p, int64_t n, const void* base,
                                                 int64_t extent) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(base);
    return n >= 0 && extent >= 0 && a >= b && a - b <= static_cast<uintptr_t>(extent) &&
           static_cast<uintptr_t>(n) <= static_cast<uintptr_t>(extent) - (a - b);
}

// Every extern dynamic shared-memory array of a kernel starts at this address.
extern __shared__ __align__(128) unsigned char rmsn_dynamic_smem[];

__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
    uint32_t v;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
    return v;
}
// [p, p + n) lies inside the block's dynamic shared memory.
__device__ __forceinline__ bool smem_span_in(const void* p, uint32_t n) {
    const uint32_t a = smem_u32(p), b = smem_u32(rmsn_dynamic_smem);
    return a >= b && a - b <= dynamic_smem_bytes() && n <= dynamic_smem_bytes() - (a - b);
}

__device__ __forceinline__ bool record_if_out(bool ok, int* status) {
    if (!ok) report_status(status, kStatusOutOfBounds);
    return ok;
}

#ifdef RMSNORM_CHECKS
#define RMSN_OK(cond, status) ::rmsn::record_if_out((cond), (status))
#else
#define RMSN_OK(cond, status) true
#endif

// A 16-byte ring read: checked against the dynamic shared memory in the
// checked build (an out-of-range read gives zeros), a plain load otherwise.
__device__ __forceinline__ uint4 ld_ring_16(const void* p, int* status) {
    if (!RMSN_OK(smem_span_in(p, 16), status)) return make_uint4(0, 0, 0, 0);
    return ld_shared_16(p);
}

}  // namespace rmsn
