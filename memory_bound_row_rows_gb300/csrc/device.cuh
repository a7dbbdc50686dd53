// Device-side building blocks for the row-softmax kernels (sm_103a).
//
// Inline PTX for the Blackwell data-movement path: mbarrier transaction
// barriers, 1-D bulk asynchronous copies global -> shared
// (cp.async.bulk ... mbarrier::complete_tx), cluster ranks, distributed
// shared memory (mapa / st.shared::cluster) and cluster barriers; plus
// 16-byte streaming loads and stores, and the element packing for
// f32 / bf16 / f16.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sr {

constexpr float kLog2e = 1.4426950408889634074f;

// ---------------------------------------------------------------------------
// Bounds-checking build (compiled with -DSR_BOUNDS_CHECK=1 and relocatable
// device code; never in the product library). Every kernel first records the
// extents of the matrices of its call in a per-block table: each matrix as
// rows of `row_bytes` valid bytes at a pitch of `ld_bytes`, readable or
// writable. Every global load, store and bulk copy then checks that all of
// its bytes lie inside the valid columns of one row of a matrix that allows
// the access. An access that does not is skipped (a load returns NaN bits),
// bit 1 of the device error word is set and the first offending address is
// kept, so that softmax_rows_last_device_error reports SR_EBOUNDS: the
// checks record, they never trap.
// ---------------------------------------------------------------------------
#ifndef SR_BOUNDS_CHECK
#define SR_BOUNDS_CHECK 0
#endif
constexpr unsigned int kErrTimeout = 1u;
constexpr unsigned int kErrBounds = 2u;

// Programmatic dependent launch (see launch_kernel in internal.h): the first
// statement of every kernel. It lets the next kernel on the stream be
// scheduled once every block of this one has started, then waits until the
// previous kernel on the stream has completed and its memory is visible; no
// global memory is touched before it.
#ifndef SR_PDL
#define SR_PDL 1
#endif
#if SR_PDL
#define SR_GRID_DEPENDENCY()                                          \
    do {                                                              \
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); \
        asm volatile("griddepcontrol.wait;" ::: "memory");            \
    } while (0)
#else
#define SR_GRID_DEPENDENCY() ((void)0)
#endif

#if SR_BOUNDS_CHECK
extern __device__ unsigned int g_error_word;
extern __device__ unsigned long long g_bounds_addr;
// Test hook: bytes taken off the end of every writable region's rows, so that
// a correct kernel's last stores fall outside and must be refused.
extern __device__ long long g_bounds_shrink;

namespace bounds {

struct Region {
    const char* base;
    int64_t rows, ld_bytes, row_bytes;
    int writable;
};
constexpr int kMaxRegions = 4;
struct Table {
    int n;
    Region r[kMaxRegions];
};
static __shared__ Table s_table;

// A matrix of `rows` rows of n elements of `es` bytes at a pitch of ld elements.
__device__ __forceinline__ Region matrix(const void* base, int64_t rows, int64_t ld, int64_t n,
                                         int es, bool writable) {
    return Region{static_cast<const char*>(base), base ? rows : 0, ld * es, n * es,
                  writable ? 1 : 0};
}
// A contiguous run of `bytes` bytes (a vector or a workspace).
__device__ __forceinline__ Region span(const void* base, int64_t bytes, bool writable) {
    return Region{static_cast<const char*>(base), base ? 1 : 0, bytes, bytes, writable ? 1 : 0};
}

template <typename... R>
__device__ __forceinline__ void begin(R... regions) {
    static_assert(sizeof...(R) <= kMaxRegions, "too many regions");
    if (threadIdx.x == 0) {
        const Region list[] = {regions...};
        s_table.n = (int)sizeof...(R);
        for (int i = 0; i < (int)sizeof...(R); ++i) {
            s_table.r[i] = list[i];
            if (list[i].writable) s_table.r[i].row_bytes -= g_bounds_shrink;
        }
    }
    __syncthreads();
}

static __device__ __noinline__ bool inside(const void* p, int64_t bytes, bool write) {
    const char* a = static_cast<const char*>(p);
    for (int i = 0; i < s_table.n; ++i) {
        const Region& g = s_table.r[i];
        if ((write && !g.writable) || g.rows <= 0 || a < g.base) continue;
        const int64_t off = a - g.base;
        if (off >= g.rows * g.ld_bytes) continue;
        const int64_t row = off / g.ld_bytes;
        if (off - row * g.ld_bytes + bytes <= g.row_bytes) return true;
    }
    atomicOr(&g_error_word, kErrBounds);
    atomicCAS(&g_bounds_addr, 0ull, (unsigned long long)(uintptr_t)p);
    return false;
}

}  // namespace bounds

#define SR_BOUNDS_BEGIN(...) ::sr::bounds::begin(__VA_ARGS__)
#define SR_READ_OK(p, bytes) ::sr::bounds::inside((p), (bytes), false)
#define SR_WRITE_OK(p, bytes) ::sr::bounds::inside((p), (bytes), true)
#else
#define SR_BOUNDS_BEGIN(...) ((void)0)
#define SR_READ_OK(p, bytes) true
#define SR_WRITE_OK(p, bytes) true
#endif
// Regions for SR_BOUNDS_BEGIN: a matrix read or written by the call (rows of
// n elements of *p's type at a pitch of ld), and a contiguous run of bytes.
#define SR_MAT_IN(p, rows, ld, n) \
    ::sr::bounds::matrix((p), (rows), (ld), (n), (int)sizeof(*(p)), false)
#define SR_MAT_OUT(p, rows, ld, n) \
    ::sr::bounds::matrix((p), (rows), (ld), (n), (int)sizeof(*(p)), true)
#define SR_SPAN_IN(p, bytes) ::sr::bounds::span((p), (bytes), false)
#define SR_SPAN_OUT(p, bytes) ::sr::bounds::span((p), (bytes), true)

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000u); }

// ---------------------------------------------------------------------------
// Element packing. A 16-byte vector holds kVec elements of storage type T.
// unpack() widens to float exactly; pack() rounds to nearest even once.
// ---------------------------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int kVec = 4;
    static constexpr bool kAccurateExp = true;
    __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ __forceinline__ static float load1(const float* p) {
        if (!SR_READ_OK(p, 4)) return __int_as_float(0x7fc00000);
        return __ldg(p);
    }
    __device__ __forceinline__ static void store1(float* p, float v) {
        if (SR_WRITE_OK(p, 4)) __stcs(p, v);
    }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
    static constexpr bool kAccurateExp = false;
    __device__ __forceinline__ static void unpack2(uint32_t w, float* f) {
        f[0] = __uint_as_float(w << 16);
        f[1] = __uint_as_float(w & 0xffff0000u);
    }
    __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
        unpack2(u.x, f + 0);
        unpack2(u.y, f + 2);
        unpack2(u.z, f + 4);
        unpack2(u.w, f + 6);
    }
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
    __device__ __forceinline__ static float load1(const __nv_bfloat16* p) {
        if (!SR_READ_OK(p, 2)) return __int_as_float(0x7fc00000);
        unsigned short s = __ldg(reinterpret_cast<const unsigned short*>(p));
        return __uint_as_float(((uint32_t)s) << 16);
    }
    __device__ __forceinline__ static void store1(__nv_bfloat16* p, float v) {
        if (SR_WRITE_OK(p, 2)) *p = __float2bfloat16_rn(v);
    }
};

template <>
struct Elem<__half> {
    static constexpr int kVec = 8;
    static constexpr bool kAccurateExp = false;
    __device__ __forceinline__ static void unpack2(uint32_t w, float* f) {
        __half2 h = *reinterpret_cast<__half2*>(&w);
        float2 v = __half22float2(h);
        f[0] = v.x;
        f[1] = v.y;
    }
    __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
        unpack2(u.x, f + 0);
        unpack2(u.y, f + 2);
        unpack2(u.z, f + 4);
        unpack2(u.w, f + 6);
    }
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
    __device__ __forceinline__ static float load1(const __half* p) {
        if (!SR_READ_OK(p, 2)) return __int_as_float(0x7fc00000);
        unsigned short s = __ldg(reinterpret_cast<const unsigned short*>(p));
        return __half2float(*reinterpret_cast<__half*>(&s));
    }
    __device__ __forceinline__ static void store1(__half* p, float v) {
        if (SR_WRITE_OK(p, 2)) *p = __float2half_rn(v);
    }
};

// ---------------------------------------------------------------------------
// Exponential of (x - shift). FP32 data uses the accurate library expf on the
// exact difference (its outputs are compared at 1e-6). 16-bit data uses one
// FMA and the hardware base-2 exponential: x*log2(e) - shift*log2(e), whose
// relative error (~1e-6) is far below one bf16/f16 unit in the last place.
// `shift_l2` is shift*log2(e), precomputed per row.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T>
__device__ __forceinline__ float exp_shifted(float x, float shift, float shift_l2) {
    if constexpr (Elem<T>::kAccurateExp) {
        return expf(x - shift);
    } else {
        return ex2_approx(fmaf(x, kLog2e, -shift_l2));
    }
}

// ---------------------------------------------------------------------------
// Warp reductions (butterfly, every lane ends with the result).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Scale factor exp(m - mref) of a partial (max m, sum s) being merged into a
// result whose max is mref, with the all -inf guard of the online merge: a
// part whose max is -inf contributes 0 (exp(-inf - (-inf)) is never formed).
// Multiplying a NaN partial sum by it still gives NaN, so NaN propagates.
__device__ __forceinline__ float merge_scale(float m, float mref) {
    return (m == neg_inf()) ? 0.0f : expf(m - mref);
}

// Online (max, sum) merge: (m, s) <- (m, s) combined with (m2, s2).
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2) {
    const float mn = fmaxf(m, m2);
    s = s * merge_scale(m, mn) + s2 * merge_scale(m2, mn);
    m = mn;
}

// 1/S for the final normalisation, NaN when the whole row was -inf (0/0 by
// the definition) so that every output of such a row is NaN.
__device__ __forceinline__ float final_rcp(float M, float S) {
    return (M == neg_inf()) ? __int_as_float(0x7fc00000) : __frcp_rn(S);
}

// ---------------------------------------------------------------------------
// Global memory: 16-byte streaming load (read-only path, no L1 allocation)
// and streaming store.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    if (!SR_READ_OK(p, 16)) return make_uint4(0x7fc00000u, 0x7fc00000u, 0x7fc00000u, 0x7fc00000u);
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void stg_stream(void* p, const uint4& v) {
    if (!SR_WRITE_OK(p, 16)) return;
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------------------
// Shared memory, mbarriers and bulk copies.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// 1-D bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
// from global memory into this CTA's shared memory; completion is signalled
// on the mbarrier as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    // A refused copy never completes: the bounded wait for it expires.
    if (!SR_READ_OK(src, bytes)) return;
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of the mbarrier to complete, for at most
// `timeout_ns` nanoseconds of wall time. Returns false on expiry.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
#pragma unroll 1
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
}

// ---------------------------------------------------------------------------
// Thread-block clusters and distributed shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// Asynchronous 16-byte store into (possibly another block's) shared memory,
// completing 16 transaction bytes on the mbarrier at `remote_bar` (both are
// shared::cluster addresses of the same destination block).
__device__ __forceinline__ void st_async_f4(uint32_t remote_addr, float4 v, uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::
            "r"(remote_addr),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
        : "memory");
}

// The same for an 8-byte pair.
__device__ __forceinline__ void st_async_f2(uint32_t remote_addr, float a, float b,
                                            uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
            remote_addr),
        "f"(a), "f"(b), "r"(remote_bar)
        : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

}  // namespace sr
