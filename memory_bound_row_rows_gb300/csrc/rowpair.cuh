// Row-pair engine: kernels for operations that read two M x N matrices A and
// B, reduce each row to one FP32 number, and write C = f(A, B, that number)
// elementwise. The softmax backward (A = y, B = dy, the number is the dot
// product) and the residual RMSNorm (A = x, B = residual, the number is the
// inverse RMS) are such operations; an Op type supplies the arithmetic:
//
//   struct Op {
//     // acc += the element's contribution to the row's reduction
//     __device__ void accumulate(float& acc, float a, float b) const;
//     // the row's number from the FP32 sum of all contributions
//     __device__ float finish(float total, int64_t N) const;
//     // per-column data of n columns (the RMSNorm weights; empty otherwise),
//     // loaded together with the row so that no load waits on the reduction
//     template <int n> struct Aux;
//     template <int n> __device__ Aux<n> load_aux(int64_t col) const;
//     // out[e] = the result at the n columns the unit covers
//     template <int n> __device__ void apply(const float* a, const float* b, float s,
//                                            const Aux<n>& aux, float* out) const;
//     // whether the ROW kernel is compiled for higher occupancy (see team_bounded)
//     static constexpr bool kBoundTeam;
//   };
//
// Three plans, each reading A and B once (ONLINE: twice) and writing C once:
//  ROW      a team of 32..512 threads per row holds the row in registers and
//           reduces with shuffles (plus one shared-memory step for teams
//           wider than a warp); one-warp teams share a block four to one.
//  CLUSTER  the C blocks of a thread-block cluster hold a row in C slices;
//           each block stores its partial into every block's shared memory
//           (distributed shared memory) and one hardware cluster barrier
//           makes them visible; every block adds the C partials in rank order,
//           so all blocks of a row use the same number.
//           Aligned rows too wide for the cluster's registers are streamed:
//           each block reads its slice to reduce it and again to write.
//  ONLINE   one block per row reads the row to reduce it, then again to write.
//
// Units: with Mode::kAligned every row of all three matrices starts on a
// 16-byte boundary and holds whole 16-byte vectors; with Mode::kShifted the
// rows of the three matrices share the same offset from a 16-byte boundary
// (the same base offset and pitch modulo 16 bytes), so each row is a head of
// fewer than VEC elements, 16-byte vectors, and a tail of fewer than VEC
// elements; the head and tail elements go one per thread. Mode::kScalar
// loads single elements. A thread's columns are the same in every row in the
// aligned mode, so its per-column data is loaded once, before the first row.
#pragma once

#include <type_traits>

#include "device.cuh"
#include "internal.h"
#include "rowpair.h"

namespace sr {
namespace rp {

// Units per thread a plan aims for, and the most it holds.
template <typename T, Mode MODE>
struct KvTarget {
    static constexpr bool kWide = MODE != Mode::kScalar;
    static constexpr int kTarget = kWide ? 4 : 8;
    static constexpr int kMax = kWide ? (sizeof(T) == 4 ? 8 : 4) : 16;
};

// One load unit: a 16-byte vector or a single element.
template <typename T, bool WIDE>
struct Unit;

template <typename T>
struct Unit<T, true> {
    static constexpr int kN = Elem<T>::kVec;
    uint4 raw;
    __device__ __forceinline__ void zero() { raw = make_uint4(0u, 0u, 0u, 0u); }
    __device__ __forceinline__ void load(const T* p) { raw = ldg_stream(p); }
    __device__ __forceinline__ void get(float* f) const { Elem<T>::unpack(raw, f); }
    // The same values, widened again from the stored vector. For 16-bit data
    // the empty asm hides that they equal an earlier get(), so the compiler
    // keeps the packed vector (4 registers) across the row's reduction
    // instead of the widened floats (8), which lets more blocks share an SM.
    __device__ __forceinline__ void get_again(float* f) const {
        uint4 r = raw;
        if constexpr (sizeof(T) == 2)
            asm volatile("" : "+r"(r.x), "+r"(r.y), "+r"(r.z), "+r"(r.w));
        Elem<T>::unpack(r, f);
    }
    __device__ __forceinline__ static void put(T* p, const float* f) {
        stg_stream(p, Elem<T>::pack(f));
    }
};

template <typename T>
struct Unit<T, false> {
    static constexpr int kN = 1;
    float v;
    __device__ __forceinline__ void zero() { v = 0.0f; }
    __device__ __forceinline__ void load(const T* p) { v = Elem<T>::load1(p); }
    __device__ __forceinline__ void get(float* f) const { f[0] = v; }
    __device__ __forceinline__ void get_again(float* f) const { f[0] = v; }
    __device__ __forceinline__ static void put(T* p, const float* f) { Elem<T>::store1(p, f[0]); }
};

// Where a row's units and its head/tail elements are.
template <typename T, Mode MODE>
struct Layout {
    static constexpr int VEC = MODE == Mode::kScalar ? 1 : Elem<T>::kVec;
    int head = 0;      // elements before the first 16-byte boundary
    int64_t nv = 0;    // units (vectors, or elements with kScalar)
    int extra = 0;     // head + tail elements
    __device__ __forceinline__ Layout(const T* row, int64_t N) {
        if constexpr (MODE == Mode::kShifted) {
            const int off = (int)((reinterpret_cast<uintptr_t>(row) & 15u) / sizeof(T));
            head = off ? VEC - off : 0;
            if (head > N) head = (int)N;
            nv = (N - head) / VEC;
            extra = (int)(N - nv * VEC);
        } else {
            nv = N / VEC;
        }
    }
    __device__ __forceinline__ int64_t unit_col(int64_t i) const { return head + i * VEC; }
    __device__ __forceinline__ int64_t extra_col(int k) const {
        return k < head ? k : head + nv * VEC + (k - head);
    }
};

template <int VEC>
__device__ __forceinline__ float fold(float* acc) {
#pragma unroll
    for (int w = VEC / 2; w > 0; w >>= 1)
#pragma unroll
        for (int e = 0; e < w; ++e) acc[e] += acc[e + w];
    return acc[0];
}

// Sum of one value per thread over the NW warps starting at warp w0, through
// red[] (callers alternate two buffers per row, so a warp may write the next
// row's partial before a slower warp has read this row's).
template <int NW>
__device__ __forceinline__ float team_sum(float v, float* red, int w0) {
    v = warp_sum(v);
    if constexpr (NW == 1) {
        return v;
    } else {
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
        __syncthreads();
        float s = red[w0];
#pragma unroll
        for (int w = 1; w < NW; ++w) s += red[w0 + w];
        return s;
    }
}

template <class Op, typename T, bool WIDE>
__device__ __forceinline__ void accumulate_unit(const Op& op, const Unit<T, WIDE>& a,
                                                const Unit<T, WIDE>& b, float* acc) {
    constexpr int VEC = Unit<T, WIDE>::kN;
    float fa[VEC], fb[VEC];
    a.get(fa);
    b.get(fb);
#pragma unroll
    for (int e = 0; e < VEC; ++e) op.accumulate(acc[e], fa[e], fb[e]);
}

template <class Op, typename T, bool WIDE>
__device__ __forceinline__ void write_unit(const Op& op, const Unit<T, WIDE>& a,
                                           const Unit<T, WIDE>& b, float s,
                                           const typename Op::template Aux<Unit<T, WIDE>::kN>& aux,
                                           T* p) {
    constexpr int VEC = Unit<T, WIDE>::kN;
    float fa[VEC], fb[VEC], f[VEC];
    a.get_again(fa);
    b.get_again(fb);
    op.template apply<VEC>(fa, fb, s, aux, f);
    Unit<T, WIDE>::put(p, f);
}

// The head/tail element a thread owns (if any) in a kShifted row.
template <class Op, typename T>
struct Extra {
    float a = 0.0f, b = 0.0f;
    int64_t col = -1;
    typename Op::template Aux<1> aux;
    __device__ __forceinline__ void load(const Op& op, const T* ra, const T* rb, int64_t c) {
        col = c;
        a = Elem<T>::load1(ra + c);
        b = Elem<T>::load1(rb + c);
        aux = op.template load_aux<1>(c);
    }
    __device__ __forceinline__ void accumulate(const Op& op, float* acc) const {
        if (col >= 0) op.accumulate(acc[0], a, b);
    }
    __device__ __forceinline__ void write(const Op& op, float s, T* rc) const {
        if (col >= 0) {
            float f;
            op.template apply<1>(&a, &b, s, aux, &f);
            Elem<T>::store1(rc + col, f);
        }
    }
};

// ---------------------------------------------------------------------------
// ROW plan.
// ---------------------------------------------------------------------------
template <class Op, typename T, Mode MODE, int TPR, int KV>
__device__ __forceinline__ void team_body(Op op, const T* __restrict__ A, const T* __restrict__ B,
                                          T* __restrict__ C, int64_t M, int64_t N, int64_t lda,
                                          int64_t ldb, int64_t ldc) {
    constexpr bool WIDE = MODE != Mode::kScalar;
    using U = Unit<T, WIDE>;
    using L = Layout<T, MODE>;
    constexpr int VEC = U::kN;
    using AuxV = typename Op::template Aux<VEC>;
    constexpr int NT = TPR < 128 ? 128 : TPR;
    constexpr int RPB = NT / TPR;  // rows per block
    constexpr int NW = TPR / 32;   // warps per team
    __shared__ float red[2][NT / 32];
    const int tid = threadIdx.x, t = tid % TPR;
    const int w0 = (tid / TPR) * NW;
    AuxV aux[KV];
    if constexpr (MODE == Mode::kAligned) {  // the same columns in every row
        const L lay(A, N);
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int64_t idx = t + TPR * k;
            if (idx < lay.nv) aux[k] = op.template load_aux<VEC>(lay.unit_col(idx));
        }
    }
    int parity = 0;
    for (int64_t r0 = (int64_t)blockIdx.x * RPB; r0 < M; r0 += (int64_t)gridDim.x * RPB) {
        const int64_t r = r0 + tid / TPR;
        const bool live = r < M;
        const T* ra = A + r * lda;
        const T* rb = B + r * ldb;
        const L lay(ra, live ? N : 0);
        U a[KV], b[KV];
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int64_t idx = t + TPR * k;
            if (idx < lay.nv) {
                a[k].load(ra + lay.unit_col(idx));
                b[k].load(rb + lay.unit_col(idx));
                if constexpr (MODE != Mode::kAligned)
                    aux[k] = op.template load_aux<VEC>(lay.unit_col(idx));
            } else {
                a[k].zero();
                b[k].zero();
            }
        }
        Extra<Op, T> ex;
        if constexpr (MODE == Mode::kShifted)
            if (t < lay.extra) ex.load(op, ra, rb, lay.extra_col(t));
        float acc[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
#pragma unroll
        for (int k = 0; k < KV; ++k) accumulate_unit<Op, T, WIDE>(op, a[k], b[k], acc);
        if constexpr (MODE == Mode::kShifted) ex.accumulate(op, acc);
        const float s = op.finish(team_sum<NW>(fold<VEC>(acc), red[parity], w0), N);
        parity ^= 1;
        T* rc = C + r * ldc;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int64_t idx = t + TPR * k;
            if (idx < lay.nv)
                write_unit<Op, T, WIDE>(op, a[k], b[k], s, aux[k], rc + lay.unit_col(idx));
        }
        if constexpr (MODE == Mode::kShifted) ex.write(op, s, rc);
    }
}

// The ROW kernel, and the same kernel compiled for at least 24 resident warps
// per SM (at most 85 registers at 256 threads), used for the operations whose
// Op sets kBoundTeam on the element types SR_PAIR_TEAM_BOUND selects: 0 none,
// 1 bf16, 2 both 16-bit types, 3 all. Unbounded, the bf16 RMSNorm kernels took
// 92-96 registers (2 blocks of 256 threads per SM); bounded, bf16 8192 x 8192
// went from 77.0 to 65.9 µs on GB300 (cold L2), while the f16 kernels and the
// backward gained nothing.
#ifndef SR_PAIR_TEAM_BOUND
#define SR_PAIR_TEAM_BOUND 1
#endif
template <class Op, typename T>
constexpr bool team_bounded() {
    return Op::kBoundTeam &&
           (SR_PAIR_TEAM_BOUND >= 3 || (SR_PAIR_TEAM_BOUND == 2 && sizeof(T) == 2) ||
            (SR_PAIR_TEAM_BOUND == 1 && std::is_same<T, __nv_bfloat16>::value));
}

template <class Op, typename T, Mode MODE, int TPR, int KV>
__global__ void __launch_bounds__(TPR < 128 ? 128 : TPR)
    team_kernel(Op op, const T* __restrict__ A, const T* __restrict__ B, T* __restrict__ C,
                int64_t M, int64_t N, int64_t lda, int64_t ldb, int64_t ldc) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(A, M, lda, N), SR_MAT_IN(B, M, ldb, N), SR_MAT_OUT(C, M, ldc, N),
                    SR_SPAN_IN(op.aux_base(), N * (int64_t)sizeof(T)));
    team_body<Op, T, MODE, TPR, KV>(op, A, B, C, M, N, lda, ldb, ldc);
}

template <class Op, typename T, Mode MODE, int TPR, int KV>
__global__ void __launch_bounds__(TPR < 128 ? 128 : TPR, 768 / (TPR < 128 ? 128 : TPR))
    team_kernel_bounded(Op op, const T* __restrict__ A, const T* __restrict__ B,
                        T* __restrict__ C, int64_t M, int64_t N, int64_t lda, int64_t ldb,
                        int64_t ldc) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(A, M, lda, N), SR_MAT_IN(B, M, ldb, N), SR_MAT_OUT(C, M, ldc, N),
                    SR_SPAN_IN(op.aux_base(), N * (int64_t)sizeof(T)));
    team_body<Op, T, MODE, TPR, KV>(op, A, B, C, M, N, lda, ldb, ldc);
}

// ---------------------------------------------------------------------------
// CLUSTER plan: csize blocks per row, `slice` units per block; the head and
// tail elements of a kShifted row belong to rank 0.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Asynchronous 4-byte store into a peer's shared memory, completing 4
// transaction bytes on the peer's mbarrier (both shared::cluster addresses).
__device__ __forceinline__ void st_async_f32(uint32_t remote_addr, float v, uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(
            remote_addr),
        "f"(v), "r"(remote_bar)
        : "memory");
}

// The partials travel by st.async and complete on each receiver's exchange
// mbarrier (no cluster barrier and no release fence in the row); a receiver's
// wait is bounded, and a block whose wait expires writes nothing more,
// records the failure in the error word and waits once more (bounded) before
// it leaves, so that a late partial cannot land after it exits.
// Resident blocks per SM the CLUSTER kernel is compiled for (at most 4 units
// per thread). Without a bound the RMSNorm kernel for bf16 took 122 registers
// (2 blocks/SM): at 4 blocks/SM bf16 2048 x 65536 went from 197 to 157 µs,
// and the other shapes measured stayed within 2 %.
#ifndef SR_PAIR_CLUSTER_MIN_BLOCKS
#define SR_PAIR_CLUSTER_MIN_BLOCKS 4
#endif
template <class Op, typename T, Mode MODE, int KV>
__global__ void __launch_bounds__(kClusterThreads, KV <= 4 ? SR_PAIR_CLUSTER_MIN_BLOCKS : 2)
    cluster_kernel(Op op, const T* __restrict__ A, const T* __restrict__ B, T* __restrict__ C,
                   int64_t M, int64_t N, int64_t lda, int64_t ldb, int64_t ldc, int csize,
                   int64_t slice, unsigned int* err, unsigned long long timeout_ns,
                   int flags) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(A, M, lda, N), SR_MAT_IN(B, M, ldb, N), SR_MAT_OUT(C, M, ldc, N),
                    SR_SPAN_IN(op.aux_base(), N * (int64_t)sizeof(T)));
    constexpr bool WIDE = MODE != Mode::kScalar;
    using U = Unit<T, WIDE>;
    using L = Layout<T, MODE>;
    constexpr int VEC = U::kN;
    using AuxV = typename Op::template Aux<VEC>;
    constexpr int NT = kClusterThreads;
    constexpr int NW = NT / 32;
    __shared__ float red[2][NW];
    __shared__ float part[2][kMaxCluster];  // part[p][q]: block q's partial of this row
    __shared__ __align__(8) unsigned long long xbar[2];
    const int tid = threadIdx.x;
    const int rank = (int)cluster_ctarank();
    const int64_t nclusters = gridDim.x / csize;
    const int64_t u0 = (int64_t)rank * slice;
    AuxV aux[KV];
    if constexpr (MODE == Mode::kAligned) {
        const L lay(A, N);
        const int64_t u1 = (u0 + slice < lay.nv) ? u0 + slice : lay.nv;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int64_t idx = u0 + tid + NT * k;
            if (idx < u1) aux[k] = op.template load_aux<VEC>(lay.unit_col(idx));
        }
    }
    if (tid == 0) {
        mbar_init(smem_addr(&xbar[0]), 1);
        mbar_init(smem_addr(&xbar[1]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    // A block may send to a peer only once the peer runs and its barriers are
    // initialised; the first row's loads overlap this start-up barrier.
    cluster_arrive_relaxed();
    bool started = false, failed = false;
    uint32_t fail_bar = 0, fail_phase = 0;
    int parity = 0;
    int64_t it = 0;
    for (int64_t r = blockIdx.x / csize; r < M; r += nclusters, ++it) {
        const T* ra = A + r * lda;
        const T* rb = B + r * ldb;
        const L lay(ra, N);
        const int64_t u1 = (u0 + slice < lay.nv) ? u0 + slice : lay.nv;
        U a[KV], b[KV];
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int64_t idx = u0 + tid + NT * k;
            if (idx < u1) {
                a[k].load(ra + lay.unit_col(idx));
                b[k].load(rb + lay.unit_col(idx));
                if constexpr (MODE != Mode::kAligned)
                    aux[k] = op.template load_aux<VEC>(lay.unit_col(idx));
            } else {
                a[k].zero();
                b[k].zero();
            }
        }
        Extra<Op, T> ex;
        if constexpr (MODE == Mode::kShifted)
            if (rank == 0 && tid < lay.extra) ex.load(op, ra, rb, lay.extra_col(tid));
        float acc[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
#pragma unroll
        for (int k = 0; k < KV; ++k) accumulate_unit<Op, T, WIDE>(op, a[k], b[k], acc);
        if constexpr (MODE == Mode::kShifted) ex.accumulate(op, acc);
        const float mine = team_sum<NW>(fold<VEC>(acc), red[parity], 0);
        if (!started) {
            cluster_wait();
            started = true;
        }
        const uint32_t xb = smem_addr(&xbar[parity]);
        const uint32_t phase = (uint32_t)((it >> 1) & 1);
        if (tid == 0) mbar_expect_tx(xb, (uint32_t)csize * 4u);
        if (tid < csize && !(flags & kFlagNoCopy))  // the test hook sends nothing
            st_async_f32(map_to_rank(smem_addr(&part[parity][rank]), (uint32_t)tid), mine,
                         map_to_rank(xb, (uint32_t)tid));
        if (!failed && !mbar_wait_bounded(xb, phase, timeout_ns)) {
            failed = true;
            fail_bar = xb;
            fail_phase = phase;
        }
        if (failed) {  // no output; keep sending, so peers do not wait in vain
            parity ^= 1;
            continue;
        }
        float total = part[parity][0];
        for (int q = 1; q < csize; ++q) total += part[parity][q];
        const float s = op.finish(total, N);
        parity ^= 1;
        T* rc = C + r * ldc;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int64_t idx = u0 + tid + NT * k;
            if (idx < u1) write_unit<Op, T, WIDE>(op, a[k], b[k], s, aux[k], rc + lay.unit_col(idx));
        }
        if constexpr (MODE == Mode::kShifted) ex.write(op, s, rc);
    }
    if (!started) cluster_wait();
    if (failed) {
        if (tid == 0) atomicOr(err, 1u);
        mbar_wait_bounded(fail_bar, fail_phase, timeout_ns);
    }
}

// ---------------------------------------------------------------------------
// Streamed CLUSTER plan, for aligned rows too wide for a cluster's registers:
// each block reduces its slice in steps of kStreamUnroll units per thread,
// exchanges the partial as cluster_kernel does, then reads the slice again to
// write. Pass 1 reads with an L2 evict-last policy and pass 2 with
// evict-first, so the resident clusters' slices stay in L2 between the passes
// (cache hints only; the results do not depend on them).
// ---------------------------------------------------------------------------
#ifndef SR_PAIR_STREAM_UNROLL
#define SR_PAIR_STREAM_UNROLL 2
#endif
constexpr int kStreamUnroll = SR_PAIR_STREAM_UNROLL;

__device__ __forceinline__ uint64_t l2_policy(bool keep) {
    uint64_t pol;
    if (keep)
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    else
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint4 ldg_policy(const void* p, uint64_t pol) {
    if (!SR_READ_OK(p, 16)) return make_uint4(0x7fc00000u, 0x7fc00000u, 0x7fc00000u, 0x7fc00000u);
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "l"(pol));
    return v;
}

template <class Op, typename T>
__global__ void __launch_bounds__(kClusterThreads, kStreamMinBlocks)
    stream_kernel(Op op, const T* __restrict__ A, const T* __restrict__ B, T* __restrict__ C,
                  int64_t M, int64_t N, int64_t lda, int64_t ldb, int64_t ldc, int csize,
                  int64_t slice, unsigned int* err, unsigned long long timeout_ns, int flags) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(A, M, lda, N), SR_MAT_IN(B, M, ldb, N), SR_MAT_OUT(C, M, ldc, N),
                    SR_SPAN_IN(op.aux_base(), N * (int64_t)sizeof(T)));
    using U = Unit<T, true>;
    constexpr int VEC = U::kN;
    using AuxV = typename Op::template Aux<VEC>;
    constexpr int NT = kClusterThreads;
    constexpr int NW = NT / 32;
    constexpr int UR = kStreamUnroll;
    __shared__ float red[2][NW];
    __shared__ float part[2][kMaxCluster];
    __shared__ __align__(8) unsigned long long xbar[2];
    const int tid = threadIdx.x;
    const int rank = (int)cluster_ctarank();
    const int64_t nclusters = gridDim.x / csize;
    const int64_t nv = N / VEC;
    const int64_t u0 = (int64_t)rank * slice;
    const int64_t u1 = (u0 + slice < nv) ? u0 + slice : nv;
    const uint64_t keep = l2_policy(true), drop = l2_policy(false);
    if (tid == 0) {
        mbar_init(smem_addr(&xbar[0]), 1);
        mbar_init(smem_addr(&xbar[1]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    cluster_arrive_relaxed();
    bool started = false, failed = false;
    uint32_t fail_bar = 0, fail_phase = 0;
    int parity = 0;
    int64_t it = 0;
    for (int64_t r = blockIdx.x / csize; r < M; r += nclusters, ++it) {
        const T* ra = A + r * lda;
        const T* rb = B + r * ldb;
        float acc[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
        for (int64_t j0 = u0 + tid; j0 < u1; j0 += (int64_t)NT * UR) {
            const int64_t rem = u1 - j0;
            U a[UR], b[UR];
#pragma unroll
            for (int j = 0; j < UR; ++j) {
                if (NT * j < rem) {
                    a[j].raw = ldg_policy(ra + (j0 + NT * j) * VEC, keep);
                    b[j].raw = ldg_policy(rb + (j0 + NT * j) * VEC, keep);
                } else {
                    a[j].zero();
                    b[j].zero();
                }
            }
#pragma unroll
            for (int j = 0; j < UR; ++j) accumulate_unit<Op, T, true>(op, a[j], b[j], acc);
        }
        const float mine = team_sum<NW>(fold<VEC>(acc), red[parity], 0);
        if (!started) {
            cluster_wait();
            started = true;
        }
        const uint32_t xb = smem_addr(&xbar[parity]);
        const uint32_t phase = (uint32_t)((it >> 1) & 1);
        if (tid == 0) mbar_expect_tx(xb, (uint32_t)csize * 4u);
        if (tid < csize && !(flags & kFlagNoCopy))  // the test hook sends nothing
            st_async_f32(map_to_rank(smem_addr(&part[parity][rank]), (uint32_t)tid), mine,
                         map_to_rank(xb, (uint32_t)tid));
        if (!failed && !mbar_wait_bounded(xb, phase, timeout_ns)) {
            failed = true;
            fail_bar = xb;
            fail_phase = phase;
        }
        if (failed) {  // no output; keep sending, so peers do not wait in vain
            parity ^= 1;
            continue;
        }
        float total = part[parity][0];
        for (int q = 1; q < csize; ++q) total += part[parity][q];
        const float s = op.finish(total, N);
        parity ^= 1;
        T* rc = C + r * ldc;
        for (int64_t j0 = u0 + tid; j0 < u1; j0 += (int64_t)NT * UR) {
            const int64_t rem = u1 - j0;
            U a[UR], b[UR];
            AuxV aux[UR];
#pragma unroll
            for (int j = 0; j < UR; ++j) {
                if (NT * j < rem) {
                    const int64_t idx = j0 + NT * j;
                    a[j].raw = ldg_policy(ra + idx * VEC, drop);
                    b[j].raw = ldg_policy(rb + idx * VEC, drop);
                    aux[j] = op.template load_aux<VEC>(idx * VEC);
                }
            }
#pragma unroll
            for (int j = 0; j < UR; ++j)
                if (NT * j < rem)
                    write_unit<Op, T, true>(op, a[j], b[j], s, aux[j], rc + (j0 + NT * j) * VEC);
        }
    }
    if (!started) cluster_wait();
    if (failed) {
        if (tid == 0) atomicOr(err, 1u);
        mbar_wait_bounded(fail_bar, fail_phase, timeout_ns);
    }
}

// ---------------------------------------------------------------------------
// ONLINE plan: one block per row, two passes.
// ---------------------------------------------------------------------------
template <class Op, typename T, Mode MODE>
__global__ void __launch_bounds__(kLoopThreads)
    loop_kernel(Op op, const T* __restrict__ A, const T* __restrict__ B, T* __restrict__ C,
                int64_t M, int64_t N, int64_t lda, int64_t ldb, int64_t ldc) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(A, M, lda, N), SR_MAT_IN(B, M, ldb, N), SR_MAT_OUT(C, M, ldc, N),
                    SR_SPAN_IN(op.aux_base(), N * (int64_t)sizeof(T)));
    constexpr bool WIDE = MODE != Mode::kScalar;
    using U = Unit<T, WIDE>;
    using L = Layout<T, MODE>;
    constexpr int VEC = U::kN;
    using AuxV = typename Op::template Aux<VEC>;
    constexpr int NT = kLoopThreads;
    constexpr int NW = NT / 32;
    constexpr int UR = kLoopUnroll;
    __shared__ float red[2][NW];
    const int tid = threadIdx.x;
    int parity = 0;
    for (int64_t r = blockIdx.x; r < M; r += gridDim.x) {
        const T* ra = A + r * lda;
        const T* rb = B + r * ldb;
        const L lay(ra, N);
        float acc[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
        for (int64_t base = 0; base < lay.nv; base += (int64_t)NT * UR) {
            U a[UR], b[UR];
#pragma unroll
            for (int j = 0; j < UR; ++j) {
                const int64_t idx = base + tid + NT * j;
                if (idx < lay.nv) {
                    a[j].load(ra + lay.unit_col(idx));
                    b[j].load(rb + lay.unit_col(idx));
                } else {
                    a[j].zero();
                    b[j].zero();
                }
            }
#pragma unroll
            for (int j = 0; j < UR; ++j) accumulate_unit<Op, T, WIDE>(op, a[j], b[j], acc);
        }
        Extra<Op, T> ex;
        if constexpr (MODE == Mode::kShifted)
            if (tid < lay.extra) ex.load(op, ra, rb, lay.extra_col(tid));
        if constexpr (MODE == Mode::kShifted) ex.accumulate(op, acc);
        const float s = op.finish(team_sum<NW>(fold<VEC>(acc), red[parity], 0), N);
        parity ^= 1;
        T* rc = C + r * ldc;
        for (int64_t base = 0; base < lay.nv; base += (int64_t)NT * UR) {
            U a[UR], b[UR];
            AuxV aux[UR];
#pragma unroll
            for (int j = 0; j < UR; ++j) {
                const int64_t idx = base + tid + NT * j;
                if (idx < lay.nv) {
                    a[j].load(ra + lay.unit_col(idx));
                    b[j].load(rb + lay.unit_col(idx));
                    aux[j] = op.template load_aux<VEC>(lay.unit_col(idx));
                }
            }
#pragma unroll
            for (int j = 0; j < UR; ++j) {
                const int64_t idx = base + tid + NT * j;
                if (idx < lay.nv)
                    write_unit<Op, T, WIDE>(op, a[j], b[j], s, aux[j], rc + lay.unit_col(idx));
            }
        }
        if constexpr (MODE == Mode::kShifted) ex.write(op, s, rc);
    }
}

// One block (or cluster) per row up to the largest grid; more rows are
// walked with a grid stride.
inline unsigned grid_for(int64_t rows, int64_t blocks_per_unit) {
    const int64_t cap = 0x7fffffff / blocks_per_unit;
    return (unsigned)((rows < cap ? rows : cap) * blocks_per_unit);
}

template <class Op, typename T, Mode MODE, int TPR, int KV>
cudaError_t launch_team_kv(const Op& op, const Args& p) {
    constexpr int NT = TPR < 128 ? 128 : TPR;
    constexpr int RPB = NT / TPR;
    const unsigned grid = grid_for((p.M + RPB - 1) / RPB, 1);
    const T* a = static_cast<const T*>(p.a);
    const T* b = static_cast<const T*>(p.b);
    T* c = static_cast<T*>(p.c);
    const LaunchShape ls{dim3(grid), dim3(NT)};
    if constexpr (team_bounded<Op, T>())
        return launch_kernel(team_kernel_bounded<Op, T, MODE, TPR, KV>, ls, p.stream, op, a, b, c,
                             p.M, p.N, p.lda, p.ldb, p.ldc);
    else
        return launch_kernel(team_kernel<Op, T, MODE, TPR, KV>, ls, p.stream, op, a, b, c, p.M,
                             p.N, p.lda, p.ldb, p.ldc);
}

template <class Op, typename T, Mode MODE, int TPR>
cudaError_t launch_team_tpr(const Op& op, const Args& p, int kv) {
    constexpr int KT = KvTarget<T, MODE>::kTarget;
    constexpr int KM = KvTarget<T, MODE>::kMax;
    if constexpr (TPR == 32) {
        if (kv == 1) return launch_team_kv<Op, T, MODE, TPR, 1>(op, p);
        if (kv == 2) return launch_team_kv<Op, T, MODE, TPR, 2>(op, p);
        if (kv == 4) return launch_team_kv<Op, T, MODE, TPR, 4>(op, p);
        if constexpr (KT > 4) if (kv == KT) return launch_team_kv<Op, T, MODE, TPR, KT>(op, p);
    } else {
        if (kv == KT) return launch_team_kv<Op, T, MODE, TPR, KT>(op, p);
        if constexpr (TPR == kTeamMaxThreads && KM > KT)
            if (kv == KM) return launch_team_kv<Op, T, MODE, TPR, KM>(op, p);
    }
    return cudaErrorInvalidValue;
}

template <class Op, typename T, Mode MODE>
cudaError_t launch_team(const Op& op, const Args& p, const Shape& sh) {
    switch (sh.tpr) {
        case 32: return launch_team_tpr<Op, T, MODE, 32>(op, p, sh.kv);
        case 64: return launch_team_tpr<Op, T, MODE, 64>(op, p, sh.kv);
        case 128: return launch_team_tpr<Op, T, MODE, 128>(op, p, sh.kv);
        case 256: return launch_team_tpr<Op, T, MODE, 256>(op, p, sh.kv);
        case 512: return launch_team_tpr<Op, T, MODE, 512>(op, p, sh.kv);
    }
    return cudaErrorInvalidValue;
}

template <class Op, typename T>
using ClusterKernel = void (*)(Op, const T*, const T*, T*, int64_t, int64_t, int64_t, int64_t,
                               int64_t, int, int64_t, unsigned int*, unsigned long long, int);

template <class Op, typename T>
cudaError_t launch_clusters(ClusterKernel<Op, T> kern, const Op& op, const Args& p,
                            const Shape& sh) {
    const void* fn = reinterpret_cast<const void*>(kern);
    cudaError_t e = ensure_smem_limit(fn, 0, sh.csize > 8);
    if (e != cudaSuccess) return e;
    if (max_active_clusters(fn, kClusterThreads, 0, sh.csize) <= 0)
        return cudaErrorInvalidConfiguration;
    return launch_kernel(kern,
                         LaunchShape{dim3(grid_for(p.M, sh.csize)), dim3(kClusterThreads), 0,
                                     sh.csize},
                         p.stream, op, static_cast<const T*>(p.a), static_cast<const T*>(p.b),
                         static_cast<T*>(p.c), p.M, p.N, p.lda, p.ldb, p.ldc, sh.csize, sh.slice,
                         p.err, p.timeout_ns, p.flags);
}

template <class Op, typename T, Mode MODE>
cudaError_t launch_cluster(const Op& op, const Args& p, const Shape& sh) {
    constexpr int KM = KvTarget<T, MODE>::kMax;
    if (sh.streamed) {
        if constexpr (MODE == Mode::kAligned)
            return launch_clusters<Op, T>(stream_kernel<Op, T>, op, p, sh);
        return cudaErrorInvalidValue;
    }
    if (sh.kv == 1) return launch_clusters<Op, T>(cluster_kernel<Op, T, MODE, 1>, op, p, sh);
    if (sh.kv == 2) return launch_clusters<Op, T>(cluster_kernel<Op, T, MODE, 2>, op, p, sh);
    if (sh.kv == 4) return launch_clusters<Op, T>(cluster_kernel<Op, T, MODE, 4>, op, p, sh);
    if constexpr (KM >= 8)
        if (sh.kv == 8) return launch_clusters<Op, T>(cluster_kernel<Op, T, MODE, 8>, op, p, sh);
    if constexpr (KM >= 16)
        if (sh.kv == 16) return launch_clusters<Op, T>(cluster_kernel<Op, T, MODE, 16>, op, p, sh);
    return cudaErrorInvalidValue;
}

template <class Op, typename T, Mode MODE>
cudaError_t launch_mode(const Op& op, const Args& p, const Shape& sh) {
    switch (sh.plan) {
        case SR_PLAN_ROW: return launch_team<Op, T, MODE>(op, p, sh);
        case SR_PLAN_CLUSTER: return launch_cluster<Op, T, MODE>(op, p, sh);
        case SR_PLAN_ONLINE:
            return launch_kernel(loop_kernel<Op, T, MODE>,
                                 LaunchShape{dim3(grid_for(p.M, 1)), dim3(kLoopThreads)}, p.stream,
                                 op, static_cast<const T*>(p.a), static_cast<const T*>(p.b),
                                 static_cast<T*>(p.c), p.M, p.N, p.lda, p.ldb, p.ldc);
    }
    return cudaErrorInvalidValue;
}

// Launch `sh` with the Op the factory makes for element type T.
template <typename T, class Op>
cudaError_t launch(const Op& op, const Args& p, const Shape& sh) {
    switch (sh.mode) {
        case (int)Mode::kAligned: return launch_mode<Op, T, Mode::kAligned>(op, p, sh);
        case (int)Mode::kShifted: return launch_mode<Op, T, Mode::kShifted>(op, p, sh);
        case (int)Mode::kScalar: return launch_mode<Op, T, Mode::kScalar>(op, p, sh);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rp
}  // namespace sr
