// WIDE plan: a row cut into slices held in the registers of the blocks of a
// thread-block cluster, one row per cluster.
//
// The split plan of "Measured optimization case studies" (Wide rows) kept on
// chip, as the CLUSTER plan does, with a different schedule. Each of the C
// blocks of a cluster loads its slice of the row straight into registers as
// packed 16-byte vectors (2 bytes per element on chip for 16-bit data), every
// warp reduces its part to an online (max, sum) pair with the all -inf guard
// of the same section, and sends the pair to every block of the cluster with
// st.async: the store lands in the receiver's shared memory and completes
// transaction bytes on the receiver's mbarrier, so no cluster barrier and no
// release fence sit in the row. Each block waits (bounded) for the C x 8
// pairs, every warp merges them in the same order into the row's (M, S), and
// exponentiates its values again against M for the output. Keeping the inputs
// instead of FP32 exponentials halves the on-chip bytes per element; the
// price is a second exponential per element (the result is still rounded
// once, from FP32). The grid has one cluster per row, so the hardware starts
// a new cluster as soon as one finishes.
//
// Aligned rows too wide for the cluster's registers (over 512 KiB) take a
// streamed variant that reads each slice twice instead (wide_bulk_kernel on
// 8-block clusters, its loads by the bulk-copy engine; wide_stream_kernel on
// 16-block clusters).
//
// Failure: a wait that expires marks the block failed; it writes nothing
// more, records the failure in the error word and, before leaving, waits once
// more (bounded) so that a late peer's pair cannot land after it exits.
#include "device.cuh"
#include "internal.h"
#include "l2prefetch.cuh"
#include "packed.cuh"
#include "wide.h"

namespace sr {
namespace {

// Cluster scheduling policy of the launch (a cudaClusterSchedulingPolicy).
#ifndef SR_WIDE_POLICY
#define SR_WIDE_POLICY 2
#endif

// Resident blocks per SM the kernel is compiled for (bounds its registers).
#ifndef SR_WIDE_MIN_BLOCKS
#define SR_WIDE_MIN_BLOCKS 4
#endif

// 1: aligned rows of exactly 1 MiB (65536 vectors) run the staged variant
// (half of each slice in shared memory; wide_staged_kernel) instead of being
// streamed. Measured on GB300 (cold L2), µs, staged against streamed: bf16
// 128 x 524288 48.3 / 56.7, 256 x 524288 86.0 / 113.7, f32 256 x 262144
// 85.4 / 115.7, 64 x 262144 28.3 / 31.0. Rows between 512 KiB and 1 MiB,
// whose slices do not split evenly, were slower staged (bf16 512 x 400008
// 170.9 / 157.0 streamed), and on rows the registers hold it gained nothing
// (within 1 %).
#ifndef SR_WIDE_STAGED
#define SR_WIDE_STAGED 1
#endif

constexpr int kWideThreads = 256;


// exp(x - m) for FP32 data: the hardware ex2 of the difference (rounded once
// in FP32) times log2(e), as in the ROW plan, instead of the library expf;
// SR_WIDE_EX2 = 0 keeps expf. 16-bit data always takes one FMA and ex2.
#ifndef SR_WIDE_EX2
#define SR_WIDE_EX2 1
#endif
template <typename T>
__device__ __forceinline__ float wide_exp(float x, float m, float m_l2) {
    if constexpr (Elem<T>::kAccurateExp && SR_WIDE_EX2) {
        return ex2_approx((x - m) * kLog2e);
    } else {
        return exp_shifted<T>(x, m, m_l2);
    }
}
constexpr int kWideWarps = kWideThreads / 32;

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Row layouts: kAligned, every row of both matrices on a 16-byte boundary
// and whole vectors (kFull when, besides, every block's slice is exactly
// 256 * KV vectors, so no vector needs a bounds check); kShifted, the rows of
// the input and the output share their offset from a 16-byte boundary, so a
// row is a head of fewer than VEC elements, 16-byte vectors and a tail of
// fewer than VEC elements; rank 0's first threads take the head and tail
// elements one each.
enum : int { kAligned = 0, kFull = 1, kShifted = 2 };

// KV: 16-byte vectors per thread; `slice`: vectors per block (<= 256 * KV).
// Slices of 5 or 6 vectors per thread (rows that would half fill 8) get
// their own kernels, compiled for SR_WIDE_MIN_BLOCKS_MID blocks per SM, so
// that more row bytes are resident per SM. Measured on GB300 (cold L2):
// bf16 4096 x 16392 57.1 -> 51.2 µs, f32 3000 x 20000 86.2 -> 76.9 µs,
// f16 2730 x 24576 46.8 -> 43.4 µs.
#ifndef SR_WIDE_MID_KV
#define SR_WIDE_MID_KV 1
#endif
#ifndef SR_WIDE_MIN_BLOCKS_MID
#define SR_WIDE_MIN_BLOCKS_MID 5
#endif
template <typename T, int KV, int MODE>
__global__ void __launch_bounds__(kWideThreads, (KV == 5 || KV == 6) ? SR_WIDE_MIN_BLOCKS_MID
                                                                     : SR_WIDE_MIN_BLOCKS)
    wide_rows_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int64_t N,
                     int64_t ld_in, int64_t ld_out, int csize, int64_t slice, unsigned int* err,
                     unsigned long long timeout_ns, int flags, int64_t ahead) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, M, ld_in, N), SR_MAT_OUT(out, M, ld_out, N));
    constexpr int VEC = Elem<T>::kVec;
    constexpr int NT = kWideThreads;
    constexpr int NW = kWideWarps;
    constexpr bool FULL = MODE == kFull;
    constexpr bool SHIFTED = MODE == kShifted;
    // pairs[p][q * NW + w]: warp w of block q for rows of parity p (a cluster
    // walks more than one row only when the grid is capped), and the two
    // exchange barriers they complete on.
    __shared__ float2 pairs[2][kMaxCluster * NW];
    __shared__ __align__(8) unsigned long long xbar[2];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)cluster_ctarank();
    const int64_t nclusters = gridDim.x / csize;
    const int64_t nvec = N / VEC;
    const int64_t u0 = (int64_t)rank * slice;
    const int npairs = csize * NW;
    const bool send = !(flags & kFlagNoCopy);  // test hook: send nothing, every wait expires

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
    int64_t it = 0;
    for (int64_t r = blockIdx.x / csize; r < M; r += nclusters, ++it) {
        const int p = (int)(it & 1);
        const uint32_t phase = (uint32_t)((it >> 1) & 1);
        const T* rin = in + r * ld_in;
        // The row's vectors start `head` elements in; `nvb` of them, then
        // `extra` = head + tail single elements.
        int head = 0, extra = 0;
        int64_t nvb = nvec;
        if constexpr (SHIFTED) {
            const int off = (int)((reinterpret_cast<uintptr_t>(rin) & 15u) / sizeof(T));
            head = off ? VEC - off : 0;
            if (head > N) head = (int)N;
            nvb = (N - head) / VEC;
            extra = (int)(N - nvb * VEC);
        }
        const T* rbody = rin + head;
        const int64_t u1 = (u0 + slice < nvb) ? u0 + slice : nvb;
        // The row `ahead` rows on (the one a cluster starts about one wave of
        // resident clusters later) is prefetched into L2 by the bulk-copy
        // engine, so that its blocks load from L2 and hold their registers
        // for less time; DRAM streams it in the background meanwhile.
        if constexpr (!SHIFTED) {
            if (tid == 0 && ahead > 0 && r + ahead < M && u1 > u0)
                bulk_prefetch_l2(in + (r + ahead) * ld_in + u0 * VEC, (uint32_t)((u1 - u0) * 16));
        }
        uint4 raw[KV];
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int64_t idx = u0 + tid + NT * k;
            if (FULL || idx < u1) raw[k] = ldg_stream(rbody + idx * VEC);
        }
        float xe = neg_inf();  // this thread's head or tail element, if any
        int64_t ce = -1;
        if constexpr (SHIFTED) {
            if (rank == 0 && tid < extra) {
                ce = tid < head ? tid : head + nvb * VEC + (tid - head);
                xe = Elem<T>::load1(rin + ce);
            }
        }
        // Warp partial (m_w, s_w): max, then sum of exp(x - m_w).
        VecMax<T> vm;
#pragma unroll
        for (int k = 0; k < KV; ++k)
            if (FULL || u0 + tid + NT * k < u1) vm.add(raw[k]);
        const float m_w = warp_max(fmaxf(vm.get(), xe));
        const float shift = (m_w == neg_inf()) ? 0.0f : m_w;
        const float shift_l2 = shift * kLog2e;
        float sa = 0.0f, sb = 0.0f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            if (FULL || u0 + tid + NT * k < u1) {
                float f[VEC];
                Elem<T>::unpack(raw[k], f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float x = wide_exp<T>(f[e], shift, shift_l2);
                    if (e & 1) sb += x; else sa += x;
                }
            }
        }
        if (SHIFTED && ce >= 0) sa += wide_exp<T>(xe, shift, shift_l2);
        const float s_w = warp_sum(sa + sb);
        if (!started) {
            cluster_wait();
            started = true;
        }
        const uint32_t xb = smem_addr(&xbar[p]);
        if (tid == 0) mbar_expect_tx(xb, (uint32_t)npairs * 8u);
        if (send && lane < csize)
            st_async_f2(map_to_rank(smem_addr(&pairs[p][rank * NW + warp]), (uint32_t)lane), m_w,
                        s_w, map_to_rank(xb, (uint32_t)lane));
        if (!failed && !mbar_wait_bounded(xb, phase, timeout_ns)) {
            failed = true;
            fail_bar = xb;
            fail_phase = phase;
        }
        if (failed) continue;  // no output; keep sending, so peers do not wait in vain
        // The row's (M, S): the same merge, in the same order, in every warp.
        float mloc = neg_inf();
        for (int i = lane; i < npairs; i += 32) mloc = fmaxf(mloc, pairs[p][i].x);
        const float Mr = warp_max(mloc);
        float sloc = 0.0f;
        for (int i = lane; i < npairs; i += 32) {
            const float2 q = pairs[p][i];
            sloc += q.y * merge_scale(q.x, Mr);
        }
        const float Sr = warp_sum(sloc);
        T* rout = out + r * ld_out;
        T* obody = rout + head;
        if constexpr (Elem<T>::kAccurateExp) {
            // FP32 data: exp of the exact difference, times the rounded 1/S.
            const float rs = final_rcp(Mr, Sr);
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int64_t idx = u0 + tid + NT * k;
                if (FULL || idx < u1) {
                    float f[VEC];
                    unpack_again<T>(raw[k], f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) f[e] = wide_exp<T>(f[e], Mr, 0.0f) * rs;
                    stg_stream(obody + idx * VEC, Elem<T>::pack(f));
                }
            }
            if (SHIFTED && ce >= 0) Elem<T>::store1(rout + ce, wide_exp<T>(xe, Mr, 0.0f) * rs);
        } else {
            // 16-bit data: 1/S folded into the exponent,
            // y = 2^(x log2(e) - (M log2(e) + log2(S))), one FMA and one ex2 per
            // element. An all -inf row gives -inf - -inf = NaN, as 0/0 does.
            const float c = fmaf(Mr, kLog2e, lg2_approx(Sr));
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int64_t idx = u0 + tid + NT * k;
                if (FULL || idx < u1) {
                    float f[VEC];
                    unpack_again<T>(raw[k], f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) f[e] = ex2_approx(fmaf(f[e], kLog2e, -c));
                    stg_stream(obody + idx * VEC, Elem<T>::pack(f));
                }
            }
            if (SHIFTED && ce >= 0) Elem<T>::store1(rout + ce, ex2_approx(fmaf(xe, kLog2e, -c)));
        }
    }
    if (!started) cluster_wait();
    if (failed) {
        if (tid == 0) atomicOr(err, 1u);
        // A late peer may still send its pair into this block's shared memory:
        // wait once more (bounded) before leaving.
        mbar_wait_bounded(fail_bar, fail_phase, timeout_ns);
    }
}

// Staged variant for aligned 1 MiB rows (16 slices of 4096 vectors), twice
// what a 16-block cluster's registers hold: each thread holds 8 vectors of its
// block's slice in registers and 8 more in shared memory, brought in by
// 16-byte cp.async copies that occupy no registers while in flight (each
// thread reads back only its own slots, so no block barrier is needed). Such
// rows stay on chip and are read from DRAM once instead of being streamed
// twice. Arithmetic, exchange, prefetch and failure path as in
// wide_rows_kernel (kFull).
constexpr int kStagedKV = 8;
constexpr int kStagedKS = 8;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    if (!SR_READ_OK(src, 16)) return;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

#ifndef SR_WIDE_STAGED_MIN_BLOCKS
#define SR_WIDE_STAGED_MIN_BLOCKS 3
#endif
template <typename T>
__global__ void __launch_bounds__(kWideThreads, SR_WIDE_STAGED_MIN_BLOCKS)
    wide_staged_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int64_t N,
                       int64_t ld_in, int64_t ld_out, int csize, int64_t slice,
                       unsigned int* err, unsigned long long timeout_ns, int flags,
                       int64_t ahead) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, M, ld_in, N), SR_MAT_OUT(out, M, ld_out, N));
    constexpr int VEC = Elem<T>::kVec;
    constexpr int NT = kWideThreads;
    constexpr int NW = kWideWarps;
    constexpr int KV = kStagedKV;
    constexpr int KS = kStagedKS;
    extern __shared__ __align__(128) unsigned char stage_buf[];  // slot k*NT + tid: 16 bytes
    __shared__ float2 pairs[2][kMaxCluster * NW];
    __shared__ __align__(8) unsigned long long xbar[2];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)cluster_ctarank();
    const int64_t nclusters = gridDim.x / csize;
    const int64_t u0 = (int64_t)rank * slice;
    const int npairs = csize * NW;
    const bool send = !(flags & kFlagNoCopy);
    const uint32_t stage = smem_addr(stage_buf) + 16u * (uint32_t)tid;

    if (tid == 0) {
        mbar_init(smem_addr(&xbar[0]), 1);
        mbar_init(smem_addr(&xbar[1]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    cluster_arrive_relaxed();
    bool started = false, failed = false;
    uint32_t fail_bar = 0, fail_phase = 0;
    int64_t it = 0;
    for (int64_t r = blockIdx.x / csize; r < M; r += nclusters, ++it) {
        const int p = (int)(it & 1);
        const uint32_t phase = (uint32_t)((it >> 1) & 1);
        const T* rin = in + r * ld_in + u0 * VEC;
        if (tid == 0 && ahead > 0 && r + ahead < M)
            bulk_prefetch_l2(in + (r + ahead) * ld_in + u0 * VEC, (uint32_t)(slice * 16));
        // Vectors NT*KV + tid + NT*k of the slice go to this thread's staging
        // slots, vectors tid + NT*k to its registers.
#pragma unroll
        for (int k = 0; k < KS; ++k)
            cp_async16(stage + 16u * (uint32_t)(NT * k), rin + (int64_t)(NT * KV + tid + NT * k) * VEC);
        asm volatile("cp.async.commit_group;" ::: "memory");
        uint4 raw[KV];
#pragma unroll
        for (int k = 0; k < KV; ++k) raw[k] = ldg_stream(rin + (int64_t)(tid + NT * k) * VEC);
        VecMax<T> vm;
#pragma unroll
        for (int k = 0; k < KV; ++k) vm.add(raw[k]);
        asm volatile("cp.async.wait_group 0;" ::: "memory");
#pragma unroll
        for (int k = 0; k < KS; ++k) vm.add(lds128(stage + 16u * (uint32_t)(NT * k)));
        const float m_w = warp_max(vm.get());
        const float shift = (m_w == neg_inf()) ? 0.0f : m_w;
        const float shift_l2 = shift * kLog2e;
        float sa = 0.0f, sb = 0.0f;
        auto add_exp = [&](const uint4& u) {
            float f[VEC];
            Elem<T>::unpack(u, f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float x = wide_exp<T>(f[e], shift, shift_l2);
                if (e & 1) sb += x; else sa += x;
            }
        };
#pragma unroll
        for (int k = 0; k < KV; ++k) add_exp(raw[k]);
#pragma unroll
        for (int k = 0; k < KS; ++k) add_exp(lds128(stage + 16u * (uint32_t)(NT * k)));
        const float s_w = warp_sum(sa + sb);
        if (!started) {
            cluster_wait();
            started = true;
        }
        const uint32_t xb = smem_addr(&xbar[p]);
        if (tid == 0) mbar_expect_tx(xb, (uint32_t)npairs * 8u);
        if (send && lane < csize)
            st_async_f2(map_to_rank(smem_addr(&pairs[p][rank * NW + warp]), (uint32_t)lane), m_w,
                        s_w, map_to_rank(xb, (uint32_t)lane));
        if (!failed && !mbar_wait_bounded(xb, phase, timeout_ns)) {
            failed = true;
            fail_bar = xb;
            fail_phase = phase;
        }
        if (failed) continue;
        float mloc = neg_inf();
        for (int i = lane; i < npairs; i += 32) mloc = fmaxf(mloc, pairs[p][i].x);
        const float Mr = warp_max(mloc);
        float sloc = 0.0f;
        for (int i = lane; i < npairs; i += 32) {
            const float2 q = pairs[p][i];
            sloc += q.y * merge_scale(q.x, Mr);
        }
        const float Sr = warp_sum(sloc);
        T* rout = out + r * ld_out + u0 * VEC;
        const float rs = Elem<T>::kAccurateExp ? final_rcp(Mr, Sr) : 0.0f;
        const float c = Elem<T>::kAccurateExp ? 0.0f : fmaf(Mr, kLog2e, lg2_approx(Sr));
        auto put = [&](const uint4& u, int64_t idx) {
            float f[VEC];
            unpack_again<T>(u, f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                if constexpr (Elem<T>::kAccurateExp)
                    f[e] = wide_exp<T>(f[e], Mr, 0.0f) * rs;
                else
                    f[e] = ex2_approx(fmaf(f[e], kLog2e, -c));
            }
            stg_stream(rout + idx * VEC, Elem<T>::pack(f));
        };
#pragma unroll
        for (int k = 0; k < KV; ++k) put(raw[k], tid + NT * k);
#pragma unroll
        for (int k = 0; k < KS; ++k) put(lds128(stage + 16u * (uint32_t)(NT * k)), NT * KV + tid + NT * k);
    }
    if (!started) cluster_wait();
    if (failed) {
        if (tid == 0) atomicOr(err, 1u);
        mbar_wait_bounded(fail_bar, fail_phase, timeout_ns);
    }
}

// Streamed variant for aligned rows too wide for the registers of a 16-block
// cluster (over 512 KiB): the looped plan of the same section (Wide rows),
// spread over a cluster. Pass 1 walks the block's slice in steps of
// kStreamChunk vectors per thread, keeping a per-thread online (max, sum):
// the step's maximum is taken in the storage format, the sum is rescaled when
// the maximum grows, and a thread whose values so far are all -inf shifts by 0
// and keeps a zero sum. The lanes' pairs merge into one pair per warp with
// the same rule, and the warp pairs are exchanged and merged exactly as in
// wide_rows_kernel. Pass 2 reads the slice again and writes the output. The
// resident clusters' rows were read moments before and fit in L2, so HBM sees
// about one read per element.
#ifndef SR_WIDE_STREAM_CHUNK
#define SR_WIDE_STREAM_CHUNK 4
#endif
#ifndef SR_WIDE_STREAM_MIN_BLOCKS
#define SR_WIDE_STREAM_MIN_BLOCKS 4
#endif
constexpr int kStreamChunk = SR_WIDE_STREAM_CHUNK;
// 1: pass 1 marks the lines it reads for late eviction from L2 and pass 2
// marks them for early eviction, so that the slices stay in L2 between the
// two passes (L2 cache-policy hints of ld; no effect on results). Measured on
// GB300, cold L2: bf16 128 x 524288 62.2 -> 54.7 µs, bf16 1024 x 262152
// 249.6 -> 197.8 µs; rows of 4 MiB and more are too wide to stay in L2
// either way.
#ifndef SR_WIDE_STREAM_HINT
#define SR_WIDE_STREAM_HINT 1
#endif
// Blocks per cluster of the streamed variant (8 or 16).
#ifndef SR_WIDE_STREAM_CLUSTER
#define SR_WIDE_STREAM_CLUSTER 8
#endif

__device__ __forceinline__ uint64_t l2_policy_keep() {
    uint64_t pol = 0;
    if (SR_WIDE_STREAM_HINT) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_policy_drop() {
    uint64_t pol = 0;
    if (SR_WIDE_STREAM_HINT) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16-byte load through the read-only path with an L2 cache policy.
__device__ __forceinline__ uint4 ldg_policy(const void* p, uint64_t pol) {
    if (!SR_READ_OK(p, 16)) return make_uint4(0x7fc00000u, 0x7fc00000u, 0x7fc00000u, 0x7fc00000u);
    uint4 v;
    if (SR_WIDE_STREAM_HINT) {
        asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
            : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
            : "l"(p), "l"(pol));
    } else {
        v = ldg_stream(p);
    }
    return v;
}

template <typename T>
__global__ void __launch_bounds__(kWideThreads, SR_WIDE_STREAM_MIN_BLOCKS)
    wide_stream_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int64_t N,
                       int64_t ld_in, int64_t ld_out, int csize, int64_t slice,
                       unsigned int* err, unsigned long long timeout_ns, int flags,
                       int64_t /* ahead: unused */) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, M, ld_in, N), SR_MAT_OUT(out, M, ld_out, N));
    constexpr int VEC = Elem<T>::kVec;
    constexpr int NT = kWideThreads;
    constexpr int NW = kWideWarps;
    constexpr int CH = kStreamChunk;
    __shared__ float2 pairs[2][kMaxCluster * NW];
    __shared__ __align__(8) unsigned long long xbar[2];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)cluster_ctarank();
    const int64_t nclusters = gridDim.x / csize;
    const int64_t nvec = N / VEC;
    const int64_t u0 = (int64_t)rank * slice;
    const int64_t u1 = (u0 + slice < nvec) ? u0 + slice : nvec;
    const int npairs = csize * NW;
    const bool send = !(flags & kFlagNoCopy);  // test hook: send nothing, every wait expires
    const uint64_t keep = l2_policy_keep(), drop = l2_policy_drop();

    if (tid == 0) {
        mbar_init(smem_addr(&xbar[0]), 1);
        mbar_init(smem_addr(&xbar[1]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    cluster_arrive_relaxed();
    bool started = false, failed = false;
    uint32_t fail_bar = 0, fail_phase = 0;
    int64_t it = 0;
    for (int64_t r = blockIdx.x / csize; r < M; r += nclusters, ++it) {
        const int p = (int)(it & 1);
        const uint32_t phase = (uint32_t)((it >> 1) & 1);
        const T* rin = in + r * ld_in;
        // Pass 1: per-thread online (m, s) over vectors u0 + tid + NT * j.
        float m = neg_inf(), s = 0.0f;
        for (int64_t j0 = u0 + tid; j0 < u1; j0 += (int64_t)NT * CH) {
            const T* q = rin + j0 * VEC;
            const int64_t rem = u1 - j0;  // vectors of this thread's step: k < rem / NT
            uint4 raw[CH];
#pragma unroll
            for (int k = 0; k < CH; ++k)
                if (NT * k < rem) raw[k] = ldg_policy(q + NT * k * VEC, keep);
            VecMax<T> vm;
#pragma unroll
            for (int k = 0; k < CH; ++k)
                if (NT * k < rem) vm.add(raw[k]);
            const float mn = fmaxf(m, vm.get());
            const float shift = (mn == neg_inf()) ? 0.0f : mn;
            const float shift_l2 = shift * kLog2e;
            float sa = 0.0f, sb = 0.0f;
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                if (NT * k < rem) {
                    float f[VEC];
                    Elem<T>::unpack(raw[k], f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float x = wide_exp<T>(f[e], shift, shift_l2);
                        if (e & 1) sb += x; else sa += x;
                    }
                }
            }
            s = s * merge_scale(m, mn) + (sa + sb);
            m = mn;
        }
        // One pair per warp (the merge is symmetric, so every lane ends with
        // the same bits).
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
            merge_ms(m, s, m2, s2);
        }
        if (!started) {
            cluster_wait();
            started = true;
        }
        const uint32_t xb = smem_addr(&xbar[p]);
        if (tid == 0) mbar_expect_tx(xb, (uint32_t)npairs * 8u);
        if (send && lane < csize)
            st_async_f2(map_to_rank(smem_addr(&pairs[p][rank * NW + warp]), (uint32_t)lane), m, s,
                        map_to_rank(xb, (uint32_t)lane));
        if (!failed && !mbar_wait_bounded(xb, phase, timeout_ns)) {
            failed = true;
            fail_bar = xb;
            fail_phase = phase;
        }
        if (failed) continue;  // no output; keep sending, so peers do not wait in vain
        float mloc = neg_inf();
        for (int i = lane; i < npairs; i += 32) mloc = fmaxf(mloc, pairs[p][i].x);
        const float Mr = warp_max(mloc);
        float sloc = 0.0f;
        for (int i = lane; i < npairs; i += 32) {
            const float2 q = pairs[p][i];
            sloc += q.y * merge_scale(q.x, Mr);
        }
        const float Sr = warp_sum(sloc);
        // Pass 2: the output, as in wide_rows_kernel.
        T* rout = out + r * ld_out;
        const float rs = Elem<T>::kAccurateExp ? final_rcp(Mr, Sr) : 0.0f;
        const float c = Elem<T>::kAccurateExp ? 0.0f : fmaf(Mr, kLog2e, lg2_approx(Sr));
        for (int64_t j0 = u0 + tid; j0 < u1; j0 += (int64_t)NT * CH) {
            const T* q = rin + j0 * VEC;
            T* o = rout + j0 * VEC;
            const int64_t rem = u1 - j0;
            uint4 raw[CH];
#pragma unroll
            for (int k = 0; k < CH; ++k)
                if (NT * k < rem) raw[k] = ldg_policy(q + NT * k * VEC, drop);
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                if (NT * k < rem) {
                    float f[VEC];
                    Elem<T>::unpack(raw[k], f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        if constexpr (Elem<T>::kAccurateExp)
                            f[e] = wide_exp<T>(f[e], Mr, 0.0f) * rs;
                        else
                            f[e] = ex2_approx(fmaf(f[e], kLog2e, -c));
                    }
                    stg_stream(o + NT * k * VEC, Elem<T>::pack(f));
                }
            }
        }
    }
    if (!started) cluster_wait();
    if (failed) {
        if (tid == 0) atomicOr(err, 1u);
        mbar_wait_bounded(fail_bar, fail_phase, timeout_ns);
    }
}

// Streamed rows with the loads done by the bulk-copy engine (streamed rows on
// 8-block clusters; SR_WIDE_BULK = 0 keeps wide_stream_kernel for all). A producer warp
// (lane 0) walks the block's chunk sequence -- for each of its rows, the
// slice's kWBUnits-vector chunks for pass 1, then the same chunks again for
// pass 2 -- and issues each as a 1-D bulk copy (L2 policy: keep for pass 1,
// drop for pass 2) into a ring of kWBSlots shared-memory slots as soon as the
// slot is free; slot i completes on full[i] (transaction bytes). The eight
// consumer warps take the chunks in the same order, move their units into
// registers, release the slot on empty[i] (one arrival per warp) and compute
// exactly as wide_stream_kernel does; the exchange is the same. Failure: a
// consumer warp whose wait for a chunk or for the exchange expires stops
// taking chunks and writing, keeps sending its pairs, and waits once more
// before it leaves, as in wide_stream_kernel; the producer stops issuing when
// a wait of its own expires or a consumer failed, and waits (bounded) for
// every copy it issued before it leaves.
#ifndef SR_WIDE_BULK
#define SR_WIDE_BULK 1
#endif
#ifndef SR_WIDE_BULK_CHUNK
#define SR_WIDE_BULK_CHUNK 16384
#endif
#ifndef SR_WIDE_BULK_SLOTS
#define SR_WIDE_BULK_SLOTS 4
#endif
constexpr int kWBChunk = SR_WIDE_BULK_CHUNK;        // bytes
constexpr int kWBUnits = kWBChunk / 16;             // vectors per chunk
constexpr int kWBSlots = SR_WIDE_BULK_SLOTS;
constexpr int kWBThreads = kWideThreads + 32;       // consumers + the producer warp
constexpr int kWBPer = kWBUnits / kWideThreads;     // vectors per consumer thread and chunk
static_assert(kWBChunk % (16 * kWideThreads) == 0, "whole vectors per consumer thread");
constexpr size_t kWBBarOff = (size_t)kWBSlots * kWBChunk;
constexpr size_t kWBSmem = kWBBarOff + 16 * kWBSlots;

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void bulk_g2s_policy(uint32_t dst, const void* src, uint32_t bytes,
                                                uint32_t bar, uint64_t pol) {
    if (!SR_READ_OK(src, bytes)) return;  // never completes: the bounded wait expires
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// MINB: resident blocks per SM it is compiled for (3, or 2 when the rows of
// the clusters resident at 3 blocks/SM would not fit in half the L2 between a
// slice's two reads).
template <typename T, int MINB>
__global__ void __launch_bounds__(kWBThreads, MINB)
    wide_bulk_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int64_t N,
                     int64_t ld_in, int64_t ld_out, int csize, int64_t slice, unsigned int* err,
                     unsigned long long timeout_ns, int flags, int64_t /* ahead: unused */) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, M, ld_in, N), SR_MAT_OUT(out, M, ld_out, N));
    constexpr int VEC = Elem<T>::kVec;
    constexpr int NT = kWideThreads;
    constexpr int NW = kWideWarps;
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ float2 pairs[2][kMaxCluster * NW];
    __shared__ __align__(8) unsigned long long xbar[2];
    __shared__ int s_fail;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)cluster_ctarank();
    const int64_t nclusters = gridDim.x / csize;
    const int64_t nvec = N / VEC;
    const int64_t u0 = (int64_t)rank * slice;
    const int64_t u1 = (u0 + slice < nvec) ? u0 + slice : nvec;
    const int64_t nch = u1 > u0 ? (u1 - u0 + kWBUnits - 1) / kWBUnits : 0;
    const int npairs = csize * NW;
    const bool send = !(flags & kFlagNoCopy);  // test hook: send nothing, every wait expires
    const uint32_t sbase = smem_addr(ring);
    const uint32_t full0 = sbase + (uint32_t)kWBBarOff;  // full[i] at full0 + 8 i
    const uint32_t empty0 = full0 + 8u * kWBSlots;       // empty[i] at empty0 + 8 i

    if (tid == 0) {
        s_fail = 0;
        mbar_init(smem_addr(&xbar[0]), 1);
        mbar_init(smem_addr(&xbar[1]), 1);
        for (int i = 0; i < kWBSlots; ++i) {
            mbar_init(full0 + 8u * i, 1);
            mbar_init(empty0 + 8u * i, NW);
        }
        fence_mbar_init();
    }
    __syncthreads();
    cluster_arrive_relaxed();

    if (warp == NW) {
        // Producer warp: the whole warp passes the cluster barrier, then lane 0
        // issues the copies in the consumers' order.
        cluster_wait();
        if (lane != 0) return;
        const uint64_t keep = l2_policy_keep(), drop = l2_policy_drop();
        int64_t j = 0;
        bool ok = true;
        for (int64_t r = blockIdx.x / csize; r < M && ok; r += nclusters) {
            const T* rin = in + r * ld_in;
            for (int pass = 0; pass < 2 && ok; ++pass) {
                for (int64_t c = 0; c < nch && ok; ++c) {
                    const int64_t cu = u0 + c * kWBUnits;
                    const uint32_t bytes = (uint32_t)((u1 - cu < kWBUnits ? u1 - cu : kWBUnits) * 16);
                    const int slot = (int)(j % kWBSlots);
                    if (j >= kWBSlots) {
                        // Wait for the consumers to release the slot, watching for their failure.
                        const uint32_t bar = empty0 + 8u * slot;
                        const uint32_t par = (uint32_t)((j / kWBSlots - 1) & 1);
                        const uint64_t t0 = global_timer_ns();
                        while (!mbar_try_wait(bar, par)) {
                            if (*(volatile int*)&s_fail || global_timer_ns() - t0 > timeout_ns) {
                                ok = false;
                                break;
                            }
                        }
                        if (!ok) break;
                    }
                    if (*(volatile int*)&s_fail) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(full0 + 8u * slot, bytes);
                    bulk_g2s_policy(sbase + (uint32_t)slot * kWBChunk, rin + cu * VEC, bytes,
                                    full0 + 8u * slot, pass == 0 ? keep : drop);
                    ++j;
                }
            }
        }
        if (!ok) atomicOr(err, 1u);
        // Before the block may exit, every issued copy must have landed.
        for (int64_t i = (j > kWBSlots ? j - kWBSlots : 0); i < j; ++i)
            mbar_wait_bounded(full0 + 8u * (uint32_t)(i % kWBSlots),
                              (uint32_t)((i / kWBSlots) & 1), timeout_ns);
        return;
    }

    // Consumer warps.
    bool started = false, failed = false;
    uint32_t fail_bar = 0, fail_phase = 0, last_bar = 0, last_phase = 0;
    int64_t it = 0, j = 0;
    auto take = [&](int64_t c, uint4 (&v)[kWBPer], int& cnt) -> bool {
        // Chunk c of the slice into registers; false once this warp has failed.
        const int slot = (int)(j % kWBSlots);
        const uint32_t par = (uint32_t)((j / kWBSlots) & 1);
        ++j;
        if (failed) return false;
        if (!mbar_wait_bounded(full0 + 8u * slot, par, timeout_ns)) {
            failed = true;
            s_fail = 1;
            fail_bar = 0;
            return false;
        }
        const int64_t cu = u0 + c * kWBUnits;
        cnt = (int)(u1 - cu < kWBUnits ? u1 - cu : kWBUnits);
        const uint32_t chunk = sbase + (uint32_t)slot * kWBChunk;
#pragma unroll
        for (int k = 0; k < kWBPer; ++k)
            if (tid + k * NT < cnt) v[k] = lds128(chunk + 16u * (tid + k * NT));
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8u * slot);
        return true;
    };
    for (int64_t r = blockIdx.x / csize; r < M; r += nclusters, ++it) {
        const int p = (int)(it & 1);
        const uint32_t phase = (uint32_t)((it >> 1) & 1);
        // Pass 1: per-thread online (m, s).
        float m = neg_inf(), s = 0.0f;
        for (int64_t c = 0; c < nch; ++c) {
            uint4 v[kWBPer];
            int cnt = 0;
            if (!take(c, v, cnt)) break;
            VecMax<T> vm;
#pragma unroll
            for (int k = 0; k < kWBPer; ++k)
                if (tid + k * NT < cnt) vm.add(v[k]);
            const float mn = fmaxf(m, vm.get());
            const float shift = (mn == neg_inf()) ? 0.0f : mn;
            const float shift_l2 = shift * kLog2e;
            float sa = 0.0f, sb = 0.0f;
#pragma unroll
            for (int k = 0; k < kWBPer; ++k) {
                if (tid + k * NT < cnt) {
                    float f[VEC];
                    Elem<T>::unpack(v[k], f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float x = wide_exp<T>(f[e], shift, shift_l2);
                        if (e & 1) sb += x; else sa += x;
                    }
                }
            }
            s = s * merge_scale(m, mn) + (sa + sb);
            m = mn;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
            merge_ms(m, s, m2, s2);
        }
        if (!started) {
            cluster_wait();
            started = true;
        }
        const uint32_t xb = smem_addr(&xbar[p]);
        last_bar = xb;
        last_phase = phase;
        if (tid == 0) mbar_expect_tx(xb, (uint32_t)npairs * 8u);
        if (send && lane < csize)
            st_async_f2(map_to_rank(smem_addr(&pairs[p][rank * NW + warp]), (uint32_t)lane), m, s,
                        map_to_rank(xb, (uint32_t)lane));
        if (!failed && !mbar_wait_bounded(xb, phase, timeout_ns)) {
            failed = true;
            s_fail = 1;
            fail_bar = xb;
            fail_phase = phase;
        }
        if (failed) continue;  // no output; keep sending, so peers do not wait in vain
        float mloc = neg_inf();
        for (int i = lane; i < npairs; i += 32) mloc = fmaxf(mloc, pairs[p][i].x);
        const float Mr = warp_max(mloc);
        float sloc = 0.0f;
        for (int i = lane; i < npairs; i += 32) {
            const float2 q = pairs[p][i];
            sloc += q.y * merge_scale(q.x, Mr);
        }
        const float Sr = warp_sum(sloc);
        // Pass 2: the output, as in wide_stream_kernel.
        T* rout = out + r * ld_out;
        const float rs = Elem<T>::kAccurateExp ? final_rcp(Mr, Sr) : 0.0f;
        const float cexp = Elem<T>::kAccurateExp ? 0.0f : fmaf(Mr, kLog2e, lg2_approx(Sr));
        for (int64_t c = 0; c < nch; ++c) {
            uint4 v[kWBPer];
            int cnt = 0;
            if (!take(c, v, cnt)) break;
            const int64_t cu = u0 + c * kWBUnits;
#pragma unroll
            for (int k = 0; k < kWBPer; ++k) {
                if (tid + k * NT < cnt) {
                    float f[VEC];
                    Elem<T>::unpack(v[k], f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        if constexpr (Elem<T>::kAccurateExp)
                            f[e] = wide_exp<T>(f[e], Mr, 0.0f) * rs;
                        else
                            f[e] = ex2_approx(fmaf(f[e], kLog2e, -cexp));
                    }
                    stg_stream(rout + (cu + tid + k * NT) * VEC, Elem<T>::pack(f));
                }
            }
        }
    }
    if (!started) cluster_wait();
    if (failed) {
        // Once more (bounded): the exchange that failed, or else the last one,
        // so that a late peer's pair does not land after this block exits.
        if (tid == 0) atomicOr(err, 1u);
        if (fail_bar != 0) mbar_wait_bounded(fail_bar, fail_phase, timeout_ns);
        else if (last_bar != 0) mbar_wait_bounded(last_bar, last_phase, timeout_ns);
    }
}

template <typename T>
using WideKernel = void (*)(const T*, T*, int64_t, int64_t, int64_t, int64_t, int, int64_t,
                            unsigned int*, unsigned long long, int, int64_t);

template <typename T>
cudaError_t launch_clusters(WideKernel<T> kern, const Problem& p, int csize, int64_t slice) {
    const void* fn = reinterpret_cast<const void*>(kern);
    cudaError_t e = ensure_smem_limit(fn, 0, csize > 8);
    if (e != cudaSuccess) return e;
    const int resident = max_active_clusters(fn, kWideThreads, 0, csize);
    if (resident <= 0) return cudaErrorInvalidConfiguration;
    // One cluster per row up to the largest grid; beyond it rows are walked
    // with a stride.
    const int64_t cap = 0x7fffffff / csize;
    // The cluster scheduling policy lets the hardware balance a cluster's
    // blocks over the SMs of a GPC (measured: 1.5 % faster than the default
    // policy on 1024 x 131072 bf16).
    const LaunchShape ls{dim3((unsigned)((p.M < cap ? p.M : cap) * csize)), dim3(kWideThreads), 0,
                         csize, SR_WIDE_POLICY};
    e = launch_kernel(kern, ls, p.stream, static_cast<const T*>(p.in), static_cast<T*>(p.out),
                      p.M, p.N, p.ld_in, p.ld_out, csize, slice, p.dev->err, p.timeout_ns,
                      p.flags,
                      (int64_t)(csize >= kAheadMinCluster ? resident * SR_WIDE_AHEAD_QUARTERS / 4 : 0));
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T, int KV>
cudaError_t launch_mode(const Problem& p, const WideShape& sh, int mode) {
    switch (mode) {
        case kAligned: return launch_clusters<T>(wide_rows_kernel<T, KV, kAligned>, p, sh.csize,
                                                 sh.slice);
        case kFull: return launch_clusters<T>(wide_rows_kernel<T, KV, kFull>, p, sh.csize, sh.slice);
        case kShifted: return launch_clusters<T>(wide_rows_kernel<T, KV, kShifted>, p, sh.csize,
                                                 sh.slice);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_typed(const Problem& p, const WideShape& sh) {
    const int64_t nvec = p.N / Elem<T>::kVec;
    const bool aligned = rows_vector_aligned(p.in, p.out, p.N, p.ld_in, p.ld_out, p.dtype);
    if (sh.staged) {
        if (!aligned) return cudaErrorInvalidValue;
        const int c = sh.csize;
        if (sh.slice != (int64_t)kWideThreads * (kStagedKV + kStagedKS) || nvec != sh.slice * c)
            return cudaErrorInvalidValue;
        auto kern = wide_staged_kernel<T>;
        const size_t smem = (size_t)kWideThreads * kStagedKS * 16;
        const void* fn = reinterpret_cast<const void*>(kern);
        cudaError_t e = ensure_smem_limit(fn, smem, c > 8);
        if (e != cudaSuccess) return e;
        const int resident = max_active_clusters(fn, kWideThreads, smem, c);
        if (resident <= 0) return cudaErrorInvalidConfiguration;
        const int64_t cap = 0x7fffffff / c;
        const LaunchShape ls{dim3((unsigned)((p.M < cap ? p.M : cap) * c)), dim3(kWideThreads),
                             smem, c, SR_WIDE_POLICY};
        return launch_kernel(kern, ls, p.stream, static_cast<const T*>(p.in),
                             static_cast<T*>(p.out), p.M, p.N, p.ld_in, p.ld_out, c, sh.slice,
                             p.dev->err, p.timeout_ns, p.flags,
                             (int64_t)(c >= kAheadMinCluster ? resident * SR_WIDE_AHEAD_QUARTERS / 4
                                                             : 0));
    }
    if (sh.streamed) {
        if (!aligned) return cudaErrorInvalidValue;
        // The bulk-copy ring on 8-block clusters; 16-block clusters (few rows) stay on
        // register loads. Measured on GB300 (cold L2, µs, bulk with 16 KiB x 3
        // slots at 3 blocks/SM against register loads): 8-block clusters: bf16
        // 512 x 400008 150.5 / 156.7, bf16 256 x 1048576 209.6 / 245.8, f32
        // 256 x 524288 209.2 / 247.3, f16 96 x 1500000 125.1 / 161.8; 16-block
        // clusters: f32 32 x 4194304 272.2 / 268.8, bf16 64 x 600008 40.1 / 36.5.
        // With 4 slots, at 3 / 2 blocks per SM: bf16 512 x 400008 145.5 / 162.5,
        // bf16 256 x 1048576 209.2 / 192.3, f16 96 x 1500000 128.0 / 115.7, f32
        // 128 x 600000 130.8 / 121.1 (32 KiB x 2 slots 169-279, 8 KiB x 6 127-218):
        // 3 blocks per SM while the resident clusters' rows fit in half the L2.
        if (SR_WIDE_BULK && sh.csize <= 8) {
            const int64_t row_bytes = p.N * (int64_t)sizeof(T);
            const bool three = (int64_t)3 * p.dev->sm_count / sh.csize * row_bytes <= p.dev->l2_bytes / 2;
            auto kern = three ? wide_bulk_kernel<T, 3> : wide_bulk_kernel<T, 2>;
            const void* fn = reinterpret_cast<const void*>(kern);
            const int c = sh.csize;
            cudaError_t e = ensure_smem_limit(fn, kWBSmem, c > 8);
            if (e != cudaSuccess) return e;
            if (max_active_clusters(fn, kWBThreads, kWBSmem, c) <= 0)
                return cudaErrorInvalidConfiguration;
            const int64_t cap = 0x7fffffff / c;
            const LaunchShape ls{dim3((unsigned)((p.M < cap ? p.M : cap) * c)), dim3(kWBThreads),
                                 kWBSmem, c, SR_WIDE_POLICY};
            return launch_kernel(kern, ls, p.stream, static_cast<const T*>(p.in),
                                 static_cast<T*>(p.out), p.M, p.N, p.ld_in, p.ld_out, c, sh.slice,
                                 p.dev->err, p.timeout_ns, p.flags, (int64_t)0);
        }
        return launch_clusters<T>(wide_stream_kernel<T>, p, sh.csize, sh.slice);
    }
    int mode = kShifted;
    if (aligned)
        mode = (sh.slice == (int64_t)kWideThreads * sh.kv && nvec == sh.slice * sh.csize) ? kFull
                                                                                          : kAligned;
    switch (sh.kv) {
        case 1: return launch_mode<T, 1>(p, sh, mode);
        case 2: return launch_mode<T, 2>(p, sh, mode);
        case 4: return launch_mode<T, 4>(p, sh, mode);
        case 8: return launch_mode<T, 8>(p, sh, mode);
#if SR_WIDE_MID_KV
        case 5: return launch_mode<T, 5>(p, sh, mode);
        case 6: return launch_mode<T, 6>(p, sh, mode);
#endif
    }
    return cudaErrorInvalidValue;
}

}  // namespace

// Shape (host logic): clusters of 2..16 blocks of 256 threads; the smallest
// power-of-two cluster whose slices give each thread at most SR_WIDE_KV
// vectors. While there are too few rows to give every SM two blocks, the
// cluster doubles (up to 8: larger clusters are scheduled poorly) as long as
// each thread keeps at least one vector. The vectors per thread are rounded
// up to 1, 2, 4 or 8. Rows up to 16 x 256 x 8 vectors (512 KiB) are held in
// registers; aligned rows of exactly twice that (1 MiB) are staged (16-block
// clusters, 8 vectors per thread in registers and 8 in shared memory); other
// wider rows are streamed by 8-block clusters (16 while the grid would not
// fill one wave of resident blocks).
bool wide_shape(int64_t M, int64_t N, int dtype, int sm_count, WideShape* out) {
    const int64_t nvec = N * elem_bytes(dtype) / 16;
    for (int c = 2; c <= kMaxCluster; c *= 2) {
        if ((nvec + c - 1) / c > (int64_t)kWideThreads * SR_WIDE_KV) continue;
        while (c < 8 && M * c < 2 * (int64_t)sm_count && nvec / (2 * c) >= kWideThreads) c *= 2;
        const int64_t per = (nvec + c - 1) / c;
        const int64_t kv = (per + kWideThreads - 1) / kWideThreads;
        out->csize = c;
        out->slice = per;
        out->kv = kv <= 1 ? 1 : kv <= 2 ? 2 : kv <= 4 ? 4
                : (SR_WIDE_MID_KV && kv <= 5) ? 5 : (SR_WIDE_MID_KV && kv <= 6) ? 6 : 8;
        out->streamed = false;
        return true;
    }
    if (SR_WIDE_STAGED && nvec == (int64_t)kMaxCluster * kWideThreads * (kStagedKV + kStagedKS)) {
        out->csize = kMaxCluster;
        out->slice = (nvec + kMaxCluster - 1) / kMaxCluster;
        out->kv = kStagedKV + kStagedKS;
        out->streamed = false;
        out->staged = true;
        return true;
    }
    int c = SR_WIDE_STREAM_CLUSTER;
    while (c < kMaxCluster && M * c < (int64_t)SR_WIDE_STREAM_MIN_BLOCKS * sm_count) c *= 2;
    out->csize = c;
    out->slice = (nvec + c - 1) / c;
    out->kv = 0;
    out->streamed = true;
    return true;
}

// Whether the WIDE plan takes these rows: aligned rows of any width, or rows
// of at most 512 KiB whose input and output share their offset from a
// 16-byte boundary.
bool wide_fits(const void* in, const void* out, int64_t N, int64_t ld_in, int64_t ld_out,
               int dtype) {
    WideShape sh;
    if (!wide_shape(1, N, dtype, 0, &sh)) return false;
    if (rows_vector_aligned(in, out, N, ld_in, ld_out, dtype)) return true;
    if (sh.streamed || sh.staged) return false;
    const int64_t es = elem_bytes(dtype);
    const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
    return a % 16 == b % 16 && a % es == 0 && (ld_in * es) % 16 == (ld_out * es) % 16;
}

cudaError_t launch_wide(const Problem& p) {
    WideShape sh;
    if (!wide_shape(p.M, p.N, p.dtype, p.dev->sm_count, &sh)) return cudaErrorInvalidValue;
    switch (p.dtype) {
        case kF32: return launch_typed<float>(p, sh);
        case kBF16: return launch_typed<__nv_bfloat16>(p, sh);
        case kF16: return launch_typed<__half>(p, sh);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sr
