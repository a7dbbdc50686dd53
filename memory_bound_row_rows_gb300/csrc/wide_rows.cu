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
// Failure: a wait that expires marks the block failed; it writes nothing
// more, records the failure in the error word and, before leaving, waits once
// more (bounded) so that a late peer's pair cannot land after it exits.
#include "device.cuh"
#include "internal.h"
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

constexpr int kWideThreads = 256;
constexpr int kWideWarps = kWideThreads / 32;

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// KV: 16-byte vectors per thread; `slice`: vectors per block (<= 256 * KV).
// FULL: every block's slice is exactly 256 * KV vectors, so no vector needs a
// bounds check (straight-line loads, math and stores).
template <typename T, int KV, bool FULL>
__global__ void __launch_bounds__(kWideThreads, SR_WIDE_MIN_BLOCKS)
    wide_rows_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int64_t N,
                     int64_t ld_in, int64_t ld_out, int csize, int64_t slice, unsigned int* err,
                     unsigned long long timeout_ns, int flags) {
    constexpr int VEC = Elem<T>::kVec;
    constexpr int NT = kWideThreads;
    constexpr int NW = kWideWarps;
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
    const int64_t u1 = (u0 + slice < nvec) ? u0 + slice : nvec;
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
        uint4 raw[KV];
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int64_t idx = u0 + tid + NT * k;
            if (FULL || idx < u1) raw[k] = ldg_stream(rin + idx * VEC);
        }
        // Warp partial (m_w, s_w): max, then sum of exp(x - m_w).
        VecMax<T> vm;
#pragma unroll
        for (int k = 0; k < KV; ++k)
            if (FULL || u0 + tid + NT * k < u1) vm.add(raw[k]);
        const float m_w = warp_max(vm.get());
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
                    const float x = exp_shifted<T>(f[e], shift, shift_l2);
                    if (e & 1) sb += x; else sa += x;
                }
            }
        }
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
                    for (int e = 0; e < VEC; ++e) f[e] = expf(f[e] - Mr) * rs;
                    stg_stream(rout + idx * VEC, Elem<T>::pack(f));
                }
            }
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
                    stg_stream(rout + idx * VEC, Elem<T>::pack(f));
                }
            }
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

template <typename T, int KV, bool FULL>
cudaError_t launch_kv(const Problem& p, int csize, int64_t slice) {
    auto kern = wide_rows_kernel<T, KV, FULL>;
    const void* fn = reinterpret_cast<const void*>(kern);
    cudaError_t e = ensure_smem_limit(fn, 0, csize > 8);
    if (e != cudaSuccess) return e;
    if (max_active_clusters(fn, kWideThreads, 0, csize) <= 0) return cudaErrorInvalidConfiguration;
    // One cluster per row up to the largest grid; beyond it rows are walked
    // with a stride.
    const int64_t cap = 0x7fffffff / csize;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.M < cap ? p.M : cap) * csize), 1, 1);
    cfg.blockDim = dim3(kWideThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = p.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Let the hardware balance a cluster's blocks over the SMs of a GPC
    // (measured: 1.5 % faster than the default policy on 1024 x 131072 bf16).
    attr[1].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
    attr[1].val.clusterSchedulingPolicyPreference = (cudaClusterSchedulingPolicy)SR_WIDE_POLICY;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, static_cast<const T*>(p.in), static_cast<T*>(p.out), p.M,
                           p.N, p.ld_in, p.ld_out, csize, slice, p.dev->err, p.timeout_ns,
                           p.flags);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const Problem& p, const WideShape& sh) {
    const int64_t nvec = p.N / Elem<T>::kVec;
    const bool full = sh.slice == (int64_t)kWideThreads * sh.kv && nvec == sh.slice * sh.csize;
    switch (sh.kv) {
        case 2:
            return full ? launch_kv<T, 2, true>(p, sh.csize, sh.slice)
                        : launch_kv<T, 2, false>(p, sh.csize, sh.slice);
        case 4:
            return full ? launch_kv<T, 4, true>(p, sh.csize, sh.slice)
                        : launch_kv<T, 4, false>(p, sh.csize, sh.slice);
        case 8:
            return full ? launch_kv<T, 8, true>(p, sh.csize, sh.slice)
                        : launch_kv<T, 8, false>(p, sh.csize, sh.slice);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

// Shape (host logic): clusters of 2..16 blocks of 256 threads; the smallest
// power-of-two cluster whose slices give each thread at most SR_WIDE_KV
// vectors, the vectors per thread rounded up to 2, 4 or 8. Rows up to
// 16 x 256 x 8 vectors (512 KiB) fit.
bool wide_shape(int64_t N, int dtype, WideShape* out) {
    const int64_t nvec = N * elem_bytes(dtype) / 16;
    for (int c = 2; c <= kMaxCluster; c *= 2) {
        const int64_t per = (nvec + c - 1) / c;
        if (per <= (int64_t)kWideThreads * SR_WIDE_KV) {
            const int64_t kv = (per + kWideThreads - 1) / kWideThreads;
            out->csize = c;
            out->slice = per;
            out->kv = kv <= 2 ? 2 : kv <= 4 ? 4 : 8;
            return true;
        }
    }
    return false;
}

cudaError_t launch_wide(const Problem& p) {
    WideShape sh;
    if (!wide_shape(p.N, p.dtype, &sh)) return cudaErrorInvalidValue;
    switch (p.dtype) {
        case kF32: return launch_typed<float>(p, sh);
        case kBF16: return launch_typed<__nv_bfloat16>(p, sh);
        case kF16: return launch_typed<__half>(p, sh);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sr
