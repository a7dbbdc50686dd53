// CTA and CLUSTER plans: rows (or row slices) staged in shared memory by
// 1-D bulk asynchronous copies, several rows ahead.
//
// CTA plan ("Fused Softmax on GPU", Triton one block per row and the
// persistent variant): one thread block per row, the persistent grid walking
// rows with a stride. Instead of a compiler-pipelined register load, one
// thread issues cp.async.bulk copies of whole rows into a ring of `stages`
// shared-memory buffers, each completing on its own mbarrier, so the next
// rows stream in while the current one is reduced.
//
// CLUSTER plan (the split plan of "Measured optimization case studies",
// Wide rows, kept on chip): a cluster of `csize` blocks owns a row; block k
// stages slice k. Each warp reduces its part to an online (max, sum) pair
// with the all -inf guard of the same section and stores the pair into every
// block's shared memory with st.async, which completes on that block's
// exchange mbarrier; each block waits (bounded) for all pairs of the row,
// merges them and writes its slice. No cluster-wide barrier (and so no cluster-scope fence)
// sits in the row loop. Every input element is read from HBM once, written
// once and exponentiated once.
//
// Per row (both plans): each warp reduces its values to (m_w, s_w) with
// e = exp(x - m_w) and publishes the pair (shared memory for the CTA plan;
// st.async into every block of the cluster for the CLUSTER plan); after one
// block barrier each warp merges all published pairs into the row's (M, S)
// itself, rescales its e by exp(m_w - M) / S and stores. Warp 1 issues the
// bulk copies, so no warp serialises the merge behind the copy engine.
//
// Every wait (bulk copy, exchange) is bounded (wall clock, `timeout_ns`); on
// expiry the block records the failure in the error word, stops at its next
// block barrier, drains its in-flight copies (again bounded) and returns; its
// peers' exchange waits then expire too.
#include "device.cuh"
#include "internal.h"

#ifndef SR_TMA_STAGE_BUDGET
#define SR_TMA_STAGE_BUDGET (96 * 1024)
#endif
#ifndef SR_TMA_MAX_STAGES
#define SR_TMA_MAX_STAGES 4
#endif
// CLUSTER plan: stage budget per block, and the resident blocks per SM the
// widest slices are compiled for (the register file holds every block's
// FP32 slice values, so it is what bounds the blocks per SM).
#ifndef SR_CLUSTER_STAGE_BUDGET
#define SR_CLUSTER_STAGE_BUDGET (96 * 1024)
#endif
#ifndef SR_CLUSTER_MIN_BLOCKS
#define SR_CLUSTER_MIN_BLOCKS 2
#endif
#ifndef SR_CLUSTER_MIN_BLOCKS_SMALL
#define SR_CLUSTER_MIN_BLOCKS_SMALL 1
#endif
#ifndef SR_CLUSTER_MIN_BLOCKS_PARKED
#define SR_CLUSTER_MIN_BLOCKS_PARKED 3
#endif
// Vectors per thread whose exponentials are parked in shared memory for the
// widest 16-bit slices (KV = 8), and the stage budget in that case.
#ifndef SR_CLUSTER_PARK
#define SR_CLUSTER_PARK 4
#endif
#ifndef SR_CLUSTER_PARK_STAGE_BUDGET
#define SR_CLUSTER_PARK_STAGE_BUDGET (32 * 1024)
#endif

namespace sr {
namespace {

constexpr int kTmaThreads = 256;

struct SmemLayout {
    uint32_t stage_bytes;
    int stages;
    uint32_t ebuf_bytes;  // FP32 exponentials parked in shared memory (0: none)
    // [stages x stage_bytes] rows | 8 stage mbarriers + 2 exchange mbarriers |
    // 2 x 32 warp partials (float2, CTA plan) | 2 x kMaxCluster x 8 partials
    // (float2, CLUSTER plan: one per warp of every block of the cluster)
    __host__ __device__ uint32_t bar_off() const { return stage_bytes * stages; }
    __host__ __device__ uint32_t red_off() const { return bar_off() + 16u * 8u; }
    __host__ __device__ uint32_t xch_off() const { return red_off() + 2u * 32u * 8u; }
    __host__ __device__ uint32_t ebuf_off() const { return xch_off() + 2u * kMaxCluster * 8u * 8u; }
    __host__ __device__ uint32_t total() const { return ebuf_off() + ebuf_bytes; }
};

// KS: of each thread's KV vectors, the last KS keep their FP32 exponentials
// in shared memory instead of registers between the exchange and the store,
// which lets more blocks share an SM's register file.
template <typename T, int NT, int KV, bool CLUSTER, int KS>
__global__ void __launch_bounds__(NT, !CLUSTER ? 1
                                       : (KS > 0 ? SR_CLUSTER_MIN_BLOCKS_PARKED
                                          : KV * Elem<T>::kVec >= 64 ? SR_CLUSTER_MIN_BLOCKS
                                                                     : SR_CLUSTER_MIN_BLOCKS_SMALL))
    tma_rows_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int64_t N,
                    int64_t ld_in, int64_t ld_out, int csize, SmemLayout L, unsigned int* err,
                    unsigned long long timeout_ns, int flags) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, M, ld_in, N), SR_MAT_OUT(out, M, ld_out, N));
    constexpr int VEC = Elem<T>::kVec;
    constexpr int NW = NT / 32;
    static_assert(NW <= 8 || !CLUSTER, "cluster exchange slots hold 8 warps per block");
    static_assert(KS >= 0 && KS <= KV, "parked vectors");
    constexpr int KR = KV - KS;  // vectors whose exponentials stay in registers
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar0 = sbase + L.bar_off();   // stage barriers
    const uint32_t xbar0 = bar0 + 8u * 8u;      // exchange barriers (cluster plan)
    float2* red = reinterpret_cast<float2*>(smem + L.red_off());
    float2* xch = reinterpret_cast<float2*>(smem + L.xch_off());
    // Parked exponentials: vector k (KV - KS <= k < KV) of thread tid, half h,
    // at ebuf[((k - (KV - KS)) * 2 + h) * NT + tid] (16-byte units): a warp's
    // 32 stores of one (k, h) cover 512 consecutive bytes.
    const uint32_t ebuf = sbase + L.ebuf_off();

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int kProducer = 32;  // warp 1, lane 0 issues and tracks the bulk copies
    const int rank = CLUSTER ? (int)cluster_ctarank() : 0;
    const int64_t unit = CLUSTER ? blockIdx.x / csize : blockIdx.x;
    const int64_t nunits = CLUSTER ? gridDim.x / csize : gridDim.x;

    // This block's slice of every row, in 16-byte vectors.
    const int64_t nvec = N / VEC;
    const int64_t per = (nvec + csize - 1) / csize;
    const int64_t v0 = (int64_t)rank * per;
    const int cnt = (int)(v0 < nvec ? (nvec - v0 < per ? nvec - v0 : per) : 0);
    const uint32_t bytes = (uint32_t)cnt * 16u;
    const bool copies = cnt > 0 && !(flags & kFlagNoCopy);

    if (tid == 0) {
        for (int s = 0; s < L.stages; ++s) mbar_init(bar0 + 8u * s, 1);
        mbar_init(xbar0, 1);
        mbar_init(xbar0 + 8u, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if constexpr (CLUSTER) cluster_sync_all();  // peers started, barriers initialised

    int64_t issued = 0, confirmed = 0;  // the producer's copies issued / seen complete
    auto issue = [&](int64_t it) {
        const int s = (int)(it % L.stages);
        const int64_t r = unit + it * nunits;
        const T* src = in + r * ld_in + v0 * VEC;
        mbar_expect_tx(bar0 + 8u * s, bytes);
        bulk_g2s(sbase + (uint32_t)s * L.stage_bytes, src, bytes, bar0 + 8u * s);
    };
    if (tid == kProducer && copies) {
        for (int s = 0; s < L.stages && unit + (int64_t)s * nunits < M; ++s) issue(issued++);
    }

    bool local_fail = false;
    for (int64_t it = 0;; ++it) {
        const int64_t r = unit + it * nunits;
        if (r >= M) break;  // uniform: every block of a cluster walks the same rows
        const int s = (int)(it % L.stages);
        const int p = (int)(it & 1);

        bool ok = !local_fail;
        if (ok && cnt > 0) {
            ok = mbar_wait_bounded(bar0 + 8u * s, (uint32_t)((it / L.stages) & 1), timeout_ns);
            if (tid == kProducer && ok) confirmed = it + 1;
            local_fail = !ok;
        }

        float v[KV][VEC];
        // Slice values into registers (vectors tid, tid+NT, ...). Vectors
        // k >= KV - KS are only read here for the max; their exponentials are
        // computed from a second read of the staged slice and parked.
        const uint32_t stage = sbase + (uint32_t)s * L.stage_bytes;
        float mx = neg_inf();
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + NT * k;
            float f[VEC];
            if (ok && idx < cnt) {
                Elem<T>::unpack(lds128(stage + 16u * idx), f);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) f[e] = neg_inf();
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                mx = fmaxf(mx, f[e]);
                if (k < KR) v[k][e] = f[e];
            }
        }

        // Warp partial: m_w, then e = exp(x - shift) and s_w (all -inf guard).
        const float m_w = warp_max(mx);
        const float shift = (m_w == neg_inf()) ? 0.0f : m_w;
        const float shift_l2 = shift * kLog2e;
        // Two partial sums per thread keep the register count low (the
        // slice values themselves fill most of the register file).
        float sa = 0.0f, sb = 0.0f;
#pragma unroll
        for (int k = 0; k < KR; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                v[k][e] = exp_shifted<T>(v[k][e], shift, shift_l2);
                if (e & 1) sb += v[k][e]; else sa += v[k][e];
            }
#pragma unroll
        for (int k = KR; k < KV; ++k) {
            const int idx = tid + NT * k;
            float f[VEC];
            if (ok && idx < cnt) {
                Elem<T>::unpack(lds128(stage + 16u * idx), f);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) f[e] = neg_inf();
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                f[e] = exp_shifted<T>(f[e], shift, shift_l2);
                if (e & 1) sb += f[e]; else sa += f[e];
            }
            const uint32_t a = ebuf + 16u * (uint32_t)(((k - KR) * 2) * NT + tid);
#pragma unroll
            for (int h = 0; h < VEC / 4; ++h)
                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a + 16u * NT * h),
                             "f"(f[4 * h]), "f"(f[4 * h + 1]), "f"(f[4 * h + 2]), "f"(f[4 * h + 3])
                             : "memory");
        }
        const float s_w = warp_sum(sa + sb);
        if constexpr (!CLUSTER) {
            if (lane == 0) red[p * 32 + warp] = make_float2(m_w, s_w);
        }
        // The stage is consumed (and, for the CTA plan, the warp partials are
        // visible); a failure anywhere in the block stops every thread here.
        if (__syncthreads_or(local_fail)) {
            local_fail = true;
            break;
        }
        // Refill the consumed stage with the row `stages` iterations ahead.
        if (tid == kProducer && copies && issued == it + L.stages &&
            unit + (it + L.stages) * nunits < M)
            issue(issued++);

        // Row (M, S): merge every warp's pair of the block (CTA) or cluster.
        float Mr, Sr;
        if constexpr (CLUSTER) {
            // Each warp stores its pair into slot [p][rank][warp] of every block
            // of the cluster; each store completes 8 bytes on the receiver's
            // exchange barrier for this parity, which expects csize * NW pairs.
            const int npairs = csize * NW;
            if (tid == 0) mbar_expect_tx(xbar0 + 8u * p, (uint32_t)npairs * 8u);
            if (lane < csize) {
                const uint32_t slot = smem_addr(xch + (p * kMaxCluster + rank) * 8 + warp);
                st_async_f2(map_to_rank(slot, lane), m_w, s_w, map_to_rank(xbar0 + 8u * p, lane));
            }
            if (!mbar_wait_bounded(xbar0 + 8u * p, (uint32_t)((it >> 1) & 1), timeout_ns)) {
                local_fail = true;  // a peer stopped; the next block barrier stops us
                continue;
            }
            float mloc = neg_inf();
            for (int i = lane; i < npairs; i += 32)
                mloc = fmaxf(mloc, xch[(p * kMaxCluster + i / NW) * 8 + i % NW].x);
            Mr = warp_max(mloc);
            float sloc = 0.0f;
            for (int i = lane; i < npairs; i += 32) {
                const float2 q = xch[(p * kMaxCluster + i / NW) * 8 + i % NW];
                sloc += q.y * merge_scale(q.x, Mr);
            }
            Sr = warp_sum(sloc);
        } else {
            const float2 q = lane < NW ? red[p * 32 + lane] : make_float2(neg_inf(), 0.0f);
            Mr = warp_max(q.x);
            Sr = warp_sum(q.y * merge_scale(q.x, Mr));
        }

        const float f = merge_scale(m_w, Mr) * final_rcp(Mr, Sr);
        T* rout = out + r * ld_out + v0 * VEC + (int64_t)tid * VEC;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            if (k >= KR) {  // bring a parked vector back
                const uint32_t a = ebuf + 16u * (uint32_t)(((k - KR) * 2) * NT + tid);
#pragma unroll
                for (int h = 0; h < VEC / 4; ++h)
                    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                 : "=f"(v[k][4 * h]), "=f"(v[k][4 * h + 1]), "=f"(v[k][4 * h + 2]),
                                   "=f"(v[k][4 * h + 3])
                                 : "r"(a + 16u * NT * h)
                                 : "memory");
            }
            if (tid + NT * k < cnt) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] *= f;
                stg_stream(rout + k * NT * VEC, Elem<T>::pack(v[k]));
            }
        }
    }

    if (tid == 0 && local_fail) atomicOr(err, 1u);
    if (tid == kProducer) {
        // Drain copies still in flight (only after a failure), bounded.
        for (int64_t j = confirmed; j < issued; ++j)
            mbar_wait_bounded(bar0 + 8u * (uint32_t)(j % L.stages), (uint32_t)((j / L.stages) & 1),
                              timeout_ns);
    }
    // No block of the cluster leaves while a peer may still store into it.
    if constexpr (CLUSTER) cluster_sync_all();
}

template <typename T, int KV, bool CLUSTER, int KS>
cudaError_t launch_kv(const Problem& p, int csize, SmemLayout L) {
    auto kern = tma_rows_kernel<T, kTmaThreads, KV, CLUSTER, KS>;
    const void* fn = reinterpret_cast<const void*>(kern);
    const size_t smem = L.total();
    cudaError_t e = ensure_smem_limit(fn, smem, csize > 8);
    if (e != cudaSuccess) return e;
    if ((int64_t)smem > p.dev->smem_optin) return cudaErrorInvalidValue;
    const T* in = static_cast<const T*>(p.in);
    T* out = static_cast<T*>(p.out);
    if constexpr (!CLUSTER) {
        const int per_sm = blocks_per_sm(fn, kTmaThreads, smem);
        if (per_sm <= 0) return cudaErrorInvalidConfiguration;
        const int64_t cap = (int64_t)per_sm * p.dev->sm_count;
        const unsigned grid = (unsigned)(p.M < cap ? p.M : cap);
        return launch_kernel(kern, LaunchShape{dim3(grid), dim3(kTmaThreads), smem}, p.stream, in,
                             out, p.M, p.N, p.ld_in, p.ld_out, 1, L, p.dev->err, p.timeout_ns,
                             p.flags);
    } else {
        const int nclusters = max_active_clusters(fn, kTmaThreads, smem, csize);
        if (nclusters <= 0) return cudaErrorInvalidConfiguration;
        const int64_t units = p.M < nclusters ? p.M : nclusters;
        return launch_kernel(
            kern, LaunchShape{dim3((unsigned)(units * csize)), dim3(kTmaThreads), smem, csize},
            p.stream, in, out, p.M, p.N, p.ld_in, p.ld_out, csize, L, p.dev->err, p.timeout_ns,
            p.flags);
    }
}

template <typename T, bool CLUSTER>
cudaError_t launch_typed(const Problem& p, int csize) {
    constexpr int VEC = Elem<T>::kVec;
    const int64_t nvec = p.N / VEC;
    const int64_t per = (nvec + csize - 1) / csize;  // vectors per block
    const int64_t kv = (per + kTmaThreads - 1) / kTmaThreads;
    SmemLayout L;
    L.stage_bytes = (uint32_t)(((per * 16) + 127) / 128 * 128);
    L.ebuf_bytes = 0u;
    auto stages_for = [&](int64_t budget, int lo) {
        int st = (int)(budget / L.stage_bytes);
        return st < lo ? lo : (st > SR_TMA_MAX_STAGES ? SR_TMA_MAX_STAGES : st);
    };
    const bool wide16 = CLUSTER && VEC == 8 && kv > 4;
    if constexpr (CLUSTER && VEC == 8) {
        // The widest 16-bit slices park part of their exponentials in shared
        // memory, so that three blocks share an SM's register file.
        if (wide16 && SR_CLUSTER_PARK > 0) {
            L.stages = stages_for(SR_CLUSTER_PARK_STAGE_BUDGET, 1);
            L.ebuf_bytes = (uint32_t)(SR_CLUSTER_PARK * kTmaThreads * VEC * 4);
            return launch_kv<T, 8, CLUSTER, SR_CLUSTER_PARK>(p, csize, L);
        }
    }
    L.stages = stages_for(CLUSTER ? SR_CLUSTER_STAGE_BUDGET : SR_TMA_STAGE_BUDGET, 2);
    if ((int64_t)L.total() > p.dev->smem_optin) return cudaErrorInvalidValue;
    if (kv <= 1) return launch_kv<T, 1, CLUSTER, 0>(p, csize, L);
    if (kv <= 2) return launch_kv<T, 2, CLUSTER, 0>(p, csize, L);
    if (kv <= 4) return launch_kv<T, 4, CLUSTER, 0>(p, csize, L);
    if (kv <= 8) return launch_kv<T, 8, CLUSTER, 0>(p, csize, L);
    return cudaErrorInvalidValue;
}

template <bool CLUSTER>
cudaError_t launch_dtype(const Problem& p, int csize) {
    switch (p.dtype) {
        case kF32: return launch_typed<float, CLUSTER>(p, csize);
        case kBF16: return launch_typed<__nv_bfloat16, CLUSTER>(p, csize);
        case kF16: return launch_typed<__half, CLUSTER>(p, csize);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_tma(const Problem& p, int cluster) {
    if (cluster <= 1) return launch_dtype<false>(p, 1);
    return launch_dtype<true>(p, cluster);
}

}  // namespace sr
