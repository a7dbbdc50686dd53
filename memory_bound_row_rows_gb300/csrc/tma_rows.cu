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
// stages slice k. Each block reduces its slice to an online (max, sum) pair
// with the all -inf guard of the same section and stores the pair into every
// peer's shared memory with st.async, which completes on the peer's exchange
// mbarrier; each block waits (bounded) for the csize pairs, merges them and
// writes its slice. No cluster-wide barrier (and so no cluster-scope fence)
// sits in the row loop. Every input element is read from HBM once, written
// once and exponentiated once.
//
// Per row (both plans): each warp reduces its values to (m_w, s_w) with
// e = exp(x - m_w); warp 0 merges the warps' pairs and publishes the block's
// pair (block barrier, or st.async to the cluster); each warp rescales its e
// by exp(m_w - M) / S and stores.
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

namespace sr {
namespace {

constexpr int kTmaThreads = 256;

struct SmemLayout {
    uint32_t stage_bytes;
    int stages;
    // [stages x stage_bytes] rows | 8 stage mbarriers + 2 exchange mbarriers |
    // 32 warp partials (float4) | 2 x kMaxCluster exchange slots (float4)
    __host__ __device__ uint32_t bar_off() const { return stage_bytes * stages; }
    __host__ __device__ uint32_t red_off() const { return bar_off() + 16u * 8u; }
    __host__ __device__ uint32_t xch_off() const { return red_off() + 32u * 16u; }
    __host__ __device__ uint32_t total() const { return xch_off() + 2u * kMaxCluster * 16u; }
};

template <typename T, int NT, int KV, bool CLUSTER>
__global__ void __launch_bounds__(NT, (CLUSTER && KV * Elem<T>::kVec >= 64) ? SR_CLUSTER_MIN_BLOCKS : 1)
    tma_rows_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int64_t N,
                    int64_t ld_in, int64_t ld_out, int csize, SmemLayout L, unsigned int* err,
                    unsigned long long timeout_ns, int flags) {
    constexpr int VEC = Elem<T>::kVec;
    constexpr int NW = NT / 32;
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar0 = sbase + L.bar_off();   // stage barriers
    const uint32_t xbar0 = bar0 + 8u * 8u;      // exchange barriers (cluster plan)
    float4* red = reinterpret_cast<float4*>(smem + L.red_off());
    float4* xch = reinterpret_cast<float4*>(smem + L.xch_off());

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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

    int64_t issued = 0, confirmed = 0;  // copies issued / seen complete (thread 0)
    auto issue = [&](int64_t it) {
        const int s = (int)(it % L.stages);
        const int64_t r = unit + it * nunits;
        const T* src = in + r * ld_in + v0 * VEC;
        mbar_expect_tx(bar0 + 8u * s, bytes);
        bulk_g2s(sbase + (uint32_t)s * L.stage_bytes, src, bytes, bar0 + 8u * s);
    };
    if (tid == 0 && copies) {
        for (int s = 0; s < L.stages && unit + (int64_t)s * nunits < M; ++s) issue(issued++);
    }

    bool local_fail = false;
    for (int64_t it = 0;; ++it) {
        const int64_t r = unit + it * nunits;
        if (r >= M) break;  // uniform: every block of a cluster walks the same rows
        const int s = (int)(it % L.stages);

        bool ok = !local_fail;
        if (ok && cnt > 0) {
            ok = mbar_wait_bounded(bar0 + 8u * s, (uint32_t)((it / L.stages) & 1), timeout_ns);
            if (tid == 0 && ok) confirmed = it + 1;
            local_fail = !ok;
        }

        // Slice values into registers (vectors tid, tid+NT, ...).
        float v[KV][VEC];
        const uint32_t stage = sbase + (uint32_t)s * L.stage_bytes;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + NT * k;
            if (ok && idx < cnt) {
                Elem<T>::unpack(lds128(stage + 16u * idx), v[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = neg_inf();
            }
        }

        // Warp partial: m_w, then e = exp(x - shift) and s_w (all -inf guard).
        float mx = v[0][0];
#pragma unroll
        for (int k = 0; k < KV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) mx = fmaxf(mx, v[k][e]);
        const float m_w = warp_max(mx);
        const float shift = (m_w == neg_inf()) ? 0.0f : m_w;
        const float shift_l2 = shift * kLog2e;
        float sv[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) sv[e] = 0.0f;
#pragma unroll
        for (int k = 0; k < KV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                v[k][e] = exp_shifted<T>(v[k][e], shift, shift_l2);
                sv[e] += v[k][e];
            }
#pragma unroll
        for (int w = VEC / 2; w > 0; w >>= 1)
#pragma unroll
            for (int e = 0; e < w; ++e) sv[e] += sv[e + w];
        const float s_w = warp_sum(sv[0]);
        if (lane == 0) red[warp] = make_float4(m_w, s_w, 0.0f, 0.0f);
        // The stage is consumed and the warp partials are visible; a failure
        // anywhere in the block stops every thread here, together.
        if (__syncthreads_or(local_fail)) {
            local_fail = true;
            break;
        }

        if (warp == 0) {
            const float4 pw = lane < NW ? red[lane] : make_float4(neg_inf(), 0.0f, 0.0f, 0.0f);
            const float mk = warp_max(pw.x);
            const float sk = warp_sum(pw.y * merge_scale(pw.x, mk));
            // Refill the consumed stage with the row `stages` iterations ahead.
            if (tid == 0 && copies && issued == it + L.stages &&
                unit + (it + L.stages) * nunits < M)
                issue(issued++);
            if constexpr (CLUSTER) {
                // Publish (mk, sk) into slot [it&1][rank] of every block of the
                // cluster; each store completes 16 bytes on the receiver's
                // exchange barrier for this parity.
                const int p = (int)(it & 1);
                if (tid == 0) mbar_expect_tx(xbar0 + 8u * p, (uint32_t)csize * 16u);
                if (lane < csize) {
                    const uint32_t slot = smem_addr(xch + p * kMaxCluster + rank);
                    st_async_f4(map_to_rank(slot, lane), make_float4(mk, sk, 0.0f, 0.0f),
                                map_to_rank(xbar0 + 8u * p, lane));
                }
            } else {
                if (lane == 0) xch[0] = make_float4(mk, sk, 0.0f, 0.0f);
            }
        }

        // Row (M, S) from the published pair(s).
        float Mr, Sr;
        if constexpr (CLUSTER) {
            const int p = (int)(it & 1);
            if (!mbar_wait_bounded(xbar0 + 8u * p, (uint32_t)((it >> 1) & 1), timeout_ns)) {
                local_fail = true;  // a peer stopped; the next block barrier stops us
                continue;
            }
            const float4 pk = lane < csize ? xch[p * kMaxCluster + lane]
                                           : make_float4(neg_inf(), 0.0f, 0.0f, 0.0f);
            Mr = warp_max(pk.x);
            Sr = warp_sum(pk.y * merge_scale(pk.x, Mr));
        } else {
            __syncthreads();
            const float4 pk = xch[0];
            Mr = pk.x;
            Sr = pk.y;
        }

        const float f = merge_scale(m_w, Mr) * final_rcp(Mr, Sr);
        T* rout = out + r * ld_out + v0 * VEC;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + NT * k;
            if (idx < cnt) {
                float y[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) y[e] = v[k][e] * f;
                stg_stream(rout + (int64_t)idx * VEC, Elem<T>::pack(y));
            }
        }
    }

    if (tid == 0) {
        if (local_fail) atomicOr(err, 1u);
        // Drain copies still in flight (only after a failure), bounded.
        for (int64_t j = confirmed; j < issued; ++j)
            mbar_wait_bounded(bar0 + 8u * (uint32_t)(j % L.stages), (uint32_t)((j / L.stages) & 1),
                              timeout_ns);
    }
    // No block of the cluster leaves while a peer may still store into it.
    if constexpr (CLUSTER) cluster_sync_all();
}

template <typename T, int KV, bool CLUSTER>
cudaError_t launch_kv(const Problem& p, int csize, const SmemLayout& L) {
    auto kern = tma_rows_kernel<T, kTmaThreads, KV, CLUSTER>;
    const void* fn = reinterpret_cast<const void*>(kern);
    const size_t smem = L.total();
    cudaError_t e = ensure_smem_limit(fn, smem, csize > 8);
    if (e != cudaSuccess) return e;
    const T* in = static_cast<const T*>(p.in);
    T* out = static_cast<T*>(p.out);
    if constexpr (!CLUSTER) {
        const int per_sm = blocks_per_sm(fn, kTmaThreads, smem);
        if (per_sm <= 0) return cudaErrorInvalidConfiguration;
        const int64_t cap = (int64_t)per_sm * p.dev->sm_count;
        const unsigned grid = (unsigned)(p.M < cap ? p.M : cap);
        kern<<<grid, kTmaThreads, smem, p.stream>>>(in, out, p.M, p.N, p.ld_in, p.ld_out, 1, L,
                                                    p.dev->err, p.timeout_ns, p.flags);
        return cudaGetLastError();
    } else {
        const int nclusters = max_active_clusters(fn, kTmaThreads, smem, csize);
        if (nclusters <= 0) return cudaErrorInvalidConfiguration;
        const int64_t units = p.M < nclusters ? p.M : nclusters;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(units * csize), 1, 1);
        cfg.blockDim = dim3(kTmaThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = p.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)csize;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, in, out, p.M, p.N, p.ld_in, p.ld_out, csize, L,
                               p.dev->err, p.timeout_ns, p.flags);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
}

template <typename T, bool CLUSTER>
cudaError_t launch_typed(const Problem& p, int csize) {
    constexpr int VEC = Elem<T>::kVec;
    const int64_t nvec = p.N / VEC;
    const int64_t per = (nvec + csize - 1) / csize;  // vectors per block
    SmemLayout L;
    L.stage_bytes = (uint32_t)(((per * 16) + 127) / 128 * 128);
    int stages = (int)((CLUSTER ? SR_CLUSTER_STAGE_BUDGET : SR_TMA_STAGE_BUDGET) / L.stage_bytes);
    stages = stages < 2 ? 2 : (stages > SR_TMA_MAX_STAGES ? SR_TMA_MAX_STAGES : stages);
    L.stages = stages;
    if ((int64_t)L.total() > p.dev->smem_optin) return cudaErrorInvalidValue;
    const int64_t kv = (per + kTmaThreads - 1) / kTmaThreads;
    if (kv <= 1) return launch_kv<T, 1, CLUSTER>(p, csize, L);
    if (kv <= 2) return launch_kv<T, 2, CLUSTER>(p, csize, L);
    if (kv <= 4) return launch_kv<T, 4, CLUSTER>(p, csize, L);
    if (kv <= 8) return launch_kv<T, 8, CLUSTER>(p, csize, L);
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
