// SMEM plan: one warp per row, the row staged in shared memory by bulk
// asynchronous copies into a ring that belongs to that warp alone.
//
// The fused single-program softmax of "Triton: Writing GPU Kernels in Python,
// Measured" (Step 2) and the persistent, prefetching grid of "Fused Softmax
// on GPU" (Persistent Triton Kernel, num_stages prefetch), rebuilt so that no
// warp ever waits for another: every warp is an independent pipeline. Lane 0
// issues cp.async.bulk copies of the warp's next rows into its own slots
// (completion on one mbarrier per slot, every wait bounded); the warp reduces
// the current row from shared memory and streams the result out with
// 16-byte stores. There is no block barrier in the row loop.
//
// Two variants:
//  * KV > 0 (rows of at most 32*KV vectors): the row is read once from shared
//    memory into registers and finished there, one exponential per element;
//  * KV == 0 (any aligned row that fits a slot): three passes over shared
//    memory: max; exp and sum; scale and store. FP32 rows keep e = exp(x - m)
//    in place of x, so each element is exponentiated once; 16-bit rows have
//    no room for FP32 values and recompute the exponential in the last pass.
//
// Grid: persistent, `warps_per_block` warps per block, blocks resident on
// every SM; warp g handles rows g, g + G, g + 2G, ... (G = total warps).
#include "device.cuh"
#include "internal.h"

namespace sr {
namespace {

template <typename T, int KV>
__global__ void __launch_bounds__(256)
    smem_rows_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int64_t N,
                     int64_t ld_in, int64_t ld_out, int slots, uint32_t slot_bytes,
                     unsigned int* err, unsigned long long timeout_ns, int flags) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, M, ld_in, N), SR_MAT_OUT(out, M, ld_out, N));
    constexpr int VEC = Elem<T>::kVec;
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const uint32_t base = smem_addr(smem);
    const uint32_t wslots = base + (uint32_t)(warp * slots) * slot_bytes;
    const uint32_t wbars = base + (uint32_t)(nw * slots) * slot_bytes + 8u * (uint32_t)(warp * slots);
    const int64_t first = (int64_t)blockIdx.x * nw + warp;
    const int64_t stride = (int64_t)gridDim.x * nw;
    const int nvec = (int)(N / VEC);
    const uint32_t bytes = (uint32_t)nvec * 16u;
    const bool copies = !(flags & kFlagNoCopy);

    if (lane == 0) {
        for (int s = 0; s < slots; ++s) mbar_init(wbars + 8u * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    int64_t issued = 0, confirmed = 0;  // lane 0's bookkeeping
    auto issue = [&](int64_t it) {
        const int s = (int)(it % slots);
        const T* src = in + (first + it * stride) * ld_in;
        mbar_expect_tx(wbars + 8u * s, bytes);
        bulk_g2s(wslots + (uint32_t)s * slot_bytes, src, bytes, wbars + 8u * s);
    };
    if (lane == 0 && copies)
        for (int s = 0; s < slots && first + s * stride < M; ++s) issue(issued++);

    bool failed = false;
    for (int64_t it = 0;; ++it) {
        const int64_t r = first + it * stride;
        if (r >= M) break;
        const int s = (int)(it % slots);
        const uint32_t slot = wslots + (uint32_t)s * slot_bytes;
        const bool ok = mbar_wait_bounded(wbars + 8u * s, (uint32_t)((it / slots) & 1), timeout_ns);
        if (!__all_sync(0xffffffffu, ok)) {
            failed = true;
            break;
        }
        if (lane == 0) confirmed = it + 1;
        T* rout = out + r * ld_out;

        if constexpr (KV > 0) {
            // Register-resident: one read of shared memory, one exp per element.
            float v[KV][VEC];
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int idx = lane + 32 * k;
                if (idx < nvec) {
                    Elem<T>::unpack(lds128(slot + 16u * idx), v[k]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) v[k][e] = neg_inf();
                }
            }
            __syncwarp();
            if (lane == 0 && copies && issued == it + slots && first + (it + slots) * stride < M)
                issue(issued++);  // the slot is consumed: refill it
            float mv[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) mv[e] = v[0][e];
#pragma unroll
            for (int k = 1; k < KV; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) mv[e] = fmaxf(mv[e], v[k][e]);
            float m = mv[0];
#pragma unroll
            for (int e = 1; e < VEC; ++e) m = fmaxf(m, mv[e]);
            m = warp_max(m);
            const float m_l2 = m * kLog2e;
            float sv[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) sv[e] = 0.0f;
#pragma unroll
            for (int k = 0; k < KV; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    v[k][e] = exp_shifted<T>(v[k][e], m, m_l2);
                    sv[e] += v[k][e];
                }
#pragma unroll
            for (int w = VEC / 2; w > 0; w >>= 1)
#pragma unroll
                for (int e = 0; e < w; ++e) sv[e] += sv[e + w];
            const float rs = __frcp_rn(warp_sum(sv[0]));
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int idx = lane + 32 * k;
                if (idx < nvec) {
                    float y[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) y[e] = v[k][e] * rs;
                    stg_stream(rout + (int64_t)idx * VEC, Elem<T>::pack(y));
                }
            }
        } else {
            // Three passes over shared memory. Pass 1: the row max.
            float mv[4] = {neg_inf(), neg_inf(), neg_inf(), neg_inf()};
            int idx = lane;
            for (; idx + 96 < nvec; idx += 128) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float f[VEC];
                    Elem<T>::unpack(lds128(slot + 16u * (idx + 32 * u)), f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) mv[u] = fmaxf(mv[u], f[e]);
                }
            }
            for (; idx < nvec; idx += 32) {
                float f[VEC];
                Elem<T>::unpack(lds128(slot + 16u * idx), f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) mv[0] = fmaxf(mv[0], f[e]);
            }
            const float m = warp_max(fmaxf(fmaxf(mv[0], mv[1]), fmaxf(mv[2], mv[3])));
            const float m_l2 = m * kLog2e;

            // Pass 2: e = exp(x - m) and its sum; FP32 rows store e in place.
            float sv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            auto exp_vec = [&](int i, float& acc) {
                float f[VEC];
                Elem<T>::unpack(lds128(slot + 16u * i), f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    f[e] = exp_shifted<T>(f[e], m, m_l2);
                    acc += f[e];
                }
                if constexpr (sizeof(T) == 4) {
                    const uint4 pk = Elem<T>::pack(f);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(slot + 16u * i),
                                 "r"(pk.x), "r"(pk.y), "r"(pk.z), "r"(pk.w)
                                 : "memory");
                }
            };
            for (idx = lane; idx + 96 < nvec; idx += 128) {
#pragma unroll
                for (int u = 0; u < 4; ++u) exp_vec(idx + 32 * u, sv[u]);
            }
            for (; idx < nvec; idx += 32) exp_vec(idx, sv[0]);
            const float rs = __frcp_rn(warp_sum((sv[0] + sv[1]) + (sv[2] + sv[3])));

            // Pass 3: scale, round once, store.
            for (idx = lane; idx < nvec; idx += 32) {
                float f[VEC];
                Elem<T>::unpack(lds128(slot + 16u * idx), f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    if constexpr (sizeof(T) == 4) {
                        f[e] = f[e] * rs;
                    } else {
                        f[e] = exp_shifted<T>(f[e], m, m_l2) * rs;
                    }
                }
                stg_stream(rout + (int64_t)idx * VEC, Elem<T>::pack(f));
            }
            // The slot was written through the generic proxy (FP32 in place);
            // order those writes before the bulk copy that refills it.
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && copies && issued == it + slots && first + (it + slots) * stride < M)
                issue(issued++);
        }
    }

    if (failed && lane == 0) {
        atomicOr(err, 1u);
        for (int64_t j = confirmed; j < issued; ++j)  // drain, bounded
            mbar_wait_bounded(wbars + 8u * (uint32_t)(j % slots), (uint32_t)((j / slots) & 1),
                              timeout_ns);
    }
}

// Tuning: bytes of rows each warp keeps in flight, and the shared memory a
// block may use (several blocks share an SM).
#ifndef SR_SMEM_WARP_INFLIGHT
#define SR_SMEM_WARP_INFLIGHT (12 * 1024)
#endif
#ifndef SR_SMEM_BLOCK_BUDGET
#define SR_SMEM_BLOCK_BUDGET (56 * 1024)
#endif
#ifndef SR_SMEM_MAX_WARPS
#define SR_SMEM_MAX_WARPS 4
#endif

template <typename T, int KV>
cudaError_t launch_kv(const Problem& p, uint32_t slot_bytes) {
    // Slots per warp: enough to keep ~SR_SMEM_WARP_INFLIGHT bytes in flight
    // beyond the row being reduced; warps per block: as many as fit the budget.
    int slots = 1 + (int)((SR_SMEM_WARP_INFLIGHT + slot_bytes - 1) / slot_bytes);
    slots = slots < 2 ? 2 : (slots > 8 ? 8 : slots);
    int nw = (int)(SR_SMEM_BLOCK_BUDGET / ((uint64_t)slots * (slot_bytes + 8)));
    nw = nw < 1 ? 1 : (nw > SR_SMEM_MAX_WARPS ? SR_SMEM_MAX_WARPS : nw);
    const size_t smem = (size_t)nw * slots * (slot_bytes + 8);
    if ((int64_t)smem > p.dev->smem_optin) return cudaErrorInvalidValue;
    auto kern = smem_rows_kernel<T, KV>;
    const void* fn = reinterpret_cast<const void*>(kern);
    cudaError_t e = ensure_smem_limit(fn, smem, false);
    if (e != cudaSuccess) return e;
    const int per_sm = blocks_per_sm(fn, nw * 32, smem);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    const int64_t need = (p.M + nw - 1) / nw;
    const int64_t cap = (int64_t)per_sm * p.dev->sm_count;
    const unsigned grid = (unsigned)(need < cap ? need : cap);
    return launch_kernel(kern, LaunchShape{dim3(grid), dim3(nw * 32), smem}, p.stream,
                         static_cast<const T*>(p.in), static_cast<T*>(p.out), p.M, p.N, p.ld_in,
                         p.ld_out, slots, slot_bytes, p.dev->err, p.timeout_ns, p.flags);
}

template <typename T>
cudaError_t launch_typed(const Problem& p) {
    constexpr int VEC = Elem<T>::kVec;
    const int64_t nvec = p.N / VEC;
    const uint32_t slot_bytes = (uint32_t)((nvec * 16 + 127) / 128 * 128);
    const int64_t kv = (nvec + 31) / 32;
    if (kv <= 1) return launch_kv<T, 1>(p, slot_bytes);
    if (kv <= 2) return launch_kv<T, 2>(p, slot_bytes);
    if (kv <= 4) return launch_kv<T, 4>(p, slot_bytes);
    if (kv <= 8) return launch_kv<T, 8>(p, slot_bytes);
    return launch_kv<T, 0>(p, slot_bytes);
}

}  // namespace

cudaError_t launch_smem(const Problem& p) {
    switch (p.dtype) {
        case kF32: return launch_typed<float>(p);
        case kBF16: return launch_typed<__nv_bfloat16>(p);
        case kF16: return launch_typed<__half>(p);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sr
