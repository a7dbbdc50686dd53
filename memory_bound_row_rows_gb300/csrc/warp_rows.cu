// WARP plan: one warp per row, the whole row resident in registers.
//
// The single-program fused softmax of "Triton: Writing GPU Kernels in Python,
// Measured" (Step 2) and of "Fused Softmax on GPU" (Triton, one block per
// row), mapped to one 32-lane warp: load the row (masked lanes read -inf),
// warp-shuffle max, exponentiate, warp-shuffle sum, scale, store. No shared
// memory and no block barriers, so a warp never waits for another one (the
// per-row barrier stalls the pages blame for PyTorch's slow rows). The grid
// is persistent ("Fused Softmax on GPU", Persistent Triton Kernel): blocks
// resident on every SM walk the rows with a grid stride.
//
// Lane l owns 16-byte vectors l, l+32, ..., so every load and store
// instruction of a warp covers 512 contiguous bytes. A row of up to
// 32 * KV * VEC elements fits; VEC == 1 is the scalar variant used when rows
// are not 16-byte aligned.
#include "device.cuh"
#include "internal.h"

namespace sr {
namespace {

constexpr int kWarpBlock = 256;  // 8 warps per block
// 1: persistent grid (resident blocks x SMs, grid-stride over rows);
// 0: one warp per row, the hardware scheduler hands out the rows.
#ifndef SR_WARP_PERSISTENT
#define SR_WARP_PERSISTENT 1
#endif

template <typename T, int VEC, int KV, bool MASKED>
__global__ void __launch_bounds__(kWarpBlock)
    warp_rows_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int N,
                     int64_t ld_in, int64_t ld_out, RowMask mask) {
    const int lane = threadIdx.x & 31;
    const int64_t first = ((int64_t)blockIdx.x * kWarpBlock + threadIdx.x) >> 5;
    const int64_t stride = ((int64_t)gridDim.x * kWarpBlock) >> 5;
    const int nvec = N / VEC;  // VEC divides N whenever VEC > 1

    for (int64_t r = first; r < M; r += stride) {
        const T* rin = in + r * ld_in;
        T* rout = out + r * ld_out;
        float v[KV][VEC];
        // Masked rows read only the vectors that hold valid entries.
        const int valid = MASKED ? (int)mask.valid(r, N) : N;

        // Row load (masked lanes read -inf, which adds exp(-inf) = 0 to the sum).
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = lane + 32 * k;
            const int rem = MASKED ? valid - idx * VEC : VEC;  // valid entries in this vector
            if (idx < nvec && (!MASKED || rem > 0)) {
                if constexpr (VEC == 1) {
                    v[k][0] = Elem<T>::load1(rin + idx);
                    if (MASKED && rem <= 0) v[k][0] = neg_inf();
                } else {
                    uint4 u = ldg_stream(rin + (int64_t)idx * VEC);
                    Elem<T>::unpack(u, v[k]);
                    if constexpr (MASKED) {
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            if (e >= rem) v[k][e] = neg_inf();
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = neg_inf();
            }
        }

        // Row max: per lane (one accumulator per vector slot), then butterfly.
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

        // Exponentiate in place and sum (VEC partial sums per lane, then a tree).
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
        const float s = warp_sum(sv[0]);
        const float rs = __frcp_rn(s);

        // Normalise, round once, store.
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = lane + 32 * k;
            if (idx < nvec) {
                if constexpr (VEC == 1) {
                    Elem<T>::store1(rout + idx, v[k][0] * rs);
                } else {
                    float y[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) y[e] = v[k][e] * rs;
                    stg_stream(rout + (int64_t)idx * VEC, Elem<T>::pack(y));
                }
            }
        }
    }
}

template <typename T, int VEC, int KV, bool MASKED>
cudaError_t launch_one_m(const Problem& p) {
    auto kern = warp_rows_kernel<T, VEC, KV, MASKED>;
    const int64_t warps_per_block = kWarpBlock / 32;
    const int64_t need = (p.M + warps_per_block - 1) / warps_per_block;
    int64_t cap = 0x7fffffff;
    if (SR_WARP_PERSISTENT) {
        const int per_sm = blocks_per_sm(reinterpret_cast<const void*>(kern), kWarpBlock, 0);
        if (per_sm <= 0) return cudaErrorInvalidConfiguration;
        cap = (int64_t)per_sm * p.dev->sm_count;
    }
    const unsigned grid = (unsigned)(need < cap ? need : cap);
    kern<<<grid, kWarpBlock, 0, p.stream>>>(static_cast<const T*>(p.in), static_cast<T*>(p.out),
                                            p.M, (int)p.N, p.ld_in, p.ld_out, p.mask);
    return cudaGetLastError();
}

template <typename T, int VEC, int KV>
cudaError_t launch_one(const Problem& p) {
    if (p.mask.active()) return launch_one_m<T, VEC, KV, true>(p);
    return launch_one_m<T, VEC, KV, false>(p);
}

// Vectors per lane: the smallest power of two that covers the row.
template <typename T, int VEC>
cudaError_t launch_vec(const Problem& p) {
    const int64_t nvec = p.N / VEC;
    const int64_t kv = (nvec + 31) / 32;
    if (kv <= 1) return launch_one<T, VEC, 1>(p);
    if (kv <= 2) return launch_one<T, VEC, 2>(p);
    if (kv <= 4) return launch_one<T, VEC, 4>(p);
    if (kv <= 8) return launch_one<T, VEC, 8>(p);
    if constexpr (32 * 8 * VEC < kWarpMaxN) {
        if (kv <= 16) return launch_one<T, VEC, 16>(p);
    }
    if constexpr (VEC == 1) {
        if (kv <= 32) return launch_one<T, VEC, 32>(p);
        if (kv <= 64) return launch_one<T, VEC, 64>(p);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_typed(const Problem& p) {
    if (rows_vector_aligned(p.in, p.out, p.N, p.ld_in, p.ld_out, p.dtype))
        return launch_vec<T, Elem<T>::kVec>(p);
    return launch_vec<T, 1>(p);
}

}  // namespace

cudaError_t launch_warp(const Problem& p) {
    switch (p.dtype) {
        case kF32: return launch_typed<float>(p);
        case kBF16: return launch_typed<__nv_bfloat16>(p);
        case kF16: return launch_typed<__half>(p);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sr
