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
// Aligned rows without a mask take a packed variant (warp_packed_kernel):
// the row stays in registers as packed 16-byte vectors and the exponential is
// computed twice, which doubles the rows in flight per SM. Its rows of at most
// 64 vectors are taken by 8 or 16 lanes each (two or four rows per warp).
//
// Lane l owns 16-byte vectors l, l+32, ..., so every load and store
// instruction of a warp covers 512 contiguous bytes. A row of up to
// 32 * KV * VEC elements fits; VEC == 1 is the scalar variant used when rows
// are not 16-byte aligned.
#include "device.cuh"
#include "internal.h"
#include "packed.cuh"

namespace sr {
namespace {

constexpr int kWarpBlock = 256;  // 8 warps per block
// 1: persistent grid (resident blocks x SMs, grid-stride over rows);
// 0: one warp per row, the hardware scheduler hands out the rows.
#ifndef SR_WARP_PERSISTENT
#define SR_WARP_PERSISTENT 1
#endif
// 1: aligned, unmasked rows take the packed variant; the resident blocks per
// SM it is compiled for.
#ifndef SR_WARP_PACKED
#define SR_WARP_PACKED 1
#endif
#ifndef SR_WARP_PACKED_MIN_BLOCKS
#define SR_WARP_PACKED_MIN_BLOCKS 6
#endif

template <typename T, int VEC, int KV, bool MASKED>
__global__ void __launch_bounds__(kWarpBlock)
    warp_rows_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int N,
                     int64_t ld_in, int64_t ld_out, RowMask mask) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, M, ld_in, N), SR_MAT_OUT(out, M, ld_out, N),
                    SR_SPAN_IN(mask.lens, M * 4));
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

// Resident blocks per SM the packed variant with 8 vectors per lane is
// compiled for (64 registers at 4).
#ifndef SR_WARP_PACKED_MIN_BLOCKS_KV8
#define SR_WARP_PACKED_MIN_BLOCKS_KV8 4
#endif
// Threads per block of the packed variant (the bounds above are for 256 and
// scale with it). Two-warp blocks retire and refill sooner than eight-warp
// blocks: bf16 16384 x 1000 ran at 13.0 against 13.5 µs, f32 32768 x 512 at
// 21.3 against 22.7 µs (GB300, cold L2); other shapes moved by under 1 %.
#ifndef SR_WARP_PACKED_BLOCK
#define SR_WARP_PACKED_BLOCK 64
#endif
constexpr int kPackedBlock = SR_WARP_PACKED_BLOCK;
constexpr int kPackedScale = 256 / SR_WARP_PACKED_BLOCK;

// Butterfly max / sum over aligned groups of W lanes (W = 32: the whole warp,
// in the same order as warp_max / warp_sum).
template <int W>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

template <int W>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Packed variant for aligned, unmasked rows: the row stays in registers as
// packed 16-byte vectors (4 registers per 16 bytes instead of one per element
// for 16-bit data), so about twice as many rows are in flight per SM; the
// exponential is computed twice, once for the sum and once for the output
// (16-bit data: 1/S folded into the exponent, one FMA and one ex2 per element),
// and the result is still rounded once, from FP32. LPR lanes take a row; the
// row loop is uniform over the warp so that every lane joins the shuffles.
template <typename T, int KV, int LPR>
__global__ void __launch_bounds__(kPackedBlock,
                                  kPackedScale * (KV <= 4   ? SR_WARP_PACKED_MIN_BLOCKS
                                                  : KV == 8 ? SR_WARP_PACKED_MIN_BLOCKS_KV8
                                                            : 2))
    warp_packed_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int N,
                       int64_t ld_in, int64_t ld_out) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, M, ld_in, N), SR_MAT_OUT(out, M, ld_out, N));
    constexpr int VEC = Elem<T>::kVec;
    constexpr int RPW = 32 / LPR;  // rows per warp
    const int lane = threadIdx.x & 31;
    const int sub = lane & (LPR - 1);
    const int64_t wfirst = ((int64_t)blockIdx.x * kPackedBlock + threadIdx.x) >> 5;
    const int64_t wstride = ((int64_t)gridDim.x * kPackedBlock) >> 5;
    const int nvec = N / VEC;
    for (int64_t w = wfirst; w * RPW < M; w += wstride) {
        const int64_t r = w * RPW + lane / LPR;
        const bool live = r < M;
        const T* rin = in + (live ? r : 0) * ld_in;
        uint4 raw[KV];
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = sub + LPR * k;
            if (live && idx < nvec) raw[k] = ldg_stream(rin + (int64_t)idx * VEC);
        }
        VecMax<T> vm;
#pragma unroll
        for (int k = 0; k < KV; ++k)
            if (live && sub + LPR * k < nvec) vm.add(raw[k]);
        const float m = group_max<LPR>(vm.get());
        const float m_l2 = m * kLog2e;
        float sa = 0.0f, sb = 0.0f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            if (live && sub + LPR * k < nvec) {
                float f[VEC];
                Elem<T>::unpack(raw[k], f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float x = exp_shifted<T>(f[e], m, m_l2);
                    if (e & 1) sb += x; else sa += x;
                }
            }
        }
        const float s = group_sum<LPR>(sa + sb);
        if (!live) continue;
        T* rout = out + r * ld_out;
        if constexpr (Elem<T>::kAccurateExp) {
            const float rs = __frcp_rn(s);
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int idx = sub + LPR * k;
                if (idx < nvec) {
                    float f[VEC];
                    unpack_again<T>(raw[k], f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) f[e] = expf(f[e] - m) * rs;
                    stg_stream(rout + (int64_t)idx * VEC, Elem<T>::pack(f));
                }
            }
        } else {
            // y = 2^(x log2(e) - (m log2(e) + log2(S))); an all -inf row gives
            // -inf - -inf = NaN, as 0/0 does.
            const float c = fmaf(m, kLog2e, lg2_approx(s));
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int idx = sub + LPR * k;
                if (idx < nvec) {
                    float f[VEC];
                    unpack_again<T>(raw[k], f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) f[e] = ex2_approx(fmaf(f[e], kLog2e, -c));
                    stg_stream(rout + (int64_t)idx * VEC, Elem<T>::pack(f));
                }
            }
        }
    }
}

template <typename T, int KV, int LPR>
cudaError_t launch_packed_lpr(const Problem& p) {
    auto kern = warp_packed_kernel<T, KV * 32 / LPR, LPR>;
    const int64_t rows_per_block = kPackedBlock / LPR;
    const int64_t need = (p.M + rows_per_block - 1) / rows_per_block;
    const int64_t cap = 0x7fffffff;
    const unsigned grid = (unsigned)(need < cap ? need : cap);
    return launch_kernel(kern, LaunchShape{dim3(grid), dim3(kPackedBlock)}, p.stream,
                         static_cast<const T*>(p.in), static_cast<T*>(p.out), p.M, (int)p.N,
                         p.ld_in, p.ld_out);
}

// No row loop: the hardware hands out rows as blocks retire (measured faster
// than a persistent grid for this variant). KV counts the vectors a lane
// holds when 32 lanes take a row. Rows of at most 64 vectors are shared by
// fewer lanes, so that each lane holds 4 vectors and every SM has more rows
// in flight. This needs rows enough for 4 blocks per SM at the narrower
// layout. Measured on GB300, cold L2: bf16 131072 x 256 went from 27.5 to
// 20.7 µs with 8 lanes per row.
template <typename T, int KV>
cudaError_t launch_packed(const Problem& p) {
    const int64_t min_blocks = 4 * (int64_t)p.dev->sm_count;
    if constexpr (KV == 1) {
        if (p.M >= min_blocks * (kWarpBlock / 8)) return launch_packed_lpr<T, 1, 8>(p);
    }
    if constexpr (KV == 2) {
        if (p.M >= min_blocks * (kWarpBlock / 16)) return launch_packed_lpr<T, 2, 16>(p);
    }
    return launch_packed_lpr<T, KV, 32>(p);
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
    return launch_kernel(kern, LaunchShape{dim3(grid), dim3(kWarpBlock)}, p.stream,
                         static_cast<const T*>(p.in), static_cast<T*>(p.out), p.M, (int)p.N,
                         p.ld_in, p.ld_out, p.mask);
}

template <typename T, int VEC, int KV>
cudaError_t launch_one(const Problem& p) {
    if (p.mask.active()) return launch_one_m<T, VEC, KV, true>(p);
    if constexpr (VEC > 1 && SR_WARP_PACKED) return launch_packed<T, KV>(p);
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
