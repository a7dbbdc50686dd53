// ONLINE plan: one thread block per row, two passes over global memory.
//
// The looped wide-row softmax of "Measured optimization case studies" (Wide
// rows): pass 1 walks the row keeping a per-thread online maximum and sum,
// rescaling the sum whenever the maximum grows, with the section's guard for
// lanes whose values so far are all -inf (shift by 0, keep a zero sum); the
// per-thread pairs are merged across the block with the same rule. Pass 2
// rereads the row (from L2 when it is still resident) and writes
// exp(x - M) / S. Scalar accesses, so any width, pitch and alignment work;
// this is the fallback for rows the other plans cannot take.
#include "device.cuh"
#include "internal.h"

namespace sr {
namespace {

constexpr int kOnlineThreads = 256;
constexpr int kChunk = 8;  // elements per thread per step of pass 1

template <typename T, bool MASKED>
__global__ void __launch_bounds__(kOnlineThreads)
    online_rows_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int64_t N,
                       int64_t ld_in, int64_t ld_out, RowMask mask) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, M, ld_in, N), SR_MAT_OUT(out, M, ld_out, N),
                    SR_SPAN_IN(mask.lens, M * 4));
    constexpr int NW = kOnlineThreads / 32;
    __shared__ float2 red[NW];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    for (int64_t r = blockIdx.x; r < M; r += gridDim.x) {
        const T* rin = in + r * ld_in;
        T* rout = out + r * ld_out;
        // Masked rows: entries at or past `valid` are -inf and never read.
        const int64_t valid = MASKED ? mask.valid(r, N) : N;

        // Pass 1: online (m, s) per thread over elements tid + NT*k.
        float m = neg_inf(), s = 0.0f;
        for (int64_t j0 = tid; j0 < valid; j0 += (int64_t)kOnlineThreads * kChunk) {
            float x[kChunk];
            float cm = neg_inf();
#pragma unroll
            for (int u = 0; u < kChunk; ++u) {
                const int64_t j = j0 + (int64_t)kOnlineThreads * u;
                x[u] = j < valid ? Elem<T>::load1(rin + j) : neg_inf();
                cm = fmaxf(cm, x[u]);
            }
            const float mn = fmaxf(m, cm);
            const float shift = (mn == neg_inf()) ? 0.0f : mn;
            float cs = 0.0f;
#pragma unroll
            for (int u = 0; u < kChunk; ++u) cs += expf(x[u] - shift);
            s = s * merge_scale(m, mn) + cs;
            m = mn;
        }

        // Merge across the warp, then across warps.
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
            merge_ms(m, s, m2, s2);
        }
        if (lane == 0) red[warp] = make_float2(m, s);
        __syncthreads();
        float Mr = red[0].x, Sr = red[0].y;
#pragma unroll
        for (int w = 1; w < NW; ++w) merge_ms(Mr, Sr, red[w].x, red[w].y);
        __syncthreads();  // red[] is reused by the next row

        // Pass 2: normalise and write.
        const float rs = final_rcp(Mr, Sr);
        for (int64_t j = tid; j < N; j += kOnlineThreads) {
            const float x = (!MASKED || j < valid) ? Elem<T>::load1(rin + j) : neg_inf();
            Elem<T>::store1(rout + j, expf(x - Mr) * rs);
        }
    }
}

template <typename T, bool MASKED>
cudaError_t launch_m(const Problem& p) {
    auto kern = online_rows_kernel<T, MASKED>;
    const int per_sm = blocks_per_sm(reinterpret_cast<const void*>(kern), kOnlineThreads, 0);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    const int64_t cap = (int64_t)per_sm * p.dev->sm_count;
    const unsigned grid = (unsigned)(p.M < cap ? p.M : cap);
    return launch_kernel(kern, LaunchShape{dim3(grid), dim3(kOnlineThreads)}, p.stream,
                         static_cast<const T*>(p.in), static_cast<T*>(p.out), p.M, p.N, p.ld_in,
                         p.ld_out, p.mask);
}

template <typename T>
cudaError_t launch_typed(const Problem& p) {
    if (p.mask.active()) return launch_m<T, true>(p);
    return launch_m<T, false>(p);
}

}  // namespace

cudaError_t launch_online(const Problem& p) {
    switch (p.dtype) {
        case kF32: return launch_typed<float>(p);
        case kBF16: return launch_typed<__nv_bfloat16>(p);
        case kF16: return launch_typed<__half>(p);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sr
