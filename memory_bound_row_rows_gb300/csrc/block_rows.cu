// ROW plan: one thread block per row, the row loaded straight into registers.
//
// The one-program-per-row fused softmax of "Fused Softmax on GPU" (Triton,
// one block per row) and of "Triton: Writing GPU Kernels in Python,
// Measured" (Step 2), written for sm_103a: every thread issues all of its
// 16-byte loads at once, the block reduces the max and the sum through
// shuffles and one shared-memory step each, and stores with 16-byte
// streaming stores. The grid has one block per row (not persistent): the
// hardware block scheduler hands rows to SMs as blocks retire, so a row that
// finishes late never holds back a whole statically assigned share, which is
// what sets the tail of a short kernel.
#include "device.cuh"
#include "internal.h"
#include "packed.cuh"

// Threads per row: the power of two that gives each thread about
// SR_ROW_TARGET_KV 16-byte vectors, within [SR_ROW_MIN_THREADS, the dtype's
// cap]. FP32 rows go up to 512 threads (64 KiB rows: on f32 4096 x 16384 this
// ran at 79.9 µs against 86.0 µs for the WIDE plan); 16-bit rows stop at 256
// threads (32 KiB), where WIDE is faster beyond.
// (8: f32 4096 x 4096 in 128-thread blocks ran at 20.3 against 20.6 µs with
// 4 vectors in 256-thread blocks, bf16 8192 x 8192 at 39.4 against 41.5 µs;
// GB300, cold L2.)
#ifndef SR_ROW_TARGET_KV
#define SR_ROW_TARGET_KV 8
#endif
#ifndef SR_ROW_MIN_THREADS
#define SR_ROW_MIN_THREADS 64
#endif
#ifndef SR_ROW_MAX_THREADS_F32
#define SR_ROW_MAX_THREADS_F32 512
#endif
#ifndef SR_ROW_MAX_THREADS_16
#define SR_ROW_MAX_THREADS_16 256
#endif
// Resident blocks per SM the packed 16-bit kernel is compiled for.
#ifndef SR_ROW_PACKED_MIN_BLOCKS
#define SR_ROW_PACKED_MIN_BLOCKS 4
#endif
constexpr int kRowMaxKV = 8;

namespace sr {
namespace {

// exp(x - m) for this kernel. FP32 data: the hardware ex2 of the difference
// (rounded once in FP32) times log2(e). Near the row maximum, where the
// outputs are large, the argument is small and the result's relative error is
// that of ex2 (about 2^-22); far from it the absolute error is far below the
// 1e-6 tolerance. Three instructions instead of the library expf's sequence:
// 2.5 % faster on 4096 x 4096 FP32, 15 % on 1024 x 3001. SR_ROW_EX2 = 0 keeps
// expf. 16-bit data as everywhere (one FMA and ex2).
#ifndef SR_ROW_EX2
#define SR_ROW_EX2 1
#endif
template <typename T>
__device__ __forceinline__ float row_exp(float x, float m, float m_l2) {
    if constexpr (Elem<T>::kAccurateExp && SR_ROW_EX2) {
        return ex2_approx((x - m) * kLog2e);
    } else {
        return exp_shifted<T>(x, m, m_l2);
    }
}

// SHIFTED (unmasked only): the input and output rows share their offset from
// a 16-byte boundary but are not aligned; each row is a head of fewer than
// VEC elements, 16-byte vectors and a tail of fewer than VEC elements, and the
// first threads of the block take the head and tail elements one each.
template <typename T, int NT, int KV, bool MASKED, bool SHIFTED = false>
__global__ void __launch_bounds__(NT)
    block_rows_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int64_t N,
                      int64_t ld_in, int64_t ld_out, RowMask mask) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, M, ld_in, N), SR_MAT_OUT(out, M, ld_out, N),
                    SR_SPAN_IN(mask.lens, M * 4));
    constexpr int VEC = Elem<T>::kVec;
    constexpr int NW = NT / 32;
    __shared__ float red_m[NW], red_s[NW];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    static_assert(!(MASKED && SHIFTED), "masked rows are aligned");

    for (int64_t r = blockIdx.x; r < M; r += gridDim.x) {
        const T* rin0 = in + r * ld_in;
        int head = 0;
        if constexpr (SHIFTED) {
            const int off = (int)((reinterpret_cast<uintptr_t>(rin0) & 15u) / sizeof(T));
            head = off ? VEC - off : 0;
            if (head > N) head = (int)N;
        }
        const T* rin = rin0 + head;  // the row's first 16-byte boundary
        const int nvec = (int)((N - head) / VEC);
        const int extra = (int)(N - (int64_t)nvec * VEC);  // head + tail elements
        float xe = neg_inf();
        int ce = -1;
        if constexpr (SHIFTED) {
            if (tid < extra) {
                ce = tid < head ? tid : head + nvec * VEC + (tid - head);
                xe = Elem<T>::load1(rin0 + ce);
            }
        }
        // Masked rows read only the vectors that hold valid entries (rows of
        // this plan are short enough for 32-bit element counts).
        const int valid = MASKED ? (int)mask.valid(r, N) : 0;
        float v[KV][VEC];
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + NT * k;
            const int rem = MASKED ? valid - idx * VEC : VEC;  // valid entries in this vector
            if (idx < nvec && (!MASKED || rem > 0)) {
                Elem<T>::unpack(ldg_stream(rin + (int64_t)idx * VEC), v[k]);
                if constexpr (MASKED) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        if (e >= rem) v[k][e] = neg_inf();
                }
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = neg_inf();
            }
        }
        float mx = v[0][0];
#pragma unroll
        for (int k = 0; k < KV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) mx = fmaxf(mx, v[k][e]);
        if constexpr (SHIFTED) mx = fmaxf(mx, xe);
        mx = warp_max(mx);
        if (lane == 0) red_m[warp] = mx;
        __syncthreads();
        float m = red_m[0];
#pragma unroll
        for (int w = 1; w < NW; ++w) m = fmaxf(m, red_m[w]);
        const float m_l2 = m * kLog2e;

        float sv[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) sv[e] = 0.0f;
#pragma unroll
        for (int k = 0; k < KV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                v[k][e] = row_exp<T>(v[k][e], m, m_l2);
                sv[e] += v[k][e];
            }
#pragma unroll
        for (int w = VEC / 2; w > 0; w >>= 1)
#pragma unroll
            for (int e = 0; e < w; ++e) sv[e] += sv[e + w];
        if constexpr (SHIFTED) {
            xe = row_exp<T>(xe, m, m_l2);  // 0 for a thread without an element
            sv[0] += xe;
        }
        const float sw = warp_sum(sv[0]);
        if (lane == 0) red_s[warp] = sw;
        __syncthreads();
        float s = red_s[0];
#pragma unroll
        for (int w = 1; w < NW; ++w) s += red_s[w];
        const float rs = __frcp_rn(s);

        T* rout0 = out + r * ld_out;
        T* rout = rout0 + head;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + NT * k;
            if (idx < nvec) {
                float y[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) y[e] = v[k][e] * rs;
                stg_stream(rout + (int64_t)idx * VEC, Elem<T>::pack(y));
            }
        }
        if constexpr (SHIFTED) {
            if (ce >= 0) Elem<T>::store1(rout0 + ce, xe * rs);
        }
    }
}

// Packed variant for aligned, unmasked 16-bit rows of more than 1024
// vectors (8 per thread at 256 threads). The unpacked kernel keeps 64 FP32
// values per thread there and needs 119 registers (2 blocks/SM). This one
// keeps the row as packed 16-byte vectors (4 registers per 8 elements), takes
// the maximum in the storage format, and computes the exponential twice: once
// for the sum and once for the output, with 1/S folded into the exponent
// (y = 2^(x log2(e) - (m log2(e) + log2(S))), one FMA and one ex2). The result
// is still rounded once, from FP32.
template <typename T, int NT, int KV>
__global__ void __launch_bounds__(NT, SR_ROW_PACKED_MIN_BLOCKS)
    block_packed_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int64_t N,
                        int64_t ld_in, int64_t ld_out) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, M, ld_in, N), SR_MAT_OUT(out, M, ld_out, N));
    constexpr int VEC = Elem<T>::kVec;
    constexpr int NW = NT / 32;
    static_assert(!Elem<T>::kAccurateExp, "16-bit data only");
    __shared__ float red_m[NW], red_s[NW];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nvec = (int)(N / VEC);
    for (int64_t r = blockIdx.x; r < M; r += gridDim.x) {
        const T* rin = in + r * ld_in;
        uint4 raw[KV];
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + NT * k;
            if (idx < nvec) raw[k] = ldg_stream(rin + (int64_t)idx * VEC);
        }
        VecMax<T> vm;
#pragma unroll
        for (int k = 0; k < KV; ++k)
            if (tid + NT * k < nvec) vm.add(raw[k]);
        const float mw = warp_max(vm.get());
        if (lane == 0) red_m[warp] = mw;
        __syncthreads();
        float m = red_m[0];
#pragma unroll
        for (int w = 1; w < NW; ++w) m = fmaxf(m, red_m[w]);
        const float m_l2 = m * kLog2e;
        float sa = 0.0f, sb = 0.0f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            if (tid + NT * k < nvec) {
                float f[VEC];
                Elem<T>::unpack(raw[k], f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float x = exp_shifted<T>(f[e], m, m_l2);
                    if (e & 1) sb += x; else sa += x;
                }
            }
        }
        const float sw = warp_sum(sa + sb);
        if (lane == 0) red_s[warp] = sw;
        __syncthreads();
        float s = red_s[0];
#pragma unroll
        for (int w = 1; w < NW; ++w) s += red_s[w];
        // An all -inf row gives -inf - -inf = NaN, as 0/0 does.
        const float c = fmaf(m, kLog2e, lg2_approx(s));
        T* rout = out + r * ld_out;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + NT * k;
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

// One block per row, capped at the largest grid dimension; rows beyond it
// are walked with a grid stride.
template <typename T>
cudaError_t launch_grid(void (*kern)(const T*, T*, int64_t, int64_t, int64_t, int64_t, RowMask),
                        int nt, const Problem& p) {
    const int64_t cap = 0x7fffffff;
    const unsigned grid = (unsigned)(p.M < cap ? p.M : cap);
    return launch_kernel(kern, LaunchShape{dim3(grid), dim3(nt)}, p.stream,
                         static_cast<const T*>(p.in), static_cast<T*>(p.out), p.M, p.N, p.ld_in,
                         p.ld_out, p.mask);
}

template <typename T, int NT, int KV>
cudaError_t launch_nt_kv(const Problem& p) {
    if (p.mask.active()) return launch_grid(block_rows_kernel<T, NT, KV, true>, NT, p);
    if (!rows_vector_aligned(p.in, p.out, p.N, p.ld_in, p.ld_out, p.dtype))
        return launch_grid(block_rows_kernel<T, NT, KV, false, true>, NT, p);
    if constexpr (!Elem<T>::kAccurateExp && KV == kRowMaxKV) {
        auto kern = block_packed_kernel<T, NT, KV>;
        const int64_t cap = 0x7fffffff;
        const unsigned grid = (unsigned)(p.M < cap ? p.M : cap);
        return launch_kernel(kern, LaunchShape{dim3(grid), dim3(NT)}, p.stream,
                             static_cast<const T*>(p.in), static_cast<T*>(p.out), p.M, p.N,
                             p.ld_in, p.ld_out);
    }
    return launch_grid(block_rows_kernel<T, NT, KV, false>, NT, p);
}

template <typename T, int NT>
cudaError_t launch_nt(const Problem& p, int64_t nvec) {
    const int64_t kv = (nvec + NT - 1) / NT;
    if (kv <= 1) return launch_nt_kv<T, NT, 1>(p);
    if (kv <= 2) return launch_nt_kv<T, NT, 2>(p);
    if (kv <= 4) return launch_nt_kv<T, NT, 4>(p);
    if (kv <= kRowMaxKV) return launch_nt_kv<T, NT, kRowMaxKV>(p);
    return cudaErrorInvalidValue;
}

inline int row_max_threads(int dtype) {
    return dtype == kF32 ? SR_ROW_MAX_THREADS_F32 : SR_ROW_MAX_THREADS_16;
}

// Up to 256 threads the block grows first (about SR_ROW_TARGET_KV vectors per
// thread), then each thread takes up to kRowMaxKV vectors, and only rows
// beyond 256 x kRowMaxKV vectors take 512 threads. On f32 8192-element rows,
// 256 x 8 ran at 76.8 µs and 512 x 4 at 89.3 µs.
inline int row_threads(int64_t nvec, int dtype) {
    int nt = SR_ROW_MIN_THREADS;
    while (nt < 256 && nt < row_max_threads(dtype) && (int64_t)nt * SR_ROW_TARGET_KV < nvec)
        nt *= 2;
    while (nt < row_max_threads(dtype) && (int64_t)nt * kRowMaxKV < nvec) nt *= 2;
    return nt;
}

template <typename T>
cudaError_t launch_typed(const Problem& p) {
    constexpr int VEC = Elem<T>::kVec;
    constexpr int kMaxNT = Elem<T>::kAccurateExp ? SR_ROW_MAX_THREADS_F32 : SR_ROW_MAX_THREADS_16;
    const int64_t nvec = p.N / VEC;
    const int nt = row_threads(nvec, p.dtype);
    if constexpr (SR_ROW_MIN_THREADS <= 32) if (nt == 32) return launch_nt<T, 32>(p, nvec);
    if constexpr (SR_ROW_MIN_THREADS <= 64) if (nt == 64) return launch_nt<T, 64>(p, nvec);
    if (nt == 128) return launch_nt<T, 128>(p, nvec);
    if constexpr (kMaxNT >= 256) if (nt == 256) return launch_nt<T, 256>(p, nvec);
    if constexpr (kMaxNT >= 512) if (nt == 512) return launch_nt<T, 512>(p, nvec);
    return cudaErrorInvalidValue;
}

}  // namespace

// Rows the ROW plan takes (aligned ones): at most kRowMaxKV vectors per thread.
bool row_plan_fits(int64_t N, int dtype) {
    const int64_t nvec = N / (16 / elem_bytes(dtype));
    return nvec <= (int64_t)kRowMaxKV * row_threads(nvec, dtype);
}

cudaError_t launch_row(const Problem& p) {
    switch (p.dtype) {
        case kF32: return launch_typed<float>(p);
        case kBF16: return launch_typed<__nv_bfloat16>(p);
        case kF16: return launch_typed<__half>(p);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sr
