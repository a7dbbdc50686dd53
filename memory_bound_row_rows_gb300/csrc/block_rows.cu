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

// Threads per row: the power of two that gives each thread about
// SR_ROW_TARGET_KV 16-byte vectors, within [SR_ROW_MIN_THREADS, SR_ROW_MAX_THREADS].
#ifndef SR_ROW_TARGET_KV
#define SR_ROW_TARGET_KV 4
#endif
#ifndef SR_ROW_MIN_THREADS
#define SR_ROW_MIN_THREADS 64
#endif
#ifndef SR_ROW_MAX_THREADS
#define SR_ROW_MAX_THREADS 256
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

// One block per row, capped at the largest grid dimension; rows beyond it
// are walked with a grid stride.
template <typename T>
cudaError_t launch_grid(void (*kern)(const T*, T*, int64_t, int64_t, int64_t, int64_t, RowMask),
                        int nt, const Problem& p) {
    const int64_t cap = 0x7fffffff;
    const unsigned grid = (unsigned)(p.M < cap ? p.M : cap);
    kern<<<grid, nt, 0, p.stream>>>(static_cast<const T*>(p.in), static_cast<T*>(p.out), p.M,
                                    p.N, p.ld_in, p.ld_out, p.mask);
    return cudaGetLastError();
}

template <typename T, int NT, int KV>
cudaError_t launch_nt_kv(const Problem& p) {
    if (p.mask.active()) return launch_grid(block_rows_kernel<T, NT, KV, true>, NT, p);
    if (!rows_vector_aligned(p.in, p.out, p.N, p.ld_in, p.ld_out, p.dtype))
        return launch_grid(block_rows_kernel<T, NT, KV, false, true>, NT, p);
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

inline int row_threads(int64_t nvec) {
    int nt = SR_ROW_MIN_THREADS;
    while (nt < SR_ROW_MAX_THREADS && (int64_t)nt * SR_ROW_TARGET_KV < nvec) nt *= 2;
    return nt;
}

template <typename T>
cudaError_t launch_typed(const Problem& p) {
    constexpr int VEC = Elem<T>::kVec;
    const int64_t nvec = p.N / VEC;
    const int nt = row_threads(nvec);
    if constexpr (SR_ROW_MIN_THREADS <= 32) if (nt == 32) return launch_nt<T, 32>(p, nvec);
    if constexpr (SR_ROW_MIN_THREADS <= 64) if (nt == 64) return launch_nt<T, 64>(p, nvec);
    if (nt == 128) return launch_nt<T, 128>(p, nvec);
    if constexpr (SR_ROW_MAX_THREADS >= 256) if (nt == 256) return launch_nt<T, 256>(p, nvec);
    if constexpr (SR_ROW_MAX_THREADS >= 512) if (nt == 512) return launch_nt<T, 512>(p, nvec);
    return cudaErrorInvalidValue;
}

}  // namespace

// Rows the ROW plan takes (aligned ones): at most kRowMaxKV vectors per thread.
bool row_plan_fits(int64_t N, int dtype) {
    const int64_t nvec = N / (16 / elem_bytes(dtype));
    return nvec <= (int64_t)kRowMaxKV * row_threads(nvec);
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
