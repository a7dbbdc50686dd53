// SPLIT plan: rows cut into chunks across many blocks, statistics through a
// workspace, two launches.
//
// The split plan of "Measured optimization case studies" (Wide rows): when
// there are fewer rows than SMs, one program per row cannot fill the GPU, so
// every row is split into chunks; the first kernel writes each chunk's
// statistics, and in the second every chunk merges its row's statistics
// itself and writes its part of the output. The statistics are online
// (max, sum) pairs merged with the same section's rule and its guard for
// chunks that are entirely -inf.
//
// stats_kernel: block (row r, chunk c) reduces its chunk to (m, s) with
//   s = sum exp(x - m) and stores it at ws[r * C + c].
// apply_kernel: block (row r, chunk c) merges ws[r * C .. r * C + C) into
//   the row's (M, S), rereads its chunk (from L2 for the few-row shapes this
//   plan is for) and writes exp(x - M) / S.
// The grid is (C, M): block x = chunk, y = row. Chunks are whole 16-byte
// vectors when rows are 16-byte aligned (VEC = 16 / sizeof(T)), else
// elements (VEC = 1).
#include <mutex>

#include "../../include/softmax_rows.h"
#include "device.cuh"
#include "internal.h"

namespace sr {
namespace {

constexpr int kSplitThreads = 256;
constexpr int kSplitNW = kSplitThreads / 32;

template <typename T, int VEC>
__device__ __forceinline__ void load_vec(const T* p, float* f) {
    if constexpr (VEC == 1) {
        f[0] = Elem<T>::load1(p);
    } else {
        Elem<T>::unpack(ldg_stream(p), f);
    }
}

// Block-wide online (max, sum) merge; every thread returns the result.
__device__ __forceinline__ void block_merge(float& m, float& s, float2* red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        merge_ms(m, s, m2, s2);
    }
    if (lane == 0) red[warp] = make_float2(m, s);
    __syncthreads();
    m = red[0].x;
    s = red[0].y;
#pragma unroll
    for (int w = 1; w < kSplitNW; ++w) merge_ms(m, s, red[w].x, red[w].y);
}

template <typename T, int VEC>
__global__ void __launch_bounds__(kSplitThreads)
    split_stats_kernel(const T* __restrict__ in, int64_t N, int64_t ld_in, int64_t chunk_units,
                       float2* __restrict__ ws) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, (int64_t)gridDim.y, ld_in, N),
                    SR_SPAN_OUT(ws, (int64_t)gridDim.x * gridDim.y * 8));
    __shared__ float2 red[kSplitNW];
    const int64_t r = blockIdx.y, c = blockIdx.x, C = gridDim.x;
    const int64_t units = N / VEC;  // VEC divides N when VEC > 1
    const int64_t u0 = c * chunk_units;
    const int64_t u1 = (u0 + chunk_units < units) ? u0 + chunk_units : units;
    const T* rin = in + r * ld_in;
    float m = neg_inf(), s = 0.0f;
    for (int64_t u = u0 + threadIdx.x; u < u1; u += kSplitThreads) {
        float f[VEC];
        load_vec<T, VEC>(rin + u * VEC, f);
        float cm = f[0];
#pragma unroll
        for (int e = 1; e < VEC; ++e) cm = fmaxf(cm, f[e]);
        const float mn = fmaxf(m, cm);
        const float shift = (mn == neg_inf()) ? 0.0f : mn;
        float cs = 0.0f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) cs += expf(f[e] - shift);
        s = s * merge_scale(m, mn) + cs;
        m = mn;
    }
    block_merge(m, s, red);
    if (threadIdx.x == 0 && SR_WRITE_OK(ws + r * C + c, 8)) ws[r * C + c] = make_float2(m, s);
}

template <typename T, int VEC>
__global__ void __launch_bounds__(kSplitThreads)
    split_apply_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t N, int64_t ld_in,
                       int64_t ld_out, int64_t chunk_units, const float2* __restrict__ ws) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, (int64_t)gridDim.y, ld_in, N),
                    SR_MAT_OUT(out, (int64_t)gridDim.y, ld_out, N),
                    SR_SPAN_IN(ws, (int64_t)gridDim.x * gridDim.y * 8));
    __shared__ float2 red[kSplitNW];
    const int64_t r = blockIdx.y, c = blockIdx.x, C = gridDim.x;
    // The row's (M, S) from all of its chunks' pairs.
    float m = neg_inf(), s = 0.0f;
    for (int64_t k = threadIdx.x; k < C; k += kSplitThreads) {
        const float2 q = SR_READ_OK(ws + r * C + k, 8) ? ws[r * C + k]
                                                       : make_float2(__int_as_float(0x7fc00000), 0.0f);
        merge_ms(m, s, q.x, q.y);
    }
    block_merge(m, s, red);
    const float rs = final_rcp(m, s);
    const float m_l2 = m * kLog2e;

    const int64_t units = N / VEC;
    const int64_t u0 = c * chunk_units;
    const int64_t u1 = (u0 + chunk_units < units) ? u0 + chunk_units : units;
    const T* rin = in + r * ld_in;
    T* rout = out + r * ld_out;
    for (int64_t u = u0 + threadIdx.x; u < u1; u += kSplitThreads) {
        float f[VEC];
        load_vec<T, VEC>(rin + u * VEC, f);
#pragma unroll
        for (int e = 0; e < VEC; ++e) f[e] = exp_shifted<T>(f[e], m, m_l2) * rs;
        if constexpr (VEC == 1) {
            Elem<T>::store1(rout + u, f[0]);
        } else {
            stg_stream(rout + u * VEC, Elem<T>::pack(f));
        }
    }
}

template <typename T, int VEC>
cudaError_t launch_vec(const Problem& p, const SplitShape& sh, float2* ws) {
    const dim3 grid((unsigned)sh.chunks, (unsigned)p.M, 1);
    const LaunchShape ls{grid, dim3(kSplitThreads)};
    const cudaError_t e = launch_kernel(split_stats_kernel<T, VEC>, ls, p.stream,
                                        static_cast<const T*>(p.in), p.N, p.ld_in, sh.chunk_units,
                                        ws);
    if (e != cudaSuccess) return e;
    return launch_kernel(split_apply_kernel<T, VEC>, ls, p.stream, static_cast<const T*>(p.in),
                         static_cast<T*>(p.out), p.N, p.ld_in, p.ld_out, sh.chunk_units,
                         static_cast<const float2*>(ws));
}

template <typename T>
cudaError_t launch_typed(const Problem& p, const SplitShape& sh, float2* ws) {
    if (sh.vec > 1) return launch_vec<T, 16 / sizeof(T)>(p, sh, ws);
    return launch_vec<T, 1>(p, sh, ws);
}

}  // namespace

// Chunking (host logic, the same on every device): about kSplitTargetBlocks
// blocks in total, chunks of at least kSplitMinUnits vectors (or elements),
// at most kSplitMaxChunks chunks per row.
SplitShape split_shape(int64_t M, int64_t N, int64_t ld_in, int64_t ld_out, int dtype,
                       const void* in, const void* out) {
    SplitShape sh;
    const bool vec = rows_vector_aligned(in, out, N, ld_in, ld_out, dtype);
    sh.vec = vec ? 16 / elem_bytes(dtype) : 1;
    const int64_t units = N / sh.vec;
    const int64_t target_blocks = kSplitTargetBlocks;
    int64_t chunks = M > 0 ? (target_blocks + M - 1) / M : 1;
    const int64_t max_chunks = (units + kSplitMinUnits - 1) / kSplitMinUnits;
    if (chunks > max_chunks) chunks = max_chunks;
    if (chunks > kSplitMaxChunks) chunks = kSplitMaxChunks;
    if (chunks < 1) chunks = 1;
    sh.chunk_units = (units + chunks - 1) / chunks;
    sh.chunks = (units + sh.chunk_units - 1) / sh.chunk_units;
    return sh;
}

// Rows go in batches of at most kSplitMaxGridRows (the grid's y dimension).
cudaError_t launch_split(const Problem& p, const SplitShape& sh, void* ws) {
    const int64_t es = elem_bytes(p.dtype);
    for (int64_t r0 = 0; r0 < p.M; r0 += kSplitMaxGridRows) {
        Problem q = p;
        q.M = (p.M - r0 < kSplitMaxGridRows) ? p.M - r0 : kSplitMaxGridRows;
        q.in = static_cast<const char*>(p.in) + r0 * p.ld_in * es;
        q.out = static_cast<char*>(p.out) + r0 * p.ld_out * es;
        float2* w = static_cast<float2*>(ws) + r0 * sh.chunks;
        cudaError_t e = cudaErrorInvalidValue;
        switch (p.dtype) {
            case kF32: e = launch_typed<float>(q, sh, w); break;
            case kBF16: e = launch_typed<__nv_bfloat16>(q, sh, w); break;
            case kF16: e = launch_typed<__half>(q, sh, w); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace sr

// ---------------------------------------------------------------------------
// softmax_rows_split_noalloc: the split plan with built-in scratch.
//
// For callers that must not allocate device memory at all: code that runs
// under a fixed memory budget reserved up front (inference servers, plugins
// living inside another framework's memory pool), code that may not change
// the device's memory footprint once it is running, and code called from
// places where a cudaMalloc would implicitly synchronise the device and
// stall other work. They pass only the input and the output; the
// statistics live in the array below, which is part of the library's device
// image: every GPU that loads the library holds it until the process exits.
// ---------------------------------------------------------------------------
namespace sr {
namespace {

// Room for this many (max, sum) pairs: M * chunks of a call must fit.
constexpr int64_t kNoAllocPairs = 65536;  // 512 KiB
static __device__ __align__(256) float2 g_noalloc_scratch[kNoAllocPairs];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64];  // the array's device address, per device, once set up

// Device address of the array on the current device (set up on first use,
// with that device current). In host code the array's name is only a
// stand-in, never a device address.
int noalloc_scratch(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SR_ECUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return SR_ECUDA;
        g_noalloc_addr[dev] = ptr;
    }
    *out = g_noalloc_addr[dev];
    return SR_OK;
}

}  // namespace
}  // namespace sr

extern "C" int softmax_rows_split_noalloc(const void* in, void* out, int64_t M, int64_t N,
                                          int64_t ld_in, int64_t ld_out, int dtype,
                                          sr_stream_t stream) {
    const int64_t need = softmax_rows_split_workspace_bytes(in, out, M, N, ld_in, ld_out, dtype);
    if (need < 0) return (int)-need;
    if (M == 0) return SR_OK;
    if (need > sr::kNoAllocPairs * (int64_t)sizeof(float2)) return SR_EINVAL;  // too big
    void* scratch = nullptr;
    const int st = sr::noalloc_scratch(&scratch);
    if (st != SR_OK) return st;
    // Nothing in the scratch has to start at zero: the first kernel writes
    // every pair the second one reads.
    return softmax_rows_split(in, out, M, N, ld_in, ld_out, dtype, scratch, need, stream);
}
