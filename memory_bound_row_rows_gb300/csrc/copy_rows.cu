// Row copy: the bandwidth ceiling the softmax kernels are measured against.
//
// The "Warpline" README (Ceilings) takes a measured device copy as the
// roofline's bandwidth denominator. This kernel moves exactly the bytes a
// row softmax moves -- M rows of row_bytes, read at one pitch and written at
// another -- with the same 16-byte streaming loads and stores as the softmax
// kernels and no arithmetic, so "as fast as a copy" can be checked on the
// same shapes and layouts. It is a measurement tool; no softmax path calls it.
//
// Work split: rows are cut into chunks of 32 lanes x kCopyUnroll 16-byte
// vectors; warps of a grid sized to fill every SM take chunks in turn, each
// lane issuing its kCopyUnroll loads before any store. Rows that are not
// 16-byte aligned (either pitch, either base, or the row length) are copied
// byte by byte in the same chunks.
#include "../../include/softmax_rows.h"
#include "device.cuh"
#include "internal.h"

namespace sr {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr int64_t kChunk = 32 * kCopyUnroll;  // units per warp chunk

template <bool VEC>
__global__ void __launch_bounds__(kCopyThreads)
    copy_rows_kernel(const char* __restrict__ in, char* __restrict__ out, int64_t M,
                     int64_t row_bytes, int64_t ld_in, int64_t ld_out) {
    SR_BOUNDS_BEGIN(::sr::bounds::matrix(in, M, ld_in, row_bytes, 1, false),
                    ::sr::bounds::matrix(out, M, ld_out, row_bytes, 1, true));
    const int lane = threadIdx.x & 31;
    const int64_t units = VEC ? row_bytes / 16 : row_bytes;
    const int64_t chunks = (units + kChunk - 1) / kChunk;
    const int64_t items = M * chunks;
    const int64_t warps = (int64_t)gridDim.x * (kCopyThreads / 32);
    for (int64_t it = ((int64_t)blockIdx.x * kCopyThreads + threadIdx.x) >> 5; it < items;
         it += warps) {
        const int64_t r = it / chunks;
        const int64_t c0 = (it - r * chunks) * kChunk + lane;
        const char* src = in + r * ld_in;
        char* dst = out + r * ld_out;
        if constexpr (VEC) {
            uint4 v[kCopyUnroll];
#pragma unroll
            for (int k = 0; k < kCopyUnroll; ++k) {
                const int64_t c = c0 + 32 * k;
                if (c < units) v[k] = ldg_stream(src + c * 16);
            }
#pragma unroll
            for (int k = 0; k < kCopyUnroll; ++k) {
                const int64_t c = c0 + 32 * k;
                if (c < units) stg_stream(dst + c * 16, v[k]);
            }
        } else {
            unsigned char b[kCopyUnroll];
#pragma unroll
            for (int k = 0; k < kCopyUnroll; ++k) {
                const int64_t c = c0 + 32 * k;
                if (c < units && SR_READ_OK(src + c, 1))
                    b[k] = (unsigned char)__ldg(reinterpret_cast<const unsigned char*>(src + c));
            }
#pragma unroll
            for (int k = 0; k < kCopyUnroll; ++k) {
                const int64_t c = c0 + 32 * k;
                if (c < units && SR_WRITE_OK(dst + c, 1)) dst[c] = (char)b[k];
            }
        }
    }
}

}  // namespace

cudaError_t launch_copy_rows(const void* in, void* out, int64_t M, int64_t row_bytes,
                             int64_t ld_in, int64_t ld_out, cudaStream_t stream, int sm_count) {
    const bool vec = reinterpret_cast<uintptr_t>(in) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(out) % 16 == 0 && row_bytes % 16 == 0 &&
                     ld_in % 16 == 0 && ld_out % 16 == 0;
    const void* fn = vec ? reinterpret_cast<const void*>(copy_rows_kernel<true>)
                         : reinterpret_cast<const void*>(copy_rows_kernel<false>);
    const int per_sm = blocks_per_sm(fn, kCopyThreads, 0);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    const int64_t units = vec ? row_bytes / 16 : row_bytes;
    const int64_t items = M * ((units + kChunk - 1) / kChunk);
    const int64_t need = (items + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
    const int64_t cap = (int64_t)per_sm * sm_count;
    const unsigned grid = (unsigned)(need < cap ? need : cap);
    const char* src = static_cast<const char*>(in);
    char* dst = static_cast<char*>(out);
    if (vec) {
        note_launch(copy_rows_kernel<true>, grid, kCopyThreads);
        copy_rows_kernel<true><<<grid, kCopyThreads, 0, stream>>>(src, dst, M, row_bytes, ld_in,
                                                                   ld_out);
    } else {
        note_launch(copy_rows_kernel<false>, grid, kCopyThreads);
        copy_rows_kernel<false><<<grid, kCopyThreads, 0, stream>>>(src, dst, M, row_bytes, ld_in,
                                                                    ld_out);
    }
    return cudaGetLastError();
}

}  // namespace sr
