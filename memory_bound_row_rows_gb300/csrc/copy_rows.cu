// Row copy: the bandwidth ceiling the softmax kernels are measured against.
//
// The "Warpline" README (Ceilings) takes a measured device copy as the
// roofline's bandwidth denominator. This kernel moves exactly the bytes a
// row softmax moves -- M rows of row_bytes, read at one pitch and written at
// another -- with the same 16-byte streaming loads and stores as the softmax
// kernels and no arithmetic, so "as fast as a copy" can be checked on the
// same shapes and layouts. It is a measurement tool; no softmax path calls it.
//
// Work split: the rows' 16-byte vectors are numbered row by row and cut into
// tiles of kCopyThreads x kCopyUnroll vectors, one tile per block of a grid
// with a block per tile (the hardware starts a new block as one retires, as
// in the ROW softmax); each thread issues its kCopyUnroll loads before any
// store. Rows that are not 16-byte aligned (either pitch, either base, or the
// row length) are copied byte by byte in the same tiles.
#include "../../include/softmax_rows.h"
#include "device.cuh"
#include "internal.h"

namespace sr {
namespace {

constexpr int kCopyThreads = 64;
constexpr int kCopyUnroll = 4;
constexpr int64_t kTile = (int64_t)kCopyThreads * kCopyUnroll;  // units per block

// Unit u of the numbering -> (row, unit within the row); 32-bit division when
// the numbering fits in 31 bits.
template <typename I>
__device__ __forceinline__ void split_unit(I u, I per_row, int64_t& r, int64_t& c) {
    const I q = u / per_row;
    r = (int64_t)q;
    c = (int64_t)(u - q * per_row);
}

template <bool VEC, typename I>
__global__ void __launch_bounds__(kCopyThreads)
    copy_rows_kernel(const char* __restrict__ in, char* __restrict__ out, int64_t M,
                     int64_t row_bytes, int64_t ld_in, int64_t ld_out) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(::sr::bounds::matrix(in, M, ld_in, row_bytes, 1, false),
                    ::sr::bounds::matrix(out, M, ld_out, row_bytes, 1, true));
    const I per_row = (I)(VEC ? row_bytes / 16 : row_bytes);
    const I total = (I)M * per_row;
    for (int64_t b = blockIdx.x; b * kTile < (int64_t)total; b += gridDim.x) {
        const I base = (I)(b * kTile) + (I)threadIdx.x;
        if constexpr (VEC) {
            uint4 v[kCopyUnroll];
            int64_t r[kCopyUnroll], c[kCopyUnroll];
#pragma unroll
            for (int k = 0; k < kCopyUnroll; ++k) {
                const I u = base + (I)(kCopyThreads * k);
                split_unit<I>(u, per_row, r[k], c[k]);
                if (u < total) v[k] = ldg_stream(in + r[k] * ld_in + c[k] * 16);
            }
#pragma unroll
            for (int k = 0; k < kCopyUnroll; ++k) {
                const I u = base + (I)(kCopyThreads * k);
                if (u < total) stg_stream(out + r[k] * ld_out + c[k] * 16, v[k]);
            }
        } else {
            unsigned char v[kCopyUnroll];
            int64_t r[kCopyUnroll], c[kCopyUnroll];
#pragma unroll
            for (int k = 0; k < kCopyUnroll; ++k) {
                const I u = base + (I)(kCopyThreads * k);
                split_unit<I>(u, per_row, r[k], c[k]);
                const char* p = in + r[k] * ld_in + c[k];
                if (u < total && SR_READ_OK(p, 1))
                    v[k] = (unsigned char)__ldg(reinterpret_cast<const unsigned char*>(p));
            }
#pragma unroll
            for (int k = 0; k < kCopyUnroll; ++k) {
                const I u = base + (I)(kCopyThreads * k);
                char* p = out + r[k] * ld_out + c[k];
                if (u < total && SR_WRITE_OK(p, 1)) *p = (char)v[k];
            }
        }
    }
}

template <bool VEC, typename I>
cudaError_t launch_copy(const char* in, char* out, int64_t M, int64_t row_bytes, int64_t ld_in,
                        int64_t ld_out, cudaStream_t stream) {
    const int64_t units = M * (VEC ? row_bytes / 16 : row_bytes);
    const int64_t need = (units + kTile - 1) / kTile;
    const unsigned grid = (unsigned)(need < 0x7fffffff ? need : 0x7fffffff);
    return launch_kernel(copy_rows_kernel<VEC, I>, LaunchShape{dim3(grid), dim3(kCopyThreads)},
                         stream, in, out, M, row_bytes, ld_in, ld_out);
}

}  // namespace

cudaError_t launch_copy_rows(const void* in, void* out, int64_t M, int64_t row_bytes,
                             int64_t ld_in, int64_t ld_out, cudaStream_t stream, int sm_count) {
    (void)sm_count;
    const bool vec = reinterpret_cast<uintptr_t>(in) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(out) % 16 == 0 && row_bytes % 16 == 0 &&
                     ld_in % 16 == 0 && ld_out % 16 == 0;
    const char* src = static_cast<const char*>(in);
    char* dst = static_cast<char*>(out);
    // 32-bit unit numbers while the last unit of the last tile fits.
    const int64_t units = M * (vec ? row_bytes / 16 : row_bytes);
    const bool narrow = units + kTile < 0x7fffffff;
    if (vec)
        return narrow ? launch_copy<true, int32_t>(src, dst, M, row_bytes, ld_in, ld_out, stream)
                      : launch_copy<true, int64_t>(src, dst, M, row_bytes, ld_in, ld_out, stream);
    return narrow ? launch_copy<false, int32_t>(src, dst, M, row_bytes, ld_in, ld_out, stream)
                  : launch_copy<false, int64_t>(src, dst, M, row_bytes, ld_in, ld_out, stream);
}

}  // namespace sr
