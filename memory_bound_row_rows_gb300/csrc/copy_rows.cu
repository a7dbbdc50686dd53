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
// store. Rows whose starts are not 16-byte aligned but sit at the same offset
// from a 16-byte boundary in the input and the output (equal base offsets
// and equal pitches modulo 16) are copied as a head of up to 15 bytes, whole
// 16-byte vectors and a tail; other unaligned rows byte by byte.
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

// How a row is cut into units: whole 16-byte vectors (aligned rows), bytes,
// or (co-aligned rows) a head, vectors and a tail: unit 0 of a row copies the
// bytes before its first 16-byte boundary, unit s >= 1 the vector at byte
// head + 16 (s - 1), or the bytes left at the end of the row.
enum CopyMode { kCopyVec = 0, kCopyBytes = 1, kCopyCoaligned = 2 };

template <int MODE>
__host__ __device__ __forceinline__ int64_t copy_units_per_row(int64_t row_bytes) {
    return MODE == kCopyVec ? row_bytes / 16 : MODE == kCopyBytes ? row_bytes : row_bytes / 16 + 2;
}

__device__ __forceinline__ void copy_bytes(const char* src, char* dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i)
        if (SR_READ_OK(src + i, 1) && SR_WRITE_OK(dst + i, 1))
            dst[i] = (char)__ldg(reinterpret_cast<const unsigned char*>(src + i));
}

template <int MODE, typename I>
__global__ void __launch_bounds__(kCopyThreads)
    copy_rows_kernel(const char* __restrict__ in, char* __restrict__ out, int64_t M,
                     int64_t row_bytes, int64_t ld_in, int64_t ld_out) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(::sr::bounds::matrix(in, M, ld_in, row_bytes, 1, false),
                    ::sr::bounds::matrix(out, M, ld_out, row_bytes, 1, true));
    const I per_row = (I)copy_units_per_row<MODE>(row_bytes);
    const I total = (I)M * per_row;
    for (int64_t b = blockIdx.x; b * kTile < (int64_t)total; b += gridDim.x) {
        const I base = (I)(b * kTile) + (I)threadIdx.x;
        if constexpr (MODE == kCopyVec) {
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
        } else if constexpr (MODE == kCopyCoaligned) {
            uint4 v[kCopyUnroll];
            int64_t src[kCopyUnroll], dst[kCopyUnroll], n[kCopyUnroll];
            bool whole[kCopyUnroll];  // a 16-byte vector (else n[k] bytes)
#pragma unroll
            for (int k = 0; k < kCopyUnroll; ++k) {
                const I u = base + (I)(kCopyThreads * k);
                int64_t r, c;
                split_unit<I>(u, per_row, r, c);
                const int64_t ri = r * ld_in, ro = r * ld_out;
                int64_t head = (16 - (int64_t)(reinterpret_cast<uintptr_t>(in + ri) & 15)) & 15;
                if (head > row_bytes) head = row_bytes;
                const int64_t off = c == 0 ? 0 : head + 16 * (c - 1);
                const int64_t end = c == 0 ? head : (off + 16 < row_bytes ? off + 16 : row_bytes);
                n[k] = (u < total && end > off) ? end - off : 0;
                src[k] = ri + off;
                dst[k] = ro + off;
                whole[k] = n[k] == 16 && c > 0;
                if (whole[k]) v[k] = ldg_stream(in + src[k]);
            }
#pragma unroll
            for (int k = 0; k < kCopyUnroll; ++k) {
                if (whole[k]) stg_stream(out + dst[k], v[k]);
                else if (n[k] > 0) copy_bytes(in + src[k], out + dst[k], n[k]);
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

// The two-input ceiling of the row-pair operations (two matrices read, one
// written): out = a XOR b, byte for byte, in the same tiles; 16-byte vectors
// when every base and pitch and the row length are multiples of 16, else bytes.
template <bool VEC, typename I>
__global__ void __launch_bounds__(kCopyThreads)
    copy_pair_kernel(const char* __restrict__ a, const char* __restrict__ b, char* __restrict__ out,
                     int64_t M, int64_t row_bytes, int64_t ld_a, int64_t ld_b, int64_t ld_out) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(::sr::bounds::matrix(a, M, ld_a, row_bytes, 1, false),
                    ::sr::bounds::matrix(b, M, ld_b, row_bytes, 1, false),
                    ::sr::bounds::matrix(out, M, ld_out, row_bytes, 1, true));
    const I per_row = (I)(VEC ? row_bytes / 16 : row_bytes);
    const I total = (I)M * per_row;
    for (int64_t blk = blockIdx.x; blk * kTile < (int64_t)total; blk += gridDim.x) {
        const I base = (I)(blk * kTile) + (I)threadIdx.x;
        int64_t r[kCopyUnroll], c[kCopyUnroll];
        if constexpr (VEC) {
            uint4 va[kCopyUnroll], vb[kCopyUnroll];
#pragma unroll
            for (int k = 0; k < kCopyUnroll; ++k) {
                const I u = base + (I)(kCopyThreads * k);
                split_unit<I>(u, per_row, r[k], c[k]);
                if (u < total) {
                    va[k] = ldg_stream(a + r[k] * ld_a + c[k] * 16);
                    vb[k] = ldg_stream(b + r[k] * ld_b + c[k] * 16);
                }
            }
#pragma unroll
            for (int k = 0; k < kCopyUnroll; ++k) {
                const I u = base + (I)(kCopyThreads * k);
                if (u < total)
                    stg_stream(out + r[k] * ld_out + c[k] * 16,
                               make_uint4(va[k].x ^ vb[k].x, va[k].y ^ vb[k].y, va[k].z ^ vb[k].z,
                                          va[k].w ^ vb[k].w));
            }
        } else {
#pragma unroll
            for (int k = 0; k < kCopyUnroll; ++k) {
                const I u = base + (I)(kCopyThreads * k);
                split_unit<I>(u, per_row, r[k], c[k]);
                const char* pa = a + r[k] * ld_a + c[k];
                const char* pb = b + r[k] * ld_b + c[k];
                char* po = out + r[k] * ld_out + c[k];
                if (u < total && SR_READ_OK(pa, 1) && SR_READ_OK(pb, 1) && SR_WRITE_OK(po, 1))
                    *po = (char)(__ldg(reinterpret_cast<const unsigned char*>(pa)) ^
                                 __ldg(reinterpret_cast<const unsigned char*>(pb)));
            }
        }
    }
}

template <bool VEC, typename I>
cudaError_t launch_pair(const char* a, const char* b, char* out, int64_t M, int64_t row_bytes,
                        int64_t ld_a, int64_t ld_b, int64_t ld_out, cudaStream_t stream) {
    const int64_t units = M * (VEC ? row_bytes / 16 : row_bytes);
    const int64_t need = (units + kTile - 1) / kTile;
    const unsigned grid = (unsigned)(need < 0x7fffffff ? need : 0x7fffffff);
    return launch_kernel(copy_pair_kernel<VEC, I>, LaunchShape{dim3(grid), dim3(kCopyThreads)},
                         stream, a, b, out, M, row_bytes, ld_a, ld_b, ld_out);
}

template <int MODE, typename I>
cudaError_t launch_copy(const char* in, char* out, int64_t M, int64_t row_bytes, int64_t ld_in,
                        int64_t ld_out, cudaStream_t stream) {
    const int64_t units = M * copy_units_per_row<MODE>(row_bytes);
    const int64_t need = (units + kTile - 1) / kTile;
    const unsigned grid = (unsigned)(need < 0x7fffffff ? need : 0x7fffffff);
    return launch_kernel(copy_rows_kernel<MODE, I>, LaunchShape{dim3(grid), dim3(kCopyThreads)},
                         stream, in, out, M, row_bytes, ld_in, ld_out);
}

template <int MODE>
cudaError_t launch_mode(const char* in, char* out, int64_t M, int64_t row_bytes, int64_t ld_in,
                        int64_t ld_out, cudaStream_t stream) {
    // 32-bit unit numbers while the last unit of the last tile fits.
    const int64_t units = M * copy_units_per_row<MODE>(row_bytes);
    if (units + kTile < 0x7fffffff)
        return launch_copy<MODE, int32_t>(in, out, M, row_bytes, ld_in, ld_out, stream);
    return launch_copy<MODE, int64_t>(in, out, M, row_bytes, ld_in, ld_out, stream);
}

}  // namespace

cudaError_t launch_copy_rows(const void* in, void* out, int64_t M, int64_t row_bytes,
                             int64_t ld_in, int64_t ld_out, cudaStream_t stream, int sm_count) {
    (void)sm_count;
    const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
    const bool vec = a % 16 == 0 && b % 16 == 0 && row_bytes % 16 == 0 && ld_in % 16 == 0 &&
                     ld_out % 16 == 0;
    const bool coaligned = a % 16 == b % 16 && ld_in % 16 == ld_out % 16;
    const char* src = static_cast<const char*>(in);
    char* dst = static_cast<char*>(out);
    if (vec) return launch_mode<kCopyVec>(src, dst, M, row_bytes, ld_in, ld_out, stream);
    if (coaligned)
        return launch_mode<kCopyCoaligned>(src, dst, M, row_bytes, ld_in, ld_out, stream);
    return launch_mode<kCopyBytes>(src, dst, M, row_bytes, ld_in, ld_out, stream);
}

cudaError_t launch_copy_pair(const void* a, const void* b, void* out, int64_t M,
                             int64_t row_bytes, int64_t ld_a, int64_t ld_b, int64_t ld_out,
                             cudaStream_t stream) {
    const bool vec = reinterpret_cast<uintptr_t>(a) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(b) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(out) % 16 == 0 && row_bytes % 16 == 0 &&
                     ld_a % 16 == 0 && ld_b % 16 == 0 && ld_out % 16 == 0;
    const char* pa = static_cast<const char*>(a);
    const char* pb = static_cast<const char*>(b);
    char* po = static_cast<char*>(out);
    const int64_t units = M * (vec ? row_bytes / 16 : row_bytes);
    const bool narrow = units + kTile < 0x7fffffff;
    if (vec)
        return narrow ? launch_pair<true, int32_t>(pa, pb, po, M, row_bytes, ld_a, ld_b, ld_out, stream)
                      : launch_pair<true, int64_t>(pa, pb, po, M, row_bytes, ld_a, ld_b, ld_out, stream);
    return narrow ? launch_pair<false, int32_t>(pa, pb, po, M, row_bytes, ld_a, ld_b, ld_out, stream)
                  : launch_pair<false, int64_t>(pa, pb, po, M, row_bytes, ld_a, ld_b, ld_out, stream);
}

}  // namespace sr
