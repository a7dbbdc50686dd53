// Helpers for kernels that keep rows in registers as packed 16-byte vectors
// (WIDE, and the WARP plan's packed variant): a running maximum compared in the
// storage format, a re-widening that keeps the packed form live, and the
// hardware base-2 logarithm.
#pragma once

#include <type_traits>

#include "device.cuh"

namespace sr {

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Running maximum over packed vectors (NaN elements are ignored, as fmaxf
// does). 16-bit data is compared in pairs in its own format (exact, one
// instruction per two elements) and widened once at the end.
template <typename T>
struct VecMax {
    uint32_t m = sizeof(T) == 2 ? (std::is_same<T, __half>::value ? 0xFC00FC00u : 0xFF80FF80u)
                                : 0xFF800000u;  // -inf (pair)
    __device__ __forceinline__ void add(const uint4& u);
    __device__ __forceinline__ float get() const;
};

template <>
__device__ __forceinline__ void VecMax<float>::add(const uint4& u) {
    const float a = fmaxf(fmaxf(__uint_as_float(u.x), __uint_as_float(u.y)),
                          fmaxf(__uint_as_float(u.z), __uint_as_float(u.w)));
    m = __float_as_uint(fmaxf(__uint_as_float(m), a));
}
template <>
__device__ __forceinline__ float VecMax<float>::get() const { return __uint_as_float(m); }

template <typename H2>
__device__ __forceinline__ H2 as_h2(uint32_t w) {
    return *reinterpret_cast<H2*>(&w);
}
template <typename H2>
__device__ __forceinline__ uint32_t from_h2(H2 h) {
    return *reinterpret_cast<uint32_t*>(&h);
}

template <>
__device__ __forceinline__ void VecMax<__nv_bfloat16>::add(const uint4& u) {
    using H2 = __nv_bfloat162;
    const H2 a = __hmax2(__hmax2(as_h2<H2>(u.x), as_h2<H2>(u.y)),
                         __hmax2(as_h2<H2>(u.z), as_h2<H2>(u.w)));
    m = from_h2(__hmax2(as_h2<H2>(m), a));
}
template <>
__device__ __forceinline__ float VecMax<__nv_bfloat16>::get() const {
    const __nv_bfloat162 h = as_h2<__nv_bfloat162>(m);
    return fmaxf(__low2float(h), __high2float(h));
}

template <>
__device__ __forceinline__ void VecMax<__half>::add(const uint4& u) {
    using H2 = __half2;
    const H2 a = __hmax2(__hmax2(as_h2<H2>(u.x), as_h2<H2>(u.y)),
                         __hmax2(as_h2<H2>(u.z), as_h2<H2>(u.w)));
    m = from_h2(__hmax2(as_h2<H2>(m), a));
}
template <>
__device__ __forceinline__ float VecMax<__half>::get() const {
    const __half2 h = as_h2<__half2>(m);
    return fmaxf(__low2float(h), __high2float(h));
}

// Values of a packed vector, widened again for the output pass. The empty
// asm hides that they equal the first pass's, so the compiler keeps the
// packed vector (4 registers) across the exchange rather than its floats.
template <typename T>
__device__ __forceinline__ void unpack_again(const uint4& raw, float* f) {
    uint4 r = raw;
    if constexpr (sizeof(T) == 2) asm volatile("" : "+r"(r.x), "+r"(r.y), "+r"(r.z), "+r"(r.w));
    Elem<T>::unpack(r, f);
}

}  // namespace sr
