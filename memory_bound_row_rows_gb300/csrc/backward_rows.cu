// Softmax backward: dx = y * (dy - sum_j y_j dy_j), row by row.
//
// "Measured optimization case studies" (Training: backward kernels through
// autograd): the softmax backward keeps the forward output y and forms
// y * (dy - sum(y * dy)), following the same row plans as the forward
// kernels. Per row that is one reduction (the dot product of y and dy) and
// one elementwise pass, which is the row-pair engine's shape (rowpair.cuh)
// with A = y, B = dy, C = dx. The dot product is held in FP32 (one FMA per
// element) and every dx is rounded once to the storage type. The
// algorithmic traffic is two reads and one write of the M x N elements.
#include "rowpair.cuh"

namespace sr {
namespace {

struct BackwardOp {
    static constexpr bool kBoundTeam = false;
    // Per-column data the op reads beside the two matrices: none.
    __device__ __forceinline__ const void* aux_base() const { return nullptr; }
    __device__ __forceinline__ void accumulate(float& acc, float y, float dy) const {
        acc = fmaf(y, dy, acc);
    }
    __device__ __forceinline__ float finish(float dot, int64_t) const { return dot; }
    template <int n>
    struct Aux {};  // no per-column data
    template <int n>
    __device__ __forceinline__ Aux<n> load_aux(int64_t) const { return {}; }
    template <int n>
    __device__ __forceinline__ void apply(const float* y, const float* dy, float dot,
                                          const Aux<n>&, float* dx) const {
#pragma unroll
        for (int e = 0; e < n; ++e) dx[e] = y[e] * (dy[e] - dot);
    }
};

}  // namespace

cudaError_t launch_backward(const rp::Args& p, const rp::Shape& sh) {
    const BackwardOp op;
    switch (p.dtype) {
        case kF32: return rp::launch<float>(op, p, sh);
        case kBF16: return rp::launch<__nv_bfloat16>(op, p, sh);
        case kF16: return rp::launch<__half>(op, p, sh);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sr
