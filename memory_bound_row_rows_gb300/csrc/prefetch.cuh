// L2 prefetch by the bulk-copy engine, for the kernels that stream a slice of
// a row twice (streamed WIDE, streamed row-pair CLUSTER).
#pragma once

#include "device.cuh"

namespace sr {

// Bulk prefetch of `bytes` of global memory into L2 (multiple of 16, start
// 16-byte aligned) by the bulk-copy engine, under an L2 eviction policy: no
// registers, no shared memory, nothing to wait for; later loads of those
// bytes hit L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes, uint64_t pol) {
    if (!SR_READ_OK(p, bytes)) return;
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p),
                 "r"(bytes), "l"(pol)
                 : "memory");
}

}  // namespace sr
