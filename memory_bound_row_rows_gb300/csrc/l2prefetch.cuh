// L2 prefetch by the bulk-copy engine, for the WIDE kernel, whose clusters
// prefetch the row a cluster will start about one wave of resident clusters
// later.
#pragma once

#include "device.cuh"

namespace sr {

// Bulk prefetch of `bytes` of global memory into L2 (multiple of 16, start
// 16-byte aligned) by the bulk-copy engine: no registers, no shared memory,
// nothing to wait for; later loads of those bytes hit L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
    if (!SR_READ_OK(p, bytes)) return;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Clusters of at least this many blocks prefetch one wave ahead (measured on
// GB300, cold L2: with 8-block clusters bf16 1024 x 131072 84.5 -> 82.6 µs and
// 82.5 -> 81.9 µs on two machines, with 16-block clusters f32 512 x 131072
// 88.2 -> 83.4 µs; 4-block clusters unchanged, 2-block clusters 0.5 % slower).
// The row-pair CLUSTER kernel does not prefetch: on the backward of f16
// 64 x 131072 (1.7 waves of 16-block clusters) it cost 5 %.
#ifndef SR_AHEAD_MIN_CLUSTER
#define SR_AHEAD_MIN_CLUSTER 4
#endif
constexpr int kAheadMinCluster = SR_AHEAD_MIN_CLUSTER;
// How far ahead, in quarter waves of resident clusters (measured on GB300,
// cold L2, bf16 1024 x 131072 / f32 512 x 131072, µs: none 84.2 / 87.5, half a
// wave 81.4 / 82.1, one wave 82.1 / 82.8, 1.5 waves 82.8 / 83.9, two waves
// 87.5 / 88.1).
#ifndef SR_WIDE_AHEAD_QUARTERS
#define SR_WIDE_AHEAD_QUARTERS 2
#endif

}  // namespace sr
