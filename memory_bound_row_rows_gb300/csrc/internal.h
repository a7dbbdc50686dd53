// Host-side interface between the C ABI (api.cu) and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "device.cuh"

namespace sr {

enum : int { kF32 = 0, kBF16 = 1, kF16 = 2 };

// Debug flags for the bounded-wait test hooks: issue no bulk copies; (SPLIT
// plan, split.h) count no block in.
constexpr int kFlagNoCopy = 1;
constexpr int kFlagNoArrive = 2;

// Rows up to this many elements run one warp per row (64 values per lane).
constexpr int64_t kWarpMaxN = 2048;
// Aligned rows of at least this many 16-byte vectors run one block per row.
constexpr int64_t kRowMinVectors = 256;
// Largest row slice a thread block stages in shared memory (CTA plan rows,
// CLUSTER slices), and largest row a warp stages in its own ring (SMEM plan).
constexpr int64_t kSliceMaxBytes = 32 * 1024;
constexpr int64_t kSmemMaxRowBytes = 32 * 1024;
// Preferred CLUSTER slice: smaller slices mean fewer registers per thread and
// more blocks per SM; clusters grow up to kMaxCluster before slices grow.
#ifndef SR_CLUSTER_SLICE_BYTES
#define SR_CLUSTER_SLICE_BYTES (32 * 1024)
#endif
// Largest cluster (non-portable size 16 needs an opt-in attribute).
constexpr int kMaxCluster = 16;

struct DeviceInfo {
    int id = -1;
    int sm_count = 0;
    int smem_optin = 0;    // max dynamic shared memory per block (opt-in)
    int smem_per_sm = 0;
    int l2_bytes = 0;
    unsigned int* err = nullptr;  // device address of the error word
};

// Masked softmax: in row r only the first valid(r) entries take part; the
// rest count as -inf, are never loaded (a 16-byte vector with no valid entry
// is skipped) and come out as zeros.
struct RowMask {
    const int32_t* lens = nullptr;  // device array of M valid lengths, or null
    int64_t period = 0;             // without lens: row r keeps r mod period + 1 entries
    __host__ __device__ bool active() const { return lens != nullptr || period > 0; }
    __device__ __forceinline__ int64_t valid(int64_t r, int64_t N) const {
        int64_t v = N;
        if (lens) {
            v = SR_READ_OK(lens + r, 4) ? lens[r] : 0;
        } else if (period > 0) {
            // 32-bit division when both fit: a 64-bit one costs as much as the
            // rest of a short row's work.
            if (r <= 0x7fffffff && period <= 0x7fffffff)
                v = (int64_t)((uint32_t)r % (uint32_t)period) + 1;
            else
                v = r % period + 1;
        }
        return v < 0 ? 0 : (v > N ? N : v);
    }
};

struct Problem {
    const void* in;
    void* out;
    int64_t M, N, ld_in, ld_out;
    int dtype;
    cudaStream_t stream;
    const DeviceInfo* dev;
    unsigned long long timeout_ns;
    int flags;
    RowMask mask = RowMask();
};

inline int elem_bytes(int dtype) { return dtype == kF32 ? 4 : 2; }

// True when every row start of `in` and `out` is 16-byte aligned and a row is
// a whole number of 16-byte vectors.
inline bool rows_vector_aligned(const void* in, const void* out, int64_t N, int64_t ld_in,
                                int64_t ld_out, int dtype) {
    const int64_t es = elem_bytes(dtype);
    return (reinterpret_cast<uintptr_t>(in) % 16 == 0) &&
           (reinterpret_cast<uintptr_t>(out) % 16 == 0) && ((ld_in * es) % 16 == 0) &&
           ((ld_out * es) % 16 == 0) && ((N * es) % 16 == 0);
}

// Cluster size for a row: the smallest power of two (at least `min_cluster`)
// whose slices fit SR_CLUSTER_SLICE_BYTES, else the smallest whose slices fit
// kSliceMaxBytes; 0 when the row is too wide (or too short to split).
inline int cluster_size_for(int64_t N, int dtype, int min_cluster) {
    const int64_t nvec = N * elem_bytes(dtype) / 16;
    for (int64_t limit : {(int64_t)SR_CLUSTER_SLICE_BYTES, kSliceMaxBytes}) {
        for (int c = min_cluster; c <= kMaxCluster; c *= 2) {
            const int64_t per = (nvec + c - 1) / c;
            if (per * 16 <= limit && nvec >= c) return c;
        }
    }
    return 0;
}

// The calling host thread's record of the last kernel it launched through the
// library (read back by softmax_rows_last_launch). launch_kernel calls it.
void note_launch(const void* func, dim3 grid, dim3 block, size_t smem, int cluster);
template <typename F>
inline void note_launch(F* func, dim3 grid, dim3 block, size_t smem = 0, int cluster = 1) {
    note_launch(reinterpret_cast<const void*>(func), grid, block, smem, cluster);
}

// How a kernel is launched: grid and block, dynamic shared memory, blocks per
// cluster and the cluster scheduling policy (-1: default). `cluster` is 0 for
// a kernel that uses no cluster features; a kernel that does (cluster
// barriers, distributed shared memory, st.async) passes its cluster size,
// 1 included, and is always launched with that cluster dimension.
// `cooperative`: every block of the grid must be resident at once (its
// blocks wait on one another); the launch fails instead of starting a grid
// the device cannot hold.
struct LaunchShape {
    dim3 grid;
    dim3 block;
    size_t smem = 0;
    int cluster = 0;
    int policy = -1;
    bool cooperative = false;
};

// Every kernel of the library is launched here. With SR_PDL the launch allows
// programmatic stream serialisation: the kernel may be scheduled while the
// previous kernel on the stream drains, and (SR_GRID_DEPENDENCY, the first
// statement of every kernel) waits for that kernel to complete and its
// memory to be visible before any global access of its own, so stream order
// holds exactly as without it; only the launch and the block dispatch
// overlap the previous kernel's tail. A cooperative launch goes without it:
// it starts once the previous kernel has completed.
template <typename... P, typename... A>
cudaError_t launch_kernel(void (*kern)(P...), const LaunchShape& ls, cudaStream_t stream,
                          A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = ls.grid;
    cfg.blockDim = ls.block;
    cfg.dynamicSmemBytes = ls.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[3];
    int n = 0;
    if (ls.cluster > 0) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)ls.cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (ls.cluster > 0 && ls.policy >= 0) {
        attr[n].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
        attr[n].val.clusterSchedulingPolicyPreference = (cudaClusterSchedulingPolicy)ls.policy;
        ++n;
    }
    if (ls.cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    } else if (SR_PDL) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)n;
    note_launch(kern, ls.grid, ls.block, ls.smem, ls.cluster > 0 ? ls.cluster : 1);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<A&&>(args)...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Resident blocks per SM for a kernel (cached per device).
int blocks_per_sm(const void* func, int threads, size_t smem);
// Resident clusters on the device for a cluster launch (cached per device).
int max_active_clusters(const void* func, int threads, size_t smem, int cluster);
// Raise a kernel's dynamic shared memory limit once per device.
cudaError_t ensure_smem_limit(const void* func, size_t smem, bool nonportable_cluster);

cudaError_t launch_warp(const Problem& p);
cudaError_t launch_tma(const Problem& p, int cluster);
cudaError_t launch_online(const Problem& p);
cudaError_t launch_smem(const Problem& p);
cudaError_t launch_row(const Problem& p);
// The copy ceiling: M rows of row_bytes from pitch ld_in to pitch ld_out (bytes).
cudaError_t launch_copy_rows(const void* in, void* out, int64_t M, int64_t row_bytes,
                             int64_t ld_in, int64_t ld_out, cudaStream_t stream, int sm_count);
// The two-input ceiling: out = a XOR b over M rows of row_bytes (pitches in bytes).
cudaError_t launch_copy_pair(const void* a, const void* b, void* out, int64_t M,
                             int64_t row_bytes, int64_t ld_a, int64_t ld_b, int64_t ld_out,
                             cudaStream_t stream);
bool row_plan_fits(int64_t N, int dtype);
int64_t host_workspace_bytes(int64_t M, int64_t N, int dtype);

int run_host(const void* h_in, void* h_out, int64_t M, int64_t N, int64_t ld_in, int64_t ld_out,
             int dtype, void* d_work, int64_t work_bytes, cudaStream_t stream,
             int (*launch)(const void*, void*, int64_t, int64_t, int64_t, int64_t, int,
                           cudaStream_t));

}  // namespace sr
