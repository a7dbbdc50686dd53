// Host-side interface of the SPLIT plan (split_rows.cu) for the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace sr {

// SPLIT plan (split_rows.cu): `lanes` groups of `parts` blocks, each group
// taking one row at a time, each block one part of part_units units (16-byte
// vectors when vec > 1, else elements). The workspace holds a ring of
// kSplitRing steps of tagged (max, sum) pairs (16 bytes) for up to
// kSplitMaxBlocks blocks: a fixed size, whatever the problem.
// Steps between a row's pass 1 and its pass 2 (kSplitLag), and the ring of
// exchange slots, which must span 2 kSplitLag steps.
#ifndef SR_SPLIT_LAG
#define SR_SPLIT_LAG 2
#endif
constexpr int kSplitLag = SR_SPLIT_LAG;
constexpr int kSplitRing = 2 * kSplitLag;
constexpr int kSplitMaxBlocks = 4096;
constexpr int64_t kSplitMinUnits = 256;
constexpr int64_t kSplitMinSteps = 8;
constexpr int64_t kSplitWorkspaceBytes = (int64_t)kSplitRing * kSplitMaxBlocks * 16;
constexpr int kSplitThreadsPerBlock = 256;
struct SplitShape {
    int lanes = 1;
    int parts = 1;
    int64_t part_units = 1;
    int vec = 1;
};
SplitShape split_shape(int64_t M, int64_t N, int64_t ld_in, int64_t ld_out, int dtype,
                       const void* in, const void* out, int max_blocks, int64_t l2_bytes);
// The SPLIT kernel for a dtype and vector width, its dynamic shared memory
// and its threads per block (for occupancy queries).
const void* split_kernel(int dtype, int vec);
size_t split_smem(int vec);
int split_threads(int vec);
cudaError_t launch_split(const Problem& p, const SplitShape& sh, void* ws);

}  // namespace sr
