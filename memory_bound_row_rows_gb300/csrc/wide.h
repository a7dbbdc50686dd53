// Host-side interface of the WIDE plan (wide_rows.cu) for the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace sr {

// WIDE plan: clusters of `csize` blocks, `slice` 16-byte vectors per block,
// `kv` vectors per thread. SR_WIDE_KV: the most vectors a thread holds in
// registers. Aligned rows of exactly twice what the registers of a 16-block
// cluster hold (1 MiB) are `staged`: each thread holds 8 vectors in
// registers and 8 more in shared memory (kv = 16). Other wider aligned rows
// are `streamed`: each block reads its slice twice (the second time mostly
// from L2) instead of holding it.
#ifndef SR_WIDE_KV
#define SR_WIDE_KV 8
#endif
struct WideShape {
    int csize = 0;
    int kv = 0;
    int64_t slice = 0;
    bool streamed = false;
    bool staged = false;  // half of each thread's vectors held in shared memory
};
bool wide_shape(int64_t M, int64_t N, int dtype, int sm_count, WideShape* out);
bool wide_fits(const void* in, const void* out, int64_t N, int64_t ld_in, int64_t ld_out,
               int dtype);
cudaError_t launch_wide(const Problem& p);

}  // namespace sr
