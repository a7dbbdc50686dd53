// SPLIT plan: every row cut into parts held by different thread blocks of one
// grid whose blocks are all resident together (a cooperative launch); the
// parts' statistics meet in a small caller-owned workspace. One launch.
//
// The split plan of "Measured optimization case studies" (Wide rows): when
// one program cannot take a whole row, the row is split across programs,
// each reduces its chunk to an online (max, sum) pair, and the pairs are
// merged with the same section's rule and its guard for chunks that are
// entirely -inf. Here a row may span any number of SMs, beyond the 16 blocks
// of a thread-block cluster, because the pairs travel through global memory.
//
// Schedule. The B = lanes x parts blocks form `lanes` groups of `parts`
// blocks; group g takes rows g, g + lanes, g + 2 lanes, ... in turn (its
// steps), block p of the group always the same part of the row. For step t a
// block
//   1. reads its part and reduces it to a pair (pass 1, loads marked to stay
//      in L2);
//   2. stores the pair, tagged with the step, in the workspace;
//   3. kLag steps later, merges the group's tagged pairs of step t (waiting,
//      bounded, for any not there yet) into the row's (M, S), and reads its
//      part again to write exp(x - M) / S (pass 2, loads marked for early
//      eviction).
// Pass 1 of step t + kLag and pass 2 of step t run in one sweep over the
// part, each step of the sweep issuing both rows' loads first, so that DRAM
// reads and writes overlap; kLag - 1 sweeps lie between storing a pair and
// needing the group's, which hides the exchange. The pass-2 read comes from
// L2: a group reads kLag more rows between a part's two reads, and the host
// picks `lanes` so that kLag + 1 rows per group fit in half of the L2. DRAM
// then sees each element read once and written once, whatever the row width.
//
// Workspace: slots[kRing][B], 16 bytes each; slot (t mod kRing, block) holds
// the block's pair of step t as two 8-byte words (max bits, t + 1) and (sum
// bits, t + 1), each stored and loaded as one relaxed 64-bit access, so a
// reader that finds its tag in both words holds that step's pair: no fence,
// no counter. The host zeroes the slots before the launch (tags start at 1).
// A block stores its pair for step t only after it has merged the pairs of
// step t - kLag, which every block of its group stored only after it had
// merged those of step t - 2 kLag: with kRing = 2 kLag slots no pair is
// overwritten while it may still be read.
//
// Two kernels run this schedule: the register sweep below for rows that are
// not 16-byte aligned (each thread's loads for a step of the sweep in
// registers), and for aligned rows a variant whose loads are 1-D bulk copies
// into a ring of shared memory fed by a producer warp (split_bulk_kernel),
// which keeps more bytes in flight than the registers can.
//
// Failure: a wait that expires sets the timeout bit of the error word; the
// block's threads leave together after the next barrier, writing nothing
// more, and the other blocks of the group then expire in turn. No block waits
// on shared memory of another block.
#include <mutex>
#include <type_traits>

#include "../../include/softmax_rows.h"
#include "device.cuh"
#include "internal.h"
#include "split.h"

namespace sr {

static_assert(kSplitLag != 2 || kSplitWorkspaceBytes == 262144, "the header documents this size");

namespace {

constexpr int kSplitThreads = kSplitThreadsPerBlock;
constexpr int kSplitNW = kSplitThreads / 32;
constexpr int kRing = kSplitRing;
constexpr int kLag = kSplitLag;  // pass 2 of step t runs kLag steps after its pass 1

// Units per thread and row in one step of a sweep (loads in flight).
#ifndef SR_SPLIT_UNROLL
#define SR_SPLIT_UNROLL 4
#endif
constexpr int kSplitUnroll = SR_SPLIT_UNROLL;

// Resident blocks per SM the register sweep is compiled for (bounds its
// registers). Measured on GB300 while the sweep also took aligned rows (cold
// L2, µs, 2 / 3 / 4 blocks per SM with 4 / 4 / 2 units per step): f32
// 32 x 4194304 272 / 327 / 300, bf16 128 x 524288 83 / 86 / 85, bf16
// 512 x 400008 251 / 249 / 236, f16 64 x 131072 38 / 46 / 48; 2 blocks per SM
// with 8 units per step 367 / 101 / 332 / 50.
#ifndef SR_SPLIT_MIN_BLOCKS
#define SR_SPLIT_MIN_BLOCKS 2
#endif

__device__ __forceinline__ uint64_t l2_keep() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_drop() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Loads through the read-only path with an L2 cache policy: one 16-byte
// vector, or one element.
__device__ __forceinline__ uint4 ld_vec(const void* p, uint64_t pol) {
    if (!SR_READ_OK(p, 16)) return make_uint4(0x7fc00000u, 0x7fc00000u, 0x7fc00000u, 0x7fc00000u);
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "l"(pol));
    return v;
}

template <typename T>
__device__ __forceinline__ float ld_one(const T* p, uint64_t pol) {
    if (!SR_READ_OK(p, sizeof(T))) return __int_as_float(0x7fc00000);
    if constexpr (sizeof(T) == 4) {
        float v;
        asm("ld.global.nc.L1::no_allocate.L2::cache_hint.f32 %0, [%1], %2;"
            : "=f"(v)
            : "l"(p), "l"(pol));
        return v;
    } else {
        unsigned short h;
        asm("ld.global.nc.L1::no_allocate.L2::cache_hint.b16 %0, [%1], %2;"
            : "=h"(h)
            : "l"(p), "l"(pol));
        if constexpr (std::is_same<T, __half>::value) return __half2float(__ushort_as_half(h));
        else return __uint_as_float(((uint32_t)h) << 16);
    }
}

// exp(x - m): for FP32 data the hardware ex2 of the FP32 difference times
// log2(e), for 16-bit data one FMA and ex2 (m_l2 = m * log2(e)), as in the
// ROW and WIDE plans.
template <typename T>
__device__ __forceinline__ float split_exp(float x, float m, float m_l2) {
    if constexpr (Elem<T>::kAccurateExp) {
        return ex2_approx((x - m) * kLog2e);
    } else {
        return exp_shifted<T>(x, m, m_l2);
    }
}

struct CtaBarrier {
    __device__ __forceinline__ static void sync() { __syncthreads(); }
};
struct ConsumerBarrier {
    __device__ __forceinline__ static void sync() {
        asm volatile("bar.sync 1, %0;" ::"n"(kSplitThreads) : "memory");
    }
};

// Block-wide online (max, sum) merge; every thread returns the result. Ends
// with a barrier, so `red` may be reused at once.
template <typename Bar = CtaBarrier>
__device__ __forceinline__ void block_merge(float& m, float& s, float2* red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        merge_ms(m, s, m2, s2);
    }
    if (lane == 0) red[warp] = make_float2(m, s);
    Bar::sync();
    m = red[0].x;
    s = red[0].y;
#pragma unroll
    for (int w = 1; w < kSplitNW; ++w) merge_ms(m, s, red[w].x, red[w].y);
    Bar::sync();
}

// The units one thread holds in one step of a sweep: kSplitUnroll 16-byte
// vectors (VEC > 1, kept packed until used) or elements (VEC == 1).
template <typename T, int VEC>
struct Units {
    uint4 v[kSplitUnroll];
    __device__ __forceinline__ void load(const T* p, int left, uint64_t pol) {
#pragma unroll
        for (int k = 0; k < kSplitUnroll; ++k)
            if (k < left) v[k] = ld_vec(p + (int64_t)k * kSplitThreads * VEC, pol);
    }
    __device__ __forceinline__ void get(int k, float* f) const { Elem<T>::unpack(v[k], f); }
};

template <typename T>
struct Units<T, 1> {
    float v[kSplitUnroll];
    __device__ __forceinline__ void load(const T* p, int left, uint64_t pol) {
#pragma unroll
        for (int k = 0; k < kSplitUnroll; ++k)
            if (k < left) v[k] = ld_one<T>(p + (int64_t)k * kSplitThreads, pol);
    }
    __device__ __forceinline__ void get(int k, float* f) const { f[0] = v[k]; }
};

// One sweep over a block's part in two rows at once: pass 1 of row `a`
// (STATS: its (m, s), returned in every thread) and pass 2 of row `b`
// (APPLY: y = exp(x - M) / S written to `bo`). The pointers address this
// thread's first unit of the part (16-byte vectors when VEC > 1, elements
// when VEC == 1); its units follow at a stride of kSplitThreads, `n` of them.
// Each step of the sweep issues both rows' loads before using either; pass 1
// takes one max over the step's units, one rescale, then the exponentials.
template <typename T, int VEC, bool STATS, bool APPLY>
__device__ __forceinline__ float2 sweep(const T* a, const T* b, T* bo, int n, uint64_t keep,
                                        uint64_t drop, float M, float S, float2* red) {
    float m = neg_inf(), s = 0.0f;
    const float rs = final_rcp(M, S);
    const float m_l2 = M * kLog2e;
    constexpr int U = kSplitUnroll;
    constexpr int64_t kStep = (int64_t)U * kSplitThreads * VEC;  // elements per sweep step
#pragma unroll 1
    for (int k0 = 0; k0 < n; k0 += U, a += kStep, b += kStep, bo += kStep) {
        const int left = n - k0;
        Units<T, VEC> ua, ub;
        if (STATS) ua.load(a, left, keep);
        if (APPLY) ub.load(b, left, drop);
        if (STATS) {
            float cm = neg_inf();
#pragma unroll
            for (int k = 0; k < U; ++k) {
                if (k < left) {
                    float f[VEC];
                    ua.get(k, f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) cm = fmaxf(cm, f[e]);
                }
            }
            const float mn = fmaxf(m, cm);
            const float shift = (mn == neg_inf()) ? 0.0f : mn;
            const float shift_l2 = shift * kLog2e;
            float cs = 0.0f;
#pragma unroll
            for (int k = 0; k < U; ++k) {
                if (k < left) {
                    float f[VEC];
                    ua.get(k, f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) cs += split_exp<T>(f[e], shift, shift_l2);
                }
            }
            s = s * merge_scale(m, mn) + cs;
            m = mn;
        }
        if (APPLY) {
#pragma unroll
            for (int k = 0; k < U; ++k) {
                if (k < left) {
                    float f[VEC];
                    ub.get(k, f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) f[e] = split_exp<T>(f[e], M, m_l2) * rs;
                    if constexpr (VEC == 1) {
                        Elem<T>::store1(bo + (int64_t)k * kSplitThreads, f[0]);
                    } else {
                        stg_stream(bo + (int64_t)k * kSplitThreads * VEC, Elem<T>::pack(f));
                    }
                }
            }
        }
    }
    if (STATS) block_merge(m, s, red);
    return make_float2(m, s);
}

// A block's (max, sum) for a step, tagged with the step, as two 8-byte words.
__device__ __forceinline__ void st_tagged(void* p, float m, float s, unsigned int tag) {
    asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p),
                 "l"(((unsigned long long)tag << 32) | __float_as_uint(m)),
                 "l"(((unsigned long long)tag << 32) | __float_as_uint(s))
                 : "memory");
}

__device__ __forceinline__ bool ld_tagged(const void* p, unsigned int tag, float& m, float& s) {
    unsigned long long a, b;
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
    m = __uint_as_float((unsigned int)a);
    s = __uint_as_float((unsigned int)b);
    return (unsigned int)(a >> 32) == tag && (unsigned int)(b >> 32) == tag;
}

// The exchange of one group: slots[kRing][B] of 16 bytes in the workspace.
struct Exchange {
    unsigned char* slots;
    int parts, B, g, b;
    __device__ Exchange(void* ws, int B_, int parts_, int g_, int b_)
        : slots(static_cast<unsigned char*>(ws)), parts(parts_), B(B_), g(g_), b(b_) {}

    // Thread 0 stores the block's pair for step t (tag t + 1).
    __device__ __forceinline__ void publish(int64_t t, float m, float s, int flags_) {
        if (threadIdx.x != 0 || (flags_ & kFlagNoArrive)) return;
        unsigned char* slot = slots + ((int64_t)(t % kRing) * B + b) * 16;
        if (SR_WRITE_OK(slot, 16)) st_tagged(slot, m, s, (unsigned int)(t + 1));
    }

    // The row's (M, S) of step q from the group's `parts` pairs, each thread
    // merging (after waiting, bounded, for them) pairs tid, tid + threads, ...;
    // false in every thread when a wait expired (the timeout bit is then set).
    // Block-wide.
    template <typename Bar = CtaBarrier>
    __device__ __forceinline__ bool merge_row(int64_t q, float& M, float& S, float2* red,
                                              int* s_fail, unsigned int* err,
                                              unsigned long long timeout_ns) {
        const unsigned int tag = (unsigned int)(q + 1);
        const unsigned char* grp = slots + ((int64_t)(q % kRing) * B + (int64_t)g * parts) * 16;
        float m = neg_inf(), s = 0.0f;
        bool ok = true;
        for (int k = threadIdx.x; k < parts && ok; k += kSplitThreads) {
            const unsigned char* slot = grp + (int64_t)k * 16;
            if (!SR_READ_OK(slot, 16)) {
                ok = false;
                break;
            }
            float pm, ps;
            if (!ld_tagged(slot, tag, pm, ps)) {
                const uint64_t t0 = global_timer_ns();
                while (!ld_tagged(slot, tag, pm, ps)) {
                    if (global_timer_ns() - t0 > timeout_ns) {
                        ok = false;
                        break;
                    }
                    __nanosleep(64);
                }
            }
            if (ok) merge_ms(m, s, pm, ps);
        }
        if (!ok) {
            *s_fail = 1;
            atomicOr(err, kErrTimeout);
        }
        Bar::sync();
        if (*s_fail) return false;
        block_merge<Bar>(m, s, red);
        M = m;
        S = s;
        return true;
    }
};

template <typename T, int VEC>
__global__ void __launch_bounds__(kSplitThreads, SR_SPLIT_MIN_BLOCKS)
    split_grid_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int64_t N,
                      int64_t ld_in, int64_t ld_out, int lanes, int parts, int64_t part_units,
                      void* ws, unsigned int* err, unsigned long long timeout_ns, int flags) {
    SR_GRID_DEPENDENCY();
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, M, ld_in, N), SR_MAT_OUT(out, M, ld_out, N),
                    SR_SPAN_OUT(ws, kSplitWorkspaceBytes));
    __shared__ float2 red[kSplitNW];
    __shared__ int s_fail;
    const int tid = threadIdx.x;
    if (tid == 0) s_fail = 0;
    const int b_idx = blockIdx.x;
    const int g = b_idx / parts, p = b_idx - g * parts;
    Exchange x(ws, (int)gridDim.x, parts, g, b_idx);
    const int64_t units = N / VEC;  // VEC divides N when VEC > 1
    const int64_t u0 = (p * part_units < units) ? p * part_units : units;
    const int64_t u1 = (u0 + part_units < units) ? u0 + part_units : units;
    const int64_t steps = (M > g) ? (M - g + lanes - 1) / lanes : 0;
    // This thread's units of the part: u0 + tid + k * threads, k < n.
    const int n = (u1 - u0 > tid) ? (int)((u1 - u0 - tid + kSplitThreads - 1) / kSplitThreads) : 0;
    const int64_t first = (u0 + tid) * VEC;  // element offset of the first one in a row
    const uint64_t keep = l2_keep(), drop = l2_drop();

    // Iteration t: merge step t - kLag's pairs, then one sweep that runs pass 1
    // of step t and pass 2 of step t - kLag, then store step t's pair.
#pragma unroll 1
    for (int64_t t = 0; t < steps + kLag; ++t) {
        const bool stats = t < steps, apply = t >= kLag;
        if (!stats && !apply) continue;  // a group with fewer rows than kLag (block-uniform)
        float rm = neg_inf(), rsum = 0.0f;  // the row's (M, S) for pass 2
        if (apply && !x.merge_row(t - kLag, rm, rsum, red, &s_fail, err, timeout_ns)) return;
        const T* a = stats ? in + (g + t * lanes) * ld_in + first : nullptr;
        const T* b = apply ? in + (g + (t - kLag) * lanes) * ld_in + first : nullptr;
        T* bo = apply ? out + (g + (t - kLag) * lanes) * ld_out + first : nullptr;
        float2 ms;
        if (stats && apply) {
            ms = sweep<T, VEC, true, true>(a, b, bo, n, keep, drop, rm, rsum, red);
        } else if (stats) {
            ms = sweep<T, VEC, true, false>(a, b, bo, n, keep, drop, rm, rsum, red);
        } else {
            ms = sweep<T, VEC, false, true>(a, b, bo, n, keep, drop, rm, rsum, red);
        }
        if (stats) x.publish(t, ms.x, ms.y, flags);
    }
}


// ---------------------------------------------------------------------------
// Aligned rows: the same schedule with the loads done by the bulk-copy
// engine. A producer warp (lane 0) walks the block's chunk sequence -- for
// every step t and every kBulkChunk-byte chunk c of the part: c of row t for
// pass 1, then c of row t - kLag for pass 2 -- and issues each chunk as a
// 1-D bulk copy (cp.async.bulk, L2 policy as in the sweep) into a ring of
// kBulkSlots slots of shared memory as soon as the slot is free; slot i
// completes on full[i] (transaction bytes). The kSplitThreads consumer
// threads take the chunks in the same order, move their units into
// registers, release the slot on empty[i] (one arrival per consumer warp)
// and then reduce or normalise them. Consumers synchronise on named barrier 1
// (the producer warp takes no part). Failure: a consumer whose wait expires
// takes no further chunk and all consumers leave together after the next
// consumer barrier; the producer stops issuing when a wait of its own expires
// or a consumer failed, and before it exits waits (bounded) for every copy it
// issued, so that no copy lands in the shared memory of a finished block.
// ---------------------------------------------------------------------------
// Chunk bytes and ring slots per block, and resident blocks per SM. Measured
// on GB300 (cold L2, µs; f32 32 x 4194304 / bf16 128 x 524288 / bf16
// 512 x 400008): 32 KiB x 3 slots, 2 blocks/SM 229 / 72 / 197; 16 KiB x 6
// 243 / 78 / 204; 8 KiB x 12 294 / 91 / 255; 48 KiB x 2 253 / 77 / 190;
// 64 KiB x 2, 1 block/SM 248 / 82 / 229; the register sweep (the kernel
// unaligned rows take) 272 / 83 / 252. A bulk L2 prefetch of the next row's
// part by the producer: 248 / 81 / 219 with 16 KiB chunks (against 243).
#ifndef SR_SPLIT_BULK_SLOTS
#define SR_SPLIT_BULK_SLOTS 3
#endif
#ifndef SR_SPLIT_BULK_CHUNK
#define SR_SPLIT_BULK_CHUNK 32768
#endif
#ifndef SR_SPLIT_BULK_MIN_BLOCKS
#define SR_SPLIT_BULK_MIN_BLOCKS 2
#endif
constexpr int kBulkSlots = SR_SPLIT_BULK_SLOTS;
constexpr int kBulkChunk = SR_SPLIT_BULK_CHUNK;
constexpr int kBulkUnits = kBulkChunk / 16;
constexpr int kBulkThreads = kSplitThreads + 32;
constexpr int kBulkPer = kBulkUnits / kSplitThreads;  // units per consumer thread and chunk
static_assert(kBulkChunk % (16 * kSplitThreads) == 0, "whole units per consumer thread");
constexpr size_t kBulkBarOffset = (size_t)kBulkSlots * kBulkChunk;
constexpr size_t kBulkSmem = kBulkBarOffset + 16 * kBulkSlots;

__device__ __forceinline__ void bulk_g2s_pol(uint32_t dst, const void* src, uint32_t bytes,
                                             uint32_t bar, uint64_t pol) {
    if (!SR_READ_OK(src, bytes)) return;  // never completes: the bounded wait expires
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive1(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kBulkThreads, SR_SPLIT_BULK_MIN_BLOCKS)
    split_bulk_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t M, int64_t N,
                      int64_t ld_in, int64_t ld_out, int lanes, int parts, int64_t part_units,
                      void* ws, unsigned int* err, unsigned long long timeout_ns, int flags) {
    SR_GRID_DEPENDENCY();
    constexpr int VEC = 16 / sizeof(T);
    SR_BOUNDS_BEGIN(SR_MAT_IN(in, M, ld_in, N), SR_MAT_OUT(out, M, ld_out, N),
                    SR_SPAN_OUT(ws, kSplitWorkspaceBytes));
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float2 red[kSplitNW];
    __shared__ int s_fail;
    const int tid = threadIdx.x;
    const uint32_t sbase = smem_addr(smem);
    const uint32_t full0 = sbase + (uint32_t)kBulkBarOffset;
    const uint32_t empty0 = full0 + 8u * kBulkSlots;
    if (tid == 0) {
        s_fail = 0;
        for (int i = 0; i < kBulkSlots; ++i) {
            mbar_init(full0 + 8u * i, 1);
            mbar_init(empty0 + 8u * i, kSplitNW);
        }
        fence_mbar_init();
    }
    __syncthreads();
    const int b_idx = blockIdx.x;
    const int g = b_idx / parts, p = b_idx - g * parts;
    const int64_t units = N / VEC;
    const int64_t u0 = (p * part_units < units) ? p * part_units : units;
    const int64_t u1 = (u0 + part_units < units) ? u0 + part_units : units;
    const int64_t steps = (M > g) ? (M - g + lanes - 1) / lanes : 0;
    const int nch = (int)((u1 - u0 + kBulkUnits - 1) / kBulkUnits);

    if (tid >= kSplitThreads) {
        // Producer warp: lane 0 issues the copies, in the consumers' order.
        if (tid != kSplitThreads) return;
        const uint64_t keep = l2_keep(), drop = l2_drop();
        int64_t j = 0;
        bool ok = true;
        for (int64_t t = 0; t < steps + kLag && ok; ++t) {
            for (int c = 0; c < nch && ok; ++c) {
                const int64_t cu = u0 + (int64_t)c * kBulkUnits;
                const uint32_t bytes = (uint32_t)((u1 - cu < kBulkUnits ? u1 - cu : kBulkUnits) * 16);
                for (int kind = 0; kind < 2 && ok; ++kind) {
                    if (kind == 0 ? t >= steps : t < kLag) continue;
                    const int64_t r = g + (kind == 0 ? t : t - kLag) * lanes;
                    const int slot = (int)(j % kBulkSlots);
                    if (j >= kBulkSlots) {
                        ok = mbar_wait_bounded(empty0 + 8u * slot,
                                               (uint32_t)((j / kBulkSlots - 1) & 1), timeout_ns);
                        if (!ok) break;
                    }
                    if (*(volatile int*)&s_fail) { ok = false; break; }
                    mbar_expect_tx(full0 + 8u * slot, bytes);
                    bulk_g2s_pol(sbase + (uint32_t)slot * kBulkChunk, in + r * ld_in + cu * VEC,
                                 bytes, full0 + 8u * slot, kind == 0 ? keep : drop);
                    ++j;
                }
            }
        }
        if (!ok) atomicOr(err, kErrTimeout);
        // Before the block may exit, every issued copy must have landed.
        for (int64_t i = (j > kBulkSlots ? j - kBulkSlots : 0); i < j; ++i)
            mbar_wait_bounded(full0 + 8u * (uint32_t)(i % kBulkSlots),
                              (uint32_t)((i / kBulkSlots) & 1), timeout_ns);
        return;
    }

    // Consumers.
    Exchange x(ws, (int)gridDim.x, parts, g, b_idx);
    const int lane = tid & 31;
    bool failed = false;
    int64_t j = 0;
#pragma unroll 1
    for (int64_t t = 0; t < steps + kLag; ++t) {
        const bool stats = t < steps, apply = t >= kLag;
        if (!stats && !apply) continue;
        float rm = neg_inf(), rsum = 0.0f;
        if (apply && !x.merge_row<ConsumerBarrier>(t - kLag, rm, rsum, red, &s_fail, err, timeout_ns))
            return;  // every consumer, after the same barrier
        const float rs = final_rcp(rm, rsum);
        const float rm_l2 = rm * kLog2e;
        T* orow = apply ? out + (g + (t - kLag) * lanes) * ld_out : nullptr;
        float m = neg_inf(), s = 0.0f;
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
            const int64_t cu = u0 + (int64_t)c * kBulkUnits;
            const int cnt = (int)(u1 - cu < kBulkUnits ? u1 - cu : kBulkUnits);
#pragma unroll 1
            for (int kind = 0; kind < 2; ++kind) {
                if (kind == 0 ? !stats : !apply) continue;
                const int slot = (int)(j % kBulkSlots);
                const uint32_t parity = (uint32_t)((j / kBulkSlots) & 1);
                ++j;
                if (failed) continue;
                if (!mbar_wait_bounded(full0 + 8u * slot, parity, timeout_ns)) {
                    failed = true;
                    s_fail = 1;
                    atomicOr(err, kErrTimeout);
                    continue;
                }
                const uint32_t chunk = sbase + (uint32_t)slot * kBulkChunk;
                uint4 v[kBulkPer];
#pragma unroll
                for (int k = 0; k < kBulkPer; ++k)
                    if (tid + k * kSplitThreads < cnt) v[k] = lds128(chunk + 16u * (tid + k * kSplitThreads));
                __syncwarp();
                if (lane == 0) mbar_arrive1(empty0 + 8u * slot);  // the slot's data is in registers
                if (kind == 0) {
                    float cm = neg_inf();
#pragma unroll
                    for (int k = 0; k < kBulkPer; ++k) {
                        if (tid + k * kSplitThreads < cnt) {
                            float f[VEC];
                            Elem<T>::unpack(v[k], f);
#pragma unroll
                            for (int e = 0; e < VEC; ++e) cm = fmaxf(cm, f[e]);
                        }
                    }
                    const float mn = fmaxf(m, cm);
                    const float shift = (mn == neg_inf()) ? 0.0f : mn;
                    const float shift_l2 = shift * kLog2e;
                    float cs = 0.0f;
#pragma unroll
                    for (int k = 0; k < kBulkPer; ++k) {
                        if (tid + k * kSplitThreads < cnt) {
                            float f[VEC];
                            Elem<T>::unpack(v[k], f);
#pragma unroll
                            for (int e = 0; e < VEC; ++e) cs += split_exp<T>(f[e], shift, shift_l2);
                        }
                    }
                    s = s * merge_scale(m, mn) + cs;
                    m = mn;
                } else {
#pragma unroll
                    for (int k = 0; k < kBulkPer; ++k) {
                        const int vi = tid + k * kSplitThreads;
                        if (vi < cnt) {
                            float f[VEC];
                            Elem<T>::unpack(v[k], f);
#pragma unroll
                            for (int e = 0; e < VEC; ++e) f[e] = split_exp<T>(f[e], rm, rm_l2) * rs;
                            stg_stream(orow + (cu + vi) * VEC, Elem<T>::pack(f));
                        }
                    }
                }
            }
        }
        ConsumerBarrier::sync();
        if (s_fail) return;  // every consumer, after the same barrier
        if (stats) {
            block_merge<ConsumerBarrier>(m, s, red);
            x.publish(t, m, s, flags);
        }
    }
}

template <typename T, int VEC>
cudaError_t launch_vec(const Problem& p, const SplitShape& sh, void* ws) {
    // Zero the slots the launch uses (slots[kRing][B], 16 bytes each).
    const int B = sh.lanes * sh.parts;
    cudaError_t e = cudaMemsetAsync(ws, 0, (size_t)kRing * B * 16, p.stream);
    if (e != cudaSuccess) return e;
    LaunchShape ls{dim3((unsigned)B), dim3(kSplitThreads)};
    ls.cooperative = true;
    if constexpr (VEC > 1) {
        ls.block = dim3(kBulkThreads);
        ls.smem = kBulkSmem;
        e = ensure_smem_limit(reinterpret_cast<const void*>(split_bulk_kernel<T>), ls.smem, false);
        if (e != cudaSuccess) return e;
        return launch_kernel(split_bulk_kernel<T>, ls, p.stream, static_cast<const T*>(p.in),
                             static_cast<T*>(p.out), p.M, p.N, p.ld_in, p.ld_out, sh.lanes,
                             sh.parts, sh.part_units, ws, p.dev->err, p.timeout_ns, p.flags);
    } else {
        return launch_kernel(split_grid_kernel<T, VEC>, ls, p.stream,
                             static_cast<const T*>(p.in), static_cast<T*>(p.out), p.M, p.N,
                             p.ld_in, p.ld_out, sh.lanes, sh.parts, sh.part_units, ws, p.dev->err,
                             p.timeout_ns, p.flags);
    }
}

template <typename T>
cudaError_t launch_typed(const Problem& p, const SplitShape& sh, void* ws) {
    if (sh.vec > 1) return launch_vec<T, 16 / sizeof(T)>(p, sh, ws);
    return launch_vec<T, 1>(p, sh, ws);
}

template <typename T>
const void* typed_kernel(int vec) {
    return vec > 1 ? reinterpret_cast<const void*>(split_bulk_kernel<T>)
                   : reinterpret_cast<const void*>(split_grid_kernel<T, 1>);
}

}  // namespace

size_t split_smem(int vec) { return vec > 1 ? kBulkSmem : 0; }
int split_threads(int vec) { return vec > 1 ? kBulkThreads : kSplitThreads; }

const void* split_kernel(int dtype, int vec) {
    switch (dtype) {
        case kF32: return typed_kernel<float>(vec);
        case kBF16: return typed_kernel<__nv_bfloat16>(vec);
        case kF16: return typed_kernel<__half>(vec);
    }
    return nullptr;
}

// Lanes and parts (host logic). `max_blocks` is how many blocks of the
// kernel the device holds at once (at most kSplitMaxBlocks), `l2_bytes` its
// L2. Lanes: when the whole input fits in half the L2, a group per row (as
// many as there are blocks); else as many groups as half the L2 allows at
// kLag + 1 rows per group (a row's parts wait for their second read while the
// group reads kLag more), but no more than leave each group kSplitMinSteps
// rows (the first kLag sweeps of a group only read and the last kLag only
// write, so a group needs a few steps to overlap them); never more than the
// rows or the blocks. Parts:
// the blocks left per group, but no part under kSplitMinUnits units; the
// parts are then evened out so that none is empty.
SplitShape split_shape(int64_t M, int64_t N, int64_t ld_in, int64_t ld_out, int dtype,
                       const void* in, const void* out, int max_blocks, int64_t l2_bytes) {
    SplitShape sh;
    const bool vec = rows_vector_aligned(in, out, N, ld_in, ld_out, dtype);
    sh.vec = vec ? 16 / elem_bytes(dtype) : 1;
    const int64_t units = N / sh.vec;
    const int64_t row_bytes = N * elem_bytes(dtype);
    if (max_blocks > kSplitMaxBlocks) max_blocks = kSplitMaxBlocks;
    if (max_blocks < 1) max_blocks = 1;
    int64_t lanes = (l2_bytes / 2) / ((kLag + 1) * (row_bytes > 0 ? row_bytes : 1));
    if (M * row_bytes <= l2_bytes / 2) {
        lanes = M;  // the whole input stays in L2 between the passes: all rows at once
    } else if (lanes > M / kSplitMinSteps) {
        lanes = M / kSplitMinSteps;
    }
    if (lanes > M) lanes = M;
    if (lanes > max_blocks) lanes = max_blocks;
    if (lanes < 1) lanes = 1;
    int64_t parts = max_blocks / lanes;
    const int64_t most = (units + kSplitMinUnits - 1) / kSplitMinUnits;
    if (parts > most) parts = most;
    if (parts < 1) parts = 1;
    sh.part_units = (units + parts - 1) / parts;
    if (sh.part_units < 1) sh.part_units = 1;
    sh.parts = (int)((units + sh.part_units - 1) / sh.part_units);
    if (sh.parts < 1) sh.parts = 1;
    sh.lanes = (int)lanes;
    return sh;
}

cudaError_t launch_split(const Problem& p, const SplitShape& sh, void* ws) {
    switch (p.dtype) {
        case kF32: return launch_typed<float>(p, sh, ws);
        case kBF16: return launch_typed<__nv_bfloat16>(p, sh, ws);
        case kF16: return launch_typed<__half>(p, sh, ws);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sr

// ---------------------------------------------------------------------------
// softmax_rows_split_noalloc: the split plan with built-in scratch.
//
// For callers that must not allocate device memory at all: code that runs
// under a fixed memory budget reserved up front (inference servers, plugins
// living inside another framework's memory pool), code that may not change
// the device's memory footprint once it is running, and code called from
// places where a cudaMalloc would implicitly synchronise the device and
// stall other work. They pass only the input and the output; the
// statistics live in the array below, which is part of the library's device
// image: every GPU that loads the library holds it until the process exits.
// ---------------------------------------------------------------------------
namespace sr {
namespace {

// The split plan's workspace, whatever the problem.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kSplitWorkspaceBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64];  // the array's device address, per device, once set up

// Device address of the array on the current device (set up on first use,
// with that device current). In host code the array's name is only a
// stand-in, never a device address.
int noalloc_scratch(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SR_ECUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return SR_ECUDA;
        g_noalloc_addr[dev] = ptr;
    }
    *out = g_noalloc_addr[dev];
    return SR_OK;
}

}  // namespace
}  // namespace sr

extern "C" int softmax_rows_split_noalloc(const void* in, void* out, int64_t M, int64_t N,
                                          int64_t ld_in, int64_t ld_out, int dtype,
                                          sr_stream_t stream) {
    const int64_t need = softmax_rows_split_workspace_bytes(in, out, M, N, ld_in, ld_out, dtype);
    if (need < 0) return (int)-need;
    if (M == 0) return SR_OK;
    if (need > sr::kSplitWorkspaceBytes) return SR_EINVAL;
    void* scratch = nullptr;
    const int st = sr::noalloc_scratch(&scratch);
    if (st != SR_OK) return st;
    return softmax_rows_split(in, out, M, N, ld_in, ld_out, dtype, scratch, need, stream);
}
