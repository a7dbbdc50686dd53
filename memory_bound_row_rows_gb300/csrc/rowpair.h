// Host-side logic of the row-pair engine (rowpair.cuh): the problem, the
// load mode the matrices allow, and the shape each plan runs with. Plain host
// code, shared by the C ABI (plan queries) and the launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/softmax_rows.h"
#include "internal.h"

namespace sr {
namespace rp {

enum class Mode : int { kAligned = 0, kShifted = 1, kScalar = 2 };

constexpr int kTeamMaxThreads = 512;
constexpr int kClusterThreads = 256;
constexpr int kLoopThreads = 512;
constexpr int kLoopUnroll = 4;

inline int kv_target(int mode) { return mode != (int)Mode::kScalar ? 4 : 8; }
inline int kv_max(int mode, int dtype) {
    return mode != (int)Mode::kScalar ? (elem_bytes(dtype) == 4 ? 8 : 4) : 16;
}

// One problem: C = f(A, B, the row's reduction), M x N, pitches in elements.
struct Args {
    const void* a;
    const void* b;
    void* c;
    int64_t M, N, lda, ldb, ldc;
    int dtype;
    cudaStream_t stream;
    unsigned int* err = nullptr;            // device error word (CLUSTER plan's bounded waits)
    unsigned long long timeout_ns = 0;      // limit of one bounded wait
    int flags = 0;                          // kFlagNoCopy: the CLUSTER plan sends no partials
    bool stream_wide = false;               // stream aligned rows of kStreamWideUnits and more
};

// How one plan runs one problem (host logic only, the same on every device).
struct Shape {
    int plan = 0;  // SR_PLAN_ROW, SR_PLAN_CLUSTER or SR_PLAN_ONLINE
    int mode = 0;  // Mode
    int tpr = 0;   // ROW: threads per row
    int kv = 0;    // ROW, CLUSTER: units per thread
    int csize = 0; // CLUSTER: blocks per row
    int64_t slice = 0;  // CLUSTER: units per block
    bool streamed = false;  // CLUSTER: slices read twice instead of held (aligned rows only)
};

// Resident blocks per SM the streamed CLUSTER kernel is compiled for.
constexpr int kStreamMinBlocks = 4;
// Aligned rows of at least this many units are streamed when the operation
// asks for it (Args::stream_wide; the RMSNorm does): f16 64 x 131072 ran at
// 15.5 against 16.8 µs and bf16 1024 x 131072 at 157.7 against 177.0 µs on
// GB300 (cold L2). The backward holds such rows in registers: streaming them
// cost it 10 %.
constexpr int64_t kStreamWideUnits = 16384;
// Aligned rows of at least this many units are streamed even when a cluster
// could hold them (never, by default: streaming rows of 8192 units helped the
// RMSNorm and hurt the backward by as much).
#ifndef SR_PAIR_STREAM_MIN_UNITS
#define SR_PAIR_STREAM_MIN_UNITS (int64_t(1) << 62)
#endif
// Streamed clusters double (8 -> 16 blocks) only while the doubled grid still
// fits one wave of resident blocks (backward f16 64 x 1048576: 102.2 -> 93.8 µs
// against doubling whenever the grid is short of a wave).
#ifndef SR_PAIR_STREAM_GROW_WAVE
#define SR_PAIR_STREAM_GROW_WAVE 1
#endif

// The load mode the three matrices allow.
inline int mode_for(const Args& p) {
    const int64_t es = elem_bytes(p.dtype);
    const uintptr_t a = reinterpret_cast<uintptr_t>(p.a), b = reinterpret_cast<uintptr_t>(p.b),
                    c = reinterpret_cast<uintptr_t>(p.c);
    const int64_t pa = p.lda * es % 16, pb = p.ldb * es % 16, pc = p.ldc * es % 16;
    if (a % 16 == 0 && b % 16 == 0 && c % 16 == 0 && pa == 0 && pb == 0 && pc == 0 &&
        (p.N * es) % 16 == 0)
        return (int)Mode::kAligned;
    if (a % 16 == b % 16 && a % 16 == c % 16 && pa == pb && pa == pc && a % es == 0)
        return (int)Mode::kShifted;
    return (int)Mode::kScalar;
}

// Most units a row of the matrices can hold (a shifted row's vectors are at
// most N / VEC).
inline int64_t max_units(const Args& p, int mode) {
    return mode == (int)Mode::kScalar ? p.N : p.N / (16 / elem_bytes(p.dtype));
}

inline int64_t pow2_at_least(int64_t v) {
    int64_t k = 1;
    while (k < v) k *= 2;
    return k;
}

// Shapes:
//  ROW: the smallest power-of-two team (32..512 threads) that gives each
//    thread at most the target units (4 vectors, or 8 elements), the units
//    per thread rounded up to a power of two; rows up to 512 x the most a
//    thread holds (8 f32 vectors, 4 16-bit vectors, 16 elements).
//  CLUSTER: 256-thread blocks; the smallest power-of-two cluster (2..16)
//    whose slices fit the target units per thread (else the most a thread
//    holds, in 16 blocks). While there are too few rows to give every SM two
//    blocks, the cluster doubles (up to 16) as long as each block keeps at
//    least one unit per thread; the units per thread follow the slice.
//    Aligned rows too wide for that are streamed: 8-block clusters (16 when
//    the doubled grid still fits one wave of resident blocks), each block
//    reading its slice once to reduce it and again to write.
inline bool shape_for(const Args& p, int plan, int sm_count, Shape* out) {
    Shape sh;
    sh.plan = plan;
    sh.mode = mode_for(p);
    const int64_t units = max_units(p, sh.mode);
    const int kt = kv_target(sh.mode);
    const int km = kv_max(sh.mode, p.dtype);
    switch (plan) {
        case SR_PLAN_ROW: {
            if (units > (int64_t)kTeamMaxThreads * km) return false;
            int tpr = 32;
            while (tpr < kTeamMaxThreads && (int64_t)tpr * kt < units) tpr *= 2;
            int64_t kv = pow2_at_least((units + tpr - 1) / tpr);
            if (tpr > 32 && kv < kt) kv = kt;
            sh.tpr = tpr;
            sh.kv = (int)kv;
            break;
        }
        case SR_PLAN_CLUSTER: {
            int c = 0, kv = kt;
            for (int cc = 2; cc <= kMaxCluster; cc *= 2)
                if ((int64_t)cc * kClusterThreads * kt >= units) {
                    c = cc;
                    break;
                }
            const bool stream_anyway =
                sh.mode == (int)Mode::kAligned &&
                (units >= SR_PAIR_STREAM_MIN_UNITS || (p.stream_wide && units >= kStreamWideUnits));
            if (c == 0 || stream_anyway) {
                if ((int64_t)kMaxCluster * kClusterThreads * km < units || stream_anyway) {
                    if (sh.mode != (int)Mode::kAligned) return false;
                    c = 8;
                    while (c < kMaxCluster &&
                           (SR_PAIR_STREAM_GROW_WAVE
                                ? p.M * c * 2 <= (int64_t)kStreamMinBlocks * sm_count
                                : p.M * c < (int64_t)kStreamMinBlocks * sm_count))
                        c *= 2;
                    sh.csize = c;
                    sh.slice = (units + c - 1) / c;
                    sh.kv = 0;
                    sh.streamed = true;
                    break;
                }
                c = kMaxCluster;
                kv = km;
            }
            while (c < kMaxCluster && p.M * c < 2 * (int64_t)sm_count &&
                   units / (2 * c) >= kClusterThreads)
                c *= 2;
            sh.csize = c;
            sh.slice = (units + c - 1) / c;
            const int64_t k = pow2_at_least((sh.slice + kClusterThreads - 1) / kClusterThreads);
            if (k > kv) return false;
            sh.kv = (int)k;
            break;
        }
        case SR_PLAN_ONLINE: break;
        default: return false;
    }
    *out = sh;
    return true;
}

// Automatic plan: ROW when the row fits a team of at most 256 threads and
// there are rows enough for the GPU (or the row is short); CLUSTER for wider
// rows and for rows too few to fill the GPU; ONLINE otherwise. Rows that need
// a 512-thread team run faster on CLUSTER (measured on GB300, cold L2:
// backward f16 4096 x 16384 58.2 against 72.6 µs, RMSNorm 65.5 against 85.0;
// f32 1024 x 16384 29.2 against 34.0 µs).
inline int choose_plan(const Args& p, int sm_count) {
    Shape sh;
    const bool row = shape_for(p, SR_PLAN_ROW, sm_count, &sh);
    const int64_t units = max_units(p, mode_for(p));
    const bool cluster_ok = row && sh.tpr == kTeamMaxThreads &&
                            shape_for(p, SR_PLAN_CLUSTER, sm_count, &sh);
    if (row && !cluster_ok && (p.M >= sm_count || units < 2 * kClusterThreads))
        return SR_PLAN_ROW;
    if (shape_for(p, SR_PLAN_CLUSTER, sm_count, &sh)) return SR_PLAN_CLUSTER;
    if (row) return SR_PLAN_ROW;
    return SR_PLAN_ONLINE;
}

}  // namespace rp

// Launchers of the two row-pair operations (backward_rows.cu, rmsnorm_rows.cu).
cudaError_t launch_backward(const rp::Args& p, const rp::Shape& sh);
cudaError_t launch_rmsnorm(const rp::Args& p, const rp::Shape& sh, const void* weight, float eps);

}  // namespace sr
