// C ABI of the row-softmax library: argument checks, plan choice, the
// per-device cache (SM count, shared-memory limits, occupancy, the device
// error word) and the launch. See include/softmax_rows.h for the contract.
#include <mutex>
#include <unordered_map>

#include "../../include/softmax_rows.h"
#include "rowpair.h"
#include "wide.h"
#include "internal.h"
#include "split.h"

namespace sr {

// Set (bit 0, kErrTimeout) by a kernel whose bounded wait (for a bulk copy,
// or for the pairs or partials of its cluster peers) expired; in the
// bounds-checking build also (bit 1, kErrBounds) by an access outside the
// call's matrices. One word per device (each device holds its own copy of
// this module's globals).
__device__ unsigned int g_error_word;
#if SR_BOUNDS_CHECK
// First address a checked access refused, and the test hook's shrink of the
// writable extents (bounds-checking build only).
__device__ unsigned long long g_bounds_addr;
__device__ long long g_bounds_shrink;
#endif

namespace {

constexpr int kMaxDevices = 64;
// Default limit for one bounded wait: far above any copy's real latency.
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices];

struct OccKey {
    int dev;
    const void* func;
    int threads;
    size_t smem;
    int cluster;
    bool operator==(const OccKey& o) const {
        return dev == o.dev && func == o.func && threads == o.threads && smem == o.smem &&
               cluster == o.cluster;
    }
};
struct OccHash {
    size_t operator()(const OccKey& k) const {
        size_t h = std::hash<const void*>()(k.func);
        h ^= (size_t)k.dev * 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
        h ^= (size_t)k.threads * 0xBF58476D1CE4E5B9ull + (h << 6) + (h >> 2);
        h ^= (size_t)k.smem * 0x94D049BB133111EBull + (h << 6) + (h >> 2);
        h ^= (size_t)k.cluster + (h << 6) + (h >> 2);
        return h;
    }
};
std::unordered_map<OccKey, int, OccHash> g_occ;
std::unordered_map<OccKey, size_t, OccHash> g_smem_set;

int current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

// Per-device properties, queried once per device.
const DeviceInfo* device_info(cudaError_t* err) {
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev_ready[d]) {
        DeviceInfo info;
        info.id = d;
        cudaError_t e;
        if ((e = cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, d)) ||
            (e = cudaDeviceGetAttribute(&info.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                        d)) ||
            (e = cudaDeviceGetAttribute(&info.smem_per_sm,
                                        cudaDevAttrMaxSharedMemoryPerMultiprocessor, d)) ||
            (e = cudaDeviceGetAttribute(&info.l2_bytes, cudaDevAttrL2CacheSize, d)) ||
            (e = cudaGetSymbolAddress(reinterpret_cast<void**>(&info.err), g_error_word))) {
            *err = e;
            return nullptr;
        }
        g_dev[d] = info;
        g_dev_ready[d] = true;
    }
    *err = cudaSuccess;
    return &g_dev[d];
}

}  // namespace

namespace {
struct LaunchRecord {
    const void* func = nullptr;
    dim3 grid, block;
    size_t smem = 0;
    int cluster = 1;
};
thread_local LaunchRecord t_last_launch;
}  // namespace

void note_launch(const void* func, dim3 grid, dim3 block, size_t smem, int cluster) {
    t_last_launch = LaunchRecord{func, grid, block, smem, cluster};
}

int blocks_per_sm(const void* func, int threads, size_t smem) {
    const OccKey key{current_device(), func, threads, smem, 0};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem) != cudaSuccess)
        return -1;
    std::lock_guard<std::mutex> lk(g_mu);
    g_occ[key] = n;
    return n;
}

int max_active_clusters(const void* func, int threads, size_t smem, int cluster) {
    const OccKey key{current_device(), func, threads, smem, cluster};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) return it->second;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cluster, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess) return -1;
    std::lock_guard<std::mutex> lk(g_mu);
    g_occ[key] = n;
    return n;
}

cudaError_t ensure_smem_limit(const void* func, size_t smem, bool nonportable_cluster) {
    const OccKey key{current_device(), func, 0, 0, nonportable_cluster ? 1 : 0};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_smem_set.find(key);
        if (it != g_smem_set.end() && it->second >= smem) return cudaSuccess;
    }
    cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    if (nonportable_cluster) {
        e = cudaFuncSetAttribute(func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    g_smem_set[key] = smem;
    return cudaSuccess;
}

namespace {

// Argument check shared by every entry point: 0 or a positive sr_status.
int check_args(const void* in, const void* out, int64_t M, int64_t N, int64_t ld_in,
               int64_t ld_out, int dtype) {
    if (dtype != SR_F32 && dtype != SR_BF16 && dtype != SR_F16) return SR_EDTYPE;
    if (M < 0 || N < 1 || ld_in < N || ld_out < N) return SR_EINVAL;
    if (M > 0 && (in == nullptr || out == nullptr)) return SR_EINVAL;
    // Index arithmetic stays in int64: the last byte addressed must fit.
    if (M > 0) {
        const __int128 ld = ld_in > ld_out ? ld_in : ld_out;
        const __int128 last = ((__int128)(M - 1) * ld + N) * elem_bytes(dtype);
        if (last > (__int128)INT64_MAX) return SR_EINVAL;
    }
    return 0;
}

// True when the rows of `in` and `out` sit at the same offset from a 16-byte
// boundary (the same base offset, pitches equal modulo 16 bytes) on element
// boundaries: such rows are read as a head, 16-byte vectors and a tail.
bool rows_congruent(const void* in, const void* out, int64_t ld_in, int64_t ld_out, int dtype) {
    const int64_t es = elem_bytes(dtype);
    const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
    return a % 16 == b % 16 && a % es == 0 && (ld_in * es) % 16 == (ld_out * es) % 16;
}

// Whether a plan can run the arguments (host logic only).
bool plan_fits(int plan, const void* in, const void* out, int64_t N, int64_t ld_in,
               int64_t ld_out, int dtype) {
    const bool vec = rows_vector_aligned(in, out, N, ld_in, ld_out, dtype);
    const int64_t row_bytes = N * elem_bytes(dtype);
    switch (plan) {
        case SR_PLAN_WARP: return N <= kWarpMaxN;
        case SR_PLAN_CTA: return vec && row_bytes <= kSliceMaxBytes;
        case SR_PLAN_CLUSTER: return vec && cluster_size_for(N, dtype, 2) > 0;
        case SR_PLAN_ONLINE: return true;
        case SR_PLAN_SMEM: return vec && row_bytes <= kSmemMaxRowBytes;
        case SR_PLAN_ROW: return (vec || rows_congruent(in, out, ld_in, ld_out, dtype)) &&
                                 row_plan_fits(N, dtype);
        case SR_PLAN_WIDE: return wide_fits(in, out, N, ld_in, ld_out, dtype);
    }
    return false;
}

// Automatic plan (from plan sweeps on GB300, cold L2):
//  - rows of 256 vectors up to the ROW plan's limit (2048 16-bit or 4096 FP32
//    vectors), aligned or at a common offset from a 16-byte boundary: ROW
//    (one block per row);
//  - shorter rows (or unaligned rows up to 2048 elements): WARP;
//  - wider rows: WIDE (one cluster per row, the row in registers up to
//    512 KiB, streamed beyond when aligned; faster than CLUSTER on every wide
//    shape measured);
//  - anything else: ONLINE.
int choose_plan(const void* in, const void* out, int64_t N, int64_t ld_in, int64_t ld_out,
                int dtype) {
    const bool vec = rows_vector_aligned(in, out, N, ld_in, ld_out, dtype);
    const int64_t nvec = N * elem_bytes(dtype) / 16;
    if ((vec || rows_congruent(in, out, ld_in, ld_out, dtype)) && nvec >= kRowMinVectors &&
        row_plan_fits(N, dtype))
        return SR_PLAN_ROW;
    if (N <= kWarpMaxN) return SR_PLAN_WARP;
    if (plan_fits(SR_PLAN_WIDE, in, out, N, ld_in, ld_out, dtype)) return SR_PLAN_WIDE;
    if (plan_fits(SR_PLAN_CLUSTER, in, out, N, ld_in, ld_out, dtype)) return SR_PLAN_CLUSTER;
    return SR_PLAN_ONLINE;
}

int run(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in, int64_t ld_out,
        int dtype, int plan, cudaStream_t stream, unsigned long long timeout_ns, int flags) {
    const int bad = check_args(in, out, M, N, ld_in, ld_out, dtype);
    if (bad) return bad;
    if (plan == SR_PLAN_AUTO) {
        plan = choose_plan(in, out, N, ld_in, ld_out, dtype);
    } else if (!plan_fits(plan, in, out, N, ld_in, ld_out, dtype)) {
        return SR_EPLAN;
    }
    if (M == 0) return SR_OK;
    cudaError_t e;
    const DeviceInfo* dev = device_info(&e);
    if (!dev) return SR_ECUDA;
    Problem p{in, out, M, N, ld_in, ld_out, dtype, stream, dev, timeout_ns, flags};
    switch (plan) {
        case SR_PLAN_WARP: e = launch_warp(p); break;
        case SR_PLAN_CTA: e = launch_tma(p, 1); break;
        case SR_PLAN_CLUSTER: e = launch_tma(p, cluster_size_for(N, dtype, 2)); break;
        case SR_PLAN_ONLINE: e = launch_online(p); break;
        case SR_PLAN_SMEM: e = launch_smem(p); break;
        case SR_PLAN_ROW: e = launch_row(p); break;
        case SR_PLAN_WIDE: e = launch_wide(p); break;
        default: return SR_EPLAN;
    }
    return e == cudaSuccess ? SR_OK : SR_ECUDA;
}

// Plans that take a row mask, and the automatic choice among them.
bool masked_plan_fits(int plan, const void* in, const void* out, int64_t N, int64_t ld_in,
                      int64_t ld_out, int dtype) {
    if (plan == SR_PLAN_ROW)  // the masked ROW kernel reads aligned rows only
        return rows_vector_aligned(in, out, N, ld_in, ld_out, dtype) && row_plan_fits(N, dtype);
    return plan == SR_PLAN_WARP || plan == SR_PLAN_ONLINE
               ? plan_fits(plan, in, out, N, ld_in, ld_out, dtype)
               : false;
}

int choose_masked_plan(const void* in, const void* out, int64_t N, int64_t ld_in, int64_t ld_out,
                       int dtype) {
    const int plan = choose_plan(in, out, N, ld_in, ld_out, dtype);
    if (plan == SR_PLAN_ROW && !rows_vector_aligned(in, out, N, ld_in, ld_out, dtype))
        return N <= kWarpMaxN ? SR_PLAN_WARP : SR_PLAN_ONLINE;
    return (plan == SR_PLAN_ROW || plan == SR_PLAN_WARP) ? plan : SR_PLAN_ONLINE;
}

// Argument check of the softmax backward: 0 or a positive sr_status.
int check_bwd_args(const void* y, const void* dy, const void* dx, int64_t M, int64_t N,
                   int64_t ld_y, int64_t ld_dy, int64_t ld_dx, int dtype) {
    if (dtype != SR_F32 && dtype != SR_BF16 && dtype != SR_F16) return SR_EDTYPE;
    if (M < 0 || N < 1 || ld_y < N || ld_dy < N || ld_dx < N) return SR_EINVAL;
    if (M > 0 && (y == nullptr || dy == nullptr || dx == nullptr)) return SR_EINVAL;
    if (M > 0 && (dx == y || dx == dy)) return SR_EINVAL;
    if (M > 0) {
        __int128 ld = ld_y > ld_dy ? ld_y : ld_dy;
        if (ld_dx > ld) ld = ld_dx;
        const __int128 last = ((__int128)(M - 1) * ld + N) * elem_bytes(dtype);
        if (last > (__int128)INT64_MAX) return SR_EINVAL;
    }
    return 0;
}

// Resolve `plan` for a row-pair operation (SR_PLAN_AUTO included): the plan,
// or a negative status.
int resolve_pair_plan(const rp::Args& p, int plan, int sm_count, rp::Shape* sh) {
    if (plan == SR_PLAN_AUTO) plan = rp::choose_plan(p, sm_count);
    if (plan != SR_PLAN_ROW && plan != SR_PLAN_CLUSTER && plan != SR_PLAN_ONLINE) return -SR_EPLAN;
    if (!rp::shape_for(p, plan, sm_count, sh)) return -SR_EPLAN;
    return plan;
}

// Plan and launch one row-pair operation (arguments already checked).
template <class Launch>
int run_pair(const rp::Args& a, int plan, Launch&& launch,
             unsigned long long timeout_ns = kDefaultTimeoutNs) {
    if (plan < SR_PLAN_AUTO || plan > SR_PLAN_ROW) return SR_EPLAN;
    rp::Shape sh;
    // Whether a plan fits does not depend on the device (only the cluster
    // size does), so a plan that cannot run is refused before any CUDA call.
    if (resolve_pair_plan(a, plan, 1, &sh) < 0) return SR_EPLAN;
    if (a.M == 0) return SR_OK;
    cudaError_t e;
    const DeviceInfo* dev = device_info(&e);
    if (!dev) return SR_ECUDA;
    const int chosen = resolve_pair_plan(a, plan, dev->sm_count, &sh);
    if (chosen < 0) return -chosen;
    rp::Args q = a;
    q.err = dev->err;
    q.timeout_ns = timeout_ns;
    return launch(q, sh) == cudaSuccess ? SR_OK : SR_ECUDA;
}

int run_bwd(const void* y, const void* dy, void* dx, int64_t M, int64_t N, int64_t ld_y,
            int64_t ld_dy, int64_t ld_dx, int dtype, int plan, cudaStream_t stream) {
    const int bad = check_bwd_args(y, dy, dx, M, N, ld_y, ld_dy, ld_dx, dtype);
    if (bad) return bad;
    const rp::Args a{y, dy, dx, M, N, ld_y, ld_dy, ld_dx, dtype, stream};
    return run_pair(a, plan, [](const rp::Args& q, const rp::Shape& sh) {
        return launch_backward(q, sh);
    });
}

// Argument check of the residual RMSNorm: 0 or a positive sr_status.
int check_rms_args(const void* x, const void* r, const void* w, const void* y, int64_t M,
                   int64_t N, int64_t ld_x, int64_t ld_r, int64_t ld_y, float eps, int dtype) {
    const int bad = check_bwd_args(x, r, y, M, N, ld_x, ld_r, ld_y, dtype);
    if (bad) return bad;
    if (!(eps >= 0.0f) || eps == INFINITY) return SR_EINVAL;
    if (M > 0 && (w == nullptr || reinterpret_cast<uintptr_t>(w) % elem_bytes(dtype) != 0))
        return SR_EINVAL;
    return 0;
}

// The plan a row-pair call would run, or a negative status (host logic; the
// current device's SM count when sm_count <= 0).
int pair_plan_query(const rp::Args& a, int plan, int sm_count) {
    if (plan < SR_PLAN_AUTO || plan > SR_PLAN_ROW) return -SR_EPLAN;
    if (sm_count <= 0) {
        cudaError_t e;
        const DeviceInfo* dev = device_info(&e);
        if (!dev) return -SR_ECUDA;
        sm_count = dev->sm_count;
    }
    rp::Shape sh;
    return resolve_pair_plan(a, plan, sm_count, &sh);
}

// Plan for matrices read and written over the host link. There every plan is
// bound by the link (about 210 GB/s host-to-device and 193 GB/s back, 340 GB/s
// both at once, the same as the copy engines). With both matrices on the host,
// one cluster per row comes closest to that. Measured on GB300 against the
// device plans: 325 vs 290 GB/s on f32 4096 x 4096, 301 vs 239 GB/s on bf16
// 16384 x 1000, and 342 vs 333 GB/s on f16 65536 x 2048. Below a few MiB the
// call is launch-bound and the device choice stays.
constexpr int64_t kMappedWideMinBytes = 8ll << 20;

int mapped_plan(const void* in, const void* out, int64_t M, int64_t N, int64_t ld_in,
                int64_t ld_out, int dtype) {
    if (M * N * elem_bytes(dtype) >= kMappedWideMinBytes &&
        plan_fits(SR_PLAN_WIDE, in, out, N, ld_in, ld_out, dtype))
        return SR_PLAN_WIDE;
    return SR_PLAN_AUTO;
}

int launch_auto(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in, int64_t ld_out,
                int dtype, cudaStream_t stream) {
    return run(in, out, M, N, ld_in, ld_out, dtype, SR_PLAN_AUTO, stream, kDefaultTimeoutNs, 0);
}

}  // namespace
}  // namespace sr

extern "C" {

int softmax_rows(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in, int64_t ld_out,
                 int dtype, sr_stream_t stream) {
    return sr::run(in, out, M, N, ld_in, ld_out, dtype, SR_PLAN_AUTO, (cudaStream_t)stream,
                   sr::kDefaultTimeoutNs, 0);
}

int softmax_rows_ex(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in,
                    int64_t ld_out, int dtype, int plan, sr_stream_t stream) {
    if (plan < SR_PLAN_AUTO || plan > SR_PLAN_WIDE) return SR_EPLAN;
    return sr::run(in, out, M, N, ld_in, ld_out, dtype, plan, (cudaStream_t)stream,
                   sr::kDefaultTimeoutNs, 0);
}

int softmax_rows_plan(const void* in, const void* out, int64_t M, int64_t N, int64_t ld_in,
                      int64_t ld_out, int dtype) {
    const int bad = sr::check_args(in, out, M, N, ld_in, ld_out, dtype);
    if (bad) return -bad;
    return sr::choose_plan(in, out, N, ld_in, ld_out, dtype);
}

int softmax_rows_plan_check(const void* in, const void* out, int64_t M, int64_t N,
                            int64_t ld_in, int64_t ld_out, int dtype, int plan) {
    const int bad = sr::check_args(in, out, M, N, ld_in, ld_out, dtype);
    if (bad) return -bad;
    if (plan == SR_PLAN_AUTO) return sr::choose_plan(in, out, N, ld_in, ld_out, dtype);
    if (plan < SR_PLAN_AUTO || plan > SR_PLAN_WIDE) return -SR_EPLAN;
    return sr::plan_fits(plan, in, out, N, ld_in, ld_out, dtype) ? plan : -SR_EPLAN;
}

int softmax_rows_last_device_error(sr_stream_t stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SR_ECUDA;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, sr::g_error_word, sizeof(word)) != cudaSuccess) return SR_ECUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(sr::g_error_word, &zero, sizeof(zero)) != cudaSuccess)
            return SR_ECUDA;
        return (word & sr::kErrBounds) ? SR_EBOUNDS : SR_EDEVICE_TIMEOUT;
    }
    return SR_OK;
}

int softmax_rows_test_expiry(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in,
                             int64_t ld_out, int dtype, int plan, uint64_t timeout_ns,
                             sr_stream_t stream) {
    if (plan != SR_PLAN_CTA && plan != SR_PLAN_CLUSTER && plan != SR_PLAN_SMEM &&
        plan != SR_PLAN_WIDE)
        return SR_EPLAN;
    return sr::run(in, out, M, N, ld_in, ld_out, dtype, plan, (cudaStream_t)stream,
                   (unsigned long long)timeout_ns, sr::kFlagNoCopy);
}

int softmax_rows_masked(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in,
                        int64_t ld_out, int dtype, const int32_t* lengths, int64_t causal_period,
                        int plan, sr_stream_t stream) {
    const int bad = sr::check_args(in, out, M, N, ld_in, ld_out, dtype);
    if (bad) return bad;
    if (causal_period < 0 || (lengths != nullptr && causal_period != 0)) return SR_EINVAL;
    if (plan == SR_PLAN_AUTO) {
        plan = sr::choose_masked_plan(in, out, N, ld_in, ld_out, dtype);
    } else if (!sr::masked_plan_fits(plan, in, out, N, ld_in, ld_out, dtype)) {
        return SR_EPLAN;
    }
    if (M == 0) return SR_OK;
    if (M > 0 && lengths == nullptr && causal_period == 0)  // no mask: the plain softmax
        return softmax_rows_ex(in, out, M, N, ld_in, ld_out, dtype, plan, stream);
    cudaError_t e;
    const sr::DeviceInfo* dev = sr::device_info(&e);
    if (!dev) return SR_ECUDA;
    sr::Problem p{in, out, M, N, ld_in, ld_out, dtype, (cudaStream_t)stream, dev,
                  sr::kDefaultTimeoutNs, 0};
    p.mask.lens = lengths;
    p.mask.period = causal_period;
    switch (plan) {
        case SR_PLAN_WARP: e = sr::launch_warp(p); break;
        case SR_PLAN_ROW: e = sr::launch_row(p); break;
        case SR_PLAN_ONLINE: e = sr::launch_online(p); break;
        default: return SR_EPLAN;
    }
    return e == cudaSuccess ? SR_OK : SR_ECUDA;
}

int64_t softmax_rows_split_workspace_bytes(const void* in, const void* out, int64_t M, int64_t N,
                                           int64_t ld_in, int64_t ld_out, int dtype) {
    const int bad = sr::check_args(in, out, M, N, ld_in, ld_out, dtype);
    if (bad) return -bad;
    return sr::kSplitWorkspaceBytes;
}

namespace sr {
namespace {

// Blocks of the SPLIT kernel the current device holds at once.
int split_max_blocks(const DeviceInfo* dev, int dtype, int vec) {
    const void* func = split_kernel(dtype, vec);
    const size_t smem = split_smem(vec);
    if (smem > 0 && ensure_smem_limit(func, smem, false) != cudaSuccess) return -1;
    const int per_sm = blocks_per_sm(func, split_threads(vec), smem);
    if (per_sm <= 0) return -1;
    const int64_t n = (int64_t)per_sm * dev->sm_count;
    return n > kSplitMaxBlocks ? kSplitMaxBlocks : (int)n;
}

int run_split(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in, int64_t ld_out,
              int dtype, void* workspace, int64_t workspace_bytes, cudaStream_t stream,
              unsigned long long timeout_ns, int flags) {
    const int bad = check_args(in, out, M, N, ld_in, ld_out, dtype);
    if (bad) return bad;
    if (M == 0) return SR_OK;
    if (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 16 != 0 ||
        workspace_bytes < kSplitWorkspaceBytes)
        return SR_EINVAL;
    if (in == out) return SR_EINVAL;  // the second pass rereads the input
    cudaError_t e;
    const DeviceInfo* dev = device_info(&e);
    if (!dev) return SR_ECUDA;
    const bool vec = rows_vector_aligned(in, out, N, ld_in, ld_out, dtype);
    const int max_blocks = split_max_blocks(dev, dtype, vec ? 2 : 1);
    if (max_blocks <= 0) return SR_ECUDA;
    const SplitShape sh = split_shape(M, N, ld_in, ld_out, dtype, in, out, max_blocks,
                                      dev->l2_bytes);
    Problem p{in, out, M, N, ld_in, ld_out, dtype, stream, dev, timeout_ns, flags};
    return launch_split(p, sh, workspace) == cudaSuccess ? SR_OK : SR_ECUDA;
}

}  // namespace
}  // namespace sr

int softmax_rows_split(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in,
                       int64_t ld_out, int dtype, void* workspace, int64_t workspace_bytes,
                       sr_stream_t stream) {
    return sr::run_split(in, out, M, N, ld_in, ld_out, dtype, workspace, workspace_bytes,
                         (cudaStream_t)stream, sr::kDefaultTimeoutNs, 0);
}

int softmax_rows_split_test_expiry(const void* in, void* out, int64_t M, int64_t N,
                                   int64_t ld_in, int64_t ld_out, int dtype, void* workspace,
                                   int64_t workspace_bytes, uint64_t timeout_ns,
                                   sr_stream_t stream) {
    return sr::run_split(in, out, M, N, ld_in, ld_out, dtype, workspace, workspace_bytes,
                         (cudaStream_t)stream, (unsigned long long)timeout_ns,
                         sr::kFlagNoArrive);
}

int softmax_rows_split_shape(const void* in, const void* out, int64_t M, int64_t N,
                             int64_t ld_in, int64_t ld_out, int dtype, int max_blocks,
                             int64_t l2_bytes, sr_split_shape* shape) {
    const int bad = sr::check_args(in, out, M, N, ld_in, ld_out, dtype);
    if (bad) return bad;
    if (shape == nullptr) return SR_EINVAL;
    if (max_blocks <= 0 || l2_bytes <= 0) {
        cudaError_t e;
        const sr::DeviceInfo* dev = sr::device_info(&e);
        if (!dev) return SR_ECUDA;
        const bool vec = sr::rows_vector_aligned(in, out, N, ld_in, ld_out, dtype);
        if (max_blocks <= 0) max_blocks = sr::split_max_blocks(dev, dtype, vec ? 2 : 1);
        if (max_blocks <= 0) return SR_ECUDA;
        if (l2_bytes <= 0) l2_bytes = dev->l2_bytes;
    }
    const sr::SplitShape sh =
        sr::split_shape(M, N, ld_in, ld_out, dtype, in, out, max_blocks, l2_bytes);
    shape->lanes = sh.lanes;
    shape->parts = sh.parts;
    shape->part_units = sh.part_units;
    shape->unit_elems = sh.vec;
    return SR_OK;
}

int64_t softmax_rows_host_workspace_bytes(int64_t M, int64_t N, int dtype) {
    if (dtype != SR_F32 && dtype != SR_BF16 && dtype != SR_F16) return -SR_EDTYPE;
    if (M < 0 || N < 1) return -SR_EINVAL;
    return sr::host_workspace_bytes(M, N, dtype);
}

int softmax_rows_host_mapped(const void* h_in, void* h_out, int64_t M, int64_t N, int64_t ld_in,
                             int64_t ld_out, int dtype, sr_stream_t stream) {
    const int bad = sr::check_args(h_in, h_out, M, N, ld_in, ld_out, dtype);
    if (bad) return bad;
    if (M == 0) return SR_OK;
    // Only memory the device can address: page-locked host memory mapped into
    // the device's address space (or managed memory). Anything else is
    // refused before a kernel could touch it.
    void* dptr[2] = {nullptr, nullptr};
    const void* hptr[2] = {h_in, h_out};
    for (int i = 0; i < 2; ++i) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, hptr[i]) != cudaSuccess) {
            (void)cudaGetLastError();  // clear the sticky-free error of an unknown pointer
            return SR_EINVAL;
        }
        if ((at.type != cudaMemoryTypeHost && at.type != cudaMemoryTypeManaged) ||
            at.devicePointer == nullptr)
            return SR_EINVAL;
        dptr[i] = at.devicePointer;
    }
    return sr::run(dptr[0], dptr[1], M, N, ld_in, ld_out, dtype,
                   sr::mapped_plan(dptr[0], dptr[1], M, N, ld_in, ld_out, dtype),
                   (cudaStream_t)stream, sr::kDefaultTimeoutNs, 0);
}

int softmax_rows_host(const void* h_in, void* h_out, int64_t M, int64_t N, int64_t ld_in,
                      int64_t ld_out, int dtype, void* d_work, int64_t work_bytes,
                      sr_stream_t stream) {
    const int bad = sr::check_args(h_in, h_out, M, N, ld_in, ld_out, dtype);
    if (bad) return bad;
    if (M == 0) return SR_OK;
    return sr::run_host(h_in, h_out, M, N, ld_in, ld_out, dtype, d_work, work_bytes,
                        (cudaStream_t)stream, sr::launch_auto);
}

int softmax_rows_backward(const void* y, const void* dy, void* dx, int64_t M, int64_t N,
                          int64_t ld_y, int64_t ld_dy, int64_t ld_dx, int dtype,
                          sr_stream_t stream) {
    return sr::run_bwd(y, dy, dx, M, N, ld_y, ld_dy, ld_dx, dtype, SR_PLAN_AUTO,
                       (cudaStream_t)stream);
}

int softmax_rows_backward_ex(const void* y, const void* dy, void* dx, int64_t M, int64_t N,
                             int64_t ld_y, int64_t ld_dy, int64_t ld_dx, int dtype, int plan,
                             sr_stream_t stream) {
    return sr::run_bwd(y, dy, dx, M, N, ld_y, ld_dy, ld_dx, dtype, plan, (cudaStream_t)stream);
}

int softmax_rows_backward_test_expiry(const void* y, const void* dy, void* dx, int64_t M,
                                      int64_t N, int64_t ld_y, int64_t ld_dy, int64_t ld_dx,
                                      int dtype, uint64_t timeout_ns, sr_stream_t stream) {
    const int bad = sr::check_bwd_args(y, dy, dx, M, N, ld_y, ld_dy, ld_dx, dtype);
    if (bad) return bad;
    sr::rp::Args a{y, dy, dx, M, N, ld_y, ld_dy, ld_dx, dtype, (cudaStream_t)stream};
    a.flags = sr::kFlagNoCopy;
    return sr::run_pair(
        a, SR_PLAN_CLUSTER,
        [](const sr::rp::Args& q, const sr::rp::Shape& sh) { return sr::launch_backward(q, sh); },
        (unsigned long long)timeout_ns);
}

int softmax_rows_backward_plan(const void* y, const void* dy, const void* dx, int64_t M,
                               int64_t N, int64_t ld_y, int64_t ld_dy, int64_t ld_dx, int dtype,
                               int plan, int sm_count) {
    const int bad = sr::check_bwd_args(y, dy, dx, M, N, ld_y, ld_dy, ld_dx, dtype);
    if (bad) return -bad;
    const sr::rp::Args a{y, dy, const_cast<void*>(dx), M, N, ld_y, ld_dy, ld_dx, dtype, nullptr};
    return sr::pair_plan_query(a, plan, sm_count);
}

int rmsnorm_residual_rows_ex(const void* x, const void* residual, const void* weight, void* y,
                             int64_t M, int64_t N, int64_t ld_x, int64_t ld_r, int64_t ld_y,
                             float eps, int dtype, int plan, sr_stream_t stream) {
    const int bad = sr::check_rms_args(x, residual, weight, y, M, N, ld_x, ld_r, ld_y, eps, dtype);
    if (bad) return bad;
    sr::rp::Args a{x, residual, y, M, N, ld_x, ld_r, ld_y, dtype, (cudaStream_t)stream};
    a.stream_wide = true;
    return sr::run_pair(a, plan, [weight, eps](const sr::rp::Args& q, const sr::rp::Shape& sh) {
        return sr::launch_rmsnorm(q, sh, weight, eps);
    });
}

int rmsnorm_residual_rows(const void* x, const void* residual, const void* weight, void* y,
                          int64_t M, int64_t N, int64_t ld_x, int64_t ld_r, int64_t ld_y,
                          float eps, int dtype, sr_stream_t stream) {
    return rmsnorm_residual_rows_ex(x, residual, weight, y, M, N, ld_x, ld_r, ld_y, eps, dtype,
                                    SR_PLAN_AUTO, stream);
}

int rmsnorm_residual_rows_plan(const void* x, const void* residual, const void* weight,
                               const void* y, int64_t M, int64_t N, int64_t ld_x, int64_t ld_r,
                               int64_t ld_y, float eps, int dtype, int plan, int sm_count) {
    const int bad = sr::check_rms_args(x, residual, weight, y, M, N, ld_x, ld_r, ld_y, eps, dtype);
    if (bad) return -bad;
    sr::rp::Args a{x, residual, const_cast<void*>(y), M, N, ld_x, ld_r, ld_y, dtype, nullptr};
    a.stream_wide = true;
    return sr::pair_plan_query(a, plan, sm_count);
}

const char* softmax_rows_strerror(int status) {
    switch (status) {
        case SR_OK: return "success";
        case SR_EINVAL: return "invalid size, pitch or pointer";
        case SR_EDTYPE: return "unknown dtype";
        case SR_ECUDA: return "CUDA runtime error";
        case SR_EDEVICE_TIMEOUT: return "a bounded device wait expired";
        case SR_EPLAN: return "plan cannot handle this shape or alignment";
        case SR_EBOUNDS: return "a device access fell outside the call's matrices (bounds check)";
    }
    return "unknown status";
}

int softmax_rows_wide_shape(int64_t M, int64_t N, int dtype, int sm_count, int* csize, int* kv,
                            int64_t* slice, int* streamed) {
    if (dtype != SR_F32 && dtype != SR_BF16 && dtype != SR_F16) return -SR_EDTYPE;
    if (M < 0 || N < 1 || sm_count < 1) return -SR_EINVAL;
    sr::WideShape sh;
    if (!sr::wide_shape(M, N, dtype, sm_count, &sh)) return -SR_EINVAL;
    if (csize) *csize = sh.csize;
    if (kv) *kv = sh.kv;
    if (slice) *slice = sh.slice;
    if (streamed) *streamed = sh.streamed ? 1 : 0;
    return 0;
}

int softmax_rows_last_launch(sr_launch_info* info) {
    const sr::LaunchRecord& r = sr::t_last_launch;
    if (info == nullptr || r.func == nullptr) return SR_EINVAL;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, r.func) != cudaSuccess) return SR_ECUDA;
    info->registers = fa.numRegs;
    info->local_bytes = (int)fa.localSizeBytes;
    info->static_smem_bytes = (int)fa.sharedSizeBytes;
    info->dynamic_smem_bytes = (int)r.smem;
    info->grid = (int)r.grid.x;
    info->block = (int)r.block.x;
    info->cluster = r.cluster;
    info->name[0] = '\0';
    const char* name = nullptr;
    if (cudaFuncGetName(&name, r.func) == cudaSuccess && name != nullptr) {
        size_t k = 0;
        for (; name[k] != '\0' && k + 1 < sizeof(info->name); ++k) info->name[k] = name[k];
        info->name[k] = '\0';
    }
    return SR_OK;
}

int softmax_rows_copy_ceiling2(const void* a, const void* b, void* out, int64_t M,
                               int64_t row_bytes, int64_t ld_a_bytes, int64_t ld_b_bytes,
                               int64_t ld_out_bytes, sr_stream_t stream) {
    if (M < 0 || row_bytes < 1 || ld_a_bytes < row_bytes || ld_b_bytes < row_bytes ||
        ld_out_bytes < row_bytes)
        return SR_EINVAL;
    if (M > 0 && (a == nullptr || b == nullptr || out == nullptr)) return SR_EINVAL;
    if (M > 0) {
        __int128 ld = ld_a_bytes > ld_b_bytes ? ld_a_bytes : ld_b_bytes;
        if (ld_out_bytes > ld) ld = ld_out_bytes;
        if ((__int128)(M - 1) * ld + row_bytes > (__int128)INT64_MAX) return SR_EINVAL;
    }
    if (M == 0) return SR_OK;
    cudaError_t e;
    const sr::DeviceInfo* dev = sr::device_info(&e);
    if (!dev) return SR_ECUDA;
    return sr::launch_copy_pair(a, b, out, M, row_bytes, ld_a_bytes, ld_b_bytes, ld_out_bytes,
                                (cudaStream_t)stream) == cudaSuccess
               ? SR_OK
               : SR_ECUDA;
}

int softmax_rows_copy_ceiling(const void* in, void* out, int64_t M, int64_t row_bytes,
                              int64_t ld_in_bytes, int64_t ld_out_bytes, sr_stream_t stream) {
    if (M < 0 || row_bytes < 1 || ld_in_bytes < row_bytes || ld_out_bytes < row_bytes)
        return SR_EINVAL;
    if (M > 0 && (in == nullptr || out == nullptr)) return SR_EINVAL;
    if (M > 0) {
        const __int128 ld = ld_in_bytes > ld_out_bytes ? ld_in_bytes : ld_out_bytes;
        if ((__int128)(M - 1) * ld + row_bytes > (__int128)INT64_MAX) return SR_EINVAL;
    }
    if (M == 0) return SR_OK;
    cudaError_t e;
    const sr::DeviceInfo* dev = sr::device_info(&e);
    if (!dev) return SR_ECUDA;
    return sr::launch_copy_rows(in, out, M, row_bytes, ld_in_bytes, ld_out_bytes,
                                (cudaStream_t)stream, dev->sm_count) == cudaSuccess
               ? SR_OK
               : SR_ECUDA;
}

int softmax_rows_build_flags(void) { return SR_BOUNDS_CHECK ? SR_BUILD_BOUNDS_CHECK : 0; }

uint64_t softmax_rows_bounds_address(void) {
#if SR_BOUNDS_CHECK
    unsigned long long a = 0;
    if (cudaMemcpyFromSymbol(&a, sr::g_bounds_addr, sizeof(a)) != cudaSuccess) return 0;
    const unsigned long long zero = 0;
    if (cudaMemcpyToSymbol(sr::g_bounds_addr, &zero, sizeof(zero)) != cudaSuccess) return 0;
    return (uint64_t)a;
#else
    return 0;
#endif
}

int softmax_rows_test_bounds_shrink(int64_t bytes) {
#if SR_BOUNDS_CHECK
    if (bytes < 0) return SR_EINVAL;
    const long long v = (long long)bytes;
    return cudaMemcpyToSymbol(sr::g_bounds_shrink, &v, sizeof(v)) == cudaSuccess ? SR_OK
                                                                                 : SR_ECUDA;
#else
    (void)bytes;
    return SR_EINVAL;
#endif
}

int softmax_rows_version(void) { return 210; }

}  // extern "C"
