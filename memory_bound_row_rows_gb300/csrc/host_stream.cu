// Host-resident matrices streamed through the device: softmax_rows_host.
//
// Rows are cut into chunks. Chunk c is copied host -> device into workspace
// slot c % S, reduced there by the usual kernels, and copied back, on three
// library-owned streams (copy-in, compute, copy-out) so that on a GB300 the
// host link carries both directions while the SMs work on a third chunk.
// Events order the stages of one chunk and keep a slot from being refilled
// before its previous chunk has been copied out. The caller's stream is
// joined at both ends: the pipeline starts after the work already queued on
// it, and it waits for the last copy-out.
#include <mutex>

#include "../../include/softmax_rows.h"
#include "internal.h"

namespace sr {
namespace {

constexpr int kMaxSlots = 4;
constexpr int kMaxDevices = 64;
// Preferred bytes of input per chunk: large enough to amortise a copy's
// fixed cost, small enough to pipeline several chunks.
constexpr int64_t kChunkTarget = 8ll << 20;

struct Pipeline {
    bool ready = false;
    cudaStream_t s_in = nullptr, s_run = nullptr, s_out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t copied_in[kMaxSlots] = {}, computed[kMaxSlots] = {}, copied_out[kMaxSlots] = {};
};

std::mutex g_pipe_mu;
Pipeline g_pipe[kMaxDevices];

cudaError_t pipeline_for(int dev, Pipeline** out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    Pipeline& p = g_pipe[dev];
    if (!p.ready) {
        cudaError_t e;
        const unsigned fl = cudaEventDisableTiming;
        if ((e = cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking)) ||
            (e = cudaStreamCreateWithFlags(&p.s_run, cudaStreamNonBlocking)) ||
            (e = cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking)) ||
            (e = cudaEventCreateWithFlags(&p.start, fl)) ||
            (e = cudaEventCreateWithFlags(&p.done, fl)))
            return e;
        for (int k = 0; k < kMaxSlots; ++k) {
            if ((e = cudaEventCreateWithFlags(&p.copied_in[k], fl)) ||
                (e = cudaEventCreateWithFlags(&p.computed[k], fl)) ||
                (e = cudaEventCreateWithFlags(&p.copied_out[k], fl)))
                return e;
        }
        p.ready = true;
    }
    *out = &p;
    return cudaSuccess;
}

// Device pitch of a staged row: the row rounded up to 16 bytes, so staged
// rows are always 16-byte aligned.
int64_t staged_pitch(int64_t N, int dtype) {
    const int64_t es = elem_bytes(dtype);
    return ((N * es + 15) / 16 * 16) / es;
}

cudaError_t copy_rows(void* dst, int64_t dld, const void* src, int64_t sld, int64_t N,
                      int64_t rows, int dtype, cudaMemcpyKind kind, cudaStream_t s) {
    const int64_t es = elem_bytes(dtype);
    if (dld == N && sld == N)
        return cudaMemcpyAsync(dst, src, (size_t)(rows * N * es), kind, s);
    return cudaMemcpy2DAsync(dst, (size_t)(dld * es), src, (size_t)(sld * es), (size_t)(N * es),
                             (size_t)rows, kind, s);
}

}  // namespace

// Workspace that lets the pipeline run at full depth (kMaxSlots chunks of up
// to kChunkTarget input bytes); any size from two staged rows up works.
int64_t host_workspace_bytes(int64_t M, int64_t N, int dtype) {
    const int64_t es = elem_bytes(dtype);
    const int64_t ldd = staged_pitch(N, dtype);
    int64_t rows = kChunkTarget / (ldd * es);
    if (rows < 1) rows = 1;
    if (rows > M) rows = M < 1 ? 1 : M;
    return (int64_t)kMaxSlots * rows * 2 * ldd * es;
}

int run_host(const void* h_in, void* h_out, int64_t M, int64_t N, int64_t ld_in, int64_t ld_out,
             int dtype, void* d_work, int64_t work_bytes, cudaStream_t stream,
             int (*launch)(const void*, void*, int64_t, int64_t, int64_t, int64_t, int,
                           cudaStream_t)) {
    const int64_t es = elem_bytes(dtype);
    const int64_t ldd = staged_pitch(N, dtype);
    const int64_t row_bytes = 2 * ldd * es;  // one staged row, in and out
    if (d_work == nullptr || work_bytes < 2 * row_bytes) return SR_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_work) % 16 != 0) return SR_EINVAL;

    // Rows per chunk and slots: at most kChunkTarget of input per chunk,
    // as many slots (2..4) as the workspace holds.
    int64_t rows = kChunkTarget / (ldd * es);
    if (rows < 1) rows = 1;
    if (rows > M) rows = M;
    int slots = (int)(work_bytes / (rows * row_bytes));
    if (slots < 2) {
        rows = work_bytes / (2 * row_bytes);
        slots = 2;
    }
    if (slots > kMaxSlots) slots = kMaxSlots;
    const int64_t nchunks = (M + rows - 1) / rows;
    if (nchunks < slots) slots = (int)(nchunks < 2 ? 2 : nchunks);

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SR_ECUDA;
    std::lock_guard<std::mutex> lk(g_pipe_mu);
    Pipeline* p = nullptr;
    if (pipeline_for(dev, &p) != cudaSuccess) return SR_ECUDA;

    char* base = static_cast<char*>(d_work);
    const int64_t slot_bytes = rows * row_bytes;
    if (cudaEventRecord(p->start, stream) || cudaStreamWaitEvent(p->s_in, p->start, 0) ||
        cudaStreamWaitEvent(p->s_run, p->start, 0) ||
        cudaStreamWaitEvent(p->s_out, p->start, 0))
        return SR_ECUDA;

    for (int64_t c = 0; c < nchunks; ++c) {
        const int k = (int)(c % slots);
        const int64_t r0 = c * rows;
        const int64_t nr = (M - r0 < rows) ? (M - r0) : rows;
        void* d_in = base + k * slot_bytes;
        void* d_out = base + k * slot_bytes + rows * ldd * es;
        const char* src = static_cast<const char*>(h_in) + r0 * ld_in * es;
        char* dst = static_cast<char*>(h_out) + r0 * ld_out * es;
        // Copy in once the slot's previous chunk has been copied out.
        if (c >= slots && cudaStreamWaitEvent(p->s_in, p->copied_out[k], 0)) return SR_ECUDA;
        if (copy_rows(d_in, ldd, src, ld_in, N, nr, dtype, cudaMemcpyHostToDevice, p->s_in) ||
            cudaEventRecord(p->copied_in[k], p->s_in))
            return SR_ECUDA;
        // Compute.
        if (cudaStreamWaitEvent(p->s_run, p->copied_in[k], 0)) return SR_ECUDA;
        const int st = launch(d_in, d_out, nr, N, ldd, ldd, dtype, p->s_run);
        if (st != SR_OK) return st;
        if (cudaEventRecord(p->computed[k], p->s_run)) return SR_ECUDA;
        // Copy out.
        if (cudaStreamWaitEvent(p->s_out, p->computed[k], 0) ||
            copy_rows(dst, ld_out, d_out, ldd, N, nr, dtype, cudaMemcpyDeviceToHost, p->s_out) ||
            cudaEventRecord(p->copied_out[k], p->s_out))
            return SR_ECUDA;
    }
    if (cudaEventRecord(p->done, p->s_out) || cudaStreamWaitEvent(stream, p->done, 0))
        return SR_ECUDA;
    return SR_OK;
}

}  // namespace sr
