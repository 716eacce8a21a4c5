// End-to-end entry point on host buffers: rows stream through a
// double-buffered device workspace in chunks, and three streams overlap the
// host->device copy of chunk c+1, the kernel on chunk c and the
// device->host copy of chunk c-1.
//
//   h2d stream:      wait compute[b] -> copy in (x, r) -> record h2d[b]
//   caller stream:   wait h2d[b], wait d2h[b] -> kernel -> record compute[b]
//   d2h stream:      wait compute[b] -> copy out y -> record d2h[b]
//
// b = c % 2.  Each wait is issued after the record it must see (chunks are
// enqueued in order), so chunk c+2 reuses buffer b only once chunk c's
// kernel has consumed the inputs and chunk c's output has left the device.
//
// When the output buffer is pinned host memory the device can address (over
// NVLink-C2C on Grace systems), the kernels store each chunk's results
// straight into it and the device->host copies are skipped: the copy
// engines then carry only the inputs, which is what bounds the pipeline.
#include "../../include/tile_rows.h"

#include <cmath>
#include <cstdint>
#include <mutex>

#include "launch.h"

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

int tensors_of(int op) { return op == TILE_OP_RESIDUAL_LAYERNORM ? 3 : 2; }

// Internal streams and events, created once per device.
struct DeviceQueues {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t h2d_ev[2] = {}, compute_ev[2] = {}, d2h_ev[2] = {};
    std::mutex mu;
};

DeviceQueues g_queues[tile::kMaxDevices];

cudaError_t ensure_queues(DeviceQueues &q) {
    if (q.ready) return cudaSuccess;
    cudaError_t err = cudaStreamCreateWithFlags(&q.h2d, cudaStreamNonBlocking);
    if (err == cudaSuccess) err = cudaStreamCreateWithFlags(&q.d2h, cudaStreamNonBlocking);
    const unsigned flags = cudaEventDisableTiming;
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&q.start, flags);
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&q.done, flags);
    for (int b = 0; b < 2 && err == cudaSuccess; ++b) {
        err = cudaEventCreateWithFlags(&q.h2d_ev[b], flags);
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&q.compute_ev[b], flags);
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&q.d2h_ev[b], flags);
    }
    if (err == cudaSuccess) q.ready = true;
    return err;
}

bool overlaps(const void *a, const void *b, size_t bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bytes && y < x + bytes;
}

}  // namespace

namespace tile {

// Rows per chunk for a workspace of `work_bytes`: as many as fit twice
// (double buffering), at most ceil(rows/8) so the pipeline has stages to
// overlap, and at least 1 (0 if not even one row fits).
long long host_chunk_rows(int op, int rows, int width, size_t work_bytes) {
    const size_t row_bytes = static_cast<size_t>(width) * sizeof(float);
    const size_t per_buffer = work_bytes / (2 * static_cast<size_t>(tensors_of(op)));
    long long fit = static_cast<long long>((per_buffer / kAlign * kAlign) / row_bytes);
    const long long stage = (static_cast<long long>(rows) + 7) / 8;
    if (fit > stage) fit = stage;
    return fit;
}

// The pipeline over caller-provided workspace (also used by the entry point
// that stages through the library's static device area).
int run_host(int op, const float *h_in, const float *h_res, float *h_out, int rows, int width,
             float eps, void *d_work, size_t work_bytes, cudaStream_t stream) {
    if (op < TILE_OP_RESIDUAL_LAYERNORM || op > TILE_OP_SOFTMAX) return TILE_ERR_OP;
    if (rows < 0 || width < 1 || width > tile_max_width()) return TILE_ERR_SHAPE;
    if (op != TILE_OP_SOFTMAX && !(std::isfinite(eps) && eps >= 0.0f)) return TILE_ERR_EPS;
    if (rows == 0) return TILE_OK;
    const bool residual = op == TILE_OP_RESIDUAL_LAYERNORM;
    if (h_in == nullptr || h_out == nullptr || (residual && h_res == nullptr) || d_work == nullptr)
        return TILE_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(d_work) & (kAlign - 1)) != 0) return TILE_ERR_ALIGN;
    const size_t total = static_cast<size_t>(rows) * static_cast<size_t>(width) * sizeof(float);
    if (overlaps(h_out, h_in, total) || (residual && overlaps(h_out, h_res, total)))
        return TILE_ERR_ALIAS;
    const long long chunk = host_chunk_rows(op, rows, width, work_bytes);
    if (chunk < 1) return TILE_ERR_WORKSPACE;

    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess && (dev < 0 || dev >= kMaxDevices)) err = cudaErrorInvalidDevice;
    if (err != cudaSuccess) {
        set_last_cuda_error(static_cast<int>(err));
        return TILE_ERR_CUDA;
    }
    DeviceQueues &q = g_queues[dev];
    std::lock_guard<std::mutex> lock(q.mu);
    err = ensure_queues(q);
    if (err != cudaSuccess) {
        set_last_cuda_error(static_cast<int>(err));
        return TILE_ERR_CUDA;
    }

    // Pinned, device-addressable output: the kernels write it directly.
    float *out_dev = nullptr;
    {
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, h_out) == cudaSuccess &&
            attr.type == cudaMemoryTypeHost && attr.devicePointer != nullptr)
            out_dev = static_cast<float *>(attr.devicePointer);
        else
            (void)cudaGetLastError();   // clear a non-sticky error of the query
    }

    const size_t buf = round_up(static_cast<size_t>(chunk) * width * sizeof(float));
    char *base = static_cast<char *>(d_work);
    float *dx[2], *dr[2], *dy[2];
    for (int b = 0; b < 2; ++b) {
        char *p = base + static_cast<size_t>(b) * tensors_of(op) * buf;
        dx[b] = reinterpret_cast<float *>(p);
        dr[b] = residual ? reinterpret_cast<float *>(p + buf) : nullptr;
        dy[b] = reinterpret_cast<float *>(p + (residual ? 2 : 1) * buf);
    }

    // Everything enqueued here runs after the work already on `stream`.
#define TILE_TRY(call)                                          \
    do {                                                        \
        err = (call);                                           \
        if (err != cudaSuccess) {                               \
            set_last_cuda_error(static_cast<int>(err));         \
            return TILE_ERR_CUDA;                               \
        }                                                       \
    } while (0)

    TILE_TRY(cudaEventRecord(q.start, stream));
    TILE_TRY(cudaStreamWaitEvent(q.h2d, q.start, 0));
    TILE_TRY(cudaStreamWaitEvent(q.d2h, q.start, 0));

    const long long nchunks = (rows + chunk - 1) / chunk;
    for (long long c = 0; c < nchunks; ++c) {
        const int b = static_cast<int>(c & 1);
        const long long r0 = c * chunk;
        const int n = static_cast<int>(rows - r0 < chunk ? rows - r0 : chunk);
        const size_t off = static_cast<size_t>(r0) * width;
        const size_t bytes = static_cast<size_t>(n) * width * sizeof(float);
        if (c >= 2) TILE_TRY(cudaStreamWaitEvent(q.h2d, q.compute_ev[b], 0));
        TILE_TRY(cudaMemcpyAsync(dx[b], h_in + off, bytes, cudaMemcpyHostToDevice, q.h2d));
        if (residual)
            TILE_TRY(cudaMemcpyAsync(dr[b], h_res + off, bytes, cudaMemcpyHostToDevice, q.h2d));
        TILE_TRY(cudaEventRecord(q.h2d_ev[b], q.h2d));

        TILE_TRY(cudaStreamWaitEvent(stream, q.h2d_ev[b], 0));
        if (out_dev != nullptr) {
            const int st = run_selected(op, dx[b], dr[b], out_dev + off, n, width, eps, stream);
            if (st != TILE_OK) return st;
            TILE_TRY(cudaEventRecord(q.compute_ev[b], stream));
            continue;
        }
        if (c >= 2) TILE_TRY(cudaStreamWaitEvent(stream, q.d2h_ev[b], 0));
        const int st = run_selected(op, dx[b], dr[b], dy[b], n, width, eps, stream);
        if (st != TILE_OK) return st;
        TILE_TRY(cudaEventRecord(q.compute_ev[b], stream));

        TILE_TRY(cudaStreamWaitEvent(q.d2h, q.compute_ev[b], 0));
        TILE_TRY(cudaMemcpyAsync(h_out + off, dy[b], bytes, cudaMemcpyDeviceToHost, q.d2h));
        TILE_TRY(cudaEventRecord(q.d2h_ev[b], q.d2h));
    }
    // The caller's stream is ordered after the last copy out (and the copies
    // in, which precede it).
    TILE_TRY(cudaEventRecord(q.done, q.d2h));
    TILE_TRY(cudaStreamWaitEvent(stream, q.done, 0));
    TILE_TRY(cudaEventRecord(q.done, q.h2d));
    TILE_TRY(cudaStreamWaitEvent(stream, q.done, 0));
#undef TILE_TRY
    return TILE_OK;
}

}  // namespace tile

extern "C" {

size_t tile_host_workspace_bytes(int op, int width, int chunk_rows) {
    if (op < TILE_OP_RESIDUAL_LAYERNORM || op > TILE_OP_SOFTMAX || width < 1 || chunk_rows < 1)
        return 0;
    return 2 * static_cast<size_t>(tensors_of(op)) *
           round_up(static_cast<size_t>(chunk_rows) * width * sizeof(float));
}

int tile_run_host_f32(int op, const float *h_in, const float *h_residual, float *h_out, int rows,
                      int width, float eps, void *d_work, size_t work_bytes,
                      cudaStream_t stream) {
    return tile::run_host(op, h_in, h_residual, h_out, rows, width, eps, d_work, work_bytes,
                          stream);
}

}  // extern "C"
