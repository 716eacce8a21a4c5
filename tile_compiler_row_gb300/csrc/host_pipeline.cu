// End-to-end entry point on host buffers: rows stream through a ring of
// device buffers ("slots") carved from the caller's workspace, in chunks,
// and three streams overlap the host->device copy of chunk c+1, the kernel
// on chunk c and the device->host copy of chunk c-1.
//
//   h2d stream:      wait compute[b] -> copy in (x, r) -> record h2d[b]
//   caller stream:   wait h2d[b], wait d2h[b] -> kernel -> record compute[b]
//   d2h stream:      wait compute[b] -> copy out y -> record d2h[b]
//
// b = c % slots.  Each wait is issued after the record it must see (chunks
// are enqueued in order), so chunk c+slots reuses slot b only once chunk c's
// kernel has consumed the inputs and chunk c's output has left the device.
// More than two slots let the copies in run ahead of a kernel that is slow
// to finish (one that writes its results over the host link).  Every chunk
// runs the plan a device call on the whole matrix would select, so the
// results are bitwise those of that call whatever the chunking.
//
// When the output buffer is pinned host memory the device can address (over
// NVLink-C2C on Grace systems), the kernels store each chunk's results
// straight into it and the device->host copies are skipped: the copy
// engines then carry only the inputs, which is what bounds the pipeline.
// When the inputs are too, there is no pipeline: one kernel reads and writes
// the host buffers directly.
#include "../../include/tile_rows.h"

#include <cmath>
#include <cstdint>
#include <mutex>

#include "launch.h"

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxSlots = 4;
// A chunk is about 1/16 of the rows (the tail after the last copy in is one
// chunk's kernel) but at least 1 MiB of each input (per-chunk overheads).
constexpr long long kStages = 16;
constexpr size_t kMinChunkBytes = size_t(1) << 20;

size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

int inputs_of(int op) { return op == TILE_OP_RESIDUAL_LAYERNORM ? 2 : 1; }
int tensors_of(int op) { return inputs_of(op) + 1; }

// Internal streams and events, created once per device.
struct DeviceQueues {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t h2d_ev[kMaxSlots] = {}, compute_ev[kMaxSlots] = {}, d2h_ev[kMaxSlots] = {};
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
    for (int b = 0; b < kMaxSlots && err == cudaSuccess; ++b) {
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

// Rows per chunk when a slot holds `tensors` row blocks: as many as fit in
// two slots, at most about rows/16 (but not below 1 MiB of one tensor) so the
// pipeline has stages to overlap, and at least 1 (0 if not even one row fits
// twice).
long long host_chunk_rows(int tensors, int rows, int width, size_t work_bytes) {
    const size_t row_bytes = static_cast<size_t>(width) * sizeof(float);
    const size_t per_buffer = work_bytes / (2 * static_cast<size_t>(tensors));
    long long fit = static_cast<long long>((per_buffer / kAlign * kAlign) / row_bytes);
    long long stage = (static_cast<long long>(rows) + kStages - 1) / kStages;
    const long long min_rows = static_cast<long long>((kMinChunkBytes + row_bytes - 1) / row_bytes);
    if (stage < min_rows) stage = min_rows;
    if (stage > rows) stage = rows;
    if (fit > stage) fit = stage;
    return fit;
}

// Chunk rows and ring slots for a workspace of `work_bytes`.  Slots hold
// the inputs, plus the output unless it is stored directly; `slots` is as
// many as fit (2 to kMaxSlots, never more than there are chunks, but at
// least 2, which host_chunk_rows guarantees fit).
void schedule(int op, int rows, int width, size_t work_bytes, bool direct, long long *chunk,
              int *slots) {
    const int per_slot = inputs_of(op) + (direct ? 0 : 1);
    const long long c = host_chunk_rows(per_slot, rows, width, work_bytes);
    *chunk = c;
    *slots = 0;
    if (c < 1) return;
    const size_t buf = round_up(static_cast<size_t>(c) * width * sizeof(float));
    const long long nchunks = (rows + c - 1) / c;
    long long fit = static_cast<long long>(work_bytes / (per_slot * buf));
    if (fit > nchunks) fit = nchunks;
    *slots = fit < 2 ? 2 : (fit > kMaxSlots ? kMaxSlots : static_cast<int>(fit));
}

// The device address of pinned, mapped host memory; nullptr for other
// memory (pageable host memory, or a pointer the runtime does not know).
void *device_address(const void *p) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) == cudaSuccess && attr.type == cudaMemoryTypeHost &&
        attr.devicePointer != nullptr)
        return attr.devicePointer;
    (void)cudaGetLastError();   // clear a non-sticky error of the query
    return nullptr;
}

// Argument checks of the host entry points that need no CUDA call and no
// workspace: op, shape, eps, NULL buffers and an output overlapping an
// input.  TILE_OK for rows == 0 too (the caller then returns at once).
int check_host_args(int op, const float *h_in, const float *h_res, const float *h_out,
                    int rows, int width, float eps) {
    if (op < TILE_OP_RESIDUAL_LAYERNORM || op > TILE_OP_SOFTMAX) return TILE_ERR_OP;
    if (rows < 0 || width < 1 || width > tile_max_width()) return TILE_ERR_SHAPE;
    if (op != TILE_OP_SOFTMAX && !(std::isfinite(eps) && eps >= 0.0f)) return TILE_ERR_EPS;
    if (rows == 0) return TILE_OK;
    const bool residual = op == TILE_OP_RESIDUAL_LAYERNORM;
    if (h_in == nullptr || h_out == nullptr || (residual && h_res == nullptr))
        return TILE_ERR_NULL;
    const size_t total = static_cast<size_t>(rows) * static_cast<size_t>(width) * sizeof(float);
    if (overlaps(h_out, h_in, total) || (residual && overlaps(h_out, h_res, total)))
        return TILE_ERR_ALIAS;
    return TILE_OK;
}

// The pipeline over caller-provided workspace (also used by the entry point
// that stages through the library's static device area).  If a CUDA call
// fails after work was enqueued, `stream` is still ordered after everything
// this call enqueued on the internal copy streams (as far as the runtime
// accepts the joins), so work the caller orders after `stream` never
// overlaps it.
int run_host(int op, const float *h_in, const float *h_res, float *h_out, int rows, int width,
             float eps, void *d_work, size_t work_bytes, cudaStream_t stream) {
    const int arg = check_host_args(op, h_in, h_res, h_out, rows, width, eps);
    if (arg != TILE_OK || rows == 0) return arg;
    const bool residual = op == TILE_OP_RESIDUAL_LAYERNORM;
    if (d_work == nullptr) return TILE_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(d_work) & (kAlign - 1)) != 0) return TILE_ERR_ALIGN;
    // Checked on the host before any CUDA call: one row of every tensor must
    // fit twice (whether or not the output later turns out to be stored
    // directly).
    if (host_chunk_rows(tensors_of(op), rows, width, work_bytes) < 1) return TILE_ERR_WORKSPACE;

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
    float *out_dev = static_cast<float *>(device_address(h_out));
    // Every buffer pinned and device-addressable: one launch of the selected
    // kernel on the host buffers themselves, which reads the inputs and
    // writes the output over the host link with no staging copies (measured
    // 10.63 ms at 65536 x 4096 residual LayerNorm against 11.03 ms for the
    // copy pipeline; the results are those of the device call, bit for bit).
    if (out_dev != nullptr) {
        const float *in_dev = static_cast<const float *>(device_address(h_in));
        const float *res_dev =
            residual ? static_cast<const float *>(device_address(h_res)) : nullptr;
        if (in_dev != nullptr && (!residual || res_dev != nullptr))
            return run_selected(op, in_dev, res_dev, out_dev, rows, width, eps, stream);
    }

    long long chunk = 0;
    int slots = 0;
    schedule(op, rows, width, work_bytes, out_dev != nullptr, &chunk, &slots);
    const int per_slot = inputs_of(op) + (out_dev != nullptr ? 0 : 1);
    const size_t buf = round_up(static_cast<size_t>(chunk) * width * sizeof(float));
    // The first and the last chunk are a quarter of a full one when that
    // still holds kMinChunkBytes of an input and there are more than two
    // chunks: the pipeline fills with one chunk's copy in and drains with
    // one chunk's kernel, so short ends shorten both.
    const long long ramp_min = static_cast<long long>(
        (kMinChunkBytes + static_cast<size_t>(width) * sizeof(float) - 1) /
        (static_cast<size_t>(width) * sizeof(float)));
    const long long ramp = (chunk / 4 >= ramp_min && rows > 2 * chunk) ? chunk / 4 : 0;
    const long long body = rows - 2 * ramp;
    const long long nchunks = ramp > 0 ? (body + chunk - 1) / chunk + 2 : (rows + chunk - 1) / chunk;
    // rows [*r0, *r0 + *n) of chunk c
    auto range = [&](long long c, long long *r0, int *n) {
        long long a, e;
        if (ramp == 0) {
            a = c * chunk;
            e = a + chunk;
        } else if (c == 0) {
            a = 0;
            e = ramp;
        } else if (c == nchunks - 1) {
            a = rows - ramp;
            e = rows;
        } else {
            a = ramp + (c - 1) * chunk;
            e = a + chunk;
            if (e > rows - ramp) e = rows - ramp;
        }
        if (e > rows) e = rows;
        *r0 = a;
        *n = static_cast<int>(e - a);
    };
    char *base = static_cast<char *>(d_work);
    float *dx[kMaxSlots], *dr[kMaxSlots], *dy[kMaxSlots];
    for (int b = 0; b < slots; ++b) {
        char *p = base + static_cast<size_t>(b) * per_slot * buf;
        dx[b] = reinterpret_cast<float *>(p);
        dr[b] = residual ? reinterpret_cast<float *>(p + buf) : nullptr;
        dy[b] = out_dev != nullptr ? nullptr
                                   : reinterpret_cast<float *>(p + (residual ? 2 : 1) * buf);
    }

    // Everything enqueued here runs after the work already on `stream`.  On
    // a failure `stream` first waits for both copy streams (best effort; the
    // error reported is the first one).
    auto join = [&]() {
        if (cudaEventRecord(q.done, q.d2h) == cudaSuccess)
            (void)cudaStreamWaitEvent(stream, q.done, 0);
        if (cudaEventRecord(q.done, q.h2d) == cudaSuccess)
            (void)cudaStreamWaitEvent(stream, q.done, 0);
    };
#define TILE_TRY(call)                                          \
    do {                                                        \
        err = (call);                                           \
        if (err != cudaSuccess) {                               \
            set_last_cuda_error(static_cast<int>(err));         \
            join();                                             \
            return TILE_ERR_CUDA;                               \
        }                                                       \
    } while (0)

    TILE_TRY(cudaEventRecord(q.start, stream));
    TILE_TRY(cudaStreamWaitEvent(q.h2d, q.start, 0));
    TILE_TRY(cudaStreamWaitEvent(q.d2h, q.start, 0));

    for (long long c = 0; c < nchunks; ++c) {
        const int b = static_cast<int>(c % slots);
        long long r0 = 0;
        int n = 0;
        range(c, &r0, &n);
        const size_t off = static_cast<size_t>(r0) * width;
        const size_t bytes = static_cast<size_t>(n) * width * sizeof(float);
        if (c >= slots) TILE_TRY(cudaStreamWaitEvent(q.h2d, q.compute_ev[b], 0));
        TILE_TRY(cudaMemcpyAsync(dx[b], h_in + off, bytes, cudaMemcpyHostToDevice, q.h2d));
        if (residual)
            TILE_TRY(cudaMemcpyAsync(dr[b], h_res + off, bytes, cudaMemcpyHostToDevice, q.h2d));
        TILE_TRY(cudaEventRecord(q.h2d_ev[b], q.h2d));

        TILE_TRY(cudaStreamWaitEvent(stream, q.h2d_ev[b], 0));
        if (out_dev != nullptr) {
            const int st =
                run_selected(op, dx[b], dr[b], out_dev + off, n, width, eps, stream, rows);
            if (st != TILE_OK) {
                join();
                return st;
            }
            TILE_TRY(cudaEventRecord(q.compute_ev[b], stream));
            continue;
        }
        if (c >= slots) TILE_TRY(cudaStreamWaitEvent(stream, q.d2h_ev[b], 0));
        const int st = run_selected(op, dx[b], dr[b], dy[b], n, width, eps, stream, rows);
        if (st != TILE_OK) {
            join();
            return st;
        }
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

int tile_host_schedule(int op, int rows, int width, size_t work_bytes, int direct_output,
                       int *chunk_rows, int *slots) {
    if (op < TILE_OP_RESIDUAL_LAYERNORM || op > TILE_OP_SOFTMAX) return TILE_ERR_OP;
    if (rows < 1 || width < 1 || width > tile_max_width()) return TILE_ERR_SHAPE;
    if (chunk_rows == nullptr || slots == nullptr) return TILE_ERR_NULL;
    if (tile::host_chunk_rows(tensors_of(op), rows, width, work_bytes) < 1)
        return TILE_ERR_WORKSPACE;
    long long c = 0;
    int k = 0;
    tile::schedule(op, rows, width, work_bytes, direct_output != 0, &c, &k);
    *chunk_rows = static_cast<int>(c);
    *slots = k;
    return TILE_OK;
}

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
