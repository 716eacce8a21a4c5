// Host-buffer entry point that allocates nothing.
//
// tile_run_host_f32 stages rows through a device workspace the caller
// allocates.  Some callers cannot allocate device memory when they need to
// run: code that runs after an application has fixed its device memory
// budget at start-up, plugin code inside a framework that owns the device
// allocator, or code that must not call cudaMalloc (which synchronises the
// device) on a latency-critical path.  This entry point gives them the same
// pipeline over a staging area that lives inside the library: a file-scope
// static device array of TILE_STATIC_STAGING_BYTES, which every GPU that
// loads the library holds until the process exits.
//
// In host code `g_static_staging` is only a host-side stand-in for the
// array, not a device address, so it is never passed to a kernel or a copy.
// Its device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call that
// runs on the device.
#include "../../include/tile_rows.h"

#include <cmath>
#include <mutex>

#include "launch.h"

namespace {

__device__ __align__(256) unsigned char g_static_staging[TILE_STATIC_STAGING_BYTES];

struct StaticStaging {
    bool ready = false;
    void *device_ptr = nullptr;    // device address of g_static_staging
    cudaEvent_t done = nullptr;    // the previous call's end on this device
    std::mutex mu;
};

StaticStaging g_staging[tile::kMaxDevices];

}  // namespace

extern "C" int tile_run_host_static_f32(int op, const float *h_in, const float *h_residual,
                                        float *h_out, int rows, int width, float eps,
                                        cudaStream_t stream) {
    // Argument errors (op, shape, eps, NULL buffers, an output overlapping
    // an input, a row too large for the area) are reported before any CUDA
    // call.
    const int arg = tile::check_host_args(op, h_in, h_residual, h_out, rows, width, eps);
    if (arg != TILE_OK || rows == 0) return arg;
    // One row of every tensor must fit the area twice (double buffering).
    if (tile_host_workspace_bytes(op, width, 1) > TILE_STATIC_STAGING_BYTES)
        return TILE_ERR_WORKSPACE;

    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess && (dev < 0 || dev >= tile::kMaxDevices)) err = cudaErrorInvalidDevice;
    if (err != cudaSuccess) {
        tile::set_last_cuda_error(static_cast<int>(err));
        return TILE_ERR_CUDA;
    }
    StaticStaging &s = g_staging[dev];
    std::lock_guard<std::mutex> lock(s.mu);
    if (!s.ready) {
        err = cudaGetSymbolAddress(&s.device_ptr, g_static_staging);
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming);
        if (err != cudaSuccess) {
            tile::set_last_cuda_error(static_cast<int>(err));
            return TILE_ERR_CUDA;
        }
        s.ready = true;
    }
    // Every call on this device uses the same area, so a call must not start
    // on the GPU before the previous one has finished with it: order this
    // call's work after the previous call's end.
    err = cudaStreamWaitEvent(stream, s.done, 0);
    if (err != cudaSuccess) {
        tile::set_last_cuda_error(static_cast<int>(err));
        return TILE_ERR_CUDA;
    }
    const int st = tile::run_host(op, h_in, h_residual, h_out, rows, width, eps, s.device_ptr,
                                  TILE_STATIC_STAGING_BYTES, stream);
    // run_host leaves `stream` ordered after everything it enqueued, on
    // success and on failure alike, so the next call waits for this one
    // either way.
    err = cudaEventRecord(s.done, stream);
    if (st != TILE_OK) return st;
    if (err != cudaSuccess) {
        tile::set_last_cuda_error(static_cast<int>(err));
        return TILE_ERR_CUDA;
    }
    return TILE_OK;
}
