// rs_bin_noalloc: binning for callers that cannot allocate device memory.
//
// Some callers of this library cannot hand it a workspace: a plug-in living inside a host
// application whose device memory is owned and budgeted by that application, or a per-frame
// loop that must not call cudaMalloc because the allocation synchronises the device and has no
// bound on its latency.  rs_bin needs scratch (offsets, sort ping-pong buffers, digit
// histograms); this entry point takes it from a fixed array that is part of the library's own
// device image instead of from the caller.
//
// The array lives at file scope below.  Every GPU on which the library's module holding it is
// loaded holds it until the process exits.  Host code cannot use the array's name as a device
// address, so the address is obtained once per device with cudaGetSymbolAddress, with that
// device current, on the first call made while it is current.  With the CUDA runtime's lazy
// module loading (its default) that lookup is also what loads the module, and with it the array,
// onto the device: the first call on a device may therefore allocate device memory and
// synchronise, and callers make it once outside their allocation-free region.  A lookup that
// fails (for example for lack of device memory) is not remembered: the next call tries again.
#include <mutex>

#include "rs_internal.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(RS_BIN_NOALLOC_SCRATCH_BYTES);
static_assert(kScratchBytes % 256 == 0, "scratch size");

static __device__ __align__(256) unsigned char g_bin_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_scratch[kMaxDevices];  // nullptr until a lookup on that device has succeeded

// Device address of g_bin_scratch on the current device, looked up on the first successful call
// per device and kept; a failed lookup is retried by the next call.
cudaError_t scratch_on_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> hold(g_lock);
    if (!g_scratch[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_bin_scratch);
        if (e != cudaSuccess || !p) {
            (void)cudaGetLastError();  // clear the sticky-free error so later calls can retry
            return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
        }
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int rs_bin_noalloc(const rs_camera* camera, const rs_projected* proj, int32_t n,
                              size_t capacity, uint64_t* d_keys_sorted, uint32_t* d_point_list,
                              uint32_t* d_tile_ranges, size_t* n_entries, void* stream) {
    size_t need = 0;
    const int rc = rs_bin_workspace_size(n, camera, capacity, &need);
    if (rc != RS_OK) return rc;
    if (need > kScratchBytes) return RS_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (scratch_on_current_device(&scratch) != cudaSuccess) return RS_ERR_CUDA;
    // rs_bin writes every byte of its workspace that it later reads, so the previous call's
    // leftovers in the shared array need no clearing.
    const int r = rs_bin(camera, proj, n, scratch, kScratchBytes, capacity, d_keys_sorted, d_point_list,
                         d_tile_ranges, n_entries, stream);
    // rs_bin waits for its stream on every other return; after a failed launch, kernels enqueued
    // before it may still be running on the shared array, so wait for them here: on return the
    // array is idle whatever the outcome
    if (r == RS_ERR_CUDA) (void)cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    return r;
}
