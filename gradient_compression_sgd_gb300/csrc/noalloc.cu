// noalloc.cu -- dgc_compress for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc: for example a plugin inside a host
// framework whose caching allocator owns the whole device-memory budget, or a
// real-time training loop that must not enter the driver's allocator (which
// can block or synchronise the device) in the middle of a step.  Such a
// caller still owns its inputs and outputs, but cannot hand the library a
// scratch workspace.  dgc_compress_noalloc runs the same DGC step as
// dgc_compress with its scratch in a fixed array that is part of the loaded
// library: GCSGD_NOALLOC_SCRATCH_BYTES on every GPU that loads the library,
// held until the process exits.
//
// The array's name is only a host-side stand-in for the device array, so the
// host looks up its device address once per device (with that device
// current) and passes that address to the kernels.  With CUDA's lazy module
// loading (the default) the array is not placed on a device when the library
// loads but when that lookup first runs there: the first call on each device
// is where the driver commits the GCSGD_NOALLOC_SCRATCH_BYTES, and it fails
// with GCSGD_ERR_CUDA ("cannot place ...") if the device has no room left.
// Callers make one warm-up call per device before their own allocator
// reserves the device's memory and before any stream capture.  The cached
// address belongs to the device's primary context: after cudaDeviceReset, or
// from another driver context on the same device, it is stale and the entry
// point must not be called.  Every call shares the
// one array; the DGC kernels rewrite everything they read from it (the plan
// and the candidate counters are set at the start of each call), so nothing
// has to be cleared between calls, but calls whose work overlaps on the GPU
// (different streams without ordering, or several host threads) race on it.
#include <mutex>

#include "common.cuh"
#include "dgc.cuh"

namespace gcsgd {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GCSGD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the static scratch on the current device (looked up on
// the first call for that device).
int noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return set_error(GCSGD_ERR_CUDA, "dgc_compress_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(GCSGD_ERR_CUDA, "dgc_compress_noalloc: device %d beyond the %d supported", dev, kMaxDevices);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e == cudaErrorMemoryAllocation) {
            (void)cudaGetLastError();  // not sticky: clear it for the caller
            return set_error(GCSGD_ERR_CUDA,
                             "dgc_compress_noalloc: cannot place the library's %zu-byte scratch array on device %d "
                             "(out of memory); make the first call on a device before reserving its memory",
                             (size_t)GCSGD_NOALLOC_SCRATCH_BYTES, dev);
        }
        if (e != cudaSuccess || !p)
            return set_error(GCSGD_ERR_CUDA, "dgc_compress_noalloc: cudaGetSymbolAddress failed: %s",
                             cudaGetErrorString(e));
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return GCSGD_OK;
}

}  // namespace
}  // namespace gcsgd

extern "C" int dgc_compress_noalloc(const int64_t* seg_offsets, int32_t n_seg, int32_t K, const float* grad,
                                    float* u, float* v, double density, float momentum, float clip_thr,
                                    int32_t clip_nodes, gcsgd_pair* out, int64_t cap, int64_t* counts,
                                    int64_t* totals, void* stream) {
    using namespace gcsgd;
    size_t need = 0;
    int rc = gcsgd_dgc_workspace_size(seg_offsets, n_seg, K, density, &need);
    if (rc != GCSGD_OK) return rc;
    if (need > (size_t)GCSGD_NOALLOC_SCRATCH_BYTES)
        return set_error(GCSGD_ERR_WORKSPACE,
                         "dgc_compress_noalloc: this layout and K need %zu bytes of scratch, more than the fixed "
                         "%zu bytes built into the library; use dgc_compress with a caller workspace",
                         need, (size_t)GCSGD_NOALLOC_SCRATCH_BYTES);
    void* ws = nullptr;
    if ((rc = noalloc_scratch(&ws)) != GCSGD_OK) return rc;
    return dgc_compress(seg_offsets, n_seg, K, grad, u, v, density, momentum, clip_thr, clip_nodes, out, cap, counts,
                        totals, ws, (size_t)GCSGD_NOALLOC_SCRATCH_BYTES, stream);
}
