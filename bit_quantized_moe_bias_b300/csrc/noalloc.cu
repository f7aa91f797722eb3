// noalloc.cu — a variant of ds4g_moe_forward for callers that cannot allocate
// device memory: code that runs where cudaMalloc is off limits (inside a
// custom allocator or memory-pool callback, a real-time loop that must never
// block on the driver's allocator, a plugin handed fixed buffers by its host
// engine).  Its scratch is a file-scope device array instead of a caller
// workspace.
#include <atomic>

#include "ds4g_internal.cuh"

namespace ds4g {

// Scratch of the per-slot decode kernels for one chunk of kDecodeMaxT tokens
// (the layout of decode_workspace(kDecodeMaxT), 4.92 MB).  Every device
// that loads the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = 5 * 1024 * 1024;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device.  In host
// code the array's name is only a host-side stand-in, so kernels must be given
// this address, never the symbol itself.  Host threads may race on the first
// lookup of a device: both find the same address, and the atomic store makes
// the cached value safe to read from any thread.  A cudaDeviceReset unloads
// the module, so the cached address is stale afterwards (documented in the
// header: the entry point is not supported after a reset).
constexpr int kMaxDevices = 64;
static std::atomic<void *> g_scratch_addr[kMaxDevices];

static ds4g_status scratch_address(void **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DS4G_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return DS4G_EUNSUPPORTED;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DS4G_ECUDA;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *ptr = p;
    return DS4G_OK;
}

}  // namespace ds4g

using namespace ds4g;

extern "C" ds4g_status ds4g_moe_forward_noalloc(const float *hidden, int T, const ds4g_layer *L,
                                                const int32_t *ids, const float *w, float *out,
                                                ds4g_stream_t s) {
    DS4G_TRACE();
    if (!hidden || !L || !ids || !w || !out || T < 1) return DS4G_EINVAL;
    if (T > DS4G_NOALLOC_MAX_T) return DS4G_ENOSPACE;
    if (!L->gate || !L->up || !L->down || !L->sh_gate || !L->sh_up || !L->sh_down) return DS4G_EINVAL;
    const bool types = (L->gate_up_type == DS4G_IQ2_XXS && L->down_type == DS4G_Q2_K) ||
                       (L->gate_up_type == DS4G_Q4_K && L->down_type == DS4G_Q4_K);
    if (!types) return DS4G_EUNSUPPORTED;
    if (L->gate_up_type == DS4G_IQ2_XXS && !L->iq2_grid) return DS4G_EINVAL;
    const uintptr_t al = (uintptr_t)hidden | (uintptr_t)ids | (uintptr_t)w | (uintptr_t)out |
                         (uintptr_t)L->gate | (uintptr_t)L->up | (uintptr_t)L->down |
                         (uintptr_t)L->sh_gate | (uintptr_t)L->sh_up | (uintptr_t)L->sh_down |
                         (uintptr_t)L->iq2_grid;
    if (al & 15) return DS4G_EALIGN;
    const int chunk = T < kDecodeMaxT ? T : kDecodeMaxT;
    const size_t need = decode_workspace(chunk);
    if (need > kNoAllocScratchBytes) return DS4G_ENOSPACE;
    void *ws = nullptr;
    const ds4g_status ar = scratch_address(&ws);
    if (ar != DS4G_OK) return ar;
    cudaStream_t st = (cudaStream_t)s;
    // The array keeps whatever the previous call left.  Only the status word
    // and the kernels' tile counters must start at zero; all of them lie
    // below kWsScratch (13 KB), and every other byte the kernels use is
    // written before it is read.  The kernels put their counters back to
    // zero, so the clear matters only after a call that a fault cut short;
    // it is 13 KB, not the 4.9 MB in use.  cudaMemsetAsync allocates nothing.
    if (cudaMemsetAsync(ws, 0, kWsScratch, st) != cudaSuccess) return DS4G_ECUDA;
    for (int t0 = 0; t0 < T; t0 += kDecodeMaxT) {
        const int n = T - t0 < kDecodeMaxT ? T - t0 : kDecodeMaxT;
        const ds4g_status rc = decode_forward(hidden + (size_t)t0 * kH, n, L, ids + (size_t)t0 * kK,
                                              w + (size_t)t0 * kK, out + (size_t)t0 * kH, ws, st, 3);
        if (rc != DS4G_OK) return rc;
    }
    return DS4G_OK;
}
