// noalloc.cu -- fd_decode_paged_noalloc: the decode call with its workspace
// in a fixed buffer owned by the library, for callers that cannot allocate
// device memory where they call us (see include/fd_api.h).
//
// The buffer is a file-scope device array, one instance per GPU that loads
// the library.  Host code may not pass the array's name to a kernel: on the
// host that name is only a stand-in, not a device address.  The address is
// looked up once per device with cudaGetSymbolAddress (with that device
// current) and then handed to fd_decode_paged as its workspace.
#include <mutex>

#include "fd_internal.h"

namespace {

constexpr size_t kScratchBytes = FD_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char fd_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the current device's buffer (looked up on first use).
fd_status scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FD_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FD_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, fd_noalloc_scratch) != cudaSuccess || !p) return FD_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return FD_OK;
}

}  // namespace

extern "C" fd_status fd_decode_paged_noalloc(const fd_plan_t *plan, const void *q, const void *k_pages,
                                             const void *v_pages, const float *k_scale, const float *v_scale,
                                             const int32_t *block_table, const int32_t *seq_lens, void *out,
                                             float *lse, int32_t *status_dev, void *stream) {
    if (!plan) return FD_ERR_INVALID_ARG;
    if (plan->workspace_bytes > kScratchBytes) return FD_ERR_WORKSPACE_TOO_SMALL;
    if (plan->ws_counters > plan->workspace_bytes) return FD_ERR_INVALID_ARG;
    void *ws = nullptr;
    const fd_status st = scratch_for_current_device(&ws);
    if (st != FD_OK) return st;
    // The work and merge counters must start at zero; the buffer holds
    // whatever the previous call (possibly one that stopped on an error)
    // left in it.
    const size_t ctr_bytes = plan->workspace_bytes - plan->ws_counters;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (ctr_bytes && cudaMemsetAsync(static_cast<unsigned char *>(ws) + plan->ws_counters, 0, ctr_bytes, s) !=
                         cudaSuccess)
        return FD_ERR_CUDA;
    return fd_decode_paged(plan, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, out, lse, ws,
                           kScratchBytes, status_dev, stream);
}
