// scan_noalloc.cu — ssm_scan_fwd_noalloc: the forward scan with its scratch
// held in a fixed array inside this library instead of a caller workspace.
//
// Who needs it: a caller that cannot allocate device memory at all — for
// example a plugin whose host framework owns every device allocation and hands
// the plugin no allocator, or a loop that is not allowed to call cudaMalloc
// because that can synchronise the device.  ssm_scan_fwd already allocates
// nothing itself, but it asks the caller for a workspace when the sequence is
// split into chunks; this entry point needs none.
//
// The scratch is one file-scope device array of SSM_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  Host
// code may not use the array's name as a device address (on the host it names
// a stand-in object), so the device address is looked up once per device with
// cudaGetSymbolAddress and cached.
#include <mutex>

#include "../../include/ssm_scan.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SSM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on
// the first call for that device.  Returns nullptr if the lookup fails.
void *scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> hold(g_lock);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" ssm_status ssm_scan_fwd_noalloc(const ssm_scan_params *p, ssm_stream_t stream) {
    if (!p) return SSM_ERR_INVALID_ARG;
    ssm_scan_params q = *p;
    q.workspace = nullptr;
    q.workspace_bytes = 0;
    const size_t need = ssm_scan_workspace_size(&q);
    if (need == 0) return SSM_ERR_INVALID_ARG;
    if (need > SSM_NOALLOC_SCRATCH_BYTES) return SSM_ERR_UNSUPPORTED;
    void *scratch = scratch_on_current_device();
    if (!scratch) return SSM_ERR_CUDA;
    q.workspace = scratch;
    q.workspace_bytes = SSM_NOALLOC_SCRATCH_BYTES;
    // ssm_scan_fwd clears the status word and the chunk flags at the head of
    // the scratch before its launches; the chunk pairs and carried states that
    // follow are written before a flag says they are out, so stale contents do
    // no harm.
    return ssm_scan_fwd(&q, stream);
}
