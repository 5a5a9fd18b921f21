// Block forward for callers that cannot allocate device memory.
//
// Some hosts of this library may not call cudaMalloc at all: code running
// under an allocator that owns every device byte (a framework's caching
// allocator that must see all allocations, a memory-capped sandbox), or code
// that is not allowed to allocate at the point where it runs the block.  For
// them dit_block_forward_static runs the same schedule and kernels as
// dit_block_forward, but its scratch (the plan's workspace: K/V of all tokens
// plus the chunk-sized slabs) is a file-scope device array of fixed size
// instead of caller-bound memory.
#include "internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB

// Device scratch shared by every call in the process; every device that
// loads this module holds it until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};  // device address, per device

}  // namespace

extern "C" dit_status_t dit_block_forward_static(const dit_plan_t *plan, float *x,
                                                 const dit_block_weights_t *w,
                                                 const float *modulation,
                                                 dit_stream_t stream) {
    if (!plan) return DIT_ERR_INVALID_ARG;
    if (plan->total > kStaticScratchBytes) return DIT_ERR_WORKSPACE_TOO_SMALL;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ds::cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return DIT_ERR_INVALID_ARG;
    if (!g_scratch_addr[dev]) {
        // Set-up, once per device, with that device current: the symbol's
        // host-side name is not a device address; ask the runtime for it.
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return ds::cuda_fail(e);
        if (major != 10 || minor != 3) return DIT_ERR_UNSUPPORTED_ARCH;
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess) return ds::cuda_fail(e);
        g_scratch_addr[dev] = ptr;
    }
    uint8_t *scratch = static_cast<uint8_t *>(g_scratch_addr[dev]);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Only the header (the status word and the attention's hand-off flags)
    // must start at zero: every other region is written before it is read
    // within one forward.
    e = cudaMemsetAsync(scratch, 0, ds::kHeaderBytes, st);
    if (e != cudaSuccess) return ds::cuda_fail(e);
    // Run the ordinary schedule with the plan pointed at the static scratch
    // for the duration of the (host-side, asynchronous) enqueue.
    dit_plan *p = const_cast<dit_plan *>(plan);
    uint8_t *saved_ws = p->ws;
    const size_t saved_bytes = p->ws_bytes;
    const bool saved_prof = p->prof;
    p->ws = scratch;
    p->ws_bytes = kStaticScratchBytes;
    p->prof = false;
    const dit_status_t r = dit_block_forward(p, x, w, modulation, stream);
    p->ws = saved_ws;
    p->ws_bytes = saved_bytes;
    p->prof = saved_prof;
    return r;
}
