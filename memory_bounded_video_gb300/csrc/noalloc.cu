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
#include <atomic>
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB
static_assert(kStaticScratchBytes == DIT_STATIC_SCRATCH_BYTES, "header and library agree");

// Device scratch shared by every call in the process; every device that
// loads this module holds it until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
// Device address of g_static_scratch per device (null until set up).
std::atomic<void *> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mu;

// Address of the scratch on device `dev` (current), setting it up on first
// use: the symbol's host-side name is not a device address, so the runtime
// is asked for it, and the header (status word and hand-off flags) is
// cleared on `st`.
dit_status_t scratch_for(int dev, cudaStream_t st, uint8_t **out) {
    void *ptr = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!ptr) {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        ptr = g_scratch_addr[dev].load(std::memory_order_relaxed);
        if (!ptr) {
            int major = 0, minor = 0;
            cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
            if (e == cudaSuccess)
                e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
            if (e != cudaSuccess) return ds::cuda_fail(e);
            if (major != 10 || minor != 3) return DIT_ERR_UNSUPPORTED_ARCH;
            e = cudaGetSymbolAddress(&ptr, g_static_scratch);
            if (e == cudaSuccess) e = cudaMemsetAsync(ptr, 0, ds::kHeaderBytes, st);
            if (e != cudaSuccess) return ds::cuda_fail(e);
            g_scratch_addr[dev].store(ptr, std::memory_order_release);
        }
    }
    *out = static_cast<uint8_t *>(ptr);
    return DIT_OK;
}

}  // namespace

namespace ds {

int *static_status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    return static_cast<int *>(g_scratch_addr[dev].load(std::memory_order_acquire));
}

}  // namespace ds

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
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *scratch = nullptr;
    dit_status_t r = scratch_for(dev, st, &scratch);
    if (r != DIT_OK) return r;
    // The hand-off flags must start at zero (a launch that gave up may have
    // left some set); every other region is written before it is read within
    // one forward.  The status word is kept, so that a wait that ran out in
    // an earlier call stays visible to dit_block_sync_status.
    e = cudaMemsetAsync(scratch + ds::kFlagsOffset, 0, ds::kHeaderBytes - ds::kFlagsOffset, st);
    if (e != cudaSuccess) return ds::cuda_fail(e);
    return ds::block_forward(plan, scratch, false, x, w, modulation, nullptr, nullptr, stream);
}
