// mk_noalloc.cu -- the allocation-free entry point.
//
// Some callers cannot allocate device memory when they run this operation:
// code embedded in a host framework that owns the whole device-memory budget
// through its own allocator and hands out no extra scratch, or a
// latency-critical loop (decode-sized batches) where cudaMalloc /
// cudaMallocAsync and their possible device-wide synchronisation are not
// allowed.  For them the library keeps one fixed scratch array in device
// memory (below) and runs the normal path with it as the workspace.
//
// The array is static device memory of MK_NOALLOC_SCRATCH_BYTES bytes.  Each
// GPU on which it is set up keeps it until the process exits (with eager
// module loading, every GPU that loads the library does).  It is shared by
// every call on that GPU and keeps the last call's contents.
//
// The array's device address is looked up once per device, with that device
// current, and kept.  A device reset gives the device a new context in which
// the array may sit elsewhere, so mk_release_workspace() -- which a caller
// runs after a reset, as it must for the workspace cache too -- forgets the
// kept addresses and the next call looks them up again.

#include <cuda_runtime.h>

#include <mutex>

#include "mk.h"

namespace {

// The fixed scratch.  In host code this name is only a host-side stand-in
// for the device array: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MK_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).
mk_status_t scratch_on_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MK_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MK_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MK_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MK_OK;
}

}  // namespace

namespace mk {
// Called by mk_release_workspace(): drop every kept device address.
void noalloc_forget_scratch() {
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < kMaxDevices; ++i) g_scratch_ptr[i] = nullptr;
}
}  // namespace mk

extern "C" mk_status_t mk_moe_dispatch_gemm_noalloc(const void* x, const float* logits, int T, int H, int E, int k,
                                                    const void* W, int F, void* y_sorted, int32_t* src_index,
                                                    int32_t* expert_offsets, float* gate_w, void* stream,
                                                    const mk_config_t* cfg) {
    // Phase stamps would land in the array, where mk_read_trace cannot find
    // them: tracing is refused rather than silently lost.
    if (cfg && cfg->trace != 0) return MK_ERR_UNSUPPORTED;
    // Sizes the fixed array cannot hold are refused before anything runs.
    const size_t need = mk_workspace_size(T, H, F, E, k, cfg);
    if (need > size_t(MK_NOALLOC_SCRATCH_BYTES)) return MK_ERR_WORKSPACE;
    void* scratch = nullptr;
    mk_status_t s = scratch_on_current_device(&scratch);
    if (s != MK_OK) return s;
    // The workspace's control block must start at zero; the array keeps
    // whatever the previous call left, so clear it on the caller's stream.
    if (need > 0 && cudaMemsetAsync(scratch, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MK_ERR_CUDA;
    // need == 0 means invalid sizes: the call below reports the exact error
    // before touching the workspace.
    return mk_moe_dispatch_gemm_ex(x, logits, T, H, E, k, W, F, y_sorted, src_index, expert_offsets, gate_w, stream,
                                   cfg, scratch, size_t(MK_NOALLOC_SCRATCH_BYTES));
}
