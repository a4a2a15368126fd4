// attn_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory.
//
// attn_bwd needs a caller-provided scratch buffer (the fp32 dQ accumulator and
// two per-row vectors).  Some callers have no way to provide one: code that is
// handed only its input and output tensors by a host framework which owns all
// device memory and forbids allocations after start-up, or a process whose
// device memory is fully budgeted when it loads.  For them this file keeps a
// fixed scratch area in a file-scope device array and runs the ordinary
// backward kernels on it.  Nothing here calls cudaMalloc, cudaFree or any
// allocating routine.
//
// The array costs kNoAllocScratchBytes of device memory on every GPU that
// loads this part of the library, until the process exits.  All calls share
// it: calls whose kernels overlap on the GPU (for example on two streams
// without ordering between them) race on it and give wrong results.  The dQ
// accumulator is zeroed by the backward preprocess kernel at the start of
// every call, so nothing left by an earlier call leaks into a later one.
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "attn_sm103a.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

struct ScratchState {
    bool ready = false;
    void* ptr = nullptr;  // device address of g_bwd_scratch on that device
};
ScratchState g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

// Once per device, with that device current: check the architecture and look
// up the device address of the scratch array.  In host code the array's name
// is only a host-side stand-in, never a usable device pointer.
attn_status scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchState& s = g_scratch[dev];
    if (!s.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        if (!(major == 10 && minor == 3)) return ATTN_ERR_UNSUPPORTED;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr)
            return ATTN_ERR_CUDA;
        s.ptr = p;
        s.ready = true;
    }
    *out = s.ptr;
    return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                        const void* dout, const float* lse, void* dq, void* dk,
                                        void* dv, int B, int H, int N, int d, float scale,
                                        int causal, attn_stream_t stream) {
    const size_t need = attn_bwd_workspace_bytes(B, H, N, d);
    if (need == 0) return ATTN_ERR_INVALID;
    if (need > kNoAllocScratchBytes) return ATTN_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const attn_status rc = scratch_for_current_device(&scratch);
    if (rc != ATTN_OK) return rc;
    return attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch, B, H, N, d, scale, causal, stream);
}
