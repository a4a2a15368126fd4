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

#include "attn_internal.h"
#include "attn_sm103a.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

// Architecture check, cached per device (a device's compute capability never
// changes).
bool g_arch_checked[kMaxDevices];
bool g_arch_ok[kMaxDevices];
std::mutex g_arch_mutex;

// The scratch array's device address on the current device.  In host code the
// array's name is only a host-side stand-in, never a usable device pointer, so
// the address is looked up with that device current.  It is looked up on every
// call rather than cached: the address belongs to the module loaded into the
// device's current context, and a context created after cudaDeviceReset (or a
// different context made current on the same device) loads the module again,
// possibly elsewhere.  The lookup allocates nothing.  On the first call in a
// context it may load the library's module into that context, which is why the
// first call should come before any stream capture.
attn_status scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(g_arch_mutex);
        if (!g_arch_checked[dev]) {
            int major = 0, minor = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
                return ATTN_ERR_CUDA;
            g_arch_ok[dev] = (major == 10 && minor == 3);
            g_arch_checked[dev] = true;
        }
        if (!g_arch_ok[dev]) return ATTN_ERR_UNSUPPORTED;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    *out = p;
    return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                        const void* dout, const float* lse, void* dq, void* dk,
                                        void* dv, int B, int H, int N, int d, float scale,
                                        int causal, attn_stream_t stream) {
    // The problem is checked the way attn_bwd checks it (same status for a bad
    // size, head dim or flag) before the scratch limit is applied.
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    const attn_status chk = static_cast<attn_status>(attn::check_problem(B, H, N, d, scale, causal));
    if (chk != ATTN_OK) return chk;
    // With the split last round of the d = 128 kernel when its partials fit in the
    // scratch too (the results are then attn_bwd's bit for bit); otherwise without
    // it, and rows of the last round's key tiles of dK, dV may differ from
    // attn_bwd's in the last bit (another summation order).
    bool split = true;
    size_t need = attn::bwd_workspace_bytes_for(B, H, N, d, true);
    if (need > kNoAllocScratchBytes) {
        split = false;
        need = attn::bwd_workspace_bytes_for(B, H, N, d, false);
    }
    if (need == 0) return ATTN_ERR_INVALID;
    if (need > kNoAllocScratchBytes) return ATTN_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const attn_status rc = scratch_for_current_device(&scratch);
    if (rc != ATTN_OK) return rc;
    return static_cast<attn_status>(
        attn::bwd_dense(q, k, v, o, dout, lse, dq, dk, dv, scratch, B, H, N, d, scale, causal, split, stream));
}
