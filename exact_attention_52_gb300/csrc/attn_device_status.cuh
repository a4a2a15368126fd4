// Device-side error reporting shared by every kernel of the library.
//
// Kernels never trap.  A wait that runs out of time raises the CTA's abort
// flag, ORs a code into a device error word and records the id of the first
// wait that gave up; the host reads and clears both with
// attn_check_device_error().
#pragma once

#include <cstdint>

namespace attn {

enum : uint32_t {
    ATTN_DEVERR_WAIT_TIMEOUT = 1u,  // a bounded mbarrier wait gave up
    ATTN_DEVERR_SMEM_ALIGN = 2u,    // dynamic shared memory was not 1024-byte aligned
    ATTN_DEVERR_RANGE = 4u,         // debug builds: a TMA coordinate or tensor-memory address
                                    // failed its range check (the access was skipped)
};

struct DevStatus {
    unsigned int* word;             // word[0]: error bits (ATTN_DEVERR_*);
                                    // word[1]: id of the first failing wait (0 = none)
    unsigned long long wait_limit_ns;
};

__device__ __forceinline__ void record_device_error(unsigned int* word, uint32_t code,
                                                    uint32_t site) {
    atomicOr(word, code);
    atomicCAS(word + 1, 0u, site);
}

__device__ __forceinline__ void record_device_error(const DevStatus& st, uint32_t code,
                                                    uint32_t site) {
    record_device_error(st.word, code, site);
}

}  // namespace attn
