// Inline-PTX building blocks for the sm_103a attention kernels: shared-memory
// mbarriers, TMA tensor copies, tcgen05 tensor-core MMAs with TMEM
// accumulators, TMEM loads/stores, and the bounded waits every kernel uses.
//
// Everything here is written against the public PTX ISA (tcgen05, cp.async.bulk
// and mbarrier chapters).  No cluster multicast is used anywhere.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_device_status.cuh"

namespace attn {

// ---------------------------------------------------------------------------
// Debug builds (ATTN_DEBUG_CHECKS): range checks on every TMA coordinate and
// tensor-memory address, standing in for a memory checker.  A failed check
// ORs ATTN_DEVERR_RANGE into the device error word, records the check's site
// id and skips the access; nothing traps.  Release builds compile them away.
// ---------------------------------------------------------------------------
#ifdef ATTN_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
// The error word of the launching call, copied in by this file's launchers.
static __device__ unsigned int* g_dbg_word;
#else
constexpr bool kDebugChecks = false;
#endif

__device__ __forceinline__ bool dbg_ok(bool cond, uint32_t site) {
#ifdef ATTN_DEBUG_CHECKS
    if (!cond) {
        if (g_dbg_word != nullptr) record_device_error(g_dbg_word, ATTN_DEVERR_RANGE, site);
        return false;
    }
#endif
    (void)site;
    return true;
}

// A 32x32b tensor-memory access of `ncols` columns by this warp: the lanes are
// the warp's own quadrant and the columns lie inside the 512 every kernel of
// the library allocates (the allocation then starts at column 0).
__device__ __forceinline__ bool dbg_tmem(uint32_t taddr, uint32_t ncols, uint32_t site) {
    if constexpr (!kDebugChecks) return true;
    const uint32_t lane = taddr >> 16, col = taddr & 0xFFFFu;
    return dbg_ok(lane == ((threadIdx.x >> 5) & 3u) * 32u && col + ncols <= 512u, site);
}

// A TMA box load at element coordinates {x, row, head, batch} of a
// {d, N, heads, B} view: x on a 16-byte boundary and inside the row, the box's
// first row inside the sequence (later rows may fall past it: they read as
// zero), head and batch inside the tensor, destination 1024-byte aligned.
__device__ __forceinline__ bool dbg_tma(uint32_t dst, int x, int row, int head, int batch, int d, int N,
                                        int heads, int B, int elem_bytes, uint32_t site) {
    if constexpr (!kDebugChecks) return true;
    return dbg_ok((dst & 1023u) == 0 && x >= 0 && (x * elem_bytes) % 16 == 0 && x < d && row >= 0 &&
                      row < N && head >= 0 && head < heads && batch >= 0 && batch < B,
                  site);
}

// Debug builds: point the range checks of the calling file at the launching
// call's error word (a small copy on the launch stream, ahead of the kernel).
inline cudaError_t dbg_set_word(unsigned int* word, cudaStream_t stream) {
#ifdef ATTN_DEBUG_CHECKS
    return cudaMemcpyToSymbolAsync(g_dbg_word, &word, sizeof(word), 0, cudaMemcpyHostToDevice, stream);
#else
    (void)word;
    (void)stream;
    return cudaSuccess;
#endif
}

// ---------------------------------------------------------------------------
// Addresses
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait by one thread.  Returns false (after raising the CTA's abort
// flag and the device error word) when the phase does not complete within the
// library's wait limit, or when another role of the CTA has already aborted.
static __device__ __noinline__ bool wait_one_impl(uint32_t bar, uint32_t parity,
                                                   volatile int* abort_flag, unsigned int* err,
                                                   unsigned long long limit, uint32_t site) {
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit) {
            *abort_flag = 1;
            record_device_error(err, ATTN_DEVERR_WAIT_TIMEOUT, site);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         const DevStatus& st, uint32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_one_impl(bar, parity, abort_flag, st.word, st.wait_limit_ns, site);
}

// Bounded wait that ignores the abort flag: used on the way out to let this
// thread's own asynchronous copies and MMAs land before the CTA exits.
static __device__ __noinline__ bool wait_drain_impl(uint32_t bar, uint32_t parity, unsigned int* err,
                                                     unsigned long long limit, uint32_t site) {
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit) {
            record_device_error(err, ATTN_DEVERR_WAIT_TIMEOUT, site);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, const DevStatus& st,
                                           uint32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_drain_impl(bar, parity, st.word, st.wait_limit_ns, site);
}

// Bounded wait taken by a whole warp together: every lane polls, the warp
// leaves only when all lanes saw the phase complete, and a time-out is decided
// by lane 0 for the whole warp, so the warp never splits before a collective
// tcgen05.ld/st.
static __device__ __noinline__ bool wait_warp_impl(uint32_t bar, uint32_t parity,
                                                    volatile int* abort_flag, unsigned int* err,
                                                    unsigned long long limit, uint32_t site) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        const bool ok = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        int stop = 0;
        if (lane_id() == 0) {
            if (it == 0) {
                t0 = global_timer_ns();
            } else if (*abort_flag) {
                stop = 1;
            } else if (global_timer_ns() - t0 > limit) {
                *abort_flag = 1;
                record_device_error(err, ATTN_DEVERR_WAIT_TIMEOUT, site);
                stop = 1;
            }
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
}

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          const DevStatus& st, uint32_t site) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    return wait_warp_impl(bar, parity, abort_flag, st.word, st.wait_limit_ns, site);
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copies, global -> shared), no multicast
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch.  pdl_wait: block until the grids this one was
// launched after have completed and their writes are visible (returns at once
// for a grid launched without the attribute).  pdl_launch_dependents: this block
// no longer holds back the launch of the grid launched after it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Plain bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// Element-wise add of a shared-memory box into global memory through a tensor
// map (fp32 add for an fp32 map); completion is tracked by bulk groups.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                                  int c2) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every committed bulk group of this thread has finished reading
// its shared-memory source.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Waits until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_group0() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Generic-proxy shared-memory writes -> visible to the async proxy (tensor core).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Tensor memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive 32-bit columns of this warp's 32 lanes (one lane per thread).
// The values are valid only after tmem_ld_wait() on the same array.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    if (!dbg_tmem(taddr, 32, 0xD01)) return;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}

// Waits for this thread's outstanding tcgen05.ld; the array is threaded
// through the asm so that no use of it can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    if (!dbg_tmem(taddr, 32, 0xD02)) return;
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

// 16 consecutive 32-bit columns (one lane per thread).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    if (!dbg_tmem(taddr, 16, 0xD03)) return;
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05.mma
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile whose
// 1024-byte swizzle atoms are 8 rows x 128 bytes:
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-47  descriptor version (1)
//   bits 49-51  base offset (0: every tile is 1024-byte aligned)
//   bits 61-63  swizzle mode (2 = 128-byte swizzle)
// K-major operand: rows are M/N, 128-byte row segments hold K; SBO = 1024 is
// the step between 8-row groups and LBO is unused.  MN-major operand: rows are
// K, 128-byte row segments hold 64 (16-bit) or 128 (8-bit) M/N elements; LBO is
// the step between such 128-byte M/N blocks and SBO = 1024 the step between
// 8-row K groups.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor (kind::f16 and kind::f8f6f4): D format in bits 4-5
// (1 = f32), A format 7-9 and B format 10-12 (kind::f16: 1 = bf16;
// kind::f8f6f4: 0 = e4m3), A/B major-ness bits 15/16 (1 = MN-major),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t ab_format, int M, int N, bool a_mn,
                                                  bool b_mn) {
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t kFmtBF16 = 1;
constexpr uint32_t kFmtE4M3 = 0;

// A shared-memory descriptor kept as its two 32-bit words.  The start address
// sits in the low word (bits 0-13, address >> 4), so a byte offset b is added
// as lo + (b >> 4): shared memory is below 256 KB, so the field never carries.
struct SmemDesc {
    uint32_t lo, hi;
};

__device__ __forceinline__ SmemDesc sw128_desc_words(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    const uint64_t d = sw128_desc(saddr, lbo, sbo);
    return SmemDesc{static_cast<uint32_t>(d), static_cast<uint32_t>(d >> 32)};
}

__device__ __forceinline__ SmemDesc desc_add(SmemDesc d, uint32_t byte_offset) {
    return SmemDesc{d.lo + (byte_offset >> 4), d.hi};
}

// Descriptor of a K-major operand without swizzle (swizzle mode 0): the
// operand is made of core matrices of 8 rows x 16 bytes (8 bf16 of K), each
// stored contiguously (row i at +16 i); LBO is the byte step between core
// matrices adjacent in K and SBO the step between adjacent 8-row groups of M/N.
// Any step, zero included, is a valid descriptor: a zero SBO makes every
// 8-row group read the same eight rows.
__device__ __forceinline__ SmemDesc noswz_desc_words(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return SmemDesc{static_cast<uint32_t>(d), static_cast<uint32_t>(d >> 32)};
}

// Warp-wide forms: every lane of a converged warp executes the call with the
// same (warp-uniform) operands and one lane, chosen by elect.sync, issues the
// instructions.  Keeping the issuing loop on the whole warp lets the compiler
// hold loop counters and descriptors in uniform registers; a loop run by one
// lane of a warp that shares its scheduler with busy softmax warps issues
// several times more slowly.
//
// Four products from one asm block: one elect.sync for the four, the first
// accumulating as `accumulate` says and the other three always accumulating.
// The offsets are compile-time constants: OA/OB are added to the low words of
// the shared-memory descriptors (16-byte units); for the TS form OA is added to
// the tensor-memory address of A (columns).
template <bool FP8, uint32_t OA0, uint32_t OA1, uint32_t OA2, uint32_t OA3, uint32_t OB0, uint32_t OB1,
          uint32_t OB2, uint32_t OB3>
__device__ __forceinline__ void mma_ss_warp4(uint32_t d_tmem, SmemDesc a, SmemDesc b, uint32_t idesc,
                                             uint32_t accumulate) {
    // D: lane 0 (M = 128 rows from lane 0), N fp32 columns inside the allocation
    if (!dbg_ok((d_tmem >> 16) == 0 && (d_tmem & 0xFFFFu) + ((idesc >> 17) & 0x3Fu) * 8u <= 512u, 0xD04))
        return;
    if constexpr (FP8) {
        asm volatile(
            "{\n\t.reg .pred p, t, e;\n\t.reg .b32 al, bl;\n\t.reg .b64 da, db;\n\t"
            "setp.ne.b32 p, %6, 0;\n\tsetp.eq.b32 t, %5, %5;\n\telect.sync _|e, 0xffffffff;\n\t"
            "add.u32 al, %1, %7;\n\tadd.u32 bl, %3, %11;\n\tmov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, p;\n\t"
            "add.u32 al, %1, %8;\n\tadd.u32 bl, %3, %12;\n\tmov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, t;\n\t"
            "add.u32 al, %1, %9;\n\tadd.u32 bl, %3, %13;\n\tmov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, t;\n\t"
            "add.u32 al, %1, %10;\n\tadd.u32 bl, %3, %14;\n\tmov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, t;\n\t"
            "}"
            ::"r"(d_tmem), "r"(a.lo), "r"(a.hi), "r"(b.lo), "r"(b.hi), "r"(idesc), "r"(accumulate),
            "n"(OA0), "n"(OA1), "n"(OA2), "n"(OA3), "n"(OB0), "n"(OB1), "n"(OB2), "n"(OB3)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p, t, e;\n\t.reg .b32 al, bl;\n\t.reg .b64 da, db;\n\t"
            "setp.ne.b32 p, %6, 0;\n\tsetp.eq.b32 t, %5, %5;\n\telect.sync _|e, 0xffffffff;\n\t"
            "add.u32 al, %1, %7;\n\tadd.u32 bl, %3, %11;\n\tmov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t"
            "add.u32 al, %1, %8;\n\tadd.u32 bl, %3, %12;\n\tmov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t"
            "add.u32 al, %1, %9;\n\tadd.u32 bl, %3, %13;\n\tmov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t"
            "add.u32 al, %1, %10;\n\tadd.u32 bl, %3, %14;\n\tmov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t"
            "}"
            ::"r"(d_tmem), "r"(a.lo), "r"(a.hi), "r"(b.lo), "r"(b.hi), "r"(idesc), "r"(accumulate),
            "n"(OA0), "n"(OA1), "n"(OA2), "n"(OA3), "n"(OB0), "n"(OB1), "n"(OB2), "n"(OB3)
            : "memory");
    }
}

template <bool FP8, uint32_t OA0, uint32_t OA1, uint32_t OA2, uint32_t OA3, uint32_t OB0, uint32_t OB1,
          uint32_t OB2, uint32_t OB3>
__device__ __forceinline__ void mma_ts_warp4(uint32_t d_tmem, uint32_t a_tmem, SmemDesc b, uint32_t idesc,
                                             uint32_t accumulate) {
    // D as above; A: 8 columns (16 bf16 or 32 e4m3 values of K per row) at each of
    // the four offsets, lanes from 0
    if (!dbg_ok((d_tmem >> 16) == 0 && (d_tmem & 0xFFFFu) + ((idesc >> 17) & 0x3Fu) * 8u <= 512u &&
                    (a_tmem >> 16) == 0 && (a_tmem & 0xFFFFu) + OA3 + 8u <= 512u,
                0xD05))
        return;
    if constexpr (FP8) {
        asm volatile(
            "{\n\t.reg .pred p, t, e;\n\t.reg .b32 ta, bl;\n\t.reg .b64 db;\n\t"
            "setp.ne.b32 p, %5, 0;\n\tsetp.eq.b32 t, %4, %4;\n\telect.sync _|e, 0xffffffff;\n\t"
            "add.u32 ta, %1, %6;\n\tadd.u32 bl, %2, %10;\n\tmov.b64 db, {bl, %3};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ta], db, %4, p;\n\t"
            "add.u32 ta, %1, %7;\n\tadd.u32 bl, %2, %11;\n\tmov.b64 db, {bl, %3};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ta], db, %4, t;\n\t"
            "add.u32 ta, %1, %8;\n\tadd.u32 bl, %2, %12;\n\tmov.b64 db, {bl, %3};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ta], db, %4, t;\n\t"
            "add.u32 ta, %1, %9;\n\tadd.u32 bl, %2, %13;\n\tmov.b64 db, {bl, %3};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ta], db, %4, t;\n\t"
            "}"
            ::"r"(d_tmem), "r"(a_tmem), "r"(b.lo), "r"(b.hi), "r"(idesc), "r"(accumulate),
            "n"(OA0), "n"(OA1), "n"(OA2), "n"(OA3), "n"(OB0), "n"(OB1), "n"(OB2), "n"(OB3)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p, t, e;\n\t.reg .b32 ta, bl;\n\t.reg .b64 db;\n\t"
            "setp.ne.b32 p, %5, 0;\n\tsetp.eq.b32 t, %4, %4;\n\telect.sync _|e, 0xffffffff;\n\t"
            "add.u32 ta, %1, %6;\n\tadd.u32 bl, %2, %10;\n\tmov.b64 db, {bl, %3};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p;\n\t"
            "add.u32 ta, %1, %7;\n\tadd.u32 bl, %2, %11;\n\tmov.b64 db, {bl, %3};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, t;\n\t"
            "add.u32 ta, %1, %8;\n\tadd.u32 bl, %2, %12;\n\tmov.b64 db, {bl, %3};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, t;\n\t"
            "add.u32 ta, %1, %9;\n\tadd.u32 bl, %2, %13;\n\tmov.b64 db, {bl, %3};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, t;\n\t"
            "}"
            ::"r"(d_tmem), "r"(a_tmem), "r"(b.lo), "r"(b.hi), "r"(idesc), "r"(accumulate),
            "n"(OA0), "n"(OA1), "n"(OA2), "n"(OA3), "n"(OB0), "n"(OB1), "n"(OB2), "n"(OB3)
            : "memory");
    }
}

// One bf16 product (kind::f16, both operands in shared memory) from the
// elected lane of a converged warp; it accumulates into D.
__device__ __forceinline__ void mma_ss_warp1_acc(uint32_t d_tmem, SmemDesc a, SmemDesc b, uint32_t idesc) {
    if (!dbg_ok((d_tmem >> 16) == 0 && (d_tmem & 0xFFFFu) + ((idesc >> 17) & 0x3Fu) * 8u <= 512u, 0xD06))
        return;
    asm volatile(
        "{\n\t.reg .pred e, t;\n\t.reg .b64 da, db;\n\t"
        "setp.eq.b32 t, %5, %5;\n\telect.sync _|e, 0xffffffff;\n\t"
        "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t}"
        ::"r"(d_tmem), "r"(a.lo), "r"(a.hi), "r"(b.lo), "r"(b.hi), "r"(idesc)
        : "memory");
}

// Arrive (once) on `bar` when every tcgen05.mma issued so far by the issuing
// lane has completed.  elect.sync over a full, converged warp picks the same
// lane every time, so that lane has issued every product of the warp.
__device__ __forceinline__ void mma_commit_warp(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// ---------------------------------------------------------------------------
// Arithmetic helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two floats -> packed bf16x2 (round to nearest even); `lo` in bits 15..0.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four floats -> four e4m3 bytes (saturating, round to nearest even); `a` in bits 7..0.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// max(a, b, c) in one instruction (three-input max, sm_100+).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (d0, d1) = (a0 * b0 + c0, a1 * b1 + c1) as one packed fp32x2 FMA.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                      float c0, float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// (d0, d1) = (a0 * b0, a1 * b1) packed.
__device__ __forceinline__ void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// (d0, d1) = (a0 + b0, a1 + b1) packed.
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// (d0, d1) = (a0 - b0, a1 - b1) packed.
__device__ __forceinline__ void fsub2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// 2^x for two floats on the FMA pipe instead of MUFU (the softmax of the
// forward pass is bound by MUFU: one ex2 per element at a quarter of the issue
// rate, so moving a few of them to the otherwise idle FMA pipe shortens it).
// x = n + r with n = round(x): adding 1.5 * 2^23 leaves n in the low mantissa
// bits of t (the float spacing there is 1), so t - 1.5 * 2^23 = n exactly and
// r = x - n lies in [-1/2, 1/2].  2^r comes from a cubic fitted here to the
// relative error of 2^r on that interval (Lawson's iteratively reweighted least
// squares; max relative error 7.5e-5, also in fp32 evaluation), and n is added
// to the exponent field: the low bits of t shifted up by 23 are n << 23 modulo
// 2^32.  x is clamped below at -125 so that the exponent field stays positive;
// results under 2^-125 (zero in every use here) come out as about 2^-125.
__device__ __forceinline__ void ex2_fma2(float& y0, float& y1, float x0, float x1) {
    constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
    constexpr float c0 = 0.99992812f, c1 = 0.69326097f, c2 = 0.24261054f, c3 = 0.055171322f;
    x0 = fmaxf(x0, -125.f);
    x1 = fmaxf(x1, -125.f);
    float t0, t1, n0, n1, r0, r1, p0, p1;
    fadd2(t0, t1, x0, x1, kRound, kRound);
    fsub2(n0, n1, t0, t1, kRound, kRound);
    fsub2(r0, r1, x0, x1, n0, n1);
    ffma2(p0, p1, r0, r1, c3, c3, c2, c2);
    ffma2(p0, p1, p0, p1, r0, r1, c1, c1);
    ffma2(p0, p1, p0, p1, r0, r1, c0, c0);
    y0 = __int_as_float(__float_as_int(p0) + (__float_as_int(t0) << 23));
    y1 = __int_as_float(__float_as_int(p1) + (__float_as_int(t1) << 23));
}

// acc + lo(w) + hi(w) where w holds two bf16 values: mixed-precision adds
// (f32 accumulator, bf16 operand), no unpacking.
__device__ __forceinline__ float add_bf16x2(float acc, uint32_t w) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %0, hi, %0;\n\t}"
        : "+f"(acc)
        : "r"(w));
    return acc;
}

__device__ __forceinline__ void red_add_f32(float* gaddr, float a) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(gaddr), "f"(a) : "memory");
}

__device__ __forceinline__ void st_global_v4(void* gaddr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(gaddr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// 32-byte store (sm_100+); gaddr must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* gaddr, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(gaddr), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// 64 bytes of one row (16 words): two 32-byte stores (rows 32-byte aligned) or
// four 16-byte ones.  A row per lane leaves a warp instruction with 32 separate
// pieces; whole 32-byte sectors halve the pieces, which at a backward item's end
// hold up the next item's loads and first products.
template <bool V8>
__device__ __forceinline__ void st_global_row64(uint8_t* gaddr, const uint32_t* w) {
    if constexpr (V8) {
        st_global_v8(gaddr, w);
        st_global_v8(gaddr + 32, w + 8);
    } else {
#pragma unroll
        for (int v = 0; v < 4; ++v) st_global_v4(gaddr + 16 * v, w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
    }
}

}  // namespace attn
