// Backward exact attention on sm_103a.  Three launches on one stream:
//
//  1. bwd_pre     D_i = sum_k dO_ik O_ik (equal to sum_j P_ij dP_ij), -LSE in
//                 log2 units, zeroed fp32 dQ accumulator.
//  2. bwd_main    one work item per (key/value head, 128-key tile j); loops over
//                 query tiles i, regenerating P from Q, K and the saved log-sum-exp
//                 (FlashAttention item 58: backward recomputes score tiles from
//                 inputs and normalisation statistics):
//                     S^T  = K Q_i^T            P^T = 2^(S^T*cs - LSE*log2(e))
//                     dP^T = V dO_i^T           dS^T = P^T (dP^T - D)
//                     dV  += P^T dO_i           dK  += dS^T Q_i
//                     dQ_i += dS K   (fp32 reductions into the accumulator)
//                 The dQ reductions are done by a dedicated writer warpgroup,
//                 the role the FlashAttention-3 digest (section 1) gives its
//                 dQ-writer warp.
//  3. dq_convert  dQ = bf16(scale * accumulator)  (the second, combining
//                 kernel of a split reduction, CUTLASS split-K item).
//
// bwd_main has two forms:
//   d = 128  bwd_main_full_kernel: persistent CTAs, whole 128x128 query tiles,
//            every product 128 wide, the steps pipelined so that the
//            exponential and dS passes overlap dP^T and dV (section 2b below).
//            Its instantiation <1, *> also splits a short last round of key
//            tiles into parts that meet in the workspace (no mask); <2, *> takes
//            per-CTA lists built on the host, with the longest causal items in
//            two parts (grouped heads whose longest items pass the per-CTA mean)
//            or causal items in groups of heads; <*, true> writes dK and dV rows
//            with 32-byte stores.
//   d = 64   bwd_main_kernel<64>: one CTA per key tile, each query tile as two
//            64-row halves with their own compute warpgroup and tensor-memory
//            region, dQ staged in shared memory and TMA-reduced (section 2).
// Both use 448 threads: warps 0-7 compute (one thread per key row), warps 8-11
// the dQ writer, warp 12 the TMA producer, warp 13 the MMA issuer.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <queue>
#include <type_traits>
#include <utility>
#include <vector>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.44269504088896340736f;

template <int D>
struct BwdTraits {
    static constexpr int NBLK = D / 64;                 // 128-byte column blocks of a K/V/Q/dO row
    static constexpr int NDQ = D / 64;                  // dQ tile computed as NDQ parts of 64 columns
    static constexpr int BLK_BYTES = kTile * 128;       // one [128 rows x 128 B] block
    static constexpr int HALF_BYTES = 64 * 128;         // 64 rows of a block (one query half)
    static constexpr int TILE_BYTES = kTile * D * 2;
    static constexpr int DS_BYTES = kTile * kTile * 2;  // dS^T [128 keys][128 queries], 2 blocks
    static constexpr int STAGES = 2;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + TILE_BYTES;
    static constexpr int OFF_Q = OFF_V + TILE_BYTES;                 // + stage * TILE_BYTES
    static constexpr int OFF_DO = OFF_Q + STAGES * TILE_BYTES;       // + stage * TILE_BYTES
    static constexpr int OFF_DS = OFF_DO + STAGES * TILE_BYTES;
    static constexpr int OFF_VEC = OFF_DS + DS_BYTES;                // -LSE2[s], D[s]: 512 B each
    static constexpr int OFF_BAR = OFF_VEC + STAGES * 2 * 512;
    // barriers: kv_full, qdo_full[2], qdo_empty[2], s_full[2], p_full[2], dq_full[2],
    //           dq_empty[2], dkv_full, done, dq_staged[2]
    static constexpr int NBARS = 1 + 2 * STAGES + 2 + 2 + 2 + 2 + 2 + 2;
    static constexpr int SMEM_BYTES = OFF_BAR + NBARS * 8 + 16;
    // Region h (h = query half) = 128 columns: S^T_h at +0, dP^T_h at +64.
    static constexpr uint32_t COL_REGION = 128, COL_DP = 64;
    static constexpr uint32_t COL_DV = 256, COL_DK = 256 + D;
    static constexpr uint32_t IDESC_SDP = make_idesc(kFmtBF16, kTile, 64, false, false);
    static constexpr uint32_t IDESC_DVK = make_idesc(kFmtBF16, kTile, D, false, true);
    static constexpr uint32_t IDESC_DQ = make_idesc(kFmtBF16, kTile, 64, true, true);
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

constexpr int kBwdThreads = 448;  // 14 warps

enum : uint32_t {
    SITE_KV = 0x201, SITE_QDO_EMPTY = 0x202, SITE_QDO_FULL = 0x203, SITE_DQ_EMPTY = 0x204,
    SITE_P_FULL = 0x205, SITE_S_FULL = 0x206, SITE_DQ_FULL = 0x207, SITE_DKV = 0x208,
    SITE_DRAIN = 0x209, SITE_DQ_STAGED = 0x20A,
};

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// 1. preprocess: one block per kAuxRows consecutive rows of one head
// ---------------------------------------------------------------------------
// Both auxiliary kernels give each row D/8 threads (8 elements, one 16-byte
// load per thread), so a warp covers 2 (D = 128) or 4 (D = 64) rows and the
// row sum is a shuffle reduction over D/8 lanes.  Npad is a multiple of 128,
// so a block never straddles two heads and the head index is one division per
// block.
constexpr int kAuxRows = 64;
constexpr int kAuxThreads = 256;

template <int D>
__global__ void __launch_bounds__(kAuxThreads) bwd_pre_kernel(const BwdPreParams p) {
    constexpr int TPR = D / 8;                   // threads per row
    constexpr int RPP = kAuxThreads / TPR;       // rows per pass
    constexpr int PASSES = kAuxRows / RPP;
    const int blocks_per_head = p.Npad / kAuxRows;
    const int bh = static_cast<int>(blockIdx.x / blocks_per_head);
    const int n0 = static_cast<int>(blockIdx.x % blocks_per_head) * kAuxRows;
    const int b = bh / p.H, h = bh - b * p.H;
    const int c = threadIdx.x % TPR, rr = threadIdx.x / TPR;
    const uint16_t* obase = static_cast<const uint16_t*>(p.o) + b * p.os.b + h * p.os.h + c * 8;
    const uint16_t* dbase = static_cast<const uint16_t*>(p.dout) + b * p.dos.b + h * p.dos.h + c * 8;
    uint4 a[PASSES], g[PASSES];
#pragma unroll
    for (int k = 0; k < PASSES; ++k) {
        const int n = n0 + k * RPP + rr;
        a[k] = g[k] = make_uint4(0u, 0u, 0u, 0u);
        if (n < p.N) {
            a[k] = *reinterpret_cast<const uint4*>(obase + n * p.os.n);
            g[k] = *reinterpret_cast<const uint4*>(dbase + n * p.dos.n);
        }
    }
    if (blockIdx.x == 0)  // arrival counters of a split last round of the main kernel
        for (int k = threadIdx.x; k < p.split_cnt_words; k += kAuxThreads) p.split_cnt[k] = 0u;
    // Zero this block's rows of the dQ accumulator (contiguous, fp32 [BH, Npad, D]).
    float4* z = reinterpret_cast<float4*>(p.dq_acc + (static_cast<size_t>(bh) * p.Npad + n0) * D);
#pragma unroll
    for (int k = threadIdx.x; k < kAuxRows * D / 4; k += kAuxThreads)
        z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < PASSES; ++k) {
        const int n = n0 + k * RPP + rr;
        float acc = bf16lo(a[k].x) * bf16lo(g[k].x) + bf16hi(a[k].x) * bf16hi(g[k].x) +
                    bf16lo(a[k].y) * bf16lo(g[k].y) + bf16hi(a[k].y) * bf16hi(g[k].y) +
                    bf16lo(a[k].z) * bf16lo(g[k].z) + bf16hi(a[k].z) * bf16hi(g[k].z) +
                    bf16lo(a[k].w) * bf16lo(g[k].w) + bf16hi(a[k].w) * bf16hi(g[k].w);
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (c == 0) {
            const size_t v = static_cast<size_t>(bh) * p.Npad + n;
            p.dsum[v] = acc;
            p.lse2[v] = n < p.N ? -p.lse[static_cast<size_t>(bh) * p.N + n] * kLog2e : -INFINITY;
        }
    }
    pdl_launch_dependents();  // the main kernel may start its set-up (it waits for this grid)
}

// ---------------------------------------------------------------------------
// 3. dQ conversion: one block per kAuxRows rows of one head, 8 elements a thread
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kAuxThreads) dq_convert_kernel(const DqConvertParams p) {
    pdl_wait();  // launched as a dependent of the main kernel: its reductions must be done
    constexpr int TPR = D / 8;
    constexpr int RPP = kAuxThreads / TPR;
    constexpr int PASSES = kAuxRows / RPP;
    const int blocks_per_head = p.Npad / kAuxRows;
    const int bh = static_cast<int>(blockIdx.x / blocks_per_head);
    const int n0 = static_cast<int>(blockIdx.x % blocks_per_head) * kAuxRows;
    const int b = bh / p.H, h = bh - b * p.H;
    const int c = threadIdx.x % TPR, rr = threadIdx.x / TPR;
    const float* src = p.dq_acc + (static_cast<size_t>(bh) * p.Npad + n0 + rr) * D + c * 8;
    uint16_t* dst = static_cast<uint16_t*>(p.dq) + b * p.dqs.b + h * p.dqs.h + c * 8;
    const float s = p.scale;
#pragma unroll
    for (int k = 0; k < PASSES; ++k) {
        const int n = n0 + k * RPP + rr;
        if (n < p.N) {
            const float4* f = reinterpret_cast<const float4*>(src + k * RPP * D);
            const float4 x = f[0], y = f[1];
            st_global_v4(dst + static_cast<long long>(n) * p.dqs.n, pack_bf16x2(x.x * s, x.y * s),
                         pack_bf16x2(x.z * s, x.w * s), pack_bf16x2(y.x * s, y.y * s),
                         pack_bf16x2(y.z * s, y.w * s));
        }
    }
}

// ---------------------------------------------------------------------------
// Work of one backward CTA: one 128-row key tile of one key/value head and the
// query tiles (of every query head of its group) that see some key of it.
// ---------------------------------------------------------------------------
struct BwdWork {
    int kv_bh, j;        // (batch, key/value head) index and key tile
    int n_q_total;       // query tiles of a head
    int q_lo, n_qh;      // query tiles [q_lo, q_lo + n_qh) see this key tile
    bool full_range;     // every query tile does
    int q_bh0;           // first query (batch, head) index of the group
    int b_idx, hk_idx;   // batch, key/value head
    int bH0;             // (batch, head) index of head 0 of this batch
    int n_steps;         // G * n_qh (a part of a split item: its share of them)
    int slot;            // a part of a split item: its index among the split round's parts; else -1
    int parts;           // parts of the item (1: whole)
    int tt0, bh_first;   // (tile step, query head) of the first step

    __device__ explicit BwdWork(const BwdParams& prm) : BwdWork(prm, static_cast<int>(blockIdx.x)) {}

    // Work item `item` of the launch's numbering (items = key tiles of every
    // key/value head), whole.
    __device__ BwdWork(const BwdParams& prm, int item) {
        const int N = prm.N;
        // Non-causal: head-major order keeps the resident CTAs on a few heads, so
        // those heads' Q, dO and fp32 dQ accumulator stay in L2 while every key
        // tile reduces into them.  Causal: low key tiles (longest loops) of every
        // head first, which keeps the tail of the launch short.
        kv_bh = prm.causal ? item % prm.BHk : item / prm.n_kv;
        j = prm.causal ? item / prm.BHk : item % prm.n_kv;
        n_q_total = (N + kTile - 1) / kTile;
        // Query tiles holding the rows that see some key of this tile (window
        // i - win_left <= key <= i + win_right; negative = no bound).
        const int kr0 = j * kTile, kr1 = min(N - 1, j * kTile + kTile - 1);
        const int qrow_lo = prm.win_right < 0 ? 0 : max(0, kr0 - prm.win_right);
        const int qrow_hi = prm.win_left < 0 ? N - 1 : min(N - 1, kr1 + prm.win_left);
        q_lo = qrow_lo / kTile;
        n_qh = qrow_lo <= qrow_hi ? qrow_hi / kTile - q_lo + 1 : 0;  // per query head
        full_range = (q_lo == 0 && n_qh == n_q_total);
        // The G query heads sharing this key/value head (G = 1 without grouping)
        // are visited one after the other; dK and dV accumulate over all of them.
        const int G = prm.H / prm.Hk;
        q_bh0 = (kv_bh / prm.Hk) * prm.H + (kv_bh % prm.Hk) * G;
        b_idx = kv_bh / prm.Hk;
        hk_idx = kv_bh % prm.Hk;
        bH0 = b_idx * prm.H;
        n_steps = G * n_qh;
        slot = -1;
        parts = 1;
        tt0 = 0;
        bh_first = q_bh0;
    }
    // Item `v` of a launch with a split last round: from split_base on, part
    // (v - split_base) % P of item split_base + (v - split_base) / P, which takes
    // steps [t0, t1) of the item's walk (query head by query head, tile by tile).
    __device__ static BwdWork split_at(const BwdParams& prm, int v) {
        if (v < prm.split_base) return BwdWork(prm, v);
        const int s = v - prm.split_base, P = prm.split_parts;
        BwdWork w(prm, prm.split_base + s / P);
        w.make_part(s % P, P, s);
        return w;
    }
    // Entry e of a dealt launch (see BwdDeal): item e & 0x3FFF, whole, or (bit 15)
    // part (e >> 14) & 1 of its two parts, with partial slot 2 * item + part.
    __device__ static BwdWork dealt(const BwdParams& prm, int e) {
        const int item = e & 0x3FFF;
        BwdWork w(prm, item);
        if (e & 0x8000) w.make_part((e >> 14) & 1, 2, 2 * item + ((e >> 14) & 1));
        return w;
    }
    __device__ void make_part(int part, int P, int part_slot) {
        const int t0 = part * n_steps / P;
        n_steps = (part + 1) * n_steps / P - t0;
        slot = part_slot;
        parts = P;
        tt0 = t0 % n_qh;
        bh_first = q_bh0 + t0 / n_qh;
    }
    // Query tile of step t (tt = step index within one query head).  Over the
    // full range each key tile starts at its own index and wraps, so CTAs that
    // run together reduce into different dQ tiles; otherwise (causal, windows)
    // the range is walked upwards, which already starts neighbouring key tiles
    // on different query tiles.
    __device__ int q_tile(int tt) const {
        if (!full_range) return q_lo + tt;
        const int i = j + tt;
        return i < n_q_total ? i : i - n_q_total;
    }
};

// ---------------------------------------------------------------------------
// 2. main kernel
// ---------------------------------------------------------------------------
// Each 128-row query tile is processed as two 64-row halves h, each with its
// own compute warpgroup and its own 128 tensor-memory columns, so that the
// tensor core computes one half's S^T/dP^T while the other half's P^T/dS^T
// are being formed, and dV/dK for a half start as soon as that half is ready.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const BwdParams prm) {
    using T = BwdTraits<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + T::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t b_kv = bar0;
    auto b_qdo_full = [&](int s) { return bar0 + 8u * (1 + s); };
    auto b_qdo_empty = [&](int s) { return bar0 + 8u * (1 + T::STAGES + s); };
    const uint32_t b_s_full = bar0 + 8u * (1 + 2 * T::STAGES);  // + 8*h
    const uint32_t b_p_full = b_s_full + 16u;                   // + 8*h
    const uint32_t b_dq_full = b_p_full + 16u;                  // + 8*p
    const uint32_t b_dq_empty = b_dq_full + 16u;                // + 8*p
    const uint32_t b_dkv_full = b_dq_empty + 16u;
    const uint32_t b_done = b_dkv_full + 8u;
    const uint32_t b_dq_staged = b_done + 8u;  // + 8*p: all writer warps staged part p

    if ((sbase & 1023u) != 0) {
        if (threadIdx.x == 0) record_device_error(prm.st, ATTN_DEVERR_SMEM_ALIGN, 0x2FF);
        return;
    }

    const int N = prm.N;
    const BwdWork w(prm);
    const int j = w.j, n_qh = w.n_qh, q_bh0 = w.q_bh0, b_idx = w.b_idx, hk_idx = w.hk_idx,
              bH0 = w.bH0, n_steps = w.n_steps;
    auto q_tile = [&](int tt) { return w.q_tile(tt); };

    if (threadIdx.x == 0) {
        mbar_init(b_kv, 1);
        for (int s = 0; s < T::STAGES; ++s) {
            mbar_init(b_qdo_full(s), 1);
            // MMA commit, and for d = 64 the dQ writer (its reductions read the stage)
            mbar_init(b_qdo_empty(s), D == 128 ? 1 : 2);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(b_s_full + 8u * h, 1);
            mbar_init(b_p_full + 8u * h, 4);    // one arrival per compute warp
            mbar_init(b_dq_full + 8u * h, 1);
            mbar_init(b_dq_empty + 8u * h, 4);  // one arrival per dQ-writer warp
            mbar_init(b_dq_staged + 8u * h, 4);
        }
        mbar_init(b_dkv_full, 1);
        mbar_init(b_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 13) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == 12 && lane == 0) {
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
        tma_prefetch_map(&tm_do);
        tma_prefetch_map(&tm_dq);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 12) {
        // ================= TMA producer =================
        if (lane == 0) {
            mbar_arrive_expect_tx(b_kv, 2 * T::TILE_BYTES);
            for (int blk = 0; blk < T::NBLK; ++blk) {
                const int B = prm.BHk / prm.Hk;
                if (dbg_tma(sbase + T::OFF_K + blk * T::BLK_BYTES, blk * 64, j * kTile, hk_idx, b_idx, D, N,
                            prm.Hk, B, 2, 0x2D1))
                    tma_load_4d(sbase + T::OFF_K + blk * T::BLK_BYTES, &tm_k, b_kv, blk * 64, j * kTile,
                                hk_idx, b_idx);
                if (dbg_tma(sbase + T::OFF_V + blk * T::BLK_BYTES, blk * 64, j * kTile, hk_idx, b_idx, D, N,
                            prm.Hk, B, 2, 0x2D2))
                    tma_load_4d(sbase + T::OFF_V + blk * T::BLK_BYTES, &tm_v, b_kv, blk * 64, j * kTile,
                                hk_idx, b_idx);
            }
            int t = 0;
            int tt = 0, bh = q_bh0;  // step t = (head bh - q_bh0) * n_qh + tt
            for (; t < n_steps; ++t, ++tt) {
                if (tt == n_qh) {
                    tt = 0;
                    ++bh;
                }
                const int s = t % T::STAGES;
                const int i = q_tile(tt);
                if (t >= T::STAGES &&
                    !wait_one(b_qdo_empty(s), ((t / T::STAGES) - 1) & 1, abort_flag, prm.st,
                              SITE_QDO_EMPTY))
                    break;
                const uint32_t bf = b_qdo_full(s);
                mbar_arrive_expect_tx(bf, 2 * T::TILE_BYTES + 1024);
                const int B = prm.BHk / prm.Hk;
                for (int blk = 0; blk < T::NBLK; ++blk) {
                    const uint32_t dq_ = sbase + T::OFF_Q + s * T::TILE_BYTES + blk * T::BLK_BYTES;
                    const uint32_t ddo = sbase + T::OFF_DO + s * T::TILE_BYTES + blk * T::BLK_BYTES;
                    if (dbg_tma(dq_, blk * 64, i * kTile, bh - bH0, b_idx, D, N, prm.H, B, 2, 0x2D3))
                        tma_load_4d(dq_, &tm_q, bf, blk * 64, i * kTile, bh - bH0, b_idx);
                    if (dbg_tma(ddo, blk * 64, i * kTile, bh - bH0, b_idx, D, N, prm.H, B, 2, 0x2D4))
                        tma_load_4d(ddo, &tm_do, bf, blk * 64, i * kTile, bh - bH0, b_idx);
                }
                const size_t vrow = static_cast<size_t>(bh) * prm.Npad + i * kTile;
                if (dbg_ok(vrow + kTile <= static_cast<size_t>(B) * prm.H * prm.Npad, 0x2D5)) {
                    bulk_load(sbase + T::OFF_VEC + s * 1024, prm.lse2 + vrow, 512, bf);
                    bulk_load(sbase + T::OFF_VEC + s * 1024 + 512, prm.dsum + vrow, 512, bf);
                }
            }
            wait_drain(b_kv, 0, prm.st, SITE_DRAIN);
            const int first = t > T::STAGES ? t - T::STAGES : 0;
            for (int u = first; u < t; ++u)
                wait_drain(b_qdo_full(u % T::STAGES), (u / T::STAGES) & 1, prm.st, SITE_DRAIN);
        }
    } else if (warp == 13) {
        // ================= MMA issuer =================
        // The whole warp walks the schedule; one elected lane issues each group of
        // four products (uniform operands, one elect.sync per group).
        __syncwarp();
        {
            const uint32_t tDV = tmem + T::COL_DV, tDK = tmem + T::COL_DK;
            const uint32_t sK = sbase + T::OFF_K, sV = sbase + T::OFF_V, sDS = sbase + T::OFF_DS;
            // K-major operand, 16 bf16 (32 bytes) of K per instruction.
            auto kmaj = [](uint32_t base, int kk) {
                return desc_add(sw128_desc_words(base, 16, 1024), (kk >> 2) * T::BLK_BYTES + (kk & 3) * 32);
            };
            // MN-major operand: rows are the reduction index, 16 rows per instruction.
            auto mnmaj = [](uint32_t base, int kk) {
                return desc_add(sw128_desc_words(base, T::BLK_BYTES, 1024), kk * 16 * 128);
            };
            auto run = [&]() -> bool {
                if (!wait_warp(b_kv, 0, abort_flag, prm.st, SITE_KV)) return false;
                for (int t = 0; t < n_steps; ++t) {
                    const int s = t % T::STAGES;
                    const uint32_t sQ = sbase + T::OFF_Q + s * T::TILE_BYTES;
                    const uint32_t sDO = sbase + T::OFF_DO + s * T::TILE_BYTES;
                    if (!wait_warp(b_qdo_full(s), (t / T::STAGES) & 1, abort_flag, prm.st, SITE_QDO_FULL))
                        return false;
                    tc_fence_after();
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t tR = tmem + h * T::COL_REGION;
                        // S^T_h = K Q_h^T  (M = 128 keys, N = 64 queries, K = d)
#pragma unroll
                        for (int q = 0; q < D / 64; ++q)
                            mma_ss_warp4<false, 0, 2, 4, 6, 0, 2, 4, 6>(
                                tR, kmaj(sK, 4 * q), kmaj(sQ + h * T::HALF_BYTES, 4 * q), T::IDESC_SDP,
                                q > 0 ? 1u : 0u);
                        if (t > 0 && h < T::NDQ) {  // dQ part h of the previous tile has left
                            if (!wait_warp(b_dq_empty + 8u * h, (t - 1) & 1, abort_flag, prm.st,
                                           SITE_DQ_EMPTY))
                                return false;
                            tc_fence_after();
                        }
                        // dP^T_h = V dO_h^T
#pragma unroll
                        for (int q = 0; q < D / 64; ++q)
                            mma_ss_warp4<false, 0, 2, 4, 6, 0, 2, 4, 6>(
                                tR + T::COL_DP, kmaj(sV, 4 * q), kmaj(sDO + h * T::HALF_BYTES, 4 * q),
                                T::IDESC_SDP, q > 0 ? 1u : 0u);
                        mma_commit_warp(b_s_full + 8u * h);
                    }
                    for (int h = 0; h < 2; ++h) {
                        if (!wait_warp(b_p_full + 8u * h, t & 1, abort_flag, prm.st, SITE_P_FULL))
                            return false;
                        tc_fence_after();
                        const uint32_t tR = tmem + h * T::COL_REGION;
                        // dV += P^T_h dO_h : A = P^T_h (tensor memory), B = dO_h (MN-major)
                        mma_ts_warp4<false, 0, 8, 16, 24, 0, 128, 256, 384>(
                            tDV, tR, mnmaj(sDO + h * T::HALF_BYTES, 0), T::IDESC_DVK, (t > 0 || h > 0) ? 1u : 0u);
                        // dK += dS^T_h Q_h : A = dS^T_h (tensor memory), B = Q_h (MN-major)
                        // (dS^T_h packed in the first columns of dP^T_h, 8 per instruction;
                        // the dQ product that reuses those columns is issued after it)
                        mma_ts_warp4<false, 0, 8, 16, 24, 0, 128, 256, 384>(
                            tDK, tR + T::COL_DP, mnmaj(sQ + h * T::HALF_BYTES, 0), T::IDESC_DVK,
                            (t > 0 || h > 0) ? 1u : 0u);
                        if constexpr (D == 128) {
                            // dQ^T for the 64 queries of half h = K^T dS^T_h (M = d, N = 64,
                            // K = keys), into the dP^T columns of region h, issued as soon as
                            // dS^T_h exists rather than after both halves
#pragma unroll
                            for (int q = 0; q < kTile / 64; ++q)
                                mma_ss_warp4<false, 0, 128, 256, 384, 0, 128, 256, 384>(
                                    tR + T::COL_DP, mnmaj(sK, 4 * q), mnmaj(sDS + h * T::BLK_BYTES, 4 * q),
                                    T::IDESC_DQ, q > 0 ? 1u : 0u);
                            mma_commit_warp(b_dq_full + 8u * h);
                        }
                    }
                    // d = 64: dQ_i = dS K (M = queries, N = d) into the dP^T columns of region 0
#pragma unroll
                    for (int p = 0; p < (D == 128 ? 0 : T::NDQ); ++p) {
#pragma unroll
                        for (int q = 0; q < kTile / 64; ++q)
                            mma_ss_warp4<false, 0, 128, 256, 384, 0, 128, 256, 384>(
                                tmem + p * T::COL_REGION + T::COL_DP, mnmaj(sDS, 4 * q),
                                mnmaj(sK + p * T::BLK_BYTES, 4 * q), T::IDESC_DQ, q > 0 ? 1u : 0u);
                        mma_commit_warp(b_dq_full + 8u * p);
                    }
                    mma_commit_warp(b_qdo_empty(s));
                }
                mma_commit_warp(b_dkv_full);
                return true;
            };
            run();
            mma_commit_warp(b_done);
            wait_drain(b_done, 0, prm.st, SITE_DRAIN);
        }
    } else if (warp < 8) {
        // ================= compute warpgroups: P^T, dS^T for query half h =================
        const int h = warp >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;  // key row within the tile
        const int kv_row = j * kTile + r;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + h * T::COL_REGION + lane_off;
        const uint32_t tDP = tS + T::COL_DP;
        const float cs = prm.cs;
        uint8_t* ds_row = smem + T::OFF_DS + h * T::BLK_BYTES + r * 128;
        const int sw = r & 7;
        const uint32_t b_sf = b_s_full + 8u * h, b_pf = b_p_full + 8u * h;
        bool ok = true;
        for (int t = 0, tt = 0; t < n_steps; ++t, ++tt) {
            if (tt == n_qh) tt = 0;
            const int s = t % T::STAGES;
            const int i = q_tile(tt);
            const float* nlse2 =
                reinterpret_cast<const float*>(smem + T::OFF_VEC + s * 1024) + h * 64;
            const float* dsum = nlse2 + 128;
            // -LSE2_i and D_i arrived with Q_i/dO_i; waiting here (the phase is already
            // complete) makes those bulk-copied bytes visible to this thread.
            if (!wait_warp(b_qdo_full(s), (t / T::STAGES) & 1, abort_flag, prm.st, SITE_QDO_FULL) ||
                !wait_warp(b_sf, t & 1, abort_flag, prm.st, SITE_S_FULL)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // query column c of this half (row qc0 + c) sees key kv_row iff
            // cmin <= c <= cmax; the mask is applied only where some row of the
            // warp needs it (boundary tiles of a causal mask or a window)
            const int qc0 = i * kTile + h * 64;
            const int cmin = prm.win_right < 0 ? -kTile : kv_row - prm.win_right - qc0;
            const int cmax = prm.win_left < 0 ? 2 * kTile : kv_row + prm.win_left - qc0;
            const bool masked = __any_sync(0xffffffffu, cmin > 0 || cmax < 63);
            auto chunk = [&](auto masked_tag, int cc) {
                constexpr bool kMasked = decltype(masked_tag)::value;
                const int c0 = cc * 32;
                uint32_t sv[32], dp[32];
                tmem_ld32(tS + c0, sv);
                tmem_ld32(tDP + c0, dp);
                tmem_ld_wait(sv);
                tmem_ld_wait(dp);
                uint32_t pk[16], dsw[16];
                const float4* nl4 = reinterpret_cast<const float4*>(nlse2 + c0);
                const float4* ds4 = reinterpret_cast<const float4*>(dsum + c0);
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 nl = nl4[e / 4];  // same address in every lane: broadcast
                    const float4 dd = ds4[e / 4];
                    const float nlv[4] = {nl.x, nl.y, nl.z, nl.w};
                    const float ddv[4] = {dd.x, dd.y, dd.z, dd.w};
#pragma unroll
                    for (int h2 = 0; h2 < 4; h2 += 2) {
                        const int c = c0 + e + h2;
                        float x0, x1, t0, t1, d0, d1;
                        ffma2(x0, x1, u2f(sv[e + h2]), u2f(sv[e + h2 + 1]), cs, cs, nlv[h2], nlv[h2 + 1]);
                        float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                        if constexpr (kMasked) {
                            if (c < cmin || c > cmax) p0 = 0.f;
                            if (c + 1 < cmin || c + 1 > cmax) p1 = 0.f;
                        }
                        pk[(e + h2) / 2] = pack_bf16x2(p0, p1);
                        fsub2(t0, t1, u2f(dp[e + h2]), u2f(dp[e + h2 + 1]), ddv[h2], ddv[h2 + 1]);
                        fmul2(d0, d1, p0, p1, t0, t1);
                        dsw[(e + h2) / 2] = pack_bf16x2(d0, d1);
                    }
                }
                // P^T chunk -> columns [16 cc, 16 cc + 16) of S^T_h (already read), and
                // the dS^T chunk likewise into dP^T_h: the A operand of dK from tensor
                // memory, so that product reads only Q from shared memory
                tmem_st16(tS + 16 * cc, pk);
                tmem_st16(tDP + 16 * cc, dsw);
                // dS^T row r, 64 bytes -> 16-byte chunks x = 4 cc .. 4 cc + 3, swizzled
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    *reinterpret_cast<uint4*>(ds_row + (((cc * 4 + v) ^ sw) << 4)) =
                        make_uint4(dsw[4 * v], dsw[4 * v + 1], dsw[4 * v + 2], dsw[4 * v + 3]);
            };
            if (masked) {
                chunk(std::true_type{}, 0);
                chunk(std::true_type{}, 1);
            } else {
                chunk(std::false_type{}, 0);
                chunk(std::false_type{}, 1);
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_pf);
        }
        // ---- epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (scaled) ----
        if (ok && wait_warp(b_dkv_full, 0, abort_flag, prm.st, SITE_DKV)) {
            tc_fence_after();
            const bool row_ok = kv_row < N;
            const Strides& ds = h ? prm.dks : prm.dvs;
            const long long roff = (b_idx * ds.b + hk_idx * ds.h + (row_ok ? kv_row : 0) * ds.n) * 2;
            const uint32_t tsrc = tmem + (h ? T::COL_DK : T::COL_DV) + lane_off;
            uint8_t* dst = static_cast<uint8_t*>(h ? prm.dk : prm.dv) + roff;
            const float f = h ? prm.scale : 1.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tsrc + 32 * c, o);
                tmem_ld_wait(o);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(u2f(o[2 * e]) * f, u2f(o[2 * e + 1]) * f);
                if (row_ok) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        st_global_v4(dst + c * 64 + v * 16, pk[4 * v], pk[4 * v + 1], pk[4 * v + 2],
                                     pk[4 * v + 3]);
                }
            }
        }
    } else {
        // ================= dQ writer warpgroup (warps 8-11) =================
        // Each 64-column dQ part leaves tensor memory into shared memory (the Q
        // and dO buffers of the stage, free once this tile's MMAs are done), in
        // the 128-byte swizzled layout of two [128 x 32] fp32 boxes, and one
        // thread adds the boxes into the fp32 accumulator with TMA reductions.
        // The stage goes back to the producer when those reductions have read it.
        const int wq = warp & 3;
        const int r = wq * 32 + lane;  // query row within tile i
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const bool leader = (warp == 8 && lane == 0);
        constexpr int SLOTS_PER_BUF = T::TILE_BYTES / (kTile * 128);  // 16 KB boxes per buffer
        bool ok = true;
        int tt = 0, bh = q_bh0;
        if constexpr (D == 128) {
            // dQ^T_h sits in tensor memory with lane = feature, column = query, so one
            // warp-wide fp32 reduction covers 32 consecutive features of one query row:
            // a whole 128-byte line of the accumulator.  The adds go straight from
            // registers to L2; nothing is staged, and the Q/dO stage is handed back by
            // the MMA issuer alone as soon as the tile's products have read it.
            float* acc_col = prm.dq_acc + static_cast<size_t>(wq * 32 + lane);
            for (int t = 0; t < n_steps && ok; ++t, ++tt) {
                if (tt == n_qh) {
                    tt = 0;
                    ++bh;
                }
                const int i = q_tile(tt);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (!wait_warp(b_dq_full + 8u * h, t & 1, abort_flag, prm.st, SITE_DQ_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tq = tmem + h * T::COL_REGION + T::COL_DP + lane_off;
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tq, v0);
                    tmem_ld32(tq + 32, v1);
                    tmem_ld_wait(v0);
                    tmem_ld_wait(v1);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(b_dq_empty + 8u * h);  // dQ^T_h has left tensor memory
                    float* row0 = acc_col + (static_cast<size_t>(bh) * prm.Npad + i * kTile + 64 * h) * D;
#pragma unroll
                    for (int q = 0; q < 32; ++q) red_add_f32(row0 + q * D, __uint_as_float(v0[q]));
#pragma unroll
                    for (int q = 0; q < 32; ++q) red_add_f32(row0 + (32 + q) * D, __uint_as_float(v1[q]));
                }
            }
        } else {
            for (int t = 0; t < n_steps && ok; ++t, ++tt) {
                if (tt == n_qh) {
                    tt = 0;
                    ++bh;
                }
                const int s = t % T::STAGES;
                const int i = q_tile(tt);
    #pragma unroll
                for (int p = 0; p < T::NDQ; ++p) {
                    if (!wait_warp(b_dq_full + 8u * p, t & 1, abort_flag, prm.st, SITE_DQ_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tq = tmem + p * T::COL_REGION + T::COL_DP + lane_off;
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tq, v0);
                    tmem_ld32(tq + 32, v1);
                    tmem_ld_wait(v0);
                    tmem_ld_wait(v1);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(b_dq_empty + 8u * p);  // part p has left tensor memory
    #pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        const int u = 2 * p + b;  // staging box
                        const uint32_t box = sbase +
                                             (u < SLOTS_PER_BUF ? T::OFF_Q + s * T::TILE_BYTES + u * 16384
                                                                : T::OFF_DO + s * T::TILE_BYTES +
                                                                      (u - SLOTS_PER_BUF) * 16384);
                        uint8_t* row = smem + (box - sbase) + r * 128;
                        const uint32_t(&v)[32] = b ? v1 : v0;
    #pragma unroll
                        for (int x = 0; x < 8; ++x)
                            *reinterpret_cast<uint4*>(row + ((x ^ (r & 7)) << 4)) =
                                make_uint4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(b_dq_staged + 8u * p);
                    if (warp == 8) {
                        // Every writer warp has staged its rows.  A bounded wait, never a bare
                        // bar.sync: a warp that gave up must not strand the others.  The
                        // outcome is made uniform across warp 8 before anyone acts on it.
                        bool staged = true;
                        if (lane == 0)
                            staged = wait_one(b_dq_staged + 8u * p, t & 1, abort_flag, prm.st,
                                              SITE_DQ_STAGED);
                        if (!__shfl_sync(0xffffffffu, staged ? 1 : 0, 0)) {
                            ok = false;
                            break;
                        }
                    }
                    if (leader) {
    #pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            const int u = 2 * p + b;
                            const uint32_t box = sbase +
                                                 (u < SLOTS_PER_BUF ? T::OFF_Q + s * T::TILE_BYTES + u * 16384
                                                                    : T::OFF_DO + s * T::TILE_BYTES +
                                                                          (u - SLOTS_PER_BUF) * 16384);
                            if (dbg_ok(p * 64 + 32 * b < D && i * kTile < prm.Npad &&
                                           bh < (prm.BHk / prm.Hk) * prm.H,
                                       0x2D6))
                                tma_reduce_add_3d(&tm_dq, box, p * 64 + 32 * b, i * kTile, bh);
                        }
                        bulk_commit_group();
                    }
                }
                if (!ok) break;
                if (leader) {
                    bulk_wait_group_read0();       // the stage's bytes have been read
                    mbar_arrive(b_qdo_empty(s));   // second arrival: the producer may refill it
                }
            }
        }
        if (leader) bulk_wait_group0();  // every reduction has landed before the CTA retires
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// 2b. main kernel for d = 128: whole 128-query tiles, pipelined across steps
// ---------------------------------------------------------------------------
// Every product is full width (N = 128 queries or features).  An M = 128,
// N = 128 product with both operands in shared memory reads 8 KB per 64-cycle
// instruction and runs at the tensor rate, where the 64-query products of the
// half-tile kernel above read 6 KB per 32 cycles of work and are held to 48
// cycles by shared-memory bandwidth; the shared-memory traffic of a step drops
// from about 450 KB to 350 KB.  Per step t (query tile i_t):
//   S^T(t)  = K Q_t^T          -> region S  (lane = key, column = query)
//   dP^T(t) = V dO_t^T         -> region dP
//   dV     += P^T(t) dO_t      (A = P^T, packed bf16 over S^T in region S)
//   dK     += dS^T(t) Q_t      (A = dS^T, packed bf16 over S^T in region S)
//   dQ^T(t) = K^T dS^T(t)      -> region dP (lane = feature, column = query)
// Compute warpgroup h owns query columns 64h .. 64h + 63 of regions S and dP:
// it packs P^T over the first 32 of its S columns and dS^T over the other 32,
// so both A operands sit in region S and region dP is free as soon as dP^T has
// been read.  Issue order of step t:
//   [P^T(t) formed] dV(t), [dS^T(t) formed] dK(t), dQ^T(t), S^T(t+1),
//   [dQ^T(t) drained], dP^T(t+1), [P^T(t+1) formed] dV(t+1) ...
// The dQ writer takes dQ^T(t) out of tensor memory while S^T(t+1) executes, so
// the drain costs the tensor pipe nothing; the exponentials of step t+1 run
// while dP^T(t+1) executes and the dS^T pass while dV(t+1) does.  The tensor
// pipe executes in issue order, so a product that overwrites a region is
// issued after the last product that reads it.
// The per-query terms -LSE log2 e (of the exponent) and -D (of dS) are not
// loaded by the compute warps: each enters S^T or dP^T through one more K = 16
// product against a tile of their bf16 parts, so S^T holds S^T - LSE log2 e / cs
// and dP^T holds dP^T - D (the per-column broadcast loads they replace shared
// the memory pipeline with the dQ reductions).
// Warps 0-3 / 4-7: compute for query columns 0-63 / 64-127 of the tile (one
// thread per key row); warps 8-11: dQ writer; warp 12: TMA and the per-query
// terms; warp 13: MMA.
struct BwdFullTraits {
    static constexpr int D = 128;
    static constexpr int BLK_BYTES = kTile * 128;        // one [128 rows x 128 B] block
    static constexpr int HALF_BYTES = 64 * 128;          // 64 rows of a block
    static constexpr int TILE_BYTES = kTile * D * 2;
    static constexpr int DS_BYTES = kTile * kTile * 2;   // dS^T [128 keys][128 queries], 2 blocks
    static constexpr int STAGES = 2;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + TILE_BYTES;
    static constexpr int OFF_Q = OFF_V + TILE_BYTES;            // + stage * TILE_BYTES
    static constexpr int OFF_DO = OFF_Q + STAGES * TILE_BYTES;  // + stage * TILE_BYTES
    static constexpr int OFF_DS = OFF_DO + STAGES * TILE_BYTES;
    // The per-query terms of the exponent (-LSE log2 e / cs) and of dS (-D) enter
    // S^T and dP^T as one more K = 16 product each: A = a row of ones over the
    // term's parts (the same 8 rows for every row group), B = each query's parts
    // (written per step by the producer warp).
    static constexpr int OFF_AUG_A = OFF_DS + DS_BYTES;         // 2 core matrices, 8 x 16 B each
    static constexpr int OFF_AUG_B = OFF_AUG_A + 2 * 128;       // [128 queries][8 bf16]
    static constexpr int OFF_BAR = OFF_AUG_B + kTile * 16;
    // barriers: kv_full, qdo_full[2], qdo_empty[2], s_full, dp_full, p_full, dq_full,
    //           dq_empty, dkv_full, done, kv_empty, aug_full, pa_full
    static constexpr int NBARS = 1 + 2 * STAGES + 10;
    static constexpr int SMEM_BYTES = OFF_BAR + NBARS * 8 + 16;
    static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 384;
    static constexpr uint32_t IDESC_SDP = make_idesc(kFmtBF16, kTile, kTile, false, false);
    static constexpr uint32_t IDESC_DVK = make_idesc(kFmtBF16, kTile, D, false, true);
    static constexpr uint32_t IDESC_DQ = make_idesc(kFmtBF16, D, kTile, true, true);
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

enum : uint32_t { SITE_DP_FULL = 0x20B, SITE_KV_EMPTY = 0x20C, SITE_AUG_FULL = 0x20D, SITE_PA_FULL = 0x20E };

// Per-CTA item lists of a dealt launch (bwd_main_full_kernel<2>), for causal
// launches whose longest items (a key tile visits every query head of its group,
// so causal items run from G n_q steps down to G) reach or pass the per-CTA mean:
// the longest are split in two parts (steps [0, n/2) and [n/2, n) of the item's
// walk, partial slots 2 item + part) and the parts and whole items are dealt
// longest first, each to the CTA with the least work so far.  Causal launches
// whose items are not split but whose Q, dO and dQ accumulators overflow the L2
// are dealt the same way in groups of heads, one group after the other (see
// bwd_deal_for).  The lists are built on the host and travel as a kernel
// parameter.
constexpr int kDealGrid = 160;   // CTAs the lists cover at most
constexpr int kDealMax = 8192;   // entries (items and parts) at most
template <int MODE>
struct BwdDealArg {};
template <>
struct BwdDealArg<2> {
    uint16_t start[kDealGrid + 1];  // CTA c takes entries [start[c], start[c + 1])
    uint16_t entry[kDealMax];       // item | part << 14 | (split ? 1 << 15 : 0)
};

// Epilogue of one warp's 32 rows (row r of this lane) of dV (h = 0) or dK (h = 1,
// written times f = scale) for a part of a split item: the part's fp32 partial
// rows (tensor memory at tsrc) go to its slot of the workspace; the item's last
// part to arrive for these rows adds up every part's partial in part order (so
// the result does not depend on which part is last), writes the bf16 rows and
// leaves the counter at zero.  Kept out of line so that the main loops'
// registers do not depend on it.
__device__ __noinline__ void split_part_epilogue(float* split_part, unsigned* split_cnt, int slot, int parts,
                                                 int h, int wq, int r, uint32_t tsrc, uint8_t* dst,
                                                 bool row_ok, float f) {
    constexpr int D = 128;
    const int lane = threadIdx.x & 31;
    const int item_slot = slot / parts;
    auto part_row = [&](int sub) { return split_part + ((static_cast<size_t>(sub) * 2 + h) * kTile + r) * D; };
    float* mine = part_row(slot);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tsrc + 32 * c, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int v = 0; v < 8; ++v)
            st_global_v4(mine + c * 32 + 4 * v, o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
    }
    __threadfence();
    __syncwarp();
    unsigned* cnt = split_cnt + (item_slot * 2 + h) * 4 + wq;
    unsigned arrived = 0;
    if (lane == 0) arrived = atomicAdd(cnt, 1u);
    arrived = __shfl_sync(0xffffffffu, arrived, 0);
    if (arrived != static_cast<unsigned>(parts - 1)) return;
    if (lane == 0) *cnt = 0u;  // every part has arrived
    __threadfence();
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
        float a[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) a[e] = 0.f;
#pragma unroll 1
        for (int q = 0; q < parts; ++q) {
            const float4* src = reinterpret_cast<const float4*>(part_row(item_slot * parts + q) + c * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const float4 x = __ldcg(src + v);
                a[4 * v] += x.x;
                a[4 * v + 1] += x.y;
                a[4 * v + 2] += x.z;
                a[4 * v + 3] += x.w;
            }
        }
        if (row_ok) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
                st_global_v4(dst + c * 64 + v * 16, pack_bf16x2(a[8 * v] * f, a[8 * v + 1] * f),
                             pack_bf16x2(a[8 * v + 2] * f, a[8 * v + 3] * f),
                             pack_bf16x2(a[8 * v + 4] * f, a[8 * v + 5] * f),
                             pack_bf16x2(a[8 * v + 6] * f, a[8 * v + 7] * f));
        }
    }
}

// v as hi + mid + lo, each rounded to bf16 (hi + mid + lo = v to about 2^-24
// relative: each remainder is exact in fp32), returned halved (exact) and
// packed as the bf16 words (hi/2 | mid/2 << 16, lo/2).
__device__ __forceinline__ uint2 split3_half_bf16(float v) {
    const uint32_t hb = pack_bf16x2(v, 0.f);
    const float r1 = v - __uint_as_float(hb << 16);
    const uint32_t mb = pack_bf16x2(r1, 0.f);
    const float r2 = r1 - __uint_as_float(mb << 16);
    const uint32_t lb = pack_bf16x2(r2, 0.f);
    const uint32_t h2 = pack_bf16x2(0.5f * __uint_as_float(hb << 16), 0.5f * __uint_as_float(mb << 16));
    return make_uint2(h2, pack_bf16x2(0.5f * __uint_as_float(lb << 16), 0.f));
}

// Pause of the dQ writer between groups of eight reductions (see the writer).
constexpr unsigned kDqPauseNs = 60;

// MODE 0: items dealt in snake order; 1: the same with a split last round; 2: the
// per-CTA lists of a BwdDeal (causal launches with long items).  V8: every dK and
// dV row starts on a 32-byte boundary (32-byte stores in the epilogue; a runtime
// choice between the two store widths measured 1-2 % slower than either alone).
template <int MODE, bool V8>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_main_full_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const BwdParams prm, const __grid_constant__ BwdDealArg<MODE> deal) {
    using T = BwdFullTraits;
    constexpr int D = T::D;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + T::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t b_kv = bar0;
    auto b_qdo_full = [&](int s) { return bar0 + 8u * (1 + s); };
    auto b_qdo_empty = [&](int s) { return bar0 + 8u * (1 + T::STAGES + s); };
    const uint32_t b_s_full = bar0 + 8u * (1 + 2 * T::STAGES);  // S^T(t) in region S
    const uint32_t b_dp_full = b_s_full + 8u;                    // dP^T(t) in region dP
    const uint32_t b_p_full = b_dp_full + 8u;                    // P^T(t), dS^T(t) formed
    const uint32_t b_dq_full = b_p_full + 8u;                    // dQ^T(t) in region dP
    const uint32_t b_dq_empty = b_dq_full + 8u;                  // dQ^T(t) read out
    const uint32_t b_dkv_full = b_dq_empty + 8u;
    const uint32_t b_done = b_dkv_full + 8u;
    const uint32_t b_kv_empty = b_done + 8u;                     // an item's K, V read for the last time
    const uint32_t b_aug_full = b_kv_empty + 8u;                 // per-query terms of the next step written
    const uint32_t b_pa_full = b_aug_full + 8u;                  // P^T(t) formed (dS^T(t) not yet)

    if ((sbase & 1023u) != 0) {
        if (threadIdx.x == 0) record_device_error(prm.st, ATTN_DEVERR_SMEM_ALIGN, 0x2FE);
        return;
    }

    const int N = prm.N;
    // Persistent CTAs: CTA c takes the items of the launch's numbering (key tiles
    // of every key/value head; non-causal head-major, causal longest first) in
    // rounds of G = gridDim.x, dealt in snake order (CTA c takes item rG + c in
    // even rounds and rG + G - 1 - c in odd ones), so that longest-first causal
    // items leave every CTA within about one item of the others.  An item's
    // epilogue (dV, dK out of tensor memory) overlaps the next item's K/V copy
    // and first products.  item_at returns -1 after the last round and -2 for a
    // round in which this CTA has no item (only the last round can be short).
    const int n_items = MODE == 1 ? prm.split_base + (prm.BHk * prm.n_kv - prm.split_base) * prm.split_parts
                                  : prm.BHk * prm.n_kv;
    auto work = [&](int v) {  // the work of item v (a part of a split item from split_base on)
        if constexpr (MODE == 1) return BwdWork::split_at(prm, v);
        else if constexpr (MODE == 2) return BwdWork::dealt(prm, v);
        else return BwdWork(prm, v);
    };
    auto item_at = [&](int r) -> int {
        if constexpr (MODE == 2) {  // entry r of this CTA's list
            const int e = deal.start[blockIdx.x] + r;
            return e < deal.start[blockIdx.x + 1] ? static_cast<int>(deal.entry[e]) : -1;
        }
        const long long base = static_cast<long long>(r) * gridDim.x;
        if (base >= n_items) return -1;
        const int c = (r & 1) ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
        return base + c < n_items ? static_cast<int>(base + c) : -2;
    };

    if (threadIdx.x == 0) {
        mbar_init(b_kv, 1);
        mbar_init(b_kv_empty, 1);
        for (int s = 0; s < T::STAGES; ++s) {
            mbar_init(b_qdo_full(s), 1);
            mbar_init(b_qdo_empty(s), 1);
        }
        mbar_init(b_s_full, 1);
        mbar_init(b_dp_full, 1);
        mbar_init(b_p_full, 8);    // one arrival per compute warp
        mbar_init(b_pa_full, 8);
        mbar_init(b_dq_full, 1);
        mbar_init(b_dq_empty, 4);  // one arrival per dQ-writer warp
        mbar_init(b_dkv_full, 1);
        mbar_init(b_done, 1);
        mbar_init(b_aug_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 13) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == 12 && lane == 0) {
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
        tma_prefetch_map(&tm_do);
    }
    if (warp == 12 && lane < 16) {
        // the constant A tile of the per-query products: row i of core matrix 0 (the
        // S^T term, ones over elements 0-2) and of core matrix 1 (the dP^T term,
        // ones over elements 4-6)
        const uint32_t one2 = 0x3F803F80u, one1 = 0x00003F80u;  // bf16 1.0 pairs
        *reinterpret_cast<uint4*>(smem + T::OFF_AUG_A + lane * 16) =
            lane < 8 ? make_uint4(one2, one1, 0u, 0u) : make_uint4(0u, 0u, one2, one1);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a dependent of the preprocess kernel: the set-up above overlapped
    // its last blocks; D, -LSE log2 e and the zeroed dQ accumulator are read below.
    pdl_wait();

    // Steps are counted over all of the CTA's items (g): the Q/dO stages and the
    // per-step barriers run on through item boundaries.
    if (warp == 12) {
        // ================= TMA producer and per-query terms =================
        // The whole warp runs the loop (lane 0 issues the copies).  Besides Q, dO,
        // K and V it writes, per step, the B tile of the per-query products: row q
        // holds halves of the three bf16 parts of -LSE log2 e / cs (the S^T term:
        // P^T = 2^(cs (S^T - LSE log2 e / cs))) and of -D (the dP^T term); lane l
        // owns rows l + 32 m.  The raw values are loaded a step ahead of the step's
        // copies and written a step after them, once dP^T of the previous step (the
        // last reader of the single tile) has completed; aug_full publishes them to
        // the MMA warp before that step's S^T.
        const int B = prm.BHk / prm.Hk;
        const float rcs = 1.f / prm.cs;
        int g = 0;   // steps loaded so far (all items)
        int k = 0;   // items whose K/V copy was issued
        bool ok = true;
        float raw_l[4], raw_d[4];  // -LSE log2 e and D of step `pend`, rows lane + 32 m
        float nxt_l[4], nxt_d[4];  // the same for step pend + 1 (in flight)
        int pend = -1;             // step whose terms are loaded but not yet written (-1: none)
        auto fetch = [&](int bh, int i) {  // step (query head bh, tile i) into nxt (bh < 0: none)
            if (bh < 0) return;
            const size_t vrow = static_cast<size_t>(bh) * prm.Npad + i * kTile + lane;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                nxt_l[m] = prm.lse2[vrow + 32 * m];
                nxt_d[m] = prm.dsum[vrow + 32 * m];
            }
        };
        // (query head, tile) of the first step of the CTA's items from round rr on
        auto first_step = [&](int rr, int& bh, int& tile) {
            bh = -1;
            tile = 0;
            for (;; ++rr) {
                const int item = item_at(rr);
                if (item == -1) return;
                if (item < 0) continue;
                const BwdWork w = work(item);
                if (w.n_steps > 0) {
                    bh = w.bh_first;
                    tile = w.q_tile(w.tt0);
                    return;
                }
            }
        };
        auto write_terms = [&]() -> bool {
            if (pend < 0) return true;
            if (pend > 0 && !wait_warp(b_dp_full, (pend - 1) & 1, abort_flag, prm.st, SITE_DP_FULL)) return false;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                float vl = raw_l[m] * rcs;
                // -inf on padding rows: a large finite negative value makes P^T zero
                // there; +inf (a row that sees no key) only meets masked entries
                if (!(vl >= -1e30f)) vl = -1e30f;
                if (!(vl <= 1e30f)) vl = 0.f;
                const uint2 a = split3_half_bf16(vl), b = split3_half_bf16(-raw_d[m]);
                *reinterpret_cast<uint4*>(smem + T::OFF_AUG_B + (lane + 32 * m) * 16) =
                    make_uint4(a.x, a.y, b.x, b.y);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_aug_full);
            pend = -1;
            return true;
        };
        // Q and dO of global step g (query tile i of query head bh); the previous
        // step's terms are written first, and those of the step after this one
        // (query head nbh, tile ni; nbh < 0: none) are fetched
        auto load_step = [&](int i, int bh, int bH0, int b_idx, int nbh, int ni) -> bool {
            if (!write_terms()) return false;
            const int s = g % T::STAGES;
            if (g >= T::STAGES &&
                !wait_warp(b_qdo_empty(s), ((g / T::STAGES) - 1) & 1, abort_flag, prm.st, SITE_QDO_EMPTY))
                return false;
            if (lane == 0) {
                const uint32_t bf = b_qdo_full(s);
                mbar_arrive_expect_tx(bf, 2 * T::TILE_BYTES);
                for (int blk = 0; blk < 2; ++blk) {
                    const uint32_t dq_ = sbase + T::OFF_Q + s * T::TILE_BYTES + blk * T::BLK_BYTES;
                    const uint32_t ddo = sbase + T::OFF_DO + s * T::TILE_BYTES + blk * T::BLK_BYTES;
                    if (dbg_tma(dq_, blk * 64, i * kTile, bh - bH0, b_idx, D, N, prm.H, B, 2, 0x2D3))
                        tma_load_4d(dq_, &tm_q, bf, blk * 64, i * kTile, bh - bH0, b_idx);
                    if (dbg_tma(ddo, blk * 64, i * kTile, bh - bH0, b_idx, D, N, prm.H, B, 2, 0x2D4))
                        tma_load_4d(ddo, &tm_do, bf, blk * 64, i * kTile, bh - bH0, b_idx);
                }
            }
            __syncwarp();
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                raw_l[m] = nxt_l[m];
                raw_d[m] = nxt_d[m];
            }
            fetch(nbh, ni);
            pend = g;
            ++g;
            return true;
        };
        {
            int bh0, tile0;
            first_step(0, bh0, tile0);
            fetch(bh0, tile0);
        }
        for (int r = 0; ok; ++r) {
            const int item = item_at(r);
            if (item == -1) break;
            if (item < 0) continue;
            const BwdWork w = work(item);
            int nx_bh, nx_tile;  // first step of the next item with steps
            first_step(r + 1, nx_bh, nx_tile);
            int tt = w.tt0, bh = w.bh_first;
            // (query head, tile) of the step after step t of this item
            auto after = [&](int t, int& nbh, int& ni) {
                if (t + 1 >= w.n_steps) {
                    nbh = nx_bh;
                    ni = nx_tile;
                } else {
                    const bool wrap = tt + 1 == w.n_qh;
                    nbh = wrap ? bh + 1 : bh;
                    ni = w.q_tile(wrap ? 0 : tt + 1);
                }
            };
            int nbh, ni;
            // the item's first Q/dO stage goes out as soon as a stage is free,
            // then K and V once the previous item's last products have read them
            after(0, nbh, ni);
            if (w.n_steps > 0 && !load_step(w.q_tile(tt), bh, w.bH0, w.b_idx, nbh, ni)) {
                ok = false;
                break;
            }
            if (k > 0 && !wait_warp(b_kv_empty, (k - 1) & 1, abort_flag, prm.st, SITE_KV_EMPTY)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(b_kv, 2 * T::TILE_BYTES);
                for (int blk = 0; blk < 2; ++blk) {
                    if (dbg_tma(sbase + T::OFF_K + blk * T::BLK_BYTES, blk * 64, w.j * kTile, w.hk_idx, w.b_idx,
                                D, N, prm.Hk, B, 2, 0x2D1))
                        tma_load_4d(sbase + T::OFF_K + blk * T::BLK_BYTES, &tm_k, b_kv, blk * 64, w.j * kTile,
                                    w.hk_idx, w.b_idx);
                    if (dbg_tma(sbase + T::OFF_V + blk * T::BLK_BYTES, blk * 64, w.j * kTile, w.hk_idx, w.b_idx,
                                D, N, prm.Hk, B, 2, 0x2D2))
                        tma_load_4d(sbase + T::OFF_V + blk * T::BLK_BYTES, &tm_v, b_kv, blk * 64, w.j * kTile,
                                    w.hk_idx, w.b_idx);
                }
            }
            __syncwarp();
            ++k;
            for (int t = 1; t < w.n_steps && ok; ++t) {
                if (++tt == w.n_qh) {
                    tt = 0;
                    ++bh;
                }
                after(t, nbh, ni);
                ok = load_step(w.q_tile(tt), bh, w.bH0, w.b_idx, nbh, ni);
            }
        }
        if (ok) write_terms();  // the last step's terms
        // Let every copy this warp started land before the CTA can exit.
        if (lane == 0) {
            if (k > 0) wait_drain(b_kv, (k - 1) & 1, prm.st, SITE_DRAIN);
            const int first = g > T::STAGES ? g - T::STAGES : 0;
            for (int u = first; u < g; ++u)
                wait_drain(b_qdo_full(u % T::STAGES), (u / T::STAGES) & 1, prm.st, SITE_DRAIN);
        }
        __syncwarp();
    } else if (warp == 13) {
        // ================= MMA issuer =================
        __syncwarp();
        {
            const uint32_t tS = tmem + T::COL_S, tDP = tmem + T::COL_DP;
            const uint32_t tDV = tmem + T::COL_DV, tDK = tmem + T::COL_DK;
            const uint32_t sK = sbase + T::OFF_K, sV = sbase + T::OFF_V, sDS = sbase + T::OFF_DS;
            // K-major operand, 16 bf16 (32 bytes) of K per instruction.
            auto kmaj = [](uint32_t base, int kk) {
                return desc_add(sw128_desc_words(base, 16, 1024), (kk >> 2) * T::BLK_BYTES + (kk & 3) * 32);
            };
            // MN-major operand: rows are the reduction index, 16 rows per instruction.
            auto mnmaj = [](uint32_t base, int kk) {
                return desc_add(sw128_desc_words(base, T::BLK_BYTES, 1024), kk * 16 * 128);
            };
            auto stage_q = [&](int g) { return sbase + T::OFF_Q + (g % T::STAGES) * T::TILE_BYTES; };
            auto stage_do = [&](int g) { return sbase + T::OFF_DO + (g % T::STAGES) * T::TILE_BYTES; };
            // The per-query term as one more product: A (no swizzle, both steps 0)
            // repeats one core matrix of ones over the term's parts in every row and
            // in both halves of K = 16, B (no swizzle, K step 0) repeats each query's
            // parts, so the product adds twice the sum of the stored half-parts.
            const SmemDesc aug_b = noswz_desc_words(sbase + T::OFF_AUG_B, 0, 128);
            const SmemDesc aug_s = noswz_desc_words(sbase + T::OFF_AUG_A, 0, 0);
            const SmemDesc aug_dp = noswz_desc_words(sbase + T::OFF_AUG_A + 128, 0, 0);
            // S^T or dP^T: M = 128 keys, N = 128 queries, K = d, both operands K-major,
            // plus the per-query term.
            auto issue_sdp = [&](uint32_t d_tmem, uint32_t a, uint32_t b, SmemDesc aug) {
#pragma unroll
                for (int q = 0; q < D / 64; ++q)
                    mma_ss_warp4<false, 0, 2, 4, 6, 0, 2, 4, 6>(d_tmem, kmaj(a, 4 * q), kmaj(b, 4 * q),
                                                                T::IDESC_SDP, q > 0 ? 1u : 0u);
                mma_ss_warp1_acc(d_tmem, aug, aug_b, T::IDESC_SDP);
            };
            // dV or dK += A B: A = packed bf16 in tensor memory (queries 0-63 at +0,
            // 64-127 at +64: each compute warpgroup packs over its own columns), B
            // MN-major (rows = queries), 16 queries per instruction.
            auto issue_acc = [&](uint32_t d_tmem, uint32_t a_tmem, uint32_t b, uint32_t accumulate) {
                mma_ts_warp4<false, 0, 8, 16, 24, 0, 128, 256, 384>(d_tmem, a_tmem, mnmaj(b, 0),
                                                                    T::IDESC_DVK, accumulate);
                mma_ts_warp4<false, 0, 8, 16, 24, 0, 128, 256, 384>(d_tmem, a_tmem + 64,
                                                                    mnmaj(b + T::HALF_BYTES, 0),
                                                                    T::IDESC_DVK, 1u);
            };
            // dQ^T = K^T dS^T: M = d, N = 128 queries, K = 128 keys, both MN-major.
            auto issue_dq = [&]() {
#pragma unroll
                for (int q = 0; q < kTile / 64; ++q)
                    mma_ss_warp4<false, 0, 128, 256, 384, 0, 128, 256, 384>(
                        tDP, mnmaj(sK, 4 * q), mnmaj(sDS, 4 * q), T::IDESC_DQ, q > 0 ? 1u : 0u);
            };
            int g0 = 0;  // global index of the item's first step
            int k = 0;   // items started
            // One item: dkv_full is committed after its last dK product, kv_empty after
            // its last dQ product (the last reader of K; V's was the last dP^T).
            auto run_item = [&](int n_steps) -> bool {
                if (!wait_warp(b_kv, k & 1, abort_flag, prm.st, SITE_KV) ||
                    !wait_warp(b_qdo_full(g0 % T::STAGES), (g0 / T::STAGES) & 1, abort_flag, prm.st,
                               SITE_QDO_FULL) ||
                    !wait_warp(b_aug_full, g0 & 1, abort_flag, prm.st, SITE_AUG_FULL))
                    return false;
                tc_fence_after();
                issue_sdp(tS, sK, stage_q(g0), aug_s);
                mma_commit_warp(b_s_full);
                if (g0 > 0) {  // the previous item's last dQ^T has left region dP
                    if (!wait_warp(b_dq_empty, (g0 - 1) & 1, abort_flag, prm.st, SITE_DQ_EMPTY)) return false;
                    tc_fence_after();
                }
                issue_sdp(tDP, sV, stage_do(g0), aug_dp);
                mma_commit_warp(b_dp_full);
                for (int t = 0; t < n_steps; ++t) {
                    const int g = g0 + t;
                    const uint32_t acc = t > 0 ? 1u : 0u;
                    // dV(t) as soon as P^T(t) is formed: it runs during the dS^T pass
                    if (!wait_warp(b_pa_full, g & 1, abort_flag, prm.st, SITE_PA_FULL)) return false;
                    tc_fence_after();
                    issue_acc(tDV, tS, stage_do(g), acc);       // dV += P^T(t) dO_t
                    if (!wait_warp(b_p_full, g & 1, abort_flag, prm.st, SITE_P_FULL)) return false;
                    tc_fence_after();
                    issue_acc(tDK, tS + 32, stage_q(g), acc);   // dK += dS^T(t) Q_t
                    // dV, dK are final after the last step's products: the epilogue may
                    // start while the last dQ product and its reductions run
                    if (t + 1 == n_steps) mma_commit_warp(b_dkv_full);
                    issue_dq();                                 // dQ^T(t), region dP
                    mma_commit_warp(b_dq_full);
                    mma_commit_warp(b_qdo_empty(g % T::STAGES));  // Q_t, dO_t read (after dQ^T(t))
                    if (t + 1 == n_steps) mma_commit_warp(b_kv_empty);
                    if (t + 1 < n_steps) {
                        const int u = g + 1;
                        if (!wait_warp(b_qdo_full(u % T::STAGES), (u / T::STAGES) & 1, abort_flag, prm.st,
                                       SITE_QDO_FULL) ||
                            !wait_warp(b_aug_full, u & 1, abort_flag, prm.st, SITE_AUG_FULL))
                            return false;
                        tc_fence_after();
                        issue_sdp(tS, sK, stage_q(u), aug_s);   // S^T(t+1) over P^T(t), dS^T(t)
                        mma_commit_warp(b_s_full);
                        if (!wait_warp(b_dq_empty, g & 1, abort_flag, prm.st, SITE_DQ_EMPTY)) return false;
                        tc_fence_after();
                        issue_sdp(tDP, sV, stage_do(u), aug_dp);  // dP^T(t+1) over dQ^T(t)
                        mma_commit_warp(b_dp_full);
                    }
                }
                return true;
            };
            for (int r = 0;; ++r) {
                const int item = item_at(r);
                if (item == -1) break;
                if (item < 0) continue;
                const BwdWork w = work(item);
                if (w.n_steps == 0) {  // nothing sees this key tile: zero dV, dK, release K/V
                    if (!wait_warp(b_kv, k & 1, abort_flag, prm.st, SITE_KV)) break;
                    mma_commit_warp(b_dkv_full);
                    mma_commit_warp(b_kv_empty);
                } else if (!run_item(w.n_steps)) {
                    break;
                }
                g0 += w.n_steps;
                ++k;
            }
            mma_commit_warp(b_done);
            wait_drain(b_done, 0, prm.st, SITE_DRAIN);
        }
    } else if (warp < 8) {
        // ================= compute: P^T, dS^T for query columns 64h .. 64h + 63 =================
        const int h = warp >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;  // key row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tSh = tmem + T::COL_S + 64 * h + lane_off;
        const uint32_t tDPh = tmem + T::COL_DP + 64 * h + lane_off;
        const float cs = prm.cs;
        uint8_t* ds_row = smem + T::OFF_DS + h * T::BLK_BYTES + r * 128;
        const int sw = r & 7;
        bool ok = true;
        int g = 0;  // global step
        int k = 0;  // items finished
        for (int rr = 0; ok; ++rr) {
        const int item = item_at(rr);
        if (item == -1) break;
        if (item < 0) continue;
        const BwdWork w = work(item);
        const int kv_row = w.j * kTile + r;
        for (int t = 0, tt = w.tt0; t < w.n_steps; ++t, ++tt, ++g) {
            if (tt == w.n_qh) tt = 0;
            const int i = w.q_tile(tt);
            if (!wait_warp(b_s_full, g & 1, abort_flag, prm.st, SITE_S_FULL)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // query column c of this warpgroup (row qc0 + c) sees key kv_row iff
            // cmin <= c <= cmax; masked only where some row of the warp needs it
            const int qc0 = i * kTile + h * 64;
            const int cmin = prm.win_right < 0 ? -kTile : kv_row - prm.win_right - qc0;
            const int cmax = prm.win_left < 0 ? 2 * kTile : kv_row + prm.win_left - qc0;
            const bool masked = __any_sync(0xffffffffu, cmin > 0 || cmax < 63);
            float p[64];  // P^T of this thread's key row and the warpgroup's 64 queries
            // Phase A: P^T = 2^(cs (S^T - LSE log2 e / cs)), the query term already in
            // S^T; packed bf16 over the S^T columns already read (the A operand of
            // dV), fp32 kept for dS^T.
            auto phase_a = [&](auto masked_tag, auto cc_tag) {
                constexpr bool kMasked = decltype(masked_tag)::value;
                constexpr int cc = decltype(cc_tag)::value;
                constexpr int c0 = cc * 32;
                uint32_t sv[32];
                tmem_ld32(tSh + c0, sv);
                tmem_ld_wait(sv);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int c = c0 + e;
                    float x0, x1;
                    fmul2(x0, x1, u2f(sv[e]), u2f(sv[e + 1]), cs, cs);
                    float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                    if constexpr (kMasked) {
                        if (c < cmin || c > cmax) p0 = 0.f;
                        if (c + 1 < cmin || c + 1 > cmax) p1 = 0.f;
                    }
                    p[c] = p0;
                    p[c + 1] = p1;
                    pk[e / 2] = pack_bf16x2(p0, p1);
                }
                tmem_st16(tSh + 16 * cc, pk);
            };
            // Phase B: dS^T = P^T (dP^T - D), the -D term already in dP^T; packed bf16
            // over the second 32 of this warpgroup's S^T columns (read in phase A; the
            // A operand of dK) and into shared memory with 128-byte swizzle (the B
            // operand of dQ^T, MN-major).
            auto phase_b = [&](auto cc_tag) {
                constexpr int cc = decltype(cc_tag)::value;
                constexpr int c0 = cc * 32;
                uint32_t dp[32];
                tmem_ld32(tDPh + c0, dp);
                tmem_ld_wait(dp);
                uint32_t dsw[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float d0, d1;
                    fmul2(d0, d1, p[c0 + e], p[c0 + e + 1], u2f(dp[e]), u2f(dp[e + 1]));
                    dsw[e / 2] = pack_bf16x2(d0, d1);
                }
                tmem_st16(tSh + 32 + 16 * cc, dsw);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    *reinterpret_cast<uint4*>(ds_row + (((cc * 4 + v) ^ sw) << 4)) =
                        make_uint4(dsw[4 * v], dsw[4 * v + 1], dsw[4 * v + 2], dsw[4 * v + 3]);
            };
            using C0 = std::integral_constant<int, 0>;
            using C1 = std::integral_constant<int, 1>;
            if (masked) {
                phase_a(std::true_type{}, C0{});
                phase_a(std::true_type{}, C1{});
            } else {
                phase_a(std::false_type{}, C0{});
                phase_a(std::false_type{}, C1{});
            }
            // P^T(t) is complete in tensor memory: dV(t) may start
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_pa_full);
            if (!wait_warp(b_dp_full, g & 1, abort_flag, prm.st, SITE_DP_FULL)) {
                ok = false;
                break;
            }
            tc_fence_after();
            phase_b(C0{});
            phase_b(C1{});
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_p_full);
        }
        // ---- epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (scaled) ----
        // Reading dV/dK out of tensor memory here precedes (in this warp's program
        // order) the arrival that lets the next item's first dV/dK product overwrite
        // them.
        if (!ok || !wait_warp(b_dkv_full, k & 1, abort_flag, prm.st, SITE_DKV)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const bool row_ok = kv_row < N;
        const Strides& ds = h ? prm.dks : prm.dvs;
        const long long roff = (w.b_idx * ds.b + w.hk_idx * ds.h + (row_ok ? kv_row : 0) * ds.n) * 2;
        const uint32_t tsrc = tmem + (h ? T::COL_DK : T::COL_DV) + lane_off;
        uint8_t* dst = static_cast<uint8_t*>(h ? prm.dk : prm.dv) + roff;
        const float f = h ? prm.scale : 1.f;
        if (MODE != 0 && w.slot >= 0) {
            split_part_epilogue(prm.split_part, prm.split_cnt, w.slot, w.parts, h, wq, r, tsrc, dst, row_ok, f);
        } else {
            const bool empty = w.n_steps == 0;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tsrc + 32 * c, o);
                tmem_ld_wait(o);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = empty ? 0u : pack_bf16x2(u2f(o[2 * e]) * f, u2f(o[2 * e + 1]) * f);
                if (row_ok) st_global_row64<V8>(dst + c * 64, pk);
            }
        }
        ++k;
        }  // items
    } else {
        // ================= dQ writer (warps 8-11) =================
        // dQ^T(t) sits in region dP with lane = feature, column = query: warp q
        // holds features 32q .. 32q + 31 of all 128 queries, so one warp-wide fp32
        // reduction covers a 128-byte line of the accumulator.  The whole tile
        // leaves tensor memory before the reductions start, so that dP^T(t+1) can
        // be issued as soon as possible.
        const int wq = warp & 3;
        const uint32_t tq = tmem + T::COL_DP + (static_cast<uint32_t>(wq * 32) << 16);
        float* acc_col = prm.dq_acc + static_cast<size_t>(wq * 32 + lane);
        bool ok = true;
        int g = 0;  // global step
        for (int rr = 0; ok; ++rr) {
            const int item = item_at(rr);
            if (item == -1) break;
            if (item < 0) continue;
            const BwdWork w = work(item);
            const bool last_item = item_at(rr + 1) < 0;
            int tt = w.tt0, bh = w.bh_first;
            for (int t = 0; t < w.n_steps; ++t, ++tt, ++g) {
                if (tt == w.n_qh) {
                    tt = 0;
                    ++bh;
                }
                const int i = w.q_tile(tt);
                if (!wait_warp(b_dq_full, g & 1, abort_flag, prm.st, SITE_DQ_FULL)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t v0[32], v1[32], v2[32], v3[32];
                tmem_ld32(tq, v0);
                tmem_ld32(tq + 32, v1);
                tmem_ld32(tq + 64, v2);
                tmem_ld32(tq + 96, v3);
                tmem_ld_wait(v0);
                tmem_ld_wait(v1);
                tmem_ld_wait(v2);
                tmem_ld_wait(v3);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(b_dq_empty);
                float* row0 = acc_col + (static_cast<size_t>(bh) * prm.Npad + i * kTile) * D;
                // The reductions go out in groups of eight with a short pause between
                // groups: a burst of 128 per thread right after the drain fills the
                // memory pipeline that the compute warps' shared-memory loads also use
                // (whole step 2.55 -> 2.27-2.30 ms at B1 H32 N8192 d128).  The CTA's
                // last step competes with nothing but the epilogue: no pauses.
                const bool pace = !(last_item && t + 1 == w.n_steps);
                auto send32 = [&](float* rows, const uint32_t (&v)[32]) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        red_add_f32(rows + q * D, __uint_as_float(v[q]));
                        if ((q & 7) == 7 && pace) __nanosleep(kDqPauseNs);
                    }
                };
                send32(row0, v0);
                send32(row0 + 32 * D, v1);
                send32(row0 + 64 * D, v2);
                send32(row0 + 96 * D, v3);
            }
        }
    }

    pdl_launch_dependents();  // the dQ conversion may be scheduled (it waits for this grid)
    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Host side of BwdDealArg<2>: the predicted end of the launch (in steps, an
// item costing its steps plus kDealItemCost) of the snake order against the
// deal with the longest items split, for a few split thresholds; the best deal
// is used when it ends at least 3 % sooner.  Results are cached per shape.
constexpr double kDealItemCost = 1.5;  // per-item overhead in steps (clock stamps: ~3.4 us / 2.3 us)
constexpr double kDealPartCost = 2.0;  // a part's fp32 partial written and summed, in steps
// Shorter items are never dealt: with items of at most 16 steps a deal made B2 H4
// N1024 and B1 H8 N2048 causal 45-50 % slower (the parts' partials and epilogues
// against a few steps of work), while items of 64 steps and more gained 14-39 %.
constexpr int kDealMinLongest = 64;
constexpr int kSplitMinPartSteps = 16;  // steps a part of the split last round keeps at least
constexpr double kDealGroupBytes = 64.0 * (1 << 20);  // Q, dO, dQ accumulator: half the L2

double snake_makespan(const std::vector<double>& cost, int grid) {
    std::vector<double> load(grid, 0.0);
    const int n = static_cast<int>(cost.size());
    for (int r = 0; static_cast<long long>(r) * grid < n; ++r)
        for (int c = 0; c < grid; ++c) {
            const long long i = static_cast<long long>(r) * grid + ((r & 1) ? grid - 1 - c : c);
            if (i < n) load[c] += cost[i];
        }
    return *std::max_element(load.begin(), load.end());
}

// Deal of the n causal items of p (item i: key tile i / BHk of key/value head
// i % BHk, longest first) with the x longest split in two, in groups of gs
// key/value heads (group g: heads [g gs, (g + 1) gs); gs >= BHk is one group):
// group by group, longest entry first onto the least-loaded CTA.  Returns the
// makespan, or -1 when the entries do not fit the table.
double build_deal(const BwdParams& p, int grid, int x, int gs, BwdDealArg<2>* out) {
    const int n = p.BHk * p.n_kv, G = p.H / p.Hk;
    struct E {
        int group;
        double cost;
        int code;
    };
    std::vector<E> es;
    es.reserve(n + x);
    for (int i = 0; i < n; ++i) {
        const int steps = G * (p.n_kv - i / p.BHk), group = (i % p.BHk) / gs;
        if (i < x) {
            es.push_back({group, steps / 2 + kDealItemCost + kDealPartCost, i | 0x8000});
            es.push_back({group, steps - steps / 2 + kDealItemCost + kDealPartCost, i | 0x8000 | 0x4000});
        } else {
            es.push_back({group, steps + kDealItemCost, i});
        }
    }
    if (static_cast<int>(es.size()) > kDealMax) return -1.0;
    std::stable_sort(es.begin(), es.end(), [](const E& a, const E& b) {
        return a.group != b.group ? a.group < b.group : a.cost > b.cost;
    });
    using L = std::pair<double, int>;  // (load, CTA)
    std::priority_queue<L, std::vector<L>, std::greater<L>> heap;
    for (int c = 0; c < grid; ++c) heap.push({0.0, c});
    std::vector<std::vector<uint16_t>> lists(grid);
    double makespan = 0.0;
    for (const E& e : es) {
        L top = heap.top();
        heap.pop();
        top.first += e.cost;
        makespan = std::max(makespan, top.first);
        lists[top.second].push_back(static_cast<uint16_t>(e.code));
        heap.push(top);
    }
    if (out != nullptr) {
        int k = 0;
        for (int c = 0; c < grid; ++c) {
            out->start[c] = static_cast<uint16_t>(k);
            for (uint16_t v : lists[c]) out->entry[k++] = v;
        }
        for (int c = grid; c <= kDealGrid; ++c) out->start[c] = static_cast<uint16_t>(k);
    }
    return makespan;
}

// Fills *out and returns true when a deal over `grid` CTAs is worth it for this
// causal launch, against the snake order over `snake_grid` CTAs (the items, when
// there are fewer than CTAs).  Two kinds of deal:
//  * split: the longest items in two parts, when that is predicted to end at
//    least 3 % sooner (longest item of kDealMinLongest steps or more);
//  * grouped (no item split): when the launch's Q, dO and fp32 dQ accumulator
//    (8 B per query row and feature) pass kDealGroupBytes, items are dealt in
//    groups of key/value heads, the smallest group (power of two) whose
//    predicted end is within 1 % of one group's, so that the heads in flight
//    keep theirs in the L2.  The longest-first order otherwise runs every head
//    at once (B2 H16 N4096: 128 MB, the size of the L2; causal B4 H32 N2048
//    grouped by 8 heads: 0.548 -> 0.417 ms, B2 H16 N4096 0.347 -> 0.339 ms).
bool bwd_deal_for(const BwdParams& p, int snake_grid, int grid, BwdDealArg<2>* out) {
    const int n = p.BHk * p.n_kv, G = p.H / p.Hk;
    if (!p.causal || grid > kDealGrid || n > 0x3FFF || n > kDealMax) return false;
    const bool may_split = p.split_cap >= 2 && G * p.n_kv >= kDealMinLongest;
    const double bytes = 8.0 * kTile * BwdFullTraits::D * static_cast<double>(n) * G;
    if (!may_split && bytes <= kDealGroupBytes) return false;
    struct Cached {
        long long key[6];
        bool use;
        BwdDealArg<2> deal;
    };
    static std::mutex mu;
    static std::vector<Cached> cache;  // a few shapes; the oldest is replaced
    static size_t next = 0;
    const long long key[6] = {p.BHk, p.n_kv, G, grid, snake_grid, p.split_cap};
    std::lock_guard<std::mutex> lock(mu);
    for (const Cached& c : cache)
        if (std::equal(key, key + 6, c.key)) {
            if (c.use) *out = c.deal;
            return c.use;
        }
    Cached c{};
    std::copy(key, key + 6, c.key);
    std::vector<double> cost(n);
    double total = 0.0;
    for (int i = 0; i < n; ++i) total += cost[i] = G * (p.n_kv - i / p.BHk) + kDealItemCost;
    const double snake = snake_makespan(cost, snake_grid), mean = total / grid;
    int best_x = -1;
    double best = snake;
    for (double thr : {0.6, 0.75, 0.9, 1.0, 1.2}) {
        if (!may_split) break;
        int x = 0;  // items are split only with two steps or more (a part never has none)
        while (x < n && cost[x] > thr * mean && cost[x] >= 2 + kDealItemCost) ++x;
        x = std::min(x, p.split_cap / 2);
        const double m = build_deal(p, grid, x, p.BHk, nullptr);
        if (m > 0.0 && m < best) {
            best = m;
            best_x = x;
        }
    }
    c.use = best_x >= 0 && best < 0.97 * snake;
    if (c.use) {
        build_deal(p, grid, best_x, p.BHk, &c.deal);
    } else if (bytes > kDealGroupBytes) {
        const double one = build_deal(p, grid, 0, p.BHk, nullptr);
        for (int gs = 1; gs < p.BHk && !c.use; gs *= 2)
            if (build_deal(p, grid, 0, gs, nullptr) <= 1.01 * one) {
                build_deal(p, grid, 0, gs, &c.deal);
                c.use = true;
            }
    }
    if (cache.size() < 8) {
        cache.push_back(c);
    } else {
        cache[next] = c;
        next = (next + 1) % cache.size();
    }
    if (c.use) *out = c.deal;
    return c.use;
}

template <int D>
cudaError_t launch_bwd_main_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& p,
                                 cudaStream_t stream) {
    using T = BwdTraits<D>;
    static const cudaError_t attr = cudaFuncSetAttribute(
        bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
    if (attr != cudaSuccess) return attr;
    const long long grid = static_cast<long long>(p.BHk) * p.n_kv;
    const cudaError_t dbg = dbg_set_word(p.st.word, stream);
    if (dbg != cudaSuccess) return dbg;
    bwd_main_kernel<D><<<static_cast<unsigned>(grid), kBwdThreads, T::SMEM_BYTES, stream>>>(tq, tk, tv, tdo, tdq,
                                                                                        p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t stream) {
    if (p.Npad % kAuxRows != 0) return cudaErrorInvalidValue;
    const long long blocks = static_cast<long long>(p.BH) * (p.Npad / kAuxRows);
    if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
    if (p.D == 64) bwd_pre_kernel<64><<<static_cast<unsigned>(blocks), kAuxThreads, 0, stream>>>(p);
    else if (p.D == 128) bwd_pre_kernel<128><<<static_cast<unsigned>(blocks), kAuxThreads, 0, stream>>>(p);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_dq_convert(const DqConvertParams& p, cudaStream_t stream) {
    if (p.Npad % kAuxRows != 0) return cudaErrorInvalidValue;
    const long long blocks = static_cast<long long>(p.BH) * (p.Npad / kAuxRows);
    if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
    // a programmatic dependent of the main kernel (see pdl_wait)
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kAuxThreads);
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (p.D == 64) return cudaLaunchKernelEx(&cfg, dq_convert_kernel<64>, p);
    if (p.D == 128) return cudaLaunchKernelEx(&cfg, dq_convert_kernel<128>, p);
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_main(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& p,
                            cudaStream_t stream) {
    if (D == 64) return launch_bwd_main_impl<64>(tq, tk, tv, tdo, tdq, p, stream);
    if (D == 128) {
        using T = BwdFullTraits;
        static const cudaError_t attr = [] {
            cudaError_t e = cudaSuccess;
            for (const void* fn : {reinterpret_cast<const void*>(bwd_main_full_kernel<0, false>),
                                   reinterpret_cast<const void*>(bwd_main_full_kernel<1, false>),
                                   reinterpret_cast<const void*>(bwd_main_full_kernel<2, false>),
                                   reinterpret_cast<const void*>(bwd_main_full_kernel<0, true>),
                                   reinterpret_cast<const void*>(bwd_main_full_kernel<1, true>),
                                   reinterpret_cast<const void*>(bwd_main_full_kernel<2, true>)})
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
            return e;
        }();
        if (attr != cudaSuccess) return attr;
        // persistent: one CTA per SM (shared memory admits one), items in snake order
        const long long items = static_cast<long long>(p.BHk) * p.n_kv;
        long long grid = items;
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (sms < grid) grid = sms;
        if (grid < 1) return cudaSuccess;
        // Split the last round when it would leave CTAs idle (no mask: every item
        // has the same steps), into P = grid / r parts per item, P >= 2; with fewer
        // items than SMs, the only round: every item in P = SMs / items parts, on
        // P times as many CTAs.  A part keeps at least kSplitMinPartSteps steps:
        // splitting 16-step items in two made B1 H4 N2048 19 % slower, 32-step
        // ones (B1 H2 N4096) 7 % faster.
        BwdParams pp = p;
        pp.split_base = static_cast<int>(items);
        pp.split_parts = 1;
        const long long rem = items < sms ? items : items % grid;
        const long long steps = static_cast<long long>(p.H / p.Hk) * p.n_kv;
        if (rem > 0 && p.causal == 0 && p.win_left < 0 && p.win_right < 0 && p.split_cap > 0) {
            long long parts = (items < sms ? sms : grid) / rem;
            if (parts > steps / kSplitMinPartSteps) parts = steps / kSplitMinPartSteps;
            if (parts * rem > p.split_cap) parts = p.split_cap / rem;
            if (parts >= 2) {
                pp.split_base = static_cast<int>(items - rem);
                pp.split_parts = static_cast<int>(parts);
                if (items < sms) grid = items * parts;
            }
        }
        const cudaError_t dbg = dbg_set_word(p.st.word, stream);
        if (dbg != cudaSuccess) return dbg;
        BwdDealArg<2> deal;
        const int deal_grid = sms < kDealGrid ? sms : kDealGrid;
        // a programmatic dependent of the preprocess kernel (see pdl_wait)
        cudaLaunchAttribute pdl;
        pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pdl.val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(kBwdThreads);
        cfg.dynamicSmemBytes = T::SMEM_BYTES;
        cfg.stream = stream;
        cfg.attrs = &pdl;
        cfg.numAttrs = 1;
        const bool v8 = p.dkv_v8 != 0;
        if (p.causal && bwd_deal_for(p, static_cast<int>(grid), deal_grid, &deal)) {
            pp.split_parts = 2;
            cfg.gridDim = dim3(static_cast<unsigned>(deal_grid));
            return v8 ? cudaLaunchKernelEx(&cfg, bwd_main_full_kernel<2, true>, tq, tk, tv, tdo, pp, deal)
                      : cudaLaunchKernelEx(&cfg, bwd_main_full_kernel<2, false>, tq, tk, tv, tdo, pp, deal);
        }
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        if (pp.split_parts > 1)
            return v8 ? cudaLaunchKernelEx(&cfg, bwd_main_full_kernel<1, true>, tq, tk, tv, tdo, pp, BwdDealArg<1>{})
                      : cudaLaunchKernelEx(&cfg, bwd_main_full_kernel<1, false>, tq, tk, tv, tdo, pp,
                                           BwdDealArg<1>{});
        return v8 ? cudaLaunchKernelEx(&cfg, bwd_main_full_kernel<0, true>, tq, tk, tv, tdo, pp, BwdDealArg<0>{})
                  : cudaLaunchKernelEx(&cfg, bwd_main_full_kernel<0, false>, tq, tk, tv, tdo, pp, BwdDealArg<0>{});
    }
    return cudaErrorInvalidValue;
}

int bwd_smem_bytes(int D) {
    if (D == 64) return BwdTraits<64>::SMEM_BYTES;
    if (D == 128) return BwdFullTraits::SMEM_BYTES;
    return 0;
}

}  // namespace attn
