// Forward exact attention on sm_103a: O = softmax(scale * Q K^T [+ causal mask]) V
// and the per-row natural log-sum-exp, computed tile by tile with the online
// softmax so that S and P never leave the SM (FlashAttention digest, sections
// 1-2; FlashAttention paper item 58: running max, running sum, and the same
// rescale applied to the output accumulator).
//
// A work item is two 128-row query tiles of one (batch, head); a CTA streams the
// item's key/value tiles through a shared-memory ring (persistent CTAs loop over
// items, see the work assignment below):
//
//   warp 8      TMA producer: Q tiles once, then K_j, V_j into the ring
//   warp 9      MMA issuer (one thread): S_g = Q_g K_j^T and O_g += P_g V_j on
//               the tensor cores, accumulators in tensor memory
//   warps 0-3   softmax for query tile 0 (one thread per row)
//   warps 4-7   softmax for query tile 1
//
// Tensor memory (512 columns x 128 lanes, lane = query row):
//   [0,128)   S_0 (fp32); after softmax P_0 packed into its first columns
//   [128,256) S_1 / P_1
//   [256,256+D)      O_0 accumulator (fp32)
//   [256+D,256+2D)   O_1 accumulator
//
// The MMA issue order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) keeps the tensor
// pipe busy while the two softmax warpgroups work on alternate tiles (the
// producer/consumer and GEMM-softmax overlap of the FlashAttention-3 digest,
// sections 1-2), adapted to tcgen05: the overlap comes from two query tiles
// ping-ponging on one MMA issuer instead of register-resident accumulators.
//
// The output rescale is lazy ("conditional rescaling" in the FlashAttention-3
// walkthrough tags): O and the row sums always share the same, possibly stale,
// maximum m_used, which keeps the result exact.  A row computes a tile maximum
// only on its first tile and otherwise lets P exceed 1; a tile whose row sum
// passes 448 (FP8: then some P could leave E4M3's range) or 2^60 (bf16, which
// keeps its relative precision at any magnitude) is redone with its own
// maximum.
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kRedoBound = 1152921504606846976.0f;  // 2^60
constexpr float kRedoBoundFP8 = 448.0f;                 // largest finite E4M3 value
// With the exponential offload on (FMAEXP), the group of four columns (offset
// within each 32) whose exponentials run on the FMA pipe (ex2_fma2) instead of
// MUFU: one group in eight.
constexpr int kFmaExpGroup = 28;

template <int D, bool FP8>
struct FwdTraits {
    static constexpr int EB = FP8 ? 1 : 2;                  // bytes per element
    static constexpr int ROW_BYTES = D * EB;
    static constexpr int NBLK = ROW_BYTES / 128;            // 128-byte swizzle blocks per row
    static constexpr int BLK_ELEMS = 128 / EB;              // elements per swizzle-block row
    static constexpr int BLK_BYTES = kTile * 128;           // one [128 rows x 128 B] block
    static constexpr int TILE_BYTES = kTile * ROW_BYTES;
    static constexpr int UMMA_K = FP8 ? 32 : 16;            // K of one tcgen05.mma
    static constexpr int KV_SLOTS = TILE_BYTES == 32768 ? 5 : 8;
    static constexpr int SMEM_Q = 2 * TILE_BYTES;
    static constexpr int SMEM_KV = KV_SLOTS * TILE_BYTES;
    // barriers: q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], o_full[2], mma_done,
    //           q_empty
    static constexpr int NBARS = 1 + 2 * KV_SLOTS + 2 + 2 + 2 + 1 + 1;
    static constexpr int SMEM_BYTES = SMEM_Q + SMEM_KV + NBARS * 8 + 16;
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + D;
    static constexpr uint32_t FMT = FP8 ? kFmtE4M3 : kFmtBF16;
    static constexpr uint32_t IDESC_S = make_idesc(FMT, kTile, kTile, false, false);
    static constexpr uint32_t IDESC_PV = make_idesc(FMT, kTile, D, false, true);
    static_assert(NBLK >= 1 && ROW_BYTES % 128 == 0, "row must be whole 128-byte blocks");
    static_assert(D % 32 == 0 && D <= 128, "head dim");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Site ids recorded when a wait gives up (kernel 1 = forward).
enum : uint32_t {
    SITE_Q = 0x101, SITE_KV_EMPTY = 0x102, SITE_KV_FULL = 0x103, SITE_P_FULL = 0x104,
    SITE_S_FULL = 0x105, SITE_O_FULL = 0x106, SITE_DRAIN = 0x107, SITE_Q_EMPTY = 0x108,
};

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

template <int D, bool FP8, bool FMAEXP>
__global__ void __launch_bounds__(320, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams prm) {
    using T = FwdTraits<D, FP8>;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint8_t* sQ = smem;
    uint8_t* sKV = smem + T::SMEM_Q;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + T::SMEM_KV);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + T::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const uint32_t bar0 = smem_u32(bars);
    const uint32_t b_q = bar0;
    auto b_kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
    auto b_kv_empty = [&](int s) { return bar0 + 8u * (1 + T::KV_SLOTS + s); };
    const uint32_t b_s_full = bar0 + 8u * (1 + 2 * T::KV_SLOTS);     // +8*g
    const uint32_t b_p_full = b_s_full + 16u;                        // +8*g
    const uint32_t b_o_full = b_p_full + 16u;                        // +8*g
    const uint32_t b_done = b_o_full + 16u;
    const uint32_t b_q_empty = b_done + 8u;  // every product reading the Q tiles of an item is done

    if ((smem_u32(smem) & 1023u) != 0) {  // swizzle atoms need 1024-byte alignment
        if (threadIdx.x == 0) record_device_error(prm.st, ATTN_DEVERR_SMEM_ALIGN, 0x1FF);
        return;
    }

    // ---- work assignment ----
    // The CTAs are persistent: CTA c takes work items c, c + G, c + 2G, ... (G =
    // gridDim.x), so that setting up barriers and tensor memory happens once and one
    // item's epilogue overlaps the next item's loads and first products.  An item is
    // a query-tile pair of one (batch, head) and, for split-KV, one split.
    // Without a mask (and for sliding windows) items are numbered head-major, so the
    // items in flight cover only a few heads and each head's K and V come from HBM
    // about once.  Causal: heaviest query tiles of every head first (longest-first
    // keeps the tail short).  Split-KV: the splits of one pair are adjacent items.
    const bool split_mode = prm.n_splits > 1;
    const bool lpt = prm.causal != 0;
    const int N = prm.N;
    // Work units of a head: query-tile pairs, or single tiles when the launch has so
    // few pairs that they would leave at least half of the SMs idle (a CTA then
    // runs one tile's chain, and twice as many CTAs share the work).
    const int n_units = prm.single ? (N + kTile - 1) / kTile : prm.n_pairs;
    const int n_items = prm.BH * n_units * prm.n_splits;
    struct Item {
        int split, bh, pair, kv_lo, n_kv, b_idx, h_idx, hk_idx;
        int lo0, lo1, n0, n1;  // key-tile range [lo_g, lo_g + n_g) of query tile g
        __device__ int lo(int g) const { return g ? lo1 : lo0; }
        __device__ int n(int g) const { return g ? n1 : n0; }
    };
    auto item_info = [&](int item) {
        Item w;
        const int cta = item / prm.n_splits;
        w.split = item % prm.n_splits;
        w.bh = lpt ? cta % prm.BH : cta / n_units;
        const int unit = n_units - 1 - (lpt ? cta / prm.BH : cta % n_units);
        w.pair = prm.single ? unit >> 1 : unit;
        const int g_only = prm.single ? unit & 1 : -1;  // the one live tile of a single item
        // Query tile g uses key tiles [lo_g, lo_g + n_g): the tiles holding
        // keys visible to some row of the tile (window i - win_left <= key <=
        // i + win_right, a negative bound meaning none), cut to the item's split.
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const int qt = 2 * w.pair + g;
            const int r0 = qt * kTile, r1 = min(N - 1, qt * kTile + kTile - 1);
            const int key_lo = prm.win_left < 0 ? 0 : max(0, r0 - prm.win_left);
            const int key_hi = prm.win_right < 0 ? N - 1 : min(N - 1, r1 + prm.win_right);
            const int lo = max(key_lo / kTile, w.split * prm.split_len);
            const int hi = min(key_hi / kTile, w.split * prm.split_len + prm.split_len - 1);
            const bool live = (g_only < 0 || g == g_only) && r0 < N && key_lo <= key_hi && hi >= lo;
            if (g == 0) {
                w.lo0 = live ? lo : 0;
                w.n0 = live ? hi - lo + 1 : 0;
            } else {
                w.lo1 = live ? lo : 0;
                w.n1 = live ? hi - lo + 1 : 0;
            }
        }
        // The item streams key tiles [kv_lo, kv_lo + n_kv): the union of both ranges
        // (they overlap or touch: the two tiles' rows are adjacent).
        w.kv_lo = w.n(0) > 0 ? (w.n(1) > 0 ? min(w.lo(0), w.lo(1)) : w.lo(0)) : w.lo(1);
        const int kv_hi = max(w.n(0) > 0 ? w.lo(0) + w.n(0) : 0, w.n(1) > 0 ? w.lo(1) + w.n(1) : 0);
        w.n_kv = (w.n(0) > 0 || w.n(1) > 0) ? kv_hi - w.kv_lo : 0;
        // Key/value head of the query head (grouped-query attention: H/Hk query heads
        // share one key/value head; Hk == H is ordinary multi-head attention).
        w.b_idx = w.bh / prm.H;
        w.h_idx = w.bh % prm.H;
        w.hk_idx = w.h_idx / (prm.H / prm.Hk);
        return w;
    };

    // The r-th item of this CTA.  Round r holds items [r G, r G + G); even rounds
    // are dealt in CTA order and odd rounds in reverse (a snake), so that with
    // items in longest-first order (causal) the CTAs' totals stay within about
    // one item of each other, as the hardware block scheduler's would, while the
    // CTAs stay resident.  Returns -1 after the last round and -2 for a round in
    // which this CTA has no item (only the last one can be short).
    auto item_at = [&](int r) -> int {
        const long long base = static_cast<long long>(r) * gridDim.x;
        if (base >= n_items) return -1;
        const int c = (r & 1) ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
        return base + c < n_items ? static_cast<int>(base + c) : -2;
    };

    if (threadIdx.x == 0) {
        mbar_init(b_q, 1);
        for (int s = 0; s < T::KV_SLOTS; ++s) {
            mbar_init(b_kv_full(s), 1);
            mbar_init(b_kv_empty(s), 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(b_s_full + 8u * g, 1);
            mbar_init(b_p_full + 8u * g, 4);  // one arrival per softmax warp
            mbar_init(b_o_full + 8u * g, 1);
        }
        mbar_init(b_done, 1);
        mbar_init(b_q_empty, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8) {
        // ================= TMA producer =================
        if (lane == 0) {
            int idx = 0;  // K/V loads issued so far (ring position), over all items
            int k = 0;    // items started
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int item = item_at(r);
                if (item == -1) break;
                if (item < 0) continue;
                const Item it = item_info(item);
                // The ring takes K_0, V_0, K_1, V_1, ... of the item in consecutive
                // slots.  K_0, V_0 and K_1 complete on their own slots' barriers (they
                // go out around the item's Q copy); from j = 1 on, V_j and K_{j+1},
                // which the MMA warp needs at the same point (PV(j), then S(j+1)), both
                // complete on V_j's barrier, so that it waits once per key tile.
                // K_{j+1}'s own barrier gets a plain arrival (no bytes), so that every
                // slot's barrier still completes one phase per use; nothing waits on it.
                auto claim = [&](int i) -> bool {  // slot of load i is free
                    const int round = i / T::KV_SLOTS;
                    return round == 0 ||
                           wait_one(b_kv_empty(i % T::KV_SLOTS), (round - 1) & 1, abort_flag, prm.st, SITE_KV_EMPTY);
                };
                auto copy = [&](int i, int j, bool v_tile, uint32_t bar) {  // tile of key tile j -> slot of load i
                    const int slot = i % T::KV_SLOTS;
                    const CUtensorMap* map = v_tile ? &tm_v : &tm_k;
                    for (int blk = 0; blk < T::NBLK; ++blk) {
                        const uint32_t dst = smem_u32(sKV + slot * T::TILE_BYTES + blk * T::BLK_BYTES);
                        if (dbg_tma(dst, blk * T::BLK_ELEMS, (it.kv_lo + j) * kTile, it.hk_idx, it.b_idx, D, N,
                                    prm.Hk, prm.BH / prm.H, T::EB, 0x1D1))
                            tma_load_4d(dst, map, bar, blk * T::BLK_ELEMS, (it.kv_lo + j) * kTile, it.hk_idx,
                                        it.b_idx);
                    }
                };
                auto load_single = [&](int j, bool v_tile) -> bool {
                    if (!claim(idx)) return false;
                    const uint32_t bar = b_kv_full(idx % T::KV_SLOTS);
                    mbar_arrive_expect_tx(bar, T::TILE_BYTES);
                    copy(idx, j, v_tile, bar);
                    ++idx;
                    return true;
                };
                auto load_v_k = [&](int j) -> bool {  // j >= 1: V_j, and K_{j+1} if the item has it
                    const bool k_next = j + 1 < it.n_kv;
                    if (!claim(idx) || (k_next && !claim(idx + 1))) return false;
                    const uint32_t bar = b_kv_full(idx % T::KV_SLOTS);
                    mbar_arrive_expect_tx(bar, (k_next ? 2 : 1) * T::TILE_BYTES);
                    copy(idx, j, true, bar);
                    if (k_next) {
                        mbar_arrive(b_kv_full((idx + 1) % T::KV_SLOTS));
                        copy(idx + 1, j + 1, false, bar);
                    }
                    idx += k_next ? 2 : 1;
                    return true;
                };
                // The item's first key tile goes out while the previous item finishes;
                // its Q tiles once the previous item's products that read Q are done.
                if (it.n_kv > 0 && !(load_single(0, false) && load_single(0, true))) {
                    ok = false;
                    break;
                }
                if (k > 0 && !wait_one(b_q_empty, (k - 1) & 1, abort_flag, prm.st, SITE_Q_EMPTY)) {
                    ok = false;
                    break;
                }
                const int q_tiles = (it.n0 > 0) + (it.n1 > 0);
                mbar_arrive_expect_tx(b_q, q_tiles * T::TILE_BYTES);
                for (int g = 0; g < 2; ++g) {
                    if (it.n(g) == 0) continue;
                    for (int blk = 0; blk < T::NBLK; ++blk) {
                        const uint32_t dst = smem_u32(sQ + g * T::TILE_BYTES + blk * T::BLK_BYTES);
                        if (dbg_tma(dst, blk * T::BLK_ELEMS, (2 * it.pair + g) * kTile, it.h_idx, it.b_idx, D,
                                    N, prm.H, prm.BH / prm.H, T::EB, 0x1D2))
                            tma_load_4d(dst, &tm_q, b_q, blk * T::BLK_ELEMS, (2 * it.pair + g) * kTile,
                                        it.h_idx, it.b_idx);
                    }
                }
                if (it.n_kv > 1) ok = load_single(1, false);
                for (int j = 1; j < it.n_kv && ok; ++j) ok = load_v_k(j);
                ++k;
            }
            // Let every copy this thread started land before the CTA can exit.
            if (k > 0) wait_drain(b_q, (k - 1) & 1, prm.st, SITE_DRAIN);
            const int first = idx > T::KV_SLOTS ? idx - T::KV_SLOTS : 0;
            for (int i = first; i < idx; ++i)
                wait_drain(b_kv_full(i % T::KV_SLOTS), (i / T::KV_SLOTS) & 1, prm.st, SITE_DRAIN);
        }
    } else if (warp == 9) {
        // ================= MMA issuer =================
        // The whole warp walks the schedule (uniform control flow and operands);
        // one elected lane issues each tcgen05 instruction.
        __syncwarp();
        {
            const uint32_t sq_base = smem_u32(sQ);
            const uint32_t skv_base = smem_u32(sKV);
            Item it{};        // the item being issued
            int ring = 0;     // ring position of the item's first K tile (K/V loads before it)
            int pdone0 = 0, pdone1 = 0;  // P tiles of query tile 0 / 1 consumed in earlier items
            // Descriptors as words: per instruction only a constant is added to the low word.
            const SmemDesc dq0 = sw128_desc_words(sq_base, 16, 1024);              // Q, K-major
            const SmemDesc dk0 = sw128_desc_words(skv_base, 16, 1024);             // K tiles, K-major
            const SmemDesc dv0 = sw128_desc_words(skv_base, T::BLK_BYTES, 1024);   // V tiles, MN-major
            auto slot_desc = [&](SmemDesc base, int idx) {
                return desc_add(base, static_cast<uint32_t>((idx % T::KV_SLOTS) * T::TILE_BYTES));
            };
            auto wait_kv = [&](int idx) {
                return wait_warp(b_kv_full(idx % T::KV_SLOTS), (idx / T::KV_SLOTS) & 1, abort_flag,
                                prm.st, SITE_KV_FULL);
            };
            // Ring index of K_j / V_j (j absolute), in the producer's load order.
            auto kidx = [&](int j) { return ring + 2 * (j - it.kv_lo); };
            // S_g = Q_g K_j^T : both operands K-major, 32 bytes of K per instruction.
            // Issued four instructions at a time: instruction kk of quad q reads the
            // 32 bytes at (4q + kk) * 32 of each row, i.e. block q, byte 32 kk.
            auto issue_s = [&](int g, int j) {
                const SmemDesc qa = desc_add(dq0, static_cast<uint32_t>(g * T::TILE_BYTES));
                const SmemDesc kb = slot_desc(dk0, kidx(j));
                constexpr int QUADS = D / T::UMMA_K / 4;
#pragma unroll
                for (int q = 0; q < QUADS; ++q)
                    mma_ss_warp4<FP8, 0, 2, 4, 6, 0, 2, 4, 6>(
                        tmem + (g ? T::COL_S1 : T::COL_S0), desc_add(qa, q * T::BLK_BYTES),
                        desc_add(kb, q * T::BLK_BYTES), T::IDESC_S, q > 0 ? 1u : 0u);
                mma_commit_warp(b_s_full + 8u * g);
            };
            // O_g += P_g V_j : P from tensor memory, V MN-major (rows = keys).
            // Instruction kk reads P columns 8 kk.. and V rows UMMA_K kk.. (UMMA_K
            // 128-byte rows each); four per quad.
            auto issue_pv = [&](int g, int j, bool first) {
                const SmemDesc vb = slot_desc(dv0, kidx(j) + 1);
                constexpr int QUADS = kTile / T::UMMA_K / 4;
                constexpr uint32_t VS = T::UMMA_K * 8;  // V rows of one instruction, 16-byte units
#pragma unroll
                for (int q = 0; q < QUADS; ++q)
                    mma_ts_warp4<FP8, 0, 8, 16, 24, 0, VS, 2 * VS, 3 * VS>(
                        tmem + (g ? T::COL_O1 : T::COL_O0), tmem + (g ? T::COL_S1 : T::COL_S0) + 32 * q,
                        desc_add(vb, static_cast<uint32_t>(4 * q * T::UMMA_K * 128)), T::IDESC_PV,
                        (!first || q > 0) ? 1u : 0u);
            };
            // P_g of the item's key tile j (relative to the tile's first) is ready
            auto wait_p = [&](int g, int jrel) {
                return wait_warp(b_p_full + 8u * g, ((g ? pdone1 : pdone0) + jrel) & 1, abort_flag, prm.st,
                                 SITE_P_FULL);
            };
            auto active = [&](int g, int j) {
                return it.n(g) > 0 && j >= it.lo(g) && j < it.lo(g) + it.n(g);
            };
            // Both query tiles start at kv_lo (no mask, causal, split): the tiles
            // differ only in where they stop, and the loop runs on relative indices.
            bool q_released = false;  // the item's q_empty commit has been made
            auto run_aligned = [&]() -> bool {
                const int kv_lo = it.kv_lo;
                const int n_max = max(it.n0, it.n1);
                if (!wait_kv(kidx(kv_lo))) return false;
                tc_fence_after();
                if (it.n(0) > 0) issue_s(0, kv_lo);
                if (it.n(1) > 0) issue_s(1, kv_lo);
                if (n_max == 1) {  // no further product reads Q
                    mma_commit_warp(b_q_empty);
                    q_released = true;
                }
                mma_commit_warp(b_kv_empty(kidx(kv_lo) % T::KV_SLOTS));
                for (int j = 0; j < it.n_kv; ++j) {
                    bool v_ready = false, k_next_ready = false;
                    if (j < it.n(0)) {
                        // V_j (and K_{j+1}) first: they have usually landed long before,
                        // and checking them while P_0(j) is still being formed keeps the
                        // check off the path from P_0(j) to PV_0(j)
                        if (!wait_kv(kidx(kv_lo + j) + 1)) return false;
                        if (!wait_p(0, j)) return false;
                        v_ready = true;
                        tc_fence_after();
                        issue_pv(0, kv_lo + j, j == 0);
                        if (j + 1 < it.n(0)) {  // K_{j+1} landed with V_j (K_1: on its own)
                            if (j == 0 && !wait_kv(kidx(kv_lo + 1))) return false;
                            k_next_ready = true;
                            tc_fence_after();
                            issue_s(0, kv_lo + j + 1);
                        } else {
                            mma_commit_warp(b_o_full);
                        }
                    }
                    if (j < it.n(1)) {
                        if (!wait_p(1, j)) return false;
                        if (!v_ready && !wait_kv(kidx(kv_lo + j) + 1)) return false;
                        tc_fence_after();
                        issue_pv(1, kv_lo + j, j == 0);
                    }
                    if (j < it.n(1)) {
                        if (j + 1 < it.n(1)) {  // K_{j+1} landed with V_j (K_1: on its own)
                            if (!k_next_ready && !(v_ready && j > 0) &&
                                !wait_kv(j == 0 ? kidx(kv_lo + 1) : kidx(kv_lo + j) + 1))
                                return false;
                            tc_fence_after();
                            issue_s(1, kv_lo + j + 1);
                        } else {
                            mma_commit_warp(b_o_full + 8u);
                        }
                    }
                    // V_j consumed (released after S_1(j+1) is issued, which then follows
                    // PV_1(j) without a commit in between)
                    mma_commit_warp(b_kv_empty((kidx(kv_lo + j) + 1) % T::KV_SLOTS));
                    if (j + 2 == n_max) {  // the item's last S products have just been issued
                        mma_commit_warp(b_q_empty);
                        q_released = true;
                    }
                    if (j + 1 < it.n_kv)
                        mma_commit_warp(b_kv_empty(kidx(kv_lo + j + 1) % T::KV_SLOTS));  // K_{j+1}
                }
                return true;
            };
            auto run_general = [&]() -> bool {
                const int kv_lo = it.kv_lo, n_kv = it.n_kv;
                if (!wait_kv(kidx(kv_lo))) return false;
                tc_fence_after();
                if (active(0, kv_lo)) issue_s(0, kv_lo);
                if (active(1, kv_lo)) issue_s(1, kv_lo);
                mma_commit_warp(b_kv_empty(kidx(kv_lo) % T::KV_SLOTS));
                for (int j = kv_lo; j < kv_lo + n_kv; ++j) {
                    const bool has_next = j + 1 < kv_lo + n_kv;
                    bool v_ready = false, k_next_ready = false;
                    auto need_k_next = [&]() -> bool {  // K_{j+1} lands with V_j (K_1: on its own)
                        if (k_next_ready || (v_ready && j > kv_lo)) return true;
                        if (!wait_kv(j == kv_lo ? kidx(kv_lo + 1) : kidx(j) + 1)) return false;
                        k_next_ready = true;
                        return true;
                    };
                    // query tile 0: PV_0(j), then S_0(j+1)
                    if (active(0, j)) {
                        if (!wait_kv(kidx(j) + 1)) return false;  // before P_0(j), as above
                        if (!wait_p(0, j - it.lo(0))) return false;
                        v_ready = true;
                        tc_fence_after();
                        issue_pv(0, j, j == it.lo(0));
                        if (active(0, j + 1)) {
                            if (!need_k_next()) return false;
                            tc_fence_after();
                            issue_s(0, j + 1);
                        } else {
                            mma_commit_warp(b_o_full);
                        }
                    } else if (active(0, j + 1)) {
                        if (!need_k_next()) return false;
                        tc_fence_after();
                        issue_s(0, j + 1);
                    }
                    // query tile 1: PV_1(j), release V_j, then S_1(j+1)
                    if (active(1, j)) {
                        if (!wait_p(1, j - it.lo(1))) return false;
                        if (!v_ready && !wait_kv(kidx(j) + 1)) return false;
                        v_ready = true;
                        tc_fence_after();
                        issue_pv(1, j, j == it.lo(1));
                    }
                    if (!v_ready && !wait_kv(kidx(j) + 1)) return false;  // loaded, never used
                    if (active(1, j)) {
                        if (active(1, j + 1)) {
                            if (!need_k_next()) return false;
                            tc_fence_after();
                            issue_s(1, j + 1);
                        } else {
                            mma_commit_warp(b_o_full + 8u);
                        }
                    } else if (active(1, j + 1)) {
                        if (!need_k_next()) return false;
                        tc_fence_after();
                        issue_s(1, j + 1);
                    }
                    // V_j consumed (released after S_1(j+1) is issued, which then
                    // follows PV_1(j) without a commit in between)
                    mma_commit_warp(b_kv_empty((kidx(j) + 1) % T::KV_SLOTS));
                    if (has_next) {
                        if (!need_k_next()) return false;
                        mma_commit_warp(b_kv_empty(kidx(j + 1) % T::KV_SLOTS));  // K_{j+1} consumed
                    }
                }
                return true;
            };
            int k = 0;  // items issued
            for (int r = 0;; ++r) {
                const int item = item_at(r);
                if (item == -1) break;
                if (item < 0) continue;
                it = item_info(item);
                q_released = false;
                if (!wait_warp(b_q, k & 1, abort_flag, prm.st, SITE_Q)) break;
                if (it.n_kv > 0) {
                    const bool aligned = (it.n(0) == 0 || it.lo(0) == it.kv_lo) &&
                                         (it.n(1) == 0 || it.lo(1) == it.kv_lo);
                    if (!(aligned ? run_aligned() : run_general())) break;
                }
                // Every product of this item that reads Q has been issued; once they are
                // done the producer may load the next item's Q tiles.
                if (!q_released) mma_commit_warp(b_q_empty);
                ring += 2 * it.n_kv;
                pdone0 += it.n0;
                pdone1 += it.n1;
                ++k;
            }
            // Every MMA issued above must finish before tensor memory is freed.
            mma_commit_warp(b_done);
            wait_drain(b_done, 0, prm.st, SITE_DRAIN);
        }
    } else {
        // ================= softmax warpgroups =================
        const int g = warp >> 2;         // query tile of this warpgroup
        const int wq = warp & 3;         // lane quarter of tensor memory
        const int row = wq * 32 + lane;  // row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + (g ? T::COL_S1 : T::COL_S0) + lane_off;
        const uint32_t tO = tmem + (g ? T::COL_O1 : T::COL_O0) + lane_off;
        const uint32_t b_sf = b_s_full + 8u * g, b_pf = b_p_full + 8u * g, b_of = b_o_full + 8u * g;
        const float cs = prm.cs;
        int s_seen = 0;  // S tiles of this query tile consumed in earlier items
        int o_seen = 0;  // outputs of this query tile written in earlier items
        bool ok = true;
        for (int r = 0; ok; ++r) {
        const int item = item_at(r);
        if (item == -1) break;
        if (item < 0) continue;
        const Item it = item_info(item);
        const int bh = it.bh, split = it.split, b_idx = it.b_idx, h_idx = it.h_idx;
        const int q_row = (2 * it.pair + g) * kTile + row;
        const int n = it.n(g);
        const int jt0 = it.lo(g);  // first key tile of this query tile
        // keys [key_min, key_max] are visible to this row
        const int key_min = prm.win_left < 0 ? 0 : q_row - prm.win_left;
        const int key_max = prm.win_right < 0 ? N - 1 : min(N - 1, q_row + prm.win_right);

        float m_used = -INFINITY;  // running max in log2 units of the scaled scores
        float l_sum = 0.f;         // running sum of 2^(s*cs - m_used), unrounded (for LSE)
        float l_pv = 0.f;          // the same sum over the rounded P that multiplies V
        for (int j = 0; j < n; ++j) {
            if (!wait_warp(b_sf, (s_seen + j) & 1, abort_flag, prm.st, SITE_S_FULL)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t s[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, s[c]);
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_wait(s[c]);

            const int kv0 = (jt0 + j) * kTile;
            const int c_lo = key_min - kv0, c_hi = key_max - kv0;  // visible columns [c_lo, c_hi]
            auto apply_mask = [&]() {
                if (c_lo > 0 || c_hi < kTile - 1) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (c * 32 + i < c_lo || c * 32 + i > c_hi) s[c][i] = f2u(-INFINITY);
                }
            };
            apply_mask();
            // Running maximum m_used (log2 units).  A tile maximum is computed only while
            // m_used is still -inf; later tiles are exponentiated against m_used, so P
            // may exceed 1.  A tile is redone with its own maximum when its row sum
            // passes a bound: 448 for FP8 (every P of the tile is at most the sum, and
            // E4M3 stops at 448), 2^60 for bf16 (a bf16 value keeps its relative
            // precision at any magnitude; the bound keeps P, O and the sums far inside
            // fp32).  m_used is raised when the tile maximum exceeds it by more than tau.
            float alpha = 1.f;
            bool rescale_o = false;
            auto update_max = [&](float tau) {
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = u2f(s[0][i]);
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = (c == 0 ? 8 : 0); i < 32; i += 2)
                        mx8[(i >> 1) & 7] = fmax3(mx8[(i >> 1) & 7], u2f(s[c][i]), u2f(s[c][i + 1]));
                const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7]));
                const float mx_s = mx * cs;
                if (mx_s > m_used + tau) {
                    alpha = ex2_approx(m_used - mx_s);  // 0 when m_used is still -inf
                    l_sum *= alpha;
                    l_pv *= alpha;
                    m_used = mx_s;
                    rescale_o = (j > 0);
                }
            };
            if (__any_sync(0xffffffffu, m_used == -INFINITY)) update_max(kRescaleThreshold);

            // P is kept in registers until the tile is accepted: its bf16 words would
            // overwrite the S columns, which a redo reads again.
            float ls[4], lr[4];
            uint32_t pk0[32], pk1[32];  // packed P: FP8 all 128 keys in pk0; bf16 keys 0-63, 64-127
            auto exp_pass = [&]() {
                const float m_sub = (m_used == -INFINITY) ? 0.f : m_used;
#pragma unroll
                for (int e = 0; e < 4; ++e) ls[e] = lr[e] = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        float x0, x1, x2, x3;
                        ffma2(x0, x1, u2f(s[c][i]), u2f(s[c][i + 1]), cs, cs, -m_sub, -m_sub);
                        ffma2(x2, x3, u2f(s[c][i + 2]), u2f(s[c][i + 3]), cs, cs, -m_sub, -m_sub);
                        float p0, p1, p2, p3;
                        if (FMAEXP && i == kFmaExpGroup) {
                            // one group of four in eight: exponentials on the FMA pipe
                            ex2_fma2(p0, p1, x0, x1);
                            ex2_fma2(p2, p3, x2, x3);
                        } else {
                            p0 = ex2_approx(x0);
                            p1 = ex2_approx(x1);
                            p2 = ex2_approx(x2);
                            p3 = ex2_approx(x3);
                        }
                        if constexpr (FP8) {
                            pk0[c * 8 + i / 4] = pack_e4m3x4(p0, p1, p2, p3);
                        } else {
                            const uint32_t w0 = pack_bf16x2(p0, p1), w1 = pack_bf16x2(p2, p3);
                            // The O normaliser sums the same bf16 values that multiply V, so
                            // O stays an exact convex combination of V rows; LSE uses the
                            // unrounded sum.
                            lr[(i >> 2) & 1] = add_bf16x2(lr[(i >> 2) & 1], w0);
                            lr[2 + ((i >> 2) & 1)] = add_bf16x2(lr[2 + ((i >> 2) & 1)], w1);
                            uint32_t* dst = c < 2 ? pk0 : pk1;
                            dst[(c & 1) * 16 + i / 2] = w0;
                            dst[(c & 1) * 16 + i / 2 + 1] = w1;
                        }
                        float a0, a1;
                        fadd2(a0, a1, p0, p1, p2, p3);
                        fadd2(ls[(i >> 2) & 1], ls[2 + ((i >> 2) & 1)], ls[(i >> 2) & 1],
                              ls[2 + ((i >> 2) & 1)], a0, a1);
                    }
            };
            exp_pass();
            {
                const float tile_sum = (ls[0] + ls[1]) + (ls[2] + ls[3]);
                if (__any_sync(0xffffffffu, !(tile_sum <= (FP8 ? kRedoBoundFP8 : kRedoBound)))) {
                    // the scores of this tile rose above m_used: redo it with its maximum
                    // (S is still in tensor memory: no P has been stored)
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, s[c]);
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld_wait(s[c]);
                    apply_mask();
                    update_max(0.f);
                    exp_pass();
                }
            }
            tmem_st32(tS, pk0);
            if constexpr (!FP8) tmem_st32(tS + 32, pk1);
            l_sum += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            l_pv += (lr[0] + lr[1]) + (lr[2] + lr[3]);
            if (__any_sync(0xffffffffu, rescale_o)) {
                // Rescale this warp's 32 output rows (alpha = 1 on rows that kept their max).
                // PV_g(j-1) has completed: S_g(j) was committed after it, and PV_g(j)
                // is issued only after this warp arrives on p_full below.  Done after
                // the S row has been consumed so that S and O are never live together.
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * c, o);
                    tmem_ld_wait(o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
                    tmem_st32(tO + 32 * c, o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_pf);
        }

        if (split_mode && ok && n == 0 && q_row < N) {
            // this split holds no key visible to the tile: an empty partial
            float4* op = reinterpret_cast<float4*>(
                prm.o_part + ((static_cast<size_t>(split) * prm.BH + bh) * N + q_row) * D);
#pragma unroll
            for (int c = 0; c < D / 4; ++c) op[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            prm.lse_part[(static_cast<size_t>(split) * prm.BH + bh) * N + q_row] = -INFINITY;
        }
        s_seen += n;
        const bool o_ready = ok && n > 0 && wait_warp(b_of, o_seen & 1, abort_flag, prm.st, SITE_O_FULL);
        if (n > 0) {
            ++o_seen;
            if (!o_ready) ok = false;
        }
        if (o_ready && split_mode) {
            // fp32 partial for the combine kernel: O over this split's keys, and its LSE
            tc_fence_after();
            const bool row_ok = q_row < N;
            const float l_norm = FP8 ? l_sum : l_pv;
            const float inv_l = l_norm > 0.f ? prm.out_scale / l_norm : 0.f;
            float* op = prm.o_part + ((static_cast<size_t>(split) * prm.BH + bh) * N +
                                      (row_ok ? q_row : 0)) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + 32 * c, o);
                tmem_ld_wait(o);
                if (row_ok) {
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        reinterpret_cast<float4*>(op + c * 32)[v] =
                            make_float4(u2f(o[4 * v]) * inv_l, u2f(o[4 * v + 1]) * inv_l,
                                        u2f(o[4 * v + 2]) * inv_l, u2f(o[4 * v + 3]) * inv_l);
                }
            }
            if (row_ok)
                prm.lse_part[(static_cast<size_t>(split) * prm.BH + bh) * N + q_row] =
                    l_sum > 0.f ? (m_used + log2f(l_sum)) * kLn2 : -INFINITY;
        } else if (o_ready) {
            tc_fence_after();
            const bool row_ok = q_row < N;
            const float l_norm = FP8 ? l_sum : l_pv;
            const float inv_l = l_norm > 0.f ? prm.out_scale / l_norm : 0.f;
            uint8_t* orow = static_cast<uint8_t*>(prm.o) +
                            (b_idx * prm.os.b + h_idx * prm.os.h + (row_ok ? q_row : 0) * prm.os.n) * 2;
            // one copy of the loop per store width, so that each keeps its own
            // register layout
            auto write_rows = [&](auto v8_tag) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * c, o);
                    tmem_ld_wait(o);
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_bf16x2(u2f(o[2 * i]) * inv_l, u2f(o[2 * i + 1]) * inv_l);
                    if (row_ok) st_global_row64<decltype(v8_tag)::value>(orow + c * 64, pk);
                }
            };
            if (prm.o_v8)
                write_rows(std::true_type{});
            else
                write_rows(std::false_type{});
            if (row_ok)
                prm.lse[static_cast<size_t>(bh) * N + q_row] =
                    l_sum > 0.f ? (m_used + log2f(l_sum)) * kLn2 : INFINITY;
        }
        }  // items
    }

    // ---- teardown: all tensor-memory traffic of this CTA is complete ----
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Merge of split-KV partials, one warp per (head, row): with m = max_s LSE_s
// and w_s = exp(LSE_s - m), O = sum_s w_s O_s / sum_s w_s and
// LSE = m + ln(sum_s w_s) -- the running-max / running-sum combination of the
// FlashAttention digest (section 2) applied to whole partial results.
__global__ void __launch_bounds__(256) splitkv_combine_kernel(const CombineParams p) {
    const int lane = threadIdx.x & 31;
    const long long rows = static_cast<long long>(p.BH) * p.N;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const int epl = p.D / 32;  // elements per lane: 2 or 4
    for (long long r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        float m = -INFINITY;
        for (int sp = 0; sp < p.S; ++sp) m = fmaxf(m, p.lse_part[sp * rows + r]);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        float wsum = 0.f;
        if (m != -INFINITY) {
            for (int sp = 0; sp < p.S; ++sp) {
                const float w = expf(p.lse_part[sp * rows + r] - m);
                wsum += w;
                const float* src = p.o_part + (sp * rows + r) * p.D + lane * epl;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (e < epl) acc[e] += w * src[e];
            }
        }
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
        const long long bh = r / p.N, n = r % p.N;
        uint16_t* dst = static_cast<uint16_t*>(p.o) + (bh / p.H) * p.os.b + (bh % p.H) * p.os.h +
                        n * p.os.n + lane * epl;
        if (epl == 4) {
            const uint32_t w0 = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            const uint32_t w1 = pack_bf16x2(acc[2] * inv, acc[3] * inv);
            *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
        } else {
            *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        }
        if (lane == 0) p.lse[r] = wsum > 0.f ? m + logf(wsum) : INFINITY;
    }
}

template <int D, bool FP8, bool FMAEXP = false>
cudaError_t launch_fwd_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, cudaStream_t stream) {
    using T = FwdTraits<D, FP8>;
    static const cudaError_t attr = cudaFuncSetAttribute(
        fwd_kernel<D, FP8, FMAEXP>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
    if (attr != cudaSuccess) return attr;
    // Persistent CTAs, one per SM (shared memory admits one), each looping over
    // items in the snake order of item_at: equal items (no mask) and longest-first
    // causal items alike end within about one item of each other.
    FwdParams pp = p;
    pp.single = 0;
    long long items = static_cast<long long>(p.BH) * p.n_pairs * p.n_splits;
    long long grid = items;
    {
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (p.n_splits == 1 && 2 * items <= sms) {  // single query tiles: twice the CTAs
            pp.single = 1;
            items = static_cast<long long>(p.BH) * ((p.N + kTile - 1) / kTile);
            grid = items;
        }
        if (sms < grid) grid = sms;
    }
    if (grid < 1) return cudaSuccess;
    const cudaError_t dbg = dbg_set_word(p.st.word, stream);
    if (dbg != cudaSuccess) return dbg;
    fwd_kernel<D, FP8, FMAEXP><<<static_cast<unsigned>(grid), 320, T::SMEM_BYTES, stream>>>(tq, tk, tv, pp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const FwdParams& p, cudaStream_t stream) {
    if (D == 64) return launch_fwd_impl<64, false>(tq, tk, tv, p, stream);
    if (D == 128) return launch_fwd_impl<128, false>(tq, tk, tv, p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_fp8(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const FwdParams& p, cudaStream_t stream) {
    if (D == 128)
        return p.exp2_offload ? launch_fwd_impl<128, true, true>(tq, tk, tv, p, stream)
                              : launch_fwd_impl<128, true>(tq, tk, tv, p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_splitkv_combine(const CombineParams& p, cudaStream_t stream) {
    // One warp per row, eight rows per block; at most 16 blocks per SM (of the
    // device the launch goes to), the warps striding over the remaining rows.
    const long long rows = static_cast<long long>(p.BH) * p.N;
    const long long blocks = (rows + 7) / 8;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long cap = 16ll * sms;
    const int grid = static_cast<int>(blocks < cap ? blocks : cap);
    if (grid < 1) return cudaSuccess;
    splitkv_combine_kernel<<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

int fwd_smem_bytes(int D, bool fp8) {
    if (fp8) return D == 128 ? FwdTraits<128, true>::SMEM_BYTES : 0;
    if (D == 64) return FwdTraits<64, false>::SMEM_BYTES;
    if (D == 128) return FwdTraits<128, false>::SMEM_BYTES;
    return 0;
}

}  // namespace attn
