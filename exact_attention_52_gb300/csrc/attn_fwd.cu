// Forward exact attention on sm_103a: O = softmax(scale * Q K^T [+ causal mask]) V
// and the per-row natural log-sum-exp, computed tile by tile with the online
// softmax so that S and P never leave the SM (FlashAttention digest, sections
// 1-2; FlashAttention paper item 58: running max, running sum, and the same
// rescale applied to the output accumulator).
//
// One CTA owns two 128-row query tiles of one (batch, head) and streams the
// key/value tiles of that head through a shared-memory ring:
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
// The output rescale is lazy: a row's running max m_used is raised only when
// the tile max exceeds it by more than 2^8 (log2 units), so P <= 256 and O,
// l share the same stale max, which keeps the result exact ("conditional
// rescaling" in the FlashAttention-3 walkthrough tags).
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;

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
    // barriers: q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], o_full[2], mma_done
    static constexpr int NBARS = 1 + 2 * KV_SLOTS + 2 + 2 + 2 + 1;
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
    SITE_S_FULL = 0x105, SITE_O_FULL = 0x106, SITE_DRAIN = 0x107,
};

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

template <int D, bool FP8>
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

    if ((smem_u32(smem) & 1023u) != 0) {  // swizzle atoms need 1024-byte alignment
        if (threadIdx.x == 0) record_device_error(prm.st, ATTN_DEVERR_SMEM_ALIGN, 0x1FF);
        return;
    }

    // ---- work assignment ----
    // Non-causal: head-major order, so the CTAs resident at any time cover
    // only a few heads and each head's K and V come from HBM about once.
    // Causal: heaviest query tiles of every head first (longest-first keeps
    // the tail of the launch short; a causal head needs half the K/V reuse).
    const int bh = prm.causal ? static_cast<int>(blockIdx.x % prm.BH)
                              : static_cast<int>(blockIdx.x / prm.n_pairs);
    const int pair = prm.n_pairs - 1 -
                     (prm.causal ? static_cast<int>(blockIdx.x / prm.BH)
                                 : static_cast<int>(blockIdx.x % prm.n_pairs));
    const int N = prm.N;
    const int n_kv_total = (N + kTile - 1) / kTile;
    int n_t[2];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const int qt = 2 * pair + g;
        n_t[g] = (qt * kTile >= N) ? 0 : (prm.causal ? min(n_kv_total, qt + 1) : n_kv_total);
    }
    const int n_kv = max(n_t[0], n_t[1]);
    // Key/value head of this query head (grouped-query attention: H/Hk query
    // heads share one key/value head; Hk == H is ordinary multi-head attention).
    const int kv_bh = (bh / prm.H) * prm.Hk + (bh % prm.H) / (prm.H / prm.Hk);

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
            const int q_tiles = (n_t[0] > 0) + (n_t[1] > 0);
            mbar_arrive_expect_tx(b_q, q_tiles * T::TILE_BYTES);
            for (int g = 0; g < 2; ++g) {
                if (n_t[g] == 0) continue;
                for (int blk = 0; blk < T::NBLK; ++blk)
                    tma_load_3d(smem_u32(sQ + g * T::TILE_BYTES + blk * T::BLK_BYTES), &tm_q, b_q,
                                blk * T::BLK_ELEMS, (2 * pair + g) * kTile, bh);
            }
            int idx = 0;
            bool ok = true;
            for (int j = 0; j < n_kv && ok; ++j) {
                for (int t = 0; t < 2; ++t, ++idx) {  // t = 0: K_j, t = 1: V_j
                    const int slot = idx % T::KV_SLOTS;
                    const int round = idx / T::KV_SLOTS;
                    if (round > 0 &&
                        !wait_one(b_kv_empty(slot), (round - 1) & 1, abort_flag, prm.st,
                                  SITE_KV_EMPTY)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(b_kv_full(slot), T::TILE_BYTES);
                    const CUtensorMap* map = t ? &tm_v : &tm_k;
                    for (int blk = 0; blk < T::NBLK; ++blk)
                        tma_load_3d(smem_u32(sKV + slot * T::TILE_BYTES + blk * T::BLK_BYTES), map,
                                    b_kv_full(slot), blk * T::BLK_ELEMS, j * kTile, kv_bh);
                }
            }
            // Let every copy this thread started land before the CTA can exit.
            wait_drain(b_q, 0, prm.st, SITE_DRAIN);
            const int first = idx > T::KV_SLOTS ? idx - T::KV_SLOTS : 0;
            for (int i = first; i < idx; ++i)
                wait_drain(b_kv_full(i % T::KV_SLOTS), (i / T::KV_SLOTS) & 1, prm.st, SITE_DRAIN);
        }
    } else if (warp == 9) {
        // ================= MMA issuer =================
        if (lane == 0) {
            const uint32_t sq_base = smem_u32(sQ);
            const uint32_t skv_base = smem_u32(sKV);
            auto slot_addr = [&](int idx) {
                return skv_base + static_cast<uint32_t>((idx % T::KV_SLOTS) * T::TILE_BYTES);
            };
            auto wait_kv = [&](int idx) {
                return wait_one(b_kv_full(idx % T::KV_SLOTS), (idx / T::KV_SLOTS) & 1, abort_flag,
                                prm.st, SITE_KV_FULL);
            };
            // S_g = Q_g K_j^T : both operands K-major, 32 bytes of K per instruction.
            auto issue_s = [&](int g, int j) {
                const uint32_t qa = sq_base + g * T::TILE_BYTES;
                const uint32_t kb = slot_addr(2 * j);
#pragma unroll
                for (int kk = 0; kk < D / T::UMMA_K; ++kk) {
                    const uint32_t off = (kk * 32) / 128 * T::BLK_BYTES + (kk * 32) % 128;
                    mma_ss<FP8>(tmem + (g ? T::COL_S1 : T::COL_S0), sw128_desc(qa + off, 16, 1024), sw128_desc(kb + off, 16, 1024),
                                T::IDESC_S, kk > 0 ? 1u : 0u);
                }
                mma_commit(b_s_full + 8u * g);
            };
            // O_g += P_g V_j : P from tensor memory, V MN-major (rows = keys).
            auto issue_pv = [&](int g, int j) {
                const uint32_t vb = slot_addr(2 * j + 1);
#pragma unroll
                for (int kk = 0; kk < kTile / T::UMMA_K; ++kk) {
                    mma_ts<FP8>(tmem + (g ? T::COL_O1 : T::COL_O0),
                                tmem + (g ? T::COL_S1 : T::COL_S0) + kk * 8,
                                sw128_desc(vb + kk * T::UMMA_K * 128, T::BLK_BYTES, 1024), T::IDESC_PV,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            auto run = [&]() -> bool {
                if (!wait_one(b_q, 0, abort_flag, prm.st, SITE_Q)) return false;
                if (!wait_kv(0)) return false;
                tc_fence_after();
                if (n_t[0] > 0) issue_s(0, 0);
                if (n_t[1] > 0) issue_s(1, 0);
                mma_commit(b_kv_empty(0));
                for (int j = 0; j < n_kv; ++j) {
                    bool v_ready = false, k_next_ready = false;
                    if (j < n_t[0]) {
                        if (!wait_one(b_p_full, j & 1, abort_flag, prm.st, SITE_P_FULL)) return false;
                        if (!wait_kv(2 * j + 1)) return false;
                        v_ready = true;
                        tc_fence_after();
                        issue_pv(0, j);
                        if (j + 1 < n_t[0]) {
                            if (!wait_kv(2 * j + 2)) return false;
                            k_next_ready = true;
                            tc_fence_after();
                            issue_s(0, j + 1);
                        } else {
                            mma_commit(b_o_full);
                        }
                    }
                    if (j < n_t[1]) {
                        if (!wait_one(b_p_full + 8u, j & 1, abort_flag, prm.st, SITE_P_FULL))
                            return false;
                        if (!v_ready && !wait_kv(2 * j + 1)) return false;
                        tc_fence_after();
                        issue_pv(1, j);
                    }
                    mma_commit(b_kv_empty((2 * j + 1) % T::KV_SLOTS));  // V_j consumed
                    if (j < n_t[1]) {
                        if (j + 1 < n_t[1]) {
                            if (!k_next_ready && !wait_kv(2 * j + 2)) return false;
                            tc_fence_after();
                            issue_s(1, j + 1);
                        } else {
                            mma_commit(b_o_full + 8u);
                        }
                    }
                    if (j + 1 < n_kv) mma_commit(b_kv_empty((2 * j + 2) % T::KV_SLOTS));  // K_{j+1}
                }
                return true;
            };
            run();
            // Every MMA issued above must finish before tensor memory is freed.
            mma_commit(b_done);
            wait_drain(b_done, 0, prm.st, SITE_DRAIN);
        }
    } else {
        // ================= softmax warpgroups =================
        const int g = warp >> 2;         // query tile of this warpgroup
        const int wq = warp & 3;         // lane quarter of tensor memory
        const int row = wq * 32 + lane;  // row within the tile
        const int q_row = (2 * pair + g) * kTile + row;
        const int n = g ? n_t[1] : n_t[0];
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + (g ? T::COL_S1 : T::COL_S0) + lane_off;
        const uint32_t tO = tmem + (g ? T::COL_O1 : T::COL_O0) + lane_off;
        const uint32_t b_sf = b_s_full + 8u * g, b_pf = b_p_full + 8u * g, b_of = b_o_full + 8u * g;
        const float cs = prm.cs;
        const int row_limit = prm.causal ? min(N, q_row + 1) : N;  // keys [0, row_limit) visible

        float m_used = -INFINITY;  // running max in log2 units of the scaled scores
        float l_sum = 0.f;         // running sum of 2^(s*cs - m_used), unrounded (for LSE)
        float l_pv = 0.f;          // the same sum over the rounded P that multiplies V
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            if (!wait_warp(b_sf, j & 1, abort_flag, prm.st, SITE_S_FULL)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t s[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, s[c]);
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_wait(s[c]);

            const int lim = row_limit - j * kTile;  // columns >= lim are masked
            if (lim < kTile) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (c * 32 + i >= lim) s[c][i] = f2u(-INFINITY);
            }
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

            float alpha = 1.f;
            bool rescale_o = false;
            if (mx_s > m_used + kRescaleThreshold) {
                alpha = ex2_approx(m_used - mx_s);  // 0 when m_used is still -inf
                l_sum *= alpha;
                l_pv *= alpha;
                m_used = mx_s;
                rescale_o = (j > 0);
            }
            const float m_sub = (m_used == -INFINITY) ? 0.f : m_used;

            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            float lr[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (FP8) {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float p0 = ex2_approx(fmaf(u2f(s[c][i + 0]), cs, -m_sub));
                        const float p1 = ex2_approx(fmaf(u2f(s[c][i + 1]), cs, -m_sub));
                        const float p2 = ex2_approx(fmaf(u2f(s[c][i + 2]), cs, -m_sub));
                        const float p3 = ex2_approx(fmaf(u2f(s[c][i + 3]), cs, -m_sub));
                        ls[0] += p0;
                        ls[1] += p1;
                        ls[2] += p2;
                        ls[3] += p3;
                        pk[c * 8 + i / 4] = pack_e4m3x4(p0, p1, p2, p3);
                    }
                tmem_st32(tS, pk);
            } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[32];
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int c = 2 * h + cc;
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            float x0, x1, x2, x3;
                            ffma2(x0, x1, u2f(s[c][i]), u2f(s[c][i + 1]), cs, cs, -m_sub, -m_sub);
                            ffma2(x2, x3, u2f(s[c][i + 2]), u2f(s[c][i + 3]), cs, cs, -m_sub, -m_sub);
                            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                            const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
                            const uint32_t w0 = pack_bf16x2(p0, p1), w1 = pack_bf16x2(p2, p3);
                            // The O normaliser sums the same bf16 values that multiply V, so
                            // O stays an exact convex combination of V rows; LSE uses the
                            // unrounded sum.
                            lr[(i >> 2) & 1] = add_bf16x2(lr[(i >> 2) & 1], w0);
                            lr[2 + ((i >> 2) & 1)] = add_bf16x2(lr[2 + ((i >> 2) & 1)], w1);
                            float a0, a1;
                            fadd2(a0, a1, p0, p1, p2, p3);
                            fadd2(ls[(i >> 2) & 1], ls[2 + ((i >> 2) & 1)], ls[(i >> 2) & 1],
                                  ls[2 + ((i >> 2) & 1)], a0, a1);
                            pk[cc * 16 + i / 2] = w0;
                            pk[cc * 16 + i / 2 + 1] = w1;
                        }
                    }
                    tmem_st32(tS + 32 * h, pk);
                }
            }
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

        if (ok && n > 0 && wait_warp(b_of, 0, abort_flag, prm.st, SITE_O_FULL)) {
            tc_fence_after();
            const bool row_ok = q_row < N;
            const float l_norm = FP8 ? l_sum : l_pv;
            const float inv_l = l_norm > 0.f ? prm.out_scale / l_norm : 0.f;
            uint8_t* orow = static_cast<uint8_t*>(prm.o) +
                            (static_cast<size_t>(bh) * N + (row_ok ? q_row : 0)) * D * 2;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + 32 * c, o);
                tmem_ld_wait(o);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(u2f(o[2 * i]) * inv_l, u2f(o[2 * i + 1]) * inv_l);
                if (row_ok) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        st_global_v4(orow + c * 64 + v * 16, pk[4 * v], pk[4 * v + 1], pk[4 * v + 2],
                                     pk[4 * v + 3]);
                }
            }
            if (row_ok)
                prm.lse[static_cast<size_t>(bh) * N + q_row] =
                    l_sum > 0.f ? (m_used + log2f(l_sum)) * kLn2 : INFINITY;
        }
    }

    // ---- teardown: all tensor-memory traffic of this CTA is complete ----
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool FP8>
cudaError_t launch_fwd_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, cudaStream_t stream) {
    using T = FwdTraits<D, FP8>;
    static const cudaError_t attr = cudaFuncSetAttribute(
        fwd_kernel<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
    if (attr != cudaSuccess) return attr;
    const long long grid = static_cast<long long>(p.BH) * p.n_pairs;
    fwd_kernel<D, FP8><<<static_cast<unsigned>(grid), 320, T::SMEM_BYTES, stream>>>(tq, tk, tv, p);
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
    if (D == 128) return launch_fwd_impl<128, true>(tq, tk, tv, p, stream);
    return cudaErrorInvalidValue;
}

int fwd_smem_bytes(int D, bool fp8) {
    if (fp8) return D == 128 ? FwdTraits<128, true>::SMEM_BYTES : 0;
    if (D == 64) return FwdTraits<64, false>::SMEM_BYTES;
    if (D == 128) return FwdTraits<128, false>::SMEM_BYTES;
    return 0;
}

}  // namespace attn
