// Parameter blocks and launcher entry points shared by the host-side C ABI
// (attn_api.cu) and the kernel translation units.  Internal: not installed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_device_status.cuh"

namespace attn {

constexpr int kTile = 128;  // rows of Q, K, V per tile (M and N of every MMA)

// Element strides of a [B, heads, N, d] view whose d dimension is contiguous.
struct Strides {
    long long b, h, n;
};

struct FwdParams {
    void* o;          // bf16 [B, H, N, D] with strides os
    Strides os;
    float* lse;       // fp32 [BH, N], natural log of the row normaliser
    int N;            // sequence length (queries = keys)
    int BH;           // batch * query heads
    int H, Hk;        // query heads, key/value heads (H % Hk == 0; Hk == H without grouping)
    int n_pairs;      // ceil(N / 256): CTAs per head (two 128-row Q tiles each)
    int causal;       // 1: causal mask (also selects longest-first launch order)
    int win_left;     // key j visible to query i iff i - win_left <= j <= i + win_right;
    int win_right;    // a negative bound is no bound (causal: -1, 0; full: -1, -1)
    float cs;         // scale * log2(e) (fp8: scale * s_q * s_k * log2(e))
    float out_scale;  // 1 (bf16) or s_v (fp8)
    // Split-KV mode (n_splits > 1): CTA s of a query-tile pair covers key tiles
    // [s * split_len, (s + 1) * split_len) and writes an fp32 partial result
    // (O normalised over its keys, and its log-sum-exp) instead of o and lse.
    int n_splits;
    int split_len;
    float* o_part;    // fp32 [n_splits, BH, N, D]
    float* lse_part;  // fp32 [n_splits, BH, N]; -inf where a split saw no key
    int exp2_offload; // FP8: one group of four exponentials in eight on the FMA pipe
    int single;       // items are single query tiles (set by the launcher when pairs would
                      // leave at least half of the SMs idle)
    int o_v8;         // every O row starts on a 32-byte boundary: 32-byte stores
    DevStatus st;
};

struct CombineParams {
    const float* o_part;    // fp32 [S, BH, N, D]
    const float* lse_part;  // fp32 [S, BH, N]
    void* o;                // bf16 [B, H, N, D] with strides os
    Strides os;
    float* lse;             // fp32 [BH, N]
    int S, BH, H, N, D;
};

struct BwdPreParams {
    const void* o;     // bf16 [B, H, N, D] with strides os
    const void* dout;  // bf16 [B, H, N, D] with strides dos
    Strides os, dos;
    const float* lse;  // fp32 [BH, N]
    float* dq_acc;     // fp32 [BH, Npad, D], zeroed here
    float* lse2;       // fp32 [BH, Npad]: -LSE * log2(e); -inf on padding rows
    float* dsum;       // fp32 [BH, Npad]: D_i = sum_k dO_ik O_ik; 0 on padding rows
    unsigned* split_cnt;  // arrival counters of split key tiles (see BwdParams), zeroed here
    int split_cnt_words;  // 0: none
    int N, Npad, BH, H, D;
};

// Split last round of the d = 128 backward (no mask only).  With G CTAs and
// n = R G + r items (key tiles), r > 0, the last round would leave G - r CTAs
// idle for a whole item.  Instead each of its r items is dealt as P = G / r
// parts (contiguous ranges of its query steps, P >= 2); every part leaves its
// fp32 dV and (unscaled) dK partial in the workspace, and the last part of an
// item to finish (counted per 32-row warp slice) adds the others' partials to
// its own and writes the item's dV and dK.  At most kBwdSplitCap parts.
constexpr int kBwdSplitCap = 160;
constexpr int kBwdSplitCntWords = kBwdSplitCap * 8;  // [item slot][dV, dK][4 warp slices]

struct BwdParams {
    const float* lse2;  // workspace (-LSE * log2(e)), see BwdPreParams
    const float* dsum;
    float* dq_acc;
    void* dk;           // bf16 [B, Hk, N, D] with strides dks
    void* dv;           // bf16 [B, Hk, N, D] with strides dvs
    Strides dks, dvs;
    int N, Npad;
    int BHk;            // batch * key/value heads: CTAs are (kv head, key tile)
    int H, Hk;          // query heads, key/value heads; each CTA loops over its H/Hk query heads
    int n_kv;           // ceil(N / 128): CTAs per key/value head
    int causal;         // causal mask (also selects longest-first launch order)
    int win_left;       // window bounds as in FwdParams (negative: none)
    int win_right;
    float cs;           // scale * log2(e)
    float scale;        // softmax scale (applied to dK here and to dQ at conversion)
    // Split last round (d = 128): virtual items v >= split_base are part v - split_base
    // of P = split_parts parts of item split_base + (v - split_base) / P.  Without a
    // split: split_base = number of items, split_parts = 1.
    int split_base;
    int split_parts;
    int split_cap;        // parts the workspace has room for (0: no split possible)
    float* split_part;    // fp32 [part][dV, dK][128 rows][D]
    unsigned* split_cnt;  // kBwdSplitCntWords counters, zero at launch
    int dkv_v8;           // every dK and dV row starts on a 32-byte boundary: 32-byte stores
    DevStatus st;
};

struct DqConvertParams {
    const float* dq_acc;  // fp32 [BH, Npad, D]
    void* dq;             // bf16 [B, H, N, D] with strides dqs
    Strides dqs;
    int N, Npad, BH, H, D;
    float scale;
};

// Launchers (return the launch's cudaError_t; no synchronisation).
cudaError_t launch_fwd_bf16(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const FwdParams& p, cudaStream_t stream);
cudaError_t launch_fwd_fp8(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const FwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t stream);
cudaError_t launch_splitkv_combine(const CombineParams& p, cudaStream_t stream);
cudaError_t launch_bwd_main(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                            const BwdParams& p, cudaStream_t stream);
cudaError_t launch_dq_convert(const DqConvertParams& p, cudaStream_t stream);
cudaError_t launch_wait_selftest(DevStatus st, cudaStream_t stream);

// Problem check shared by the entry points (sizes, head dim, scale, causal
// flag); returns an attn_status value (0 = valid).
int check_problem(int B, int H, int N, int d, float scale, int causal);

// The dense backward with or without the split last round of the d = 128
// kernel (without it the workspace has no room for its partials): the workspace
// size it needs, and the call (an attn_status value).
size_t bwd_workspace_bytes_for(int B, int H, int N, int d, bool split);
int bwd_dense(const void* q, const void* k, const void* v, const void* o, const void* dout,
              const float* lse, void* dq, void* dk, void* dv, void* workspace, int B, int H, int N,
              int d, float scale, int causal, bool split, cudaStream_t stream);

// Shared-memory bytes a launcher requests (for tests of the host logic).
int fwd_smem_bytes(int D, bool fp8);
int bwd_smem_bytes(int D);

}  // namespace attn
