// C ABI of libattn_sm103a.so: argument validation, TMA tensor maps, launch
// sequencing and the device error word.  The declarations and their contract
// are in include/attn_sm103a.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_sm103a.h"
#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

// Device error word: [0] error bits, [1] id of the first wait that gave up.
__device__ unsigned int g_err_word[2];

constexpr unsigned long long kDefaultWaitLimitNs = 1000000000ull;
unsigned long long g_wait_limit_ns = kDefaultWaitLimitNs;
int g_exp2_offload = 0;  // attn_set_exp2_offload

constexpr int kMaxDevices = 64;

// Architecture check, cached per device (a device's compute capability never
// changes).
struct DeviceArch {
    bool probed = false;
    bool supported = false;
};
DeviceArch g_dev[kMaxDevices];
std::mutex g_dev_mutex;

// Current device: check the architecture and look up the device address of the
// error word.  The address is looked up on every call, not cached: it belongs
// to the module loaded into the device's current context, and a context made
// after cudaDeviceReset (or another context made current on the same device)
// loads the module again, possibly at another address.  The lookup allocates
// nothing.
struct DeviceState {
    unsigned int* err = nullptr;  // device address of g_err_word in the current context
};

attn_status device_state(DeviceState* out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(g_dev_mutex);
        DeviceArch& a = g_dev[dev];
        if (!a.probed) {
            int major = 0, minor = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
                return ATTN_ERR_CUDA;
            a.supported = (major == 10 && minor == 3);
            a.probed = true;
        }
        if (!a.supported) return ATTN_ERR_UNSUPPORTED;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    out->err = static_cast<unsigned int*>(p);
    return ATTN_OK;
}

DevStatus dev_status(const DeviceState& s) {
    DevStatus st;
    st.word = s.err;
    st.wait_limit_ns = g_wait_limit_ns;
    return st;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so that the
// library has no link-time dependency on libcuda.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// 4-D view {d, N, heads, B} of a [B, heads, N, d] tensor with element strides
// s (d contiguous); box {128 bytes of d, 128 rows, 1, 1}, 128-byte swizzle,
// rows >= N read as zero.
bool make_map(CUtensorMap* m, const void* base, bool fp8, int d, int N, int heads, int B,
              const Strides& st) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t eb = fp8 ? 1 : 2;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.n) * eb, static_cast<cuuint64_t>(st.h) * eb,
                                   static_cast<cuuint64_t>(st.b) * eb};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / eb), 128u, 1u, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view {d, Npad, B*H} of the fp32 dQ accumulator; box {32, box_rows, 1}
// (128 bytes x box_rows rows), 128-byte swizzle, used for TMA reductions.
bool make_map_acc(CUtensorMap* m, const float* base, int d, int Npad, int BH, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Npad),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                   static_cast<cuuint64_t>(Npad) * d * 4};
    const cuuint32_t box[3] = {32u, static_cast<cuuint32_t>(box_rows), 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every row of a bf16 tensor (base + element strides s) starts on a 32-byte
// boundary: the epilogues then write rows with 32-byte stores.
int rows_v8(const void* base, const Strides& s) {
    return (reinterpret_cast<uintptr_t>(base) & 31u) == 0 && (s.b * 2) % 32 == 0 && (s.h * 2) % 32 == 0 &&
                   (s.n * 2) % 32 == 0
               ? 1
               : 0;
}

Strides dense(int heads, int N, int d) {
    Strides s;
    s.n = d;
    s.h = static_cast<long long>(N) * d;
    s.b = static_cast<long long>(heads) * N * d;
    return s;
}

// Strides usable by TMA and by the 16-byte vector stores: non-negative,
// multiples of 16 bytes, below 2^40 bytes.
bool strides_ok(const Strides& s, int elem_bytes) {
    for (long long x : {s.b, s.h, s.n}) {
        if (x < 0 || (x * elem_bytes) % 16 != 0 || x * elem_bytes >= (1ll << 40)) return false;
    }
    return true;
}

constexpr long long kMaxElems = (1ll << 40);  // keeps every byte offset well inside 64 bits

attn_status check_sizes(int B, int H, int N, int d, float scale, int causal) {
    if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID;
    if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    if (d <= 0) return ATTN_ERR_INVALID;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    const long long bh = static_cast<long long>(B) * H;
    if (bh > (1ll << 31) - 1) return ATTN_ERR_INVALID;
    if (bh * N * d > kMaxElems) return ATTN_ERR_INVALID;
    const long long ctas = bh * ((N + 2 * kTile - 1) / (2 * kTile));
    const long long ctas_bwd = bh * ((N + kTile - 1) / kTile);
    if (ctas > 0x7fffffffll / 16 || ctas_bwd > 0x7fffffffll) return ATTN_ERR_INVALID;
    return ATTN_OK;
}

attn_status check_group(int H, int Hk) {
    return (Hk >= 1 && Hk <= H && H % Hk == 0) ? ATTN_OK : ATTN_ERR_INVALID;
}

attn_status check_window(int wl, int wr) { return (wl >= -1 && wr >= -1) ? ATTN_OK : ATTN_ERR_INVALID; }

long long npad(int N) { return (static_cast<long long>(N) + kTile - 1) / kTile * kTile; }

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct BwdLayout {
    size_t dq_acc, lse2, dsum, split_cnt, split_part, total;
    int split_cap;  // parts of split items the workspace holds (0: none)
};

// fp32 dQ accumulator, -LSE log2 e, D; for d = 128 (split) also the counters and
// partials of split items: at most min(kBwdSplitCap, items * min(10, ceil(N / 128)))
// parts, items <= B * H * ceil(N / 128) (an item is split at most ten ways, and
// never into more parts than its steps).
BwdLayout bwd_layout(int B, int H, int N, int d, bool split) {
    const size_t rows = static_cast<size_t>(B) * H * npad(N);
    BwdLayout L;
    L.dq_acc = 0;
    L.lse2 = round256(rows * d * sizeof(float));
    L.dsum = L.lse2 + round256(rows * sizeof(float));
    L.split_cnt = L.split_part = L.dsum + round256(rows * sizeof(float));
    L.total = L.split_cnt;
    L.split_cap = 0;
    if (split && d == 128) {
        const long long tiles = npad(N) / kTile;
        const long long room = static_cast<long long>(B) * H * tiles * (tiles < 10 ? tiles : 10);
        L.split_cap = static_cast<int>(room < kBwdSplitCap ? room : kBwdSplitCap);
        if (L.split_cap > 0) {
            L.split_part = L.split_cnt + round256(kBwdSplitCntWords * sizeof(unsigned));
            L.total = L.split_part + round256(static_cast<size_t>(L.split_cap) * 2 * kTile * d * sizeof(float));
        }
    }
    return L;
}

__global__ void wait_selftest_kernel(DevStatus st) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);  // nothing ever arrives on it
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x < 32) {
        wait_warp(b, 0, &abort_flag, st, 0x901);
    } else if (threadIdx.x == 32) {
        wait_one(b, 0, &abort_flag, st, 0x902);
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// Launch paths shared by the entry points (all arguments validated here)
// ---------------------------------------------------------------------------

// Split-KV partial buffers (null: single pass).
struct SplitArgs {
    int n_splits = 1;
    int split_len = 0;
    float* o_part = nullptr;
    float* lse_part = nullptr;
};

attn_status fwd_run(const void* q, const Strides& qs, const void* k, const Strides& ks, const void* v,
                    const Strides& vs, void* o, const Strides& os, float* lse, int B, int H, int Hk,
                    int N, int d, float scale, int win_left, int win_right, attn_stream_t stream,
                    const SplitArgs& split = SplitArgs()) {
    const int causal = (win_left == -1 && win_right == 0) ? 1 : 0;
    attn_status rc = check_sizes(B, H, N, d, scale, causal);
    if (rc != ATTN_OK) return rc;
    if ((rc = check_group(H, Hk)) != ATTN_OK || (rc = check_window(win_left, win_right)) != ATTN_OK)
        return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_INVALID;
    if (!strides_ok(qs, 2) || !strides_ok(ks, 2) || !strides_ok(vs, 2) || !strides_ok(os, 2))
        return ATTN_ERR_INVALID;
    DeviceState ds;
    if ((rc = device_state(&ds)) != ATTN_OK) return rc;
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, q, false, d, N, H, B, qs) || !make_map(&tk, k, false, d, N, Hk, B, ks) ||
        !make_map(&tv, v, false, d, N, Hk, B, vs))
        return ATTN_ERR_CUDA;
    FwdParams p;
    p.o = o;
    p.os = os;
    p.lse = lse;
    p.N = N;
    p.BH = B * H;
    p.H = H;
    p.Hk = Hk;
    p.n_pairs = (N + 2 * kTile - 1) / (2 * kTile);
    p.causal = causal;
    p.win_left = win_left;
    p.win_right = win_right;
    p.cs = scale * 1.44269504088896340736f;
    p.out_scale = 1.f;
    p.n_splits = split.n_splits;
    p.split_len = split.n_splits > 1 ? split.split_len : (N + kTile - 1) / kTile;
    p.o_part = split.o_part;
    p.lse_part = split.lse_part;
    p.exp2_offload = 0;
    p.single = 0;
    p.o_v8 = rows_v8(o, os);
    p.st = dev_status(ds);
    return launch_fwd_bf16(d, tq, tk, tv, p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
}

// Number of key-tile splits: none while the CTAs already cover most SMs
// (the partials and the combine then cost more than they give back), else
// the smallest power of two that covers them, at most one split per key tile
// and at most kMaxSplits.
constexpr int kMaxSplits = 16;
int auto_splits(int BH, int N, int num_sms) {
    const long long ctas = static_cast<long long>(BH) * ((N + 2 * kTile - 1) / (2 * kTile));
    const int n_kv = (N + kTile - 1) / kTile;
    int s = 1;
    while (s < kMaxSplits && s < n_kv && ctas * s * 4 < 3ll * num_sms) s *= 2;
    return s < n_kv ? s : n_kv;
}

size_t splitkv_bytes(int B, int H, int N, int d, int S) {
    const size_t rows = static_cast<size_t>(B) * H * N;
    return round256(static_cast<size_t>(S) * rows * d * sizeof(float)) +
           round256(static_cast<size_t>(S) * rows * sizeof(float));
}

// Validated view of the backward workspace.
struct BwdCall {
    DeviceState ds;
    float* dq_acc = nullptr;
    float* lse2 = nullptr;
    float* dsum = nullptr;
    unsigned* split_cnt = nullptr;
    float* split_part = nullptr;
    int split_cap = 0;
    int BH = 0, Np = 0;
};

attn_status bwd_prepare(void* workspace, int B, int H, int N, int d, float scale, int causal, bool split,
                        BwdCall* c) {
    attn_status rc = check_sizes(B, H, N, d, scale, causal);
    if (rc != ATTN_OK) return rc;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return ATTN_ERR_INVALID;
    if ((rc = device_state(&c->ds)) != ATTN_OK) return rc;
    const BwdLayout L = bwd_layout(B, H, N, d, split);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    c->dq_acc = reinterpret_cast<float*>(ws + L.dq_acc);
    c->lse2 = reinterpret_cast<float*>(ws + L.lse2);
    c->dsum = reinterpret_cast<float*>(ws + L.dsum);
    c->split_cap = L.split_cap;
    if (L.split_cap > 0) {
        c->split_cnt = reinterpret_cast<unsigned*>(ws + L.split_cnt);
        c->split_part = reinterpret_cast<float*>(ws + L.split_part);
    }
    c->BH = B * H;
    c->Np = static_cast<int>(npad(N));
    return ATTN_OK;
}

attn_status bwd_pre_run(const void* o, const Strides& os, const void* dout, const Strides& dos,
                        const float* lse, void* workspace, int B, int H, int N, int d, bool split,
                        attn_stream_t stream) {
    for (const void* p : {o, dout, static_cast<const void*>(lse)})
        if (!aligned16(p)) return ATTN_ERR_INVALID;
    if (!strides_ok(os, 2) || !strides_ok(dos, 2)) return ATTN_ERR_INVALID;
    BwdCall c;
    attn_status rc = bwd_prepare(workspace, B, H, N, d, 1.f, 0, split, &c);
    if (rc != ATTN_OK) return rc;
    BwdPreParams pp;
    pp.split_cnt = c.split_cnt;
    pp.split_cnt_words = c.split_cap > 0 ? kBwdSplitCntWords : 0;
    pp.o = o;
    pp.dout = dout;
    pp.os = os;
    pp.dos = dos;
    pp.lse = lse;
    pp.dq_acc = c.dq_acc;
    pp.lse2 = c.lse2;
    pp.dsum = c.dsum;
    pp.N = N;
    pp.Npad = c.Np;
    pp.BH = c.BH;
    pp.H = H;
    pp.D = d;
    return launch_bwd_pre(pp, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK
                                                                                     : ATTN_ERR_CUDA;
}

attn_status bwd_main_run(const void* q, const Strides& qs, const void* k, const Strides& ks,
                         const void* v, const Strides& vs, const void* dout, const Strides& dos,
                         void* dk, const Strides& dks, void* dv, const Strides& dvs, void* workspace,
                         int B, int H, int Hk, int N, int d, float scale, int win_left, int win_right,
                         bool split, attn_stream_t stream) {
    for (const void* p : {q, k, v, dout, static_cast<const void*>(dk), static_cast<const void*>(dv)})
        if (!aligned16(p)) return ATTN_ERR_INVALID;
    for (const Strides* st : {&qs, &ks, &vs, &dos, &dks, &dvs})
        if (!strides_ok(*st, 2)) return ATTN_ERR_INVALID;
    attn_status rc;
    if ((rc = check_group(H, Hk)) != ATTN_OK || (rc = check_window(win_left, win_right)) != ATTN_OK)
        return rc;
    const int causal = (win_left == -1 && win_right == 0) ? 1 : 0;
    BwdCall c;
    if ((rc = bwd_prepare(workspace, B, H, N, d, scale, causal, split, &c)) != ATTN_OK) return rc;
    CUtensorMap tq, tk, tv, tdo, tdq;
    if (!make_map(&tq, q, false, d, N, H, B, qs) || !make_map(&tk, k, false, d, N, Hk, B, ks) ||
        !make_map(&tv, v, false, d, N, Hk, B, vs) || !make_map(&tdo, dout, false, d, N, H, B, dos) ||
        !make_map_acc(&tdq, c.dq_acc, d, c.Np, c.BH, d == 128 ? 64 : 128))
        return ATTN_ERR_CUDA;
    BwdParams bp;
    bp.lse2 = c.lse2;
    bp.dsum = c.dsum;
    bp.dq_acc = c.dq_acc;
    bp.dk = dk;
    bp.dv = dv;
    bp.dks = dks;
    bp.dvs = dvs;
    bp.N = N;
    bp.Npad = c.Np;
    bp.BHk = B * Hk;
    bp.H = H;
    bp.Hk = Hk;
    bp.n_kv = (N + kTile - 1) / kTile;
    bp.causal = causal;
    bp.win_left = win_left;
    bp.win_right = win_right;
    bp.cs = scale * 1.44269504088896340736f;
    bp.scale = scale;
    bp.split_base = bp.BHk * bp.n_kv;  // the launcher decides on a split
    bp.split_parts = 1;
    bp.split_cap = c.split_cap;
    bp.split_part = c.split_part;
    bp.split_cnt = c.split_cnt;
    bp.dkv_v8 = rows_v8(dk, dks) && rows_v8(dv, dvs);
    bp.st = dev_status(c.ds);
    return launch_bwd_main(d, tq, tk, tv, tdo, tdq, bp, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
}

attn_status dq_convert_run(void* dq, const Strides& dqs, void* workspace, int B, int H, int N, int d,
                           float scale, attn_stream_t stream) {
    if (!aligned16(dq) || !strides_ok(dqs, 2)) return ATTN_ERR_INVALID;
    BwdCall c;
    attn_status rc = bwd_prepare(workspace, B, H, N, d, scale, 0, false, &c);
    if (rc != ATTN_OK) return rc;
    DqConvertParams cp;
    cp.dq_acc = c.dq_acc;
    cp.dq = dq;
    cp.dqs = dqs;
    cp.N = N;
    cp.Npad = c.Np;
    cp.BH = c.BH;
    cp.H = H;
    cp.D = d;
    cp.scale = scale;
    return launch_dq_convert(cp, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
}

// The whole backward: everything is validated before the first launch, so a
// bad argument leaves the stream untouched.
attn_status bwd_run(const void* q, const Strides& qs, const void* k, const Strides& ks, const void* v,
                    const Strides& vs, const void* o, const Strides& os, const void* dout,
                    const Strides& dos, const float* lse, void* dq, const Strides& dqs, void* dk,
                    const Strides& dks, void* dv, const Strides& dvs, void* workspace, int B, int H,
                    int Hk, int N, int d, float scale, int win_left, int win_right,
                    attn_stream_t stream, bool split = true) {
    const int causal = (win_left == -1 && win_right == 0) ? 1 : 0;
    attn_status rc = check_sizes(B, H, N, d, scale, causal);
    if (rc != ATTN_OK) return rc;
    if ((rc = check_group(H, Hk)) != ATTN_OK || (rc = check_window(win_left, win_right)) != ATTN_OK)
        return rc;
    for (const void* p : {q, k, v, o, dout, static_cast<const void*>(lse), static_cast<const void*>(dq),
                          static_cast<const void*>(dk), static_cast<const void*>(dv)})
        if (!aligned16(p)) return ATTN_ERR_INVALID;
    for (const Strides* st : {&qs, &ks, &vs, &os, &dos, &dqs, &dks, &dvs})
        if (!strides_ok(*st, 2)) return ATTN_ERR_INVALID;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return ATTN_ERR_INVALID;
    if ((rc = bwd_pre_run(o, os, dout, dos, lse, workspace, B, H, N, d, split, stream)) != ATTN_OK) return rc;
    if ((rc = bwd_main_run(q, qs, k, ks, v, vs, dout, dos, dk, dks, dv, dvs, workspace, B, H, Hk, N, d,
                           scale, win_left, win_right, split, stream)) != ATTN_OK)
        return rc;
    return dq_convert_run(dq, dqs, workspace, B, H, N, d, scale, stream);
}

Strides from_abi(const attn_strides_t& s) {
    Strides r;
    r.b = s.b;
    r.h = s.h;
    r.n = s.n;
    return r;
}

}  // namespace

int check_problem(int B, int H, int N, int d, float scale, int causal) {
    return static_cast<int>(check_sizes(B, H, N, d, scale, causal));
}

size_t bwd_workspace_bytes_for(int B, int H, int N, int d, bool split) {
    if (check_sizes(B, H, N, d, 1.f, 0) != ATTN_OK) return 0;
    return bwd_layout(B, H, N, d, split).total;
}

int bwd_dense(const void* q, const void* k, const void* v, const void* o, const void* dout,
              const float* lse, void* dq, void* dk, void* dv, void* workspace, int B, int H, int N,
              int d, float scale, int causal, bool split, cudaStream_t stream) {
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    const Strides ds = dense(H, N, d);
    return static_cast<int>(bwd_run(q, ds, k, ds, v, ds, o, ds, dout, ds, lse, dq, ds, dk, ds, dv, ds,
                                    workspace, B, H, H, N, d, scale, -1, causal ? 0 : -1, stream, split));
}

cudaError_t launch_wait_selftest(DevStatus st, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 64, 0, stream>>>(st);
    return cudaGetLastError();
}

}  // namespace attn

using namespace attn;

extern "C" {

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int N, int d, float scale, int causal, attn_stream_t stream) {
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    const Strides ds = dense(H, N, d);
    return fwd_run(q, ds, k, ds, v, ds, o, ds, lse, B, H, H, N, d, scale, -1, causal ? 0 : -1, stream);
}

attn_status attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int Hk, int N, int d, float scale, int causal, attn_stream_t stream) {
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    if (check_group(H, Hk) != ATTN_OK) return ATTN_ERR_INVALID;
    const Strides qs = dense(H, N, d), ks = dense(Hk, N, d);
    return fwd_run(q, qs, k, ks, v, ks, o, qs, lse, B, H, Hk, N, d, scale, -1, causal ? 0 : -1, stream);
}

attn_status attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                            int H, int Hk, int N, int d, float scale, int window_left,
                            int window_right, attn_stream_t stream) {
    if (check_group(H, Hk) != ATTN_OK) return ATTN_ERR_INVALID;
    const Strides qs = dense(H, N, d), ks = dense(Hk, N, d);
    return fwd_run(q, qs, k, ks, v, ks, o, qs, lse, B, H, Hk, N, d, scale, window_left, window_right,
                   stream);
}

attn_status attn_fwd_strided(const void* q, attn_strides_t qs, const void* k, attn_strides_t ks,
                             const void* v, attn_strides_t vs, void* o, attn_strides_t os, float* lse,
                             int B, int H, int Hk, int N, int d, float scale, int window_left,
                             int window_right, attn_stream_t stream) {
    return fwd_run(q, from_abi(qs), k, from_abi(ks), v, from_abi(vs), o, from_abi(os), lse, B, H, Hk,
                   N, d, scale, window_left, window_right, stream);
}

size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int N, int d, int num_splits) {
    if (check_sizes(B, H, N, d, 1.f, 0) != ATTN_OK) return 0;
    if (num_splits < 0 || num_splits > kMaxSplits) return 0;
    if (num_splits == 0) num_splits = kMaxSplits;  // enough for any automatic choice
    return splitkv_bytes(B, H, N, d, num_splits);
}

attn_status attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                             void* workspace, int B, int H, int N, int d, float scale, int causal,
                             int num_splits, attn_stream_t stream) {
    attn_status rc = check_sizes(B, H, N, d, scale, causal);
    if (rc != ATTN_OK) return rc;
    if (num_splits < 0 || num_splits > kMaxSplits) return ATTN_ERR_INVALID;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return ATTN_ERR_INVALID;
    const int BH = B * H;
    const int n_kv = (N + kTile - 1) / kTile;
    int S = num_splits;
    if (S == 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        S = auto_splits(BH, N, sms);
    }
    if (S > n_kv) S = n_kv;
    const Strides ds = dense(H, N, d);
    const int wr = causal ? 0 : -1;
    if (S <= 1) return fwd_run(q, ds, k, ds, v, ds, o, ds, lse, B, H, H, N, d, scale, -1, wr, stream);
    SplitArgs sp;
    sp.split_len = (n_kv + S - 1) / S;
    sp.n_splits = (n_kv + sp.split_len - 1) / sp.split_len;  // no empty trailing split
    const size_t rows = static_cast<size_t>(BH) * N;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    sp.o_part = reinterpret_cast<float*>(ws);
    sp.lse_part = reinterpret_cast<float*>(
        ws + round256(static_cast<size_t>(sp.n_splits) * rows * d * sizeof(float)));
    if ((rc = fwd_run(q, ds, k, ds, v, ds, o, ds, lse, B, H, H, N, d, scale, -1, wr, stream, sp)) !=
        ATTN_OK)
        return rc;
    CombineParams c;
    c.o_part = sp.o_part;
    c.lse_part = sp.lse_part;
    c.o = o;
    c.os = ds;
    c.lse = lse;
    c.S = sp.n_splits;
    c.BH = BH;
    c.H = H;
    c.N = N;
    c.D = d;
    return launch_splitkv_combine(c, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
}

attn_status attn_fwd_fp8(const void* q8, const void* k8, const void* v8, float sq, float sk, float sv,
                         void* o, float* lse, int B, int H, int N, int d, float scale, int causal,
                         attn_stream_t stream) {
    attn_status rc = check_sizes(B, H, N, d, scale, causal);
    if (rc != ATTN_OK) return rc;
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    for (float s : {sq, sk, sv})
        if (!(s > 0.f) || !std::isfinite(s)) return ATTN_ERR_INVALID;
    if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_INVALID;
    DeviceState ds;
    if ((rc = device_state(&ds)) != ATTN_OK) return rc;
    const Strides st = dense(H, N, d);
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, q8, true, d, N, H, B, st) || !make_map(&tk, k8, true, d, N, H, B, st) ||
        !make_map(&tv, v8, true, d, N, H, B, st))
        return ATTN_ERR_CUDA;
    FwdParams p;
    p.o = o;
    p.os = st;
    p.lse = lse;
    p.N = N;
    p.BH = B * H;
    p.H = H;
    p.Hk = H;
    p.n_pairs = (N + 2 * kTile - 1) / (2 * kTile);
    p.causal = causal;
    p.win_left = -1;
    p.win_right = causal ? 0 : -1;
    p.cs = scale * sq * sk * 1.44269504088896340736f;
    p.out_scale = sv;
    p.n_splits = 1;
    p.split_len = (N + kTile - 1) / kTile;
    p.o_part = nullptr;
    p.lse_part = nullptr;
    p.exp2_offload = g_exp2_offload;
    p.single = 0;
    p.o_v8 = rows_v8(o, st);
    p.st = dev_status(ds);
    return launch_fwd_fp8(d, tq, tk, tv, p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
}

size_t attn_bwd_workspace_bytes(int B, int H, int N, int d) {
    return bwd_workspace_bytes_for(B, H, N, d, true);
}

attn_status attn_bwd_preprocess(const void* o, const void* dout, const float* lse, void* workspace,
                                int B, int H, int N, int d, attn_stream_t stream) {
    if (check_sizes(B, H, N, d, 1.f, 0) != ATTN_OK) return check_sizes(B, H, N, d, 1.f, 0);
    const Strides ds = dense(H, N, d);
    return bwd_pre_run(o, ds, dout, ds, lse, workspace, B, H, N, d, true, stream);
}

attn_status attn_bwd_main(const void* q, const void* k, const void* v, const void* dout, void* dk,
                          void* dv, void* workspace, int B, int H, int N, int d, float scale,
                          int causal, attn_stream_t stream) {
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    if (check_sizes(B, H, N, d, scale, causal) != ATTN_OK) return check_sizes(B, H, N, d, scale, causal);
    const Strides ds = dense(H, N, d);
    return bwd_main_run(q, ds, k, ds, v, ds, dout, ds, dk, ds, dv, ds, workspace, B, H, H, N, d, scale,
                        -1, causal ? 0 : -1, true, stream);
}

attn_status attn_bwd_dq_convert(void* dq, void* workspace, int B, int H, int N, int d, float scale,
                                attn_stream_t stream) {
    if (check_sizes(B, H, N, d, scale, 0) != ATTN_OK) return check_sizes(B, H, N, d, scale, 0);
    return dq_convert_run(dq, dense(H, N, d), workspace, B, H, N, d, scale, stream);
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, void* workspace, int B, int H,
                     int N, int d, float scale, int causal, attn_stream_t stream) {
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    if (check_sizes(B, H, N, d, scale, causal) != ATTN_OK) return check_sizes(B, H, N, d, scale, causal);
    const Strides ds = dense(H, N, d);
    return bwd_run(q, ds, k, ds, v, ds, o, ds, dout, ds, lse, dq, ds, dk, ds, dv, ds, workspace, B, H,
                   H, N, d, scale, -1, causal ? 0 : -1, stream);
}

attn_status attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv,
                         void* workspace, int B, int H, int Hk, int N, int d, float scale, int causal,
                         attn_stream_t stream) {
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    if (check_group(H, Hk) != ATTN_OK) return ATTN_ERR_INVALID;
    if (check_sizes(B, H, N, d, scale, causal) != ATTN_OK) return check_sizes(B, H, N, d, scale, causal);
    const Strides qs = dense(H, N, d), ks = dense(Hk, N, d);
    return bwd_run(q, qs, k, ks, v, ks, o, qs, dout, qs, lse, dq, qs, dk, ks, dv, ks, workspace, B, H,
                   Hk, N, d, scale, -1, causal ? 0 : -1, stream);
}

attn_status attn_bwd_window(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv,
                            void* workspace, int B, int H, int Hk, int N, int d, float scale,
                            int window_left, int window_right, attn_stream_t stream) {
    if (check_group(H, Hk) != ATTN_OK) return ATTN_ERR_INVALID;
    if (check_sizes(B, H, N, d, scale, 0) != ATTN_OK) return check_sizes(B, H, N, d, scale, 0);
    const Strides qs = dense(H, N, d), ks = dense(Hk, N, d);
    return bwd_run(q, qs, k, ks, v, ks, o, qs, dout, qs, lse, dq, qs, dk, ks, dv, ks, workspace, B, H,
                   Hk, N, d, scale, window_left, window_right, stream);
}

attn_status attn_bwd_strided(const void* q, attn_strides_t qs, const void* k, attn_strides_t ks,
                             const void* v, attn_strides_t vs, const void* o, attn_strides_t os,
                             const void* dout, attn_strides_t dos, const float* lse, void* dq,
                             attn_strides_t dqs, void* dk, attn_strides_t dks, void* dv,
                             attn_strides_t dvs, void* workspace, int B, int H, int Hk, int N, int d,
                             float scale, int window_left, int window_right, attn_stream_t stream) {
    return bwd_run(q, from_abi(qs), k, from_abi(ks), v, from_abi(vs), o, from_abi(os), dout,
                   from_abi(dos), lse, dq, from_abi(dqs), dk, from_abi(dks), dv, from_abi(dvs),
                   workspace, B, H, Hk, N, d, scale, window_left, window_right, stream);
}

attn_status attn_check_device_error(attn_stream_t stream, unsigned int* site) {
    if (site) *site = 0;
    DeviceState ds;
    attn_status rc = device_state(&ds);
    if (rc != ATTN_OK) return rc;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    unsigned int host[2] = {0, 0};
    const unsigned int zero[2] = {0, 0};
    if (cudaMemcpy(host, ds.err, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(ds.err, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (site) *site = host[1];
    return host[0] ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

void attn_set_exp2_offload(int on) { g_exp2_offload = on ? 1 : 0; }

void attn_set_wait_limit_ns(unsigned long long ns) {
    g_wait_limit_ns = ns ? ns : kDefaultWaitLimitNs;
}

attn_status attn_selftest_wait_timeout(attn_stream_t stream) {
    DeviceState ds;
    attn_status rc = device_state(&ds);
    if (rc != ATTN_OK) return rc;
    return launch_wait_selftest(dev_status(ds), reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
}

const char* attn_status_string(attn_status s) {
    switch (s) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID: return "ATTN_ERR_INVALID";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
        case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    }
    return "ATTN_ERR_UNKNOWN";
}

int attn_build_flags(void) { return kDebugChecks ? 1 : 0; }

int attn_kernel_smem_bytes(int which, int d) {
    if (which == 0) return fwd_smem_bytes(d, false);
    if (which == 1) return fwd_smem_bytes(d, true);
    if (which == 2) return bwd_smem_bytes(d);
    return 0;
}

}  // extern "C"
