/*
 * attn_sm103a.h -- C ABI of libattn_sm103a.so: exact softmax attention on one
 * NVIDIA GB300 (sm_103a), forward, backward and FP8 forward.
 *
 * What is computed (per batch b and head h, all rows independent):
 *   S = scale * Q K^T, with the causal mask "key j visible to query i iff
 *   j <= i" when causal = 1; P = softmax(S) row-wise; O = P V;
 *   LSE_i = ln(sum_j exp(S_ij)) (natural log, of the scaled scores).
 * The forward pass is tiled with the online-softmax recurrence -- running
 * maximum and running sum of exponentials, combined after rescaling to a
 * common maximum, with the same rescale applied to the output accumulator --
 * so the N x N matrices S and P are never written to memory
 * (xtrax digest "q02 FlashAttention", sections 1-2; ai.engineer topic page,
 * items 57 "Online Normalizer Calculation for Softmax" and 58
 * "FlashAttention").  The backward pass recomputes P from Q, K and the saved
 * LSE (item 58) and uses dV = P^T dO, dP = dO V^T, D_i = sum_k dO_ik O_ik,
 * dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q.
 *
 * Conventions shared by every entry point:
 *  - Layout: Q, K, V, O, dO, dQ, dK, dV are dense row-major [B, H, N, d]
 *    (d contiguous); LSE is dense [B, H, N].  Sequence lengths of queries and
 *    keys are equal (N).  d is 64 or 128 (FP8: 128).
 *  - Pointers are DEVICE pointers, 16-byte aligned, owned by the caller; the
 *    library allocates nothing and keeps no pointer after a call returns.
 *    Outputs whose rows all start on a 32-byte boundary (O of the forward, dK
 *    and dV of the backward) are written with 32-byte stores, others with
 *    16-byte ones; the results are the same bits.
 *  - Work is enqueued asynchronously on `stream` (0 = legacy default stream);
 *    nothing synchronises.  Outputs are valid once the stream reaches that
 *    point.
 *  - Errors are returned, never thrown or printed.  Invalid arguments return
 *    ATTN_ERR_INVALID (or ATTN_ERR_UNSUPPORTED for a valid but unbuilt shape
 *    or a device other than sm_103) before anything is launched.  A launch
 *    failure returns ATTN_ERR_CUDA.  Kernels never trap: a pipeline wait that
 *    does not complete within the wait limit (default 1 s) makes the kernel
 *    record the fact and return; attn_check_device_error() reports it.
 */
#ifndef ATTN_SM103A_H_
#define ATTN_SM103A_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* attn_stream_t; /* same type as cudaStream_t */

/* Element strides of a [B, heads, N, d] view whose d dimension is contiguous
 * (stride 1).  A dense [B, heads, N, d] tensor has n = d, h = N*d,
 * b = heads*N*d; PyTorch's [B, N, heads, d] layout has n = heads*d, h = d,
 * b = N*heads*d.  Every stride times the element size must be a multiple of
 * 16 bytes. */
typedef struct {
    int64_t b, h, n;
} attn_strides_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID = -1,     /* bad pointer, size, alignment or scale */
    ATTN_ERR_UNSUPPORTED = -2, /* d or dtype not built, or device is not sm_103 */
    ATTN_ERR_CUDA = -3,        /* a CUDA runtime or driver call failed */
    ATTN_ERR_TIMEOUT = -4      /* a kernel's bounded wait gave up (device error word) */
} attn_status;

/*
 * Forward pass, bf16 in and out, fp32 accumulation.
 *   q, k, v : bf16 [B, H, N, d] inputs.
 *   o       : bf16 [B, H, N, d] output, O = P V rounded to nearest even.
 *   lse     : fp32 [B, H, N] output, natural log-sum-exp of the scaled scores
 *             (the statistic attn_bwd consumes).
 *   scale   : softmax scale, finite and > 0 (usually 1/sqrt(d)).
 *   causal  : 0 or 1.
 * Source: FlashAttention digest sections 1-2 (tiling, online softmax, fused
 * single kernel); ai.engineer items 41 (query-row tiles across blocks, delayed
 * normalisation), 58, 59 (causal mask) and 60 (-inf guards).
 */
attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, float scale, int causal, attn_stream_t stream);

/*
 * Bytes of device scratch attn_bwd needs for (B, H, N, d): an fp32 dQ
 * accumulator [B*H, Npad, d] plus two fp32 vectors [B*H, Npad] (LSE in log2
 * units and D), Npad = N rounded up to 128; for d = 128 also 5 KB of counters
 * and room for fp32 dV/dK partials of min(160, B*H*T*min(10, T)) parts of
 * split key-tile items, T = Npad/128 (128 KB each; see attn_bwd).  Every
 * region starts on a 256-byte boundary.  Returns 0 for invalid sizes.
 */
size_t attn_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass for O = softmax(scale Q K^T [+mask]) V.
 *   q, k, v, o, dout : bf16 [B, H, N, d] inputs (o and lse from attn_fwd).
 *   lse              : fp32 [B, H, N] from attn_fwd.
 *   dq, dk, dv       : bf16 [B, H, N, d] outputs.
 *   workspace        : device scratch of attn_bwd_workspace_bytes() bytes,
 *                      256-byte aligned, caller-owned; overwritten.
 * Three kernels run in order on `stream`: preprocess (D, LSE, zeroed dQ
 * accumulator), main (recompute P, accumulate dV, dK in tensor memory, add
 * dQ partial tiles into the accumulator with fp32 reductions), and dQ
 * conversion.  dQ's summation order varies from run to run (scatter-add
 * item 52); dK and dV are deterministic.  d = 128 without a mask: the main
 * kernel's CTAs (one per SM) take key tiles in rounds; when the last round
 * (or the only one, with fewer key tiles than SMs) has fewer key tiles than
 * CTAs, each of them is shared by several CTAs (its query tiles split into
 * parts), whose fp32 dV/dK partials are added in the workspace in part order
 * by the last part to finish.  Causal with few key/value heads: the longest
 * key tiles are split in two the same way when that shortens the launch.
 * Causal launches whose Q, dO and dQ accumulator pass 64 MiB take their key
 * tiles in groups of heads, so that the heads in flight stay in the L2.
 * The main kernel and the conversion are launched as programmatic dependents
 * of the kernel before each (their set-up overlaps its tail; they wait for it
 * to complete before touching memory), which stream capture keeps.
 * Source: ai.engineer item 58 (backward regenerates score tiles from saved
 * normalisation statistics); FlashAttention-3 digest section 1 (dQ-writer
 * warp and atomic accumulation); the gradient formulas are the calculus of
 * the forward definition (the pages' own statement of them is cut off).
 */
attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, void* workspace, int B,
                     int H, int N, int d, float scale, int causal, attn_stream_t stream);

/*
 * The three stages of attn_bwd, for callers that schedule or time them
 * separately.  They must run in this order on one stream with the same
 * workspace and sizes; attn_bwd is exactly these three calls.
 *   attn_bwd_preprocess : D_i = sum_k dO_ik O_ik, LSE in log2 units, padded
 *                         rows, and a zeroed fp32 dQ accumulator, all in the
 *                         workspace.  Reads o, dout, lse.
 *   attn_bwd_main       : recomputes P, writes dk, dv (bf16) and adds every
 *                         partial dQ tile into the workspace accumulator.
 *   attn_bwd_dq_convert : dq = bf16(scale * accumulator).
 * Same argument rules and errors as attn_bwd.
 */
attn_status attn_bwd_preprocess(const void* o, const void* dout, const float* lse, void* workspace,
                                int B, int H, int N, int d, attn_stream_t stream);
attn_status attn_bwd_main(const void* q, const void* k, const void* v, const void* dout, void* dk,
                          void* dv, void* workspace, int B, int H, int N, int d, float scale,
                          int causal, attn_stream_t stream);
attn_status attn_bwd_dq_convert(void* dq, void* workspace, int B, int H, int N, int d, float scale,
                                attn_stream_t stream);

/*
 * attn_bwd without a workspace argument, for callers that cannot allocate
 * device memory -- for example code that a host framework hands only its
 * input and output tensors while the framework owns all device memory and
 * allows no allocation after start-up.  The pages describe no such variant;
 * it has no counterpart there.
 *   Arguments and results are those of attn_bwd, with the scratch taken
 *   from a fixed 64 MiB array inside the library instead of `workspace`.
 *   The problem is checked first, as attn_bwd checks it, with the same
 *   status (ATTN_ERR_INVALID for bad sizes, scale or flag,
 *   ATTN_ERR_UNSUPPORTED for a head dim other than 64 or 128); a valid
 *   problem is then rejected with ATTN_ERR_UNSUPPORTED, before anything is
 *   launched, when even the scratch without the split last round's partials
 *   exceeds 64 MiB (about 129k padded rows at d = 128, e.g.
 *   B*H*ceil(N/128)*128 <= 129,000).  Where attn_bwd_workspace_bytes() fits
 *   the 64 MiB the results are attn_bwd's bit for bit; between the two sizes
 *   the d = 128 main kernel runs without the split last round, and dK, dV
 *   rows of its last round's key tiles may differ from attn_bwd's in the last
 *   bit (another summation order).  Pointer and launch errors are those of
 *   attn_bwd.
 *   Every call looks up the array's device address in the current context
 *   (a lookup, no allocation), so the entry point stays valid after
 *   cudaDeviceReset or a change of context.  The first call in a context may
 *   load the library's device code into it: make that first call before any
 *   stream capture.  Every GPU that loads this part of the library keeps the
 *   64 MiB until the process exits.  Nothing is allocated by any call.
 *   All calls on a device share the one array: calls that overlap on the GPU
 *   (unordered streams) race and give wrong results.  Each call zeroes the
 *   part that must start at zero, so earlier calls do not leak into later ones.
 */
attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                             const void* dout, const float* lse, void* dq, void* dk, void* dv,
                             int B, int H, int N, int d, float scale, int causal,
                             attn_stream_t stream);

/*
 * Grouped-query attention (GQA; multi-query attention when Hk = 1): Hk
 * key/value heads shared by H query heads, H a multiple of Hk; query head h
 * reads key/value head h / (H / Hk).  q, o: [B, H, N, d]; k, v: [B, Hk, N, d];
 * lse: [B, H, N].  attn_fwd / attn_bwd are the Hk = H case.
 * attn_bwd_gqa: dq [B, H, N, d]; dk, dv [B, Hk, N, d], each the sum over the
 * query heads of its group; workspace = attn_bwd_workspace_bytes(B, H, N, d).
 * One backward CTA per (batch, key/value head, 128-key tile) visits all query
 * heads of the group in turn, so dK and dV need no cross-CTA reduction.
 * Source: FlashAttention-3 walkthrough (runtime parameter num_heads_k; GQA/MQA
 * listed among its features).  Errors as attn_fwd / attn_bwd, plus
 * ATTN_ERR_INVALID when Hk < 1 or H % Hk != 0.
 */
attn_status attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int Hk, int N, int d, float scale, int causal, attn_stream_t stream);
attn_status attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv,
                         void* workspace, int B, int H, int Hk, int N, int d, float scale, int causal,
                         attn_stream_t stream);

/*
 * Split-KV forward for problems too small to fill the GPU (few heads, long
 * sequences): the key tiles of every query-tile pair are divided among
 * `num_splits` CTAs, each writing an fp32 partial (O over its keys and that
 * log-sum-exp) to `workspace`; a combine kernel then merges the partials with
 * the running-max / running-sum rule and writes o (bf16) and lse as attn_fwd.
 *   num_splits : 1..16, or 0 to choose (about two waves of CTAs); 1 is attn_fwd.
 *   workspace  : attn_fwd_splitkv_workspace_bytes(B, H, N, d, num_splits) bytes,
 *                256-byte aligned, caller-owned (num_splits = 0: room for 16).
 * Two launches on `stream`.  Source: ai.engineer item 59 (small-query work
 * split across thread blocks plus a separate combining kernel); FlashAttention-3
 * tuning page (num_splits runtime parameter); the merge is the online-softmax
 * combination of the FlashAttention digest, section 2.
 */
size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int N, int d, int num_splits);
attn_status attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                             void* workspace, int B, int H, int N, int d, float scale, int causal,
                             int num_splits, attn_stream_t stream);

/*
 * Sliding-window (local) attention, with grouped heads as in attn_fwd_gqa:
 * key j is visible to query i iff i - window_left <= j <= i + window_right;
 * -1 removes that bound (window_left = -1, window_right = 0 is causal;
 * -1, -1 is no mask).  Key tiles outside every row's window are skipped in
 * both passes.  Arguments otherwise as attn_fwd_gqa / attn_bwd_gqa; bounds
 * below -1 give ATTN_ERR_INVALID.
 * Source: FlashAttention-3 tuning page (Is_local, window_size_left /
 * window_size_right runtime parameters).
 */
attn_status attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                            int H, int Hk, int N, int d, float scale, int window_left,
                            int window_right, attn_stream_t stream);
attn_status attn_bwd_window(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv,
                            void* workspace, int B, int H, int Hk, int N, int d, float scale,
                            int window_left, int window_right, attn_stream_t stream);

/*
 * The general entry points: grouped heads, sliding window, and any strides
 * per tensor (q, o, dout, dq over H heads; k, v, dk, dv over Hk heads).
 * window_left / window_right as attn_fwd_window (-1, -1: no mask; -1, 0:
 * causal).  lse stays dense [B, H, N].  Every other entry point is a special
 * case of these two.  Strides that are negative, or not multiples of 16
 * bytes, give ATTN_ERR_INVALID.
 * Source: FlashAttention-3 walkthrough (batch / seqlen / num_heads /
 * num_heads_k / head_dim runtime parameters); ai.engineer items on tensor
 * storage, strides and views (the tensor is a view over storage given by its
 * strides).
 */
attn_status attn_fwd_strided(const void* q, attn_strides_t qs, const void* k, attn_strides_t ks,
                             const void* v, attn_strides_t vs, void* o, attn_strides_t os, float* lse,
                             int B, int H, int Hk, int N, int d, float scale, int window_left,
                             int window_right, attn_stream_t stream);
attn_status attn_bwd_strided(const void* q, attn_strides_t qs, const void* k, attn_strides_t ks,
                             const void* v, attn_strides_t vs, const void* o, attn_strides_t os,
                             const void* dout, attn_strides_t dos, const float* lse, void* dq,
                             attn_strides_t dqs, void* dk, attn_strides_t dks, void* dv,
                             attn_strides_t dvs, void* workspace, int B, int H, int Hk, int N, int d,
                             float scale, int window_left, int window_right, attn_stream_t stream);

/*
 * FP8 forward pass: OCP E4M3 inputs with per-tensor fp32 scales.
 *   q8, k8, v8 : uint8 E4M3 codes [B, H, N, d]; the value read is s * code
 *                (sq, sk, sv finite and > 0).
 *   o          : bf16 [B, H, N, d] output; lse : fp32 [B, H, N] as attn_fwd.
 * Scores use fp32 accumulation of the E4M3 products; P is rounded to E4M3
 * (saturating) before the P V product, which accumulates in fp32.  d = 128.
 * Source: FlashAttention-3 digest (FP8 forward); ai.engineer item 33
 * (affine quantisation r = S(q - Z), here Z = 0).
 */
attn_status attn_fwd_fp8(const void* q8, const void* k8, const void* v8, float sq, float sk,
                         float sv, void* o, float* lse, int B, int H, int N, int d, float scale,
                         int causal, attn_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the library's device error
 * word on the current device.  Returns ATTN_ERR_TIMEOUT if any kernel's
 * bounded wait gave up since the last check (the results of that launch are
 * undefined), ATTN_ERR_CUDA if synchronisation failed, else ATTN_OK.
 * `site` (may be NULL) receives the id of the first wait that gave up.
 */
attn_status attn_check_device_error(attn_stream_t stream, unsigned int* site);

/*
 * Wait limit, in nanoseconds, that every pipeline wait of later launches
 * uses before it gives up (default 1e9).  0 restores the default.
 */
void attn_set_wait_limit_ns(unsigned long long ns);

/*
 * Exponential offload of the FP8 forward (later attn_fwd_fp8 calls; default
 * off): with on != 0, one group of four score columns in eight computes its
 * exponentials on the FMA pipe (2^x = 2^n 2^r, n = round(x), 2^r from a cubic
 * with relative error below 7.5e-5) instead of the MUFU unit.  Results stay
 * within the FP8 tolerance either way.  Off by default because it measured
 * slower on GB300 (B1 H16 N16384 d128 causal: 0.588 vs 0.533 ms): the softmax
 * pass is bound by instruction issue and latency, not by MUFU throughput.
 * Source: kernaut-resources wiki, FlashAttention-3 code walkthrough README,
 * technique tag "software-exp" (exponentials emulated on the FMA units).
 */
void attn_set_exp2_offload(int on);

/*
 * Self-test of the bounded-wait path: launches one CTA whose warps wait on a
 * barrier nothing ever completes, with the current wait limit.  The kernel
 * returns after the limit; attn_check_device_error() must then report
 * ATTN_ERR_TIMEOUT.  No fault, trap or hang is involved.
 */
attn_status attn_selftest_wait_timeout(attn_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* attn_status_string(attn_status s);

/* Dynamic shared memory (bytes) one CTA of the given kernel requests:
 * which = 0 forward bf16, 1 forward fp8, 2 backward main; 0 if not built. */
int attn_kernel_smem_bytes(int which, int d);

/* How this copy of the library was built.  Bit 0: device-side range checks
 * (libattn_sm103a_debug.so): every TMA box coordinate is checked against the
 * tensor's extents and 16-byte rule, and every tensor-memory access and MMA
 * operand address against the warp's lane quadrant and the 512 allocated
 * columns.  A failed check skips the access and makes the next
 * attn_check_device_error() return ATTN_ERR_TIMEOUT with the check's site id
 * (0xD01-0xD05 tensor memory, 0x1D1-0x1D2 and 0x2D1-0x2D6 TMA and bulk copies);
 * it never traps.  The checks stand in for a memory checker in tests; the
 * release library has none (bit 0 clear).  The pages describe no such build. */
int attn_build_flags(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_SM103A_H_ */
