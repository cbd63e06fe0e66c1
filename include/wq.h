/*
 * wq.h -- C ABI of the W8A8 INT8 fused Mixture-of-Experts layer (libwq.so).
 *
 * Sources of the method:
 *   [CW]  "[Feature] DeepSeek V3/R1 INT8 Quantization (channel-wise)",
 *         sglang pull request 3888, sections Modifications and Performance
 *         (fused MoE with channel-wise INT8 weights, int32 or fp32
 *         accumulator).
 *   [MT]  "老显卡福音！美团技术团队开源首发INT8无损满血版DeepSeek R1"
 *         (jiqizhixin, the Meituan INT8 DeepSeek R1 article), section
 *         量化技术的探索 (block-wise [128,128] weights with per-token-group
 *         activations; channel-wise weights with per-token activations and
 *         one dequantization after the INT8 matmul).
 *   [EP]  "[WIP] feat: support cutlass_moe_fp8 for deepepmoe", sglang pull
 *         request 8273, review comments (expert offsets = cumulative counts
 *         with a leading zero; ep_scatter; gather after the second GEMM;
 *         workspace sized from the problem instead of a fixed 1 GB).
 *   [LL]  "Support DeepSeek-R1 w4a8 low latency deepep", sglang pull request
 *         8311, Highlights and review (masked per-expert layout with
 *         per-expert problem sizes; a per-expert host loop to scatter
 *         results is a bottleneck; cudagraph-compatible).
 *
 * Conventions (all entry points):
 *   - Every pointer is a DEVICE pointer owned by the caller, except where an
 *     argument is marked "host".  The library never allocates device memory;
 *     scratch comes from a caller-provided workspace whose size the matching
 *     *_workspace_size() function returns.
 *   - bf16 tensors are passed as uint16_t bit patterns.  All matrices are
 *     row-major and contiguous unless a leading dimension (in elements) is
 *     given.
 *   - Every call is asynchronous on the given CUDA stream (cudaStream_t, may
 *     be NULL for the legacy default stream), performs no host
 *     synchronisation and reads no device data on the host, so it can be
 *     recorded into a CUDA graph.  Grouped GEMMs over many small segments
 *     (the masked layout) run two engines concurrently: the second on a
 *     stream of the library's own, forked from and joined back into the
 *     caller's stream through events (recorded into a graph like any other
 *     stream work).  That stream and its two events are created once per
 *     device, on first use outside a graph capture, and kept for the
 *     process; without them both engines run on the caller's stream.
 *   - Return value: WQ_OK (0) when the work was enqueued, otherwise a
 *     negative WQ_ERR_* code and nothing was enqueued.  Argument errors are
 *     detected on the host before any launch.
 *   - Errors only visible on the device (an expert id out of range, a
 *     bounded wait that gave up) are written to the caller's int32 device
 *     word `status` (first error wins; the caller zeroes it).  Kernels that
 *     detect such an error skip the offending element and never trap.
 *   - Floating point: float32 IEEE arithmetic, every multiply, add and divide
 *     rounded to nearest even and never fused, in the order each function
 *     states; results are bit-reproducible run to run.
 *   - Devices: compute capability 10.3 (GB300, sm_103a) only.
 */
#ifndef WQ_H
#define WQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define WQ_API __attribute__((visibility("default")))
#else
#define WQ_API
#endif

typedef struct CUstream_st *wq_stream_t; /* identical to cudaStream_t */

enum {
  WQ_OK = 0,
  WQ_ERR_INVALID_ARG = -1,   /* null pointer, negative size, bad enum value   */
  WQ_ERR_UNSUPPORTED = -2,   /* shape/alignment outside what the kernels take */
  WQ_ERR_DEVICE = -3,        /* no device, or not compute capability 10.3     */
  WQ_ERR_LAUNCH = -4,        /* a CUDA launch or copy failed                  */
  WQ_ERR_WORKSPACE = -5,     /* workspace smaller than *_workspace_size()     */
  WQ_ERR_INDEX = -6,         /* device: an index (expert id) out of range     */
  WQ_ERR_TIMEOUT = -7        /* device: a bounded pipeline wait gave up       */
};

enum { WQ_SCHEME_CHANNEL = 0, WQ_SCHEME_BLOCK = 1 };
enum { WQ_ACC_I32 = 0, WQ_ACC_F32 = 1 };
enum { WQ_OUT_BF16 = 0, WQ_OUT_I32 = 1 };

/* Checks that `device` exists and is compute capability 10.3 and makes it
 * current for the calling thread.  Returns WQ_OK or WQ_ERR_DEVICE. */
WQ_API int wq_init(int device);

/* Static text for a status code (never NULL). */
WQ_API const char *wq_status_string(int code);

/* Number of kernels this library has enqueued in the process so far (all
 * devices and threads; monotone).  Accounting only: a caller differences it
 * around a region to count the library's launches there.  The pages have no
 * counterpart. */
WQ_API uint64_t wq_kernel_launches(void);

/* Failure-path self-test of the bounded pipeline waits.  Takes the arguments
 * of wq_grouped_gemm_w8a8_f16codes for the block scheme (bf16 out, workspace
 * wq_grouped_gemm_workspace_size(R, E)) and launches the block-wise CTA-pair
 * engine with a wait on a barrier that nothing completes, placed before any
 * copy or MMA is issued.  The wait gives up after its 1 s limit; the kernel
 * writes WQ_ERR_TIMEOUT into *status (device, required) and releases tensor
 * memory.  out is not written.  The call itself returns WQ_OK once the launch
 * is enqueued, and the device context stays usable for the next call.  The
 * pages have no counterpart. */
WQ_API int wq_selftest_wait_timeout(const uint16_t *A16, const float *sa, const int8_t *W,
                                    const float *sw, const int32_t *offsets, int E, int64_t R,
                                    int64_t N, int64_t K, void *out, void *ws, size_t ws_bytes,
                                    int32_t *status, wq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Online activation quantization [MT] (and offline weight quantization).
 *
 * Per row of x (bf16 [T][K], leading dimension ldx elements):
 *   a = max |x_j|;  s = max(a, 1e-10f) / 127;  q_j = clamp(rint(x_j / s), -127, 127)
 * (ties to even, symmetric range, -128 never produced).
 * Outputs: q int8 [T][K] contiguous, s float [T].
 * Requirements: K % 8 == 0, ldx % 8 == 0, x 16-byte aligned, q 8-byte aligned.
 * T == 0 or K == 0 enqueues nothing.  Also used for channel-wise weights
 * (one row per output channel). */
WQ_API int wq_quantize_per_token(const uint16_t *x, int64_t T, int64_t K, int64_t ldx,
                          int8_t *q, float *s, wq_stream_t stream);

/* Per-token-group variant [MT] (block-wise scheme): the same rule on each
 * run of `group` consecutive elements of a row.  s is float [T][K/group].
 * Requirements: group in {32, 64, 128, 256}, K % group == 0, plus the
 * alignment rules above. */
WQ_API int wq_quantize_per_token_group(const uint16_t *x, int64_t T, int64_t K, int64_t ldx,
                                int group, int8_t *q, float *s, wq_stream_t stream);

/* Offline FP8 -> BF16 -> INT8 weight conversion [MT] (量化技术的探索: the
 * released weights are FP8; they are dequantized to BF16, then quantized to
 * INT8 per [128,128] block or per output channel).  w8: FP8 e4m3 bytes
 * [N][K] (no infinities; NaN bytes give unspecified codes); s8: float one
 * scale per [128,128] block [N/128][K/128].  Each value is (e4m3 value *
 * block scale) rounded to float32 then to bf16, and the bf16 matrix is
 * quantized by the rule above: scheme WQ_SCHEME_CHANNEL -> q int8 [N][K],
 * s float [N]; WQ_SCHEME_BLOCK -> s float [N/128][K/128].  The bf16 values
 * never reach memory.  Requirements: N % 128 == 0, K % 128 == 0 (channel:
 * K <= 16384), w8 and q 16-byte aligned. */
WQ_API int wq_convert_fp8_weights(const uint8_t *w8, const float *s8, int64_t N, int64_t K,
                                  int scheme, int8_t *q, float *s, wq_stream_t stream);

/* Offline [128,128] block weight quantization [MT]: w bf16 [N][K] ->
 * q int8 [N][K], s float [N/128][K/128]; the rule above over each block.
 * Requirements: N % 128 == 0, K % 128 == 0, w 16-byte aligned. */
WQ_API int wq_quantize_weight_block(const uint16_t *w, int64_t N, int64_t K, int8_t *q, float *s,
                             wq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Routing: top-k of the softmax over E router logits, renormalised over the
 * chosen experts (the pages consume topk_idx [EP]; the router is this
 * layer's configuration).  Per token t (logits float [T][E]):
 *   ids[t][0..k) = the k largest logits, descending, equal logits -> lower id;
 *   m = logit of ids[t][0];  e_j = exp(l_j - m) (Cody-Waite exp, see below);
 *   S = ((e_0 + e_1) + e_2) + ...;  w[t][j] = e_j / S.
 * exp: n = rint(x*log2e); r = (x - n*ln2_hi) - n*ln2_lo; degree-7 Taylor
 * polynomial in Horner form; times 2^floor(n/2) times 2^(n-floor(n/2));
 * x >= 89 -> inf, x <= -104 -> 0.
 * Outputs ids int32 [T][k], w float [T][k].  Requirements: 1 <= E <= 1024,
 * 1 <= k <= min(E, 32). */
WQ_API int wq_route_topk(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                  wq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Alignment [EP]: group the T*k (token, slot) pairs by expert.  Pair
 * p = t*k + j goes to expert ids[p].
 *   counts[e]      int32 [E]    pairs routed to e;
 *   offsets        int32 [E+1]  0, then cumulative ceil(counts/pad_m)*pad_m;
 *   sorted_pair[r] int32 [T*k + E*(pad_m-1)]  pair held by permuted row r,
 *                  pairs of one expert in ascending p; -1 on padding rows
 *                  and on every row at or past offsets[E];
 *   pair_to_row[p] int32 [T*k]  inverse map (-1 for a pair whose id is out
 *                  of range; such pairs also set status = WQ_ERR_INDEX).
 * Deterministic (a stable counting sort; no atomics decide an order).
 * Requirements: 1 <= E <= 4096, 1 <= pad_m <= 1024, T*k < 2^31.
 * Workspace: wq_moe_align_workspace_size(T, k, E) bytes. */
WQ_API size_t wq_moe_align_workspace_size(int T, int k, int E);
WQ_API int wq_moe_align(const int32_t *ids, int T, int k, int E, int pad_m, int32_t *counts,
                 int32_t *offsets, int32_t *sorted_pair, int32_t *pair_to_row, void *ws,
                 size_t ws_bytes, int32_t *status, wq_stream_t stream);

/* Permute (ep_scatter [EP]): for each of the R rows of sorted_pair,
 *   A[r] = q[sorted_pair[r] / k],  sa[r][g] = s[sorted_pair[r] / k][g];
 * rows with sorted_pair = -1 get zero codes and zero scales.
 * q int8 [T][K], s float [T][groups] -> A int8 [R][K], sa float [R][groups].
 * Requirements: K % 16 == 0, 16-byte aligned q and A, groups >= 1. */
WQ_API int wq_moe_permute(const int8_t *q, const float *s, int groups, int T, int k, int64_t K,
                   const int32_t *sorted_pair, int64_t R, int8_t *A, float *sa,
                   wq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Grouped W8A8 GEMM with dequantization epilogue [CW][MT].
 * Rows [offsets[e], offsets[e+1]) of A (int8 [R][K]) use expert e's weight
 * W[e] (int8 [E][N][K], one row per output channel):  C = A_e W_e^T (exact).
 *   CHANNEL + I32: v = (float(C) * sa[r]) * sw[e][n]            sa [R], sw [E][N]
 *   CHANNEL + F32: C_t = int32 sum over K tile t (128 wide);
 *                  acc = 0; for t ascending: acc = acc + float(C_t);
 *                  v = (acc * sa[r]) * sw[e][n]
 *   BLOCK (acc ignored, fp32): for kb ascending:
 *                  acc = acc + float(C_kb) * (sa[r][kb] * sw[e][n/128][kb])
 *                  sa [R][K/128], sw [E][N/128][K/128]
 * out: bf16 [R][N] (v rounded to nearest even) or, with WQ_OUT_I32 and
 * CHANNEL+I32 only, the raw int32 C.  Rows outside every expert's segment
 * are not written.  float(.) rounds to nearest even.
 * Requirements: N % 128 == 0, K % 128 == 0, 16-byte aligned A, W, out.
 * Workspace: wq_grouped_gemm_workspace_size(R, E) bytes. */
WQ_API size_t wq_grouped_gemm_workspace_size(int64_t R, int E);
WQ_API int wq_grouped_gemm_w8a8(const int8_t *A, const float *sa, const int8_t *W, const float *sw,
                         const int32_t *offsets, int E, int64_t R, int64_t N, int64_t K,
                         int scheme, int acc, int out_type, void *out, void *ws,
                         size_t ws_bytes, int32_t *status, wq_stream_t stream);

/* Grouped W8A8 GEMM without a workspace argument.  The pages have no
 * counterpart: this entry point exists for callers that may not allocate
 * device memory at run time (a plug-in inside a host framework that owns
 * the device memory pool and gives plug-ins no allocator; a serving loop that
 * cannot accept cudaMalloc's implicit device synchronisation once started).
 * Arguments, results and requirements are those of wq_grouped_gemm_w8a8
 * minus ws/ws_bytes.  The scratch lives in a static device array of
 * WQ_NOALLOC_SCRATCH_BYTES that every GPU loading libwq.so holds until the
 * process exits; the first call on a device looks up that array's address
 * (cudaGetSymbolAddress) with the device current.  All calls on a device
 * share the array; calls that overlap on the GPU race on it.  Arguments are
 * checked first, exactly as wq_grouped_gemm_w8a8 checks them (same codes);
 * then a problem whose scratch need (wq_grouped_gemm_workspace_size(R, E))
 * exceeds the array returns WQ_ERR_UNSUPPORTED before any work is enqueued.
 * Nothing is allocated. */
#define WQ_NOALLOC_SCRATCH_BYTES (256 * 1024)
WQ_API int wq_grouped_gemm_w8a8_noalloc(const int8_t *A, const float *sa, const int8_t *W,
                                        const float *sw, const int32_t *offsets, int E, int64_t R,
                                        int64_t N, int64_t K, int scheme, int acc, int out_type,
                                        void *out, int32_t *status, wq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Activation codes stored as fp16 values ("fp16 codes"): the same integers in
 * [-127, 127] as the int8 codes, two bytes each, with each row's squared L2
 * norm (sum of code^2, int32).  This is the form the CTA-pair GEMM engines
 * read directly (TMA straight into the MMA layout); the one-call layer uses
 * it when experts hold many rows and both GEMM widths are multiples of 256.
 *
 * wq_moe_permute_f16: as wq_moe_permute, writing A16 uint16 (fp16 bits)
 *   [R][K] and norm2 int32 [R] (padding rows: zero codes, scale, norm).
 * wq_silu_mul_quant_f16: as wq_silu_mul_quant (group 0: one scale per row;
 *   32/64/128/256: per-group scales, sh [R][I/group]), writing hq16 (fp16
 *   bits) [R][I]; with group 0 also norm2 int32 [R] (with a group, norm2 is
 *   not written and may be NULL).
 * wq_grouped_gemm_w8a8_f16codes: as wq_grouped_gemm_w8a8 with A given as
 *   fp16 codes.  Channel scheme (acc WQ_ACC_I32 or WQ_ACC_F32; out_type
 *   WQ_OUT_I32 only with WQ_ACC_I32): a_norm2 must be the exact row sums of
 *   squares (they decide whether the single-pass float32 sums are provably
 *   exact, else the launch is recomputed exactly).  Block scheme (sa
 *   [R][K/128], sw [E][N/128][K/128], bf16 output): a_norm2 is not read and
 *   may be NULL; every 128-wide K block's sum is exact in float32.
 *   Requirements: N % 256 == 0, K % 128 == 0, K <= 65536.
 *   Workspace: wq_grouped_gemm_workspace_size(R, E). */
WQ_API int wq_moe_permute_f16(const int8_t *q, const float *s, int groups, int T, int k, int64_t K,
                              const int32_t *sorted_pair, int64_t R, uint16_t *A16, float *sa,
                              int32_t *norm2, wq_stream_t stream);
WQ_API int wq_silu_mul_quant_f16(const uint16_t *gu, int64_t R, int64_t I, int group,
                                 uint16_t *hq16, float *sh, int32_t *norm2, wq_stream_t stream);
WQ_API int wq_grouped_gemm_w8a8_f16codes(const uint16_t *A16, const int32_t *a_norm2,
                                         const float *sa, const int8_t *W, const float *sw,
                                         const int32_t *offsets, int E, int64_t R, int64_t N,
                                         int64_t K, int scheme, int acc, int out_type, void *out,
                                         void *ws, size_t ws_bytes, int32_t *status,
                                         wq_stream_t stream);

/* Fused gate_up GEMM -> SiLU-and-mul -> re-quantization, block-wise scheme
 * ("[Feature] DeepSeek V3/R1 INT8 Quantization (channel-wise)", Performance:
 * the accumulator and epilogue cost set the throughput; Meituan INT8 DeepSeek
 * R1 article, 量化技术的探索: activations quantized per token per 128-group,
 * weights per [128,128] block).  A16 fp16 codes [R][K] with sa [R][K/128],
 * W13 int8 [E][2I][K] (gate rows [0, I), up rows [I, 2I)) with sw13
 * [E][2I/128][K/128], segments from offsets [E+1].  The result is exactly
 *   wq_silu_mul_quant_f16(gu, R, I, 128, ...) of
 *   gu = wq_grouped_gemm_w8a8_f16codes(..., N = 2I, WQ_SCHEME_BLOCK, bf16 out)
 * (gate and up rounded to bf16 before SiLU), written as hq16 fp16 codes
 * [R][I] and sh float [R][I/128]; gu itself never reaches memory.  Each
 * 128-column group of h depends on one gate and one up weight block only, so
 * the two CTAs of a pair compute the matching blocks and finish the group.
 * scheme must be WQ_SCHEME_BLOCK: the channel scheme re-quantizes h with one
 * scale per whole row of I columns, which no single tile sees
 * (WQ_ERR_UNSUPPORTED).
 * Requirements: I % 128 == 0, K % 128 == 0, K <= 65536, 16-byte aligned
 * A16, W13 and hq16.  Workspace: wq_grouped_gemm_silu_quant_workspace_size(R, E)
 * bytes (the grouped GEMM's plus a silu table).
 * hq16 and sh rows outside every segment are not written. */
WQ_API size_t wq_grouped_gemm_silu_quant_workspace_size(int64_t R, int E);
WQ_API int wq_grouped_gemm_w8a8_silu_quant_f16codes(const uint16_t *A16, const float *sa,
                                                    const int8_t *W13, const float *sw13,
                                                    const int32_t *offsets, int E, int64_t R,
                                                    int64_t I, int64_t K, int scheme,
                                                    uint16_t *hq16, float *sh, void *ws,
                                                    size_t ws_bytes, int32_t *status,
                                                    wq_stream_t stream);

/* Per-token quantization into fp16 codes with row norms (the rule of
 * wq_quantize_per_token, Meituan INT8 DeepSeek R1 article, 量化技术的探索:
 * online per-token activation quantization): codes as fp16 bits q16 [T][K]
 * (row pitch K), s float32 [T] and norm2 int32 [T] = sum of code^2 of each
 * row, the input form of wq_grouped_gemm_w8a8_f16codes (a dense W8A8 linear
 * with one expert reads it directly).
 * Requirements: K % 8 == 0, ldx % 8 == 0, K <= 65536, 16-byte aligned x and
 * q16. */
WQ_API int wq_quantize_per_token_f16(const uint16_t *x, int64_t T, int64_t K, int64_t ldx,
                                     uint16_t *q16, float *s, int32_t *norm2, wq_stream_t stream);

/* Quantization and permute in one pass, scatter form (the quantization rule
 * of wq_quantize_per_token / wq_quantize_per_token_group, Meituan INT8
 * DeepSeek R1 article, 量化技术的探索; the ep_scatter placement of
 * "[WIP] feat: support cutlass_moe_fp8 for deepepmoe", review).  Each token
 * of x bf16 [T][K] is quantized once (group 0: one scale per token; 32, 64,
 * 128 or 256: one per group) and its codes, as fp16 bits, go to every row
 * r = pair_to_row[t * k + j] (j < k, the map wq_moe_align returns):
 * A16 [R][K] (row pitch K), sa [R] or [R][K/group], and with group 0 also
 * norm2 int32 [R] = the row's sum of code^2 (with a group norm2 is not
 * written and may be NULL).  The result equals wq_quantize_per_token(_group)
 * followed by wq_moe_permute_f16 on every row some pair maps to; rows no pair
 * maps to (alignment padding) are not written, and map entries outside
 * [0, R) are skipped.
 * Requirements: 1 <= k <= 32, K % 8 == 0, K % group == 0, K <= 65536,
 * 16-byte aligned x and A16. * wq_quantize_permute: the same with int8 codes A int8 [R][K] (row pitch K)
 * and no norms; 16-byte aligned x and A. */
WQ_API int wq_quantize_permute_f16(const uint16_t *x, int64_t T, int64_t K, int group,
                                   const int32_t *pair_to_row, int k, int64_t R, uint16_t *A16,
                                   float *sa, int32_t *norm2, wq_stream_t stream);
WQ_API int wq_quantize_permute(const uint16_t *x, int64_t T, int64_t K, int group,
                               const int32_t *pair_to_row, int k, int64_t R, int8_t *A, float *sa,
                               wq_stream_t stream);

/* Masked layout [LL]: A int8 [E][Mmax][K] with per-row scales sa
 * ([E][Mmax] or [E][Mmax][K/128]) and valid counts masked_m int32 [E]
 * (device).  Expert e computes rows [0, min(masked_m[e], Mmax)) with the
 * epilogues above; out is [E][Mmax][N]; rows at or past masked_m[e] are not
 * written.  Negative counts count as zero.
 * Workspace: wq_grouped_gemm_masked_workspace_size(E, Mmax) bytes. */
WQ_API size_t wq_grouped_gemm_masked_workspace_size(int E, int Mmax);
WQ_API int wq_grouped_gemm_w8a8_masked(const int8_t *A, const float *sa, const int32_t *masked_m,
                                int E, int Mmax, const int8_t *W, const float *sw, int64_t N,
                                int64_t K, int scheme, int acc, int out_type, void *out,
                                void *ws, size_t ws_bytes, int32_t *status,
                                wq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Activation between the GEMMs (the "activation" of the scatter -> GEMM ->
 * activation -> GEMM -> gather flow [EP]) with re-quantization.
 * gu bf16 [R][2I]: g = gu[r][c], u = gu[r][I + c] (gate half first),
 *   h = (g / (1 + exp(-g))) * u        (exp as in wq_route_topk)
 * then the quantization rule per row (group = 0) or per `group` elements
 * (group in {32, 64, 128, 256}).  hq int8 [R][I], sh float [R] or [R][I/group].
 * Requirements: I % 8 == 0 (and I % group == 0), 16-byte aligned gu. */
WQ_API int wq_silu_mul_quant(const uint16_t *gu, int64_t R, int64_t I, int group, int8_t *hq,
                      float *sh, wq_stream_t stream);

/* Combine (the gather after the second GEMM [EP]; one launch instead of a
 * per-expert host loop [LL]):
 *   out[t] = bf16( acc ),  acc = 0; for j ascending: acc = acc + w[t][j] * y[pair_to_row[t*k+j]]
 * y bf16 [*][H], pair_to_row int32 [T*k] (a -1 entry contributes nothing),
 * w float [T][k], out bf16 [T][H].  Requirements: 1 <= k <= 32, H % 8 == 0,
 * 16-byte aligned y and out (k > 32: WQ_ERR_UNSUPPORTED). */
WQ_API int wq_moe_combine(const uint16_t *y, const int32_t *pair_to_row, const float *w, int T, int k,
                   int64_t H, uint16_t *out, wq_stream_t stream);

/* ---------------------------------------------------------------------------
 * The whole layer in one call, on one stream, no host synchronisation:
 *   route -> quantize (per token, or per 128-group for BLOCK) -> align ->
 *   permute -> GEMM1 (W13 [E][2I][H]) -> SiLU-mul + re-quantize ->
 *   GEMM2 (W2 [E][H][I]) -> combine.
 * x bf16 [T][H], logits float [T][E]; sw13/sw2 as in wq_grouped_gemm_w8a8
 * for the scheme; out bf16 [T][H].  Requirements: those of the steps, and
 * H % 128 == 0, I % 128 == 0.  Workspace: wq_moe_forward_workspace_size(). */
WQ_API size_t wq_moe_forward_workspace_size(int T, int H, int I, int E, int k, int scheme);
WQ_API int wq_moe_forward(const uint16_t *x, const float *logits, const int8_t *W13, const float *sw13,
                   const int8_t *W2, const float *sw2, int T, int H, int I, int E, int k,
                   int scheme, int acc, uint16_t *out, void *ws, size_t ws_bytes,
                   int32_t *status, wq_stream_t stream);

/* Same layer with HOST activations x_host bf16 [T][H] and logits_host
 * float [T][E], result in out_host bf16 [T][H].  When all three buffers are
 * pinned host memory mapped into the device's address space (16-byte
 * aligned x_host and out_host), the quantization kernel reads x_host, the
 * router reads logits_host and the combine writes out_host across the
 * CPU-GPU link, with no staging copies.  Otherwise the inputs are copied to
 * the workspace on `stream` and the result copied back (asynchronous for
 * pinned memory).  Either way the caller synchronises the stream before
 * reading out_host and leaves x_host and logits_host unchanged until then.
 * Workspace: wq_moe_forward_host_workspace_size() (it covers both cases). */
WQ_API size_t wq_moe_forward_host_workspace_size(int T, int H, int I, int E, int k, int scheme);
WQ_API int wq_moe_forward_host(const uint16_t *x_host, const float *logits_host, const int8_t *W13,
                        const float *sw13, const int8_t *W2, const float *sw2, int T, int H,
                        int I, int E, int k, int scheme, int acc, uint16_t *out_host,
                        void *ws, size_t ws_bytes, int32_t *status, wq_stream_t stream);

/* Masked-layout layer [LL]: already-quantized activations a int8
 * [E][Mmax][H] with scales sa ([E][Mmax], or [E][Mmax][H/128] for BLOCK) and
 * valid counts masked_m [E] -> y bf16 [E][Mmax][H] (GEMM1 -> SiLU-mul +
 * re-quantize -> GEMM2 on the valid rows; other rows not written).
 * Workspace: wq_moe_forward_masked_workspace_size().  With the CHANNEL
 * scheme and Mmax > 64 it also holds an fp16 copy of each GEMM's valid input
 * rows (E * Mmax * max(H, I) * 2 bytes, 235 MB at 32 x 512 x 7168), which
 * the tensor-core engine loads as token tiles. */
WQ_API size_t wq_moe_forward_masked_workspace_size(int E, int Mmax, int H, int I, int scheme);
WQ_API int wq_moe_forward_masked(const int8_t *a, const float *sa, const int32_t *masked_m, int E,
                          int Mmax, const int8_t *W13, const float *sw13, const int8_t *W2,
                          const float *sw2, int H, int I, int scheme, int acc, uint16_t *y,
                          void *ws, size_t ws_bytes, int32_t *status, wq_stream_t stream);

/* ---------------------------------------------------------------------------
 * W4A8 on the masked layout [LL] ("Support DeepSeek-R1 w4a8 low latency
 * deepep", Highlights: a w4a8 weight path for the masked low-latency layer).
 * The page fixes no int4 format; this library reads it as the channel-wise
 * rule of the INT8 weights with 7 in place of 127:
 *   per output channel n: s4[n] = max(max_k |w[n][k]|, 1e-10) / 7,
 *   q[n][k] = clamp(rint(w[n][k] / s4[n]), -7, 7)   (ties to even),
 * stored two codes a byte, code 2j in bits 0-3 and code 2j+1 in bits 4-7 of
 * byte j (two's complement nibbles): W4 uint8 [N][K/2] per expert.
 * Activations are the int8 per-token codes of wq_quantize_per_token.
 *
 * wq_quantize_weight_int4: w bf16 [N][K] -> q4 uint8 [N][K/2], s4 float [N].
 *   Requirements: K % 8 == 0, 16-byte aligned w, 4-byte aligned q4.
 * wq_grouped_gemm_w4a8_masked: as wq_grouped_gemm_w8a8_masked (channel
 *   scheme, int32 accumulator) with W4 uint8 [E][N][K/2] and s4 [E][N]:
 *   C = sum_k a[e][r][k] * q[e][n][k] exactly (|C| <= 127 * 7 * K), then
 *   out = bf16((float(C) * sa[e][r]) * s4[e][n]), or C itself for
 *   WQ_OUT_I32.  Rows at or past masked_m[e] are not written.
 *   Requirements: N % 128 == 0, K % 128 == 0, K <= 16384 (every float32
 *   partial sum of the tensor-core pass is then an exact integer), 16-byte
 *   aligned A, W4 and out.  Workspace:
 *   wq_grouped_gemm_masked_workspace_size(E, Mmax).
 * wq_moe_forward_masked_w4a8: the masked layer of wq_moe_forward_masked
 *   (channel scheme, int32 accumulator) with int4 W13 [E][2I][H/2] (s13
 *   [E][2I]) and W2 [E][H][I/2] (s2 [E][H]).  Requirements: H, I multiples
 *   of 128 and at most 16384.  Workspace:
 *   wq_moe_forward_masked_w4a8_workspace_size(). */
WQ_API int wq_quantize_weight_int4(const uint16_t *w, int64_t N, int64_t K, uint8_t *q4,
                                   float *s4, wq_stream_t stream);
WQ_API int wq_grouped_gemm_w4a8_masked(const int8_t *A, const float *sa, const int32_t *masked_m,
                                       int E, int Mmax, const uint8_t *W4, const float *s4,
                                       int64_t N, int64_t K, int out_type, void *out, void *ws,
                                       size_t ws_bytes, int32_t *status, wq_stream_t stream);
WQ_API size_t wq_moe_forward_masked_w4a8_workspace_size(int E, int Mmax, int H, int I);
WQ_API int wq_moe_forward_masked_w4a8(const int8_t *a, const float *sa, const int32_t *masked_m,
                                      int E, int Mmax, const uint8_t *W13, const float *s13,
                                      const uint8_t *W2, const float *s2, int H, int I,
                                      uint16_t *y, void *ws, size_t ws_bytes, int32_t *status,
                                      wq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Dense W8A8 INT8 linear [CW] (Modifications, "Norm Linear": the model's
 * non-MoE linear layers run as a w8a8 INT8 GEMM).  out = dequant(quant(x)
 * W^T): the activation quantization of the scheme (per token, or per token
 * per 128-group for the block scheme), the INT8 GEMM and its dequantization
 * exactly as wq_grouped_gemm_w8a8 with one expert.
 *   x bf16 [T][K] (leading dimension ldx), W int8 [N][K], sw float [N]
 *   (channel) or [N/128][K/128] (block), out bf16 [T][N] contiguous.
 * Requirements: K % 128 == 0, N % 128 == 0, K <= 65536, ldx % 8 == 0, x, W
 * and out 16-byte aligned.  T == 0 enqueues nothing.
 * Workspace: wq_linear_w8a8_workspace_size(T, K, N, scheme) (0: the shape is
 * not supported).  Device-side errors go to *status (may be NULL). */
WQ_API size_t wq_linear_w8a8_workspace_size(int64_t T, int64_t K, int64_t N, int scheme);
WQ_API int wq_linear_w8a8(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, const int8_t *W,
                          const float *sw, int64_t N, int scheme, int acc, uint16_t *out, void *ws,
                          size_t ws_bytes, int32_t *status, wq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* WQ_H */
