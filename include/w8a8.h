/*
 * w8a8.h -- C ABI of the GB300 (sm_103a) W8A8_DYNAMIC linear-layer and
 * MoE-expert library (libw8a8.so).
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子"
 *        §一 quantisation recipe (activations per-token symmetric INT8,
 *            weights per-channel symmetric INT8; W13 = gate_proj + up_proj,
 *            W2 = down_proj);
 *        §二 Dense path: load-time transpose + format cast of the INT8
 *            weight, npu_dynamic_quant, npu_quant_matmul, output dtype BF16;
 *        §三 MoE path: npu_grouped_matmul over group_list (rows per expert),
 *            W13 GMM -> SwiGLU -> Requant -> W2 GMM, and the rule that an
 *            input that already carries a per-token scale is not quantised
 *            again;
 *        §四 operator contract: INT8 x1, INT8 x2, FLOAT32 per-token scale,
 *            BF16 output.
 *   [P2] "Qwen3.8-FP8 on Ascend 950: Why Weights Become MXFP8 at Load Time",
 *        Deep Dive 4 (load-time repack into persistent buffers whose addresses
 *        stay fixed for graph replay) and 6 (MoE weights prepared one expert
 *        at a time); "Where It Breaks or Falls Back" (error conventions).
 *
 * Conventions for every call:
 *   - Tensor pointers are DEVICE pointers owned by the caller, row-major and
 *     contiguous.  BF16 tensors are passed as uint16_t bit patterns.
 *   - Work is enqueued on `stream` and returns without synchronising; the
 *     library allocates nothing and never synchronises in these calls.  The
 *     caller keeps every buffer alive until the stream work completes.
 *   - Argument errors are detected on the host and returned synchronously;
 *     nothing is launched then.  Errors that depend on device data (a bad
 *     group_list, a packed weight that does not match the call, an exhausted
 *     wait) are written to the status word at the start of the caller's
 *     workspace; read them with w8a8_read_device_status().
 *   - Workspaces must be zero-filled once before their first use; every call
 *     leaves the parts that must start at zero (arrival counters, split-K
 *     sums) zeroed again, and the status word too unless an error was
 *     recorded (w8a8_read_device_status() clears it).  One workspace serves
 *     one stream at a time.
 *   - K (the reduction depth) must be a multiple of 16 and at most
 *     W8A8_MAX_K; M, N and group sizes are arbitrary (>= 0 / >= 1).
 *   - Integer results (INT8 payloads, INT32 accumulators) and FP32 scales are
 *     exact; BF16 outputs are the binary32 epilogue rounded to nearest-even.
 */
#ifndef W8A8_H
#define W8A8_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define W8A8_API __attribute__((visibility("default")))
#else
#define W8A8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t), passed through untouched; NULL = legacy default stream. */
typedef struct CUstream_st* w8a8_stream_t;

typedef enum {
  W8A8_OK = 0,
  W8A8_ERR_NULL = 1,           /* a required pointer is NULL */
  W8A8_ERR_SHAPE = 2,          /* a size is negative, zero where it must not be, or too large */
  W8A8_ERR_ALIGN = 3,          /* K % 16 != 0, or a pointer is not 16-byte aligned */
  W8A8_ERR_WORKSPACE = 4,      /* workspace NULL or smaller than the matching *_workspace_bytes() */
  W8A8_ERR_GROUP_LIST = 5,     /* device: a count < 0 or the counts do not sum to R */
  W8A8_ERR_DEVICE_TIMEOUT = 6, /* device: a bounded wait gave up */
  W8A8_ERR_CUDA = 7,           /* a CUDA runtime call failed (launch error etc.) */
  W8A8_ERR_UNSUPPORTED = 8,    /* the device is not sm_103 / a mode is not built */
  W8A8_ERR_PACKED = 9,         /* device: packed weight header does not match the call */
  W8A8_ERR_TOPK_IDS = 10       /* device: a topk id outside [0,E), or a routed row index outside [0,T*k) */
} w8a8_status;

#define W8A8_MAX_K 65536
#define W8A8_MAX_EXPERTS 1024
#define W8A8_STATUS_BYTES 256 /* the status word at the start of every workspace */

/* Human-readable name of a status code (static string). */
W8A8_API const char* w8a8_status_string(int status);

/* Library version (major*10000 + minor*100 + patch). */
W8A8_API int w8a8_version(void);

/* ------------------------------------------------------------------------ */
/* Weight prepack -- [P1] §二 (INT8 weight [N,K] transposed and cast to the  */
/* kernel's layout once at load time, reused by every forward) and [P2] Deep */
/* Dive 4 and 6 (persistent repacked buffers; MoE experts one at a time).    */
/* ------------------------------------------------------------------------ */

/* Pack flags. */
#define W8A8_PACK_GATE_UP 1u /* W13 [E,2I,K]: interleave gate rows [0,I) and up rows [I,2I)
                                in blocks of 64 so one tile holds matching gate/up channels;
                                requires N even and (N/2) % 64 == 0 */
#define W8A8_PACK_F16 2u     /* also store an integer-valued FP16 copy of the weights, which
                                one large-M tensor-core engine reads; without it large-M
                                calls run on the CTA-pair engine that widens the INT8 weights
                                in tensor memory (a third of the memory) */

/* Bytes of the packed buffer for E experts of [N,K] INT8 weights (E = 1 for a dense layer). */
W8A8_API size_t w8a8_prepacked_bytes(int64_t E, int64_t N, int64_t K, uint32_t flags);

/* w [E,N,K] int8 row-major (the checkpoint layout: output channel major, K
 * contiguous) -> packed (device buffer of w8a8_prepacked_bytes() bytes,
 * 256-byte aligned).  The packed buffer starts with a header recording
 * E, N, K and flags; later calls check it on the device.  Runs once per weight
 * at load time; the source may be freed after the stream work completes. */
W8A8_API w8a8_status w8a8_prepack_weight(const int8_t* w, int64_t E, int64_t N, int64_t K, uint32_t flags,
                                void* packed, w8a8_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Offline weight quantisation -- [P1] §一 (the msModelSlim recipe: weight   */
/* scope per_channel, dtype int8, symmetric) and §二 (the checkpoint weight  */
/* is already INT8 when loaded: it was quantised once, offline, from BF16).  */
/* Per output channel n of W [E,N,K] over its K inputs:                      */
/* s[e,n] = max_k |W[e,n,k]| / 127 (binary32 divide),                        */
/* q = clamp(rint(W / s), -127, 127), ties to even; an all-zero channel gets */
/* s = 0 and q = 0 -- the activation recipe applied to each channel.         */
/* ------------------------------------------------------------------------ */

/* w [E,N,K] bf16 -> q [E,N,K] int8 (the checkpoint layout) and scale [E,N]
 * fp32.  K % 16 == 0 (<= W8A8_MAX_K), w and q 16-byte aligned. */
W8A8_API w8a8_status w8a8_quantize_weight(const uint16_t* w, int64_t E, int64_t N, int64_t K, int8_t* q,
                                          float* scale, w8a8_stream_t stream);

/* The same quantisation written straight into a packed buffer (as
 * w8a8_prepack_weight would pack the INT8 weight, flags alike: the W13
 * gate/up interleave and the fp16 copy), one pass over the BF16 weight;
 * scale [E,N] in the ORIGINAL channel order (what the contractions take).
 * packed: w8a8_prepacked_bytes(E, N, K, flags) bytes, 256-byte aligned. */
W8A8_API w8a8_status w8a8_quantize_prepack_weight(const uint16_t* w, int64_t E, int64_t N, int64_t K,
                                                  uint32_t flags, void* packed, float* scale,
                                                  w8a8_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Dynamic per-token quantisation -- [P1] §二 npu_dynamic_quant and §三      */
/* HiddenStatesDynamicQuant: amax = max_k |x[m,k]|, scale[m] = amax / 127    */
/* (binary32 divide), q = clamp(rint(x / scale), -127, 127), rint = ties to  */
/* even; a row of zeros gets scale 0 and q = 0.                              */
/* ------------------------------------------------------------------------ */

/* x [M,K] bf16 -> q [M,K] int8, scale [M] fp32.  M >= 0, K % 16 == 0, x and q 16-byte aligned. */
W8A8_API w8a8_status w8a8_dynamic_quant(const uint16_t* x, int64_t M, int64_t K, int8_t* q, float* scale,
                               w8a8_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Dense quantised matmul -- [P1] §二 npu_quant_matmul and §四:              */
/* acc[m,n] = sum_k q[m,k] * W[n,k] (exact INT32);                          */
/* y[m,n] = bf16_rne(((float)acc * x_scale[m]) * w_scale[n] + bias[n]).      */
/* ------------------------------------------------------------------------ */

W8A8_API size_t w8a8_quant_matmul_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* q [M,K] int8, x_scale [M] fp32, w_packed (from w8a8_prepack_weight with E = 1,
 * flags 0 or W8A8_PACK_F16), w_scale [N] fp32, bias [N] bf16 or NULL -> y [M,N] bf16.
 * ws: zero-filled device workspace of at least w8a8_quant_matmul_workspace_bytes(). */
W8A8_API w8a8_status w8a8_quant_matmul(const int8_t* q, const float* x_scale, int64_t M, int64_t K,
                              const void* w_packed, const float* w_scale, int64_t N,
                              const uint16_t* bias, uint16_t* y, void* ws, size_t ws_bytes,
                              w8a8_stream_t stream);

/* Same contraction, writing the exact INT32 accumulators acc [M,N] instead of
 * the dequantised output (validation entry point for bit-exact checks). */
W8A8_API w8a8_status w8a8_int8_matmul_acc(const int8_t* q, int64_t M, int64_t K, const void* w_packed,
                                 int64_t N, int32_t* acc, void* ws, size_t ws_bytes,
                                 w8a8_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Grouped matmul -- [P1] §三 npu_grouped_matmul(x, weight, scale,           */
/* per_token_scale, group_list): group_list[e] = number of rows of expert e; */
/* rows are contiguous per expert in expert order; rows of expert e use      */
/* W[e] and w_scale[e,:]; experts with 0 rows are skipped.                   */
/* ------------------------------------------------------------------------ */

W8A8_API size_t w8a8_grouped_matmul_workspace_bytes(int64_t E, int64_t R, int64_t N, int64_t K);

/* q [R,K] int8, x_scale [R] fp32, group_list [E] int64 (device) counts,
 * w_packed (E experts, flags 0 or W8A8_PACK_F16), w_scale [E,N] fp32 -> y [R,N] bf16.
 * Counts < 0 or a sum != R set W8A8_ERR_GROUP_LIST on the device and write nothing. */
W8A8_API w8a8_status w8a8_grouped_matmul(const int8_t* q, const float* x_scale, const int64_t* group_list,
                                int64_t E, int64_t R, int64_t K, const void* w_packed,
                                const float* w_scale, int64_t N, uint16_t* y, void* ws,
                                size_t ws_bytes, w8a8_stream_t stream);

/* Grouped contraction writing the exact INT32 accumulators acc [R,N] (validation). */
W8A8_API w8a8_status w8a8_grouped_matmul_acc(const int8_t* q, const int64_t* group_list, int64_t E,
                                    int64_t R, int64_t K, const void* w_packed, int64_t N,
                                    int32_t* acc, void* ws, size_t ws_bytes, w8a8_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Static W8A8 -- [P1] closing comparison of the static recipe: npu_quantize */
/* with a fixed input_scale s and input_offset o; at load time               */
/* deq_scale[n] = s * weight_scale[n] and                                    */
/* quant_bias[n] = round(fp_bias[n] / deq_scale[n] - sum_k Qw[n,k] * o)      */
/* (the correction of x = s * (q - o)); npu_quant_matmul(x, W, deq_scale,    */
/* bias=quant_bias) -> BF16.                                                 */
/*   quantise: q = clamp(rint(x / s) + o, -128, 127) (binary32 divide, ties  */
/*             to even, the integer offset added after rounding)             */
/*   prepare:  binary32 steps a = bias / deq (0 without a bias or where deq  */
/*             is 0), c = float(sum_k Qw) * o, quant_bias = rint(a - c),     */
/*             saturated to int32                                            */
/*   matmul:   y = bf16_rne(float(acc + quant_bias[n]) * deq_scale[n])       */
/* s > 0 and finite, o in [-128, 127]; both per tensor.                      */
/* ------------------------------------------------------------------------ */

/* x [M,K] bf16 -> q [M,K] int8.  K % 16 == 0, x and q 16-byte aligned. */
W8A8_API w8a8_status w8a8_static_quant(const uint16_t* x, int64_t M, int64_t K, float input_scale,
                                       int32_t input_offset, int8_t* q, w8a8_stream_t stream);

/* Load time: w [N,K] int8 (checkpoint layout), weight_scale [N] fp32, bias
 * [N] bf16 or NULL -> deq_scale [N] fp32 and quant_bias [N] int32 (device
 * buffers).  K % 16 == 0, w 16-byte aligned. */
W8A8_API w8a8_status w8a8_static_prepare(const int8_t* w, int64_t N, int64_t K, const float* weight_scale,
                                         float input_scale, int32_t input_offset, const uint16_t* bias,
                                         float* deq_scale, int32_t* quant_bias, w8a8_stream_t stream);

/* q [M,K] int8 from w8a8_static_quant, w_packed as for w8a8_quant_matmul,
 * deq_scale / quant_bias from w8a8_static_prepare -> y [M,N] bf16.  Workspace
 * as w8a8_quant_matmul_workspace_bytes(M, N, K). */
W8A8_API w8a8_status w8a8_static_quant_matmul(const int8_t* q, int64_t M, int64_t K, const void* w_packed,
                                              const float* deq_scale, const int32_t* quant_bias, int64_t N,
                                              uint16_t* y, void* ws, size_t ws_bytes, w8a8_stream_t stream);

/* ------------------------------------------------------------------------ */
/* MXFP8 quantisation -- [P2] sections 3 and 5: weights re-quantised to      */
/* MXFP8 at load, activation rows at run time (group sizes [1,1,32]): an E4M3 */
/* payload with one E8M0 (power-of-two) scale per 32 values along K, the     */
/* normal scale algorithm: per group shared = floor(log2 max|v|) - 8,        */
/* clamped to [-127, 127], scale byte = shared + 127 (0 for a group of zeros, */
/* 0xFF for a group holding a NaN); elements v / 2^shared rounded to E4M3,   */
/* nearest even, saturating at +-448.                                        */
/* ------------------------------------------------------------------------ */

/* x [M,K] bf16 -> q [M,K] E4M3 bytes, scale [M,K/32] E8M0 bytes.  K % 32 == 0,
 * x and q 16-byte aligned.  Weights [N,K] (or [E*N,K]) take the same call. */
W8A8_API w8a8_status w8a8_mx_quant(const uint16_t* x, int64_t M, int64_t K, uint8_t* q, uint8_t* scale,
                                   w8a8_stream_t stream);

/* MXFP8 contraction ([P2] section 5, npu_quant_matmul with both E8M0
 * scales): qa [M,K] E4M3 + sa [M,K/32] E8M0 (from w8a8_mx_quant of the
 * activations), qw [N,K] E4M3 + sw [N,K/32] (of the weights) ->
 * y[m,n] = bf16( sum_g 2^(sa[m,g]-127) 2^(sw[n,g]-127) sum_{k in g} qa[m,k] qw[n,k] ),
 * accumulated in binary32 (so within a bound of the exact sum, not bit-exact).
 * K % 128 == 0; all pointers 16-byte aligned.  With K % 512 == 0 and N % 8 == 0
 * it runs on the block-scaled tensor cores (tcgen05 kind::mxf8f6f4, both
 * scales applied inside the MMA; w8a8_last_engine() reports W8A8_ENGINE_TC),
 * otherwise on the warp-level FP8 instruction (W8A8_ENGINE_WARP).  The call
 * has no workspace, so an exhausted bounded wait on the tensor-core path
 * (which only a stalled GPU produces) leaves y incomplete without a status. */
W8A8_API w8a8_status w8a8_mx_matmul(const uint8_t* qa, const uint8_t* sa, int64_t M, int64_t K, const uint8_t* qw,
                                    const uint8_t* sw, int64_t N, uint16_t* y, w8a8_stream_t stream);

/* ------------------------------------------------------------------------ */
/* MoE expert FFN -- [P1] §三 runner chain: (quantise only if no per-token   */
/* scale was supplied) -> W13 grouped matmul -> SwiGLU -> per-token INT8     */
/* requant -> W2 grouped matmul -> BF16.                                     */
/*   y13 = grouped(x, W13) rounded to bf16, gate = channels [0,I), up = [I,2I) */
/*   h   = bf16_rne((g * sigmoid(g)) * u), sigmoid(g) = 1 / (1 + exp(-g)) in  */
/*         binary32, exp by Cody-Waite reduction + degree-7 Taylor polynomial */
/*         evaluated with fused multiply-adds (Cody & Waite, 1980)            */
/*   (hq, hs) = dynamic quant of h over I;  y = grouped(hq, W2) -> bf16        */
/* ------------------------------------------------------------------------ */

W8A8_API size_t moe_workspace_bytes(int64_t R, int64_t H, int64_t I, int64_t E);

/* x: bf16 [R,H] when x_scale == NULL (quantised here), else int8 [R,H] already
 * quantised with per-token scales x_scale [R] (used as is, not quantised again).
 * group_list [E] int64 device counts; w13_packed from W8A8_PACK_GATE_UP
 * (+ optional W8A8_PACK_F16) of W13 [E,2I,H]; w13_scale [E,2I] in the ORIGINAL
 * channel order; w2_packed of W2 [E,H,I]; w2_scale [E,H]; y [R,H] bf16.
 * I % 64 == 0, H % 16 == 0. */
W8A8_API w8a8_status moe_w13_swiglu_requant_w2(const void* x, const float* x_scale,
                                      const int64_t* group_list, int64_t E, int64_t R, int64_t H,
                                      int64_t I, const void* w13_packed, const float* w13_scale,
                                      const void* w2_packed, const float* w2_scale, void* ws,
                                      size_t ws_bytes, uint16_t* y, w8a8_stream_t stream);

/* Offsets (bytes from ws) of the MoE intermediates kept in the workspace after
 * a call: 0 xq int8 [R,H], 1 xs fp32 [R], 2 h bf16 [R,I], 3 hq int8 [R,I],
 * 4 hs fp32 [R], 5 xq as fp16 [R,H], 6 hq as fp16 [R,I].  The codes are kept
 * in the form the contraction reads: int8 (0, 3) on shapes the warp engine
 * takes, integer-valued fp16 (5, 6) on shapes a tensor-core engine takes
 * (R >= 64 * E).  Returns -1 for an unknown index or a copy the shape does not
 * keep.  (Validation aid.) */
W8A8_API int64_t moe_workspace_offset(int64_t R, int64_t H, int64_t I, int64_t E, int which);

/* ------------------------------------------------------------------------ */
/* MoE routing around the expert chain -- [P1] §三: the DeepEP INT8 dispatch */
/* quantises each token's BF16 hidden row once (INT8 + one per-token scale); */
/* the Ascend runner input regroups the routed rows by expert, its           */
/* expert_tokens (rows per expert) being the grouped matmul's group_list;    */
/* topk_ids and topk_weights travel with the dispatch output.                */
/*   Every (token t, slot j) pair of topk_ids [T,k] is one routed row,       */
/*   R = T*k.  Routed rows are ordered by expert, then token, then slot:     */
/*   pos[t*k+j] is the routed row of (t, j), group_list[e] the number of     */
/*   pairs naming expert e.                                                  */
/*   combine: y[t,c] = bf16_rne(s) with s = 0, then for j = 0..k-1 in order  */
/*   s = s + w[t,j] * float(y_routed[pos[t,j], c]), every product and sum     */
/*   rounded to binary32 (no fused multiply-add).                            */
/* ------------------------------------------------------------------------ */

/* Workspace of moe_permute_quant (status word + per-chunk expert counts). */
W8A8_API size_t moe_route_workspace_bytes(int64_t T, int64_t k, int64_t E);

/* x: bf16 [T,H] token rows when x_scale == NULL (each token quantised once,
 * as w8a8_dynamic_quant would), else int8 [T,H] with per-token scales
 * x_scale [T] fp32 (copied, not quantised again).  topk_ids int64 [T,k].
 * Out (caller-owned device buffers): xq int8 [T*k,H] routed rows, xs fp32
 * [T*k], group_list int64 [E], pos int32 [T,k].  H % 16 == 0, x and xq 16-byte
 * aligned, k >= 1, T*k <= INT32_MAX, 1 <= E <= W8A8_MAX_EXPERTS.  ws: zero-filled,
 * at least moe_route_workspace_bytes(T, k, E).  An id outside [0,E) sets
 * W8A8_ERR_TOPK_IDS on the device: its pair gets pos = -1 and no routed row,
 * so the counts sum to less than T*k and a grouped call given them refuses
 * them. */
W8A8_API w8a8_status moe_permute_quant(const void* x, const float* x_scale, const int64_t* topk_ids,
                                       int64_t T, int64_t k, int64_t E, int64_t H, int8_t* xq, float* xs,
                                       int64_t* group_list, int32_t* pos, void* ws, size_t ws_bytes,
                                       w8a8_stream_t stream);

/* y_routed bf16 [T*k,H], pos int32 [T,k] (as moe_permute_quant writes it),
 * topk_weights fp32 [T,k] -> y bf16 [T,H].  H % 8 == 0, y_routed and y 16-byte
 * aligned.  ws: zero-filled, at least W8A8_STATUS_BYTES (only the status word
 * is used).  A pos outside [0,T*k) sets W8A8_ERR_TOPK_IDS on the device and its
 * term is left out of the sum. */
W8A8_API w8a8_status moe_unpermute_combine(const uint16_t* y_routed, const int32_t* pos,
                                           const float* topk_weights, int64_t T, int64_t k, int64_t H,
                                           uint16_t* y, void* ws, size_t ws_bytes, w8a8_stream_t stream);

/* The whole MoE layer from token rows and router output:
 * moe_permute_quant -> moe_w13_swiglu_requant_w2 on the routed rows (already
 * quantised, so not quantised again) -> moe_unpermute_combine.  Arguments as
 * in those calls; y bf16 [T,H].  I % 64 == 0, H % 16 == 0. */
W8A8_API size_t moe_layer_workspace_bytes(int64_t T, int64_t k, int64_t H, int64_t I, int64_t E);
W8A8_API w8a8_status moe_layer(const void* x, const float* x_scale, const int64_t* topk_ids,
                               const float* topk_weights, int64_t T, int64_t k, int64_t E, int64_t H,
                               int64_t I, const void* w13_packed, const float* w13_scale,
                               const void* w2_packed, const float* w2_scale, void* ws, size_t ws_bytes,
                               uint16_t* y, w8a8_stream_t stream);

/* Offsets (bytes from ws) of what moe_layer leaves in its workspace: 0..6 as
 * moe_workspace_offset with R = T*k (on shapes the tensor-core engine takes,
 * the routed codes are kept only as their fp16 copy, index 5), 7 group_list
 * int64 [E], 8 pos int32 [T,k], 9 y_routed bf16 [T*k,H].  -1 for an unknown
 * index.  (Validation aid.) */
W8A8_API int64_t moe_layer_workspace_offset(int64_t T, int64_t k, int64_t H, int64_t I, int64_t E, int which);

/* ------------------------------------------------------------------------ */
/* Dense quantised matmul without a caller workspace.  The pages have no     */
/* counterpart: this exists for callers that cannot allocate device memory   */
/* (a plugin interface without an allocator, a host that reserved all HBM    */
/* for its own pools, code where cudaMalloc is not allowed).                 */
/* ------------------------------------------------------------------------ */

/* Same arguments and result as w8a8_quant_matmul, minus the workspace.  The
 * scratch lives in a fixed 8 MiB device array inside the library (held by every
 * GPU that loads it until exit): problems whose split-K partial sums do not fit
 * (roughly M*N > 2M) run without splitting K, and a problem whose per-tile
 * counters alone do not fit (M*N beyond about 2^31) returns W8A8_ERR_WORKSPACE
 * before any launch.  The first call on a device
 * looks up the array's address, clears its status word, and should come
 * before any stream capture.  All calls share the array: calls that overlap
 * on the GPU race.  Errors found on the device go to the array's status
 * word (the first one stays); read them with
 * w8a8_quant_matmul_noalloc_status().  Allocates nothing. */
W8A8_API w8a8_status w8a8_quant_matmul_noalloc(const int8_t* q, const float* x_scale, int64_t M, int64_t K,
                                               const void* w_packed, const float* w_scale, int64_t N,
                                               const uint16_t* bias, uint16_t* y, w8a8_stream_t stream);

/* Synchronises `stream`, returns the status word that w8a8_quant_matmul_noalloc
 * calls on the current device wrote (W8A8_OK if none, else the first device
 * error since the last read, e.g. W8A8_ERR_PACKED for a packed weight whose
 * header does not match the call) and clears it.  Copies through the array's
 * symbol into a host local: allocates nothing. */
W8A8_API w8a8_status w8a8_quant_matmul_noalloc_status(w8a8_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Device status                                                             */
/* ------------------------------------------------------------------------ */

/* Synchronises `stream`, returns the status word that kernels wrote into the
 * workspace `ws` (W8A8_OK if none) and clears it.  `ws` is any workspace
 * passed to the calls above. */
W8A8_API w8a8_status w8a8_read_device_status(void* ws, w8a8_stream_t stream);

/* Self-check of the device-side failure path (the failure table at the end
 * of [P2], "Where It Breaks or Falls Back": a condition the operation cannot
 * meet comes back as an error code, not a crash).  Launches one CTA that waits
 * on an mbarrier nobody arrives on, with the bounded-wait helper of the
 * tensor-core kernels and a limit of `limit_us` microseconds (1 .. 2,000,000).
 * When the wait gives up the kernel writes W8A8_ERR_DEVICE_TIMEOUT to the status
 * word of `ws` (a zero-filled workspace of at least W8A8_STATUS_BYTES) and
 * returns; nothing else is in flight, so the context stays usable.  Read the
 * outcome with w8a8_read_device_status(). */
W8A8_API w8a8_status w8a8_selftest_bounded_wait(void* ws, uint32_t limit_us, w8a8_stream_t stream);

/* Engines a contraction can run on. */
enum {
  W8A8_ENGINE_NONE = 0,    /* no contraction launched yet on this thread (or M == 0) */
  W8A8_ENGINE_WARP = 1,    /* warp-level mma.sync engine (any shape) */
  W8A8_ENGINE_DECODE = 2,  /* tcgen05 decode engine: dense, M <= 64, int8 weights widened in tensor memory */
  W8A8_ENGINE_TC = 3,      /* tcgen05 engine for large M reading the fp16 weight copy (W8A8_PACK_F16) */
  W8A8_ENGINE_TC_I8 = 4    /* tcgen05 engine for large M on CTA pairs reading the INT8 weights, widened in
                              tensor memory (packs without the fp16 copy) */
};

/* The engine the last contraction launched by the calling host thread ran on
 * (w8a8_quant_matmul, w8a8_int8_matmul_acc, w8a8_grouped_matmul,
 * w8a8_grouped_matmul_acc, and the W2 contraction of
 * moe_w13_swiglu_requant_w2).  A host-side record: no device access, never
 * fails. */
W8A8_API int w8a8_last_engine(void);

#ifdef __cplusplus
}
#endif

#endif /* W8A8_H */
