/*
 * w8a8_oracle.c -- plain, slow, obviously-correct CPU oracle for the
 * W8A8_DYNAMIC linear layer and its MoE-expert counterpart.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  The product path
 * (the CUDA library) shares no code, header, table or helper with it.
 *
 * Sources (web pages; cited by title and section):
 *   [P1] "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子"
 *        §一  (quantisation recipe: act per_token int8 symmetric,
 *              weight per_channel int8 symmetric; W13 = gate_proj + up_proj,
 *              W2 = down_proj)
 *        §二  (Dense: npu_dynamic_quant -> INT8 [M,K] + per-token scale [M];
 *              npu_quant_matmul(q, W, weight_scale, pertoken_scale, bias,
 *              output_dtype=bf16) -> BF16 [M,N])
 *        §三  (MoE: npu_grouped_matmul over group_list = rows per expert;
 *              routed rows -> W13 grouped matmul -> SwiGLU -> requant -> W2
 *              grouped matmul -> BF16; an input that already carries a
 *              per-token scale is not quantised again)
 *        §四  (Atlas A3 operator contract: INT8 x1, INT8 x2, FLOAT32 per-token
 *              scale, BF16 output)
 *   [P2] "Qwen3.8-FP8 on Ascend 950: Why Weights Become MXFP8 at Load Time",
 *        sections 3 (re-quantisation to MXFP8) and 5 (MXFP8 activations and
 *        weights in the quantized matmul).
 *   [P3] "超大 MoE 的低比特推理：INT4、FP4 与量化感知训练", section
 *        on why quantisation-aware training is needed (its fake-quant
 *        helper takes the group absmax over qmax as the scale, divides by
 *        it, rounds half to even and clamps).
 *
 * Arithmetic (readings where the pages are silent are marked READING):
 *   quant    amax = max_k |x|, s = amax / 127 (binary32 divide),
 *            q = clamp(rint(x / s), -127, 127), rint = ties-to-even;
 *            READING: divide by s (not multiply by a reciprocal), as in [P3];
 *            READING: a row with amax == 0 gets s = 0 and q = 0.
 *   gemm     acc[m,n] = sum_k int32(q[m,k]) * int32(W[n,k])  (exact int32).
 *   epilogue t = float(acc) (RNE); t = t * s_x[m]; t = t * s_w[n];
 *            t = t + float(bias[n]) if bias; y = bf16_rne(t).  No FMA.
 *            READING: scale order x-scale first, bias added after scaling.
 *   grouped  group_list holds per-expert ROW COUNTS (not offsets); rows of
 *            expert e are [sum_{j<e} cnt_j, + cnt_e); counts >= 0, sum == R.
 *   swiglu   g = y13[r, j], u = y13[r, I + j] (bf16 values of the W13 output,
 *            gate = first I output channels, up = last I);
 *            h = bf16_rne((g * sigmoid(g)) * u), sigmoid(g) = 1 / (1 + exp(-g))
 *            in binary32, exp = the specification in oracle_exp_f32 below.
 *   requant  quant applied to h over its I columns.
 *   W2       grouped GEMM with W2 [E,H,I], no bias, BF16 out.
 *   skip     a non-NULL x_scale means x is already INT8 + per-token scale and
 *            is not quantised again.
 *   route / permute / combine (token rows in, token rows out): see the
 *            readings above oracle_moe_route.
 *   per-channel weight quantisation from BF16: above oracle_quantize_weight.
 *   static W8A8 (fixed input scale and offset, deq_scale, quant_bias):
 *            above oracle_static_quant.
 *   MXFP8 (E4M3 + one E8M0 scale per 32 along K, [P2] sections 3 and 5):
 *            above oracle_e4m3_from_f32.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp -shared
 * (contraction off: no hidden FMA may change a rounding).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_SHAPE 2
#define ORC_ERR_GROUP_LIST 5
#define ORC_ERR_ALLOC 9
#define ORC_ERR_TOPK_IDS 10

/* Largest reduction depth for which |acc| <= K * 128 * 127 < 2^31. */
#define ORC_MAX_K 131072

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------- bf16 -- */

float oracle_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even. */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
    return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays a quiet NaN */
  uint32_t keep_lsb = (u >> 16) & 1u;
  u += 0x7fffu + keep_lsb;
  return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------- exp (binary32) -- */
/*
 * e^x by Cody & Waite argument reduction (W. J. Cody, W. Waite, "Software
 * Manual for the Elementary Functions", 1980) and the degree-7 Taylor
 * polynomial of e^r, evaluated by Horner's rule with fused multiply-adds:
 *
 *   n  = rint(x * log2e)                 log2e  = binary32(1 / ln 2)
 *   r  = fma(-n, ln2_hi, x)              ln2_hi = ln 2 cut to 15 significant
 *   r  = fma(-n, ln2_lo, r)                       bits, so n*ln2_hi is exact
 *                                        ln2_lo = binary32(ln 2 - ln2_hi)
 *   p  = c7; p = fma(p, r, c_k) for k = 6..0,  c_k = binary32(1 / k!)
 *   e^x = (p * 2^(n/2)) * 2^(n - n/2)    (n/2 truncates; both factors normal)
 *
 * x > 89 gives +inf, x < -104 gives +0, NaN propagates.  Every step is a
 * correctly rounded binary32 operation, so any implementation that follows
 * these steps gets the same bits.  The constants are the mathematical values
 * above rounded to binary32 (hex given for checking).
 */
static float pow2_normal(int k) { /* 2^k for -126 <= k <= 127 */
  uint32_t u = (uint32_t)(k + 127) << 23;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

float oracle_exp_f32(float x) {
  if (x != x) return x;
  if (x > 89.0f) return INFINITY;
  if (x < -104.0f) return 0.0f;
  const float log2e = 1.44269502162933349609375f;          /* 0x3fb8aa3b */
  const float ln2_hi = 0.693145751953125f;                 /* 0x3f317200 */
  const float ln2_lo = 1.428606765330187045037746429443359375e-6f; /* 0x35bfbe8e */
  const float c7 = 1.98412701138295233249664306640625e-4f; /* 0x39500d01 = 1/5040 */
  const float c6 = 1.38888892251998186111450195312500e-3f; /* 0x3ab60b61 = 1/720  */
  const float c5 = 8.33333376795053482055664062500000e-3f; /* 0x3c088889 = 1/120  */
  const float c4 = 4.16666679084300994873046875000000e-2f; /* 0x3d2aaaab = 1/24   */
  const float c3 = 1.66666671633720397949218750000000e-1f; /* 0x3e2aaaab = 1/6    */
  const float c2 = 0.5f;
  const float c1 = 1.0f;
  const float c0 = 1.0f;
  float t = x * log2e;
  float n = rintf(t);
  float r = fmaf(-n, ln2_hi, x);
  r = fmaf(-n, ln2_lo, r);
  float p = c7;
  p = fmaf(p, r, c6);
  p = fmaf(p, r, c5);
  p = fmaf(p, r, c4);
  p = fmaf(p, r, c3);
  p = fmaf(p, r, c2);
  p = fmaf(p, r, c1);
  p = fmaf(p, r, c0);
  int ni = (int)n;
  int n1 = ni / 2; /* C division truncates toward zero */
  int n2 = ni - n1;
  return (p * pow2_normal(n1)) * pow2_normal(n2);
}

/* ------------------------------------------------ dynamic per-token quant -- */

/* [P1] §二 npu_dynamic_quant: BF16 x [M,K] -> INT8 q [M,K] + fp32 scale [M]. */
int oracle_dynamic_quant(const uint16_t* x, int64_t M, int64_t K, int8_t* q, float* scale) {
  if (M < 0 || K <= 0) return ORC_ERR_SHAPE;
  int64_t m;
#pragma omp parallel for schedule(static)
  for (m = 0; m < M; ++m) {
    const uint16_t* xr = x + m * K;
    int8_t* qr = q + m * K;
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      float a = fabsf(oracle_bf16_to_f32(xr[k]));
      if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    scale[m] = s;
    for (int64_t k = 0; k < K; ++k) {
      int8_t v = 0;
      if (s > 0.0f) {
        float t = oracle_bf16_to_f32(xr[k]) / s;
        float r = rintf(t);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        v = (int8_t)r;
      }
      qr[k] = v;
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------- INT8 GEMM, int32 -- */

/* acc[m,n] = sum_k q[m,k] * W[n,k]; W is [N,K] row-major (the checkpoint
 * layout of [P1] §二, output channel major). */
int oracle_int8_gemm_acc(const int8_t* q, int64_t M, int64_t K, const int8_t* w, int64_t N,
                         int32_t* acc) {
  if (M < 0 || N <= 0 || K <= 0 || K > ORC_MAX_K) return ORC_ERR_SHAPE;
  int64_t m;
#pragma omp parallel for schedule(static)
  for (m = 0; m < M; ++m) {
    const int8_t* qr = q + m * K;
    for (int64_t n = 0; n < N; ++n) {
      const int8_t* wr = w + n * K;
      int32_t a = 0;
      for (int64_t k = 0; k < K; ++k) a += (int32_t)qr[k] * (int32_t)wr[k];
      acc[m * N + n] = a;
    }
  }
  return ORC_OK;
}

/* One output element of the fused dequant epilogue ([P1] §二, §四). */
static uint16_t epilogue_one(int32_t acc, float sx, float sw, const uint16_t* bias, int64_t n) {
  float t = (float)acc;
  t = t * sx;
  t = t * sw;
  if (bias) t = t + oracle_bf16_to_f32(bias[n]);
  return oracle_f32_to_bf16(t);
}

int oracle_epilogue(const int32_t* acc, int64_t M, int64_t N, const float* x_scale,
                    const float* w_scale, const uint16_t* bias, uint16_t* y) {
  if (M < 0 || N <= 0) return ORC_ERR_SHAPE;
  int64_t m;
#pragma omp parallel for schedule(static)
  for (m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n)
      y[m * N + n] = epilogue_one(acc[m * N + n], x_scale[m], w_scale[n], bias, n);
  return ORC_OK;
}

/* [P1] §二 npu_quant_matmul: INT8 x INT8 -> INT32 -> * x_scale * w_scale (+bias) -> BF16. */
int oracle_quant_matmul(const int8_t* q, const float* x_scale, int64_t M, int64_t K,
                        const int8_t* w, const float* w_scale, int64_t N, const uint16_t* bias,
                        uint16_t* y) {
  if (M < 0 || N <= 0 || K <= 0 || K > ORC_MAX_K) return ORC_ERR_SHAPE;
  int64_t m;
#pragma omp parallel for schedule(static)
  for (m = 0; m < M; ++m) {
    const int8_t* qr = q + m * K;
    for (int64_t n = 0; n < N; ++n) {
      const int8_t* wr = w + n * K;
      int32_t a = 0;
      for (int64_t k = 0; k < K; ++k) a += (int32_t)qr[k] * (int32_t)wr[k];
      y[m * N + n] = epilogue_one(a, x_scale[m], w_scale[n], bias, n);
    }
  }
  return ORC_OK;
}

/* ------------------------------------------- per-channel weight quant -- */
/*
 * [P1] §一 (msModelSlim recipe: weight scope per_channel, dtype int8,
 * symmetric) and §二 (the checkpoint weight [N,K] is already INT8 at load:
 * the quantisation happened offline, from the BF16 weight).
 * READING: per channel = per output channel n, over its K inputs; the
 * symmetric recipe is the activation one: s[n] = amax_k |W[n,k]| / 127,
 * q = clamp(rint(W / s), -127, 127), ties to even; an all-zero channel gets
 * s = 0 and q = 0.  W is BF16 [E,N,K] (E = 1 for a dense layer); scales are
 * fp32 [E,N] in channel order.
 */
int oracle_quantize_weight(const uint16_t* w, int64_t E, int64_t N, int64_t K, int8_t* q, float* scale) {
  if (E <= 0 || N <= 0 || K <= 0) return ORC_ERR_SHAPE;
  for (int64_t e = 0; e < E; ++e) {
    /* each expert's N channels, one at a time: the per-row quantiser on one row */
    for (int64_t n = 0; n < N; ++n) {
      const int64_t row = e * N + n;
      const int rc = oracle_dynamic_quant(w + row * K, 1, K, q + row * K, scale + row);
      if (rc) return rc;
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------- static W8A8 -- */
/*
 * [P1] closing comparison of the static recipe: BF16 X is quantised by
 * npu_quantize with a fixed (calibrated) input_scale / input_offset; at load
 * time deq_scale = input_scale * weight_scale and
 * quant_bias = round(fp_bias / deq_scale - sum_k(Qw[n,k]) * input_offset)
 * (int32); npu_quant_matmul(x, W, deq_scale, bias=quant_bias) gives BF16 Y.
 * The correction term is that of x = input_scale * (q - input_offset).
 *
 * READING (quantise): q = clamp(rint(x / s) + o, -128, 127): binary32 divide,
 *   ties to even, the integer offset added to the integer code (exact), the
 *   full int8 range (the code is no longer symmetric).  s, o per tensor.
 * READING (prepare): a = float(bias[n]) / deq[n] (0 without a bias),
 *   c = float(sum_k Qw[n,k]) * float(o) (the sum is exact), quant_bias =
 *   rint(a - c) (binary32 steps, ties to even), saturated to int32.
 *   deq[n] = s * weight_scale[n] (binary32).  Where deq is 0 (an all-zero
 *   weight channel) the bias cannot be expressed: a = 0 (y is 0 there).
 * READING (matmul): y = bf16_rne(float(acc + quant_bias[n]) * deq[n]); the
 *   integer bias is added to the accumulator before the one conversion.
 */
int oracle_static_quant(const uint16_t* x, int64_t M, int64_t K, float s, int32_t o, int8_t* q) {
  if (M < 0 || K <= 0 || !(s > 0.0f)) return ORC_ERR_SHAPE;
  int64_t m;
#pragma omp parallel for schedule(static)
  for (m = 0; m < M; ++m)
    for (int64_t k = 0; k < K; ++k) {
      const float t = oracle_bf16_to_f32(x[m * K + k]) / s;
      double c = (double)rintf(t) + (double)o;
      if (c > 127.0) c = 127.0;
      if (c < -128.0) c = -128.0;
      if (t != t) c = 0.0; /* NaN input: not produced by the generator */
      q[m * K + k] = (int8_t)c;
    }
  return ORC_OK;
}

int oracle_static_prepare(const int8_t* w, int64_t N, int64_t K, const float* w_scale, float s, int32_t o,
                          const uint16_t* bias, float* deq, int32_t* quant_bias) {
  if (N <= 0 || K <= 0) return ORC_ERR_SHAPE;
  for (int64_t n = 0; n < N; ++n) {
    int64_t sum = 0;
    for (int64_t k = 0; k < K; ++k) sum += w[n * K + k];
    deq[n] = s * w_scale[n];
    const float a = (bias && deq[n] != 0.0f) ? oracle_bf16_to_f32(bias[n]) / deq[n] : 0.0f;
    const float c = (float)sum * (float)o;
    const float t = rintf(a - c);
    double v = (double)t;
    if (v > 2147483647.0) v = 2147483647.0;
    if (v < -2147483648.0) v = -2147483648.0;
    quant_bias[n] = (int32_t)v;
  }
  return ORC_OK;
}

int oracle_static_quant_matmul(const int8_t* q, int64_t M, int64_t K, const int8_t* w, int64_t N,
                               const float* deq, const int32_t* quant_bias, uint16_t* y) {
  if (M < 0 || N <= 0 || K <= 0 || K > ORC_MAX_K) return ORC_ERR_SHAPE;
  int32_t* acc = malloc((size_t)(M > 0 ? M : 1) * (size_t)N * sizeof(int32_t));
  if (!acc) return ORC_ERR_ALLOC;
  int rc = oracle_int8_gemm_acc(q, M, K, w, N, acc);
  if (rc == ORC_OK)
    for (int64_t m = 0; m < M; ++m)
      for (int64_t n = 0; n < N; ++n) {
        const float t = (float)((int64_t)acc[m * N + n] + (int64_t)quant_bias[n]);
        y[m * N + n] = oracle_f32_to_bf16(t * deq[n]);
      }
  free(acc);
  return rc;
}

/* ---------------------------------------------------------- grouped GEMM -- */

int oracle_check_group_list(const int64_t* group_list, int64_t E, int64_t R) {
  int64_t total = 0;
  for (int64_t e = 0; e < E; ++e) {
    if (group_list[e] < 0) return ORC_ERR_GROUP_LIST;
    total += group_list[e];
  }
  return total == R ? ORC_OK : ORC_ERR_GROUP_LIST;
}

/* [P1] §三 npu_grouped_matmul(x, weight, scale, per_token_scale, group_list):
 * rows of expert e use W[e] ([E,N,K]) and w_scale[e] ([E,N]).  acc (optional,
 * [R,N] int32) receives the exact accumulators. */
int oracle_grouped_matmul(const int8_t* q, const float* x_scale, const int64_t* group_list,
                          int64_t E, int64_t R, int64_t K, const int8_t* w,
                          const float* w_scale, int64_t N, uint16_t* y, int32_t* acc) {
  if (E <= 0 || R < 0 || N <= 0 || K <= 0 || K > ORC_MAX_K) return ORC_ERR_SHAPE;
  if (oracle_check_group_list(group_list, E, R) != ORC_OK) return ORC_ERR_GROUP_LIST;
  int64_t off = 0;
  for (int64_t e = 0; e < E; ++e) {
    const int64_t rows = group_list[e];
    const int8_t* we = w + e * N * K;
    const float* se = w_scale + e * N;
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = off; r < off + rows; ++r) {
      const int8_t* qr = q + r * K;
      for (int64_t n = 0; n < N; ++n) {
        const int8_t* wr = we + n * K;
        int32_t a = 0;
        for (int64_t k = 0; k < K; ++k) a += (int32_t)qr[k] * (int32_t)wr[k];
        if (acc) acc[r * N + n] = a;
        y[r * N + n] = epilogue_one(a, x_scale[r], se[n], NULL, n);
      }
    }
    off += rows;
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------- SwiGLU -- */

/* [P1] §三 runner chain "W13 Grouped MatMul -> SwiGLU": y13 [R, 2I] bf16 ->
 * h [R, I] bf16. */
int oracle_swiglu(const uint16_t* y13, int64_t R, int64_t I, uint16_t* h) {
  if (R < 0 || I <= 0) return ORC_ERR_SHAPE;
  int64_t r;
#pragma omp parallel for schedule(static)
  for (r = 0; r < R; ++r) {
    for (int64_t j = 0; j < I; ++j) {
      float g = oracle_bf16_to_f32(y13[r * 2 * I + j]);
      float u = oracle_bf16_to_f32(y13[r * 2 * I + I + j]);
      float e = oracle_exp_f32(-g);
      float sig = 1.0f / (1.0f + e);
      float v = (g * sig) * u;
      h[r * I + j] = oracle_f32_to_bf16(v);
    }
  }
  return ORC_OK;
}

/* ---------------------------------------------------- MoE expert FFN chain -- */
/*
 * [P1] §三: Routed Hidden -> (quant if no per-token scale) -> W13 GMM ->
 * SwiGLU -> Requant -> W2 GMM -> BF16.
 *   x        bf16 [R,H] when x_scale == NULL, else int8 [R,H]
 *   x_scale  fp32 [R] or NULL
 *   w13      int8 [E,2I,H], s13 fp32 [E,2I];  w2 int8 [E,H,I], s2 fp32 [E,H]
 *   y        bf16 [R,H]
 * Optional intermediates (NULL to skip): xq [R,H] int8, xs [R], y13 [R,2I]
 * bf16, h [R,I] bf16, hq [R,I] int8, hs [R].
 */
int oracle_moe_w13_swiglu_requant_w2(const void* x, const float* x_scale,
                                     const int64_t* group_list, int64_t E, int64_t R,
                                     int64_t H, int64_t I, const int8_t* w13, const float* s13,
                                     const int8_t* w2, const float* s2, uint16_t* y,
                                     int8_t* xq_out, float* xs_out, uint16_t* y13_out,
                                     uint16_t* h_out, int8_t* hq_out, float* hs_out) {
  if (E <= 0 || R < 0 || H <= 0 || I <= 0) return ORC_ERR_SHAPE;
  if (oracle_check_group_list(group_list, E, R) != ORC_OK) return ORC_ERR_GROUP_LIST;
  const size_t r = (size_t)R;
  int8_t* xq = malloc(r * (size_t)H + 1);
  float* xs = malloc(r * sizeof(float) + 4);
  uint16_t* y13 = malloc(r * 2 * (size_t)I * sizeof(uint16_t) + 2);
  uint16_t* h = malloc(r * (size_t)I * sizeof(uint16_t) + 2);
  int8_t* hq = malloc(r * (size_t)I + 1);
  float* hs = malloc(r * sizeof(float) + 4);
  int rc = ORC_ERR_ALLOC;
  if (!xq || !xs || !y13 || !h || !hq || !hs) goto done;

  if (x_scale == NULL) {
    rc = oracle_dynamic_quant((const uint16_t*)x, R, H, xq, xs);
    if (rc) goto done;
  } else {
    memcpy(xq, x, r * (size_t)H);
    memcpy(xs, x_scale, r * sizeof(float));
  }
  rc = oracle_grouped_matmul(xq, xs, group_list, E, R, H, w13, s13, 2 * I, y13, NULL);
  if (rc) goto done;
  rc = oracle_swiglu(y13, R, I, h);
  if (rc) goto done;
  rc = oracle_dynamic_quant(h, R, I, hq, hs);
  if (rc) goto done;
  rc = oracle_grouped_matmul(hq, hs, group_list, E, R, I, w2, s2, H, y, NULL);
  if (rc) goto done;

  if (xq_out) memcpy(xq_out, xq, r * (size_t)H);
  if (xs_out) memcpy(xs_out, xs, r * sizeof(float));
  if (y13_out) memcpy(y13_out, y13, r * 2 * (size_t)I * sizeof(uint16_t));
  if (h_out) memcpy(h_out, h, r * (size_t)I * sizeof(uint16_t));
  if (hq_out) memcpy(hq_out, hq, r * (size_t)I);
  if (hs_out) memcpy(hs_out, hs, r * sizeof(float));
done:
  free(xq);
  free(xs);
  free(y13);
  free(h);
  free(hq);
  free(hs);
  return rc;
}

/* ------------------------------------------- routing permute and combine -- */
/*
 * [P1] §三 (DeepEP INT8 dispatch and the Ascend runner input): the dispatch
 * turns each token's BF16 hidden row into INT8 + one per-token scale, and the
 * runner input regroups the routed rows by expert with expert_tokens (rows
 * per expert) as its group list; topk_ids / topk_weights come with it.
 *
 * READING (route): every (token t, slot j) pair of topk_ids [T,k] is one
 *   routed row; R = T*k.  Rows are ordered by expert, then token, then slot;
 *   pos[t*k + j] is the routed row of (t, j) and group_list[e] the number of
 *   pairs naming expert e.  An id outside [0, E) is an error.
 * READING (permute + quant): a token is quantised once over its H columns
 *   (the dispatch quantises before it sends) and its codes and scale are
 *   copied to each of its routed rows; an INT8 token with a scale is copied
 *   as it is.
 * READING (combine): y[t, c] = bf16_rne(s), s = 0 then, for j = 0..k-1 in
 *   order, s = s + w[t,j] * float(y_routed[pos[t,j], c]) with each product
 *   and sum rounded to binary32 (no FMA); the weights are binary32.
 */
int oracle_moe_route(const int64_t* topk_ids, int64_t T, int64_t k, int64_t E,
                     int64_t* group_list, int32_t* pos) {
  if (T < 0 || k <= 0 || E <= 0 || T * k > (int64_t)INT32_MAX) return ORC_ERR_SHAPE;
  const int64_t n = T * k;
  for (int64_t i = 0; i < n; ++i)
    if (topk_ids[i] < 0 || topk_ids[i] >= E) return ORC_ERR_TOPK_IDS;
  int64_t row = 0;
  for (int64_t e = 0; e < E; ++e) {
    int64_t cnt = 0;
    for (int64_t i = 0; i < n; ++i) /* i = t*k + j: token-major, then slot */
      if (topk_ids[i] == e) {
        pos[i] = (int32_t)row;
        ++row;
        ++cnt;
      }
    group_list[e] = cnt;
  }
  return ORC_OK;
}

/* x: BF16 [T,H] (x_scale NULL) or INT8 [T,H] with x_scale [T].
 * Out: xq [T*k,H] int8, xs [T*k], group_list [E], pos [T*k]. */
int oracle_moe_permute_quant(const void* x, const float* x_scale, const int64_t* topk_ids,
                             int64_t T, int64_t k, int64_t E, int64_t H, int8_t* xq, float* xs,
                             int64_t* group_list, int32_t* pos) {
  if (H <= 0) return ORC_ERR_SHAPE;
  int rc = oracle_moe_route(topk_ids, T, k, E, group_list, pos);
  if (rc) return rc;
  const size_t t_rows = (size_t)T;
  int8_t* qt = malloc(t_rows * (size_t)H + 1);
  float* st = malloc(t_rows * sizeof(float) + 4);
  rc = ORC_ERR_ALLOC;
  if (!qt || !st) goto done;
  if (x_scale == NULL) {
    rc = oracle_dynamic_quant((const uint16_t*)x, T, H, qt, st);
    if (rc) goto done;
  } else {
    memcpy(qt, x, t_rows * (size_t)H);
    memcpy(st, x_scale, t_rows * sizeof(float));
  }
  for (int64_t t = 0; t < T; ++t)
    for (int64_t j = 0; j < k; ++j) {
      const int64_t r = pos[t * k + j];
      memcpy(xq + r * H, qt + t * H, (size_t)H);
      xs[r] = st[t];
    }
  rc = ORC_OK;
done:
  free(qt);
  free(st);
  return rc;
}

/* y_routed: BF16 [R,H] with R = T*k; pos [T*k]; w fp32 [T*k] -> y BF16 [T,H]. */
int oracle_moe_unpermute_combine(const uint16_t* y_routed, const int32_t* pos, const float* w,
                                 int64_t T, int64_t k, int64_t H, uint16_t* y) {
  if (T < 0 || k <= 0 || H <= 0) return ORC_ERR_SHAPE;
  const int64_t R = T * k;
  for (int64_t i = 0; i < R; ++i)
    if (pos[i] < 0 || pos[i] >= R) return ORC_ERR_SHAPE;
  int64_t t;
#pragma omp parallel for schedule(static)
  for (t = 0; t < T; ++t)
    for (int64_t c = 0; c < H; ++c) {
      float s = 0.0f;
      for (int64_t j = 0; j < k; ++j) {
        const float v = oracle_bf16_to_f32(y_routed[(int64_t)pos[t * k + j] * H + c]);
        const float p = w[t * k + j] * v;
        s = s + p;
      }
      y[t * H + c] = oracle_f32_to_bf16(s);
    }
  return ORC_OK;
}

/* Whole MoE layer from token rows and router output: permute + quant, the
 * expert chain on the routed rows (pre-quantised, so not quantised again),
 * then the weighted combine.  y_routed_out [T*k,H] (optional) receives the
 * expert chain's BF16 output. */
int oracle_moe_layer(const void* x, const float* x_scale, const int64_t* topk_ids,
                     const float* topk_weights, int64_t T, int64_t k, int64_t E, int64_t H,
                     int64_t I, const int8_t* w13, const float* s13, const int8_t* w2,
                     const float* s2, uint16_t* y, uint16_t* y_routed_out) {
  if (T < 0 || k <= 0 || E <= 0 || H <= 0 || I <= 0) return ORC_ERR_SHAPE;
  const size_t R = (size_t)(T * k);
  int8_t* xq = malloc(R * (size_t)H + 1);
  float* xs = malloc(R * sizeof(float) + 4);
  int64_t* gl = malloc((size_t)E * sizeof(int64_t));
  int32_t* pos = malloc(R * sizeof(int32_t) + 4);
  uint16_t* yr = malloc(R * (size_t)H * sizeof(uint16_t) + 2);
  int rc = ORC_ERR_ALLOC;
  if (!xq || !xs || !gl || !pos || !yr) goto done;
  rc = oracle_moe_permute_quant(x, x_scale, topk_ids, T, k, E, H, xq, xs, gl, pos);
  if (rc) goto done;
  rc = oracle_moe_w13_swiglu_requant_w2(xq, xs, gl, E, (int64_t)R, H, I, w13, s13, w2, s2, yr,
                                        NULL, NULL, NULL, NULL, NULL, NULL);
  if (rc) goto done;
  rc = oracle_moe_unpermute_combine(yr, pos, topk_weights, T, k, H, y);
  if (rc) goto done;
  if (y_routed_out) memcpy(y_routed_out, yr, R * (size_t)H * sizeof(uint16_t));
done:
  free(xq);
  free(xs);
  free(gl);
  free(pos);
  free(yr);
  return rc;
}

/* ------------------------------------------------------------ MXFP8 -- */
/*
 * [P2] "Qwen3.8-FP8 on Ascend 950: Why Weights Become MXFP8 at Load Time",
 * sections 3 and 5: the MXFP8 contract -- an E4M3 payload with one E8M0
 * (power-of-two) scale per 32 values along the reduction axis K, for the
 * weights (re-quantised at load) and for each activation row (quantised at
 * run time, group sizes [1,1,32]); the matmul consumes both scales.
 *
 * READING (scale): the pages name the scale algorithm only as "0, the normal
 * case".  Taken as the OCP Microscaling rule: for each group of 32 values,
 * shared = floor(log2(max |v|)) - 8 (8 = the largest E4M3 exponent),
 * clamped to [-127, 127]; the E8M0 byte is shared + 127; a group of zeros
 * gets byte 0.  Elements: v / 2^shared (exact) rounded to E4M3 to nearest,
 * ties to even, saturating at +-448 (the E4M3 "fn" variant: no infinities,
 * NaN = S.1111.111).
 * READING (matmul): y[m,n] = bf16_rne( sum_g Sa[m,g] * Sw[n,g] *
 * sum_{k in g} a[m,k] * w[n,k] ) with the sum taken in float64 here (the
 * products of E4M3 values and powers of two are exact); a tensor-core
 * implementation accumulates in binary32, so parity is within a bound.
 */
static double pow2d(int e) { return ldexp(1.0, e); }

/* E4M3 (fn) byte of a binary32 value: round to nearest even, saturate. */
uint8_t oracle_e4m3_from_f32(float v) {
  if (v != v) return 0x7F;
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  const double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;             /* largest finite: 1.75 * 2^8 */
  if (a < pow2d(-6)) {                            /* subnormal steps of 2^-9 */
    const double m = nearbyint(a / pow2d(-9));    /* 0..8; 8 is the smallest normal */
    return sign | (uint8_t)m;
  }
  int e;
  (void)frexp(a, &e);
  e -= 1;                                         /* a in [2^e, 2^(e+1)) */
  double m = nearbyint((a / pow2d(e) - 1.0) * 8.0);  /* 3 mantissa bits */
  if (m == 8.0) {
    m = 0.0;
    e += 1;
  }
  if (e > 8) return sign | 0x7E;
  return sign | (uint8_t)(((e + 7) << 3) | (int)m);
}

float oracle_e4m3_to_f32(uint8_t b) {
  const int sign = b & 0x80;
  const int ex = (b >> 3) & 0xF;
  const int man = b & 0x7;
  if (ex == 0xF && man == 0x7) return NAN;
  double v = ex == 0 ? man * pow2d(-9) : (1.0 + man / 8.0) * pow2d(ex - 7);
  return (float)(sign ? -v : v);
}

/* x bf16 [M,K] (K % 32 == 0) -> q E4M3 [M,K], scale E8M0 [M,K/32]. */
int oracle_mx_quant(const uint16_t* x, int64_t M, int64_t K, uint8_t* q, uint8_t* scale) {
  if (M < 0 || K <= 0 || K % 32 != 0) return ORC_ERR_SHAPE;
  const int64_t G = K / 32;
  int64_t m;
#pragma omp parallel for schedule(static)
  for (m = 0; m < M; ++m)
    for (int64_t g = 0; g < G; ++g) {
      const uint16_t* xs = x + m * K + g * 32;
      float amax = 0.0f;
      int nan = 0;
      for (int i = 0; i < 32; ++i) {
        const float v = oracle_bf16_to_f32(xs[i]);
        if (v != v) nan = 1;
        else if (fabsf(v) > amax) amax = fabsf(v);
      }
      int shared = -127;
      if (amax > 0.0f) {
        int e;
        (void)frexp((double)amax, &e);
        shared = (e - 1) - 8;
        if (shared < -127) shared = -127;
        if (shared > 127) shared = 127;
      }
      scale[m * G + g] = nan ? 0xFF : (uint8_t)(shared + 127);
      for (int i = 0; i < 32; ++i) {
        const double v = (double)oracle_bf16_to_f32(xs[i]) / pow2d(shared);
        q[m * K + g * 32 + i] = oracle_e4m3_from_f32((float)v);
      }
    }
  return ORC_OK;
}

/* bf16 bits of a double, rounded to nearest even (normal range). */
static uint16_t bf16_from_f64(double x) {
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  int e;
  (void)frexp(fabs(x), &e);
  const double ulp = pow2d((e - 1) - 7);
  const double r = nearbyint(x / ulp) * ulp;      /* exact: a bf16 value */
  const float f = (float)r;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

/* qa E4M3 [M,K] + sa E8M0 [M,K/32], qw E4M3 [N,K] + sw E8M0 [N,K/32] -> y bf16 [M,N]. */
int oracle_mx_matmul(const uint8_t* qa, const uint8_t* sa, int64_t M, int64_t K, const uint8_t* qw,
                     const uint8_t* sw, int64_t N, uint16_t* y) {
  if (M < 0 || N <= 0 || K <= 0 || K % 32 != 0) return ORC_ERR_SHAPE;
  const int64_t G = K / 32;
  int64_t m;
#pragma omp parallel for schedule(static)
  for (m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t g = 0; g < G; ++g) {
        double part = 0.0;
        for (int i = 0; i < 32; ++i)
          part += (double)oracle_e4m3_to_f32(qa[m * K + g * 32 + i]) *
                  (double)oracle_e4m3_to_f32(qw[n * K + g * 32 + i]);
        acc += part * pow2d((int)sa[m * G + g] - 127) * pow2d((int)sw[n * G + g] - 127);
      }
      y[m * N + n] = bf16_from_f64(acc);
    }
  return ORC_OK;
}
