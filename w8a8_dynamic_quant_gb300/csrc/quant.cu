// quant.cu -- K1: dynamic per-token INT8 quantisation of BF16 activations.
//
// Page "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子":
//   §一 recipe: activations per_token, int8, symmetric;
//   §二 npu_dynamic_quant(x) -> INT8 [M,K] + per-token scale [M];
//   §三 HiddenStatesDynamicQuant (the same operation on MoE hidden states and
//       as the Requant after SwiGLU).
//   amax = max_k |x|, s = amax / 127 (binary32 divide), q = clamp(rint(x/s),
//   -127, 127) with ties to even; an all-zero row gets s = 0, q = 0.
//
// HBM-bound: 2 bytes read + 1 byte written per element (+4 bytes per row).
// The MoE routing permute uses the same kernels with a scatter: a token row is
// quantised once and its codes and scale go to each of its k routed rows (the
// DeepEP INT8 dispatch of §三 quantises before it sends), and the offline
// weight quantisation (§一: weight per_channel, int8, symmetric) uses them
// with each output channel as a row, written straight into a packed buffer.
// Each row is read once with 16-byte vector loads and held in registers
// between the absmax pass and the quantise pass; absmax is reduced with warp
// shuffles (and shared memory across the warps of a CTA).
#include <type_traits>

#include "kernels.cuh"

namespace w8a8 {

namespace {

// max |x| over 8 bf16 (two per 32-bit word): sign bits cleared, then packed bf16 maxima; the larger
// half of the result, widened to binary32 (exact).
__device__ __forceinline__ float absmax8(const uint4& v) {
  uint32_t m01, m23, m;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(m01) : "r"(v.x & 0x7fff7fffu), "r"(v.y & 0x7fff7fffu));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(m23) : "r"(v.z & 0x7fff7fffu), "r"(v.w & 0x7fff7fffu));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(m01), "r"(m23));
  return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
}

// y + 1.5 * 2^23 rounds y (|y| < 2^22) to an integer, ties to even, held in the low mantissa bits: the
// sum's low byte is the two's-complement int8 code and (sum - 1.5 * 2^23) the code as a float.
constexpr float kRoundMagic = 12582912.0f;

// The 8 codes of a chunk of 8 bf16 (x[e] = element e), as sums m[e] = code + kRoundMagic.
// rint(x / s) with the quotient rounded to binary32 first (round half to even), clamped to +-127;
// s > 0 and rs = the binary32 reciprocal of s, or s = rs = 0 (an all-zero row: every code 0).  y = x * rs is within |x / s| * 2^-23 + 2^-18 <= 2^-15 of
// the correctly rounded quotient (|x / s| <= 128), so when y is more than 2^-14 from the nearest
// half-integer both lie strictly inside the same rounding interval and round to the same integer, with
// |code| <= 127 (|y| <= 127 * (1 + 2^-22)); otherwise (rare), and for non-finite y, the whole chunk
// takes the quotient itself and the clamp.
// Two binary32 values in one 64-bit register, for the paired instructions below (each lane of
// mul/add/fma.rn.f32x2 is the correctly rounded binary32 operation of its own operands).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ void codes8(const uint4& v, float s, float rs, float (&m)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const uint64_t rs2 = pk2(rs, rs), mg2 = pk2(kRoundMagic, kRoundMagic), nmg2 = pk2(-kRoundMagic, -kRoundMagic),
                 neg1 = pk2(-1.0f, -1.0f);
  float dmax = 0.0f;  // max |y - rint(y)| over the chunk; NaN if any y is not finite
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // elements 2i, 2i+1 side by side
    const uint64_t x2 = pk2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
    uint64_t y2, m2, r2, t2;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y2) : "l"(x2), "l"(rs2));         // y = x * rs
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(m2) : "l"(y2), "l"(mg2));         // m = y + magic
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r2) : "l"(m2), "l"(nmg2));        // rint(y), exact
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(t2) : "l"(r2), "l"(neg1), "l"(y2));  // y - rint(y), exact
    float t0, t1;
    upk2(t2, t0, t1);
    upk2(m2, m[2 * i], m[2 * i + 1]);
    asm("max.NaN.f32 %0, %0, %1;" : "+f"(dmax) : "f"(fabsf(t0)));
    asm("max.NaN.f32 %0, %0, %1;" : "+f"(dmax) : "f"(fabsf(t1)));
  }
  if (__builtin_expect(!(dmax < 0.5f - 0x1p-14f), 0)) {
    float x[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int r = max(-127, min(127, __float2int_rn(__fdiv_rn(x[e], s))));
      m[e] = __fadd_rn(static_cast<float>(r), kRoundMagic);
    }
  }
}

// int8 codes of a chunk (low bytes of the sums) packed in a uint2.
__device__ __forceinline__ uint2 pack_i8(const float (&m)[8]) {
  uint32_t u[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) u[e] = __float_as_uint(m[e]);
  return make_uint2(__byte_perm(__byte_perm(u[0], u[1], 0x0040), __byte_perm(u[2], u[3], 0x0040), 0x5410),
                    __byte_perm(__byte_perm(u[4], u[5], 0x0040), __byte_perm(u[6], u[7], 0x0040), 0x5410));
}

// the codes as integer-valued fp16 (exact) packed in a uint4.
__device__ __forceinline__ uint4 pack_f16(const float (&m)[8]) {
  uint32_t h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm("cvt.rn.f16x2.f32 %0, %1, %2;"
        : "=r"(h[i])
        : "f"(__fsub_rn(m[2 * i + 1], kRoundMagic)), "f"(__fsub_rn(m[2 * i], kRoundMagic)));
  return make_uint4(h[0], h[1], h[2], h[3]);
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Where a quantised row goes: n() destinations, codes to row(m, j), the scale to scale_row(m, j); an
// index < 0 is skipped.
// Plain quantisation: row m of the output.
struct RowId {
  __device__ __forceinline__ int n() const { return 1; }
  __device__ __forceinline__ int64_t row(int64_t m, int) const { return m; }
  __device__ __forceinline__ int64_t scale_row(int64_t m, int) const { return m; }
};
// The MoE routing permute: the k routed rows dst[m*k + j] of token m, each with the same codes and scale
// (an index < 0 belongs to a pair whose expert id was rejected).
struct RowScatter {
  const int32_t* dst;
  int k;
  __device__ __forceinline__ int n() const { return k; }
  __device__ __forceinline__ int64_t row(int64_t m, int j) const { return dst[m * k + j]; }
  __device__ __forceinline__ int64_t scale_row(int64_t m, int j) const { return dst[m * k + j]; }
};
// Weight channels into a packed buffer: channel m = e*N + c goes to its packed row (the W13 gate/up
// interleave when asked), its scale stays in channel order.
struct RowPack {
  int64_t N;
  bool gate_up;
  __device__ __forceinline__ int n() const { return 1; }
  __device__ __forceinline__ int64_t row(int64_t m, int) const {
    if (!gate_up) return m;
    const int64_t e = m / N, c = m % N, I = N / 2;
    // inverse of gate_up_orig_row: gate channel c -> block c/64, first half; up channel -> second half
    const int64_t g = c < I ? c : c - I;
    return e * N + (g / kGateUpBlock) * 2 * kGateUpBlock + (c < I ? 0 : kGateUpBlock) + g % kGateUpBlock;
  }
  __device__ __forceinline__ int64_t scale_row(int64_t m, int) const { return m; }
};

// OUT: 0 = int8 codes into q; 1 = the same codes as fp16 into q16; 2 = both (each code computed once).
// s = rs = 0 (an all-zero row) gives zero codes.
template <int OUT, class D>
__device__ __forceinline__ void store8(const uint4& v, float s, float rs, int64_t row, int64_t K, int64_t idx,
                                       void* q, uint16_t* q16, const D& d) {
  float m[8];
  codes8(v, s, rs, m);
  uint2 c = make_uint2(0u, 0u);
  uint4 f = make_uint4(0u, 0u, 0u, 0u);
  if constexpr (OUT != 1) c = pack_i8(m);
  if constexpr (OUT != 0) f = pack_f16(m);
  for (int j = 0; j < d.n(); ++j) {
    const int64_t r = d.row(row, j);
    if (r < 0) continue;
    if (OUT != 1) reinterpret_cast<uint2*>(static_cast<int8_t*>(q) + r * K)[idx] = c;
    if (OUT != 0) reinterpret_cast<uint4*>(q16 + r * K)[idx] = f;
  }
}
// The same for a plain row (one destination, row m of the output) whose output rows were located once:
// q8 / q16r point at chunk 0 of the row.
template <int OUT>
__device__ __forceinline__ void store8_row(const uint4& v, float s, float rs, int64_t idx, uint2* q8, uint4* q16r) {
  float m[8];
  codes8(v, s, rs, m);
  if constexpr (OUT != 1) q8[idx] = pack_i8(m);
  if constexpr (OUT != 0) q16r[idx] = pack_f16(m);
}

template <class D>
__device__ __forceinline__ void store_scale(float s, int64_t row, float* scale, const D& d) {
  for (int j = 0; j < d.n(); ++j) {
    const int64_t r = d.scale_row(row, j);
    if (r >= 0) scale[r] = s;
  }
}

// Every quantisation kernel is launched with programmatic stream serialization
// and opens with pdl_enter: it lets the kernel after it (the decode
// contraction, whose weight stream reads nothing written here) start its
// prologue at once, and it waits for the kernel before it -- which may still
// read the codes and scales this launch overwrites -- before its first access
// to global memory.
__device__ __forceinline__ void pdl_enter() {
  pdl_trigger();
  pdl_wait();
}

// Barrier of row group grp (32 G threads): named barrier 1 + grp, with the id as an immediate so that the
// kernel reserves only the barriers it uses (a register id reserves all sixteen, which caps the CTAs per SM).
template <int G>
__device__ __forceinline__ void group_sync(int grp) {
  switch (grp) {
    case 0: asm volatile("bar.sync 1, %0;" ::"n"(32 * G) : "memory"); break;
    case 1: asm volatile("bar.sync 2, %0;" ::"n"(32 * G) : "memory"); break;
    case 2: asm volatile("bar.sync 3, %0;" ::"n"(32 * G) : "memory"); break;
    default: asm volatile("bar.sync 4, %0;" ::"n"(32 * G) : "memory"); break;
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Rows in groups of G warps (32 G threads per row), CH 16-byte chunks of 8 bf16 per thread (K <= 256 G CH).
// A CTA of 256 threads holds 8 / G groups; group g of CTA b takes rows b (8/G) + g, then every
// gridDim.x (8/G) rows; four CTAs per SM keep 32 rows' loads in flight.  absmax: warp shuffles, then (G > 1) the
// group's warps meet in shared memory behind a named barrier of the group alone.  G is chosen so that
// each thread holds about 64 elements of its row: the per-row work (the reduction, the binary32 divide
// and reciprocal) is then a small part of the per-element work.
template <int CH, int G, int OUT, class D>
__global__ void __launch_bounds__(256, 4) quant_rows(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                     void* __restrict__ q, uint16_t* __restrict__ q16,
                                                     float* __restrict__ scale, D d) {
  pdl_enter();
  // Rows of at most 4 chunks a thread load the group's next row before quantising the current one; rows of
  // 8 chunks do not (the second row's registers would halve the warps an SM holds, which hides more of the
  // memory latency than the prefetch: 27.0 against 30.0 us for 8192 x 4096).
  constexpr bool kPrefetch = CH <= 4;
  constexpr int NG = 8 / G;
  __shared__ float red[NG][2][G];
  const int lane = threadIdx.x & 31;
  const int grp = static_cast<int>(threadIdx.x) / (32 * G);
  const int gl = static_cast<int>(threadIdx.x) % (32 * G);  // thread of the group
  const int64_t nchunk = K / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * NG;
  uint4 v[CH], vn[kPrefetch ? CH : 1];
  auto load_row = [&](int64_t r, uint4* dst) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + r * K);
#pragma unroll
    for (int c = 0; c < CH; ++c) {  // every load of the row in flight before any is used
      const int64_t idx = gl + 32 * G * c;
      dst[c] = (r < M && idx < nchunk) ? ldg_stream(xr + idx) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  int64_t row = static_cast<int64_t>(blockIdx.x) * NG + grp;
  if constexpr (kPrefetch) load_row(row, v);
  int buf = 0;
  for (; row < M; row += stride) {
    if constexpr (kPrefetch) load_row(row + stride, vn);
    else load_row(row, v);
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < CH; ++c) amax = fmaxf(amax, absmax8(v[c]));
    amax = warp_max(amax);
    if constexpr (G > 1) {
      // (red[grp][buf] was last read two rows ago, before the group's previous barrier)
      if (lane == 0) red[grp][buf][gl >> 5] = amax;
      group_sync<G>(grp);
      amax = red[grp][buf][0];
#pragma unroll
      for (int w = 1; w < G; ++w) amax = fmaxf(amax, red[grp][buf][w]);
    }
    const float s = __fdiv_rn(amax, 127.0f);
    const float rs = s > 0.0f ? __frcp_rn(s) : 0.0f;
    if (gl == 0) store_scale(s, row, scale, d);
    if constexpr (std::is_same<D, RowId>::value) {  // one destination: its row located once
      uint2* q8 = OUT != 1 ? reinterpret_cast<uint2*>(static_cast<int8_t*>(q) + row * K) : nullptr;
      uint4* qh = OUT != 0 ? reinterpret_cast<uint4*>(q16 + row * K) : nullptr;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int64_t idx = gl + 32 * G * c;
        if (idx < nchunk) store8_row<OUT>(v[c], s, rs, idx, q8, qh);
      }
    } else {
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int64_t idx = gl + 32 * G * c;
        if (idx < nchunk) store8<OUT>(v[c], s, rs, row, K, idx, q, q16, d);
      }
    }
    if constexpr (kPrefetch) {
#pragma unroll
      for (int c = 0; c < CH; ++c) v[c] = vn[c];
    }
    buf ^= 1;
  }
}

// Any K: two passes over the row (the second read mostly hits L2).
template <int OUT, class D>
__global__ void __launch_bounds__(256) quant_cta_rows_any(const uint16_t* __restrict__ x, int64_t M,
                                                          int64_t K, void* __restrict__ q, uint16_t* __restrict__ q16,
                                                          float* __restrict__ scale, D d) {
  pdl_enter();
  __shared__ float red[8];
  const int64_t nchunk = K / 8;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * K);
    float amax = 0.0f;
    for (int64_t idx = threadIdx.x; idx < nchunk; idx += 256) amax = fmaxf(amax, absmax8(xr[idx]));
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
    const float s = __fdiv_rn(amax, 127.0f);
    const float rs = s > 0.0f ? __frcp_rn(s) : 0.0f;
    if (threadIdx.x == 0) store_scale(s, row, scale, d);
    for (int64_t idx = threadIdx.x; idx < nchunk; idx += 256) {
      store8<OUT>(xr[idx], s, rs, row, K, idx, q, q16, d);
    }
    __syncthreads();
  }
}

// CTAs of quant_rows<CH, G, OUT, D> resident per SM (queried once per instantiation).
template <int CH, int G, int OUT, class D>
int rows_ctas_per_sm() {
  static int per_sm = 0;
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quant_rows<CH, G, OUT, D>, 256, 0) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 1;
    }
    per_sm = n;
  }
  return per_sm;
}

template <int CH, int G, int OUT, class D>
cudaError_t launch_rows(const uint16_t* x, int64_t M, int64_t K, void* q, uint16_t* q16, float* scale, D d,
                        cudaStream_t stream, int num_sms) {
  constexpr int NG = 8 / G;
  const int64_t ctas = (M + NG - 1) / NG;  // as many as rows need, at most as many as are resident at once
  const int64_t grid = std::min<int64_t>(ctas, static_cast<int64_t>(num_sms) * rows_ctas_per_sm<CH, G, OUT, D>());
  return launch_pdl(quant_rows<CH, G, OUT, D>, dim3(static_cast<unsigned>(grid)), dim3(256), 0, stream, x, M, K, q,
                    q16, scale, d);
}

template <int OUT, class D>
cudaError_t launch_quant_t(const uint16_t* x, int64_t M, int64_t K, void* q, uint16_t* q16, float* scale,
                           D d, cudaStream_t stream, int num_sms) {
  if (M == 0) return cudaSuccess;
  const int64_t nchunk = K / 8;
  if (nchunk > 256 * 8) {  // K > 16384: more than 8 chunks per thread even for a whole CTA per row
    const dim3 g(static_cast<unsigned>(std::min<int64_t>(M, static_cast<int64_t>(num_sms) * 64)));
    return launch_pdl(quant_cta_rows_any<OUT, D>, g, dim3(256), 0, stream, x, M, K, q, q16, scale, d);
  }
  // the narrowest group holding the row in at most 8 chunks per thread ...
  int G = 1;
  while (G < 8 && nchunk > 32 * G * 8) G *= 2;
  // ... widened while the rows alone would occupy fewer CTAs than there are SMs (few rows: latency-bound)
  while (G < 8 && (M + 8 / G - 1) / (8 / G) < num_sms) G *= 2;
  if (G == 1) {
    const int64_t ch = (nchunk + 31) / 32;
    if (ch <= 1) return launch_rows<1, 1, OUT>(x, M, K, q, q16, scale, d, stream, num_sms);
    if (ch <= 2) return launch_rows<2, 1, OUT>(x, M, K, q, q16, scale, d, stream, num_sms);
    if (ch <= 4) return launch_rows<4, 1, OUT>(x, M, K, q, q16, scale, d, stream, num_sms);
    return launch_rows<8, 1, OUT>(x, M, K, q, q16, scale, d, stream, num_sms);
  }
  if (G == 2) return launch_rows<8, 2, OUT>(x, M, K, q, q16, scale, d, stream, num_sms);
  if (G == 4) return launch_rows<8, 4, OUT>(x, M, K, q, q16, scale, d, stream, num_sms);
  const int64_t ch = (nchunk + 255) / 256;
  if (ch <= 1) return launch_rows<1, 8, OUT>(x, M, K, q, q16, scale, d, stream, num_sms);
  if (ch <= 2) return launch_rows<2, 8, OUT>(x, M, K, q, q16, scale, d, stream, num_sms);
  if (ch <= 4) return launch_rows<4, 8, OUT>(x, M, K, q, q16, scale, d, stream, num_sms);
  return launch_rows<8, 8, OUT>(x, M, K, q, q16, scale, d, stream, num_sms);
}

}  // namespace

cudaError_t launch_dynamic_quant(const uint16_t* x, int64_t M, int64_t K, int8_t* q, float* scale,
                                 cudaStream_t stream, int num_sms) {
  return launch_quant_t<0>(x, M, K, q, nullptr, scale, RowId{}, stream, num_sms);
}

cudaError_t launch_dynamic_quant_f16(const uint16_t* x, int64_t M, int64_t K, uint16_t* q_f16, float* scale,
                                     cudaStream_t stream, int num_sms) {
  return launch_quant_t<1>(x, M, K, nullptr, q_f16, scale, RowId{}, stream, num_sms);
}

cudaError_t launch_quant_scatter(const uint16_t* x, int64_t T, int64_t H, const int32_t* dst, int k, int8_t* q,
                                 uint16_t* q_f16, float* scale, int out, cudaStream_t stream, int num_sms) {
  const RowScatter d{dst, k};
  if (out == 0) return launch_quant_t<0>(x, T, H, q, nullptr, scale, d, stream, num_sms);
  if (out == 1) return launch_quant_t<1>(x, T, H, nullptr, q_f16, scale, d, stream, num_sms);
  return launch_quant_t<2>(x, T, H, q, q_f16, scale, d, stream, num_sms);
}

cudaError_t launch_quant_pack(const uint16_t* w, int64_t E, int64_t N, int64_t K, uint32_t flags, void* packed,
                              float* scale, cudaStream_t stream, int num_sms) {
  const PackLayout L = pack_layout(E, N, K, flags);
  uint8_t* b = static_cast<uint8_t*>(packed);
  const RowPack d{N, (flags & W8A8_PACK_GATE_UP) != 0u};
  int8_t* q = reinterpret_cast<int8_t*>(b + L.i8_offset);
  const cudaError_t e = L.f16_offset
      ? launch_quant_t<2>(w, E * N, K, q, reinterpret_cast<uint16_t*>(b + L.f16_offset), scale, d, stream, num_sms)
      : launch_quant_t<0>(w, E * N, K, q, nullptr, scale, d, stream, num_sms);
  if (e != cudaSuccess) return e;
  return launch_pack_header(E, N, K, flags, packed, stream);
}

}  // namespace w8a8
