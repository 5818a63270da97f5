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
__device__ __forceinline__ void codes8(const uint4& v, float s, float rs, float (&m)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float x[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
  float dmax = 0.0f;  // max |y - rint(y)| over the chunk; NaN if any y is not finite
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float y = __fmul_rn(x[e], rs);
    m[e] = __fadd_rn(y, kRoundMagic);
    const float t = __fsub_rn(y, __fsub_rn(m[e], kRoundMagic));  // y - rint(y), exact
    asm("max.NaN.f32 %0, %0, %1;" : "+f"(dmax) : "f"(fabsf(t)));
  }
  if (__builtin_expect(!(dmax < 0.5f - 0x1p-14f), 0)) {
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

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One row per warp; CH 16-byte chunks per lane (K <= 256 * CH).  At least four CTAs (32 warps, 32 rows of
// loads in flight) per SM.
template <int CH, int OUT, class D>
__global__ void __launch_bounds__(256, 4) quant_warp_rows(const uint16_t* __restrict__ x, int64_t M,
                                                       int64_t K, void* __restrict__ q, uint16_t* __restrict__ q16,
                                                       float* __restrict__ scale, D d) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t nchunk = K / 8;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; row < M;
       row += warps_total) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * K);
    uint4 v[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {  // every load of the row in flight before any is used
      const int64_t idx = lane + 32 * c;
      v[c] = idx < nchunk ? ldg_stream(xr + idx) : make_uint4(0u, 0u, 0u, 0u);
    }
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < CH; ++c) amax = fmaxf(amax, absmax8(v[c]));
    amax = warp_max(amax);
    const float s = __fdiv_rn(amax, 127.0f);
    const float rs = s > 0.0f ? __frcp_rn(s) : 0.0f;
    if (lane == 0) store_scale(s, row, scale, d);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int64_t idx = lane + 32 * c;
      if (idx < nchunk) {
        store8<OUT>(v[c], s, rs, row, K, idx, q, q16, d);
      }
    }
  }
}

// One row per CTA of 256 threads; CH 16-byte chunks per thread (K <= 2048 * CH).  A CTA takes rows
// blockIdx.x, + gridDim.x, ...; the loads of its next row are issued before the current one is reduced
// and quantised, so an SM keeps reading while it computes.
template <int CH, int OUT, class D>
__global__ void __launch_bounds__(256) quant_cta_rows(const uint16_t* __restrict__ x, int64_t M,
                                                      int64_t K, void* __restrict__ q, uint16_t* __restrict__ q16,
                                                      float* __restrict__ scale, D d) {
  pdl_enter();
  __shared__ float red[2][8];
  const int64_t nchunk = K / 8;
  uint4 v[CH];
  auto load_row = [&](int64_t row, uint4 (&dst)[CH]) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * K);
#pragma unroll
    for (int c = 0; c < CH; ++c) {  // every load of the row in flight before any is used
      const int64_t idx = threadIdx.x + 256 * c;
      dst[c] = (row < M && idx < nchunk) ? ldg_stream(xr + idx) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  load_row(blockIdx.x, v);
  int buf = 0;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    uint4 vn[CH];
    load_row(row + gridDim.x, vn);
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < CH; ++c) amax = fmaxf(amax, absmax8(v[c]));
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) red[buf][threadIdx.x >> 5] = amax;
    __syncthreads();  // (red[buf] was last read two rows ago, before the previous barrier)
    amax = red[buf][0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[buf][w]);
    const float s = __fdiv_rn(amax, 127.0f);
    const float rs = s > 0.0f ? __frcp_rn(s) : 0.0f;
    if (threadIdx.x == 0) store_scale(s, row, scale, d);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int64_t idx = threadIdx.x + 256 * c;
      if (idx < nchunk) store8<OUT>(v[c], s, rs, row, K, idx, q, q16, d);
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) v[c] = vn[c];
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

// CTAs of quant_cta_rows<CH, OUT, D> resident per SM (queried once).
template <int CH, int OUT, class D>
int cta_rows_per_sm() {
  static int per_sm = 0;
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quant_cta_rows<CH, OUT, D>, 256, 0) != cudaSuccess ||
        n < 1) {
      cudaGetLastError();
      n = 1;
    }
    per_sm = n;
  }
  return per_sm;
}

template <int OUT, class D>
cudaError_t launch_quant_t(const uint16_t* x, int64_t M, int64_t K, void* q, uint16_t* q16, float* scale,
                           D d, cudaStream_t stream, int num_sms) {
  if (M == 0) return cudaSuccess;
  const int64_t nchunk = K / 8;
  const int64_t max_grid = static_cast<int64_t>(num_sms) * 64;
  if (nchunk <= 32 * 8) {
    // warp per row, 8 rows per CTA
    const int64_t blocks = std::min<int64_t>((M + 7) / 8, max_grid);
    const int ch = static_cast<int>((nchunk + 31) / 32);
    dim3 g(static_cast<unsigned>(blocks)), b(256);
    if (ch <= 1) return launch_pdl(quant_warp_rows<1, OUT, D>, g, b, 0, stream, x, M, K, q, q16, scale, d);
    else if (ch <= 2) return launch_pdl(quant_warp_rows<2, OUT, D>, g, b, 0, stream, x, M, K, q, q16, scale, d);
    else if (ch <= 4) return launch_pdl(quant_warp_rows<4, OUT, D>, g, b, 0, stream, x, M, K, q, q16, scale, d);
    else return launch_pdl(quant_warp_rows<8, OUT, D>, g, b, 0, stream, x, M, K, q, q16, scale, d);
  } else {
    // as many CTAs as are resident at once; each then works through its rows
    const int ch = static_cast<int>((nchunk + 255) / 256);
    dim3 b(256);
    auto grid = [&](int per_sm) {
      return dim3(static_cast<unsigned>(std::min<int64_t>(M, static_cast<int64_t>(num_sms) * per_sm)));
    };
    if (ch <= 2)
      return launch_pdl(quant_cta_rows<2, OUT, D>, grid(cta_rows_per_sm<2, OUT, D>()), b, 0, stream, x, M, K, q,
                        q16, scale, d);
    if (ch <= 4)
      return launch_pdl(quant_cta_rows<4, OUT, D>, grid(cta_rows_per_sm<4, OUT, D>()), b, 0, stream, x, M, K, q,
                        q16, scale, d);
    if (ch <= 8)
      return launch_pdl(quant_cta_rows<8, OUT, D>, grid(cta_rows_per_sm<8, OUT, D>()), b, 0, stream, x, M, K, q,
                        q16, scale, d);
    const dim3 g(static_cast<unsigned>(std::min<int64_t>(M, max_grid)));
    return launch_pdl(quant_cta_rows_any<OUT, D>, g, b, 0, stream, x, M, K, q, q16, scale, d);
  }
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
