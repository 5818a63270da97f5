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
// Each row is read once with 16-byte vector loads and held in registers
// between the absmax pass and the quantise pass; absmax is reduced with warp
// shuffles (and shared memory across the warps of a CTA).
#include "kernels.cuh"

namespace w8a8 {

namespace {

__device__ __forceinline__ float absmax8(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
    m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xffff0000u)));
  }
  return m;
}

// rint(x / s) with the quotient rounded to binary32 first (round half to even), clamped to +-127;
// s > 0, rs = the binary32 reciprocal of s.  y = x * rs is within |x / s| * 2^-23 + 2^-18 <= 2^-15 of
// the correctly rounded quotient (|x / s| <= 128), so when y is more than 2^-14 from the nearest
// half-integer both lie strictly inside the same rounding interval and round to the same integer;
// otherwise (rare), and for non-finite y, the quotient itself is computed.
__device__ __forceinline__ int q1(float xf, float s, float rs) {
  const float y = __fmul_rn(xf, rs);
  const float frac = __fsub_rn(y, floorf(y));  // exact for |y| < 2^23
  const int r = fabsf(frac - 0.5f) > 0x1p-14f ? __float2int_rn(y) : __float2int_rn(__fdiv_rn(xf, s));
  return max(-127, min(127, r));
}

// 8 bf16 -> 8 int8 packed in a uint2.
__device__ __forceinline__ uint2 quant8(const uint4& v, float s, float rs) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[2] = {0u, 0u};
  if (s > 0.0f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int lo = q1(__uint_as_float(w[i] << 16), s, rs);
      const int hi = q1(__uint_as_float(w[i] & 0xffff0000u), s, rs);
      const uint32_t pair = (static_cast<uint32_t>(lo) & 0xffu) | ((static_cast<uint32_t>(hi) & 0xffu) << 8);
      out[i >> 1] |= pair << ((i & 1) * 16);
    }
  }
  return make_uint2(out[0], out[1]);
}

// 8 bf16 -> 8 integer-valued fp16 (same codes as quant8) packed in a uint4.
__device__ __forceinline__ uint4 quant8_f16(const uint4& v, float s, float rs) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[4] = {0u, 0u, 0u, 0u};
  if (s > 0.0f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int lo = q1(__uint_as_float(w[i] << 16), s, rs);
      const int hi = q1(__uint_as_float(w[i] & 0xffff0000u), s, rs);
      out[i] = static_cast<uint32_t>(__half_as_ushort(__int2half_rn(lo))) |
               (static_cast<uint32_t>(__half_as_ushort(__int2half_rn(hi))) << 16);
    }
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// OUT: 0 = int8 codes into q; 1 = the same codes as fp16 into q16; 2 = both (each code computed once).
__device__ __forceinline__ void store8(const uint4& v, float s, float rs, int64_t row, int64_t K, int64_t idx,
                                       void* q, uint16_t* q16, int out) {
  if (out == 0) {
    reinterpret_cast<uint2*>(static_cast<int8_t*>(q) + row * K)[idx] = quant8(v, s, rs);
  } else if (out == 1) {
    reinterpret_cast<uint4*>(q16 + row * K)[idx] = quant8_f16(v, s, rs);
  } else {
    uint32_t b[4] = {0u, 0u, 0u, 0u}, h[4] = {0u, 0u, 0u, 0u};  // byte pairs / fp16 pairs of v.x .. v.w
    if (s > 0.0f) {
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int lo = q1(__uint_as_float(w[i] << 16), s, rs);
        const int hi = q1(__uint_as_float(w[i] & 0xffff0000u), s, rs);
        b[i] = (static_cast<uint32_t>(lo) & 0xffu) | ((static_cast<uint32_t>(hi) & 0xffu) << 8);
        h[i] = static_cast<uint32_t>(__half_as_ushort(__int2half_rn(lo))) |
               (static_cast<uint32_t>(__half_as_ushort(__int2half_rn(hi))) << 16);
      }
    }
    reinterpret_cast<uint2*>(static_cast<int8_t*>(q) + row * K)[idx] = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
    reinterpret_cast<uint4*>(q16 + row * K)[idx] = make_uint4(h[0], h[1], h[2], h[3]);
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

// One row per warp; CH 16-byte chunks per lane (K <= 256 * CH).
template <int CH, int OUT>
__global__ void __launch_bounds__(256) quant_warp_rows(const uint16_t* __restrict__ x, int64_t M,
                                                       int64_t K, void* __restrict__ q, uint16_t* __restrict__ q16,
                                                       float* __restrict__ scale) {
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
    if (lane == 0) scale[row] = s;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int64_t idx = lane + 32 * c;
      if (idx < nchunk) {
        store8(v[c], s, rs, row, K, idx, q, q16, OUT);
      }
    }
  }
}

// One row per CTA of 256 threads; CH 16-byte chunks per thread (K <= 2048 * CH).
template <int CH, int OUT>
__global__ void __launch_bounds__(256) quant_cta_rows(const uint16_t* __restrict__ x, int64_t M,
                                                      int64_t K, void* __restrict__ q, uint16_t* __restrict__ q16,
                                                      float* __restrict__ scale) {
  pdl_enter();
  __shared__ float red[8];
  const int64_t nchunk = K / 8;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * K);
    uint4 v[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {  // every load of the row in flight before any is used
      const int64_t idx = threadIdx.x + 256 * c;
      v[c] = idx < nchunk ? ldg_stream(xr + idx) : make_uint4(0u, 0u, 0u, 0u);
    }
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < CH; ++c) amax = fmaxf(amax, absmax8(v[c]));
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
    const float s = __fdiv_rn(amax, 127.0f);
    const float rs = s > 0.0f ? __frcp_rn(s) : 0.0f;
    if (threadIdx.x == 0) scale[row] = s;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int64_t idx = threadIdx.x + 256 * c;
      if (idx < nchunk) {
        store8(v[c], s, rs, row, K, idx, q, q16, OUT);
      }
    }
    __syncthreads();  // red[] is reused by the next row
  }
}

// Any K: two passes over the row (the second read mostly hits L2).
template <int OUT>
__global__ void __launch_bounds__(256) quant_cta_rows_any(const uint16_t* __restrict__ x, int64_t M,
                                                          int64_t K, void* __restrict__ q, uint16_t* __restrict__ q16,
                                                          float* __restrict__ scale) {
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
    if (threadIdx.x == 0) scale[row] = s;
    for (int64_t idx = threadIdx.x; idx < nchunk; idx += 256) {
      store8(xr[idx], s, rs, row, K, idx, q, q16, OUT);
    }
    __syncthreads();
  }
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), dim3 g, dim3 b, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = g;
  cfg.blockDim = b;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

template <int OUT>
cudaError_t launch_quant_t(const uint16_t* x, int64_t M, int64_t K, void* q, uint16_t* q16, float* scale,
                           cudaStream_t stream, int num_sms) {
  if (M == 0) return cudaSuccess;
  const int64_t nchunk = K / 8;
  const int64_t max_grid = static_cast<int64_t>(num_sms) * 64;
  if (nchunk <= 32 * 8) {
    // warp per row, 8 rows per CTA
    const int64_t blocks = std::min<int64_t>((M + 7) / 8, max_grid);
    const int ch = static_cast<int>((nchunk + 31) / 32);
    dim3 g(static_cast<unsigned>(blocks)), b(256);
    if (ch <= 1) return launch_pdl(quant_warp_rows<1, OUT>, g, b, stream, x, M, K, q, q16, scale);
    else if (ch <= 2) return launch_pdl(quant_warp_rows<2, OUT>, g, b, stream, x, M, K, q, q16, scale);
    else if (ch <= 4) return launch_pdl(quant_warp_rows<4, OUT>, g, b, stream, x, M, K, q, q16, scale);
    else return launch_pdl(quant_warp_rows<8, OUT>, g, b, stream, x, M, K, q, q16, scale);
  } else {
    const int64_t blocks = std::min<int64_t>(M, max_grid);
    const int ch = static_cast<int>((nchunk + 255) / 256);
    dim3 g(static_cast<unsigned>(blocks)), b(256);
    if (ch <= 2) return launch_pdl(quant_cta_rows<2, OUT>, g, b, stream, x, M, K, q, q16, scale);
    else if (ch <= 4) return launch_pdl(quant_cta_rows<4, OUT>, g, b, stream, x, M, K, q, q16, scale);
    else if (ch <= 8) return launch_pdl(quant_cta_rows<8, OUT>, g, b, stream, x, M, K, q, q16, scale);
    else return launch_pdl(quant_cta_rows_any<OUT>, g, b, stream, x, M, K, q, q16, scale);
  }
}

}  // namespace

cudaError_t launch_dynamic_quant(const uint16_t* x, int64_t M, int64_t K, int8_t* q, float* scale,
                                 cudaStream_t stream, int num_sms) {
  return launch_quant_t<0>(x, M, K, q, nullptr, scale, stream, num_sms);
}

cudaError_t launch_dynamic_quant_dual(const uint16_t* x, int64_t M, int64_t K, int8_t* q, uint16_t* q_f16,
                                      float* scale, cudaStream_t stream, int num_sms) {
  return launch_quant_t<2>(x, M, K, q, q_f16, scale, stream, num_sms);
}

}  // namespace w8a8
