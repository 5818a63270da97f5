// static.cu -- the static W8A8 variant.
//
// Page "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子", closing comparison
// of the static recipe: npu_quantize with a fixed (calibrated) input_scale
// and input_offset turns BF16 X into INT8; at load time
// deq_scale = input_scale * weight_scale and
// quant_bias = round(fp_bias / deq_scale - sum_k(Qw[n,k]) * input_offset),
// the correction that x = input_scale * (q - input_offset) calls for; then
// npu_quant_matmul(x, W, deq_scale, bias=quant_bias) -> BF16.  The contraction
// is the dense one (its epilogue adds quant_bias to the accumulator);
// this file holds the quantiser and the load-time preparation.
//
//   quantise  q = clamp(rint(x / s) + o, -128, 127) (binary32 divide, ties to
//             even, the integer offset added after rounding), computed with
//             a reciprocal multiply and the division only where the two could
//             round differently.  Elementwise and HBM-bound: 2 bytes read,
//             1 written per element.
//   prepare   one warp per output channel: the exact int8 row sum, then the
//             binary32 steps deq = s * w_scale, a = bias / deq (0 without a
//             bias or where deq is 0), c = float(sum) * o, rint(a - c)
//             saturated to int32.  Reads the INT8 weight once.
#include "kernels.cuh"

namespace w8a8 {

namespace {

// rint(x / s) of the binary32 quotient without a division where that is safe: y = x * rs with rs =
// fl(1/s) is within |x/s| * 2^-23 * (1 + 2^-25) of the exact quotient, so for |y| <= 1024 it is within
// 2^-13; when y is more than 2^-12 from the nearest half-integer, the exact quotient and its binary32
// rounding lie strictly inside the same rounding interval and round to the same integer.  Beyond 1024
// every code clamps whichever way the quotient rounds (|o| <= 128).  Otherwise (rare), and for NaN,
// the division itself.
__device__ __forceinline__ int static_code(float x, float s, float rs, int o) {
  const float y = __fmul_rn(x, rs);
  float r;
  if (fabsf(y) > 1024.0f) {
    r = y;
  } else {
    r = rintf(y);
    if (!(fabsf(__fsub_rn(y, r)) <= 0.5f - 0x1p-12f)) {
      const float t = __fdiv_rn(x, s);
      if (t != t) return 0;
      r = rintf(t);
    }
  }
  const float c = fminf(fmaxf(__fadd_rn(r, static_cast<float>(o)), -128.0f), 127.0f);  // exact below 2^24
  return static_cast<int>(c);
}

__device__ __forceinline__ uint32_t static_code4(const uint32_t* w2, float s, float rs, int o) {
  uint32_t out = 0u;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float x = __uint_as_float(h == 0 ? (w2[i] << 16) : (w2[i] & 0xffff0000u));
      out |= (static_cast<uint32_t>(static_code(x, s, rs, o)) & 0xffu) << (8 * (2 * i + h));
    }
  }
  return out;
}

// Thread per 8 elements (16 bytes in, 8 out), grid-stride.
__global__ void __launch_bounds__(256) static_quant_kernel(const uint16_t* __restrict__ x, int64_t n8, float s, int o,
                                                           int8_t* __restrict__ q) {
  pdl_trigger();
  pdl_wait();
  const float rs = __frcp_rn(s);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * 256) {
    const uint4 v = reinterpret_cast<const uint4*>(x)[i];
    const uint32_t lo[2] = {v.x, v.y}, hi[2] = {v.z, v.w};
    reinterpret_cast<uint2*>(q)[i] = make_uint2(static_code4(lo, s, rs, o), static_code4(hi, s, rs, o));
  }
}

// Warp per channel.
__global__ void __launch_bounds__(256) static_prepare_kernel(const int8_t* __restrict__ w, int64_t N, int64_t K,
                                                             const float* __restrict__ w_scale, float s, int o,
                                                             const uint16_t* __restrict__ bias,
                                                             float* __restrict__ deq, int32_t* __restrict__ qb) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * 8;
  for (int64_t n = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5); n < N; n += nwarps) {
    const uint4* row = reinterpret_cast<const uint4*>(w + n * K);
    int32_t sum = 0;
    for (int64_t c = lane; c < K / 16; c += 32) {
      const uint4 v = row[c];
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int b = 0; b < 4; ++b) sum += static_cast<int8_t>((u[i] >> (8 * b)) & 0xffu);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) {
      const float d = __fmul_rn(s, w_scale[n]);
      const float a = (bias != nullptr && d != 0.0f) ? __fdiv_rn(bf16_bits_to_f32(bias[n]), d) : 0.0f;
      const float c = __fmul_rn(__int2float_rn(sum), static_cast<float>(o));
      const float t = rintf(__fsub_rn(a, c));
      int32_t v;
      if (t != t) v = 0;
      else if (t >= 2147483648.0f) v = INT32_MAX;
      else if (t < -2147483648.0f) v = INT32_MIN;
      else v = static_cast<int32_t>(t);
      deq[n] = d;
      qb[n] = v;
    }
  }
}

}  // namespace

cudaError_t launch_static_quant(const uint16_t* x, int64_t M, int64_t K, float s, int o, int8_t* q,
                                cudaStream_t stream, int num_sms) {
  const int64_t n8 = M * K / 8;
  if (n8 == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n8 + 255) / 256, static_cast<int64_t>(num_sms) * 8);
  return launch_pdl(static_quant_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, x, n8, s, o, q);
}

cudaError_t launch_static_prepare(const int8_t* w, int64_t N, int64_t K, const float* w_scale, float s, int o,
                                  const uint16_t* bias, float* deq, int32_t* qb, cudaStream_t stream, int num_sms) {
  const int64_t blocks = std::min<int64_t>((N + 7) / 8, static_cast<int64_t>(num_sms) * 16);
  return launch_pdl(static_prepare_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, w, N, K, w_scale,
                    s, o, bias, deq, qb);
}

}  // namespace w8a8
