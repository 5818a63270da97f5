// mx.cu -- MXFP8 quantisation (E4M3 payload, one E8M0 scale per 32 values along K).
//
// Page "Qwen3.8-FP8 on Ascend 950: Why Weights Become MXFP8 at Load Time",
// sections 3 and 5: weights are re-quantised to MXFP8 at load and every
// activation row at run time (group sizes [1,1,32]); the scale algorithm is
// the normal one.  Per group of 32: shared = floor(log2 amax) - 8 (8 = the
// largest E4M3 exponent), clamped to [-127, 127], stored as the E8M0 byte
// shared + 127 (0 for a group of zeros, 0xFF if the group holds a NaN);
// elements v / 2^shared (exact) rounded to E4M3 to nearest, ties to even,
// saturating at +-448.
//
// HBM-bound: 2 bytes read, 1 + 1/32 written per element.  Four threads own a
// group (8 values, 16 bytes each); the amax meets through two shuffles.
#include "kernels.cuh"

namespace w8a8 {

namespace {

// floor(log2 |a|) of a finite binary32 a > 0 (normal or subnormal), from its bits.
__device__ __forceinline__ int floor_log2(float a) {
  const uint32_t u = __float_as_uint(a) & 0x7fffffffu;
  const int field = static_cast<int>(u >> 23);
  if (field > 0) return field - 127;
  return -149 + (31 - __clz(u));  // subnormal: mantissa * 2^-149
}

// Two binary32 values -> two E4M3 bytes (round to nearest even, saturating), lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(256) mx_quant_kernel(const uint16_t* __restrict__ x, int64_t n8,
                                                       uint8_t* __restrict__ q, uint8_t* __restrict__ scale) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * 256;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * 256 + (threadIdx.x & ~31); base < n8; base += stride) {
    const int64_t i = base + lane;  // 8 values; four consecutive i form one group (n8 % 4 == 0)
    const bool in = i < n8;
    const uint4 v = in ? reinterpret_cast<const uint4*>(x)[i] : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
    float amax = 0.0f;
    bool nan = false;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      nan = nan || (f[k] != f[k]);
      amax = fmaxf(amax, fabsf(f[k]));  // fmaxf passes over a NaN
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      nan = __shfl_xor_sync(0xffffffffu, nan ? 1 : 0, o) != 0 || nan;
    }
    int shared = -127;
    if (amax > 0.0f) shared = min(127, max(-127, floor_log2(amax) - 8));
    // 2^-shared as binary32: exponent field 127 - shared (1..254) for shared <= 126, and the subnormal
    // 2^-127 for shared = 127; multiplying by it is exact (the results stay within 2^9)
    const float inv = shared < 127 ? __uint_as_float(static_cast<uint32_t>(127 - shared) << 23)
                                   : __uint_as_float(0x00400000u);
    uint32_t lo = 0u, hi = 0u;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      lo |= e4m3x2(__fmul_rn(f[2 * k], inv), __fmul_rn(f[2 * k + 1], inv)) << (16 * k);
      hi |= e4m3x2(__fmul_rn(f[4 + 2 * k], inv), __fmul_rn(f[4 + 2 * k + 1], inv)) << (16 * k);
    }
    if (in) {
      reinterpret_cast<uint2*>(q)[i] = make_uint2(lo, hi);
      if ((lane & 3) == 0) scale[i >> 2] = nan ? 0xFFu : (amax > 0.0f ? static_cast<uint8_t>(shared + 127) : 0u);
    }
  }
}

}  // namespace

cudaError_t launch_mx_quant(const uint16_t* x, int64_t M, int64_t K, uint8_t* q, uint8_t* scale, cudaStream_t stream,
                            int num_sms) {
  const int64_t n8 = M * K / 8;
  if (n8 == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n8 + 255) / 256, static_cast<int64_t>(num_sms) * 8);
  return launch_pdl(mx_quant_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, x, n8, q, scale);
}

}  // namespace w8a8
