// common.cuh -- device helpers shared by the kernels of libw8a8.so (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/w8a8.h"

namespace w8a8 {

// ------------------------------------------------------------ layout facts --

constexpr int kNumSMsHint = 152;      // GB300; the host reads the real count
constexpr int kChunkK = 1024;         // fp32 partial sums of <= 1024 products of
                                      // |int8*int8| <= 2^14 stay <= 2^24: exact
constexpr uint32_t kPackMagic = 0x4B503857u;  // "W8PK"
constexpr uint32_t kPackVersion = 1u;
constexpr int kPackHeaderBytes = 256;
constexpr int kGateUpBlock = 64;      // W13 interleave block (gate 64 rows, then up 64 rows)

// Header at the start of every packed weight buffer.
struct PackedHeader {
  uint32_t magic;
  uint32_t version;
  int64_t E, N, K;
  uint32_t flags;
  uint32_t reserved;
  uint64_t i8_offset;   // bytes from the buffer start to the int8 payload [E,N,K] (packed row order)
  uint64_t f16_offset;  // bytes to the fp16 payload [E,N,K], 0 if absent
};

__host__ __device__ inline uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

// Status word: the first 16 bytes of every workspace.
struct DeviceStatus {
  uint32_t code;    // first error code set wins
  uint32_t detail;  // e.g. the expert index of a bad count
  uint32_t pad[2];
};
constexpr int kStatusBytes = 256;

__device__ __forceinline__ void set_status(DeviceStatus* st, uint32_t code, uint32_t detail) {
  if (st == nullptr) return;
  if (atomicCAS(&st->code, 0u, code) == 0u) st->detail = detail;
}

// Packed-row -> original-row map for the gate/up interleave of W13:
// packed rows [128b, 128b+64) are gate rows [64b, 64b+64), packed rows
// [128b+64, 128b+128) are up rows [I+64b, I+64b+64).
__host__ __device__ __forceinline__ int64_t gate_up_orig_row(int64_t p, int64_t I) {
  const int64_t b = p / (2 * kGateUpBlock);
  const int64_t i = p % (2 * kGateUpBlock);
  return i < kGateUpBlock ? b * kGateUpBlock + i : I + b * kGateUpBlock + (i - kGateUpBlock);
}

// ------------------------------------------------------------ conversions --

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
// Two values rounded to bf16 (round to nearest even, as f32_to_bf16_bits) in one instruction: lo in bits
// 0-15, hi in bits 16-31.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2_bits(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four signed bytes -> two f16x2 words holding the same integers exactly.
// Each byte b is biased to u = b + 128 (xor 0x80), placed as the low mantissa
// byte of the half 0x64uu (= 1024 + u), and 1152 = 1024 + 128 is subtracted.
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t v, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = v ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
  const uint32_t bias = 0x64806480u;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

// ------------------------------------------------- binary32 exp for SwiGLU --
// e^x by Cody & Waite argument reduction (Cody, Waite, "Software Manual for
// the Elementary Functions", 1980) and the degree-7 Taylor polynomial of e^r
// in Horner form with fused multiply-adds:
//   n = rint(x * fl(1/ln2)); r = fma(-n, ln2_hi, x); r = fma(-n, ln2_lo, r)
//   ln2_hi = ln 2 cut to 15 significant bits (n*ln2_hi exact),
//   ln2_lo = fl(ln 2 - ln2_hi); c_k = fl(1/k!);
//   e^x = (p * 2^(n/2)) * 2^(n - n/2) with n/2 truncated toward zero.
// x > 89 -> +inf, x < -104 -> 0, NaN -> NaN.  Each step is a correctly
// rounded binary32 operation, so the result is fully determined by these steps.
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }

// Branch-free: the steps run on x clamped to [-104, 89] with NaN propagated.  The clamp alone gives the
// specified results outside that range: the steps at x = 89 overflow to +inf (e^89 > FLT_MAX) and at
// x = -104 round to +0 (e^-104 < 2^-150), the results for every x > 89 and x < -104; a NaN runs through
// the steps and comes out NaN.  (Checked against the form that selects those results explicitly, on
// every binary32 value in [-112, -100] and [84, 96] and at the infinities.)  Without branches or selects
// the compiler can interleave the steps of neighbouring elements.
__device__ __forceinline__ float exp_cw(float x_in) {
  float x;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(x) : "f"(x_in), "f"(-104.0f));
  asm("min.NaN.f32 %0, %0, %1;" : "+f"(x) : "f"(89.0f));
  const float log2e = __int_as_float(0x3fb8aa3b);
  const float ln2_hi = __int_as_float(0x3f317200);
  const float ln2_lo = __int_as_float(0x35bfbe8e);
  const float c7 = __int_as_float(0x39500d01);  // 1/5040
  const float c6 = __int_as_float(0x3ab60b61);  // 1/720
  const float c5 = __int_as_float(0x3c088889);  // 1/120
  const float c4 = __int_as_float(0x3d2aaaab);  // 1/24
  const float c3 = __int_as_float(0x3e2aaaab);  // 1/6
  // n = rint(x * log2e) by the magic-number add (|x * log2e| < 2^22: the sum's low mantissa bits hold n,
  // rounded half to even as rint rounds), which also gives n as an integer without a conversion
  const float nm = __fadd_rn(__fmul_rn(x, log2e), 12582912.0f);
  const float n = __fsub_rn(nm, 12582912.0f);
  const int ni = __float_as_int(nm) - 0x4b400000;
  float r = __fmaf_rn(-n, ln2_hi, x);
  r = __fmaf_rn(-n, ln2_lo, r);
  float p = c7;
  p = __fmaf_rn(p, r, c6);
  p = __fmaf_rn(p, r, c5);
  p = __fmaf_rn(p, r, c4);
  p = __fmaf_rn(p, r, c3);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const int n1 = ni / 2;
  const int n2 = ni - n1;
  return __fmul_rn(__fmul_rn(p, pow2i(n1)), pow2i(n2));
}

// h = bf16((g * sigmoid(g)) * u), sigmoid(g) = 1 / (1 + exp(-g)) (the correctly rounded reciprocal, the
// same value as the correctly rounded quotient 1 / (1 + e)); swiglu_f32 stops before the bf16 rounding.
__device__ __forceinline__ float swiglu_f32(float g, float u) {
  const float e = exp_cw(-g);
  const float sig = __frcp_rn(__fadd_rn(1.0f, e));
  return __fmul_rn(__fmul_rn(g, sig), u);
}
__device__ __forceinline__ uint16_t swiglu_bf16(float g, float u) { return f32_to_bf16_bits(swiglu_f32(g, u)); }

// Dequant epilogue of one element: bf16(((float)acc * sx) * sw (+ bias)).
__device__ __forceinline__ float dequant(int32_t acc, float sx, float sw) {
  return __fmul_rn(__fmul_rn(__int2float_rn(acc), sx), sw);
}

// The same with an integer bias added to the accumulator first (static W8A8: quant_bias, with sx = 1
// and sw = deq_scale): float(acc + qb) * sx * sw with the sum exact -- in 32 bits, or in 64 bits where
// the 32-bit sum would wrap (rare: |acc| < 2^31 and |qb| < 2^31 both hold).
__device__ __forceinline__ float dequant_q(int32_t acc, int32_t qb, float sx, float sw) {
  const int32_t s = static_cast<int32_t>(static_cast<uint32_t>(acc) + static_cast<uint32_t>(qb));
  float f;
  if (__builtin_expect(((acc ^ s) & (qb ^ s)) < 0, 0)) f = __ll2float_rn(static_cast<long long>(acc) + qb);
  else f = __int2float_rn(s);
  return __fmul_rn(__fmul_rn(f, sx), sw);
}

// ------------------------------------------------------------- PTX helpers --

// Programmatic dependent launch.  pdl_trigger: a kernel launched after this
// one with programmatic stream serialization may be scheduled from now on (it
// still waits for this grid before it touches anything this grid reads or
// writes).  pdl_wait: blocks the calling thread until the grids this one
// depends on have completed and their writes are visible; returns at once for
// a kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Host: launch with programmatic stream serialization (the kernel must pdl_wait before it touches memory
// that kernels before it on the stream use).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*k)(KArgs...), dim3 g, dim3 b, size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = g;
  cfg.blockDim = b;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// D(16x8,f32) += A(16x16,f16,row) * B(16x8,f16,col)
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

}  // namespace w8a8
