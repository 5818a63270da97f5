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

// Running max |x| over bf16 values, two lanes packed in a 32-bit word: max.xorsign.abs compares the
// operands' magnitudes and returns the larger one (its sign the XOR of the two signs, so that only the
// magnitude of the result means anything).  KeepNaN: a NaN operand makes the lane NaN (the pass that
// finds rows holding a NaN); else it is passed over, as max passes it over (the absmax of such a row).
template <bool KeepNaN>
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t m;
  if constexpr (KeepNaN) asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
  else asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
  return m;
}
// acc folded with the 8 bf16 of a chunk.
template <bool KeepNaN>
__device__ __forceinline__ uint32_t absmax8_acc(const uint4& v, uint32_t acc) {
  return absmax_bf16x2<KeepNaN>(
      absmax_bf16x2<KeepNaN>(absmax_bf16x2<KeepNaN>(v.x, v.y), absmax_bf16x2<KeepNaN>(v.z, v.w)), acc);
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
// The larger magnitude of the two lanes, widened to binary32 (exact); NaN if a lane is NaN.
__device__ __forceinline__ float absmax_of(uint32_t acc) {
  return fmax_nan(__uint_as_float((acc << 16) & 0x7fff0000u), __uint_as_float(acc & 0x7fff0000u));
}

// y + 1.5 * 2^23 rounds y (|y| < 2^22) to an integer, ties to even, held in the low mantissa bits: the
// sum's low byte is the two's-complement int8 code and (sum - 1.5 * 2^23) the code as a float.
constexpr float kRoundMagic = 12582912.0f;

// The 8 codes of a chunk of 8 bf16 (x[e] = element e), as sums m[e] = code + kRoundMagic: rint(x / s)
// with the quotient rounded to binary32 first (round half to even), clamped to +-127.  s = RN(amax / 127)
// of the row, rs = RN(1 / s) (0 when s = 0).
//
// Fast path, for rows without a NaN whose s is 0 or in [2^-120, FLT_MAX]: the quotient by one
// correction of the reciprocal product (Markstein's step): y0 = RN(x * rs), r = x - y0 * s (exact, one
// fma), y = RN(y0 + r * rs).  Over the whole domain the kernel meets there -- every positive finite bf16
// amax whose s lies in that range and every bf16 x with |x| <= amax, 531 million pairs, negative x by
// symmetry -- rint(y) = rint(RN(x / s)) for every pair, checked exhaustively on the GPU against the
// correctly rounded divide (rint(y0) misses 5,784 of them, all at quotients within a few ulps of a
// half-integer).  |x / s| <= 127 (1 + 2^-23), so no code passes 127 and no clamp
// is needed.  s = 0 means every x is +-0: y = 0.
//
// Other rows (rare): a row holding a NaN (its absmax passes NaNs over) takes the fast path but sends
// each chunk holding a NaN down the exact path: the binary32 quotient itself, rint, clamp, a NaN quotient
// giving code 0; a row holding an infinity has s = inf, where every quotient is 0 or NaN: all codes 0;
// a row with 0 < s < 2^-120 takes the exact path throughout.
//
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

__device__ __forceinline__ void codes8_fast(const uint4& v, float s, float rs, float (&m)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const uint64_t rs2 = pk2(rs, rs), ns2 = pk2(-s, -s), mg2 = pk2(kRoundMagic, kRoundMagic);
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // elements 2i, 2i+1 side by side
    const uint64_t x2 = pk2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
    uint64_t y0, r2, y2, m2;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y0) : "l"(x2), "l"(rs2));               // y0 = x * rs
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r2) : "l"(y0), "l"(ns2), "l"(x2));  // r = x - y0 * s, exact
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(y2) : "l"(r2), "l"(rs2), "l"(y0));  // y = y0 + r * rs
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(m2) : "l"(y2), "l"(mg2));               // m = rint(y) + magic
    upk2(m2, m[2 * i], m[2 * i + 1]);
  }
}
__device__ __forceinline__ void codes8_exact(const uint4& v, float s, float (&m)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float x = __uint_as_float(e & 1 ? w[e >> 1] & 0xffff0000u : w[e >> 1] << 16);
    const int r = max(-127, min(127, __float2int_rn(__fdiv_rn(x, s))));
    m[e] = __fadd_rn(static_cast<float>(r), kRoundMagic);
  }
}
enum RowMode : int { kRowFast = 0, kRowFastNaN = 1, kRowZero = 2, kRowExact = 3 };
// The mode of a row (see above); nan_row: the row holds a NaN.
__device__ __forceinline__ int row_mode(float s, bool nan_row) {
  constexpr float kMaxFinite = 3.4028234663852886e38f;
  if (s == 0.0f || (s >= 0x1p-120f && s <= kMaxFinite)) return nan_row ? kRowFastNaN : kRowFast;
  return s > kMaxFinite ? kRowZero : kRowExact;
}
struct Codes8 {
  float m[8];
};
__device__ __forceinline__ Codes8 codes8_rare(const uint4& v, float s, float rs, int mode) {
  Codes8 c;
  if (mode == kRowFastNaN) {
    codes8_fast(v, s, rs, c.m);
    const float a = absmax_of(absmax8_acc<true>(v, 0u));
    if (a != a) codes8_exact(v, s, c.m);
  } else if (mode == kRowZero) {
#pragma unroll
    for (int e = 0; e < 8; ++e) c.m[e] = kRoundMagic;
  } else {
    codes8_exact(v, s, c.m);
  }
  return c;
}
// Callers branch on the mode once per row, so that the common rows' chunk loop sees the constant kRowFast.
__device__ __forceinline__ void codes8(const uint4& v, float s, float rs, int mode, float (&m)[8]) {
  if (mode == kRowFast) {
    codes8_fast(v, s, rs, m);
  } else {
    const Codes8 c = codes8_rare(v, s, rs, mode);
#pragma unroll
    for (int e = 0; e < 8; ++e) m[e] = c.m[e];
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
  const uint64_t nmg2 = pk2(-kRoundMagic, -kRoundMagic);
  uint32_t h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint64_t c2;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(c2) : "l"(pk2(m[2 * i], m[2 * i + 1])), "l"(nmg2));  // the codes, exact
    float lo, hi;
    upk2(c2, lo, hi);
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h[i]) : "f"(hi), "f"(lo));
  }
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
__device__ __forceinline__ void store8(const uint4& v, float s, float rs, int mode, int64_t row, int64_t K,
                                       int64_t idx, void* q, uint16_t* q16, const D& d) {
  float m[8];
  codes8(v, s, rs, mode, m);
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
__device__ __forceinline__ void store8_row(const uint4& v, float s, float rs, int mode, int64_t idx, uint2* q8,
                                           uint4* q16r) {
  float m[8];
  codes8(v, s, rs, mode, m);
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
// The same with NaN propagated.
__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
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
  __shared__ float red_nan[NG][G];  // second exchange, rows holding a NaN only
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
    uint32_t am2 = 0u;
#pragma unroll
    for (int c = 0; c < CH; ++c) am2 = absmax8_acc<true>(v[c], am2);
    float amax = warp_max_nan(absmax_of(am2));  // NaN if the row holds one
    if constexpr (G > 1) {
      // (red[grp][buf] was last read two rows ago, before the group's previous barrier)
      if (lane == 0) red[grp][buf][gl >> 5] = amax;
      group_sync<G>(grp);
      amax = red[grp][buf][0];
#pragma unroll
      for (int w = 1; w < G; ++w) amax = fmax_nan(amax, red[grp][buf][w]);
    }
    const bool nan_row = amax != amax;
    if (nan_row) {  // rare: the absmax over the row's other values (the group's threads all come here)
      am2 = 0u;
#pragma unroll
      for (int c = 0; c < CH; ++c) am2 = absmax8_acc<false>(v[c], am2);
      amax = warp_max(absmax_of(am2));
      if constexpr (G > 1) {
        // (red_nan[grp] was last read before the barrier of this row's first exchange)
        if (lane == 0) red_nan[grp][gl >> 5] = amax;
        group_sync<G>(grp);
        amax = red_nan[grp][0];
#pragma unroll
        for (int w = 1; w < G; ++w) amax = fmaxf(amax, red_nan[grp][w]);
      }
    }
    const float s = __fdiv_rn(amax, 127.0f);
    const float rs = s > 0.0f ? __frcp_rn(s) : 0.0f;
    const int mode = row_mode(s, nan_row);
    if (gl == 0) store_scale(s, row, scale, d);
    if constexpr (std::is_same<D, RowId>::value) {  // one destination: its row located once
      uint2* q8 = OUT != 1 ? reinterpret_cast<uint2*>(static_cast<int8_t*>(q) + row * K) : nullptr;
      uint4* qh = OUT != 0 ? reinterpret_cast<uint4*>(q16 + row * K) : nullptr;
      if (mode == kRowFast) {
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int64_t idx = gl + 32 * G * c;
          if (idx < nchunk) store8_row<OUT>(v[c], s, rs, kRowFast, idx, q8, qh);
        }
      } else {
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int64_t idx = gl + 32 * G * c;
          if (idx < nchunk) store8_row<OUT>(v[c], s, rs, mode, idx, q8, qh);
        }
      }
    } else {
      if (mode == kRowFast) {
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int64_t idx = gl + 32 * G * c;
          if (idx < nchunk) store8<OUT>(v[c], s, rs, kRowFast, row, K, idx, q, q16, d);
        }
      } else {
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int64_t idx = gl + 32 * G * c;
          if (idx < nchunk) store8<OUT>(v[c], s, rs, mode, row, K, idx, q, q16, d);
        }
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
  __shared__ float red[2][8];
  const int64_t nchunk = K / 8;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * K);
    uint32_t am2 = 0u;
    for (int64_t idx = threadIdx.x; idx < nchunk; idx += 256) am2 = absmax8_acc<true>(xr[idx], am2);
    float amax = warp_max_nan(absmax_of(am2));
    if ((threadIdx.x & 31) == 0) red[0][threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0][0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmax_nan(amax, red[0][w]);
    const bool nan_row = amax != amax;
    if (nan_row) {  // rare: the absmax over the row's other values, from a third read of the row
      am2 = 0u;
      for (int64_t idx = threadIdx.x; idx < nchunk; idx += 256) am2 = absmax8_acc<false>(xr[idx], am2);
      amax = warp_max(absmax_of(am2));
      if ((threadIdx.x & 31) == 0) red[1][threadIdx.x >> 5] = amax;
      __syncthreads();
      amax = red[1][0];
#pragma unroll
      for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[1][w]);
    }
    const float s = __fdiv_rn(amax, 127.0f);
    const float rs = s > 0.0f ? __frcp_rn(s) : 0.0f;
    const int mode = row_mode(s, nan_row);
    if (threadIdx.x == 0) store_scale(s, row, scale, d);
    for (int64_t idx = threadIdx.x; idx < nchunk; idx += 256) {
      store8<OUT>(xr[idx], s, rs, mode, row, K, idx, q, q16, d);
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
