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
//
// The MXFP8 contraction y[m,n] = bf16(sum_g Sa[m,g] Sw[n,g] sum_{k in g}
// a[m,k] w[n,k]) (section 5: npu_quant_matmul with both E8M0 scales, group
// sizes [1,1,32]) runs here on the warp-level FP8 tensor instruction: one
// m16n8k32 E4M3 product per 32-value group, its binary32 partial scaled by
// the group's two powers of two and added into binary32 accumulators.
// 128x128 CTA tiles, 128-deep stages staged by cp.async, eight warps of
// 64x32.
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


constexpr int MXM_BM = 128, MXM_BN = 128, MXM_BK = 128;  // BK in elements = bytes
constexpr int MXM_STRIDE = MXM_BK + 16;                    // padded row: conflict-free fragment loads
constexpr int MXM_THREADS = 256;
constexpr int MXM_TILE_BYTES = MXM_BM * MXM_STRIDE;        // one operand tile of a stage
constexpr int MXM_SC_BYTES = MXM_BM * (MXM_BK / 32);       // its scale bytes
constexpr int MXM_STAGE_BYTES = 2 * MXM_TILE_BYTES + 2 * MXM_SC_BYTES;
constexpr size_t MXM_SMEM = 2 * static_cast<size_t>(MXM_STAGE_BYTES);

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}

// 2^(b - 127) of an E8M0 byte (0xFF: NaN).
__device__ __forceinline__ float e8m0(uint32_t b) {
  if (b == 0xFFu) return __uint_as_float(0x7fc00000u);
  return b == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

__device__ __forceinline__ void mma_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(MXM_THREADS, 1) mx_matmul_kernel(const uint8_t* __restrict__ qa,
                                                                   const uint8_t* __restrict__ sa, int M, int K,
                                                                   const uint8_t* __restrict__ qw,
                                                                   const uint8_t* __restrict__ sw, int N,
                                                                   uint16_t* __restrict__ y) {
  extern __shared__ __align__(16) uint8_t mxm_smem[];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int wm = warp >> 2, wn = warp & 3;  // warp tile: rows wm*64 .. +64, cols wn*32 .. +32
  const int m0 = blockIdx.y * MXM_BM, n0 = blockIdx.x * MXM_BN;
  const int G = K / 32;
  const int nkb = K / MXM_BK;

  pdl_trigger();
  pdl_wait();

  auto stage_ptr = [&](int s) { return mxm_smem + static_cast<size_t>(s) * MXM_STAGE_BYTES; };
  auto load_stage = [&](int s, int kb) {
    uint8_t* st = stage_ptr(s);
    uint8_t* As = st;
    uint8_t* Bs = st + MXM_TILE_BYTES;
    uint8_t* SAs = st + 2 * MXM_TILE_BYTES;
    uint8_t* SBs = SAs + MXM_SC_BYTES;
    for (int c = tid; c < MXM_BM * (MXM_BK / 16); c += MXM_THREADS) {
      const int row = c >> 3, ch = c & 7;
      const int ga = m0 + row, gb = n0 + row;
      const uint8_t* srca = qa + static_cast<int64_t>(ga < M ? ga : 0) * K + kb * MXM_BK + ch * 16;
      const uint8_t* srcb = qw + static_cast<int64_t>(gb < N ? gb : 0) * K + kb * MXM_BK + ch * 16;
      cp_async_16(smem_u32(As + row * MXM_STRIDE + ch * 16), srca, ga < M ? 16 : 0);
      cp_async_16(smem_u32(Bs + row * MXM_STRIDE + ch * 16), srcb, gb < N ? 16 : 0);
    }
    if (tid < MXM_BM) {  // the four group scales of row tid of each operand
      const int ga = m0 + tid, gb = n0 + tid;
      cp_async_4(smem_u32(SAs + tid * 4), sa + static_cast<int64_t>(ga < M ? ga : 0) * G + kb * 4, ga < M ? 4 : 0);
      cp_async_4(smem_u32(SBs + tid * 4), sw + static_cast<int64_t>(gb < N ? gb : 0) * G + kb * 4, gb < N ? 4 : 0);
    }
    cp_async_commit();
  };

  float acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0.0f;

  load_stage(0, 0);
  for (int kb = 0; kb < nkb; ++kb) {
    if (kb + 1 < nkb) {
      load_stage((kb + 1) & 1, kb + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint8_t* st = stage_ptr(kb & 1);
    const uint8_t* As = st;
    const uint8_t* Bs = st + MXM_TILE_BYTES;
    const uint8_t* SAs = st + 2 * MXM_TILE_BYTES;
    const uint8_t* SBs = SAs + MXM_SC_BYTES;
#pragma unroll
    for (int g = 0; g < MXM_BK / 32; ++g) {
      uint32_t af[4][4], bf[4][2];
      float sr[4][2], sc[4][2];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int r0 = wm * 64 + mt * 16 + gid;
        const uint8_t* p0 = As + r0 * MXM_STRIDE + g * 32 + tig * 4;
        const uint8_t* p1 = p0 + 8 * MXM_STRIDE;
        af[mt][0] = *reinterpret_cast<const uint32_t*>(p0);
        af[mt][1] = *reinterpret_cast<const uint32_t*>(p1);
        af[mt][2] = *reinterpret_cast<const uint32_t*>(p0 + 16);
        af[mt][3] = *reinterpret_cast<const uint32_t*>(p1 + 16);
        sr[mt][0] = e8m0(SAs[r0 * 4 + g]);
        sr[mt][1] = e8m0(SAs[(r0 + 8) * 4 + g]);
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int c0 = wn * 32 + nt * 8;
        const uint8_t* p = Bs + (c0 + gid) * MXM_STRIDE + g * 32 + tig * 4;
        bf[nt][0] = *reinterpret_cast<const uint32_t*>(p);
        bf[nt][1] = *reinterpret_cast<const uint32_t*>(p + 16);
        sc[nt][0] = e8m0(SBs[(c0 + tig * 2) * 4 + g]);
        sc[nt][1] = e8m0(SBs[(c0 + tig * 2 + 1) * 4 + g]);
      }
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          mma_e4m3(d, af[mt], bf[nt][0], bf[nt][1]);
          acc[mt][nt][0] = __fadd_rn(acc[mt][nt][0], __fmul_rn(__fmul_rn(d[0], sr[mt][0]), sc[nt][0]));
          acc[mt][nt][1] = __fadd_rn(acc[mt][nt][1], __fmul_rn(__fmul_rn(d[1], sr[mt][0]), sc[nt][1]));
          acc[mt][nt][2] = __fadd_rn(acc[mt][nt][2], __fmul_rn(__fmul_rn(d[2], sr[mt][1]), sc[nt][0]));
          acc[mt][nt][3] = __fadd_rn(acc[mt][nt][3], __fmul_rn(__fmul_rn(d[3], sr[mt][1]), sc[nt][1]));
        }
    }
    __syncthreads();  // every warp is done with this stage before it is refilled
  }

#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int m = m0 + wm * 64 + mt * 16 + gid + (r >= 2 ? 8 : 0);
        const int n = n0 + wn * 32 + nt * 8 + tig * 2 + (r & 1);
        if (m < M && n < N) y[static_cast<int64_t>(m) * N + n] = f32_to_bf16_bits(acc[mt][nt][r]);
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

cudaError_t launch_mx_matmul(const uint8_t* qa, const uint8_t* sa, int64_t M, int64_t K, const uint8_t* qw,
                             const uint8_t* sw, int64_t N, uint16_t* y, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  // per device: set on every call, like the other engines
  const cudaError_t e = cudaFuncSetAttribute(mx_matmul_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(MXM_SMEM));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((N + MXM_BN - 1) / MXM_BN), static_cast<unsigned>((M + MXM_BM - 1) / MXM_BM));
  return launch_pdl(mx_matmul_kernel, grid, dim3(MXM_THREADS), MXM_SMEM, stream, qa, sa, static_cast<int>(M),
                    static_cast<int>(K), qw, sw, static_cast<int>(N), y);
}

}  // namespace w8a8
