// gemm_dec.cu -- exact INT8 contraction for decode-sized batches (M <= 64
// tokens), where the weight stream from HBM is the whole cost.
//
// Page "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子": §二
// npu_quant_matmul (INT8 x INT8 -> INT32, * x_scale * w_scale (+bias) ->
// BF16) and §四 (decode, small M, gets its own tiling).
//
// The weights stay INT8 in HBM (one byte per element, row-major, K
// contiguous).  Eight converter warps stream them with 16-byte loads straight
// into registers -- lane r of a warp reads its own row r, 64 contiguous bytes
// (a full DRAM burst) per half stage -- keep three 128-deep K stages of loads
// in flight, widen each row to integer-valued FP16 and store it into tensor
// memory, where tcgen05.mma reads its A operand.
// No copy engine and no shared-memory staging touch the large operand (the
// tensor-copy engine's per-row request rate caps a weight stream far below the
// HBM share of one SM).  The 64-token activation slice of each stage is widened
// into two 128-byte-swizzled K-major FP16 tiles in shared memory (the B
// operand).  The MMA is M = 128 weight rows x N = 64 tokens x K = 16 into an
// FP32 TMEM accumulator; each CTA covers at most 1024 of K, so the accumulator
// holds an exact integer (|partial| <= 1024 * 2^14 = 2^24).
//
// K is split over `ksplit` CTAs per 128-row block.  The launch is cooperative
// (every CTA resident at once), so the split-K reduction needs no second
// kernel: each CTA stores its exact int32 partial tile token-major into the
// workspace with coalesced stores, bumps an arrival counter for its row block
// and waits (bounded) until all `ksplit` partials are in; then every CTA sums
// its share of the rows over the partials with 16-byte loads issued together,
// applies the dequant epilogue and writes BF16 (or the INT32 sums).  A second
// counter tells the last reader to zero both counters.
//
// Warps: 0 TMEM owner + MMA issuer; 1-8 converters, then epilogue (warp w
// owns TMEM lanes 32*(w%4).. and K half / token half (w-1)/4).  All waits are
// bounded.
#include <mutex>

#include "kernels.cuh"
#include "tc_common.cuh"

namespace w8a8 {

namespace {

using namespace tc;

constexpr int DC_ROWS = 128;  // weight rows per CTA (MMA M)
constexpr int DC_TOK = 64;    // token columns (MMA N)
constexpr int DC_BK = 128;    // K per stage
constexpr int DC_SF = 3;      // fp16 / TMEM stages
constexpr int DC_PF = 3;      // stages of loads in flight per converter thread
constexpr uint32_t DC_B_SUB = DC_TOK * 128;    // one 64-K fp16 sub-tile (8 KB)
constexpr uint32_t DC_B_BYTES = 2 * DC_B_SUB;  // 128 K of fp16 activations
constexpr uint32_t DC_RING_BYTES = DC_SF * DC_B_BYTES;
constexpr int DC_CONV_WARPS = 8;
constexpr int DC_THREADS = 32 * (1 + DC_CONV_WARPS);
constexpr uint32_t DC_TMEM_COLS = 256;
constexpr uint32_t DC_A_COLS = DC_BK / 2;         // 64 columns of fp16 pairs per A stage
constexpr uint32_t DC_D_COL = DC_SF * DC_A_COLS;  // accumulator columns [192, 256)
constexpr int DC_MAX_KB = kChunkK / DC_BK;        // 8 stages = 1024 of K per CTA
constexpr int DC_MAX_KSPLIT = 16;
constexpr uint32_t kIdescDec = (1u << 4) | (uint32_t(DC_TOK >> 3) << 17) | (uint32_t(DC_ROWS >> 4) << 24);
static_assert(DC_B_BYTES % 1024 == 0, "1024-byte aligned stages");
static_assert(DC_D_COL + DC_TOK <= DC_TMEM_COLS, "tensor memory budget");

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// 16 int8 (one 16-byte chunk) -> 8 words of fp16 pairs.
__device__ __forceinline__ void widen16(const uint4& x, uint32_t* h) {
  s8x4_to_f16x4(x.x, h[0], h[1]);
  s8x4_to_f16x4(x.y, h[2], h[3]);
  s8x4_to_f16x4(x.z, h[4], h[5]);
  s8x4_to_f16x4(x.w, h[6], h[7]);
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Workspace of the decode engine: partial tiles [nblk][ksplit][DC_TOK][DC_ROWS]
// int32 (token-major), then two arrival counters per row block.
struct DecWs {
  int32_t* part;
  uint32_t* cnt_in;
  uint32_t* cnt_out;
};

template <int MODE>
__global__ void __launch_bounds__(DC_THREADS, 1)
dec_gemm_kernel(const GemmArgs a, const DecWs ws) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_ready[DC_SF];
  __shared__ __align__(8) uint64_t bar_emptyf[DC_SF];
  __shared__ __align__(8) uint64_t bar_accf;
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;
  __shared__ int s_bad;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int rank = blockIdx.x;  // split of K
  const int ksplit = gridDim.x;
  const int rb = blockIdx.y;    // 128-row weight block
  const int64_t M = a.R, N = a.N, K = a.K;
  const int64_t KC = K / 16;
  const int nkb = static_cast<int>((K + DC_BK - 1) / DC_BK);
  const int kb0 = static_cast<int>(static_cast<int64_t>(nkb) * rank / ksplit);
  const int kb1 = static_cast<int>(static_cast<int64_t>(nkb) * (rank + 1) / ksplit);
  const int my = kb1 - kb0;

  uint8_t* ringb = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t ringb_base = smem_u32(ringb);
  int32_t* my_part = ws.part + (static_cast<int64_t>(rb) * ksplit + rank) * (DC_TOK * DC_ROWS);

  if (tid == 0) {
    s_abort = 0;
    s_bad = 0;
    const PackedHeader* h = static_cast<const PackedHeader*>(a.packed);
    if (h->magic != kPackMagic || h->version != kPackVersion || h->E != 1 || h->N != N || h->K != K ||
        (h->flags & W8A8_PACK_GATE_UP) != 0u)
      s_bad = W8A8_ERR_PACKED;
    for (int f = 0; f < DC_SF; ++f) {
      mbar_init(smem_u32(&bar_ready[f]), DC_CONV_WARPS);
      mbar_init(smem_u32(&bar_emptyf[f]), 1);
    }
    mbar_init(smem_u32(&bar_accf), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem_base)),
                 "r"(DC_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const bool run = (s_bad == 0);
  if (!run && tid == 0 && rank == 0 && rb == 0) set_status(a.status, static_cast<uint32_t>(s_bad), 0u);

  if (run && warp == 0) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      for (int i = 0; i < my && !s_abort; ++i) {
        const int f = i % DC_SF;
        const uint32_t ph = static_cast<uint32_t>(i / DC_SF) & 1u;
        if (!mbar_wait(smem_u32(&bar_ready[f]), ph, &s_abort, a.status, 12u)) break;
        tc_fence_after();
        const uint32_t bsub0 = ringb_base + f * DC_B_BYTES;
#pragma unroll
        for (int kk = 0; kk < DC_BK / 16; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(bsub0 + (kk >> 2) * DC_B_SUB) + 2u * (kk & 3);
          tc_mma_tmem_a(tmem_base + DC_D_COL, tmem_base + f * DC_A_COLS + 8u * kk, bdesc, kIdescDec,
                        (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&bar_emptyf[f]));
      }
      tc_commit(smem_u32(&bar_accf));
    }
  } else if (run) {
    // ------------------------------------------------ converters, then epilogue
    const int q = warp & 3;           // TMEM lane quadrant
    const int half = (warp - 1) >> 2;  // K half of each stage (chunks 4*half..4*half+3)
    const int row = 32 * q + lane;     // weight row inside the block == TMEM lane
    const int ct = tid - 32;           // 0..255
    // this lane's weight row (row-major int8 payload, K contiguous); rows past N read as zero
    const int64_t grow = static_cast<int64_t>(rb) * DC_ROWS + row;
    const bool row_ok = grow < N;
    const uint8_t* wrow = reinterpret_cast<const uint8_t*>(a.packed) +
                          static_cast<const PackedHeader*>(a.packed)->i8_offset + (row_ok ? grow : 0) * K;
    const uint8_t* xq = reinterpret_cast<const uint8_t*>(a.q);
    uint4 wr[DC_PF][4];
    uint4 xr[DC_PF][2];
    // loads of stage i into register buffer B (B is a compile-time constant at every use)
#define DC_LOAD(B, I)                                                                                  \
    do {                                                                                               \
      const int ld_i = (I);                                                                              \
      if (ld_i < my) {                                                                                   \
        const int64_t kc0 = static_cast<int64_t>(kb0 + ld_i) * (DC_BK / 16) + 4 * half;                 \
        _Pragma("unroll") for (int c = 0; c < 4; ++c) {                                                \
          wr[B][c] = (row_ok && kc0 + c < KC) ? ldg_nc(wrow + (kc0 + c) * 16) : make_uint4(0, 0, 0, 0);     \
        }                                                                                              \
        _Pragma("unroll") for (int j = 0; j < 2; ++j) {                                                \
          const int p = ct + 256 * j;                                                                  \
          const int t = p >> 3, c = p & 7;                                                             \
          const int64_t k = static_cast<int64_t>(kb0 + ld_i) * DC_BK + 16 * c;                           \
          xr[B][j] = (t < M && k < K) ? ldg_nc(xq + t * K + k) : make_uint4(0, 0, 0, 0);               \
        }                                                                                              \
      }                                                                                                \
    } while (0)
    // widen stage i from register buffer B into TMEM A / smem B stage i % DC_SF, refill B with stage i + DC_PF
#define DC_STEP(B, I)                                                                                  \
    if ((I) < my && ok) {                                                                              \
      const int st_i = (I);                                                                              \
      const int f = st_i % DC_SF;                                                                        \
      const uint32_t phf = static_cast<uint32_t>(st_i / DC_SF) & 1u;                                    \
      int got = 0;                                                                                     \
      if (lane == 0) got = mbar_wait(smem_u32(&bar_emptyf[f]), phf ^ 1u, &s_abort, a.status, 15u) ? 1 : 0; \
      got = __shfl_sync(0xffffffffu, got, 0);                                                          \
      if (!got) {                                                                                      \
        ok = false;                                                                                    \
      } else {                                                                                         \
        uint32_t v[32];                                                                                \
        _Pragma("unroll") for (int c = 0; c < 4; ++c) widen16(wr[B][c], &v[8 * c]);                   \
        uint8_t* bt = ringb + f * DC_B_BYTES;                                                          \
        _Pragma("unroll") for (int j = 0; j < 2; ++j) {                                                \
          const int p = ct + 256 * j;                                                                  \
          const int t = p >> 3, c = p & 7;                                                             \
          uint32_t hh[8];                                                                              \
          widen16(xr[B][j], hh);                                                                       \
          uint8_t* brow = bt + (c >> 2) * DC_B_SUB + t * 128;                                          \
          const int cc = (c & 3) * 2;                                                                  \
          *reinterpret_cast<uint4*>(brow + ((cc ^ (t & 7)) << 4)) = make_uint4(hh[0], hh[1], hh[2], hh[3]); \
          *reinterpret_cast<uint4*>(brow + (((cc + 1) ^ (t & 7)) << 4)) = make_uint4(hh[4], hh[5], hh[6], hh[7]); \
        }                                                                                              \
        DC_LOAD(B, st_i + DC_PF);                                                                        \
        tmem_st32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + f * DC_A_COLS + 32u * half, v);   \
        tmem_wait_st();                                                                                \
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");                                   \
        tc_fence_before();                                                                             \
        __syncwarp();                                                                                  \
        if (lane == 0) mbar_arrive(smem_u32(&bar_ready[f]));                                          \
      }                                                                                                \
    }
    static_assert(DC_PF == 3, "the pipeline below is written for three register buffers");
    bool ok = true;
    DC_LOAD(0, 0);
    DC_LOAD(1, 1);
    DC_LOAD(2, 2);
    for (int i = 0; i < my && ok; i += DC_PF) {
      DC_STEP(0, i)
      DC_STEP(1, i + 1)
      DC_STEP(2, i + 2)
    }
#undef DC_STEP
#undef DC_LOAD
    // exact partial -> workspace, token-major (lanes store consecutive rows);
    // this warp drains tokens [32*half, 32*half + 32)
    int got = 1;
    if (my > 0) {
      if (lane == 0) got = mbar_wait(smem_u32(&bar_accf), 0u, &s_abort, a.status, 14u) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
    }
    if (my > 0 && got && ok) {
      tc_fence_after();
      uint32_t d[32];
      tmem_ld32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + DC_D_COL + 32u * half, d);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 32; ++c) my_part[(32 * half + c) * DC_ROWS + row] = __float2int_rn(__uint_as_float(d[c]));
    } else {
#pragma unroll 8
      for (int c = 0; c < 32; ++c) my_part[(32 * half + c) * DC_ROWS + row] = 0;
    }
    tc_fence_before();
  }
  __syncwarp();
  __threadfence();
  __syncthreads();

  // ---- all partials of this row block in: bounded wait on the arrival counter
  __shared__ int s_ready;
  if (tid == 0) {
    atomicAdd(&ws.cnt_in[rb], 1u);
    int ok = 1;
    if (ld_acquire_u32(&ws.cnt_in[rb]) < static_cast<uint32_t>(ksplit)) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_u32(&ws.cnt_in[rb]) < static_cast<uint32_t>(ksplit)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          set_status(a.status, W8A8_ERR_DEVICE_TIMEOUT, 16u);
          ok = 0;
          break;
        }
      }
    }
    s_ready = ok;
  }
  __syncthreads();

  // ---- split-K reduction and epilogue: this CTA owns row chunks [c0, c1) of 8 rows
  if (run && s_ready && !s_abort) {
    const int c0 = (DC_ROWS / 8) * rank / ksplit;
    const int c1 = (DC_ROWS / 8) * (rank + 1) / ksplit;
    const int nch = c1 - c0;
    const int32_t* blk = ws.part + static_cast<int64_t>(rb) * ksplit * (DC_TOK * DC_ROWS);
    for (int task = tid; task < DC_TOK * nch; task += DC_THREADS) {
      const int t = task / nch;
      const int r0 = (c0 + task % nch) * 8;
      if (t >= M) continue;
      int sum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      // all partial loads of a batch are issued before any is consumed
      for (int j0 = 0; j0 < ksplit; j0 += 8) {
        int4 lo[8], hi[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j0 + j < ksplit) {
            const int4* src = reinterpret_cast<const int4*>(blk + static_cast<int64_t>(j0 + j) * (DC_TOK * DC_ROWS) +
                                                            t * DC_ROWS + r0);
            lo[j] = __ldcg(src);
            hi[j] = __ldcg(src + 1);
          } else {
            lo[j] = make_int4(0, 0, 0, 0);
            hi[j] = make_int4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          sum[0] += lo[j].x; sum[1] += lo[j].y; sum[2] += lo[j].z; sum[3] += lo[j].w;
          sum[4] += hi[j].x; sum[5] += hi[j].y; sum[6] += hi[j].z; sum[7] += hi[j].w;
        }
      }
      const int64_t n0 = static_cast<int64_t>(rb) * DC_ROWS + r0;
      if (n0 >= N) continue;
      if constexpr (MODE == EPI_ACC) {
        int32_t* dst = static_cast<int32_t*>(a.out) + t * N + n0;
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (n0 + r < N) dst[r] = sum[r];
      } else {
        const float sx = a.x_scale[t];
        uint16_t o[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          float fv = 0.0f;
          if (n0 + r < N) {
            fv = dequant(sum[r], sx, a.w_scale[n0 + r]);
            if (a.bias) fv = __fadd_rn(fv, bf16_bits_to_f32(a.bias[n0 + r]));
          }
          o[r] = f32_to_bf16_bits(fv);
        }
        uint16_t* dst = static_cast<uint16_t*>(a.out) + t * N + n0;
        if (((reinterpret_cast<uintptr_t>(dst) & 15u) == 0u) && n0 + 8 <= N) {
          *reinterpret_cast<uint4*>(dst) = make_uint4(o[0] | (uint32_t(o[1]) << 16), o[2] | (uint32_t(o[3]) << 16),
                                                      o[4] | (uint32_t(o[5]) << 16), o[6] | (uint32_t(o[7]) << 16));
        } else {
#pragma unroll
          for (int r = 0; r < 8; ++r)
            if (n0 + r < N) dst[r] = o[r];
        }
      }
    }
  }
  __syncthreads();
  // the last CTA of the row block to finish reading zeroes both counters
  if (tid == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(&ws.cnt_out[rb], 1u);
    if (prev == static_cast<uint32_t>(ksplit - 1)) {
      atomicExch(&ws.cnt_in[rb], 0u);
      atomicExch(&ws.cnt_out[rb], 0u);
    }
  }

  if (s_abort) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 20000000ull) {
    }
  }
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(DC_TMEM_COLS)
                 : "memory");
  }
}

constexpr size_t kDecSmem = DC_RING_BYTES + 1024;

// CTAs of the decode kernel that can be resident at once on the current device.
int dec_resident_ctas() {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev] == 0) {
    int per_sm = 0, sms = 0;
    cudaFuncSetAttribute(dec_gemm_kernel<EPI_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(kDecSmem));
    cudaFuncSetAttribute(dec_gemm_kernel<EPI_ACC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(kDecSmem));
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dec_gemm_kernel<EPI_BF16>, DC_THREADS, kDecSmem) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[dev] = per_sm * sms;
  }
  return cache[dev];
}

template <int MODE>
cudaError_t launch_dec_mode(const GemmArgs& a, const DecWs& ws, int ksplit, int nblk, cudaStream_t stream) {
  auto k = dec_gemm_kernel<MODE>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ksplit), static_cast<unsigned>(nblk), 1);
  cfg.blockDim = dim3(DC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = kDecSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, a, ws);
}

}  // namespace

size_t dec_ws_bytes(int64_t N) {
  const int64_t nblk = (N + DC_ROWS - 1) / DC_ROWS;
  return align_up(static_cast<uint64_t>(nblk) * DC_MAX_KSPLIT * DC_TOK * DC_ROWS * 4, 256) +
         align_up(static_cast<uint64_t>(nblk) * 2 * 4, 256);
}

// K split for the decode engine: every CTA covers at most 1024 of K (one
// exact fp32 chunk) and all nblk * ksplit CTAs must be resident at once; among
// those, the largest split (most CTAs streaming weights).  0 = shape unsuited.
int dec_plan_ksplit(int64_t M, int64_t N, int64_t K, int num_sms) {
  (void)num_sms;
  if (M < 1 || M > DC_TOK || K > static_cast<int64_t>(DC_MAX_KSPLIT) * kChunkK) return 0;
  const int64_t nkb = (K + DC_BK - 1) / DC_BK;
  const int64_t nblk = (N + DC_ROWS - 1) / DC_ROWS;
  const int resident = dec_resident_ctas();
  int best = 0;
  for (int ks = 1; ks <= DC_MAX_KSPLIT; ++ks) {
    if (ks > nkb || nblk * ks > resident) break;
    if ((nkb + ks - 1) / ks <= DC_MAX_KB) best = ks;
  }
  return best;
}

cudaError_t launch_dec_gemm(const GemmArgs& a, int ksplit, void* dec_ws, cudaStream_t stream) {
  if (a.R == 0) return cudaSuccess;
  const int nblk = static_cast<int>((a.N + DC_ROWS - 1) / DC_ROWS);
  DecWs ws;
  uint8_t* b = static_cast<uint8_t*>(dec_ws);
  ws.part = reinterpret_cast<int32_t*>(b);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(
      b + align_up(static_cast<uint64_t>(nblk) * DC_MAX_KSPLIT * DC_TOK * DC_ROWS * 4, 256));
  ws.cnt_in = cnt;
  ws.cnt_out = cnt + nblk;
  if (a.mode == EPI_ACC) return launch_dec_mode<EPI_ACC>(a, ws, ksplit, nblk, stream);
  return launch_dec_mode<EPI_BF16>(a, ws, ksplit, nblk, stream);
}

}  // namespace w8a8
