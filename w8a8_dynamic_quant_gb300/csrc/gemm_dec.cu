// gemm_dec.cu -- exact INT8 contraction for decode-sized batches (M <= 64
// tokens), where the weight stream from HBM is the whole cost.
//
// Page "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子": §二
// npu_quant_matmul (INT8 x INT8 -> INT32, * x_scale * w_scale (+bias) ->
// BF16) and §四 (decode, small M, gets its own tiling).
//
// The weights stay INT8 in HBM (one byte per element).  Per 128-deep K step a
// TMA copy brings a 128-row x 128-byte int8 weight tile and the 64-token x
// 128-byte int8 activation tile into shared memory with the 128-byte swizzle:
// rows of 128 bytes keep the copy engine's row requests per byte low (its rate
// is bounded by rows, not bytes), and the swizzle makes the converters' row
// reads bank-conflict-free.  Four converter warps widen each weight row to 128
// integer-valued FP16 and store them straight into tensor memory, where
// tcgen05.mma reads its A operand (no shared-memory write for the large
// operand), and widen the activations into two 128-byte-swizzled K-major FP16
// tiles (the B operand).  The int8 ring (6 stages) and the FP16/TMEM ring (3
// stages) have their own barriers, so an int8 stage is refilled as soon as it
// has been widened.  The MMA is M = 128 weight rows x N = 64 tokens x K = 16
// into an FP32 TMEM accumulator; each CTA covers at most 1024 of K, so the
// accumulator holds an exact integer (|partial| <= 1024 * 2^14 = 2^24).
//
// K is split over `ksplit` CTAs per 128-row block.  The launch is cooperative
// (every CTA resident at once), so the split-K reduction needs no second
// kernel: each CTA stores its exact int32 partial tile token-major into the
// workspace with coalesced stores, bumps an arrival counter for its row block
// and waits (bounded) until all `ksplit` partials are in; then every CTA sums
// its share of the rows over the partials with 16-byte loads, applies the
// dequant epilogue and writes BF16 (or the INT32 sums).  A second counter
// tells the last reader to zero both counters, leaving the workspace clean.
//
// Warps: 0 TMA producer, 1 TMEM owner + MMA issuer, 2-5 converters, then
// epilogue (warp w owns TMEM lanes 32*(w%4)..).  All waits are bounded.
#include <mutex>

#include "kernels.cuh"
#include "tc_common.cuh"

namespace w8a8 {

namespace {

using namespace tc;

constexpr int DC_ROWS = 128;  // weight rows per CTA (MMA M)
constexpr int DC_TOK = 64;    // token columns (MMA N)
constexpr int DC_BK = 128;    // K (int8 bytes) per stage
constexpr int DC_S8 = 6;      // int8 stages
constexpr int DC_SF = 3;      // fp16 / TMEM stages
constexpr uint32_t DC_W_BYTES = DC_ROWS * DC_BK;  // 16 KB
constexpr uint32_t DC_X_BYTES = DC_TOK * DC_BK;   // 8 KB
constexpr uint32_t DC_S8_BYTES = DC_W_BYTES + DC_X_BYTES;
constexpr uint32_t DC_B_SUB = DC_TOK * 128;       // one 64-K fp16 sub-tile (8 KB)
constexpr uint32_t DC_B_BYTES = 2 * DC_B_SUB;     // 128 K of fp16 activations
constexpr uint32_t DC_RING_BYTES = DC_S8 * DC_S8_BYTES + DC_SF * DC_B_BYTES;
constexpr int DC_THREADS = 192;
constexpr int DC_CONV_WARPS = 4;
constexpr uint32_t DC_TMEM_COLS = 256;
constexpr uint32_t DC_A_COLS = DC_BK / 2;          // 64 columns of fp16 pairs per A stage
constexpr uint32_t DC_D_COL = DC_SF * DC_A_COLS;   // accumulator columns [192, 256)
constexpr int DC_MAX_KB = kChunkK / DC_BK;         // 8 stages = 1024 of K per CTA
constexpr int DC_MAX_KSPLIT = 16;
constexpr uint32_t kIdescDec = (1u << 4) | (uint32_t(DC_TOK >> 3) << 17) | (uint32_t(DC_ROWS >> 4) << 24);
static_assert(DC_S8_BYTES % 1024 == 0 && DC_B_BYTES % 1024 == 0, "1024-byte aligned stages");
static_assert(DC_D_COL + DC_TOK <= DC_TMEM_COLS, "tensor memory budget");

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
dec_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const GemmArgs a,
                const DecWs ws) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full8[DC_S8];
  __shared__ __align__(8) uint64_t bar_free8[DC_S8];
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
  const int nkb = static_cast<int>((K + DC_BK - 1) / DC_BK);
  const int kb0 = static_cast<int>(static_cast<int64_t>(nkb) * rank / ksplit);
  const int kb1 = static_cast<int>(static_cast<int64_t>(nkb) * (rank + 1) / ksplit);
  const int my = kb1 - kb0;

  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring8 = ring;                        // int8 stages
  uint8_t* ringb = ring + DC_S8 * DC_S8_BYTES;  // fp16 B stages
  const uint32_t ring8_base = smem_u32(ring8);
  const uint32_t ringb_base = smem_u32(ringb);
  int32_t* my_part = ws.part + (static_cast<int64_t>(rb) * ksplit + rank) * (DC_TOK * DC_ROWS);

  if (tid == 0) {
    s_abort = 0;
    s_bad = 0;
    const PackedHeader* h = static_cast<const PackedHeader*>(a.packed);
    if (h->magic != kPackMagic || h->version != kPackVersion || h->E != 1 || h->N != N || h->K != K ||
        (h->flags & W8A8_PACK_GATE_UP) != 0u)
      s_bad = W8A8_ERR_PACKED;
    for (int s = 0; s < DC_S8; ++s) {
      mbar_init(smem_u32(&bar_full8[s]), 1);
      mbar_init(smem_u32(&bar_free8[s]), DC_CONV_WARPS);
    }
    for (int f = 0; f < DC_SF; ++f) {
      mbar_init(smem_u32(&bar_ready[f]), DC_CONV_WARPS);
      mbar_init(smem_u32(&bar_emptyf[f]), 1);
    }
    mbar_init(smem_u32(&bar_accf), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int i = 0; i < my && !s_abort; ++i) {
        const int s = i % DC_S8;
        const uint32_t ph = static_cast<uint32_t>(i / DC_S8) & 1u;
        if (!mbar_wait(smem_u32(&bar_free8[s]), ph ^ 1u, &s_abort, a.status, 11u)) break;
        const uint32_t full = smem_u32(&bar_full8[s]);
        mbar_expect_tx(full, DC_S8_BYTES);
        const uint32_t st = ring8_base + s * DC_S8_BYTES;
        tma_load_2d(st, &tmW, (kb0 + i) * DC_BK, rb * DC_ROWS, full);
        tma_load_2d(st + DC_W_BYTES, &tmX, (kb0 + i) * DC_BK, 0, full);
      }
    }
  } else if (run && warp == 1) {
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
    const int q = warp & 3;
    const int row = 32 * q + lane;  // weight row inside the block == TMEM lane
    const int ct = tid - 64;        // 0..127
    for (int i = 0; i < my; ++i) {
      const int s = i % DC_S8;
      const uint32_t ph8 = static_cast<uint32_t>(i / DC_S8) & 1u;
      const int f = i % DC_SF;
      const uint32_t phf = static_cast<uint32_t>(i / DC_SF) & 1u;
      int got = 0;
      if (lane == 0)
        got = (mbar_wait(smem_u32(&bar_full8[s]), ph8, &s_abort, a.status, 13u) &&
               mbar_wait(smem_u32(&bar_emptyf[f]), phf ^ 1u, &s_abort, a.status, 15u))
                  ? 1
                  : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      const uint8_t* st = ring8 + s * DC_S8_BYTES;
      // weight row (128 int8 in swizzled 16-byte chunks) -> 128 fp16 -> TMEM lane `row`
      uint32_t v[64];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 w4 = *reinterpret_cast<const uint4*>(st + row * 128 + ((c ^ (row & 7)) << 4));
        widen16(w4, &v[8 * c]);
      }
      // activations: 64 tokens x 8 chunks of 16 int8 -> fp16 sub-tiles (K 0-63 | K 64-127)
      uint8_t* bt = ringb + f * DC_B_BYTES;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int p = ct + 128 * j;
        const int t = p >> 3, c = p & 7;
        const uint4 x4 = *reinterpret_cast<const uint4*>(st + DC_W_BYTES + t * 128 + ((c ^ (t & 7)) << 4));
        uint32_t h[8];
        widen16(x4, h);
        uint8_t* brow = bt + (c >> 2) * DC_B_SUB + t * 128;
        const int cc = (c & 3) * 2;
        *reinterpret_cast<uint4*>(brow + ((cc ^ (t & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(brow + (((cc + 1) ^ (t & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_free8[s]));  // int8 stage consumed
      tmem_st64(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + f * DC_A_COLS, v);
      tmem_wait_st();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_ready[f]));
    }
    // exact partial -> workspace, token-major (lanes store consecutive rows)
    int got = 1;
    if (my > 0) {
      if (lane == 0) got = mbar_wait(smem_u32(&bar_accf), 0u, &s_abort, a.status, 14u) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
    }
    if (my > 0 && got) {
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < DC_TOK / 32; ++j) {
        uint32_t d[32];
        tmem_ld32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + DC_D_COL + 32u * j, d);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) my_part[(32 * j + c) * DC_ROWS + row] = __float2int_rn(__uint_as_float(d[c]));
      }
    } else {
#pragma unroll 8
      for (int t = 0; t < DC_TOK; ++t) my_part[t * DC_ROWS + row] = 0;
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
      for (int j = 0; j < ksplit; ++j) {
        const int4* src = reinterpret_cast<const int4*>(blk + static_cast<int64_t>(j) * (DC_TOK * DC_ROWS) +
                                                        t * DC_ROWS + r0);
        const int4 lo = __ldcg(src);
        const int4 hi = __ldcg(src + 1);
        sum[0] += lo.x; sum[1] += lo.y; sum[2] += lo.z; sum[3] += lo.w;
        sum[4] += hi.x; sum[5] += hi.y; sum[6] += hi.z; sum[7] += hi.w;
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
  if (warp == 1) {
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
cudaError_t launch_dec_mode(const CUtensorMap& mw, const CUtensorMap& mx, const GemmArgs& a, const DecWs& ws,
                            int ksplit, int nblk, cudaStream_t stream) {
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
  return cudaLaunchKernelEx(&cfg, k, mw, mx, a, ws);
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
  CUtensorMap mw, mx;
  const uint8_t* packed = static_cast<const uint8_t*>(a.packed);
  const void* w_i8 = packed + pack_layout(1, a.N, a.K, 0u).i8_offset;
  if (!encode_map_2d(&mw, w_i8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.N, a.K, DC_BK, DC_ROWS,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_map_2d(&mx, a.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.R, a.K, DC_BK, DC_TOK, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int nblk = static_cast<int>((a.N + DC_ROWS - 1) / DC_ROWS);
  DecWs ws;
  uint8_t* b = static_cast<uint8_t*>(dec_ws);
  ws.part = reinterpret_cast<int32_t*>(b);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(
      b + align_up(static_cast<uint64_t>(nblk) * DC_MAX_KSPLIT * DC_TOK * DC_ROWS * 4, 256));
  ws.cnt_in = cnt;
  ws.cnt_out = cnt + nblk;
  if (a.mode == EPI_ACC) return launch_dec_mode<EPI_ACC>(mw, mx, a, ws, ksplit, nblk, stream);
  return launch_dec_mode<EPI_BF16>(mw, mx, a, ws, ksplit, nblk, stream);
}

}  // namespace w8a8
