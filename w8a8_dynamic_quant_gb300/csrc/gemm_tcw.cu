// gemm_tcw.cu -- exact INT8 grouped contraction on the 5th-generation tensor
// cores with the weights read as INT8 and widened on chip: the MoE prefill
// W13 (+ SwiGLU) and W2 for packed weights without an FP16 copy.
//
// Page "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子": §三
// npu_grouped_matmul over group_list (INT8 x INT8 -> INT32, then * x_scale *
// w_scale -> BF16) and the W13 -> SwiGLU step; §四 (prefill, large M).
//
// Role.  The grouped contractions of MoE prefill normally read an FP16 copy of
// the weights (gemm_tc.cu).  This engine serves packed weights that carry no
// such copy: the weights stay INT8 in HBM (a third of the memory of INT8 +
// FP16) and are widened to integer-valued FP16 in tensor memory, where
// tcgen05.mma reads its A operand; the activations arrive as FP16 (the
// quantisation writes that copy) in shared memory as the B operand.  The
// tile is therefore transposed: D[weight row n, token t] = sum_k W[n,k] x[t,k],
// M = 128 weight rows, N = 128 tokens of one expert, K = 16 per instruction.
// Products |a*b| <= 2^14 are exact in FP32 and a fresh accumulator is started
// every 1024 of K, so every accumulator holds an exact integer.
//
// Tensor memory (512 columns): four A stages of 128 K (64 columns each, two
// FP16 per column) and two 128-column accumulators that alternate per
// 1024-deep chunk.  Shared memory: four stages of a 128-token x 128-K FP16
// activation tile (two 64-K sub-tiles, 128-byte swizzle) and a 128-row x
// 128-byte INT8 weight tile (128-byte swizzle), brought in by TMA.  The two
// CTAs of a cluster are scheduled together and take weight blocks 2p and 2p+1
// of the same tokens; each loads the activation tile itself with plain tensor
// copies (the second request is served from L2) and the CTAs exchange
// nothing, so each stage is freed by its own CTA's MMA commit.
//
// Warp roles (448 threads, one CTA per SM, persistent over tiles):
//   warp 0       TMA producer
//   warp 1       TMEM owner and MMA issuer
//   warps 2-5    converters: lane r of warp w widens weight row 32*(w%4)+r of
//                the stage into TMEM lane 32*(w%4)+r
//   warps 6-13   epilogue: warp w reads TMEM lanes 32*(w%4).. (weight rows)
//                and one half (64 tokens) of the tile's columns
// W13 + SwiGLU: the gate/up interleave puts gate channel j in tile row j%64
// and up channel j in row 64 + j%64, so the up warps hand their BF16 values
// to the gate warps through shared memory (mbarrier hand-off per tile).
// Every mbarrier wait is bounded (2 s): on expiry the CTA sets
// W8A8_ERR_DEVICE_TIMEOUT, lets in-flight copies land, frees TMEM and returns.
#include "kernels.cuh"
#include "tc_common.cuh"

namespace w8a8 {

namespace {

using namespace tc;

constexpr int W_BN = 128;  // weight rows per tile (MMA M)
constexpr int W_BT = 128;  // tokens per tile (MMA N)
constexpr int W_BK = 128;  // K per stage
constexpr int W_STAGES = 4;
constexpr int W_KB_PER_CHUNK = kChunkK / W_BK;  // 16
constexpr uint32_t W_X_SUB = W_BT * 64 * 2;     // fp16 activation sub-tile of 64 K (16 KB, one swizzle row per token)
constexpr uint32_t W_X_BYTES = 2 * W_X_SUB;      // 128 K of activations (32 KB)
constexpr uint32_t W_W_BYTES = W_BN * W_BK;      // int8 weight tile (16 KB)
constexpr uint32_t W_STAGE_BYTES = W_X_BYTES + W_W_BYTES;
constexpr int W_THREADS = 448;
constexpr int W_EPI0 = 6;  // first epilogue warp
constexpr int W_EPI_WARPS = 8;
constexpr int W_CONV_WARPS = 4;
constexpr uint32_t W_A_COLS = W_BK / 2;            // TMEM columns per A stage
constexpr uint32_t W_D_COL = W_STAGES * W_A_COLS;  // accumulators at [256, 384) and [384, 512)
static_assert(W_BK == 128, "a stage is one 128-byte weight row and two 64-K activation sub-tiles");
constexpr uint32_t W_TMEM_COLS = 512;
constexpr int W_GROUP_N = 16;  // n-blocks per rasterisation group (8 pairs)
constexpr int W_CLUSTER = 2;
constexpr int kMaxE = 1024;
constexpr uint32_t W_UP_BYTES = 2 * 2 * 64 * 32 * 2;  // up values: [gate warp pair][half][64 tokens][32 lanes] bf16
// kind::f16 instruction descriptor: D = F32, A = B = F16, both K-major, N = 128, M = 128.
constexpr uint32_t kIdescW = (1u << 4) | (uint32_t(W_BT >> 3) << 17) | (uint32_t(W_BN >> 4) << 24);
static_assert(W_D_COL + 2 * W_BT <= W_TMEM_COLS, "tensor memory budget");
static_assert(W_X_BYTES % 1024 == 0 && W_STAGE_BYTES % 1024 == 0, "1024-byte aligned tiles");

__device__ __forceinline__ float bf16_round(float v) { return bf16_bits_to_f32(f32_to_bf16_bits(v)); }

// 16 int8 (one 16-byte chunk) -> 8 words of fp16 pairs.
__device__ __forceinline__ void widen16(const uint4& x, uint32_t* h) {
  s8x4_to_f16x4(x.x, h[0], h[1]);
  s8x4_to_f16x4(x.y, h[2], h[3]);
  s8x4_to_f16x4(x.z, h[4], h[5]);
  s8x4_to_f16x4(x.w, h[6], h[7]);
}

struct WTile {
  int e, tb, nb, cnt;
  int64_t row0;  // first routed row of the tile's tokens
};

// Work unit t -> (expert, 128-token block of the expert, pair of 128-row weight blocks); CTA `rank` of the
// cluster takes weight block 2p + rank (past the expert's rows when NB is odd: computed, not stored).
// Rasterised in groups of up to W_GROUP_N weight blocks, the token block varying slower, so the clusters
// in flight share activation blocks and a group's weight blocks stay in L2 while the token blocks sweep
// past them.
__device__ __forceinline__ WTile wt_decode(int t, int E, int NB, const int* s_unit_prefix, const int* s_row_off,
                                           int rank) {
  WTile ti;
  ti.e = expert_of(t, E, s_unit_prefix);
  const int local = t - s_unit_prefix[ti.e];
  ti.cnt = s_row_off[ti.e + 1] - s_row_off[ti.e];
  const int TB = (ti.cnt + W_BT - 1) / W_BT;
  const int NP = (NB + 1) / 2;
  constexpr int GP = W_GROUP_N / 2;
  const int g = local / (TB * GP);
  const int rem = local - g * TB * GP;
  const int gp = min(GP, NP - g * GP);
  ti.tb = rem / gp;
  ti.nb = 2 * (g * GP + rem % gp) + rank;
  ti.row0 = static_cast<int64_t>(s_row_off[ti.e]) + static_cast<int64_t>(ti.tb) * W_BT;
  return ti;
}

template <int MODE>
__global__ void __cluster_dims__(W_CLUSTER, 1, 1) __launch_bounds__(W_THREADS, 1)
tcw_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[W_STAGES];   // both tiles of the stage landed
  __shared__ __align__(8) uint64_t bar_conv[W_STAGES];   // the stage's weights are in tensor memory
  __shared__ __align__(8) uint64_t bar_empty[W_STAGES];  // the MMAs reading the stage are done
  __shared__ __align__(8) uint64_t bar_accf[2];
  __shared__ __align__(8) uint64_t bar_acce[2];
  __shared__ __align__(8) uint64_t bar_up[4];      // SwiGLU, per (warp pair, token half): up values written
  __shared__ __align__(8) uint64_t bar_upfree[4];  // ... and read by the gate warp
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;
  __shared__ int s_bad;
  __shared__ int s_unit_prefix[kMaxE + 1];
  __shared__ int s_row_off[kMaxE + 1];
  __shared__ int s_warp[W_THREADS / 32];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = static_cast<int>(a.E);
  const int64_t N = a.N;
  const int64_t K = a.K;
  const int NB = static_cast<int>((N + W_BN - 1) / W_BN);
  const int nkb = static_cast<int>((K + W_BK - 1) / W_BK);
  const int nchunk = (nkb + W_KB_PER_CHUNK - 1) / W_KB_PER_CHUNK;

  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t stage_base = smem_u32(stages);
  uint16_t* upbuf = reinterpret_cast<uint16_t*>(stages + W_STAGES * W_STAGE_BYTES);
  uint32_t rank, cluster_id, nclusters;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(cluster_id));
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(nclusters));
  const int c0 = static_cast<int>(cluster_id), cstep = static_cast<int>(nclusters);

  if (tid == 0) {
    s_abort = 0;
    s_bad = 0;
    const PackedHeader* h = static_cast<const PackedHeader*>(a.packed);
    if (h->magic != kPackMagic || h->version != kPackVersion || h->E != a.E || h->N != a.N || h->K != a.K ||
        ((h->flags ^ a.pack_flags) & W8A8_PACK_GATE_UP) != 0u)
      s_bad = W8A8_ERR_PACKED;
    for (int s = 0; s < W_STAGES; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_conv[s]), W_CONV_WARPS);
      mbar_init(smem_u32(&bar_empty[s]), 1);  // this CTA's MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bar_accf[b]), 1);
      mbar_init(smem_u32(&bar_acce[b]), W_EPI_WARPS);
    }
    for (int p = 0; p < 4; ++p) {
      mbar_init(smem_u32(&bar_up[p]), 1);
      mbar_init(smem_u32(&bar_upfree[p]), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem_base)),
                 "r"(W_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // ---- per-expert rows and work units (128 tokens x 128 weight rows)
  int units_total;
  const int rows_total = scan_groups<W_THREADS, kMaxE>(
      a, E, [NB](int c) { return ((c + W_BT - 1) / W_BT) * ((NB + 1) / 2); }, s_row_off, s_unit_prefix, s_warp, &s_bad,
      &units_total);
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  int bad = s_bad;
  if (rows_total != a.R) bad |= W8A8_ERR_GROUP_LIST << 8;
  if (bad && tid == 0 && blockIdx.x == 0) set_status(a.status, (bad & 0xff) ? (bad & 0xff) : (bad >> 8), 0u);
  const int units = bad ? 0 : units_total;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = c0; t < units && !s_abort; t += cstep) {
        const WTile ti = wt_decode(t, E, NB, s_unit_prefix, s_row_off, static_cast<int>(rank));
        const int yx = static_cast<int>(ti.row0);
        const int yw = static_cast<int>(static_cast<int64_t>(ti.e) * N + static_cast<int64_t>(ti.nb) * W_BN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(smem_u32(&bar_empty[stage]), phase ^ 1u, &s_abort, a.status, 1u)) break;
          const uint32_t full = smem_u32(&bar_full[stage]);
          mbar_expect_tx(full, W_STAGE_BYTES);
          const uint32_t sa = stage_base + stage * W_STAGE_BYTES;
          // the tile's token rows (two 64-K sub-tiles) and its weight rows
          tma_load_2d(sa, &tmX, kb * W_BK, yx, full);
          tma_load_2d(sa + W_X_SUB, &tmX, kb * W_BK + 64, yx, full);
          tma_load_2d(sa + W_X_BYTES, &tmW, kb * W_BK, yw, full);
          if (++stage == W_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: every stage's last fill has been consumed, so no copy into this CTA is still in flight
      // when it leaves.
      for (int i = 0; i < W_STAGES && !s_abort; ++i) {
        if (!mbar_wait(smem_u32(&bar_empty[stage]), phase ^ 1u, &s_abort, a.status, 5u)) break;
        if (++stage == W_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_count = 0;
      for (int t = c0; t < units && !s_abort; t += cstep) {
        for (int c = 0; c < nchunk && !s_abort; ++c) {
          const uint32_t b = acc_count & 1u;
          const uint32_t use = acc_count >> 1;
          if (!mbar_wait(smem_u32(&bar_acce[b]), (use & 1u) ^ 1u, &s_abort, a.status, 2u)) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + W_D_COL + b * W_BT;
          const int kb_end = min(nkb, (c + 1) * W_KB_PER_CHUNK);
          bool ok = true;
          for (int kb = c * W_KB_PER_CHUNK; kb < kb_end; ++kb) {
            if (!mbar_wait(smem_u32(&bar_conv[stage]), phase, &s_abort, a.status, 3u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sx = stage_base + stage * W_STAGE_BYTES;
#pragma unroll
            for (int k = 0; k < W_BK / 16; ++k)
              tc_mma_tmem_a(d_tmem, tmem_base + stage * W_A_COLS + 8u * k,
                            smem_desc_sw128(sx + (k >> 2) * W_X_SUB) + 2u * (k & 3), kIdescW,
                            (kb > c * W_KB_PER_CHUNK || k > 0) ? 1u : 0u);
            tc_commit(smem_u32(&bar_empty[stage]));  // frees the stage
            if (++stage == W_STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          tc_commit(smem_u32(&bar_accf[b]));
          ++acc_count;
          if (!ok) break;
        }
      }
    }
  } else if (warp < W_EPI0) {
    // ------------------------------------------------------------- converters
    const int q = warp & 3;
    const int row = 32 * q + lane;  // weight row of the tile == TMEM lane
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = c0; t < units && ok; t += cstep) {
      for (int kb = 0; kb < nkb; ++kb) {
        // every lane observes the completed load itself
        const int got = mbar_wait(smem_u32(&bar_full[stage]), phase, &s_abort, a.status, 6u) ? 1 : 0;
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        // weight row `row`: 128 bytes, 16-byte chunk c stored at chunk c ^ (row & 7) (128-byte swizzle)
        const uint8_t* wrow = stages + stage * W_STAGE_BYTES + W_X_BYTES + row * W_BK;
        uint32_t v[2][32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            widen16(*reinterpret_cast<const uint4*>(wrow + (((4 * half + c) ^ (row & 7)) << 4)), &v[half][8 * c]);
          tmem_st32(lane_addr + stage * W_A_COLS + 32 * half, v[half]);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar_conv[stage]));
        if (++stage == W_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int h = (warp - W_EPI0) >> 2;  // token half of the tile: columns [64h, 64h + 64)
    const int n_loc = 32 * q + lane;     // weight row of the tile
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    uint32_t acc_count = 0, ntile = 0;
    for (int t = c0; t < units && !s_abort; t += cstep) {
      const WTile ti = wt_decode(t, E, NB, s_unit_prefix, s_row_off, static_cast<int>(rank));
      int sums[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) sums[i] = 0;
      bool ok = true;
      for (int c = 0; c < nchunk; ++c) {
        const uint32_t b = acc_count & 1u;
        const uint32_t use = acc_count >> 1;
        int got = 0;
        if (lane == 0) got = mbar_wait(smem_u32(&bar_accf[b]), use & 1u, &s_abort, a.status, 4u) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t col0 = W_D_COL + b * W_BT + 64 * h;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          uint32_t v[32];
          tmem_ld32(lane_addr + col0 + 32 * j, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) sums[32 * j + i] += __float2int_rn(__uint_as_float(v[i]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar_acce[b]));
        ++acc_count;
      }
      if (!ok) break;

      const int64_t rowh = ti.row0 + 64 * h;                 // routed row of token 0 of this half
      const int tvalid = min(64, ti.cnt - ti.tb * W_BT - 64 * h);  // tokens of the half that have rows
      const int64_t n = static_cast<int64_t>(ti.nb) * W_BN + n_loc;  // packed weight row in the expert
      if constexpr (MODE == EPI_ACC) {
        if (n < N) {
          int32_t* dst = static_cast<int32_t*>(a.out) + rowh * N + n;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i < tvalid) dst[i * N] = sums[i];
        }
      } else if constexpr (MODE == EPI_BF16) {
        if (n < N) {
          const float sw = a.w_scale[static_cast<int64_t>(ti.e) * N + n];
          const float bias = a.bias ? bf16_bits_to_f32(a.bias[n]) : 0.0f;
          uint16_t* dst = static_cast<uint16_t*>(a.out) + rowh * N + n;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            if (i < tvalid) {
              float f = dequant(sums[i], a.x_scale[rowh + i], sw);
              if (a.bias) f = __fadd_rn(f, bias);
              dst[i * N] = f32_to_bf16_bits(f);
            }
          }
        }
      } else {  // EPI_SWIGLU: tile rows [0,64) gate channels, [64,128) up channels of j = nb*64 + [0,64)
        const int p = q & 1;
        const int64_t I = N / 2;
        const int64_t j = static_cast<int64_t>(ti.nb) * kGateUpBlock + 32 * p + lane;
        const float* sw = a.w_scale + static_cast<int64_t>(ti.e) * N;
        uint16_t* ub = upbuf + (p * 2 + h) * 64 * 32 + lane;
        const uint32_t bu = smem_u32(&bar_up[p * 2 + h]);
        const uint32_t bf = smem_u32(&bar_upfree[p * 2 + h]);
        const uint32_t par = ntile & 1u;
        int got = 0;
        if (q >= 2) {  // up warp: BF16 up values into shared memory for the gate warp
          if (lane == 0) got = mbar_wait(bf, par ^ 1u, &s_abort, a.status, 7u) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, got, 0)) break;
          const float swu = j < I ? sw[I + j] : 0.0f;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            float u = 0.0f;
            if (i < tvalid && j < I) u = dequant(sums[i], a.x_scale[rowh + i], swu);
            ub[i * 32] = f32_to_bf16_bits(u);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bu);
        } else {  // gate warp: h = SwiGLU(bf16 gate, bf16 up)
          if (lane == 0) got = mbar_wait(bu, par, &s_abort, a.status, 8u) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, got, 0)) break;
          if (j < I) {
            const float swg = sw[j];
            uint16_t* dst = static_cast<uint16_t*>(a.out) + rowh * I + j;
#pragma unroll
            for (int i = 0; i < 64; ++i) {
              if (i < tvalid) {
                const float g = bf16_round(dequant(sums[i], a.x_scale[rowh + i], swg));
                dst[i * I] = swiglu_bf16(g, bf16_bits_to_f32(ub[i * 32]));
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bf);
        }
        ++ntile;
      }
    }
  }

  // ---- teardown: on abort, give in-flight copies and MMAs time to land first.  Lanes that skipped the
  // single-lane role loops reconverge before the block-wide barrier, so TMEM is not freed while the
  // epilogue warps still read it.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (s_abort) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 20000000ull) {
    }
  }
  cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(W_TMEM_COLS)
                 : "memory");
  }
}

template <int MODE>
cudaError_t launch_tcw_mode(const CUtensorMap& mx, const CUtensorMap& mw, const GemmArgs& a, int grid, size_t smem,
                            cudaStream_t stream) {
  auto k = tcw_gemm_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k<<<grid, W_THREADS, smem, stream>>>(mx, mw, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tcw_gemm(const GemmArgs& a, const void* a_f16, int num_sms, cudaStream_t stream) {
  if (a.R == 0) return cudaSuccess;
  // fp16 activations [R, K] and the int8 weight payload [E*N, K]; rows past the ends read as zero
  CUtensorMap mx, mw;
  const uint8_t* w_i8 = static_cast<const uint8_t*>(a.packed) + pack_layout(a.E, a.N, a.K, 0).i8_offset;
  if (!encode_map_2d(&mx, a_f16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.R, a.K, 64, W_BT,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_map_2d(&mw, w_i8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.E * a.N, a.K, W_BK, W_BN,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int64_t nb = (a.N + W_BN - 1) / W_BN;
  const int64_t units = ((a.R + W_BT - 1) / W_BT + (a.group_list != nullptr ? a.E : 0)) * ((nb + 1) / 2);
  const int64_t clusters = std::max<int64_t>(1, std::min<int64_t>(units, num_sms / W_CLUSTER));
  const int grid = static_cast<int>(clusters * W_CLUSTER);
  const size_t smem = static_cast<size_t>(W_STAGES) * W_STAGE_BYTES + W_UP_BYTES + 1024;
  switch (a.mode) {
    case EPI_ACC: return launch_tcw_mode<EPI_ACC>(mx, mw, a, grid, smem, stream);
    case EPI_SWIGLU: return launch_tcw_mode<EPI_SWIGLU>(mx, mw, a, grid, smem, stream);
    default: return launch_tcw_mode<EPI_BF16>(mx, mw, a, grid, smem, stream);
  }
}

}  // namespace w8a8
