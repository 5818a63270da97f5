// gemm_tc.cu -- exact INT8 contraction on the 5th-generation tensor cores
// (tcgen05) for large-M shapes: the dense prefill linear and the grouped
// expert GEMMs of MoE prefill.
//
// Page "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子": §二
// npu_quant_matmul (INT8 x INT8 -> INT32, then * x_scale * w_scale (+bias) ->
// BF16), §三 npu_grouped_matmul over group_list and the W13 -> SwiGLU step,
// §四 (prefill, large M, gets its own tiling).
//
// Engine.  sm_103a has no integer tcgen05.mma kind, so the int8 operands are
// fed as integer-valued FP16 (exact) to tcgen05.mma.kind::f16 with FP32
// accumulators in tensor memory.  Products |a*b| <= 2^14 are exact and a
// fresh accumulator is started every 1024 K (|partial| <= 2^24, all partial
// sums exactly representable), so every accumulator holds an exact integer.
// Two TMEM accumulators of 128 lanes x 256 columns alternate between
// consecutive 1024-deep chunks; the epilogue warps drain a finished chunk into
// int32 registers while the MMA fills the other one.
//
// Data movement.  Both operands are K-major FP16 tiles brought in by TMA
// (cp.async.bulk.tensor, 128-byte swizzle).  A tile is 256 rows of one expert
// x 256 weight rows (dense: one expert of R rows), computed on a CTA pair
// (tcgen05 cta_group::2): the even CTA holds activation rows [0,128) and
// weight rows [0,128) of every 64-deep stage, the odd CTA rows [128,256) and
// weight rows [128,256), 32 KB per CTA and stage, six stages.  One elected
// lane of the even CTA's MMA warp issues tcgen05.mma M=256 N=256 K=16 over
// both CTAs' shared memory four times per stage; each CTA's tensor memory
// receives its 128 rows of the accumulator.  Both CTAs' copies complete on
// the even CTA's full barrier; the MMA commit frees the stage in both CTAs;
// both CTAs' epilogues release an accumulator on the even CTA's barrier.  The
// second 128 rows of an expert's last tile may lie past its rows: computed,
// not stored.
//
// Warp roles (320 threads, one CTA per SM, persistent over output tiles):
//   warp 0     TMA producer
//   warp 1     TMEM owner and (even CTA) MMA issuer
//   warps 2-9  epilogue: warp w reads TMEM lanes 32*(w%4).. and one half
//              (128 columns) of the tile; each thread owns one output row.
// Every mbarrier wait is bounded (%globaltimer, 2 s): on expiry the CTA sets
// W8A8_ERR_DEVICE_TIMEOUT in the status word, lets in-flight copies land,
// frees its TMEM and returns.
#include "kernels.cuh"
#include "tc_common.cuh"

namespace w8a8 {

namespace {

constexpr int TC_BN = 256;
constexpr int TC_BK = 64;  // fp16 elements = 128 bytes = one swizzle row
constexpr int TC_GROUP_N = 16;  // n-blocks per rasterisation group
constexpr int TC_KB_PER_CHUNK = kChunkK / TC_BK;  // 16
constexpr int TC_THREADS = 320;
constexpr int TC_EPI_WARPS = 8;
constexpr uint32_t TC_TMEM_COLS = 512;  // two 256-column fp32 accumulators
constexpr int TC_CLUSTER = 2;
constexpr uint16_t TC_PAIR_MASK = 0x3;
constexpr int kMaxE = 1024;

using namespace tc;

// Per-channel factors of a 128-column output segment, staged in shared memory by each epilogue warp for
// the BF16 epilogue: weight scale, integer bias (static W8A8) and float bias (0 where absent).
struct __align__(16) SegFactors {
  float w[128];
  int32_t qb[128];
  float b[128];
  int narrow;  // every |qb| <= 2^31 - 1 - 16384*K: acc + qb cannot leave int32 (|acc| <= 16384*K)
  int pad[3];  // keeps every element of an array of these 16-byte aligned (16-byte shared loads)
};
static_assert(sizeof(SegFactors) % 16 == 0, "SegFactors must keep 16-byte alignment in arrays");

// Warp-cooperative: the factors of columns [n_base, n_base + 128) of expert e into f (lane l takes
// columns l, l+32, l+64, l+96).  The caller's __syncwarp() makes them visible to the warp.
__device__ __forceinline__ void stage_factors(const GemmArgs& a, int e, int64_t n_base, int lane, SegFactors& f) {
  const int64_t N = a.N;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = lane + 32 * i;
    const int64_t n = n_base + c;
    const bool in = n < N;
    f.w[c] = in ? a.w_scale[static_cast<int64_t>(e) * N + n] : 0.0f;
    f.qb[c] = (in && a.qbias != nullptr) ? a.qbias[n] : 0;
    f.b[c] = (in && a.bias != nullptr) ? bf16_bits_to_f32(a.bias[n]) : 0.0f;
  }
  if (a.qbias != nullptr) {
    const int64_t room = 2147483647LL - 16384LL * a.K;
    bool ok = true;
#pragma unroll
    for (int i = 0; i < 4; ++i) ok = ok && (f.qb[lane + 32 * i] <= room && -static_cast<int64_t>(f.qb[lane + 32 * i]) <= room);
    const bool all = __all_sync(0xffffffffu, ok);
    if (lane == 0) f.narrow = all ? 1 : 0;
  }
}

// The same for the SwiGLU epilogue: columns [n_base, n_base + 128) of W13 hold gate channels j0 + [0,64)
// and up channels j0 + [0,64), j0 = (n_base / 128) * 64; f.w[c] takes the gate scale of channel j0 + c
// (c < 64) or the up scale of channel j0 + c - 64, in the original channel order of w_scale.
__device__ __forceinline__ void stage_factors_swiglu(const GemmArgs& a, int e, int64_t n_base, int lane,
                                                     SegFactors& f) {
  const int64_t N = a.N, I = N / 2;
  const int64_t j0 = (n_base / 128) * kGateUpBlock;
  const float* sw = a.w_scale + static_cast<int64_t>(e) * N;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = lane + 32 * i;
    f.w[c] = c < kGateUpBlock ? sw[j0 + c] : sw[I + j0 + c - kGateUpBlock];
  }
}

// Stores one output row segment of a finished tile: global row gr, 128
// columns from n_base (expert e's weight rows), from the exact int32 sums.
// fac: the segment's factors staged in shared memory (BF16 epilogue), or nullptr to read them from
// global memory.  A missing x_scale reads as 1 (static W8A8, with qbias).
template <int MODE>
__device__ __forceinline__ void store_row(const GemmArgs& a, int e, int64_t gr, int64_t n_base, const int (&sums)[128],
                                          const SegFactors* fac = nullptr) {
  const int64_t N = a.N;
  if constexpr (MODE == EPI_ACC) {
    int32_t* dst = static_cast<int32_t*>(a.out) + gr * N + n_base;
    const bool vec = ((reinterpret_cast<uintptr_t>(a.out) & 15u) == 0u) && ((N & 3) == 0) && (n_base + 128 <= N);
#pragma unroll
    for (int c4 = 0; c4 < 32; ++c4) {
      if (vec) {
        reinterpret_cast<int4*>(dst)[c4] =
            make_int4(sums[4 * c4], sums[4 * c4 + 1], sums[4 * c4 + 2], sums[4 * c4 + 3]);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (n_base + 4 * c4 + k < N) dst[4 * c4 + k] = sums[4 * c4 + k];
      }
    }
  } else if constexpr (MODE == EPI_BF16) {
    const float sx = a.x_scale != nullptr ? a.x_scale[gr] : 1.0f;
    const float* sw = a.w_scale + static_cast<int64_t>(e) * N;
    uint16_t* dst = static_cast<uint16_t*>(a.out) + gr * N + n_base;
    const bool vec = ((reinterpret_cast<uintptr_t>(a.out) & 15u) == 0u) && ((N & 7) == 0) && (n_base + 128 <= N);
#pragma unroll
    for (int c8 = 0; c8 < 16; ++c8) {
      uint16_t v[8];
      if (fac != nullptr) {  // staged factors: broadcast 16-byte shared loads
        const float4 w0 = reinterpret_cast<const float4*>(fac->w)[2 * c8];
        const float4 w1 = reinterpret_cast<const float4*>(fac->w)[2 * c8 + 1];
        const float w8[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        int32_t q8[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        float b8[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        if (a.qbias != nullptr) {
          const int4 q0 = reinterpret_cast<const int4*>(fac->qb)[2 * c8];
          const int4 q1 = reinterpret_cast<const int4*>(fac->qb)[2 * c8 + 1];
          q8[0] = q0.x; q8[1] = q0.y; q8[2] = q0.z; q8[3] = q0.w;
          q8[4] = q1.x; q8[5] = q1.y; q8[6] = q1.z; q8[7] = q1.w;
        }
        if (a.bias != nullptr) {
          const float4 b0 = reinterpret_cast<const float4*>(fac->b)[2 * c8];
          const float4 b1 = reinterpret_cast<const float4*>(fac->b)[2 * c8 + 1];
          b8[0] = b0.x; b8[1] = b0.y; b8[2] = b0.z; b8[3] = b0.w;
          b8[4] = b1.x; b8[5] = b1.y; b8[6] = b1.z; b8[7] = b1.w;
        }
        const bool narrow = a.qbias != nullptr && fac->narrow;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float f;
          if (narrow) f = __fmul_rn(__fmul_rn(__int2float_rn(sums[8 * c8 + k] + q8[k]), sx), w8[k]);
          else if (a.qbias != nullptr) f = dequant_q(sums[8 * c8 + k], q8[k], sx, w8[k]);
          else f = dequant(sums[8 * c8 + k], sx, w8[k]);
          if (a.bias) f = __fadd_rn(f, b8[k]);
          v[k] = f32_to_bf16_bits(f);  // columns past N (factors 0) are not stored
        }
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int64_t n = n_base + 8 * c8 + k;
          float f = 0.0f;
          if (n < N) {
            f = a.qbias != nullptr ? dequant_q(sums[8 * c8 + k], a.qbias[n], sx, sw[n]) : dequant(sums[8 * c8 + k], sx, sw[n]);
            if (a.bias) f = __fadd_rn(f, bf16_bits_to_f32(a.bias[n]));
          }
          v[k] = f32_to_bf16_bits(f);
        }
      }
      if (vec) {
        reinterpret_cast<uint4*>(dst)[c8] =
            make_uint4(v[0] | (uint32_t(v[1]) << 16), v[2] | (uint32_t(v[3]) << 16),
                       v[4] | (uint32_t(v[5]) << 16), v[6] | (uint32_t(v[7]) << 16));
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (n_base + 8 * c8 + k < N) dst[8 * c8 + k] = v[k];
      }
    }
  } else {  // EPI_SWIGLU: columns [0,64) gate j, [64,128) up j, j = j0 + [0,64); factors staged in fac
    const float sx = a.x_scale[gr];
    const int64_t I = N / 2;
    const int64_t j0 = (n_base / 128) * kGateUpBlock;
    uint16_t* dst = static_cast<uint16_t*>(a.out) + gr * I + j0;
    const bool vec = ((reinterpret_cast<uintptr_t>(a.out) & 15u) == 0u) && ((I & 7) == 0);
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      const float4 g0 = reinterpret_cast<const float4*>(fac->w)[2 * c8];
      const float4 g1 = reinterpret_cast<const float4*>(fac->w)[2 * c8 + 1];
      const float4 u0 = reinterpret_cast<const float4*>(fac->w + kGateUpBlock)[2 * c8];
      const float4 u1 = reinterpret_cast<const float4*>(fac->w + kGateUpBlock)[2 * c8 + 1];
      const float wg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      const float wu[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      uint32_t h[4];
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        const int jj = 8 * c8 + k;
        // gate and up of two channels rounded to bf16 (two per instruction), then h in binary32, rounded
        // to bf16 two at a time
        const uint32_t gb = f32x2_to_bf16x2_bits(dequant(sums[jj], sx, wg[k]), dequant(sums[jj + 1], sx, wg[k + 1]));
        const uint32_t ub = f32x2_to_bf16x2_bits(dequant(sums[kGateUpBlock + jj], sx, wu[k]),
                                                 dequant(sums[kGateUpBlock + jj + 1], sx, wu[k + 1]));
        const float ha = swiglu_f32(__uint_as_float(gb << 16), __uint_as_float(ub << 16));
        const float hb = swiglu_f32(__uint_as_float(gb & 0xffff0000u), __uint_as_float(ub & 0xffff0000u));
        h[k / 2] = f32x2_to_bf16x2_bits(ha, hb);
      }
      if (vec) {
        reinterpret_cast<uint4*>(dst)[c8] = make_uint4(h[0], h[1], h[2], h[3]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[8 * c8 + k] = static_cast<uint16_t>(h[k / 2] >> (16 * (k & 1)));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// The contraction on CTA pairs (layout in the file comment).
constexpr int P_BM = 256;       // rows per pair tile
constexpr int P_HALF = 128;     // rows of A and of B held by each CTA
constexpr int P_STAGES = 6;
constexpr uint32_t P_HALF_BYTES = P_HALF * TC_BK * 2;  // 16 KB
constexpr uint32_t P_STAGE_BYTES = 2 * P_HALF_BYTES;   // this CTA's A rows and B rows
constexpr uint32_t kIdescPair = (1u << 4) | (uint32_t(TC_BN >> 3) << 17) | (uint32_t(P_BM >> 4) << 24);

template <int MODE>
__global__ void __cluster_dims__(TC_CLUSTER, 1, 1) __launch_bounds__(TC_THREADS, 1)
tc_pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[P_STAGES];   // even CTA: both CTAs' copies of the stage landed
  __shared__ __align__(8) uint64_t bar_empty[P_STAGES];  // the pair MMAs reading the stage are done
  __shared__ __align__(8) uint64_t bar_accf[2];
  __shared__ __align__(8) uint64_t bar_acce[2];          // even CTA: both CTAs drained the accumulator
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;
  __shared__ int s_bad;
  __shared__ int s_unit_prefix[kMaxE + 1];
  __shared__ int s_row_off[kMaxE + 1];
  __shared__ int s_warp[TC_THREADS / 32];
  __shared__ __align__(16) SegFactors s_fac[TC_EPI_WARPS];  // one per epilogue warp

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = static_cast<int>(a.E);
  const int64_t N = a.N;
  const int64_t K = a.K;
  const int NB = static_cast<int>((N + TC_BN - 1) / TC_BN);
  const int nkb = static_cast<int>((K + TC_BK - 1) / TC_BK);
  const int nchunk = (nkb + TC_KB_PER_CHUNK - 1) / TC_KB_PER_CHUNK;

  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t stage_base = smem_u32(stages);
  uint32_t rank, cluster_id, nclusters;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(cluster_id));
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(nclusters));

  if (tid == 0) {
    s_abort = 0;
    s_bad = 0;
    const PackedHeader* h = static_cast<const PackedHeader*>(a.packed);
    if (h->magic != kPackMagic || h->version != kPackVersion || h->E != a.E || h->N != a.N || h->K != a.K ||
        ((h->flags ^ a.pack_flags) & W8A8_PACK_GATE_UP) != 0u || (h->flags & W8A8_PACK_F16) == 0u)
      s_bad = W8A8_ERR_PACKED;
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bar_accf[b]), 1);
      mbar_init(smem_u32(&bar_acce[b]), TC_CLUSTER * TC_EPI_WARPS);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem_base)),
                 "r"(TC_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  // ---- per-expert rows and work units (256-row tiles)
  int units_total;
  const int rows_total = scan_groups<TC_THREADS, kMaxE>(
      a, E, [NB](int c) { return ((c + P_BM - 1) / P_BM) * NB; }, s_row_off, s_unit_prefix, s_warp, &s_bad,
      &units_total);
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers and tensor memory exist before either touches the other's
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  int bad = s_bad;
  if (rows_total != a.R) bad |= W8A8_ERR_GROUP_LIST << 8;
  if (bad && tid == 0 && blockIdx.x == 0) set_status(a.status, (bad & 0xff) ? (bad & 0xff) : (bad >> 8), 0u);
  const int units = bad ? 0 : units_total;

  // Unit t -> expert e, 256-row block mb of the expert, n-block nb; rasterised in groups of TC_GROUP_N
  // n-blocks (n-block fastest, then the m-block), so the pairs in flight share activation blocks and the
  // group's weight blocks stay resident in L2 while the expert's m-blocks sweep past them.
  auto tile_of = [&](int t, int& e, int& mb, int& nb) {
    e = expert_of(t, E, s_unit_prefix);
    const int local = t - s_unit_prefix[e];
    const int MB = (s_row_off[e + 1] - s_row_off[e] + P_BM - 1) / P_BM;
    const int g = local / (MB * TC_GROUP_N);
    const int rem = local - g * MB * TC_GROUP_N;
    const int gn = min(TC_GROUP_N, NB - g * TC_GROUP_N);
    mb = rem / gn;
    nb = g * TC_GROUP_N + rem % gn;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = static_cast<int>(cluster_id); t < units && !s_abort; t += static_cast<int>(nclusters)) {
        int e, mb, nb;
        tile_of(t, e, mb, nb);
        const int ya = s_row_off[e] + mb * P_BM + static_cast<int>(rank) * P_HALF;
        const int yb = static_cast<int>(static_cast<int64_t>(e) * N + static_cast<int64_t>(nb) * TC_BN) +
                       static_cast<int>(rank) * P_HALF;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(smem_u32(&bar_empty[stage]), phase ^ 1u, &s_abort, a.status, 1u)) break;
          const uint32_t full = smem_u32(&bar_full[stage]);
          if (rank == 0) mbar_expect_tx(full, TC_CLUSTER * P_STAGE_BYTES);
          const uint32_t full_even = smem_cluster_addr(full, 0);
          const uint32_t sa = stage_base + stage * P_STAGE_BYTES;
          tma_load_2d_pair(sa, &tmA, kb * TC_BK, ya, full_even);
          tma_load_2d_pair(sa + P_HALF_BYTES, &tmB, kb * TC_BK, yb, full_even);
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: the last fill of every stage has been consumed, so no copy into this CTA and no MMA
      // arrival on its barriers is still in flight when the cluster leaves.
      for (int i = 0; i < P_STAGES && !s_abort; ++i) {
        if (!mbar_wait(smem_u32(&bar_empty[stage]), phase ^ 1u, &s_abort, a.status, 5u)) break;
        if (++stage == P_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer (even CTA, whole warp)
    if (rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_count = 0;
      for (int t = static_cast<int>(cluster_id); t < units && !s_abort; t += static_cast<int>(nclusters)) {
        for (int c = 0; c < nchunk && !s_abort; ++c) {
          const uint32_t b = acc_count & 1u;
          const uint32_t use = acc_count >> 1;
          if (!warp_wait(smem_u32(&bar_acce[b]), (use & 1u) ^ 1u, &s_abort, a.status, 2u)) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + b * TC_BN;
          const int kb_end = min(nkb, (c + 1) * TC_KB_PER_CHUNK);
          bool ok = true;
          for (int kb = c * TC_KB_PER_CHUNK; kb < kb_end; ++kb) {
            if (!warp_wait(smem_u32(&bar_full[stage]), phase, &s_abort, a.status, 3u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = stage_base + stage * P_STAGE_BYTES;
            const uint64_t adesc = smem_desc_sw128(sa);
            const uint64_t bdesc = smem_desc_sw128(sa + P_HALF_BYTES);
#pragma unroll
            for (int k = 0; k < TC_BK / 16; ++k)
              tc_mma_pair(d_tmem, adesc + 2u * k, bdesc + 2u * k, kIdescPair,
                          (kb > c * TC_KB_PER_CHUNK || k > 0) ? 1u : 0u);
            tc_commit_pair_mc(smem_u32(&bar_empty[stage]), TC_PAIR_MASK);  // frees the stage in both CTAs
            if (++stage == P_STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          tc_commit_pair_mc(smem_u32(&bar_accf[b]), TC_PAIR_MASK);
          ++acc_count;
          if (!ok) break;
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r_loc = 32 * q + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    uint32_t acc_count = 0;
    for (int t = static_cast<int>(cluster_id); t < units && !s_abort; t += static_cast<int>(nclusters)) {
      int e, mb, nb;
      tile_of(t, e, mb, nb);
      SegFactors& fac = s_fac[warp - 2];
      __syncwarp();  // every lane is done with the previous tile's factors
      if constexpr (MODE == EPI_BF16) {
        // the segment's factors, loaded while the tile's MMAs run (read by this warp only)
        stage_factors(a, e, static_cast<int64_t>(nb) * TC_BN + half * 128, lane, fac);
        __syncwarp();
      } else if constexpr (MODE == EPI_SWIGLU) {
        stage_factors_swiglu(a, e, static_cast<int64_t>(nb) * TC_BN + half * 128, lane, fac);
        __syncwarp();
      }
      int sums[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) sums[i] = 0;
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
        const uint32_t col0 = b * TC_BN + half * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t v[32];
          tmem_ld32(lane_addr + col0 + 32 * j, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) sums[32 * j + i] += __float2int_rn(__uint_as_float(v[i]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(smem_cluster_addr(smem_u32(&bar_acce[b]), 0));
        ++acc_count;
      }
      if (!ok) break;
      const int m0 = mb * P_BM + static_cast<int>(rank) * P_HALF;  // first row of this CTA inside the expert
      const int64_t n_base = static_cast<int64_t>(nb) * TC_BN + half * 128;
      if (m0 + r_loc < s_row_off[e + 1] - s_row_off[e] && n_base < N)
        store_row<MODE>(a, e, static_cast<int64_t>(s_row_off[e]) + m0 + r_loc, n_base, sums, &fac);
    }
  }

  // ---- teardown, then the pair leaves together.
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
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TC_TMEM_COLS)
                 : "memory");
  }
}

__global__ void __launch_bounds__(256) s8_to_f16_kernel(const int8_t* __restrict__ src, uint16_t* __restrict__ dst,
                                                       int64_t n16) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 v = reinterpret_cast<const uint4*>(src)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) s8x4_to_f16x4(w[k], h[2 * k], h[2 * k + 1]);
    uint4* d = reinterpret_cast<uint4*>(dst) + 2 * i;
    d[0] = make_uint4(h[0], h[1], h[2], h[3]);
    d[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// 2-D fp16 tensor [rows, K] (K contiguous), box = box_rows x 64, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int box_rows) {
  return encode_map_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rows, K, TC_BK, box_rows,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int MODE>
cudaError_t launch_tc_mode(const CUtensorMap& ma, const CUtensorMap& mb, const GemmArgs& a, int grid, size_t smem,
                           cudaStream_t stream) {
  void (*k)(CUtensorMap, CUtensorMap, GemmArgs) = tc_pair_gemm_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k<<<grid, TC_THREADS, smem, stream>>>(ma, mb, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_gemm(const GemmArgs& a, const void* a_f16, const void* b_f16, int num_sms, cudaStream_t stream) {
  if (a.R == 0) return cudaSuccess;
  CUtensorMap ma, mb;
  if (!make_map(&ma, a_f16, a.R, a.K, P_HALF)) return cudaErrorInvalidValue;
  if (!make_map(&mb, b_f16, a.E * a.N, a.K, P_HALF)) return cudaErrorInvalidValue;
  // work units: 256-row blocks of every expert (at most one partial block per expert) x n-blocks
  const int64_t units =
      ((a.R + P_BM - 1) / P_BM + (a.group_list != nullptr ? a.E : 0)) * ((a.N + TC_BN - 1) / TC_BN);
  const int64_t clusters = std::max<int64_t>(1, std::min<int64_t>(units, num_sms / TC_CLUSTER));
  const int grid = static_cast<int>(clusters * TC_CLUSTER);
  const size_t smem = static_cast<size_t>(P_STAGES) * P_STAGE_BYTES + 1024;
  switch (a.mode) {
    case EPI_ACC: return launch_tc_mode<EPI_ACC>(ma, mb, a, grid, smem, stream);
    case EPI_SWIGLU: return launch_tc_mode<EPI_SWIGLU>(ma, mb, a, grid, smem, stream);
    default: return launch_tc_mode<EPI_BF16>(ma, mb, a, grid, smem, stream);
  }
}

cudaError_t launch_s8_to_f16(const int8_t* src, uint16_t* dst, int64_t n, cudaStream_t stream, int num_sms) {
  if (n == 0) return cudaSuccess;
  const int64_t n16 = n / 16;
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((n16 + 255) / 256, static_cast<int64_t>(num_sms) * 8));
  s8_to_f16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(src, dst, n16);
  return cudaGetLastError();
}

}  // namespace w8a8
