// mx_tc.cu -- MXFP8 contraction on the block-scaled 5th-generation tensor
// cores: tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale on CTA pairs.
//
// Page "Qwen3.8-FP8 on Ascend 950: Why Weights Become MXFP8 at Load Time",
// section 5: at run time both operands are MXFP8 (E4M3 payload, one E8M0
// scale per 32 values along K; group sizes [1,1,32]) and the matmul is
// y[m,n] = bf16(sum_g Sa[m,g] Sw[n,g] sum_{k in g} a[m,k] w[n,k]).  The
// block-scaled MMA applies both powers of two inside the tensor core and
// accumulates in binary32 over the whole K.
//
// Tile.  As in the INT8 pair engine (gemm_tcp.cu): the weights are the MMA's
// M side, 256 rows per CTA pair (128 in each CTA), and a block of up to 192
// tokens is N -- the even CTA holds the block's first n/2 tokens, the odd CTA
// the rest -- with n the block's token count rounded up to 16.  A stage is
// 128 of K: the CTA's 128 x 128-byte weight tile and its 96 x 128-byte token
// tile (128-byte swizzle), 28 KB, by TMA into a five-stage ring; both CTAs'
// copies complete on the even CTA's barrier.  One MMA instruction covers 32 of
// K, so a stage is four MMAs, each with its own scale byte (the
// instruction's scale-data id selects byte kb of the 32-bit scale words).
//
// Scale factors in tensor memory.  The tensor core reads the scale of matrix
// row r (weight row, or token column of B) from lane r % 32 -- the value
// is replicated in all four lane quadrants -- and column r / 32 of the scale
// area, byte = the K-block; a probe on this GPU confirmed the layout
// numerically.  The row-major E8M0 scale matrices [rows, K/32] are brought
// by TMA in groups of four stages (16 bytes a row) into a two-slot
// shared-memory ring; per stage four scale warps per CTA (one per lane
// quadrant) read their rows' 32-bit words (the four K-blocks of the stage)
// and store them with tcgen05.st: 4 columns for the CTA's 128 weight rows and
// 6 for the block's 192 token columns (the token scales are the same in both
// CTAs), into a four-slot tensor-memory ring, and then arrive on the even
// CTA's barrier.
//
// Tensor memory (512 columns): two 192-column accumulators at 0 and 256
// (alternating per tile, so the epilogue drains one while the MMAs fill the
// other), scale slots of 16 columns at 192, 208, 224 and 240 (weight scales
// at +0, token scales at +8).
//
// Warp roles (448 threads, one CTA per SM, persistent over tiles):
//   warp 0       TMA producer (operand tiles, scale groups)
//   warp 1       TMEM owner; one elected lane of the even CTA's warp issues the MMAs
//   warps 2-5    scale warps
//   warps 6-13   epilogue: warp w reads TMEM lanes 32*(w%4).. (weight rows)
//                and one half (96 tokens) of the columns, rounds to BF16 and
//                writes through shared memory as 16-byte pieces of rows
// Every mbarrier wait is bounded (2 s): on expiry the CTA sets
// W8A8_ERR_DEVICE_TIMEOUT, lets in-flight copies land, frees TMEM and returns.
#include "kernels.cuh"
#include "tc_common.cuh"

namespace w8a8 {

namespace {

using namespace tc;

constexpr int X_WROWS = 256;  // weight rows per pair tile (MMA M)
constexpr int X_WHALF = 128;
constexpr int X_NT = 192;     // most tokens per tile (MMA N)
constexpr int X_NHALF = 96;
constexpr int X_BK = 128;     // K per stage (bytes = E4M3 values)
constexpr int X_STAGES = 5;
// Scale slots in tensor memory.  A slot is reused four stages later, after the commit that frees the shared-
// memory stage of its previous user; with fewer slots than ring stages that commit's barrier cannot have
// moved on to a later phase before the scale warps wait for it.
constexpr int X_SF_SLOTS = 4;
constexpr int X_SF_GROUP = 4;      // stages per scale group (16 scale bytes a row)
constexpr uint32_t X_W_BYTES = X_WHALF * X_BK;  // 16 KB
constexpr uint32_t X_X_BYTES = X_NHALF * X_BK;  // 12 KB
constexpr uint32_t X_STAGE_BYTES = X_W_BYTES + X_X_BYTES;
constexpr uint32_t X_SFW_BYTES = X_WHALF * 16;  // weight scales of a group (2 KB)
constexpr uint32_t X_SFX_BYTES = X_NT * 16;     // token scales of a group (3 KB)
constexpr uint32_t X_SF_BYTES = X_SFW_BYTES + X_SFX_BYTES;
constexpr uint32_t X_OUT_BYTES = 8 * X_NHALF * 32 * 2;  // epilogue staging, [96 tokens][32 channels] per warp
constexpr int X_THREADS = 448;
constexpr int X_SCALE_WARPS = 4;
constexpr int X_EPI0 = 6;
constexpr int X_EPI_WARPS = 8;
constexpr int X_CLUSTER = 2;
constexpr uint16_t X_PAIR_MASK = 0x3;
constexpr uint32_t X_TMEM_COLS = 512;
static_assert(X_STAGE_BYTES % 1024 == 0 && X_W_BYTES % 1024 == 0, "1024-byte tiles");
static_assert(X_NHALF % 8 == 0, "whole 8-row swizzle atoms per CTA");

__host__ __device__ constexpr uint32_t x_acc_col(uint32_t b) { return 256u * b; }
__host__ __device__ constexpr uint32_t x_sf_col(int s) { return 192u + 16u * static_cast<uint32_t>(s); }
static_assert(X_SF_SLOTS < X_STAGES && x_sf_col(X_SF_SLOTS - 1) + 16u <= x_acc_col(1) &&
                  x_acc_col(0) + 192u <= x_sf_col(0) && x_acc_col(1) + 192u <= 512u,
              "tensor memory budget");

// kind::mxf8f6f4 block-scaled instruction descriptor: A = B = E4M3 (format 0), both K-major, scale format
// UE8M0 (bit 23), M = 256, N = n, scale-data ids of A (bits 29-30) and B (bits 4-5) = kb.
__device__ __forceinline__ uint32_t idesc_mx(int n, uint32_t kb) {
  return (kb << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(X_WROWS >> 4) << 24) | (kb << 29);
}

// Issued by the elected lane of the (converged) MMA warp, as the issue helpers of tc_common.cuh.
__device__ __forceinline__ void tc_mma_pair_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %6, 0;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}\n"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void tmem_st2(uint32_t taddr, uint32_t a, uint32_t b) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1,%2};" ::"r"(taddr), "r"(a), "r"(b) : "memory");
}

// Rows [0, rows) of a warp's staging buffer [rows][32] bf16 to out[(row0 + r) * ld + c0 + c], c < min(32, ld - c0):
// 16-byte stores of 64-byte row pieces when they fit, else 2-byte stores.
__device__ __forceinline__ void x_store_rows(const uint16_t* stg, uint16_t* out, int64_t row0, int64_t ld,
                                             int64_t c0, int rows, int lane) {
  const int64_t ncols = ld - c0 < 32 ? ld - c0 : 32;
  if (ncols <= 0 || rows <= 0) return;
  if (ncols == 32 && (ld & 7) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0u) {
    const int c = (lane & 3) * 8;
#pragma unroll 4
    for (int r = lane >> 2; r < rows; r += 8)
      *reinterpret_cast<uint4*>(out + (row0 + r) * ld + c0 + c) = *reinterpret_cast<const uint4*>(stg + r * 32 + c);
  } else {
    for (int r = 0; r < rows; ++r)
      if (lane < ncols) out[(row0 + r) * ld + c0 + lane] = stg[r * 32 + lane];
  }
}

struct XArgs {
  int64_t M, N, K;
  uint16_t* y;
  DeviceStatus* status;
};

struct XTile {
  int tb, wb, n_eff, tvalid;
  int64_t row0;
};

__device__ __forceinline__ XTile x_decode(int t, int TB, int64_t M) {
  XTile ti;
  ti.wb = t / TB;
  ti.tb = t - ti.wb * TB;
  ti.tvalid = static_cast<int>(min(static_cast<int64_t>(X_NT), M - static_cast<int64_t>(ti.tb) * X_NT));
  ti.n_eff = (ti.tvalid + 15) & ~15;
  ti.row0 = static_cast<int64_t>(ti.tb) * X_NT;
  return ti;
}

__global__ void __cluster_dims__(X_CLUSTER, 1, 1) __launch_bounds__(X_THREADS, 1)
mx_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
             const __grid_constant__ CUtensorMap tmSX, const __grid_constant__ CUtensorMap tmSW, const XArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[X_STAGES];     // even CTA: both CTAs' operand tiles of the stage landed
  __shared__ __align__(8) uint64_t bar_empty[X_STAGES];    // the MMAs reading the stage (and its scale slot) are done
  __shared__ __align__(8) uint64_t bar_sffull[2];          // this CTA's scale group landed
  __shared__ __align__(8) uint64_t bar_sfempty[2];         // this CTA's scale warps read the group
  __shared__ __align__(8) uint64_t bar_sfready[X_SF_SLOTS];  // even CTA: both CTAs' scales of the stage are in TMEM
  __shared__ __align__(8) uint64_t bar_accf[2];
  __shared__ __align__(8) uint64_t bar_acce[2];            // even CTA: both CTAs drained the accumulator
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int64_t M = a.M, N = a.N, K = a.K;
  const int TB = static_cast<int>((M + X_NT - 1) / X_NT);
  const int WB = static_cast<int>((N + X_WROWS - 1) / X_WROWS);
  const int units = TB * WB;
  const int nkb = static_cast<int>((K + X_BK - 1) / X_BK);

  uint8_t* stages = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t stage_base = smem_u32(stages);
  uint8_t* sfbuf = stages + X_STAGES * X_STAGE_BYTES;     // [2][weight scales 128 x 16 B, token scales 192 x 16 B]
  uint16_t* outbuf = reinterpret_cast<uint16_t*>(sfbuf + 2 * X_SF_BYTES);
  uint32_t rank, cluster_id, nclusters;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(cluster_id));
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(nclusters));
  const int c0 = static_cast<int>(cluster_id), cstep = static_cast<int>(nclusters);

  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < X_STAGES; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bar_sffull[s]), 1);
      mbar_init(smem_u32(&bar_sfempty[s]), X_SCALE_WARPS);
    }
    for (int s = 0; s < X_SF_SLOTS; ++s) mbar_init(smem_u32(&bar_sfready[s]), X_CLUSTER * X_SCALE_WARPS);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bar_accf[b]), 1);
      mbar_init(smem_u32(&bar_acce[b]), X_CLUSTER * X_EPI_WARPS);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmSX);
    tma_prefetch_desc(&tmSW);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem_base)),
                 "r"(X_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers and tensor memory exist before either touches the other's
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t g = 0;  // stages issued so far
      for (int t = c0; t < units && !s_abort; t += cstep) {
        const XTile ti = x_decode(t, TB, M);
        const int yx = static_cast<int>(ti.row0) + static_cast<int>(rank) * (ti.n_eff >> 1);
        const int yw = ti.wb * X_WROWS + static_cast<int>(rank) * X_WHALF;
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          if (kb % X_SF_GROUP == 0) {  // the scales of this stage and the next three
            const uint32_t grp = g / X_SF_GROUP;  // groups start at kb % 4 == 0 of every tile (nkb % 4 == 0)
            const uint32_t sl = grp & 1u;
            if (!mbar_wait(smem_u32(&bar_sfempty[sl]), ((grp >> 1) & 1u) ^ 1u, &s_abort, a.status, 11u)) break;
            const uint32_t sf = smem_u32(&bar_sffull[sl]);
            mbar_expect_tx(sf, X_SF_BYTES);
            const uint32_t sb = smem_u32(sfbuf + sl * X_SF_BYTES);
            tma_load_2d(sb, &tmSW, kb * (X_BK / 32), yw, sf);
            tma_load_2d(sb + X_SFW_BYTES, &tmSX, kb * (X_BK / 32), static_cast<int>(ti.row0), sf);
          }
          const int stage = static_cast<int>(g % X_STAGES);
          if (!mbar_wait(smem_u32(&bar_empty[stage]), ((g / X_STAGES) & 1u) ^ 1u, &s_abort, a.status, 1u)) break;
          const uint32_t full = smem_u32(&bar_full[stage]);
          if (rank == 0) mbar_expect_tx(full, X_CLUSTER * X_STAGE_BYTES);
          const uint32_t full_even = smem_cluster_addr(full, 0);
          const uint32_t sa = stage_base + stage * X_STAGE_BYTES;
          tma_load_2d_pair(sa, &tmW, kb * X_BK, yw, full_even);
          tma_load_2d_pair(sa + X_W_BYTES, &tmX, kb * X_BK, yx, full_even);
        }
      }
      // Drain: the last fill of every stage has been consumed.
      for (uint32_t i = 0; i < X_STAGES && !s_abort; ++i, ++g) {
        const int stage = static_cast<int>(g % X_STAGES);
        if (!mbar_wait(smem_u32(&bar_empty[stage]), ((g / X_STAGES) & 1u) ^ 1u, &s_abort, a.status, 5u)) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer (even CTA, whole warp)
    if (rank == 0) {
      uint32_t g = 0, acc_count = 0;
      bool ok = true;
      for (int t = c0; t < units && ok && !s_abort; t += cstep) {
        const XTile ti = x_decode(t, TB, M);
        const uint32_t b = acc_count & 1u;
        const uint32_t use = acc_count >> 1;
        if (!warp_wait(smem_u32(&bar_acce[b]), (use & 1u) ^ 1u, &s_abort, a.status, 2u)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + x_acc_col(b);
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int stage = static_cast<int>(g % X_STAGES);
          const int slot = static_cast<int>(g % X_SF_SLOTS);
          if (!warp_wait(smem_u32(&bar_full[stage]), (g / X_STAGES) & 1u, &s_abort, a.status, 3u) ||
              !warp_wait(smem_u32(&bar_sfready[slot]), (g / X_SF_SLOTS) & 1u, &s_abort, a.status, 6u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = stage_base + stage * X_STAGE_BYTES;
          const uint64_t adesc = smem_desc_sw128(sa);
          const uint64_t bdesc = smem_desc_sw128(sa + X_W_BYTES);
          const uint32_t sfa = tmem_base + x_sf_col(slot), sfb = sfa + 8u;
#pragma unroll
          for (int k = 0; k < X_BK / 32; ++k)
            tc_mma_pair_mx(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc_mx(ti.n_eff, static_cast<uint32_t>(k)), sfa,
                           sfb, (kb > 0 || k > 0) ? 1u : 0u);
          tc_commit_pair_mc(smem_u32(&bar_empty[stage]), X_PAIR_MASK);  // frees the stage and scale slot in both
        }
        tc_commit_pair_mc(smem_u32(&bar_accf[b]), X_PAIR_MASK);
        ++acc_count;
      }
    }
  } else if (warp < X_EPI0) {
    // ------------------------------------------------------------- scale warps (both CTAs)
    const int q = warp & 3;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    const uint32_t sfready_even0 = smem_cluster_addr(smem_u32(&bar_sfready[0]), 0);
    uint32_t g = 0;
    bool ok = true;
    // The group's 16 scale bytes of this lane's rows (weights: rows lane + 32c, c < 4; tokens: c < 6), read
    // from shared memory once per group as whole 16-byte rows (a warp reads 512 contiguous bytes: no bank
    // conflict) and kept in registers for the group's four stages.
    uint4 wv[4], xv[6];
    for (int t = c0; t < units && ok; t += cstep) {
      for (int kb = 0; kb < nkb && ok; ++kb, ++g) {
        const uint32_t grp = g / X_SF_GROUP;
        const uint32_t sl = grp & 1u;
        const int w4 = static_cast<int>(g % X_SF_GROUP);  // which 32-bit word of the group's 16 bytes a row
        if (w4 == 0) {  // groups start at kb % 4 == 0 of every tile (nkb % 4 == 0)
          const int got = mbar_wait(smem_u32(&bar_sffull[sl]), (grp >> 1) & 1u, &s_abort, a.status, 12u) ? 1 : 0;
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          const uint4* sw128 = reinterpret_cast<const uint4*>(sfbuf + sl * X_SF_BYTES);
          const uint4* sx128 = reinterpret_cast<const uint4*>(sfbuf + sl * X_SF_BYTES + X_SFW_BYTES);
#pragma unroll
          for (int c = 0; c < 4; ++c) wv[c] = sw128[32 * c + lane];
#pragma unroll
          for (int c = 0; c < 6; ++c) xv[c] = sx128[32 * c + lane];
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bar_sfempty[sl]));  // this warp is done with the group's bytes
        }
        auto word = [w4](const uint4& v) { return w4 == 0 ? v.x : w4 == 1 ? v.y : w4 == 2 ? v.z : v.w; };
        // lane i of every quadrant holds, in column c, the scales of row 32c + i (weights: 4 columns, tokens: 6)
        const uint32_t w0 = word(wv[0]), w1 = word(wv[1]), w2 = word(wv[2]), w3 = word(wv[3]);
        const uint32_t x0 = word(xv[0]), x1 = word(xv[1]), x2 = word(xv[2]), x3 = word(xv[3]);
        const uint32_t x4 = word(xv[4]), x5 = word(xv[5]);
        const int slot = static_cast<int>(g % X_SF_SLOTS);
        if (g >= X_SF_SLOTS) {  // the slot was last read by the MMAs of stage g - 4
          const uint32_t gp = g - X_SF_SLOTS;
          const int free_ok =
              mbar_wait(smem_u32(&bar_empty[gp % X_STAGES]), (gp / X_STAGES) & 1u, &s_abort, a.status, 13u) ? 1 : 0;
          if (!__all_sync(0xffffffffu, free_ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        const uint32_t col = lane_addr + x_sf_col(slot);
        tmem_st4(col, w0, w1, w2, w3);
        tmem_st4(col + 8u, x0, x1, x2, x3);
        tmem_st2(col + 12u, x4, x5);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(sfready_even0 + 8u * static_cast<uint32_t>(slot));
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    const int ew = warp - X_EPI0;
    const int q = warp & 3;
    const int h = ew >> 2;  // token half: columns [96h, 96h + 96)
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    const uint32_t acce_even = smem_cluster_addr(smem_u32(&bar_acce[0]), 0);
    uint16_t* stg = outbuf + ew * X_NHALF * 32;
    uint32_t acc_count = 0;
    for (int t = c0; t < units && !s_abort; t += cstep) {
      const XTile ti = x_decode(t, TB, M);
      const uint32_t b = acc_count & 1u;
      const uint32_t use = acc_count >> 1;
      int got = 0;
      if (lane == 0) got = mbar_wait(smem_u32(&bar_accf[b]), use & 1u, &s_abort, a.status, 4u) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      tc_fence_after();
      const uint32_t col0 = x_acc_col(b) + X_NHALF * h;
#pragma unroll
      for (int j = 0; j < X_NHALF / 16; ++j) {
        uint32_t v[16];
        tmem_ld16(lane_addr + col0 + 16 * j, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) stg[(16 * j + i) * 32 + lane] = f32_to_bf16_bits(__uint_as_float(v[i]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce_even + 8u * b);
      ++acc_count;
      const int tv = min(X_NHALF, ti.tvalid - X_NHALF * h);
      const int64_t n0 = static_cast<int64_t>(ti.wb) * X_WROWS + static_cast<int64_t>(rank) * X_WHALF + 32 * q;
      x_store_rows(stg, a.y, ti.row0 + X_NHALF * h, N, n0, tv, lane);
      __syncwarp();  // the staging buffer is read before the next tile writes it
    }
  }

  // ---- teardown: on abort, give in-flight copies and MMAs time to land first, then the pair leaves together.
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
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(X_TMEM_COLS)
                 : "memory");
  }
}

constexpr size_t kMxTcSmem = static_cast<size_t>(X_STAGES) * X_STAGE_BYTES + 2 * X_SF_BYTES + X_OUT_BYTES + 1024;

}  // namespace

bool mx_tc_supported(int64_t M, int64_t N, int64_t K) {
  return M > 0 && N > 0 && K > 0 && K % (X_BK * X_SF_GROUP) == 0 && N % 8 == 0 && M <= INT32_MAX && N <= INT32_MAX;
}

cudaError_t launch_mx_tc(const uint8_t* qa, const uint8_t* sa, int64_t M, int64_t K, const uint8_t* qw,
                         const uint8_t* sw, int64_t N, uint16_t* y, DeviceStatus* status, int num_sms,
                         cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  // E4M3 tokens [M,K] in boxes of 96 rows x 128 bytes; E4M3 weights [N,K] in boxes of 128 rows x 128 bytes;
  // E8M0 scales [rows, K/32] in boxes of 16 bytes (four stages) x 192 token rows / 128 weight rows
  CUtensorMap mx, mw, msx, msw;
  if (!encode_map_2d(&mx, qa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, M, K, X_BK, X_NHALF, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_map_2d(&mw, qw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, N, K, X_BK, X_WHALF, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_map_2d(&msx, sa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, M, K / 32, 16, X_NT, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_map_2d(&msw, sw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, N, K / 32, 16, X_WHALF, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const int64_t units = ((M + X_NT - 1) / X_NT) * ((N + X_WROWS - 1) / X_WROWS);
  const int64_t clusters = std::max<int64_t>(1, std::min<int64_t>(units, num_sms / X_CLUSTER));
  const int grid = static_cast<int>(clusters * X_CLUSTER);
  cudaError_t e = cudaFuncSetAttribute(mx_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kMxTcSmem));
  if (e != cudaSuccess) return e;
  XArgs xa;
  xa.M = M;
  xa.N = N;
  xa.K = K;
  xa.y = y;
  xa.status = status;
  mx_tc_kernel<<<grid, X_THREADS, kMxTcSmem, stream>>>(mx, mw, msx, msw, xa);
  return cudaGetLastError();
}

}  // namespace w8a8
