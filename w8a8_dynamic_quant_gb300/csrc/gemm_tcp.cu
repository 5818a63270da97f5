// gemm_tcp.cu -- exact INT8 contraction on CTA pairs of the 5th-generation
// tensor cores with the weights read as INT8: the dense prefill linear and
// the grouped expert GEMMs of MoE prefill (W13 + SwiGLU, W2), for packed
// weights with or without an FP16 copy (only the INT8 payload is read).
//
// Page "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子": §二
// npu_quant_matmul (INT8 x INT8 -> INT32, then * x_scale * w_scale (+bias) ->
// BF16; the weight stays INT8 after loading), §三 npu_grouped_matmul over
// group_list and the W13 -> SwiGLU step, §四 (prefill, large M, gets its own
// tiling).
//
// Engine.  sm_103a has no integer tcgen05.mma kind, so the codes are fed as
// integer-valued FP16 (exact) to tcgen05.mma.kind::f16 with FP32 accumulators
// in tensor memory; products |a*b| <= 2^14 are exact and a fresh accumulator
// is started every 1024 of K, so every accumulator holds an exact integer.
//
// Tile.  The weights are the MMA's M side: a CTA pair (tcgen05 cta_group::2)
// owns 256 weight rows of one expert, 128 in each CTA, and a block of up to
// 192 of the expert's tokens as N -- the even CTA holds the first half of the
// block's tokens, the odd CTA the second.  N is the block's token count
// rounded up to 16, so an expert's ragged last block costs at most 15 rows of
// work.  Per CTA and 128 of K a stage holds the 128 x 128-byte INT8 weight
// tile and the two 64-K FP16 sub-tiles of its token rows (128-byte swizzle),
// 40 KB, brought by TMA into a ring of four stages (five for the INT32
// output, whose epilogue needs no shared memory).  The BF16 epilogues stage
// each warp's results in shared memory as [token][32 channels] and write them
// as 16-byte pieces of output rows: one thread per channel storing 2 bytes
// per token row cost about 80 cycles a store.  Four converter warps widen
// the weight tile -- lane r takes row r -- to integer-valued FP16 and store it
// into tensor memory, where the MMA reads its A operand, so the large operand
// is never written back to shared memory.  Per SM and 128 of K this moves
// 16 KB of weights and 24 KB of tokens through shared memory for 6.3 MFLOP,
// about 100 bytes per clock at the full tensor rate.
//
// Tensor memory (512 columns per CTA): two accumulators of 192 columns at 0
// and 256, and two A buffers of 128 K (64 columns of FP16 pairs) at 192 and
// 448.  The accumulators alternate per 1024-deep chunk of K, so the epilogue
// drains one while the MMAs fill the other.  Stage g of the ring (counted over
// the whole run) is widened into A buffer g%2, so the commit that frees stage
// g-2 of the shared-memory ring also frees the buffer stage g reuses: one
// commit per stage frees both.
//
// Synchronisation.  TMA: each CTA's weight tile completes on its own barrier
// (its converters wait for it); both CTAs' token tiles complete on the even
// CTA's barrier.  Converters of both CTAs arrive on the even CTA's A-buffer
// barrier once per stage; the even CTA's MMA warp (one elected lane) issues tcgen05.mma.cta_group::2
// M = 256 N = 16..192 K = 16 and frees shared-memory stages (with their A
// slots) and accumulators in both CTAs by multicast commits.  Both CTAs'
// epilogue warps release an accumulator on the even CTA's barrier.
//
// Warp roles (448 threads, one CTA per SM, persistent over tiles):
//   warp 0       TMA producer
//   warp 1       TMEM owner; one elected lane of the even CTA's warp issues the MMAs
//   warps 2-5    converters: lane r of warp w widens weight row 32*(w%4)+r
//   warps 6-13   epilogue: warp w reads TMEM lanes 32*(w%4).. (weight rows)
//                and one half (96 tokens) of the accumulator's columns
// W13 + SwiGLU: the gate/up interleave puts gate channel j in tile row j%64
// and up channel j in row 64 + j%64 of a CTA's 128 rows, so a gate warp and
// its up warp meet through shared memory: the gate warp passes its BF16 gate
// values of the second 48 tokens of its half, the up warp its BF16 up values
// of the first 48, and each computes SwiGLU for 48 tokens (the SwiGLU math is
// spread over all four SM sub-partitions) in a compact loop over values kept
// in shared memory.
// Every mbarrier wait is bounded (2 s): on expiry the CTA sets
// W8A8_ERR_DEVICE_TIMEOUT, lets in-flight copies land, frees TMEM and returns.
#include "kernels.cuh"
#include "tc_common.cuh"

namespace w8a8 {

namespace {

using namespace tc;

constexpr int P_WROWS = 256;  // weight rows per pair tile (MMA M)
constexpr int P_WHALF = 128;  // weight rows per CTA
constexpr int P_NT = 192;     // most tokens per tile (MMA N)
constexpr int P_NHALF = 96;   // token rows per CTA
constexpr int P_BK = 128;     // K per shared-memory stage
constexpr int P_MAX_STAGES = 5;
constexpr int p_stages(int mode) { return mode == EPI_ACC ? 5 : 4; }
constexpr int P_KB_PER_CHUNK = kChunkK / P_BK;  // 8
constexpr uint32_t P_X_SUB = P_NHALF * 64 * 2;  // 64-K fp16 token sub-tile (12 KB)
constexpr uint32_t P_X_BYTES = 2 * P_X_SUB;     // 24 KB
constexpr uint32_t P_W_BYTES = P_WHALF * P_BK;  // 16 KB
constexpr uint32_t P_STAGE_BYTES = P_W_BYTES + P_X_BYTES;
constexpr int P_THREADS = 448;
constexpr int P_CONV_WARPS = 4;
constexpr int P_EPI0 = 6;
constexpr int P_EPI_WARPS = 8;
constexpr int P_CLUSTER = 2;
constexpr uint16_t P_PAIR_MASK = 0x3;
constexpr uint32_t P_TMEM_COLS = 512;
// accumulator b at column 256*b; A buffer p (128 K, 64 columns) at 192 + 256*p
__host__ __device__ constexpr uint32_t p_acc_col(uint32_t b) { return 256u * b; }
__host__ __device__ constexpr uint32_t p_abuf_col(uint32_t p) { return 192u + 256u * p; }
static_assert(p_abuf_col(1) + 64u <= 512u && p_acc_col(1) + 192u <= p_abuf_col(1) && p_acc_col(0) + 192u <= p_abuf_col(0),
              "tensor memory budget");
constexpr int kMaxE = 1024;
constexpr int P_XCH = P_NHALF / 2;  // SwiGLU tokens each warp of a gate/up pair hands to the other
// SwiGLU buffers: [gate warp pair][token half][gate give, gate keep, up give, up keep][48 tokens][32 lanes] bf16
constexpr uint32_t P_XCH_BYTES = 4 * 4 * P_XCH * 32 * 2;
// BF16 output staging: per epilogue warp [96 tokens][32 channels] bf16
constexpr uint32_t P_OUT_BYTES = P_EPI_WARPS * P_NHALF * 32 * 2;
__host__ __device__ constexpr uint32_t p_epi_bytes(int mode) {
  return mode == EPI_SWIGLU ? P_XCH_BYTES : mode == EPI_BF16 ? P_OUT_BYTES : 0u;
}
static_assert(P_STAGE_BYTES % 1024 == 0 && P_W_BYTES % 1024 == 0 && P_X_SUB % 1024 == 0, "1024-byte tiles");
static_assert(P_NHALF % 8 == 0, "whole 8-row swizzle atoms per CTA");

// kind::f16 instruction descriptor: D = F32, A = B = F16, both K-major, M = 256, N = n (multiple of 16).
__device__ __forceinline__ uint32_t idesc_pair(int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(P_WROWS >> 4) << 24);
}

// D(tmem, both CTAs) (+)= A(tmem, both CTAs) * B(smem desc, both CTAs), kind::f16 on a CTA pair: each CTA's
// tensor memory holds its 128 rows of A (K packed two fp16 per column) and of D; B rows [0,N/2) in the even
// CTA, [N/2,N) in the odd one.
// Issued by the elected lane of the (converged) MMA warp, as the issue helpers of tc_common.cuh.
__device__ __forceinline__ void tc_mma_pair_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                   uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 16 int8 (one 16-byte chunk) -> 8 words of fp16 pairs.
__device__ __forceinline__ void widen16(const uint4& x, uint32_t* h) {
  s8x4_to_f16x4(x.x, h[0], h[1]);
  s8x4_to_f16x4(x.y, h[2], h[3]);
  s8x4_to_f16x4(x.z, h[4], h[5]);
  s8x4_to_f16x4(x.w, h[6], h[7]);
}

// Rows [0, rows) of a warp's staging buffer [rows][32] bf16 (shared memory) to out[(row0 + r) * ld + c0 + c],
// c < min(32, ld - c0): 16-byte stores of whole 64-byte row pieces when they fit (8 rows a warp instruction),
// else one 2-byte store a lane and row.
__device__ __forceinline__ void store_rows(const uint16_t* stg, uint16_t* out, int64_t row0, int64_t ld, int64_t c0,
                                           int rows, int lane) {
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

struct PTile {
  int e, tb, wb, cnt;
  int n_eff;     // MMA N: the block's token count rounded up to 16
  int tvalid;    // tokens of the block that belong to the expert
  int64_t row0;  // first routed row of the block
};

// Work unit t -> (expert, 256-row weight block, token block), rasterised in groups of up to P_GROUP_W weight
// blocks: inside a group the weight block varies fastest, then the token block.  The pairs in flight then
// work on a few token blocks against the group's weight blocks, which stay in L2 while the expert's token
// blocks sweep past them, and each token block is fetched from HBM about once per group.  (With the token
// block fastest over a whole expert, the dense prefill shape read its 126 MB of operands 7 times from DRAM:
// the output writes pushed the activations out of L2 between weight blocks.)
constexpr int P_GROUP_W = 16;
__device__ __forceinline__ PTile p_decode(int t, int E, int WB, const int* s_unit_prefix, const int* s_row_off) {
  PTile ti;
  ti.e = expert_of(t, E, s_unit_prefix);
  const int local = t - s_unit_prefix[ti.e];
  ti.cnt = s_row_off[ti.e + 1] - s_row_off[ti.e];
  const int TB = (ti.cnt + P_NT - 1) / P_NT;
  const int g = local / (TB * P_GROUP_W);
  const int rem = local - g * TB * P_GROUP_W;
  const int gw = min(P_GROUP_W, WB - g * P_GROUP_W);
  ti.tb = rem / gw;
  ti.wb = g * P_GROUP_W + rem % gw;
  ti.tvalid = min(P_NT, ti.cnt - ti.tb * P_NT);
  ti.n_eff = (ti.tvalid + 15) & ~15;
  ti.row0 = static_cast<int64_t>(s_row_off[ti.e]) + static_cast<int64_t>(ti.tb) * P_NT;
  return ti;
}

// 14 warps: the register file is split over the four SM sub-partitions, one of which holds four of the
// warps, so 128 registers a thread is the most the launch allows.
template <int MODE>
__global__ void __cluster_dims__(P_CLUSTER, 1, 1) __launch_bounds__(P_THREADS, 1)
tcp_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const GemmArgs a) {
  constexpr int STAGES = p_stages(MODE);
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_wfull[P_MAX_STAGES];  // this CTA's weight tile landed
  __shared__ __align__(8) uint64_t bar_xfull[P_MAX_STAGES];  // even CTA: both CTAs' token tiles landed
  __shared__ __align__(8) uint64_t bar_empty[P_MAX_STAGES];  // the MMAs reading the stage (and its A buffer) are done
  __shared__ __align__(8) uint64_t bar_aready[2];             // even CTA: both CTAs widened the stage into A buffer
  __shared__ __align__(8) uint64_t bar_accf[2];
  __shared__ __align__(8) uint64_t bar_acce[2];          // even CTA: both CTAs drained the accumulator
  // SwiGLU exchange, per (warp pair, token half): gate values written / read, up values written / read
  __shared__ __align__(8) uint64_t bar_gfull[4];
  __shared__ __align__(8) uint64_t bar_gfree[4];
  __shared__ __align__(8) uint64_t bar_ufull[4];
  __shared__ __align__(8) uint64_t bar_ufree[4];
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;
  __shared__ int s_bad;
  __shared__ int s_unit_prefix[kMaxE + 1];
  __shared__ int s_row_off[kMaxE + 1];
  __shared__ int s_warp[P_THREADS / 32];
  __shared__ float s_sx[P_EPI_WARPS][P_NHALF];           // token scales of each epilogue warp's tile half

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = static_cast<int>(a.E);
  const int64_t N = a.N;
  const int64_t K = a.K;
  const int WB = static_cast<int>((N + P_WROWS - 1) / P_WROWS);
  const int nkb = static_cast<int>((K + P_BK - 1) / P_BK);
  const int nchunk = (nkb + P_KB_PER_CHUNK - 1) / P_KB_PER_CHUNK;

  // (pointer arithmetic on the shared array keeps the shared address space known to the compiler)
  uint8_t* stages = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  // after the ring: the SwiGLU exchange buffers, or the BF16 output staging
  uint16_t* xch = reinterpret_cast<uint16_t*>(stages + STAGES * P_STAGE_BYTES);
  const uint32_t stage_base = smem_u32(stages);
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
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&bar_wfull[s]), 1);
      mbar_init(smem_u32(&bar_xfull[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) mbar_init(smem_u32(&bar_aready[s]), P_CLUSTER * P_CONV_WARPS);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bar_accf[b]), 1);
      mbar_init(smem_u32(&bar_acce[b]), P_CLUSTER * P_EPI_WARPS);
    }
    for (int p = 0; p < 4; ++p) {
      mbar_init(smem_u32(&bar_gfull[p]), 1);
      mbar_init(smem_u32(&bar_gfree[p]), 1);
      mbar_init(smem_u32(&bar_ufull[p]), 1);
      mbar_init(smem_u32(&bar_ufree[p]), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem_base)),
                 "r"(P_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  // ---- per-expert rows and work units (token blocks x 256-row weight blocks)
  int units_total;
  const int rows_total = scan_groups<P_THREADS, kMaxE>(
      a, E, [WB](int c) { return ((c + P_NT - 1) / P_NT) * WB; }, s_row_off, s_unit_prefix, s_warp, &s_bad,
      &units_total);
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers and tensor memory exist before either touches the other's
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  int bad = s_bad;
  if (rows_total != a.R) bad |= W8A8_ERR_GROUP_LIST << 8;
  if (bad && tid == 0 && blockIdx.x == 0) set_status(a.status, (bad & 0xff) ? (bad & 0xff) : (bad >> 8), 0u);
  const int units = bad ? 0 : units_total;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = c0; t < units && !s_abort; t += cstep) {
        const PTile ti = p_decode(t, E, WB, s_unit_prefix, s_row_off);
        // this CTA's token rows: the first or the second half of the block's n_eff tokens
        const int yx = static_cast<int>(ti.row0) + static_cast<int>(rank) * (ti.n_eff >> 1);
        const int yw = static_cast<int>(static_cast<int64_t>(ti.e) * N + static_cast<int64_t>(ti.wb) * P_WROWS) +
                       static_cast<int>(rank) * P_WHALF;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(smem_u32(&bar_empty[stage]), phase ^ 1u, &s_abort, a.status, 1u)) break;
          const uint32_t sa = stage_base + stage * P_STAGE_BYTES;
          const uint32_t wf = smem_u32(&bar_wfull[stage]);
          mbar_expect_tx(wf, P_W_BYTES);
          tma_load_2d(sa, &tmW, kb * P_BK, yw, wf);
          const uint32_t xf = smem_u32(&bar_xfull[stage]);
          if (rank == 0) mbar_expect_tx(xf, P_CLUSTER * P_X_BYTES);
          const uint32_t xf_even = smem_cluster_addr(xf, 0);
          tma_load_2d_pair(sa + P_W_BYTES, &tmX, kb * P_BK, yx, xf_even);
          tma_load_2d_pair(sa + P_W_BYTES + P_X_SUB, &tmX, kb * P_BK + 64, yx, xf_even);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: the last fill of every stage has been consumed, so no copy into this CTA and no arrival on
      // the even CTA's barriers from this CTA's copies is still in flight when the pair leaves.
      for (int i = 0; i < STAGES && !s_abort; ++i) {
        if (!mbar_wait(smem_u32(&bar_empty[stage]), phase ^ 1u, &s_abort, a.status, 5u)) break;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer (even CTA, whole warp)
    if (rank == 0) {
      uint32_t g = 0;  // stages consumed so far: ring index g % STAGES, A buffer g % 2
      uint32_t acc_count = 0;
      for (int t = c0; t < units && !s_abort; t += cstep) {
        const PTile ti = p_decode(t, E, WB, s_unit_prefix, s_row_off);
        const uint32_t idesc = idesc_pair(ti.n_eff);
        bool ok = true;
        for (int c = 0; c < nchunk && ok; ++c) {
          const uint32_t b = acc_count & 1u;
          const uint32_t use = acc_count >> 1;
          if (!warp_wait(smem_u32(&bar_acce[b]), (use & 1u) ^ 1u, &s_abort, a.status, 2u)) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + p_acc_col(b);
          const int kb_end = min(nkb, (c + 1) * P_KB_PER_CHUNK);
          for (int kb = c * P_KB_PER_CHUNK; kb < kb_end && ok; ++kb, ++g) {
            const int stage = static_cast<int>(g % STAGES);
            if (!warp_wait(smem_u32(&bar_xfull[stage]), (g / STAGES) & 1u, &s_abort, a.status, 3u) ||
                !warp_wait(smem_u32(&bar_aready[g & 1u]), (g >> 1) & 1u, &s_abort, a.status, 6u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sx = stage_base + stage * P_STAGE_BYTES + P_W_BYTES;
            const uint32_t abuf = tmem_base + p_abuf_col(g & 1u);
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // the two 64-K token sub-tiles of the stage
              const uint64_t bdesc = smem_desc_sw128(sx + h * P_X_SUB);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                tc_mma_pair_tmem_a(d_tmem, abuf + 32u * h + 8u * k, bdesc + 2u * k, idesc,
                                   (kb > c * P_KB_PER_CHUNK || h > 0 || k > 0) ? 1u : 0u);
            }
            // frees the stage and its two A slots in both CTAs
            tc_commit_pair_mc(smem_u32(&bar_empty[stage]), P_PAIR_MASK);
          }
          tc_commit_pair_mc(smem_u32(&bar_accf[b]), P_PAIR_MASK);
          ++acc_count;
        }
        if (!ok) break;
      }
    }
  } else if (warp < P_EPI0) {
    // ------------------------------------------------------------- converters (both CTAs)
    const int q = warp & 3;
    const int row = 32 * q + lane;  // weight row of this CTA's half == TMEM lane
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    const uint32_t aready_even0 = smem_cluster_addr(smem_u32(&bar_aready[0]), 0);
    uint32_t g = 0;  // stages widened so far (as in the MMA issuer)
    bool ok = true;
    for (int t = c0; t < units && ok; t += cstep) {
      for (int kb = 0; kb < nkb && ok; ++kb, ++g) {
        const int stage = static_cast<int>(g % STAGES);
        // every lane observes the completed weight copy itself
        const int got = mbar_wait(smem_u32(&bar_wfull[stage]), (g / STAGES) & 1u, &s_abort, a.status, 7u) ? 1 : 0;
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        // weight row `row`: 128 bytes, 16-byte chunk c stored at chunk c ^ (row & 7) (128-byte swizzle)
        const uint8_t* wrow = stages + stage * P_STAGE_BYTES + row * P_BK;
        uint32_t v[64];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          widen16(*reinterpret_cast<const uint4*>(wrow + ((c ^ (row & 7)) << 4)), &v[8 * c]);
        if (g >= 2) {
          // A buffer g % 2 was last read by stage g - 2: wait for the commit that freed that stage
          const uint32_t gp = g - 2;
          const int free_ok =
              mbar_wait(smem_u32(&bar_empty[gp % STAGES]), (gp / STAGES) & 1u, &s_abort, a.status, 8u) ? 1 : 0;
          if (!__all_sync(0xffffffffu, free_ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        tmem_st64(lane_addr + p_abuf_col(g & 1u), v);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(aready_even0 + 8u * (g & 1u));
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    const int ew = warp - P_EPI0;
    const int q = warp & 3;
    const int h = ew >> 2;              // token half of the tile: columns [96h, 96h + 96)
    const int n_loc = 32 * q + lane;    // weight row of this CTA's half
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    const uint32_t acce_even = smem_cluster_addr(smem_u32(&bar_acce[0]), 0);
    float* sxw = s_sx[ew];
    uint32_t acc_count = 0, ntile = 0;
    // W13 + SwiGLU: the SwiGLU of a tile's tokens runs in slices before each chunk wait of the next tile
    // (and what is left after its last chunk), so it overlaps that tile's MMAs instead of holding up the
    // accumulator hand-over.  The tile whose SwiGLU is outstanding:
    struct PendingSwiglu {
      bool on = false;
      int i = 0, nown = 0;       // next token of the 48, tokens with rows
      uint32_t par = 0;          // the tile's exchange phase
      int64_t row = 0, j = 0;    // first output row, this lane's channel
      uint16_t* keep = nullptr;  // my kept values (h replaces them in place)
      const uint16_t* other = nullptr;
    } pd;
    const bool sw_up = (q >= 2);
    const int sw_pi = (q & 1) * 2 + h;
    const int sw_slice = (P_XCH + nchunk - 1) / nchunk;
    // SwiGLU of up to `budget` outstanding tokens; false when the CTA aborts.
    auto swiglu_work = [&](int budget) -> bool {
      if (!pd.on) return true;
      if (pd.i == 0) {  // the partner's hand-over of that tile
        int got = 0;
        const uint32_t o_full = smem_u32(sw_up ? &bar_gfull[sw_pi] : &bar_ufull[sw_pi]);
        if (lane == 0) got = mbar_wait(o_full, pd.par, &s_abort, a.status, 10u) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, got, 0)) return false;
      }
      const int end = min(P_XCH, pd.i + budget);
#pragma unroll 4
      for (int i = pd.i; i < end; ++i) {
        const float mine = bf16_bits_to_f32(pd.keep[i * 32]);
        const float theirs = bf16_bits_to_f32(pd.other[i * 32]);
        pd.keep[i * 32] = sw_up ? swiglu_bf16(theirs, mine) : swiglu_bf16(mine, theirs);  // h, in place
      }
      pd.i = end;
      if (pd.i == P_XCH) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(sw_up ? &bar_gfree[sw_pi] : &bar_ufree[sw_pi]));
        // h of my 48 tokens, [token][32 channels j], to 16-byte stores of 64-byte row pieces
        store_rows(pd.keep - lane, static_cast<uint16_t*>(a.out), pd.row, N / 2, pd.j - lane, pd.nown, lane);
        pd.on = false;
      }
      return true;
    };
    for (int t = c0; t < units && !s_abort; t += cstep) {
      const PTile ti = p_decode(t, E, WB, s_unit_prefix, s_row_off);
      const int64_t rowh = ti.row0 + P_NHALF * h;                    // routed row of column 96h
      const int tv = min(P_NHALF, ti.tvalid - P_NHALF * h);         // tokens of the half that have rows
      if (MODE != EPI_ACC) {  // the half's token scales, loaded while the tile's MMAs run
        for (int i = lane; i < P_NHALF; i += 32)
          sxw[i] = i < tv ? (a.x_scale != nullptr ? a.x_scale[rowh + i] : 1.0f) : 0.0f;
        __syncwarp();
      }
      int sums[P_NHALF];
#pragma unroll
      for (int i = 0; i < P_NHALF; ++i) sums[i] = 0;
      bool ok = true;
      for (int c = 0; c < nchunk; ++c) {
        if (MODE == EPI_SWIGLU && !swiglu_work(sw_slice)) {
          ok = false;
          break;
        }
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
        const uint32_t col0 = p_acc_col(b) + P_NHALF * h;
#pragma unroll
        for (int j = 0; j < P_NHALF / 16; ++j) {
          uint32_t v[16];
          tmem_ld16(lane_addr + col0 + 16 * j, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) sums[16 * j + i] += __float2int_rn(__uint_as_float(v[i]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acce_even + 8u * b);
        ++acc_count;
      }
      if (!ok) break;
      if (MODE == EPI_SWIGLU && !swiglu_work(P_XCH)) break;  // the previous tile's SwiGLU, all of what is left

      // Results are computed first (register and shared-memory reads only) and stored afterwards, so the
      // reads and the arithmetic of different tokens overlap instead of queueing behind each global store.
      const int64_t n = static_cast<int64_t>(ti.wb) * P_WROWS + static_cast<int64_t>(rank) * P_WHALF + n_loc;
      if constexpr (MODE == EPI_ACC) {
        if (n < N) {
          int32_t* dst = static_cast<int32_t*>(a.out) + rowh * N + n;
#pragma unroll
          for (int i = 0; i < P_NHALF; ++i)
            if (i < tv) dst[i * N] = sums[i];
        }
      } else if constexpr (MODE == EPI_BF16) {
        const bool nin = n < N;
        const float sw = nin ? a.w_scale[static_cast<int64_t>(ti.e) * N + n] : 0.0f;
        const float bias = (nin && a.bias != nullptr) ? bf16_bits_to_f32(a.bias[n]) : 0.0f;
        const int32_t qb = (nin && a.qbias != nullptr) ? a.qbias[n] : 0;
        // through shared memory, [token][this warp's 32 channels], to 16-byte stores of 64-byte row pieces
        uint16_t* stg = xch + ew * P_NHALF * 32;
#pragma unroll
        for (int i = 0; i < P_NHALF; ++i) {
          float f = a.qbias != nullptr ? dequant_q(sums[i], qb, sxw[i], sw) : dequant(sums[i], sxw[i], sw);
          if (a.bias) f = __fadd_rn(f, bias);
          stg[i * 32 + lane] = f32_to_bf16_bits(f);
        }
        __syncwarp();
        store_rows(xch + ew * P_NHALF * 32, static_cast<uint16_t*>(a.out), rowh, N, n - lane, tv, lane);
        __syncwarp();  // the staging buffer is read before the next tile writes it
      } else {  // EPI_SWIGLU: rows [0,64) of this CTA's half are gate channels, [64,128) the matching up channels
        const int64_t I = N / 2;
        const int64_t j = (static_cast<int64_t>(ti.wb) * 2 + rank) * kGateUpBlock + 32 * (q & 1) + lane;
        const float swv = j < I ? a.w_scale[static_cast<int64_t>(ti.e) * N + (sw_up ? I : 0) + j] : 0.0f;
        // buffers of this pair: gate warp's hand-over (gate of tokens [48, 96)) and keep (gate of [0, 48)),
        // up warp's hand-over (up of [0, 48)) and keep (up of [48, 96))
        uint16_t* pair_buf = xch + sw_pi * 4 * P_XCH * 32 + lane;
        uint16_t* give = pair_buf + (sw_up ? 2 : 0) * P_XCH * 32;
        uint16_t* keep = pair_buf + (sw_up ? 3 : 1) * P_XCH * 32;
        const uint32_t par = ntile & 1u;
        // my BF16 values into the hand-over and keep buffers, once the partner has read the previous
        // tile's hand-over (this warp's own SwiGLU of that tile is complete: it ran above)
        int got = 0;
        const uint32_t b_free = smem_u32(sw_up ? &bar_ufree[sw_pi] : &bar_gfree[sw_pi]);
        if (lane == 0) got = mbar_wait(b_free, par ^ 1u, &s_abort, a.status, 9u) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, got, 0)) break;
        // gate warp: hands over tokens [48, 96), keeps [0, 48); up warp the other way round (compile-time
        // offsets in each branch keep sums[] in registers)
        if (sw_up) {
#pragma unroll
          for (int i = 0; i < P_XCH; ++i) {
            give[i * 32] = f32_to_bf16_bits(dequant(sums[i], sxw[i], swv));
            keep[i * 32] = f32_to_bf16_bits(dequant(sums[P_XCH + i], sxw[P_XCH + i], swv));
          }
        } else {
#pragma unroll
          for (int i = 0; i < P_XCH; ++i) {
            give[i * 32] = f32_to_bf16_bits(dequant(sums[P_XCH + i], sxw[P_XCH + i], swv));
            keep[i * 32] = f32_to_bf16_bits(dequant(sums[i], sxw[i], swv));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(sw_up ? &bar_ufull[sw_pi] : &bar_gfull[sw_pi]));
        // this tile's SwiGLU becomes the outstanding work of the next tile's chunks
        const int own0 = sw_up ? P_XCH : 0;
        pd.on = true;
        pd.i = 0;
        pd.nown = min(P_XCH, tv - own0);
        pd.par = par;
        pd.row = rowh + own0;
        pd.j = j;
        pd.keep = keep;
        pd.other = pair_buf + (sw_up ? 0 : 2) * P_XCH * 32;
        ++ntile;
      }
      __syncwarp();  // the scales of this tile are read before the next tile overwrites them
    }
    if (MODE == EPI_SWIGLU && !s_abort) swiglu_work(P_XCH);  // the last tile's SwiGLU
  }

  // ---- teardown: on abort, give in-flight copies and MMAs time to land first, then the pair leaves
  // together (no copy or remote arrival may target a CTA that has left).
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
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(P_TMEM_COLS)
                 : "memory");
  }
}

template <int MODE>
cudaError_t launch_tcp_mode(const CUtensorMap& mx, const CUtensorMap& mw, const GemmArgs& a, int grid, size_t smem,
                            cudaStream_t stream) {
  auto k = tcp_gemm_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k<<<grid, P_THREADS, smem, stream>>>(mx, mw, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tcp_gemm(const GemmArgs& a, const void* a_f16, int num_sms, cudaStream_t stream) {
  if (a.R == 0) return cudaSuccess;
  // fp16 token rows [R, K] in boxes of 96 rows x 64 K, and the int8 weight payload [E*N, K] in boxes of
  // 128 rows x 128 K; rows past the ends read as zero
  CUtensorMap mx, mw;
  const uint8_t* w_i8 = static_cast<const uint8_t*>(a.packed) + pack_layout(a.E, a.N, a.K, 0).i8_offset;
  if (!encode_map_2d(&mx, a_f16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.R, a.K, 64, P_NHALF,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_map_2d(&mw, w_i8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.E * a.N, a.K, P_BK, P_WHALF,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int64_t wb = (a.N + P_WROWS - 1) / P_WROWS;
  const int64_t units = ((a.R + P_NT - 1) / P_NT + (a.group_list != nullptr ? a.E : 0)) * wb;
  const int64_t clusters = std::max<int64_t>(1, std::min<int64_t>(units, num_sms / P_CLUSTER));
  const int grid = static_cast<int>(clusters * P_CLUSTER);
  auto smem = [](int mode) { return static_cast<size_t>(p_stages(mode)) * P_STAGE_BYTES + p_epi_bytes(mode) + 1024; };
  switch (a.mode) {
    case EPI_ACC: return launch_tcp_mode<EPI_ACC>(mx, mw, a, grid, smem(EPI_ACC), stream);
    case EPI_SWIGLU: return launch_tcp_mode<EPI_SWIGLU>(mx, mw, a, grid, smem(EPI_SWIGLU), stream);
    default: return launch_tcp_mode<EPI_BF16>(mx, mw, a, grid, smem(EPI_BF16), stream);
  }
}

}  // namespace w8a8
