// gemm_dec.cu -- exact INT8 contraction for decode-sized batches (M <= 64
// tokens), where the weight stream from HBM is the whole cost.
//
// Page "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子": §二
// npu_quant_matmul (INT8 x INT8 -> INT32, * x_scale * w_scale (+bias) ->
// BF16) and §四 (decode, small M, gets its own tiling).
//
// The weights stay INT8 in HBM (one byte per element, row-major, K
// contiguous).  A CTA owns 128 weight rows and a K slice of at most 7 stages
// of 128.  With one CTA per SM, an SM streams at the HBM rate only with about
// 100 KB of reads in flight, so one thread issues tensor-copy (TMA) loads of
// the CTA's WHOLE weight slice at once: per stage a 128-row x 128-byte tile,
// 128-byte swizzled, on its own mbarrier.  When the host made the packed
// buffer itself (it keeps a record of the packs it wrote), the loads are
// issued before the header check instead of after it.
//
// Tensor memory (512 columns) holds every weight stage of the slice at once
// (7 x 64 columns) beside the accumulator (64 columns).  So eight converter
// warps widen each weight stage as it lands -- lane r reads weight row r
// (conflict-free thanks to the swizzle), widens it to integer-valued FP16 and
// stores it into the stage's own A columns -- without waiting for the
// activations, which the kernel before (the quantisation) may still be
// writing.  Once that kernel has finished, the activation tiles of the slice
// (64 tokens x 128 bytes per stage, TMA, 128-byte swizzled, one mbarrier per
// stage) are requested; the converters, in two groups of four warps taking
// alternate stages, widen each into a 128-byte-swizzled K-major FP16 tile in
// the bytes the int8 weight tiles occupied (the B operand), and each stage's
// MMAs follow as soon as its tile is ready.  The MMA is M = 128 weight rows x
// N = 64 tokens x K = 16 into an FP32 TMEM accumulator; the CTA's K slice is
// at most 896, so the accumulator holds an exact integer (|partial| <= 896 *
// 128^2 < 2^24).  The whole MMA warp runs the issue loop and one elected
// lane issues: with every operand warp-uniform, the issue keeps pace with
// the tensor core at this small N, which a single diverged lane does not.
//
// Split-K reduction: each CTA drains its exact partial tile to shared memory
// and adds it into the row block's int32 sum tile in global memory (L2) with
// one bulk reduce-add copy; it then bumps the row block's arrival counter
// (release).  The CTA that arrives last reads the complete sums, applies the
// dequant epilogue, writes BF16 (or the INT32 sums) and zeroes the sum tile and
// the counter for the next call.  Integer addition is exact in any order.
//
// Warps: 0 TMEM owner, TMA producer (lane 0) and MMA issuer (the whole warp);
// 1-8 converters (warp w owns TMEM lanes 32*(w%4).. and K part / token part
// (w-1)/4).  All waits are bounded.
#include "kernels.cuh"
#include "tc_common.cuh"

namespace w8a8 {

namespace {

using namespace tc;

constexpr int DC_ROWS = 128;  // weight rows per CTA (MMA M)
constexpr int DC_TOK = 64;    // token columns (MMA N)
constexpr int DC_BK = 128;    // K per stage
constexpr uint32_t DC_B_SUB = DC_TOK * 128;    // one 64-K fp16 sub-tile (8 KB)
constexpr uint32_t DC_B_BYTES = 2 * DC_B_SUB;  // 128 K of fp16 activations
constexpr int DC_CONV_WARPS = 8;
constexpr int DC_THREADS = 32 * (1 + DC_CONV_WARPS);
constexpr int DC_NPART = DC_CONV_WARPS / 4;          // converter warps per TMEM lane quadrant
constexpr int DC_WCH = 8 / DC_NPART;                 // 16-byte weight chunks per lane per stage
constexpr int DC_TPW = DC_TOK / DC_NPART;            // accumulator columns (tokens) drained per warp
constexpr int DC_XGROUPS = 2;                        // converter groups widening alternate activation stages
constexpr int DC_XWARPS = DC_CONV_WARPS / DC_XGROUPS;
constexpr int DC_XCH = 512 / (32 * DC_XWARPS);       // 16-byte activation chunks per lane per stage
constexpr uint32_t DC_TMEM_COLS = 512;
constexpr uint32_t DC_A_COLS = DC_BK / 2;  // 64 columns of fp16 pairs per A stage
constexpr int DC_MAX_KB = 7;               // stages per CTA: 896 of K
constexpr uint32_t DC_D_COL = DC_MAX_KB * DC_A_COLS;  // every A stage resident; accumulator at [448, 512)
constexpr uint32_t DC_W_STAGE = DC_ROWS * DC_BK;  // int8 weight tile (16 KB)
constexpr uint32_t DC_X_STAGE = DC_TOK * DC_BK;   // int8 activation tile (8 KB)
constexpr uint32_t DC_TILE_I32 = DC_TOK * DC_ROWS * 4;  // int32 partial / sum tile (32 KB)
constexpr int DC_MAX_KSPLIT = 16;  // at most 16 partial tiles added into one sum tile
constexpr int DC_SUM_PER_THREAD = DC_TOK * DC_ROWS / 4 / (32 * DC_CONV_WARPS);  // int4 of the sum tile per thread
constexpr uint32_t kIdescDec = (1u << 4) | (uint32_t(DC_TOK >> 3) << 17) | (uint32_t(DC_ROWS >> 4) << 24);
static_assert(DC_B_BYTES % 1024 == 0 && DC_W_STAGE % 1024 == 0 && DC_X_STAGE % 1024 == 0, "1024-byte aligned tiles");
static_assert(DC_D_COL + DC_TOK <= DC_TMEM_COLS, "tensor memory budget");
static_assert(DC_MAX_KB * DC_BK * 128 * 128 <= (1 << 24), "exact fp32 accumulator");
static_assert(DC_MAX_KB * DC_W_STAGE >= DC_TILE_I32, "the partial tile reuses the weight tiles");
static_assert(DC_B_BYTES == DC_W_STAGE, "a stage's fp16 activation tile replaces its int8 weight tile");
static_assert(DC_SUM_PER_THREAD * 4 * 32 * DC_CONV_WARPS == DC_TOK * DC_ROWS, "sum tile split over the converters");
static_assert(DC_XWARPS == 4 && DC_XCH == 4 && DC_TOK == 64, "activation widening: 4 warps x 4 rounds of 8 tokens x 4 chunks");

// 16 int8 (one 16-byte chunk) -> 8 words of fp16 pairs.
__device__ __forceinline__ void widen16(const uint4& x, uint32_t* h) {
  s8x4_to_f16x4(x.x, h[0], h[1]);
  s8x4_to_f16x4(x.y, h[2], h[3]);
  s8x4_to_f16x4(x.z, h[4], h[5]);
  s8x4_to_f16x4(x.w, h[6], h[7]);
}

// TMA loads of a CTA's whole K slice of weights (stages [kb0, kb0 + my) of row block rb) and of the
// matching activation tiles, one mbarrier per stage and operand.
__device__ __forceinline__ void issue_weights(const CUtensorMap* wmap, uint64_t* bar_w, uint8_t* wtiles, int kb0,
                                              int my, int rb) {
  for (int s = 0; s < my; ++s) {
    const uint32_t fb = smem_u32(&bar_w[s]);
    mbar_expect_tx(fb, DC_W_STAGE);
    tma_load_2d(smem_u32(wtiles + s * DC_W_STAGE), wmap, (kb0 + s) * DC_BK, rb * DC_ROWS, fb);
  }
}
__device__ __forceinline__ void issue_activations(const CUtensorMap* xmap, uint64_t* bar_x, uint8_t* xtiles,
                                                  int kb0, int my) {
  for (int s = 0; s < my; ++s) {
    const uint32_t fb = smem_u32(&bar_x[s]);
    mbar_expect_tx(fb, DC_X_STAGE);
    tma_load_2d(smem_u32(xtiles + s * DC_X_STAGE), xmap, (kb0 + s) * DC_BK, 0, fb);
  }
}
// With programmatic stream serialization this kernel may start while the
// kernel before it (the activation quantisation) still runs: everything that
// kernel writes -- the int8 codes and the scales -- is read only after
// pdl_wait, and every global write of this kernel follows that wait (through
// the activation tiles the whole computation waits for).

// The partial tile (shared memory) added into the row block's sum tile (global) by the bulk copy engine.
__device__ __forceinline__ void bulk_reduce_add_s32(int32_t* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.s32 [%0], [%1], %2;"
               ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Workspace of the decode engine: per row block the int32 sum tile [DC_TOK][DC_ROWS] and an arrival counter,
// both zero between calls.
struct DecWs {
  int32_t* sums;
  uint32_t* cnt;
};

template <int MODE>
__global__ void __launch_bounds__(DC_THREADS, 1)
dec_gemm_kernel(const GemmArgs a, const DecWs ws, const __grid_constant__ CUtensorMap wmap,
                const __grid_constant__ CUtensorMap xmap) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_w[DC_MAX_KB];      // weight tile of the stage landed
  __shared__ __align__(8) uint64_t bar_x[DC_MAX_KB];      // activation tile of the stage landed
  __shared__ __align__(8) uint64_t bar_ready[DC_MAX_KB];  // both operands of the stage widened
  __shared__ __align__(8) uint64_t bar_accf;
  __shared__ __align__(8) uint64_t bar_sum;              // the complete sums landed (last CTA)
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;
  __shared__ int s_last;
  // epilogue inputs of this row block, loaded by the converter warps before their first stage
  __shared__ float s_sw[DC_ROWS];
  __shared__ float s_bias[DC_ROWS];
  __shared__ int32_t s_qb[DC_ROWS];
  __shared__ float s_sx[DC_TOK];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int ct = tid - 32;      // converter thread index (warps 1..DC_CONV_WARPS)
  const int rank = blockIdx.x;  // split of K
  const int ksplit = gridDim.x;
  const int rb = blockIdx.y;    // 128-row weight block
  const int64_t M = a.R, N = a.N, K = a.K;
  const int nkb = static_cast<int>((K + DC_BK - 1) / DC_BK);
  const int kb0 = static_cast<int>(static_cast<int64_t>(nkb) * rank / ksplit);
  const int kb1 = static_cast<int>(static_cast<int64_t>(nkb) * (rank + 1) / ksplit);
  const int my = kb1 - kb0;

  // int8 weights [DC_MAX_KB][DC_ROWS][DC_BK], swizzled; once every weight stage sits in tensor memory the
  // same bytes hold the fp16 activation tiles [DC_MAX_KB][2][DC_TOK][64] (the MMA's B operand)
  // (offset from smem_raw, so that the compiler keeps every access below in the shared space)
  uint8_t* wtiles = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t btiles_base = smem_u32(wtiles);
  uint8_t* xtiles = wtiles + DC_MAX_KB * DC_W_STAGE;  // int8 activations [DC_MAX_KB][DC_TOK][DC_BK], swizzled
  int32_t* ptile = reinterpret_cast<int32_t*>(wtiles);  // int32 partial [DC_TOK][DC_ROWS], after the main loop

  if (tid == 0) {
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&xmap);
    s_abort = 0;
    s_last = 0;
    for (int s = 0; s < DC_MAX_KB; ++s) {
      mbar_init(smem_u32(&bar_w[s]), 1);
      mbar_init(smem_u32(&bar_x[s]), 1);
      mbar_init(smem_u32(&bar_ready[s]), DC_XWARPS);
    }
    mbar_init(smem_u32(&bar_accf), 1);
    mbar_init(smem_u32(&bar_sum), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (a.pack_known) issue_weights(&wmap, bar_w, wtiles, kb0, my, rb);
  }
  // The next kernel on the stream may be scheduled now: it waits for this grid before it touches memory
  // this grid uses, and its own prologue (a following contraction's weight stream) overlaps this one's tail.
  pdl_trigger();
  const PackedHeader* hdr = static_cast<const PackedHeader*>(a.packed);
  const bool run = hdr->magic == kPackMagic && hdr->version == kPackVersion && hdr->E == 1 && hdr->N == N &&
                   hdr->K == K && (hdr->flags & W8A8_PACK_GATE_UP) == 0u;
  if (tid == 0 && run && !a.pack_known) issue_weights(&wmap, bar_w, wtiles, kb0, my, rb);
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
  if (!run && tid == 0 && rank == 0 && rb == 0) set_status(a.status, W8A8_ERR_PACKED, 0u);

  if (run && warp == 0) {
    // activations: the previous grid writes them, so they are requested only after it has finished
    if (lane == 0) {
      pdl_wait();
      issue_activations(&xmap, bar_x, xtiles, kb0, my);
    }
    __syncwarp();
    // ------------------------------------------------------------- MMA issuer (whole warp)
    for (int i = 0; i < my; ++i) {
      if (!warp_wait(smem_u32(&bar_ready[i]), 0u, &s_abort, a.status, 12u)) break;
      tc_fence_after();
      const uint64_t bdesc0 = smem_desc_sw128(btiles_base + i * DC_B_BYTES);
#pragma unroll
      for (int kk = 0; kk < DC_BK / 16; ++kk)
        tc_mma_tmem_a(tmem_base + DC_D_COL, tmem_base + i * DC_A_COLS + 8u * kk,
                      bdesc0 + static_cast<uint64_t>((kk >> 2) * (DC_B_SUB >> 4) + 2 * (kk & 3)), kIdescDec,
                      (i > 0 || kk > 0) ? 1u : 0u);
    }
    tc_commit(smem_u32(&bar_accf));
  } else if (run) {
    // ------------------------------------------------ converters, then the partial tile
    const int q = warp & 3;            // TMEM lane quadrant
    const int part = (warp - 1) >> 2;  // K part of each weight stage (chunks DC_WCH*part..) / token part
    const int row = 32 * q + lane;     // weight row inside the block == TMEM lane
    if (MODE != EPI_ACC && ct < DC_ROWS) {  // epilogue inputs of the row block, while the weights stream
      const int64_t n = static_cast<int64_t>(rb) * DC_ROWS + ct;
      s_sw[ct] = n < N ? a.w_scale[n] : 0.0f;
      s_bias[ct] = (a.bias != nullptr && n < N) ? bf16_bits_to_f32(a.bias[n]) : 0.0f;
      s_qb[ct] = (a.qbias != nullptr && n < N) ? a.qbias[n] : 0;
    }
    // Weights: every stage of the slice is widened into its own tensor-memory A stage as it lands,
    // independent of the activations (which the previous grid may still be writing).
    bool ok = true;
    for (int i = 0; i < my && ok; ++i) {
      // every lane observes the completed load of stage i itself
      const int got = mbar_wait(smem_u32(&bar_w[i]), 0u, &s_abort, a.status, 13u) ? 1 : 0;
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      uint32_t v[8 * DC_WCH];
      const uint8_t* wst = wtiles + i * DC_W_STAGE + row * DC_BK;
#pragma unroll
      for (int c = 0; c < DC_WCH; ++c)
        widen16(*reinterpret_cast<const uint4*>(wst + (((DC_WCH * part + c) ^ (row & 7)) << 4)), &v[8 * c]);
      tmem_st32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + i * DC_A_COLS +
                    static_cast<uint32_t>(8 * DC_WCH * part),
                v);
    }
    tmem_wait_st();
    tc_fence_before();
    // every converter is done reading the int8 weight tiles: their bytes now take the fp16 activations
    asm volatile("bar.sync 1, %0;" ::"n"(32 * DC_CONV_WARPS) : "memory");
    if (MODE != EPI_ACC && ct >= DC_ROWS && ct < DC_ROWS + DC_TOK) {  // token scales: the previous grid's output
      pdl_wait();
      s_sx[ct - DC_ROWS] = ct - DC_ROWS < M ? (a.x_scale != nullptr ? a.x_scale[ct - DC_ROWS] : 1.0f) : 0.0f;
    }
    // Activations: group g of DC_XWARPS warps widens stages g, g + DC_XGROUPS, ...  A warp instruction
    // covers 8 tokens x 4 chunks of 16 int8: lane l takes token t0 + 16 jj (t0 = 8 (gw / 2) + l / 4) and
    // source chunk cs = l % 4 + 4 ((t0 % 2) ^ (gw % 2)), so that every 8 consecutive lanes (2 tokens)
    // read the 8 distinct 16-byte positions of a 128-byte row and write 8 distinct positions: no bank
    // conflict on the loads or the stores.  Its 32 fp16 bytes are chunks 2 (cs % 4) and 2 (cs % 4) + 1 of
    // the token's row in 64-K sub-tile cs / 4.
    const int xg = (warp - 1) / DC_XWARPS, gw = (warp - 1) % DC_XWARPS;
    const int sw = lane >> 2;  // t & 7 for every token this lane takes
    const int cs = (lane & 3) + 4 * ((sw & 1) ^ (gw & 1));
    const int t0 = 8 * (gw >> 1) + sw;
    const int x_off = t0 * DC_BK + ((cs ^ sw) << 4);
    const int b_off = (cs >> 2) * DC_B_SUB + t0 * 128;
    const int lo_pos = ((2 * (cs & 3)) ^ sw) << 4, hi_pos = ((2 * (cs & 3) + 1) ^ sw) << 4;
    for (int i = xg; i < my && ok; i += DC_XGROUPS) {
      const int got = mbar_wait(smem_u32(&bar_x[i]), 0u, &s_abort, a.status, 16u) ? 1 : 0;
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      uint8_t* bt = wtiles + i * DC_B_BYTES;
      const uint8_t* xst = xtiles + i * DC_X_STAGE;
#pragma unroll
      for (int jj = 0; jj < DC_XCH; ++jj) {  // tokens t0 + 16 jj
        uint32_t hh[8];
        widen16(*reinterpret_cast<const uint4*>(xst + x_off + 16 * DC_BK * jj), hh);
        uint8_t* brow = bt + b_off + 16 * 128 * jj;
        *reinterpret_cast<uint4*>(brow + lo_pos) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
        *reinterpret_cast<uint4*>(brow + hi_pos) = make_uint4(hh[4], hh[5], hh[6], hh[7]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_ready[i]));
    }
    // exact partial -> shared memory, token-major; this warp drains tokens
    // [DC_TPW*part, DC_TPW*(part+1)).  Once the last MMA has completed, the activation tiles (in the
    // weight tiles' bytes) are free to hold the partial.
    int got = 1;
    if (my > 0) {
      if (lane == 0) got = mbar_wait(smem_u32(&bar_accf), 0u, &s_abort, a.status, 14u) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
    }
    if (my > 0 && got && ok) {
      tc_fence_after();
      uint32_t d[DC_TPW];
      tmem_ld32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + DC_D_COL + static_cast<uint32_t>(DC_TPW * part),
                d);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < DC_TPW; ++c)
        ptile[(DC_TPW * part + c) * DC_ROWS + row] = __float2int_rn(__uint_as_float(d[c]));
    } else {
#pragma unroll 8
      for (int c = 0; c < DC_TPW; ++c) ptile[(DC_TPW * part + c) * DC_ROWS + row] = 0;
    }
    tc_fence_before();
    // ---- split-K: the partial tile joins the row block's sums in global memory; the last CTA to arrive
    // holds the complete sums
    if (ksplit > 1) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the bulk copy reads ptile
      asm volatile("bar.sync 1, %0;" ::"n"(32 * DC_CONV_WARPS) : "memory");
      if (ct == 0) {
        if (!s_abort) {
          // the first M token rows of the partial: the rest stays zero
          bulk_reduce_add_s32(ws.sums + static_cast<int64_t>(rb) * (DC_TOK * DC_ROWS), smem_u32(ptile),
                              static_cast<uint32_t>(M) * DC_ROWS * 4);
          // arrival: release of the sums added above; the last to arrive acquires everyone else's
          asm volatile("fence.acq_rel.gpu;" ::: "memory");
          const uint32_t prev = atomicAdd(&ws.cnt[rb], 1u);
          if (prev == static_cast<uint32_t>(ksplit - 1)) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            asm volatile("fence.proxy.async.global;" ::: "memory");
            s_last = 1;
            ws.cnt[rb] = 0u;  // for the next call
          }
        }
      }
    } else if (ct == 0) {
      s_last = 1;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * DC_CONV_WARPS) : "memory");

    // ---- epilogue of the complete sums: thread ct takes (token, 4 rows) pieces ct, ct + 256, ...
    if (s_last && !s_abort) {
      int4* gsum = reinterpret_cast<int4*>(ws.sums + static_cast<int64_t>(rb) * (DC_TOK * DC_ROWS));
      const int4* lsum = reinterpret_cast<const int4*>(ptile);
      if (ksplit > 1) {  // the complete sums (first M token rows) into the partial tile's bytes, one bulk copy
        if (ct == 0) {
          const uint32_t bytes = static_cast<uint32_t>(M) * DC_ROWS * 4;
          mbar_expect_tx(smem_u32(&bar_sum), bytes);
          asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                       ::"r"(smem_u32(ptile)), "l"(gsum), "r"(bytes), "r"(smem_u32(&bar_sum))
                       : "memory");
        }
      }
      int got_sum = 1;  // one lane waits, the warp proceeds converged
      if (ksplit > 1 && lane == 0) got_sum = mbar_wait(smem_u32(&bar_sum), 0u, &s_abort, a.status, 17u) ? 1 : 0;
      const bool have = __shfl_sync(0xffffffffu, got_sum, 0) != 0;
      // every piece of this thread covers the same 4 rows r0..r0+3: their epilogue inputs once, in registers
      const int r0 = (ct & 31) * 4;
      const int64_t n0 = static_cast<int64_t>(rb) * DC_ROWS + r0;
      float sw4[4], bias4[4];
      int32_t qb4[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        sw4[r] = s_sw[r0 + r];
        bias4[r] = s_bias[r0 + r];
        qb4[r] = s_qb[r0 + r];
      }
      const bool has_qb = a.qbias != nullptr, has_bias = a.bias != nullptr;
      const bool vec = n0 + 4 <= N &&
                       (N % 4 == 0 || M == 1) && (reinterpret_cast<uintptr_t>(a.out) & (MODE == EPI_ACC ? 15u : 7u)) == 0u;
      // Compact loops, not unrolled: this code runs once per row block and call, on whichever SM arrives
      // last, so its instruction fetch (not its arithmetic) is what the unrolled form would pay for.
      if (have && n0 < N) {
#pragma unroll 1
        for (int t = ct >> 5; t < M; t += 32 * DC_CONV_WARPS / 32) {  // pieces ct + 256 u: token (ct + 256 u) / 32
          const int4 v = lsum[t * 32 + (ct & 31)];
          const int sum[4] = {v.x, v.y, v.z, v.w};
          if constexpr (MODE == EPI_ACC) {
            int32_t* dst = static_cast<int32_t*>(a.out) + t * N + n0;
            if (vec) {
              __stcg(reinterpret_cast<int4*>(dst), v);
            } else {
              for (int r = 0; r < 4; ++r)
                if (n0 + r < N) dst[r] = sum[r];
            }
          } else {
            const float sx = s_sx[t];
            float fv[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              fv[r] = has_qb ? dequant_q(sum[r], qb4[r], sx, sw4[r]) : dequant(sum[r], sx, sw4[r]);
              fv[r] = has_bias ? __fadd_rn(fv[r], bias4[r]) : fv[r];
            }
            const uint2 h = make_uint2(f32x2_to_bf16x2_bits(fv[0], fv[1]), f32x2_to_bf16x2_bits(fv[2], fv[3]));
            uint16_t* dst = static_cast<uint16_t*>(a.out) + t * N + n0;
            if (vec) {
              __stcg(reinterpret_cast<uint2*>(dst), h);
            } else {
              const uint16_t hs[4] = {static_cast<uint16_t>(h.x), static_cast<uint16_t>(h.x >> 16),
                                      static_cast<uint16_t>(h.y), static_cast<uint16_t>(h.y >> 16)};
              for (int r = 0; r < 4; ++r)
                if (n0 + r < N) dst[r] = hs[r];
            }
          }
        }
      }
      if (ksplit > 1 && have) {  // the sum tile's first M token rows back to zero for the next call
#pragma unroll 1
        for (int task = ct; task < M * (DC_ROWS / 4); task += 32 * DC_CONV_WARPS) __stcg(gsum + task, make_int4(0, 0, 0, 0));
        asm volatile("fence.proxy.async.global;" ::: "memory");  // the next call's bulk reduce-adds see zeros
      }
    }
  }

  if (tid == 0 && ((!run && a.pack_known) || s_abort)) {
    // loads issued for a buffer that failed the header check, or an aborted CTA: let the copies land
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 20000000ull) {
    }
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(DC_TMEM_COLS)
                 : "memory");
  }
}

// Weight and activation tiles: more than half of the SM's shared memory, which keeps a CTA (it holds all
// 512 tensor-memory columns) alone on its SM (a second one would stall in its allocation).
constexpr size_t kDecSmem = static_cast<size_t>(DC_MAX_KB) * (DC_W_STAGE + DC_X_STAGE) + 1024;
static_assert(kDecSmem > 114 * 1024 && kDecSmem <= 227 * 1024, "shared memory budget");

void dec_set_attributes() {
  for (auto k : {dec_gemm_kernel<EPI_BF16>, dec_gemm_kernel<EPI_ACC>}) {
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kDecSmem));
  }
}

template <int MODE>
cudaError_t launch_dec_mode(const GemmArgs& a, const DecWs& ws, const CUtensorMap& wmap, const CUtensorMap& xmap,
                            const DecPlan& plan, int nblk, cudaStream_t stream) {
  dec_set_attributes();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.ksplit), static_cast<unsigned>(nblk), 1);
  cfg.blockDim = dim3(DC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = kDecSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  // may start before the previous kernel on the stream ends, if that kernel allows it (the activation
  // quantisation and this kernel do); the kernel waits for it before reading what it wrote
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dec_gemm_kernel<MODE>, a, ws, wmap, xmap);
}

}  // namespace

size_t dec_ws_bytes(int64_t N) {
  const int64_t nblk = (N + DC_ROWS - 1) / DC_ROWS;
  return align_up(static_cast<uint64_t>(nblk) * DC_TILE_I32, 256) + align_up(static_cast<uint64_t>(nblk) * 4, 256);
}

// K split for the decode engine: every CTA covers at most DC_MAX_KB stages of K, all CTAs fit in one wave
// (one per SM) and at most DC_MAX_KSPLIT partials meet in one sum tile.  Among the splits that allow: the
// fewest stages per CTA, then the fewest CTAs.  ksplit 0 = shape unsuited.
DecPlan dec_plan(int64_t M, int64_t N, int64_t K, int num_sms) {
  DecPlan best;
  if (M < 1 || M > DC_TOK || N < 1 || K < 1) return best;
  const int64_t nkb = (K + DC_BK - 1) / DC_BK;
  const int64_t nblk = (N + DC_ROWS - 1) / DC_ROWS;
  const int64_t max_split = std::min<int64_t>(std::min<int64_t>(nkb, num_sms / nblk), DC_MAX_KSPLIT);
  if (max_split < 1) return best;
  const int64_t stages = (nkb + max_split - 1) / max_split;
  if (stages > DC_MAX_KB) return best;
  best.ksplit = static_cast<int>((nkb + stages - 1) / stages);  // the fewest splits with that many stages
  return best;
}

cudaError_t launch_dec_gemm(const GemmArgs& a, const DecPlan& plan, void* dec_ws, cudaStream_t stream) {
  if (a.R == 0) return cudaSuccess;
  const int64_t nkb = (a.K + DC_BK - 1) / DC_BK;
  if (plan.ksplit < 1 || plan.ksplit > nkb || (nkb + plan.ksplit - 1) / plan.ksplit > DC_MAX_KB)
    return cudaErrorInvalidValue;
  const int nblk = static_cast<int>((a.N + DC_ROWS - 1) / DC_ROWS);
  DecWs ws;
  uint8_t* b = static_cast<uint8_t*>(dec_ws);
  ws.sums = reinterpret_cast<int32_t*>(b);
  ws.cnt = reinterpret_cast<uint32_t*>(b + align_up(static_cast<uint64_t>(nblk) * DC_TILE_I32, 256));
  // tensor maps of the int8 weight payload [N, K] and the int8 activations [R, K]; rows past the ends read as zero
  CUtensorMap wmap, xmap;
  const uint8_t* w_i8 = static_cast<const uint8_t*>(a.packed) + pack_layout(1, a.N, a.K, 0).i8_offset;
  if (!encode_map_2d(&wmap, w_i8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.N, a.K, DC_BK, DC_ROWS,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_map_2d(&xmap, a.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.R, a.K, DC_BK, DC_TOK,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (a.mode == EPI_ACC) return launch_dec_mode<EPI_ACC>(a, ws, wmap, xmap, plan, nblk, stream);
  return launch_dec_mode<EPI_BF16>(a, ws, wmap, xmap, plan, nblk, stream);
}

}  // namespace w8a8
