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
// writing.  Once that kernel has finished, the MMA thread requests the
// slice's activation tiles (64 tokens x 128 bytes per stage, TMA, 128-byte
// swizzled, one mbarrier per stage); the converters widen each into a
// 128-byte-swizzled K-major FP16 tile in the bytes the int8 weight tiles
// occupied (the B operand), and each stage's MMAs follow as soon as its tile
// is ready.  After the activations arrive, only their widening, the MMAs and the
// reduction remain.  The MMA is M = 128 weight rows x N = 64 tokens x K = 16
// into an FP32 TMEM accumulator; the CTA's K slice is at most 896, so the
// accumulator holds an exact integer (|partial| <= 896 * 128^2 < 2^24).
//
// Split-K reduction, which waits on no other CTA's progress beyond the
// cluster barrier: the K splits of a row block form clusters of up to eight
// CTAs; after a cluster barrier each CTA sums, for its share of the tokens
// (64 / cluster size), the cluster's partial tiles straight out of the other
// CTAs' shared memory (distributed shared memory), every remote load of a
// thread in flight at once.  Only when a row block has more K splits than one
// cluster holds (clusters of at least four then) does a second step follow:
// each CTA stores its share in its own workspace slot and bumps the arrival
// counter of that share (release); the CTA that arrives last adds the other
// clusters' slots.  The CTA holding the complete sums applies
// the dequant epilogue and writes BF16 (or the INT32 sums) and resets the
// counter.  Integer addition is exact in any order.
//
// Warps: 0 TMEM owner, TMA producer and MMA issuer (lane 0); 1-8 converters (warp w owns
// TMEM lanes 32*(w%4).. and K part / token part (w-1)/4).  All waits are
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
constexpr uint32_t DC_B_SUB = DC_TOK * 128;    // one 64-K fp16 sub-tile (8 KB)
constexpr uint32_t DC_B_BYTES = 2 * DC_B_SUB;  // 128 K of fp16 activations
#ifndef DC_CONV_WARPS_OVERRIDE
constexpr int DC_CONV_WARPS = 8;
#else
constexpr int DC_CONV_WARPS = DC_CONV_WARPS_OVERRIDE;
#endif
constexpr int DC_THREADS = 32 * (1 + DC_CONV_WARPS);
constexpr int DC_NPART = DC_CONV_WARPS / 4;          // converter warps per TMEM lane quadrant
constexpr int DC_WCH = 8 / DC_NPART;                 // 16-byte weight chunks per lane per stage
constexpr int DC_XCH = 512 / (32 * DC_CONV_WARPS);   // 16-byte activation chunks per thread per stage
constexpr int DC_TPW = DC_TOK / DC_NPART;            // accumulator columns (tokens) drained per warp
static_assert(DC_CONV_WARPS == 8 || DC_CONV_WARPS == 16, "8 or 16 converter warps");
constexpr uint32_t DC_TMEM_COLS = 512;
constexpr uint32_t DC_A_COLS = DC_BK / 2;  // 64 columns of fp16 pairs per A stage
constexpr int DC_MAX_KB = 7;               // stages per CTA: 896 of K
constexpr uint32_t DC_D_COL = DC_MAX_KB * DC_A_COLS;  // every A stage resident; accumulator at [448, 512)
constexpr uint32_t DC_W_STAGE = DC_ROWS * DC_BK;  // int8 weight tile (16 KB)
constexpr uint32_t DC_X_STAGE = DC_TOK * DC_BK;   // int8 activation tile (8 KB)
constexpr uint32_t DC_TILE_I32 = DC_TOK * DC_ROWS * 4;  // int32 partial tile (32 KB)
constexpr int DC_MAX_KSPLIT = 16;
constexpr int DC_CLUSTER = 8;       // most CTAs per cluster (consecutive K splits)
constexpr int DC_MIN_SLOT_CLUSTER = 4;  // clusters that meet through workspace slots hold at least 4 CTAs
constexpr int DC_SLOT_I32 = DC_TOK / DC_MIN_SLOT_CLUSTER * DC_ROWS;  // int32 per workspace slot
constexpr uint32_t kIdescDec = (1u << 4) | (uint32_t(DC_TOK >> 3) << 17) | (uint32_t(DC_ROWS >> 4) << 24);
static_assert(DC_B_BYTES % 1024 == 0 && DC_W_STAGE % 1024 == 0 && DC_X_STAGE % 1024 == 0, "1024-byte aligned tiles");
static_assert(DC_D_COL + DC_TOK <= DC_TMEM_COLS, "tensor memory budget");
static_assert(DC_MAX_KB * DC_BK * 127 * 127 < (1 << 24), "exact fp32 accumulator");
static_assert(DC_MAX_KB * DC_W_STAGE >= DC_TILE_I32, "the partial tile reuses the weight tiles");
static_assert(DC_B_BYTES == DC_W_STAGE, "a stage's fp16 activation tile replaces its int8 weight tile");

// 32 lanes x N consecutive 32-bit TMEM columns (N = 16 or 32).
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&v)[N]) {
  if constexpr (N == 32) {
    tmem_st32(taddr, v);
  } else {
    static_assert(N == 16, "16 or 32 columns");
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
  }
}
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&v)[N]) {
  if constexpr (N == 32) {
    tmem_ld32(taddr, v);
  } else {
    static_assert(N == 16, "16 or 32 columns");
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
  }
}

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

// Workspace of the decode engine: per row block and K split a slot for the
// cluster-summed int32 piece [tokens of the CTA][DC_ROWS], and per row block
// eight arrival counters (one per cluster rank), zero between calls.
struct DecWs {
  int32_t* slots;
  uint32_t* cnt;
};

__device__ __forceinline__ void cluster_sync() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Remote load without a memory clobber, so that a thread's loads of several CTAs' tiles are all in
// flight before the first result is used (volatile keeps them after the cluster barrier before them).
__device__ __forceinline__ int4 ld_dsmem_v4(uint32_t addr) {
  int4 v;
  asm volatile("ld.shared::cluster.v4.s32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

template <int MODE>
__global__ void __launch_bounds__(DC_THREADS, 1)
dec_gemm_kernel(const GemmArgs a, const DecWs ws, const __grid_constant__ CUtensorMap wmap,
                const __grid_constant__ CUtensorMap xmap) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_w[DC_MAX_KB];      // weight tile of the stage landed
  __shared__ __align__(8) uint64_t bar_x[DC_MAX_KB];      // activation tile of the stage landed
  __shared__ __align__(8) uint64_t bar_ready[DC_MAX_KB];  // both operands of the stage widened
  __shared__ __align__(8) uint64_t bar_accf;
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
  uint8_t* wtiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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
      mbar_init(smem_u32(&bar_ready[s]), DC_CONV_WARPS);
    }
    mbar_init(smem_u32(&bar_accf), 1);
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
    if (lane == 0) {
      // activations: the previous grid writes them, so they are requested only after it has finished (the
      // MMAs need them first of all, so their issuer requests them)
      pdl_wait();
      issue_activations(&xmap, bar_x, xtiles, kb0, my);
      // ----------------------------------------------------------- MMA issuer
      for (int i = 0; i < my && !s_abort; ++i) {
        if (!mbar_wait(smem_u32(&bar_ready[i]), 0u, &s_abort, a.status, 12u)) break;
        tc_fence_after();
        const uint32_t bsub0 = btiles_base + i * DC_B_BYTES;
#pragma unroll
        for (int kk = 0; kk < DC_BK / 16; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(bsub0 + (kk >> 2) * DC_B_SUB) + 2u * (kk & 3);
          tc_mma_tmem_a(tmem_base + DC_D_COL, tmem_base + i * DC_A_COLS + 8u * kk, bdesc, kIdescDec,
                        (i > 0 || kk > 0) ? 1u : 0u);
        }
      }
      tc_commit(smem_u32(&bar_accf));
    }
  } else if (run) {
    // ------------------------------------------------ converters, then the partial tile
    const int q = warp & 3;           // TMEM lane quadrant
    const int part = (warp - 1) >> 2;  // K part of each stage (chunks DC_WCH*part..) / token part
    const int row = 32 * q + lane;    // weight row inside the block == TMEM lane
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
      tmem_st_cols<8 * DC_WCH>(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + i * DC_A_COLS +
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
    for (int i = 0; i < my && ok; ++i) {
      const int got = mbar_wait(smem_u32(&bar_x[i]), 0u, &s_abort, a.status, 16u) ? 1 : 0;
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      uint8_t* bt = wtiles + i * DC_B_BYTES;
      const uint8_t* xst = xtiles + i * DC_X_STAGE;
#pragma unroll
      for (int jj = 0; jj < DC_XCH; ++jj) {
        const int p = ct + 32 * DC_CONV_WARPS * jj;
        const int t = p >> 3, c = p & 7;
        uint32_t hh[8];
        widen16(*reinterpret_cast<const uint4*>(xst + t * DC_BK + ((c ^ (t & 7)) << 4)), hh);
        uint8_t* brow = bt + (c >> 2) * DC_B_SUB + t * 128;
        const int cc = (c & 3) * 2;
        // The eight threads of a token write 16-byte chunks cc and cc+1 of its row in both 64-K sub-tiles
        // (which sit on the same banks); threads c >= 4 store the odd chunk first, so each store
        // instruction covers all eight chunk positions of the row: no bank conflict.
        const int first = cc + (c >> 2), second = cc + 1 - (c >> 2);
        const uint4 lo = make_uint4(hh[0], hh[1], hh[2], hh[3]), hi = make_uint4(hh[4], hh[5], hh[6], hh[7]);
        *reinterpret_cast<uint4*>(brow + ((first ^ (t & 7)) << 4)) = (c >> 2) ? hi : lo;
        *reinterpret_cast<uint4*>(brow + ((second ^ (t & 7)) << 4)) = (c >> 2) ? lo : hi;
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
      tmem_ld_cols<DC_TPW>(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + DC_D_COL +
                               static_cast<uint32_t>(DC_TPW * part),
                           d);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < DC_TPW; ++c)
        ptile[(DC_TPW * part + c) * DC_ROWS + row] = __float2int_rn(__uint_as_float(d[c]));
    } else {
#pragma unroll 8
      for (int c = 0; c < DC_TPW; ++c) ptile[(DC_TPW * part + c) * DC_ROWS + row] = 0;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
  }
  __syncwarp();
  __syncthreads();

  // ---- split-K, step 1: the CTAs of a cluster (consecutive K splits of the row block) sum their partial
  // tiles through distributed shared memory; CTA cr of the cluster takes tokens [cr*tq, (cr+1)*tq)
  uint32_t csize, cr;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(csize));
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(cr));
  const int tq = DC_TOK / static_cast<int>(csize);
  const int ntask = tq * (DC_ROWS / 4);  // (token, 4 rows) pieces of this CTA
  constexpr int kPer = (DC_TOK * DC_ROWS / 4 + DC_THREADS - 1) / DC_THREADS;
  cluster_sync();  // every partial tile of the cluster is in place
  int4 sums[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    sums[u] = make_int4(0, 0, 0, 0);
    const int task = tid + DC_THREADS * u;
    if (task >= ntask) continue;
    const uint32_t off = static_cast<uint32_t>(((static_cast<int>(cr) * tq + (task >> 5)) * DC_ROWS + (task & 31) * 4) * 4);
    int4 v[DC_CLUSTER];  // all remote loads in flight together
#pragma unroll
    for (int c = 0; c < DC_CLUSTER; ++c)
      v[c] = c < static_cast<int>(csize) ? ld_dsmem_v4(mapa_shared(smem_u32(ptile), static_cast<uint32_t>(c)) + off)
                                         : make_int4(0, 0, 0, 0);
#pragma unroll
    for (int c = 0; c < DC_CLUSTER; ++c) {
      sums[u].x += v[c].x;
      sums[u].y += v[c].y;
      sums[u].z += v[c].z;
      sums[u].w += v[c].w;
    }
  }
  cluster_sync();  // no CTA reuses or releases its tile while the others still read it

  // ---- step 2: the clusters of the row block meet through the workspace; each CTA stores its sums in its
  // own slot and arrives (release); the last to arrive for these tokens adds the others' slots
  const int ncl = ksplit / static_cast<int>(csize);
  const int cg = rank / static_cast<int>(csize);
  if (ncl > 1) {
    int4* my_slot = reinterpret_cast<int4*>(ws.slots) + (static_cast<int64_t>(rb) * ksplit + rank) * (DC_SLOT_I32 / 4);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int task = tid + DC_THREADS * u;
      if (task < ntask) __stcg(my_slot + task, sums[u]);
    }
    __syncthreads();
    if (tid == 0) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      const uint32_t prev = atomicAdd(&ws.cnt[rb * DC_CLUSTER + cr], 1u);
      if (prev == static_cast<uint32_t>(ncl - 1)) {
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        s_last = 1;
        ws.cnt[rb * DC_CLUSTER + cr] = 0u;  // for the next call
      }
    }
  } else if (tid == 0) {
    s_last = 1;
  }
  __syncthreads();

  // ---- the CTA holding the complete sums adds the other clusters' slots
  if (ncl > 1 && s_last) {
    for (int g = 0; g < ncl; ++g) {
      if (g == cg) continue;
      const int4* slot = reinterpret_cast<const int4*>(ws.slots) +
                         (static_cast<int64_t>(rb) * ksplit + g * static_cast<int>(csize) + cr) * (DC_SLOT_I32 / 4);
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int task = tid + DC_THREADS * u;
        if (task >= ntask) continue;
        const int4 v = __ldcg(slot + task);
        sums[u].x += v.x;
        sums[u].y += v.y;
        sums[u].z += v.z;
        sums[u].w += v.w;
      }
    }
  }

  // ---- epilogue of this CTA's tokens over the complete sums
  if (s_last && run && !s_abort) {
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int task = tid + DC_THREADS * u;
      const int t = static_cast<int>(cr) * tq + (task >> 5);
      const int64_t n0 = static_cast<int64_t>(rb) * DC_ROWS + (task & 31) * 4;
      if (task >= ntask || t >= M || n0 >= N) continue;
      const int sum[4] = {sums[u].x, sums[u].y, sums[u].z, sums[u].w};
      if constexpr (MODE == EPI_ACC) {
        int32_t* dst = static_cast<int32_t*>(a.out) + t * N + n0;
        if (((reinterpret_cast<uintptr_t>(dst) & 15u) == 0u) && n0 + 4 <= N) {
          *reinterpret_cast<int4*>(dst) = sums[u];
        } else {
#pragma unroll
          for (int r = 0; r < 4; ++r)
            if (n0 + r < N) dst[r] = sum[r];
        }
      } else {
        const int r0 = (task & 31) * 4;
        const float sx = s_sx[t];
        uint16_t o[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          float fv = a.qbias != nullptr ? dequant_q(sum[r], s_qb[r0 + r], sx, s_sw[r0 + r])
                                        : dequant(sum[r], sx, s_sw[r0 + r]);
          if (a.bias) fv = __fadd_rn(fv, s_bias[r0 + r]);
          o[r] = f32_to_bf16_bits(fv);
        }
        uint16_t* dst = static_cast<uint16_t*>(a.out) + t * N + n0;
        if (((reinterpret_cast<uintptr_t>(dst) & 7u) == 0u) && n0 + 4 <= N) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(o[0] | (uint32_t(o[1]) << 16), o[2] | (uint32_t(o[3]) << 16));
        } else {
#pragma unroll
          for (int r = 0; r < 4; ++r)
            if (n0 + r < N) dst[r] = o[r];
        }
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

// Clusters of `cs` decode CTAs that can be resident at once on the current device.
int dec_resident_clusters(int cs) {
  static std::mutex mu;
  static int cache[64][DC_CLUSTER + 1] = {};
  int dev = 0;
  if (cs < 1 || cs > DC_CLUSTER || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev][cs] == 0) {
    dec_set_attributes();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
    cfg.blockDim = dim3(DC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = kDecSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, dec_gemm_kernel<EPI_BF16>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[dev][cs] = n;
  }
  return cache[dev][cs];
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
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(plan.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start before the previous kernel on the stream ends, if that kernel allows it (the activation
  // quantisation and this kernel do); the kernel waits for it before reading what it wrote
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, dec_gemm_kernel<MODE>, a, ws, wmap, xmap);
}

}  // namespace

size_t dec_ws_bytes(int64_t N) {
  const int64_t nblk = (N + DC_ROWS - 1) / DC_ROWS;
  return align_up(static_cast<uint64_t>(nblk) * DC_MAX_KSPLIT * DC_SLOT_I32 * 4, 256) +
         align_up(static_cast<uint64_t>(nblk) * DC_CLUSTER * 4, 256);
}

// K split and cluster size for the decode engine.  Every CTA covers at most DC_MAX_KB stages of K and all
// clusters fit in one wave.  Splits 1, 2, 4 and 8 form one cluster per row block (the reduction is one
// distributed-shared-memory step); 16 splits form two clusters of 8 that meet through workspace slots.
// When clusters of 8 cannot all be resident, 8 or 16 splits fall back to clusters of 4.  Among the
// candidates: the fewest stages per CTA, then the fewest clusters per row block.  ksplit 0 = shape
// unsuited.
DecPlan dec_plan(int64_t M, int64_t N, int64_t K, int num_sms) {
  (void)num_sms;
  DecPlan best;
  if (M < 1 || M > DC_TOK) return best;
  const int64_t nkb = (K + DC_BK - 1) / DC_BK;
  const int64_t nblk = (N + DC_ROWS - 1) / DC_ROWS;
  int64_t best_stages = DC_MAX_KB + 1;
  int best_ncl = 1 << 30;
  static const int kSplits[] = {1, 2, 4, 8, 16};
  for (int ks : kSplits) {
    if (ks > nkb) break;
    const int64_t stages = (nkb + ks - 1) / ks;
    for (int cs : {8, 4, 2, 1}) {
      if (cs > ks || ks % cs != 0) continue;
      if (ks > cs && cs < DC_MIN_SLOT_CLUSTER) continue;
      if (nblk * (ks / cs) > dec_resident_clusters(cs)) continue;
      const int ncl = ks / cs;
      if (stages < best_stages || (stages == best_stages && ncl < best_ncl)) {
        best_stages = stages;
        best_ncl = ncl;
        best.ksplit = ks;
        best.cluster = cs;
      }
      break;  // the largest cluster that fits for this split
    }
  }
  if (best_stages > DC_MAX_KB) best = DecPlan{};
  return best;
}

cudaError_t launch_dec_gemm(const GemmArgs& a, const DecPlan& plan, void* dec_ws, cudaStream_t stream) {
  if (a.R == 0) return cudaSuccess;
  const int ks = plan.ksplit, cs = plan.cluster;
  if (ks < 1 || ks > DC_MAX_KSPLIT || cs < 1 || cs > DC_CLUSTER || (cs & (cs - 1)) != 0 || ks % cs != 0 ||
      (ks > cs && cs < DC_MIN_SLOT_CLUSTER))
    return cudaErrorInvalidValue;
  const int nblk = static_cast<int>((a.N + DC_ROWS - 1) / DC_ROWS);
  DecWs ws;
  uint8_t* b = static_cast<uint8_t*>(dec_ws);
  ws.slots = reinterpret_cast<int32_t*>(b);
  ws.cnt = reinterpret_cast<uint32_t*>(b + align_up(static_cast<uint64_t>(nblk) * DC_MAX_KSPLIT * DC_SLOT_I32 * 4, 256));
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
