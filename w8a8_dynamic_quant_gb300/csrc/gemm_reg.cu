// gemm_reg.cu -- exact INT8 contraction on the warp-level tensor-core path.
//
// Page "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子":
//   §二 npu_quant_matmul: acc = q x W^T in INT32, then * x_scale[m] * w_scale[n]
//       (+ bias) -> BF16; §四 INT8 x1/x2, FLOAT32 per-token scale, BF16 out;
//   §三 npu_grouped_matmul over group_list (rows per expert, may be 0) and the
//       W13 -> SwiGLU step of the expert FFN.
//
// Engine.  Every int8 is exactly representable as an fp16 integer and every
// product |a*b| <= 2^14 is exact in fp32, so the contraction runs on
// mma.sync m16n8k16 f16 with fp32 accumulators that are drained into int32
// registers after at most 1024 products (|partial| <= 1024 * 2^14 = 2^24,
// every partial sum an exactly representable integer).  The int8 tiles are
// staged in shared memory by cp.async (4-stage ring, XOR-swizzled 16-byte
// chunks), loaded with ldmatrix in the int8 fragment layout and widened to
// fp16 in registers; both operands use the same k permutation inside each
// 32-wide k block, so the sum is unchanged.
//
// Orientation.  The weight rows are the MMA "M" side (16-row fragments) and
// the tokens the "N" side (8-column fragments): decode shapes with few tokens
// fill the 16-row side from the weights.  A CTA tile is 128 weight rows x
// BMT tokens (BMT = 8, 32 or 64, chosen from the rows per group).
//
// Scheduling.  Persistent CTAs walk a flat tile list (expert, n-block,
// m-block, k-split) built in shared memory from the device group_list (block
// prefix scans); empty experts own no tiles.  Split-K partials are summed with
// int32 atomics into a zeroed workspace; the last CTA of an output tile (an
// arrival counter) finishes the epilogue and zeroes the partials again.
#include "kernels.cuh"

namespace w8a8 {

namespace {

constexpr int BK = 64;       // K bytes per pipeline stage
// Ring depth and CTAs per SM of the 8-token tile (MoE decode); measured on GB300 at 8 x 2, against
// 4 x 2 (70 % of HBM on the MoE decode layer) and 6..20 stages with 1..4 CTAs per SM.
#ifndef REG_STAGES_V8
#define REG_STAGES_V8 8
#endif
#ifndef REG_GRID_V8
#define REG_GRID_V8 2
#endif
constexpr int STAGES = 4;  // pipeline depth of the 32- and 64-token tiles
constexpr int kMaxE = 1024;

template <int WM, int WN, int WARPS_W, int WARPS_T>
struct Tile {
  static constexpr int kThreads = 32 * WARPS_W * WARPS_T;
  static constexpr int BNW = 16 * WM * WARPS_W;  // weight rows per CTA tile
  static constexpr int BMT = 8 * WN * WARPS_T;   // tokens per CTA tile
  static constexpr int kStageW = BNW * BK;
  static constexpr int kStageT = BMT * BK;
  static constexpr int kStageBytes = kStageW + kStageT;
  // the 8-token tile streams weights for decode-sized groups: a deeper ring keeps more bytes in flight
  static constexpr int kStages = (WM == 1 && WN == 1) ? REG_STAGES_V8 : STAGES;
  static constexpr int kPipeBytes = kStages * kStageBytes;
  static constexpr int kEpiStride = BNW + 4;     // int32 words per staged token row
  static constexpr int kEpiBytes = BMT * kEpiStride * 4;
  static constexpr int kSmem = kPipeBytes > kEpiBytes ? kPipeBytes : kEpiBytes;
};

__device__ __forceinline__ int swz(int row, int ch) { return row * BK + ((ch ^ ((row >> 1) & 3)) << 4); }

template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int& total, int* s_warp) {
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[w] = x;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) {
    const int s = s_warp[i];
    if (i < w) before += s;
    tot += s;
  }
  __syncthreads();
  total = tot;
  return before + x - v;
}

__device__ __forceinline__ float bf16_round(float v) { return bf16_bits_to_f32(f32_to_bf16_bits(v)); }

template <int WM, int WN, int WARPS_W, int WARPS_T, int MODE>
__global__ void __launch_bounds__(32 * WARPS_W * WARPS_T)
reg_gemm_kernel(const GemmArgs a, const int ksplit) {
  using T = Tile<WM, WN, WARPS_W, WARPS_T>;
  constexpr int NT = T::kThreads;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_tile_prefix[kMaxE + 1];
  __shared__ int s_row_off[kMaxE + 1];
  __shared__ int s_warp[NT / 32];
  __shared__ int s_bad;
  __shared__ int s_is_last;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int wW = warp % WARPS_W;
  const int wT = warp / WARPS_W;
  const int E = static_cast<int>(a.E);
  const int64_t N = a.N;
  const int64_t K = a.K;
  const int NB = static_cast<int>((N + T::BNW - 1) / T::BNW);

  // Launched with programmatic stream serialization: the next kernel may be scheduled now, and this one
  // touches memory only once the kernel before it (which may write the activations, the scales or the
  // group list) has finished.
  pdl_trigger();
  pdl_wait();

  // ---- the packed weight must match the call
  if (tid == 0) {
    s_bad = 0;
    const PackedHeader* h = static_cast<const PackedHeader*>(a.packed);
    if (h->magic != kPackMagic || h->version != kPackVersion || h->E != a.E || h->N != a.N ||
        h->K != a.K || ((h->flags ^ a.pack_flags) & W8A8_PACK_GATE_UP) != 0u)
      s_bad = W8A8_ERR_PACKED;
  }
  // ---- per-expert row and tile prefix sums (block scan over <= kMaxE experts)
  constexpr int kPer = (kMaxE + NT - 1) / NT;
  int rows_loc = 0, tiles_loc = 0, neg = 0;
  int cnts[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = tid * kPer + i;
    int64_t c = 0;
    if (e < E) c = a.group_list ? a.group_list[e] : a.R;
    if (c < 0 || c > a.R) neg = 1;
    const int ci = (c < 0 || c > a.R) ? 0 : static_cast<int>(c);
    cnts[i] = ci;
    rows_loc += ci;
    tiles_loc += ((ci + T::BMT - 1) / T::BMT) * NB * ksplit;
  }
  int rows_total, tiles_total;
  int row_before = block_exclusive_scan<NT>(rows_loc, rows_total, s_warp);
  int tile_before = block_exclusive_scan<NT>(tiles_loc, tiles_total, s_warp);
  if (neg) atomicOr(&s_bad, W8A8_ERR_GROUP_LIST << 8);
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = tid * kPer + i;
    if (e < E) {
      s_row_off[e] = row_before;
      s_tile_prefix[e] = tile_before;
    }
    row_before += cnts[i];
    tile_before += ((cnts[i] + T::BMT - 1) / T::BMT) * NB * ksplit;
  }
  if (tid == 0) {
    s_row_off[E] = rows_total;
    s_tile_prefix[E] = tiles_total;
  }
  __syncthreads();
  {
    int bad = s_bad;
    if (rows_total != a.R) bad |= W8A8_ERR_GROUP_LIST << 8;
    if (bad) {
      if (tid == 0 && blockIdx.x == 0)
        set_status(a.status, (bad & 0xff) ? (bad & 0xff) : (bad >> 8), 0u);
      return;
    }
  }

  const PackedHeader* hdr = static_cast<const PackedHeader*>(a.packed);
  const int8_t* w_i8 = reinterpret_cast<const int8_t*>(static_cast<const uint8_t*>(a.packed) + hdr->i8_offset);
  const int kb_total = static_cast<int>((K + BK - 1) / BK);
  const bool vec_out = ((reinterpret_cast<uintptr_t>(a.out) & 15u) == 0u) && ((N & 7) == 0);
  int* S = reinterpret_cast<int*>(smem);

  for (int t = blockIdx.x; t < tiles_total; t += gridDim.x) {
    // ---- tile -> (expert, n-block, m-block, k-split)
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tile_prefix[mid] <= t) lo = mid; else hi = mid;
    }
    const int e = lo;
    int local = t - s_tile_prefix[e];
    const int ks = local % ksplit;
    local /= ksplit;
    const int cnt = s_row_off[e + 1] - s_row_off[e];
    const int mblocks = (cnt + T::BMT - 1) / T::BMT;
    const int mb = local % mblocks;
    const int nb = local / mblocks;

    const int64_t n0 = static_cast<int64_t>(nb) * T::BNW;
    const int rows_w = static_cast<int>(N - n0 < T::BNW ? N - n0 : static_cast<int64_t>(T::BNW));
    const int64_t r0 = static_cast<int64_t>(s_row_off[e]) + static_cast<int64_t>(mb) * T::BMT;
    const int rows_t = min(T::BMT, cnt - mb * T::BMT);
    const int kb0 = static_cast<int>(static_cast<int64_t>(kb_total) * ks / ksplit);
    const int kb1 = static_cast<int>(static_cast<int64_t>(kb_total) * (ks + 1) / ksplit);
    const int nkb = kb1 - kb0;
    const int8_t* wbase = w_i8 + (static_cast<int64_t>(e) * N + n0) * K;
    const int8_t* tbase = a.q + r0 * K;

    auto load_stage = [&](int stage, int kb) {
      uint8_t* sW = smem + stage * T::kStageBytes;
      uint8_t* sT = sW + T::kStageW;
      const int64_t kbyte = static_cast<int64_t>(kb) * BK;
#pragma unroll
      for (int c = tid; c < T::BNW * 4; c += NT) {
        const int row = c >> 2, ch = c & 3;
        const int64_t k = kbyte + ch * 16;
        const bool ok = (row < rows_w) && (k < K);
        cp_async_16(smem_u32(sW + swz(row, ch)), ok ? wbase + static_cast<int64_t>(row) * K + k : wbase, ok ? 16 : 0);
      }
#pragma unroll
      for (int c = tid; c < T::BMT * 4; c += NT) {
        const int row = c >> 2, ch = c & 3;
        const int64_t k = kbyte + ch * 16;
        const bool ok = (row < rows_t) && (k < K);
        cp_async_16(smem_u32(sT + swz(row, ch)), ok ? tbase + static_cast<int64_t>(row) * K + k : a.q, ok ? 16 : 0);
      }
    };

    float accf[WM][WN][4];
    int acci[WM][WN][4];
#pragma unroll
    for (int i = 0; i < WM; ++i)
#pragma unroll
      for (int j = 0; j < WN; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          accf[i][j][c] = 0.0f;
          acci[i][j][c] = 0;
        }
    auto drain = [&]() {
#pragma unroll
      for (int i = 0; i < WM; ++i)
#pragma unroll
        for (int j = 0; j < WN; ++j)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            acci[i][j][c] += __float2int_rn(accf[i][j][c]);
            accf[i][j][c] = 0.0f;
          }
    };

#pragma unroll
    for (int s = 0; s < T::kStages - 1; ++s) {
      if (s < nkb) load_stage(s, kb0 + s);
      cp_async_commit();
    }
    int since_drain = 0;
    for (int i = 0; i < nkb; ++i) {
      cp_async_wait<T::kStages - 2>();
      __syncthreads();
      {
        const int nxt = i + T::kStages - 1;
        if (nxt < nkb) load_stage(nxt % T::kStages, kb0 + nxt);
        cp_async_commit();
      }
      const uint8_t* sW = smem + (i % T::kStages) * T::kStageBytes;
      const uint8_t* sT = sW + T::kStageW;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t af[WM][4];
#pragma unroll
        for (int mi = 0; mi < WM; ++mi) {
          const int row = wW * 16 * WM + 16 * mi + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int ch = 2 * kk + (lane >> 4);
          ldmatrix_x4(smem_u32(sW + swz(row, ch)), af[mi][0], af[mi][1], af[mi][2], af[mi][3]);
        }
        uint32_t bfr[WN][2];
        if constexpr (WN % 2 == 0) {
#pragma unroll
          for (int nj = 0; nj < WN; nj += 2) {
            const int row = wT * 8 * WN + 8 * nj + (lane & 7) + 8 * (lane >> 4);
            const int ch = 2 * kk + ((lane >> 3) & 1);
            ldmatrix_x4(smem_u32(sT + swz(row, ch)), bfr[nj][0], bfr[nj][1], bfr[nj + 1][0], bfr[nj + 1][1]);
          }
        } else {
          const int row = wT * 8 * WN + (lane & 7);
          const int ch = 2 * kk + ((lane >> 3) & 1);
          ldmatrix_x2(smem_u32(sT + swz(row, ch)), bfr[0][0], bfr[0][1]);
        }
#pragma unroll
        for (int step = 0; step < 2; ++step) {
          uint32_t a16[WM][4];
#pragma unroll
          for (int mi = 0; mi < WM; ++mi) {
            uint32_t l0, h0, l1, h1;
            s8x4_to_f16x4(af[mi][2 * step], l0, h0);
            s8x4_to_f16x4(af[mi][2 * step + 1], l1, h1);
            a16[mi][0] = l0;
            a16[mi][1] = l1;
            a16[mi][2] = h0;
            a16[mi][3] = h1;
          }
#pragma unroll
          for (int nj = 0; nj < WN; ++nj) {
            uint32_t bl, bh;
            s8x4_to_f16x4(bfr[nj][step], bl, bh);
#pragma unroll
            for (int mi = 0; mi < WM; ++mi) mma_f16_16816(accf[mi][nj], a16[mi], bl, bh);
          }
        }
      }
      if (++since_drain == kChunkK / BK) {
        drain();
        since_drain = 0;
      }
    }
    drain();
    cp_async_wait<0>();
    __syncthreads();  // pipeline smem is free: stage the int32 tile token-major

    {
      const int g = lane >> 2, tq = lane & 3;
#pragma unroll
      for (int mi = 0; mi < WM; ++mi)
#pragma unroll
        for (int nj = 0; nj < WN; ++nj) {
          const int rc = wW * 16 * WM + 16 * mi + g;
          const int tk = wT * 8 * WN + 8 * nj + 2 * tq;
          S[tk * T::kEpiStride + rc] = acci[mi][nj][0];
          S[(tk + 1) * T::kEpiStride + rc] = acci[mi][nj][1];
          S[tk * T::kEpiStride + rc + 8] = acci[mi][nj][2];
          S[(tk + 1) * T::kEpiStride + rc + 8] = acci[mi][nj][3];
        }
    }
    __syncthreads();

    if (ksplit > 1) {
      for (int c = tid; c < T::BMT * T::BNW; c += NT) {
        const int m = c / T::BNW, n = c % T::BNW;
        if (m < rows_t && n < rows_w) atomicAdd(&a.ws_acc[(r0 + m) * N + n0 + n], S[m * T::kEpiStride + n]);
      }
      __threadfence();
      __syncthreads();
      const int out_t = t / ksplit;
      if (tid == 0) {
        if (out_t >= a.ws_count_len) {
          set_status(a.status, W8A8_ERR_WORKSPACE, static_cast<uint32_t>(out_t));
          s_is_last = 0;
        } else {
          const unsigned prev = atomicAdd(&a.ws_count[out_t], 1u);
          s_is_last = (prev == static_cast<unsigned>(ksplit - 1)) ? 1 : 0;
        }
      }
      __syncthreads();
      if (!s_is_last) continue;
      __threadfence();
      for (int c = tid; c < T::BMT * T::BNW; c += NT) {
        const int m = c / T::BNW, n = c % T::BNW;
        if (m < rows_t && n < rows_w) {
          int* p = &a.ws_acc[(r0 + m) * N + n0 + n];
          S[m * T::kEpiStride + n] = __ldcg(p);
          *p = 0;
        }
      }
      if (tid == 0) a.ws_count[out_t] = 0u;
      __syncthreads();
    }

    // ---- epilogue from the staged int32 tile
    if constexpr (MODE == EPI_ACC) {
      int32_t* out = static_cast<int32_t*>(a.out);
      for (int c = tid; c < T::BMT * (T::BNW / 8); c += NT) {
        const int m = c / (T::BNW / 8), n8 = (c % (T::BNW / 8)) * 8;
        if (m >= rows_t) continue;
        int32_t* dst = out + (r0 + m) * N + n0 + n8;
        const int* src = S + m * T::kEpiStride + n8;
        if (vec_out && n8 + 8 <= rows_w) {
          reinterpret_cast<int4*>(dst)[0] = make_int4(src[0], src[1], src[2], src[3]);
          reinterpret_cast<int4*>(dst)[1] = make_int4(src[4], src[5], src[6], src[7]);
        } else {
          for (int k = 0; k < 8; ++k)
            if (n8 + k < rows_w) dst[k] = src[k];
        }
      }
    } else if constexpr (MODE == EPI_BF16) {
      uint16_t* out = static_cast<uint16_t*>(a.out);
      const float* sw = a.w_scale + static_cast<int64_t>(e) * N;
      for (int c = tid; c < T::BMT * (T::BNW / 8); c += NT) {
        const int m = c / (T::BNW / 8), n8 = (c % (T::BNW / 8)) * 8;
        if (m >= rows_t) continue;
        const float sx = a.x_scale != nullptr ? a.x_scale[r0 + m] : 1.0f;
        uint16_t* dst = out + (r0 + m) * N + n0 + n8;
        const int* src = S + m * T::kEpiStride + n8;
        uint16_t v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int64_t n = n0 + n8 + k;
          float f = 0.0f;
          if (n8 + k < rows_w) {
            f = a.qbias != nullptr ? dequant_q(src[k], a.qbias[n], sx, sw[n]) : dequant(src[k], sx, sw[n]);
            if (a.bias) f = __fadd_rn(f, bf16_bits_to_f32(a.bias[n]));
          }
          v[k] = f32_to_bf16_bits(f);
        }
        if (vec_out && n8 + 8 <= rows_w) {
          *reinterpret_cast<uint4*>(dst) =
              make_uint4(v[0] | (uint32_t(v[1]) << 16), v[2] | (uint32_t(v[3]) << 16),
                         v[4] | (uint32_t(v[5]) << 16), v[6] | (uint32_t(v[7]) << 16));
        } else {
          for (int k = 0; k < 8; ++k)
            if (n8 + k < rows_w) dst[k] = v[k];
        }
      }
    } else {  // EPI_SWIGLU: tile rows [0,64) gate j, [64,128) up j, j = nb*64 + [0,64)
      static_assert(MODE != EPI_SWIGLU || T::BNW == 2 * kGateUpBlock, "gate/up tile");
      uint16_t* out = static_cast<uint16_t*>(a.out);
      const int64_t I = N / 2;
      const float* sw = a.w_scale + static_cast<int64_t>(e) * N;
      const bool vec_h = ((reinterpret_cast<uintptr_t>(a.out) & 15u) == 0u) && ((I & 7) == 0);
      for (int c = tid; c < T::BMT * (kGateUpBlock / 8); c += NT) {
        const int m = c / (kGateUpBlock / 8), j8 = (c % (kGateUpBlock / 8)) * 8;
        if (m >= rows_t) continue;
        const float sx = a.x_scale[r0 + m];
        const int64_t jb = static_cast<int64_t>(nb) * kGateUpBlock + j8;
        const int* src = S + m * T::kEpiStride + j8;
        uint16_t v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float gte = bf16_round(dequant(src[k], sx, sw[jb + k]));
          const float up = bf16_round(dequant(src[kGateUpBlock + k], sx, sw[I + jb + k]));
          v[k] = swiglu_bf16(gte, up);
        }
        uint16_t* dst = out + (r0 + m) * I + jb;
        if (vec_h) {
          *reinterpret_cast<uint4*>(dst) =
              make_uint4(v[0] | (uint32_t(v[1]) << 16), v[2] | (uint32_t(v[3]) << 16),
                         v[4] | (uint32_t(v[5]) << 16), v[6] | (uint32_t(v[7]) << 16));
        } else {
          for (int k = 0; k < 8; ++k) dst[k] = v[k];
        }
      }
    }
    __syncthreads();  // S aliases the pipeline of the next tile
  }
}

// Tile variants: (WM, WN, WARPS_W, WARPS_T)
//   V8  = 1,1,8,1 : 128 rows x  8 tokens (decode-sized groups)
//   V32 = 2,2,4,2 : 128 rows x 32 tokens
//   V64 = 2,4,4,2 : 128 rows x 64 tokens
template <int MODE>
cudaError_t launch_variant(const GemmArgs& a, const GemmPlan& p, cudaStream_t stream) {
  switch (p.variant) {
    case 8: {
      auto k = reg_gemm_kernel<1, 1, 8, 1, MODE>;
      if (cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(p.smem)))
        return e;
      return launch_pdl(k, dim3(p.grid), dim3(256), p.smem, stream, a, p.ksplit);
    }
    case 32: {
      auto k = reg_gemm_kernel<2, 2, 4, 2, MODE>;
      if (cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(p.smem)))
        return e;
      return launch_pdl(k, dim3(p.grid), dim3(256), p.smem, stream, a, p.ksplit);
    }
    default: {
      auto k = reg_gemm_kernel<2, 4, 4, 2, MODE>;
      if (cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(p.smem)))
        return e;
      return launch_pdl(k, dim3(p.grid), dim3(256), p.smem, stream, a, p.ksplit);
    }
  }
}

int bmt_of(int variant) { return variant == 8 ? 8 : variant == 32 ? 32 : 64; }
size_t smem_of(int variant) {
  return variant == 8 ? Tile<1, 1, 8, 1>::kSmem : variant == 32 ? Tile<2, 2, 4, 2>::kSmem : Tile<2, 4, 4, 2>::kSmem;
}

int64_t upper_tiles(int64_t E, int64_t R, int64_t N, bool grouped, int bmt) {
  const int64_t nb = (N + 127) / 128;
  const int64_t mblocks = (R + bmt - 1) / bmt + (grouped ? E : 0);
  return mblocks * nb;
}

}  // namespace

GemmPlan plan_reg_gemm(const GemmArgs& a, int num_sms) {
  GemmPlan p{};
  const double avg = a.E > 0 ? static_cast<double>(a.R) / static_cast<double>(a.E) : 0.0;
  p.variant = avg <= 8.0 ? 8 : (avg <= 32.0 ? 32 : 64);
  const int bmt = bmt_of(p.variant);
  const bool grouped = a.group_list != nullptr;
  const int64_t est = std::max<int64_t>(1, ((a.R + bmt - 1) / bmt) * ((a.N + 127) / 128));
  int ks = 1;
  if (a.ws_acc != nullptr && est < num_sms && a.K >= 512) {
    ks = static_cast<int>(std::min<int64_t>({8, (2 * num_sms + est - 1) / est, a.K / 256}));
    ks = std::max(ks, 1);
  }
  p.ksplit = ks;
  const int64_t ub = upper_tiles(a.E, a.R, a.N, grouped, bmt) * ks;
  const int per_sm = p.variant == 8 ? REG_GRID_V8 : 2;
  p.grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ub, static_cast<int64_t>(num_sms) * per_sm)));
  p.smem = smem_of(p.variant);
  return p;
}

size_t reg_gemm_ws_bytes(int64_t E, int64_t R, int64_t N, int64_t K, int num_sms) {
  (void)K;
  (void)num_sms;
  // partial sums [R,N] int32 + one counter per output tile (smallest BMT bounds the count)
  const size_t acc = align_up(static_cast<uint64_t>(R) * N * 4, 256);
  const size_t cnt = align_up(static_cast<uint64_t>(upper_tiles(E, R, N, E > 1, 8)) * 4, 256);
  return acc + cnt;
}

cudaError_t launch_reg_gemm(const GemmArgs& a, const GemmPlan& p, cudaStream_t stream) {
  if (a.R == 0) return cudaSuccess;
  switch (a.mode) {
    case EPI_ACC: return launch_variant<EPI_ACC>(a, p, stream);
    case EPI_SWIGLU: return launch_variant<EPI_SWIGLU>(a, p, stream);
    default: return launch_variant<EPI_BF16>(a, p, stream);
  }
}

}  // namespace w8a8
