// route.cu -- MoE routing on either side of the expert chain.
//
// Page "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子" §三: the DeepEP INT8
// dispatch hands the Ascend runner INT8 hidden rows with their per-token
// scales, topk_ids / topk_weights and the rows per expert (expert_tokens, the
// grouped matmul's group_list); the runner input is those rows regrouped by
// expert, and after W2 each token's rows are summed with its router weights.
//
//   route    every (token t, slot j) pair of topk_ids [T,k] is one routed row;
//            rows are ordered by expert, then token, then slot.  A stable
//            counting sort: per chunk of pairs a count per expert, one scan
//            over (expert, chunk) for the chunk offsets and the group list,
//            then each chunk walks its pairs in order, ranking equal experts
//            inside a warp with a match mask.
//   scatter  the routed copies of already-quantised token rows (codes and
//            scale unchanged; the BF16 case quantises in quant.cu).
//   combine  y[t,c] = bf16(sum over j in slot order of w[t,j] * y_routed[pos[t,j], c]),
//            binary32 products and sums.
//
// All of it is bound by memory or latency: the sort reads the ids twice
// (8 bytes a pair each time) and writes a 4-byte row index; the combine reads
// k routed rows per token and writes one.
#include "tc_common.cuh"

namespace w8a8 {

namespace {

constexpr int kRouteChunk = 512;  // pairs per routing block (one warp)

__device__ __forceinline__ void pdl_enter() {
  pdl_trigger();
  pdl_wait();
}

int64_t route_blocks(int64_t n) { return std::max<int64_t>(1, (n + kRouteChunk - 1) / kRouteChunk); }

constexpr int kIdsPerLane = kRouteChunk / 32;

// The ids of chunk b held by one lane: lane + 32u for u < kIdsPerLane, all loaded before any is used.
// -1 marks a position past the end, -2 an id outside [0,E).
__device__ __forceinline__ void load_chunk_ids(const int64_t* __restrict__ ids, int64_t n, int E, int64_t base,
                                               int lane, int (&id)[kIdsPerLane]) {
  int64_t raw[kIdsPerLane];
#pragma unroll
  for (int u = 0; u < kIdsPerLane; ++u) {
    const int64_t p = base + lane + 32 * u;
    raw[u] = p < n ? ids[p] : -1;
  }
#pragma unroll
  for (int u = 0; u < kIdsPerLane; ++u) {
    const int64_t p = base + lane + 32 * u;
    id[u] = p >= n ? -1 : (raw[u] >= 0 && raw[u] < E) ? static_cast<int>(raw[u]) : -2;
  }
}

// counts[e * nb + b] = pairs of chunk b that name expert e.  An id outside [0,E) is not counted and
// records W8A8_ERR_TOPK_IDS with its pair index.
__global__ void __launch_bounds__(32) route_count(const int64_t* __restrict__ ids, int64_t n, int E, int nb,
                                                  int32_t* __restrict__ counts, DeviceStatus* status) {
  pdl_enter();
  extern __shared__ int32_t cnt[];
  const int lane = threadIdx.x;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kRouteChunk;
  int id[kIdsPerLane];
  load_chunk_ids(ids, n, E, base, lane, id);
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
#pragma unroll
  for (int u = 0; u < kIdsPerLane; ++u) {
    if (id[u] >= 0) atomicAdd(&cnt[id[u]], 1);
    else if (id[u] == -2) set_status(status, W8A8_ERR_TOPK_IDS, static_cast<uint32_t>(base + lane + 32 * u));
  }
  __syncwarp();
  for (int e = lane; e < E; e += 32) counts[static_cast<int64_t>(e) * nb + blockIdx.x] = cnt[e];
}

__device__ __forceinline__ int32_t warp_sum_i(int32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int32_t warp_incl_scan_i(int32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t x = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += x;
  }
  return v;
}

// Lanes of the warp whose key equals this lane's: one ballot per key bit (nbits bits cover every expert
// id), so the cost does not grow with the number of distinct keys in the warp.  Lanes with valid ==
// false match only themselves.
__device__ __forceinline__ unsigned match_key(int key, bool valid, int nbits, int lane) {
  unsigned m = __ballot_sync(0xffffffffu, valid);
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (key >> b) & 1;
    const unsigned bb = __ballot_sync(0xffffffffu, bit);
    m &= bit ? bb : ~bb;
  }
  return valid ? m : (1u << lane);
}

constexpr int kScanCache = 4;  // chunks of 32 counts whose loads a lane issues together

// One CTA of 1024 threads.  Warp w takes experts w, w + 32, ...: the total of expert e over the
// chunks (loads of a warp all in flight together), then the exclusive prefix of the totals over the
// experts (the expert's first routed row), group_list[e] = total, and counts[e * nb + b] replaced by
// the first routed row of chunk b's pairs for expert e.
__global__ void __launch_bounds__(1024) route_scan(int32_t* __restrict__ counts, int E, int nb,
                                                   int64_t* __restrict__ group_list) {
  pdl_enter();
  __shared__ int32_t tot[W8A8_MAX_EXPERTS];
  __shared__ int32_t warp_sum[32];
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  for (int e = w; e < E; e += 32) {
    const int32_t* ce = counts + static_cast<int64_t>(e) * nb;
    int32_t c[kScanCache];
#pragma unroll
    for (int u = 0; u < kScanCache; ++u) c[u] = 32 * u + lane < nb ? ce[32 * u + lane] : 0;
    int32_t t = 0;
#pragma unroll
    for (int u = 0; u < kScanCache; ++u) t += c[u];
    for (int b0 = 32 * kScanCache; b0 < nb; b0 += 32) t += b0 + lane < nb ? ce[b0 + lane] : 0;
    t = warp_sum_i(t);
    if (lane == 0) tot[e] = t;
  }
  __syncthreads();
  const int e = threadIdx.x;
  const int32_t mine = e < E ? tot[e] : 0;
  const int32_t incl = warp_incl_scan_i(mine, lane);
  if (lane == 31) warp_sum[w] = incl;
  __syncthreads();
  if (w == 0) warp_sum[lane] = warp_incl_scan_i(warp_sum[lane], lane);
  __syncthreads();
  const int32_t first = incl - mine + (w > 0 ? warp_sum[w - 1] : 0);
  __syncthreads();  // every thread has read tot[] before it is overwritten with the first rows
  if (e < E) {
    group_list[e] = mine;
    tot[e] = first;
  }
  __syncthreads();
  for (int e2 = w; e2 < E; e2 += 32) {
    int32_t* ce = counts + static_cast<int64_t>(e2) * nb;
    int32_t run = tot[e2];
    for (int b0 = 0; b0 < nb; b0 += 32) {
      const bool in = b0 + lane < nb;
      const int32_t c = in ? ce[b0 + lane] : 0;
      const int32_t inc = warp_incl_scan_i(c, lane);
      if (in) ce[b0 + lane] = run + inc - c;
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
  }
}

// Chunk b's pairs in order, 32 at a time: lanes naming the same expert share a match mask, a lane's
// rank among them is the number of lower lanes in it, and the lowest of them advances the expert's
// cursor by their number.  A pair with a bad id gets pos = -1.
__global__ void __launch_bounds__(32) route_assign(const int64_t* __restrict__ ids, int64_t n, int E, int nbits,
                                                   int nb, const int32_t* __restrict__ first_row,
                                                   int32_t* __restrict__ pos) {
  pdl_enter();
  extern __shared__ int32_t cur[];
  const int lane = threadIdx.x;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kRouteChunk;
  int id[kIdsPerLane];
  load_chunk_ids(ids, n, E, base, lane, id);
  for (int e = lane; e < E; e += 32) cur[e] = first_row[static_cast<int64_t>(e) * nb + blockIdx.x];
  __syncwarp();
#pragma unroll
  for (int u = 0; u < kIdsPerLane; ++u) {
    const int64_t p = base + lane + 32 * u;
    const bool ok = id[u] >= 0;
    const int key = ok ? id[u] : 0;
    const unsigned mask = match_key(key, ok, nbits, lane);
    const int rank = __popc(mask & ((1u << lane) - 1u));
    const int32_t r = ok ? cur[key] + rank : -1;
    __syncwarp();
    if (ok && rank == 0) cur[key] += __popc(mask);
    __syncwarp();
    if (p < n) pos[p] = r;
  }
}

// Routing of up to kSmallMaxPairs pairs (decode-sized batches) in one CTA of 1024 threads, in shared memory: the ids as
// 16-bit keys, warp w owning the contiguous segment [w*S, (w+1)*S) of pairs; per-warp counts per
// expert, then (thread e for expert e) the expert totals, their prefix and each warp's first row per
// expert, then each warp ranks its segment in order.  One launch, one read of the ids.
constexpr int kSmallThreads = 1024;
constexpr int64_t kSmallMaxPairs = 8192;  // beyond this one SM's issue rate loses to the 3-kernel sort
constexpr size_t kSmallMaxSmem = 200 * 1024;
constexpr uint16_t kNoKey = 0xffffu;

int64_t small_seg(int64_t n) { return ((n + 31) / 32 + 31) / 32 * 32; }
size_t small_smem(int64_t n, int E) {
  return static_cast<size_t>(32) * E * 4 + static_cast<size_t>(align_up(static_cast<uint64_t>(32 * small_seg(n)) * 2, 16));
}

__global__ void __launch_bounds__(kSmallThreads) route_small(const int64_t* __restrict__ ids, int64_t n, int E,
                                                             int nbits, int S, int64_t* __restrict__ group_list,
                                                             int32_t* __restrict__ pos, DeviceStatus* status) {
  pdl_enter();
  extern __shared__ __align__(16) uint8_t route_smem[];
  int32_t* off = reinterpret_cast<int32_t*>(route_smem);                        // [32][E]
  uint16_t* key = reinterpret_cast<uint16_t*>(route_smem + static_cast<size_t>(32) * E * 4);  // [32*S]
  __shared__ int32_t warp_sum[32];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int w = tid >> 5;
  for (int i = tid; i < 32 * E; i += kSmallThreads) off[i] = 0;
  const int64_t total = 32LL * S;
  for (int64_t i0 = 0; i0 < total; i0 += 8 * kSmallThreads) {
    int64_t raw[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t p = i0 + u * kSmallThreads + tid;
      raw[u] = p < n ? ids[p] : -1;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t p = i0 + u * kSmallThreads + tid;
      if (p >= total) continue;
      uint16_t k = kNoKey;
      if (p < n) {
        if (raw[u] >= 0 && raw[u] < E) k = static_cast<uint16_t>(raw[u]);
        else set_status(status, W8A8_ERR_TOPK_IDS, static_cast<uint32_t>(p));
      }
      key[p] = k;
    }
  }
  __syncthreads();
  const int64_t seg = static_cast<int64_t>(w) * S;
  for (int x = 0; x < S; x += 32) {
    const int kk = key[seg + x + lane];
    const bool valid = kk != kNoKey;
    const unsigned m = match_key(kk, valid, nbits, lane);
    if (valid && (m & ((1u << lane) - 1u)) == 0u) off[w * E + kk] += __popc(m);
    __syncwarp();
  }
  __syncthreads();
  const int e = tid;
  int32_t tot = 0;
  if (e < E)
    for (int ww = 0; ww < 32; ++ww) tot += off[ww * E + e];
  const int32_t incl = warp_incl_scan_i(tot, lane);
  if (lane == 31) warp_sum[w] = incl;
  __syncthreads();
  if (w == 0) warp_sum[lane] = warp_incl_scan_i(warp_sum[lane], lane);
  __syncthreads();
  if (e < E) {
    group_list[e] = tot;
    int32_t run = incl - tot + (w > 0 ? warp_sum[w - 1] : 0);
    for (int ww = 0; ww < 32; ++ww) {
      const int32_t c = off[ww * E + e];
      off[ww * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int x = 0; x < S; x += 32) {
    const int64_t p = seg + x + lane;
    const int kk = key[p];
    const bool valid = kk != kNoKey;
    const unsigned m = match_key(kk, valid, nbits, lane);
    const int rank = __popc(m & ((1u << lane) - 1u));
    const int32_t r = valid ? off[w * E + kk] + rank : -1;
    __syncwarp();
    if (valid && rank == 0) off[w * E + kk] += __popc(m);
    __syncwarp();
    if (p < n) pos[p] = r;
  }
}

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Routed copies of INT8 token rows: thread per 16 codes of a token; out 0 int8, 1 fp16, 2 both.
__global__ void __launch_bounds__(256) scatter_rows_i8(const int8_t* __restrict__ xq, const float* __restrict__ xs,
                                                       int64_t T, int64_t H, const int32_t* __restrict__ dst, int k,
                                                       int8_t* __restrict__ q, uint16_t* __restrict__ q16,
                                                       float* __restrict__ scale, int out) {
  pdl_enter();
  const int64_t nc = H / 16;
  const int64_t total = T * nc;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * 256) {
    const int64_t t = i / nc;
    const int64_t c = i - t * nc;
    const uint4 v = ldg_nc(xq + t * H + c * 16);
    uint4 f0 = make_uint4(0u, 0u, 0u, 0u), f1 = f0;
    if (out != 0) {
      s8x4_to_f16x4(v.x, f0.x, f0.y);
      s8x4_to_f16x4(v.y, f0.z, f0.w);
      s8x4_to_f16x4(v.z, f1.x, f1.y);
      s8x4_to_f16x4(v.w, f1.z, f1.w);
    }
    const float s = c == 0 ? xs[t] : 0.0f;
    for (int j = 0; j < k; ++j) {
      const int64_t r = dst[t * k + j];
      if (r < 0) continue;
      if (out != 1) *reinterpret_cast<uint4*>(q + r * H + c * 16) = v;
      if (out != 0) {
        uint4* d = reinterpret_cast<uint4*>(q16 + r * H + c * 16);
        d[0] = f0;
        d[1] = f1;
      }
      if (c == 0) scale[r] = s;
    }
  }
}

// Combine.  Work item = (token t, slice of kCbCols columns); a unit = one item's slots j0 .. j0+7.
// Warp-specialised: warp 0 copies each unit's routed row slices (2 KB each) into a shared-memory
// stage with cp.async.bulk, completing on the stage's full barrier; warps 1-4 (8 columns a thread)
// wait on it, sum the unit's slots in slot order, and release the stage on its empty barrier.  The
// row indices and weights of the units to copy are loaded kCbAhead units ahead, so no global round
// trip sits between a stage being released and its next copy.  No CTA-wide barrier in the loop.
constexpr int kCbConsumers = 128;
constexpr int kCbThreads = 32 + kCbConsumers;
constexpr int kCbCols = 8 * kCbConsumers;  // 1024 columns per item
constexpr int kCbSlots = 8;
constexpr int kCbStages = 4;
constexpr int kCbAhead = 4;
constexpr int kCbRowBytes = kCbCols * 2;
constexpr int kCbStageBytes = kCbSlots * kCbRowBytes;

struct CbMeta {
  float w[kCbSlots];
  uint32_t ok;  // bit u: slot u of the unit holds a routed row
  uint32_t pad[3];
};
constexpr size_t kCbSmem = static_cast<size_t>(kCbStages) * kCbStageBytes + kCbStages * sizeof(CbMeta) +
                           2 * kCbStages * 8 + 16;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar)
               : "memory");
}

// Bounded wait used only to drain copies still in flight after a CTA has given up.
__device__ __forceinline__ void drain_wait(uint32_t a, uint32_t parity) {
  const uint64_t t0 = tc::globaltimer_ns();
  while (!tc::mbar_try_wait(a, parity) && tc::globaltimer_ns() - t0 < tc::kWaitLimitNs) {
  }
}

__global__ void __launch_bounds__(kCbThreads) combine_kernel(const uint16_t* __restrict__ yr,
                                                             const int32_t* __restrict__ pos,
                                                             const float* __restrict__ w, int T, int k, int H,
                                                             uint16_t* __restrict__ y, DeviceStatus* status) {
  extern __shared__ __align__(128) uint8_t cb_smem[];
  uint8_t* data = cb_smem;
  CbMeta* meta = reinterpret_cast<CbMeta*>(cb_smem + static_cast<size_t>(kCbStages) * kCbStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + kCbStages);
  uint64_t* empty = full + kCbStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kCbStages);
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int nslice = (H + kCbCols - 1) / kCbCols;
  const int nitems = T * nslice;  // < 2^31: checked by the host
  const int nbatch = (k + kCbSlots - 1) / kCbSlots;
  const int my_items = static_cast<int>(blockIdx.x) < nitems ? (nitems - 1 - static_cast<int>(blockIdx.x)) /
                                                                   static_cast<int>(gridDim.x) + 1
                                                             : 0;
  const int nunits = my_items * nbatch;
  const int64_t R = static_cast<int64_t>(T) * k;
  if (tid == 0) {
    for (int s = 0; s < kCbStages; ++s) {
      tc::mbar_init(smem_u32(&full[s]), 1);
      tc::mbar_init(smem_u32(&empty[s]), kCbConsumers / 32);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();

  if (tid < 32) {
    // ---------------------------------------------------------------- producer warp
    // unit q of this CTA: item blockIdx.x + (q / nbatch) * gridDim.x, slots (q % nbatch) * 8 + u
    auto load_slot = [&](int q, int32_t& r, float& wt) {
      r = -1;
      wt = 0.0f;
      if (q >= nunits || lane >= kCbSlots) return;
      const int64_t t = (static_cast<int>(blockIdx.x) + (q / nbatch) * static_cast<int>(gridDim.x)) / nslice;
      const int j = (q % nbatch) * kCbSlots + lane;
      if (j < k) {
        r = pos[t * k + j];
        wt = w[t * k + j];
        if (r < 0 || r >= R) {
          set_status(status, W8A8_ERR_TOPK_IDS, static_cast<uint32_t>(t * k + j));
          r = -1;
        }
      }
    };
    int32_t ar[kCbAhead];
    float aw[kCbAhead];
#pragma unroll
    for (int a = 0; a < kCbAhead; ++a) load_slot(a, ar[a], aw[a]);
    int q = 0;
    for (; q < nunits; ++q) {
      const int s = q % kCbStages;
      if (q >= kCbStages) {  // wait until the consumers have released the unit that last used stage s
        const uint32_t parity = static_cast<uint32_t>(((q / kCbStages) - 1) & 1);
        if (!tc::mbar_wait(smem_u32(&empty[s]), parity, abort_flag, status, 0x43000001u)) break;
      }
      const int item = static_cast<int>(blockIdx.x) + (q / nbatch) * static_cast<int>(gridDim.x);
      const int t = item / nslice;
      const int col0 = (item - t * nslice) * kCbCols;
      const uint32_t bytes = static_cast<uint32_t>((H - col0 < kCbCols ? H - col0 : kCbCols) * 2);
      const int32_t r = ar[0];
      const bool ok = r >= 0;
      const unsigned okm = __ballot_sync(0xffffffffu, ok);
      if (lane < kCbSlots) meta[s].w[lane] = aw[0];
      if (lane == 0) meta[s].ok = okm;
      __threadfence_block();
      __syncwarp();
      if (lane == 0) tc::mbar_expect_tx(smem_u32(&full[s]), bytes * __popc(okm));
      __syncwarp();
      if (ok)
        bulk_g2s(smem_u32(data + static_cast<size_t>(s) * kCbStageBytes + lane * kCbRowBytes),
                 yr + static_cast<int64_t>(r) * H + col0, bytes, smem_u32(&full[s]));
#pragma unroll
      for (int a = 0; a + 1 < kCbAhead; ++a) {
        ar[a] = ar[a + 1];
        aw[a] = aw[a + 1];
      }
      load_slot(q + kCbAhead, ar[kCbAhead - 1], aw[kCbAhead - 1]);
    }
    if (q < nunits && lane == 0) {
      // gave up: let the copies already started land before the CTA's shared memory goes away
      for (int d = q - 1; d >= 0 && d >= q - kCbStages; --d)
        drain_wait(smem_u32(&full[d % kCbStages]), static_cast<uint32_t>((d / kCbStages) & 1));
    }
    return;
  }

  // ------------------------------------------------------------------ consumer warps
  const int ct = tid - 32;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
  int batch = 0, item = static_cast<int>(blockIdx.x);
  for (int q = 0; q < nunits; ++q) {
    const int s = q % kCbStages;
    const uint32_t parity = static_cast<uint32_t>((q / kCbStages) & 1);
    if (!tc::mbar_wait(smem_u32(&full[s]), parity, abort_flag, status, 0x43000002u)) break;
    const uint32_t okm = meta[s].ok;
    const uint8_t* st = data + static_cast<size_t>(s) * kCbStageBytes + ct * 16;
#pragma unroll
    for (int u = 0; u < kCbSlots; ++u) {
      if (!((okm >> u) & 1u)) continue;
      const float wt = meta[s].w[u];
      const uint4 v = *reinterpret_cast<const uint4*>(st + u * kCbRowBytes);
      const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(wt, bf16_bits_to_f32(static_cast<uint16_t>(x[i] & 0xffffu))));
        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(wt, bf16_bits_to_f32(static_cast<uint16_t>(x[i] >> 16))));
      }
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(smem_u32(&empty[s]));
    if (++batch == nbatch) {
      const int t = item / nslice;
      const int c = (item - t * nslice) * kCbCols + ct * 8;
      if (c < H) {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          o[i] = static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * i])) |
                 (static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * i + 1])) << 16);
        *reinterpret_cast<uint4*>(y + static_cast<int64_t>(t) * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
      batch = 0;
      item += static_cast<int>(gridDim.x);
    }
  }
}

// CTAs of combine_kernel resident per SM (queried once; every device of the part is alike).  The
// shared-memory attribute is set before each launch.
int combine_per_sm() {
  static int per_sm = 0;
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, combine_kernel, kCbThreads, kCbSmem) != cudaSuccess ||
        n < 1) {
      cudaGetLastError();
      n = 1;
    }
    per_sm = n;
  }
  return per_sm;
}

}  // namespace

int64_t route_scratch_ints(int64_t n, int64_t E) { return E * route_blocks(n); }

cudaError_t launch_route(const int64_t* topk_ids, int64_t n, int E, int32_t* counts, int64_t* group_list,
                         int32_t* pos, DeviceStatus* status, cudaStream_t stream) {
  if (n == 0) return cudaMemsetAsync(group_list, 0, static_cast<size_t>(E) * sizeof(int64_t), stream);
  int nbits = 0;
  while ((1 << nbits) < E) ++nbits;
  const size_t ssmem = small_smem(n, E);
  if (n <= kSmallMaxPairs && ssmem <= kSmallMaxSmem) {
    const cudaError_t ea = cudaFuncSetAttribute(route_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                static_cast<int>(kSmallMaxSmem));
    if (ea != cudaSuccess) return ea;
    return launch_pdl(route_small, dim3(1), dim3(kSmallThreads), ssmem, stream, topk_ids, n, E, nbits,
                      static_cast<int>(small_seg(n)), group_list, pos, status);
  }
  const int nb = static_cast<int>(route_blocks(n));
  const size_t smem = static_cast<size_t>(E) * sizeof(int32_t);
  cudaError_t e = launch_pdl(route_count, dim3(nb), dim3(32), smem, stream, topk_ids, n, E, nb, counts, status);
  if (e != cudaSuccess) return e;
  e = launch_pdl(route_scan, dim3(1), dim3(1024), 0, stream, counts, E, nb, group_list);
  if (e != cudaSuccess) return e;
  return launch_pdl(route_assign, dim3(nb), dim3(32), smem, stream, topk_ids, n, E, nbits, nb,
                    static_cast<const int32_t*>(counts), pos);
}

cudaError_t launch_scatter_rows_i8(const int8_t* xq_tok, const float* xs_tok, int64_t T, int64_t H,
                                   const int32_t* dst, int k, int8_t* q, uint16_t* q_f16, float* scale, int out,
                                   cudaStream_t stream, int num_sms) {
  const int64_t total = T * (H / 16);
  if (total == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(num_sms) * 8);
  return launch_pdl(scatter_rows_i8, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, xq_tok, xs_tok, T,
                    H, dst, k, q, q_f16, scale, out);
}

cudaError_t launch_combine(const uint16_t* y_routed, const int32_t* pos, const float* w, int64_t T, int k,
                           int64_t H, uint16_t* y, DeviceStatus* status, cudaStream_t stream, int num_sms) {
  const int64_t nslice = (H + kCbCols - 1) / kCbCols;
  const int64_t items = T * nslice;
  if (items == 0) return cudaSuccess;
  const cudaError_t ea = cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(kCbSmem));
  if (ea != cudaSuccess) return ea;
  const int64_t blocks = std::min<int64_t>(items, static_cast<int64_t>(num_sms) * combine_per_sm());
  return launch_pdl(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kCbThreads), kCbSmem, stream,
                    y_routed, pos, w, static_cast<int>(T), k, static_cast<int>(H), y, status);
}

}  // namespace w8a8
