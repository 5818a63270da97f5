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
#include "kernels.cuh"

namespace w8a8 {

namespace {

constexpr int kRouteChunk = 512;  // pairs per routing block (one warp)

__device__ __forceinline__ void pdl_enter() {
  pdl_trigger();
  pdl_wait();
}

int64_t route_blocks(int64_t n) { return std::max<int64_t>(1, (n + kRouteChunk - 1) / kRouteChunk); }

// counts[e * nb + b] = pairs of chunk b that name expert e.  An id outside [0,E) is not counted and
// records W8A8_ERR_TOPK_IDS with its pair index.
__global__ void __launch_bounds__(32) route_count(const int64_t* __restrict__ ids, int64_t n, int E, int nb,
                                                  int32_t* __restrict__ counts, DeviceStatus* status) {
  pdl_enter();
  extern __shared__ int32_t cnt[];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kRouteChunk;
  for (int i = lane; i < kRouteChunk; i += 32) {
    const int64_t p = base + i;
    if (p >= n) break;
    const int64_t id = ids[p];
    if (id >= 0 && id < E) atomicAdd(&cnt[id], 1);
    else set_status(status, W8A8_ERR_TOPK_IDS, static_cast<uint32_t>(p));
  }
  __syncwarp();
  for (int e = lane; e < E; e += 32) counts[static_cast<int64_t>(e) * nb + blockIdx.x] = cnt[e];
}

// One CTA of 1024 threads, thread e for expert e: total of expert e over the chunks, the exclusive
// prefix of the totals over the experts (the expert's first routed row), group_list[e] = total, and
// counts[e * nb + b] replaced by the first routed row of chunk b's pairs for expert e.
__global__ void __launch_bounds__(1024) route_scan(int32_t* __restrict__ counts, int E, int nb,
                                                   int64_t* __restrict__ group_list) {
  pdl_enter();
  __shared__ int32_t warp_sum[32];
  const int e = threadIdx.x;
  const int lane = e & 31;
  const int w = e >> 5;
  int32_t total = 0;
  if (e < E)
    for (int b = 0; b < nb; ++b) total += counts[static_cast<int64_t>(e) * nb + b];
  int32_t incl = total;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[w] = incl;
  __syncthreads();
  if (w == 0) {
    int32_t ws = warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, ws, o);
      if (lane >= o) ws += v;
    }
    warp_sum[lane] = ws;
  }
  __syncthreads();
  if (e < E) {
    group_list[e] = total;
    int32_t run = incl - total + (w > 0 ? warp_sum[w - 1] : 0);
    for (int b = 0; b < nb; ++b) {
      const int64_t i = static_cast<int64_t>(e) * nb + b;
      const int32_t c = counts[i];
      counts[i] = run;
      run += c;
    }
  }
}

// Chunk b's pairs in order, 32 at a time: lanes naming the same expert share a match mask, a lane's
// rank among them is the number of lower lanes in it, and the lowest of them advances the expert's
// cursor by their number.  A pair with a bad id gets pos = -1.
__global__ void __launch_bounds__(32) route_assign(const int64_t* __restrict__ ids, int64_t n, int E, int nb,
                                                   const int32_t* __restrict__ first_row, int32_t* __restrict__ pos) {
  pdl_enter();
  extern __shared__ int32_t cur[];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) cur[e] = first_row[static_cast<int64_t>(e) * nb + blockIdx.x];
  __syncwarp();
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kRouteChunk;
  for (int w = 0; w < kRouteChunk && base + w < n; w += 32) {
    const int64_t p = base + w + lane;
    int key = E + lane;  // never an expert: a lane past the end or with a bad id matches no other lane
    if (p < n) {
      const int64_t id = ids[p];
      if (id >= 0 && id < E) key = static_cast<int>(id);
    }
    const unsigned mask = __match_any_sync(0xffffffffu, key);
    const bool ok = key < E;
    const int rank = __popc(mask & ((1u << lane) - 1u));
    const int32_t r = ok ? cur[key] + rank : -1;
    __syncwarp();
    if (ok && rank == 0) cur[key] += __popc(mask);
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

constexpr int kCombineThreads = 128;  // 8 columns (16 bytes) a thread
constexpr int kCombineBatch = 8;      // routed rows loaded before any is summed

// Block per (token, slice of 1024 columns).  Terms are summed in slot order; every load of a batch
// of slots is in flight before the first is used.
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const uint16_t* __restrict__ yr,
                                                                  const int32_t* __restrict__ pos,
                                                                  const float* __restrict__ w, int64_t T, int k,
                                                                  int64_t H, uint16_t* __restrict__ y,
                                                                  DeviceStatus* status) {
  pdl_enter();
  const int64_t n8 = H / 8;
  const int64_t nslice = (n8 + kCombineThreads - 1) / kCombineThreads;
  const int64_t t = blockIdx.x / nslice;
  const int64_t c = (blockIdx.x - t * nslice) * kCombineThreads + threadIdx.x;
  if (t >= T || c >= n8) return;
  const int64_t R = T * k;
  float s[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) s[e] = 0.0f;
  for (int j0 = 0; j0 < k; j0 += kCombineBatch) {
    uint4 v[kCombineBatch];
    float wj[kCombineBatch];
    bool ok[kCombineBatch];
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      const int j = j0 + u;
      ok[u] = false;
      wj[u] = 0.0f;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (j < k) {
        const int64_t r = pos[t * k + j];
        if (r >= 0 && r < R) {
          ok[u] = true;
          wj[u] = w[t * k + j];
          v[u] = ldg_nc(yr + r * H + c * 8);
        } else if (c == 0) {
          set_status(status, W8A8_ERR_TOPK_IDS, static_cast<uint32_t>(t * k + j));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      if (!ok[u]) continue;
      const uint32_t x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        s[2 * i] = __fadd_rn(s[2 * i], __fmul_rn(wj[u], bf16_bits_to_f32(static_cast<uint16_t>(x[i] & 0xffffu))));
        s[2 * i + 1] = __fadd_rn(s[2 * i + 1], __fmul_rn(wj[u], bf16_bits_to_f32(static_cast<uint16_t>(x[i] >> 16))));
      }
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = static_cast<uint32_t>(f32_to_bf16_bits(s[2 * i])) | (static_cast<uint32_t>(f32_to_bf16_bits(s[2 * i + 1])) << 16);
  *reinterpret_cast<uint4*>(y + t * H + c * 8) = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

int64_t route_scratch_ints(int64_t n, int64_t E) { return E * route_blocks(n); }

cudaError_t launch_route(const int64_t* topk_ids, int64_t n, int E, int32_t* counts, int64_t* group_list,
                         int32_t* pos, DeviceStatus* status, cudaStream_t stream) {
  if (n == 0) return cudaMemsetAsync(group_list, 0, static_cast<size_t>(E) * sizeof(int64_t), stream);
  const int nb = static_cast<int>(route_blocks(n));
  const size_t smem = static_cast<size_t>(E) * sizeof(int32_t);
  cudaError_t e = launch_pdl(route_count, dim3(nb), dim3(32), smem, stream, topk_ids, n, E, nb, counts, status);
  if (e != cudaSuccess) return e;
  e = launch_pdl(route_scan, dim3(1), dim3(1024), 0, stream, counts, E, nb, group_list);
  if (e != cudaSuccess) return e;
  return launch_pdl(route_assign, dim3(nb), dim3(32), smem, stream, topk_ids, n, E, nb,
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
                           int64_t H, uint16_t* y, DeviceStatus* status, cudaStream_t stream) {
  const int64_t nslice = (H / 8 + kCombineThreads - 1) / kCombineThreads;
  const int64_t blocks = T * nslice;
  if (blocks == 0) return cudaSuccess;
  return launch_pdl(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kCombineThreads), 0, stream, y_routed,
                    pos, w, T, k, H, y, status);
}

}  // namespace w8a8
