// prepack.cu -- K0: load-time weight re-layout.
//
// Page "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子", §二: the INT8
// checkpoint weight [N,K] is transposed and format-cast once after loading and
// the result is reused by every forward (no per-forward re-quantisation).
// Page "Qwen3.8-FP8 on Ascend 950: Why Weights Become MXFP8 at Load Time",
// Deep Dive 4: repacked buffers are persistent so graph-captured addresses
// stay valid; Deep Dive 6: MoE stacks are prepared expert by expert.
//
// Packed buffer = 256-byte header, then the int8 payload [E,N,K] in packed row
// order (K contiguous: the K-major operand layout both MMA engines read), then
// optionally an integer-valued fp16 copy [E,N,K] for the tensor-core engine.
// Packed row order is the identity, or for W13 the gate/up interleave in
// blocks of 64 rows so that one 128-row tile holds gate channels j..j+63 and
// the matching up channels.  Pure copy: HBM-bound, one pass.
#include "kernels.cuh"

namespace w8a8 {

namespace {

__device__ __forceinline__ void write_header(uint8_t* packed, int64_t E, int64_t N, int64_t K, uint32_t flags,
                                             uint64_t i8_off, uint64_t f16_off) {
  PackedHeader hd;
  hd.magic = kPackMagic;
  hd.version = kPackVersion;
  hd.E = E;
  hd.N = N;
  hd.K = K;
  hd.flags = flags;
  hd.reserved = 0u;
  hd.i8_offset = i8_off;
  hd.f16_offset = f16_off;
  *reinterpret_cast<PackedHeader*>(packed) = hd;
}

// The header of a buffer whose payload the kernel before it wrote (the weight quantiser).  Launched
// without programmatic serialization and never letting its dependents start early: a contraction
// launched right after it reads the packed weights before its own wait, so it must start only after
// this kernel and, through stream order, the payload writer have completed.
__global__ void pack_header_kernel(int64_t E, int64_t N, int64_t K, uint32_t flags, uint8_t* packed, uint64_t i8_off,
                                   uint64_t f16_off) {
  write_header(packed, E, N, K, flags, i8_off, f16_off);
  __threadfence();
}

__global__ void __launch_bounds__(256) prepack_kernel(const int8_t* __restrict__ w, int64_t E, int64_t N,
                                                      int64_t K, uint32_t flags, uint8_t* __restrict__ packed,
                                                      uint64_t i8_off, uint64_t f16_off) {
  const int64_t chunks_per_row = K / 16;
  const int64_t total = E * N * chunks_per_row;
  const bool gate_up = (flags & W8A8_PACK_GATE_UP) != 0u;
  const int64_t I = N / 2;
  int8_t* dst8 = reinterpret_cast<int8_t*>(packed + i8_off);
  uint16_t* dst16 = f16_off ? reinterpret_cast<uint16_t*>(packed + f16_off) : nullptr;
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < total;
       c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = c / chunks_per_row;  // packed row over E*N
    const int64_t kc = c % chunks_per_row;
    const int64_t e = row / N;
    const int64_t p = row % N;
    const int64_t src_row = gate_up ? gate_up_orig_row(p, I) : p;
    const uint4 v = *reinterpret_cast<const uint4*>(w + (e * N + src_row) * K + kc * 16);
    *reinterpret_cast<uint4*>(dst8 + row * K + kc * 16) = v;
    if (dst16) {
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      uint32_t h[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) s8x4_to_f16x4(wv[i], h[2 * i], h[2 * i + 1]);
      uint4* d = reinterpret_cast<uint4*>(dst16 + row * K + kc * 16);
      d[0] = make_uint4(h[0], h[1], h[2], h[3]);
      d[1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) write_header(packed, E, N, K, flags, i8_off, f16_off);
  // A contraction launched right after this kernel with programmatic stream
  // serialization reads the packed weights before it waits for this grid.
  // This kernel never lets its dependents start early, so they start only
  // after every CTA has exited; each CTA's writes are made visible first.
  __threadfence();
}

}  // namespace

PackLayout pack_layout(int64_t E, int64_t N, int64_t K, uint32_t flags) {
  PackLayout L;
  L.i8_offset = kPackHeaderBytes;
  const uint64_t i8_bytes = static_cast<uint64_t>(E) * N * K;
  L.f16_offset = (flags & W8A8_PACK_F16) ? align_up(L.i8_offset + i8_bytes, 256) : 0;
  L.total = (flags & W8A8_PACK_F16) ? L.f16_offset + 2 * i8_bytes : L.i8_offset + i8_bytes;
  L.total = align_up(L.total, 256);
  return L;
}

cudaError_t launch_prepack(const int8_t* w, int64_t E, int64_t N, int64_t K, uint32_t flags, void* packed,
                           cudaStream_t stream, int num_sms) {
  const PackLayout L = pack_layout(E, N, K, flags);
  const int64_t total = E * N * (K / 16);
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(num_sms) * 16));
  prepack_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      w, E, N, K, flags, static_cast<uint8_t*>(packed), L.i8_offset, L.f16_offset);
  return cudaGetLastError();
}

cudaError_t launch_pack_header(int64_t E, int64_t N, int64_t K, uint32_t flags, void* packed, cudaStream_t stream) {
  const PackLayout L = pack_layout(E, N, K, flags);
  pack_header_kernel<<<1, 1, 0, stream>>>(E, N, K, flags, static_cast<uint8_t*>(packed), L.i8_offset, L.f16_offset);
  return cudaGetLastError();
}

}  // namespace w8a8
