// noalloc.cu -- w8a8_quant_matmul_noalloc: the dense quantised matmul for
// callers that cannot allocate device memory.
//
// Some callers have no way to obtain a device workspace: code running inside
// a plugin interface that hands out no allocator, hosts that reserved all of
// the GPU's memory up front for their own pools (serving engines that size
// their caches to the whole HBM), and code that must not call cudaMalloc
// because it would synchronise the device or is not allowed at that point.
// For them this entry point takes only inputs and outputs; the scratch the
// contraction needs (a status word, split-K partial sums and arrival counters)
// lives in a file-scope device array of fixed size that every GPU loading the
// library keeps until the process exits.
//
// Rules of use:
//   - the array holds kNoAllocScratchBytes: the status word, the arrival
//     counters and, when they fit (roughly M * N <= 2 million), the split-K
//     partial sums; larger problems run without splitting K, and only a
//     problem whose counters alone would not fit (M * N beyond about 2^31)
//     is rejected with W8A8_ERR_WORKSPACE before anything is launched;
//   - the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current and clears the status
//     word; make that first call before any stream capture;
//   - all calls share the one array and it keeps the last call's contents:
//     each call zeroes the arrival counters on its stream first, and the
//     partial sums are zero again after every call; calls that overlap on
//     the GPU (different streams, no ordering) race on the array;
//   - errors found on the device (a packed header that does not match the
//     call, an exhausted bounded wait) go to the array's status word, where
//     the first one stays until w8a8_quant_matmul_noalloc_status() reads and
//     clears it -- the same contract as a workspace's status word;
//   - nothing here allocates: no cudaMalloc, cudaFree or allocating library
//     routine is called.
#include <mutex>

#include "kernels.cuh"

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the array on the current device (looked up once per device, when the status word
// is also cleared).
w8a8_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return W8A8_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return W8A8_ERR_CUDA;
    if (cudaMemset(p, 0, w8a8::kStatusBytes) != cudaSuccess) return W8A8_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return W8A8_OK;
}

}  // namespace

using namespace w8a8;

extern "C" W8A8_API w8a8_status w8a8_quant_matmul_noalloc(const int8_t* q, const float* x_scale, int64_t M,
                                                          int64_t K, const void* w_packed, const float* w_scale,
                                                          int64_t N, const uint16_t* bias, uint16_t* y,
                                                          w8a8_stream_t stream) {
  if (M < 0 || M > INT32_MAX || N <= 0 || N > INT32_MAX) return W8A8_ERR_SHAPE;
  if (K <= 0 || K > W8A8_MAX_K) return W8A8_ERR_SHAPE;
  if (K % 16 != 0) return W8A8_ERR_ALIGN;
  if (M == 0) return W8A8_OK;
  if (!q || !x_scale || !w_packed || !w_scale || !y) return W8A8_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(w_packed) & 255u))
    return W8A8_ERR_ALIGN;

  // scratch layout: status word, one counter per output tile, partial sums [M,N] int32 (split-K) when they
  // fit; without room for them K is not split
  const size_t count_off = kStatusBytes;
  const int64_t count_len = ((M + 7) / 8) * ((N + 127) / 128);
  const size_t acc_off = count_off + align_up(static_cast<uint64_t>(count_len) * 4, 256);
  if (acc_off > kNoAllocScratchBytes) return W8A8_ERR_WORKSPACE;
  const bool split_room = acc_off + align_up(static_cast<uint64_t>(M) * N * 4, 256) <= kNoAllocScratchBytes;

  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return W8A8_ERR_CUDA;
  if (major != 10 || minor != 3) return W8A8_ERR_UNSUPPORTED;

  void* base = nullptr;
  if (w8a8_status s = scratch_address(&base)) return s;
  uint8_t* b = static_cast<uint8_t*>(base);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // what must start at zero: the arrival counters (the status word keeps the first error until it is read)
  if (cudaMemsetAsync(b + count_off, 0, static_cast<size_t>(count_len) * 4, st) != cudaSuccess)
    return W8A8_ERR_CUDA;

  GemmArgs a;
  a.q = q;
  a.x_scale = x_scale;
  a.group_list = nullptr;
  a.E = 1;
  a.R = M;
  a.K = K;
  a.N = N;
  a.packed = w_packed;
  a.pack_flags = 0u;
  a.w_scale = w_scale;
  a.bias = bias;
  a.out = y;
  a.mode = EPI_BF16;
  a.status = reinterpret_cast<DeviceStatus*>(b);
  a.ws_acc = split_room ? reinterpret_cast<int32_t*>(b + acc_off) : nullptr;  // nullptr: the plan keeps K whole
  a.ws_count = reinterpret_cast<uint32_t*>(b + count_off);
  a.ws_count_len = count_len;
  const GemmPlan p = plan_reg_gemm(a, sms);
  return launch_reg_gemm(a, p, st) == cudaSuccess ? W8A8_OK : W8A8_ERR_CUDA;
}

extern "C" W8A8_API w8a8_status w8a8_quant_matmul_noalloc_status(w8a8_stream_t stream) {
  void* base = nullptr;
  if (w8a8_status s = scratch_address(&base)) return s;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return W8A8_ERR_CUDA;
  DeviceStatus s;
  if (cudaMemcpyFromSymbol(&s, g_noalloc_scratch, sizeof(s)) != cudaSuccess) return W8A8_ERR_CUDA;
  if (s.code != 0u) {
    const DeviceStatus zero = {};
    if (cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof(zero)) != cudaSuccess) return W8A8_ERR_CUDA;
  }
  return static_cast<w8a8_status>(s.code);
}
