// capi.cu -- the extern "C" boundary of libw8a8.so (declared in include/w8a8.h).
//
// Host side only: argument validation (errors returned before any launch, in
// the spirit of the error table of page "Qwen3.8-FP8 on Ascend 950: Why
// Weights Become MXFP8 at Load Time", "Where It Breaks or Falls Back", but
// with no fallback path), workspace layouts, tile-plan choice (decode- vs
// prefill-sized tiles, as the operator host of page "DeepSeek-V4 W8A8 执行链
// 从量化权重到 Ascend INT8 算子" §四 picks a tiling per M/N/K) and stream-ordered
// launches.  Nothing here allocates or synchronises except
// w8a8_read_device_status().
#include <cstring>
#include <mutex>

#include "kernels.cuh"

using namespace w8a8;

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxE = 1024;

struct DevInfo {
  int sms = 0;
  int supported = -1;  // -1 unknown, 0 no, 1 yes
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

w8a8_status device_info(int& sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return W8A8_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.supported < 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return W8A8_ERR_CUDA;
    d.supported = (major == 10 && minor == 3) ? 1 : 0;
  }
  if (!d.supported) return W8A8_ERR_UNSUPPORTED;
  sms = d.sms;
  return W8A8_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0u; }
inline w8a8_status cuda_status(cudaError_t e) { return e == cudaSuccess ? W8A8_OK : W8A8_ERR_CUDA; }

// Shapes that go to the tcgen05 engine (the tiling choice by M of page
// "DeepSeek-V4 W8A8 执行链从量化权重到 Ascend INT8 算子" §四: prefill vs decode).
constexpr int64_t kTcMinM = 128;           // dense rows
constexpr int64_t kTcMinRowsPerGroup = 64;  // grouped: average rows per expert

bool tc_shape(int64_t E, int64_t R) {
  return E <= 1 ? R >= kTcMinM : R >= kTcMinRowsPerGroup * E;
}

// Host record of the packed buffers this process made, so a call can tell
// (without reading device memory) whether a buffer carries the fp16 copy the
// tcgen05 engine reads.  Buffers not found here use the warp-level engine.
struct PackRecord {
  const void* ptr;
  int64_t E, N, K;
  uint32_t flags;
};
constexpr int kMaxPackRecords = 4096;
PackRecord g_packs[kMaxPackRecords];
int g_npacks = 0;
int g_pack_next = 0;
std::mutex g_pack_mu;

void record_pack(const void* ptr, int64_t E, int64_t N, int64_t K, uint32_t flags) {
  std::lock_guard<std::mutex> lk(g_pack_mu);
  for (int i = 0; i < g_npacks; ++i)
    if (g_packs[i].ptr == ptr) {
      g_packs[i] = PackRecord{ptr, E, N, K, flags};
      return;
    }
  if (g_npacks < kMaxPackRecords) {
    g_packs[g_npacks++] = PackRecord{ptr, E, N, K, flags};
  } else {
    g_packs[g_pack_next] = PackRecord{ptr, E, N, K, flags};
    g_pack_next = (g_pack_next + 1) % kMaxPackRecords;
  }
}

// Device address of the fp16 copy of a packed buffer, or nullptr.
const void* pack_f16(const void* ptr, int64_t E, int64_t N, int64_t K, uint32_t need_flags) {
  std::lock_guard<std::mutex> lk(g_pack_mu);
  for (int i = 0; i < g_npacks; ++i) {
    const PackRecord& r = g_packs[i];
    if (r.ptr == ptr && r.E == E && r.N == N && r.K == K && (r.flags & W8A8_PACK_F16) &&
        (r.flags & W8A8_PACK_GATE_UP) == (need_flags & W8A8_PACK_GATE_UP))
      return static_cast<const uint8_t*>(ptr) + pack_layout(E, N, K, r.flags).f16_offset;
  }
  return nullptr;
}

// True when this process packed `ptr` itself with these sizes and gate/up order.
bool pack_recorded(const void* ptr, int64_t E, int64_t N, int64_t K, uint32_t need_flags) {
  std::lock_guard<std::mutex> lk(g_pack_mu);
  for (int i = 0; i < g_npacks; ++i) {
    const PackRecord& r = g_packs[i];
    if (r.ptr == ptr && r.E == E && r.N == N && r.K == K &&
        (r.flags & W8A8_PACK_GATE_UP) == (need_flags & W8A8_PACK_GATE_UP))
      return true;
  }
  return false;
}

w8a8_status check_k(int64_t K) {
  if (K <= 0 || K > W8A8_MAX_K) return W8A8_ERR_SHAPE;
  if (K % 16 != 0) return W8A8_ERR_ALIGN;
  return W8A8_OK;
}

// Workspace of one contraction: status word, split-K partials + counters, and
// (for shapes the tcgen05 engine takes) the activations as fp16.
struct GemmWs {
  size_t status = 0, acc = 0, count = 0, a16 = 0, dec = 0, total = 0;
  int64_t count_len = 0;
};
GemmWs gemm_ws_layout(int64_t E, int64_t R, int64_t N, int64_t K, bool with_a16 = true) {
  GemmWs L;
  L.status = 0;
  L.acc = kStatusBytes;
  const size_t acc_bytes = align_up(static_cast<uint64_t>(R) * N * 4, 256);
  L.count = L.acc + acc_bytes;
  const int64_t nb = (N + 127) / 128;
  L.count_len = ((R + 7) / 8 + (E > 1 ? E : 0)) * nb;
  L.a16 = L.count + align_up(static_cast<uint64_t>(L.count_len) * 4, 256);
  L.dec = L.a16 + ((with_a16 && tc_shape(E, R)) ? align_up(static_cast<uint64_t>(R) * K * 2, 256) : 0);
  // decode engine (dense, at most 64 rows): split-K partial tiles + counters
  L.total = L.dec + ((with_a16 && E <= 1 && R <= 64) ? dec_ws_bytes(N) : 0);
  return L;
}

void bind_ws(GemmArgs& a, void* ws, const GemmWs& L) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  a.status = reinterpret_cast<DeviceStatus*>(b + L.status);
  a.ws_acc = reinterpret_cast<int32_t*>(b + L.acc);
  a.ws_count = reinterpret_cast<uint32_t*>(b + L.count);
  a.ws_count_len = L.count_len;
}

struct MoeWs {
  size_t xq, xs, h, hq, hs, xq16, hq16, gemm, total;
  GemmWs g;
};
// The codes of the routed rows and of h: int8 for the warp engine, or on shapes the tensor-core engines
// take only as the integer-valued fp16 they read (xq16, hq16; xq and hq are then 0: not kept).
MoeWs moe_layout(int64_t R, int64_t H, int64_t I, int64_t E) {
  MoeWs L;
  const bool tc = tc_shape(E, R);
  size_t off = kStatusBytes;
  L.xq = L.hq = L.xq16 = L.hq16 = 0;
  if (!tc) { L.xq = off; off = align_up(off + static_cast<uint64_t>(R) * H, 256); }
  L.xs = off; off = align_up(off + static_cast<uint64_t>(R) * 4, 256);
  L.h = off;  off = align_up(off + static_cast<uint64_t>(R) * I * 2, 256);
  if (!tc) { L.hq = off; off = align_up(off + static_cast<uint64_t>(R) * I, 256); }
  L.hs = off; off = align_up(off + static_cast<uint64_t>(R) * 4, 256);
  if (tc) {
    L.xq16 = off; off = align_up(off + static_cast<uint64_t>(R) * H * 2, 256);
    L.hq16 = off; off = align_up(off + static_cast<uint64_t>(R) * I * 2, 256);
  }
  // one split-K region serves both contractions (they run one after the other);
  // the fp16 activations of the tcgen05 engine live in xq16 / hq16 instead
  const GemmWs g13 = gemm_ws_layout(E, R, 2 * I, H, false);
  const GemmWs g2 = gemm_ws_layout(E, R, H, I, false);
  L.g = g13.total >= g2.total ? g13 : g2;
  L.gemm = off;
  L.total = off + L.g.total;
  return L;
}

// Workspace of the MoE layer from token rows: the expert chain's workspace first (its status word is
// the layer's), then the routing results, the routing scratch and the chain's routed output.
struct LayerWs {
  MoeWs m;
  size_t group_list, pos, counts, y_routed, total;
};
LayerWs layer_layout(int64_t T, int64_t k, int64_t H, int64_t I, int64_t E) {
  LayerWs L;
  const int64_t R = T * k;
  L.m = moe_layout(R, H, I, E);
  size_t off = align_up(L.m.total, 256);
  L.group_list = off; off = align_up(off + static_cast<uint64_t>(E) * 8, 256);
  L.pos = off;        off = align_up(off + static_cast<uint64_t>(R) * 4, 256);
  L.counts = off;     off = align_up(off + static_cast<uint64_t>(route_scratch_ints(R, E)) * 4, 256);
  L.y_routed = off;   off = align_up(off + static_cast<uint64_t>(R) * H * 2, 256);
  L.total = off;
  return L;
}

// Sizes shared by the routing calls: T tokens with k choices each, R = T*k routed rows.
w8a8_status check_route_shape(int64_t T, int64_t k, int64_t E) {
  if (T < 0 || k < 1 || k > INT32_MAX || E < 1 || E > kMaxE) return W8A8_ERR_SHAPE;
  if (T > 0 && k > INT32_MAX / T) return W8A8_ERR_SHAPE;
  return W8A8_OK;
}

// The combine numbers its work items (token, 1024 columns) with 32-bit integers.
bool combine_grid_ok(int64_t T, int64_t H) { return T * ((H / 8 + 127) / 128) <= INT32_MAX; }

// One contraction on the engine its shape calls for: tcgen05 (activations
// widened to fp16 in the workspace) when the shape is large and the weight
// carries its fp16 copy, else the warp-level engine.
thread_local int t_last_engine = W8A8_ENGINE_NONE;

w8a8_status run_gemm(GemmArgs a, void* ws, const GemmWs& L, cudaStream_t stream, int sms) {
  bind_ws(a, ws, L);
  a.status = static_cast<DeviceStatus*>(ws);
  // the workspace holds an fp16 copy of the codes only for shapes a tensor-core engine takes
  const bool tc_rows = L.dec > L.a16;
  uint16_t* a16 = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + L.a16);
  const void* b16 = tc_rows ? pack_f16(a.packed, a.E, a.N, a.K, a.pack_flags) : nullptr;
  if (b16 != nullptr) {  // the packed fp16 weight copy (CTA pairs, dense or grouped)
    if (w8a8_status e = cuda_status(launch_s8_to_f16(a.q, a16, a.R * a.K, stream, sms))) return e;
    t_last_engine = W8A8_ENGINE_TC;
    return cuda_status(launch_tc_gemm(a, a16, b16, sms, stream));
  }
  if (tc_rows) {  // without the fp16 copy: CTA pairs with the int8 weights widened in TMEM (dense or grouped)
    if (w8a8_status e = cuda_status(launch_s8_to_f16(a.q, a16, a.R * a.K, stream, sms))) return e;
    t_last_engine = W8A8_ENGINE_TC_I8;
    return cuda_status(launch_tcp_gemm(a, a16, sms, stream));
  }
  if (a.group_list == nullptr && a.mode != EPI_SWIGLU && L.dec < L.total) {
    const DecPlan dp = dec_plan(a.R, a.N, a.K, sms);  // dense decode: int8 weights widened in TMEM
    if (dp.ksplit > 0) {
      a.pack_known = pack_recorded(a.packed, a.E, a.N, a.K, a.pack_flags) ? 1 : 0;
      t_last_engine = W8A8_ENGINE_DECODE;
      return cuda_status(launch_dec_gemm(a, dp, static_cast<uint8_t*>(ws) + L.dec, stream));
    }
  }
  t_last_engine = W8A8_ENGINE_WARP;
  const GemmPlan p = plan_reg_gemm(a, sms);
  return cuda_status(launch_reg_gemm(a, p, stream));
}

// The expert chain on routed rows (workspace laid out by moe_layout at `ws`).  x16_ready: the routed
// codes are already in the workspace's fp16 copy (the layer's permute wrote them there), so an INT8
// input is not widened again.
w8a8_status moe_chain(const void* x, const float* x_scale, bool x16_ready, const int64_t* group_list, int64_t E,
                      int64_t R, int64_t H, int64_t I, const void* w13_packed, const float* w13_scale,
                      const void* w2_packed, const float* w2_scale, void* ws, uint16_t* y, cudaStream_t st,
                      int sms) {
  const MoeWs L = moe_layout(R, H, I, E);
  uint8_t* b = static_cast<uint8_t*>(ws);
  void* gws = b + L.gemm;

  const int8_t* xq = static_cast<const int8_t*>(x);
  const float* xs = x_scale;
  uint16_t* h = reinterpret_cast<uint16_t*>(b + L.h);
  int8_t* hq = L.hq ? reinterpret_cast<int8_t*>(b + L.hq) : nullptr;  // warp engine only
  float* hs = reinterpret_cast<float*>(b + L.hs);
  // tensor-core engines for shapes that take them: the packed fp16 weight copies when both packs carry
  // them, else the int8 weights widened in tensor memory
  const bool tc = L.xq16 != 0;
  const void* w13_16 = tc ? pack_f16(w13_packed, E, 2 * I, H, W8A8_PACK_GATE_UP) : nullptr;
  const void* w2_16 = tc ? pack_f16(w2_packed, E, H, I, 0u) : nullptr;
  const bool f16w = w13_16 != nullptr && w2_16 != nullptr;
  uint16_t* xq16 = tc ? reinterpret_cast<uint16_t*>(b + L.xq16) : nullptr;
  uint16_t* hq16 = tc ? reinterpret_cast<uint16_t*>(b + L.hq16) : nullptr;

  if (x_scale == nullptr) {  // BF16 input: quantise once; an INT8 input with its scale is used as is
    float* s = reinterpret_cast<float*>(b + L.xs);
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    int8_t* q = tc ? nullptr : reinterpret_cast<int8_t*>(b + L.xq);
    const cudaError_t e = tc ? launch_dynamic_quant_f16(xb, R, H, xq16, s, st, sms)
                             : launch_dynamic_quant(xb, R, H, q, s, st, sms);
    if (e != cudaSuccess) return W8A8_ERR_CUDA;
    xq = q;
    xs = s;
  } else if (tc && !x16_ready) {
    if (w8a8_status e = cuda_status(launch_s8_to_f16(xq, xq16, R * H, st, sms))) return e;
  }

  GemmArgs a13;
  a13.q = xq;
  a13.x_scale = xs;
  a13.group_list = group_list;
  a13.E = E;
  a13.R = R;
  a13.K = H;
  a13.N = 2 * I;
  a13.packed = w13_packed;
  a13.pack_flags = W8A8_PACK_GATE_UP;
  a13.w_scale = w13_scale;
  a13.out = h;
  a13.mode = EPI_SWIGLU;
  bind_ws(a13, gws, L.g);
  a13.status = static_cast<DeviceStatus*>(ws);
  const cudaError_t e13 = f16w ? launch_tc_gemm(a13, xq16, w13_16, sms, st)
                         : tc ? launch_tcp_gemm(a13, xq16, sms, st)
                             : launch_reg_gemm(a13, plan_reg_gemm(a13, sms), st);
  if (e13 != cudaSuccess) return W8A8_ERR_CUDA;

  const cudaError_t eq = tc ? launch_dynamic_quant_f16(h, R, I, hq16, hs, st, sms)
                            : launch_dynamic_quant(h, R, I, hq, hs, st, sms);
  if (eq != cudaSuccess) return W8A8_ERR_CUDA;

  GemmArgs a2;
  a2.q = hq;
  a2.x_scale = hs;
  a2.group_list = group_list;
  a2.E = E;
  a2.R = R;
  a2.K = I;
  a2.N = H;
  a2.packed = w2_packed;
  a2.pack_flags = 0u;
  a2.w_scale = w2_scale;
  a2.out = y;
  a2.mode = EPI_BF16;
  bind_ws(a2, gws, L.g);
  a2.status = static_cast<DeviceStatus*>(ws);
  const cudaError_t e2 = f16w ? launch_tc_gemm(a2, hq16, w2_16, sms, st)
                        : tc ? launch_tcp_gemm(a2, hq16, sms, st)
                            : launch_reg_gemm(a2, plan_reg_gemm(a2, sms), st);
  t_last_engine = f16w ? W8A8_ENGINE_TC : tc ? W8A8_ENGINE_TC_I8 : W8A8_ENGINE_WARP;
  return e2 == cudaSuccess ? W8A8_OK : W8A8_ERR_CUDA;
}


}  // namespace

extern "C" {

const char* w8a8_status_string(int s) {
  switch (s) {
    case W8A8_OK: return "W8A8_OK";
    case W8A8_ERR_NULL: return "W8A8_ERR_NULL: a required pointer is NULL";
    case W8A8_ERR_SHAPE: return "W8A8_ERR_SHAPE: a size is out of range";
    case W8A8_ERR_ALIGN: return "W8A8_ERR_ALIGN: K % 16 != 0 or a pointer is not 16-byte aligned";
    case W8A8_ERR_WORKSPACE: return "W8A8_ERR_WORKSPACE: workspace missing or too small";
    case W8A8_ERR_GROUP_LIST: return "W8A8_ERR_GROUP_LIST: group_list has a negative count or does not sum to R";
    case W8A8_ERR_DEVICE_TIMEOUT: return "W8A8_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
    case W8A8_ERR_CUDA: return "W8A8_ERR_CUDA: a CUDA runtime call failed";
    case W8A8_ERR_UNSUPPORTED: return "W8A8_ERR_UNSUPPORTED: needs a compute capability 10.3 (GB300) device";
    case W8A8_ERR_PACKED: return "W8A8_ERR_PACKED: packed weight header does not match the call";
    case W8A8_ERR_TOPK_IDS: return "W8A8_ERR_TOPK_IDS: a topk id outside [0,E) or a routed row index outside [0,T*k)";
    default: return "W8A8 unknown status";
  }
}

int w8a8_version(void) { return 100; }

size_t w8a8_prepacked_bytes(int64_t E, int64_t N, int64_t K, uint32_t flags) {
  if (E <= 0 || N <= 0 || K <= 0) return 0;
  return pack_layout(E, N, K, flags).total;
}

w8a8_status w8a8_prepack_weight(const int8_t* w, int64_t E, int64_t N, int64_t K, uint32_t flags,
                                void* packed, w8a8_stream_t stream) {
  if (!w || !packed) return W8A8_ERR_NULL;
  if (E <= 0 || N <= 0 || E > kMaxE) return W8A8_ERR_SHAPE;
  if (w8a8_status s = check_k(K)) return s;
  if (flags & ~(W8A8_PACK_GATE_UP | W8A8_PACK_F16)) return W8A8_ERR_SHAPE;
  if ((flags & W8A8_PACK_GATE_UP) && (N % 2 != 0 || (N / 2) % kGateUpBlock != 0)) return W8A8_ERR_SHAPE;
  if (!aligned16(w) || (reinterpret_cast<uintptr_t>(packed) & 255u)) return W8A8_ERR_ALIGN;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
  const w8a8_status st =
      cuda_status(launch_prepack(w, E, N, K, flags, packed, reinterpret_cast<cudaStream_t>(stream), sms));
  if (st == W8A8_OK) record_pack(packed, E, N, K, flags);
  return st;
}

w8a8_status w8a8_quantize_weight(const uint16_t* w, int64_t E, int64_t N, int64_t K, int8_t* q, float* scale,
                                 w8a8_stream_t stream) {
  if (!w || !q || !scale) return W8A8_ERR_NULL;
  if (E <= 0 || N <= 0 || E > kMaxE || N > INT32_MAX || E * N > INT32_MAX) return W8A8_ERR_SHAPE;
  if (w8a8_status s = check_k(K)) return s;
  if (!aligned16(w) || !aligned16(q)) return W8A8_ERR_ALIGN;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
  return cuda_status(launch_dynamic_quant(w, E * N, K, q, scale, reinterpret_cast<cudaStream_t>(stream), sms));
}

w8a8_status w8a8_quantize_prepack_weight(const uint16_t* w, int64_t E, int64_t N, int64_t K, uint32_t flags,
                                         void* packed, float* scale, w8a8_stream_t stream) {
  if (!w || !packed || !scale) return W8A8_ERR_NULL;
  if (E <= 0 || N <= 0 || E > kMaxE || N > INT32_MAX || E * N > INT32_MAX) return W8A8_ERR_SHAPE;
  if (w8a8_status s = check_k(K)) return s;
  if (flags & ~(W8A8_PACK_GATE_UP | W8A8_PACK_F16)) return W8A8_ERR_SHAPE;
  if ((flags & W8A8_PACK_GATE_UP) && (N % 2 != 0 || (N / 2) % kGateUpBlock != 0)) return W8A8_ERR_SHAPE;
  if (!aligned16(w) || (reinterpret_cast<uintptr_t>(packed) & 255u)) return W8A8_ERR_ALIGN;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
  const w8a8_status st = cuda_status(
      launch_quant_pack(w, E, N, K, flags, packed, scale, reinterpret_cast<cudaStream_t>(stream), sms));
  if (st == W8A8_OK) record_pack(packed, E, N, K, flags);
  return st;
}

w8a8_status w8a8_dynamic_quant(const uint16_t* x, int64_t M, int64_t K, int8_t* q, float* scale,
                               w8a8_stream_t stream) {
  if (M < 0 || M > INT32_MAX) return W8A8_ERR_SHAPE;
  if (w8a8_status s = check_k(K)) return s;
  if (M == 0) return W8A8_OK;
  if (!x || !q || !scale) return W8A8_ERR_NULL;
  if (!aligned16(x) || !aligned16(q)) return W8A8_ERR_ALIGN;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
  return cuda_status(launch_dynamic_quant(x, M, K, q, scale, reinterpret_cast<cudaStream_t>(stream), sms));
}

size_t w8a8_quant_matmul_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N <= 0 || K <= 0) return 0;
  return gemm_ws_layout(1, M, N, K).total;
}

static w8a8_status dense_common(const int8_t* q, const float* x_scale, int64_t M, int64_t K, const void* w_packed,
                                const float* w_scale, int64_t N, const uint16_t* bias, void* out, int mode,
                                void* ws, size_t ws_bytes, w8a8_stream_t stream, const int32_t* qbias = nullptr) {
  if (M < 0 || M > INT32_MAX || N <= 0 || N > INT32_MAX) return W8A8_ERR_SHAPE;
  if (w8a8_status s = check_k(K)) return s;
  if (M == 0) return W8A8_OK;
  if (!q || !w_packed || !out || !ws) return (!ws && q && w_packed && out) ? W8A8_ERR_WORKSPACE : W8A8_ERR_NULL;
  if (mode == EPI_BF16 && (!w_scale || (!x_scale && !qbias))) return W8A8_ERR_NULL;
  if (!aligned16(q) || (reinterpret_cast<uintptr_t>(w_packed) & 255u)) return W8A8_ERR_ALIGN;
  const GemmWs L = gemm_ws_layout(1, M, N, K);
  if (ws_bytes < L.total || !aligned16(ws)) return W8A8_ERR_WORKSPACE;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
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
  a.qbias = qbias;
  a.out = out;
  a.mode = mode;
  return run_gemm(a, ws, L, reinterpret_cast<cudaStream_t>(stream), sms);
}

w8a8_status w8a8_quant_matmul(const int8_t* q, const float* x_scale, int64_t M, int64_t K, const void* w_packed,
                              const float* w_scale, int64_t N, const uint16_t* bias, uint16_t* y, void* ws,
                              size_t ws_bytes, w8a8_stream_t stream) {
  return dense_common(q, x_scale, M, K, w_packed, w_scale, N, bias, y, EPI_BF16, ws, ws_bytes, stream);
}

w8a8_status w8a8_int8_matmul_acc(const int8_t* q, int64_t M, int64_t K, const void* w_packed, int64_t N,
                                 int32_t* acc, void* ws, size_t ws_bytes, w8a8_stream_t stream) {
  return dense_common(q, nullptr, M, K, w_packed, nullptr, N, nullptr, acc, EPI_ACC, ws, ws_bytes, stream);
}

w8a8_status w8a8_mx_quant(const uint16_t* x, int64_t M, int64_t K, uint8_t* q, uint8_t* scale,
                          w8a8_stream_t stream) {
  if (M < 0 || M > INT32_MAX || K <= 0 || K > W8A8_MAX_K) return W8A8_ERR_SHAPE;
  if (K % 32 != 0) return W8A8_ERR_ALIGN;
  if (M == 0) return W8A8_OK;
  if (!x || !q || !scale) return W8A8_ERR_NULL;
  if (!aligned16(x) || !aligned16(q)) return W8A8_ERR_ALIGN;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
  return cuda_status(launch_mx_quant(x, M, K, q, scale, reinterpret_cast<cudaStream_t>(stream), sms));
}

w8a8_status w8a8_mx_matmul(const uint8_t* qa, const uint8_t* sa, int64_t M, int64_t K, const uint8_t* qw,
                           const uint8_t* sw, int64_t N, uint16_t* y, w8a8_stream_t stream) {
  if (M < 0 || M > INT32_MAX || N <= 0 || N > INT32_MAX || K <= 0 || K > W8A8_MAX_K) return W8A8_ERR_SHAPE;
  if (K % 128 != 0) return W8A8_ERR_ALIGN;
  if (M == 0) return W8A8_OK;
  if (!qa || !sa || !qw || !sw || !y) return W8A8_ERR_NULL;
  if (!aligned16(qa) || !aligned16(qw) || !aligned16(sa) || !aligned16(sw)) return W8A8_ERR_ALIGN;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
  if (mx_tc_supported(M, N, K)) {  // block-scaled tensor cores
    t_last_engine = W8A8_ENGINE_TC;
    return cuda_status(launch_mx_tc(qa, sa, M, K, qw, sw, N, y, nullptr, sms, reinterpret_cast<cudaStream_t>(stream)));
  }
  t_last_engine = W8A8_ENGINE_WARP;
  return cuda_status(launch_mx_matmul(qa, sa, M, K, qw, sw, N, y, reinterpret_cast<cudaStream_t>(stream)));
}

static bool static_params_ok(float s, int32_t o) { return s > 0.0f && s < 3.0e38f && o >= -128 && o <= 127; }

w8a8_status w8a8_static_quant(const uint16_t* x, int64_t M, int64_t K, float input_scale, int32_t input_offset,
                              int8_t* q, w8a8_stream_t stream) {
  if (M < 0 || M > INT32_MAX || !static_params_ok(input_scale, input_offset)) return W8A8_ERR_SHAPE;
  if (w8a8_status s = check_k(K)) return s;
  if (M == 0) return W8A8_OK;
  if (!x || !q) return W8A8_ERR_NULL;
  if (!aligned16(x) || !aligned16(q)) return W8A8_ERR_ALIGN;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
  return cuda_status(launch_static_quant(x, M, K, input_scale, input_offset, q, reinterpret_cast<cudaStream_t>(stream),
                                         sms));
}

w8a8_status w8a8_static_prepare(const int8_t* w, int64_t N, int64_t K, const float* w_scale, float input_scale,
                                int32_t input_offset, const uint16_t* bias, float* deq_scale, int32_t* quant_bias,
                                w8a8_stream_t stream) {
  if (N <= 0 || N > INT32_MAX || !static_params_ok(input_scale, input_offset)) return W8A8_ERR_SHAPE;
  if (w8a8_status s = check_k(K)) return s;
  if (!w || !w_scale || !deq_scale || !quant_bias) return W8A8_ERR_NULL;
  if (!aligned16(w)) return W8A8_ERR_ALIGN;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
  return cuda_status(launch_static_prepare(w, N, K, w_scale, input_scale, input_offset, bias, deq_scale, quant_bias,
                                           reinterpret_cast<cudaStream_t>(stream), sms));
}

w8a8_status w8a8_static_quant_matmul(const int8_t* q, int64_t M, int64_t K, const void* w_packed,
                                     const float* deq_scale, const int32_t* quant_bias, int64_t N, uint16_t* y,
                                     void* ws, size_t ws_bytes, w8a8_stream_t stream) {
  if (M > 0 && !quant_bias) return W8A8_ERR_NULL;
  return dense_common(q, nullptr, M, K, w_packed, deq_scale, N, nullptr, y, EPI_BF16, ws, ws_bytes, stream,
                      quant_bias);
}

size_t w8a8_grouped_matmul_workspace_bytes(int64_t E, int64_t R, int64_t N, int64_t K) {
  if (E <= 0 || R < 0 || N <= 0 || K <= 0) return 0;
  return gemm_ws_layout(E, R, N, K).total;
}

static w8a8_status grouped_common(const int8_t* q, const float* x_scale, const int64_t* group_list, int64_t E,
                                  int64_t R, int64_t K, const void* w_packed, const float* w_scale, int64_t N,
                                  void* out, int mode, void* ws, size_t ws_bytes, w8a8_stream_t stream) {
  if (E <= 0 || E > kMaxE || R < 0 || R > INT32_MAX || N <= 0 || N > INT32_MAX) return W8A8_ERR_SHAPE;
  if (w8a8_status s = check_k(K)) return s;
  if (R == 0) return W8A8_OK;
  if (!q || !group_list || !w_packed || !out) return W8A8_ERR_NULL;
  if (mode == EPI_BF16 && (!x_scale || !w_scale)) return W8A8_ERR_NULL;
  if (!ws) return W8A8_ERR_WORKSPACE;
  if (!aligned16(q) || (reinterpret_cast<uintptr_t>(w_packed) & 255u)) return W8A8_ERR_ALIGN;
  const GemmWs L = gemm_ws_layout(E, R, N, K);
  if (ws_bytes < L.total || !aligned16(ws)) return W8A8_ERR_WORKSPACE;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
  GemmArgs a;
  a.q = q;
  a.x_scale = x_scale;
  a.group_list = group_list;
  a.E = E;
  a.R = R;
  a.K = K;
  a.N = N;
  a.packed = w_packed;
  a.pack_flags = 0u;
  a.w_scale = w_scale;
  a.out = out;
  a.mode = mode;
  return run_gemm(a, ws, L, reinterpret_cast<cudaStream_t>(stream), sms);
}

w8a8_status w8a8_grouped_matmul(const int8_t* q, const float* x_scale, const int64_t* group_list, int64_t E,
                                int64_t R, int64_t K, const void* w_packed, const float* w_scale, int64_t N,
                                uint16_t* y, void* ws, size_t ws_bytes, w8a8_stream_t stream) {
  return grouped_common(q, x_scale, group_list, E, R, K, w_packed, w_scale, N, y, EPI_BF16, ws, ws_bytes, stream);
}

w8a8_status w8a8_grouped_matmul_acc(const int8_t* q, const int64_t* group_list, int64_t E, int64_t R, int64_t K,
                                    const void* w_packed, int64_t N, int32_t* acc, void* ws, size_t ws_bytes,
                                    w8a8_stream_t stream) {
  return grouped_common(q, nullptr, group_list, E, R, K, w_packed, nullptr, N, acc, EPI_ACC, ws, ws_bytes, stream);
}

size_t moe_workspace_bytes(int64_t R, int64_t H, int64_t I, int64_t E) {
  if (R < 0 || H <= 0 || I <= 0 || E <= 0) return 0;
  return moe_layout(R, H, I, E).total;
}

int64_t moe_workspace_offset(int64_t R, int64_t H, int64_t I, int64_t E, int which) {
  if (R < 0 || H <= 0 || I <= 0 || E <= 0) return -1;
  const MoeWs L = moe_layout(R, H, I, E);
  switch (which) {
    case 0: return L.xq ? static_cast<int64_t>(L.xq) : -1;
    case 1: return static_cast<int64_t>(L.xs);
    case 2: return static_cast<int64_t>(L.h);
    case 3: return L.hq ? static_cast<int64_t>(L.hq) : -1;
    case 4: return static_cast<int64_t>(L.hs);
    case 5: return L.xq16 ? static_cast<int64_t>(L.xq16) : -1;
    case 6: return L.hq16 ? static_cast<int64_t>(L.hq16) : -1;
    default: return -1;
  }
}

w8a8_status moe_w13_swiglu_requant_w2(const void* x, const float* x_scale, const int64_t* group_list, int64_t E,
                                      int64_t R, int64_t H, int64_t I, const void* w13_packed,
                                      const float* w13_scale, const void* w2_packed, const float* w2_scale,
                                      void* ws, size_t ws_bytes, uint16_t* y, w8a8_stream_t stream) {
  if (E <= 0 || E > kMaxE || R < 0 || R > INT32_MAX || H <= 0 || I <= 0) return W8A8_ERR_SHAPE;
  if (w8a8_status s = check_k(H)) return s;
  if (w8a8_status s = check_k(I)) return s;
  if (I % kGateUpBlock != 0) return W8A8_ERR_SHAPE;
  if (R == 0) return W8A8_OK;
  if (!x || !group_list || !w13_packed || !w13_scale || !w2_packed || !w2_scale || !y) return W8A8_ERR_NULL;
  if (!ws) return W8A8_ERR_WORKSPACE;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(w13_packed) & 255u) ||
      (reinterpret_cast<uintptr_t>(w2_packed) & 255u))
    return W8A8_ERR_ALIGN;
  const MoeWs L = moe_layout(R, H, I, E);
  if (ws_bytes < L.total || !aligned16(ws)) return W8A8_ERR_WORKSPACE;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
  return moe_chain(x, x_scale, false, group_list, E, R, H, I, w13_packed, w13_scale, w2_packed, w2_scale, ws, y,
                   reinterpret_cast<cudaStream_t>(stream), sms);
}

size_t moe_route_workspace_bytes(int64_t T, int64_t k, int64_t E) {
  if (check_route_shape(T, k, E) != W8A8_OK) return 0;
  return kStatusBytes + align_up(static_cast<uint64_t>(route_scratch_ints(T * k, E)) * 4, 256);
}

w8a8_status moe_permute_quant(const void* x, const float* x_scale, const int64_t* topk_ids, int64_t T, int64_t k,
                              int64_t E, int64_t H, int8_t* xq, float* xs, int64_t* group_list, int32_t* pos,
                              void* ws, size_t ws_bytes, w8a8_stream_t stream) {
  if (w8a8_status s = check_route_shape(T, k, E)) return s;
  if (H <= 0 || H > INT32_MAX) return W8A8_ERR_SHAPE;
  if (H % 16 != 0) return W8A8_ERR_ALIGN;
  if (!group_list) return W8A8_ERR_NULL;
  if (!ws) return W8A8_ERR_WORKSPACE;
  if (T > 0 && (!x || !topk_ids || !xq || !xs || !pos)) return W8A8_ERR_NULL;
  if (!aligned16(x) || !aligned16(xq)) return W8A8_ERR_ALIGN;
  if (ws_bytes < moe_route_workspace_bytes(T, k, E) || !aligned16(ws)) return W8A8_ERR_WORKSPACE;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* b = static_cast<uint8_t*>(ws);
  const int64_t n = T * k;
  if (w8a8_status e = cuda_status(launch_route(topk_ids, n, static_cast<int>(E), reinterpret_cast<int32_t*>(b + kStatusBytes),
                                               group_list, pos, static_cast<DeviceStatus*>(ws), st)))
    return e;
  if (n == 0) return W8A8_OK;
  const cudaError_t e = x_scale == nullptr
      ? launch_quant_scatter(static_cast<const uint16_t*>(x), T, H, pos, static_cast<int>(k), xq, nullptr, xs, 0, st, sms)
      : launch_scatter_rows_i8(static_cast<const int8_t*>(x), x_scale, T, H, pos, static_cast<int>(k), xq, nullptr,
                               xs, 0, st, sms);
  return cuda_status(e);
}

w8a8_status moe_unpermute_combine(const uint16_t* y_routed, const int32_t* pos, const float* topk_weights, int64_t T,
                                  int64_t k, int64_t H, uint16_t* y, void* ws, size_t ws_bytes,
                                  w8a8_stream_t stream) {
  if (w8a8_status s = check_route_shape(T, k, 1)) return s;
  if (H <= 0 || H > INT32_MAX || !combine_grid_ok(T, H)) return W8A8_ERR_SHAPE;
  if (H % 8 != 0) return W8A8_ERR_ALIGN;
  if (T == 0) return W8A8_OK;
  if (!y_routed || !pos || !topk_weights || !y) return W8A8_ERR_NULL;
  if (!ws) return W8A8_ERR_WORKSPACE;
  if (!aligned16(y_routed) || !aligned16(y)) return W8A8_ERR_ALIGN;
  if (ws_bytes < static_cast<size_t>(kStatusBytes) || !aligned16(ws)) return W8A8_ERR_WORKSPACE;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
  return cuda_status(launch_combine(y_routed, pos, topk_weights, T, static_cast<int>(k), H, y,
                                    static_cast<DeviceStatus*>(ws), reinterpret_cast<cudaStream_t>(stream), sms));
}

size_t moe_layer_workspace_bytes(int64_t T, int64_t k, int64_t H, int64_t I, int64_t E) {
  if (check_route_shape(T, k, E) != W8A8_OK || H <= 0 || I <= 0) return 0;
  return layer_layout(T, k, H, I, E).total;
}

int64_t moe_layer_workspace_offset(int64_t T, int64_t k, int64_t H, int64_t I, int64_t E, int which) {
  if (check_route_shape(T, k, E) != W8A8_OK || H <= 0 || I <= 0) return -1;
  const LayerWs L = layer_layout(T, k, H, I, E);
  switch (which) {
    case 7: return static_cast<int64_t>(L.group_list);
    case 8: return static_cast<int64_t>(L.pos);
    case 9: return static_cast<int64_t>(L.y_routed);
    default: return moe_workspace_offset(T * k, H, I, E, which);
  }
}

w8a8_status moe_layer(const void* x, const float* x_scale, const int64_t* topk_ids, const float* topk_weights,
                      int64_t T, int64_t k, int64_t E, int64_t H, int64_t I, const void* w13_packed,
                      const float* w13_scale, const void* w2_packed, const float* w2_scale, void* ws, size_t ws_bytes,
                      uint16_t* y, w8a8_stream_t stream) {
  if (w8a8_status s = check_route_shape(T, k, E)) return s;
  if (H <= 0 || I <= 0 || !combine_grid_ok(T, H)) return W8A8_ERR_SHAPE;
  if (w8a8_status s = check_k(H)) return s;
  if (w8a8_status s = check_k(I)) return s;
  if (I % kGateUpBlock != 0) return W8A8_ERR_SHAPE;
  if (T == 0) return W8A8_OK;
  if (!x || !topk_ids || !topk_weights || !w13_packed || !w13_scale || !w2_packed || !w2_scale || !y)
    return W8A8_ERR_NULL;
  if (!ws) return W8A8_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(y) || (reinterpret_cast<uintptr_t>(w13_packed) & 255u) ||
      (reinterpret_cast<uintptr_t>(w2_packed) & 255u))
    return W8A8_ERR_ALIGN;
  const LayerWs L = layer_layout(T, k, H, I, E);
  if (ws_bytes < L.total || !aligned16(ws)) return W8A8_ERR_WORKSPACE;
  int sms = 0;
  if (w8a8_status s = device_info(sms)) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* b = static_cast<uint8_t*>(ws);
  DeviceStatus* status = static_cast<DeviceStatus*>(ws);
  const int64_t R = T * k;
  const int kk = static_cast<int>(k);
  int64_t* gl = reinterpret_cast<int64_t*>(b + L.group_list);
  int32_t* pos = reinterpret_cast<int32_t*>(b + L.pos);
  int8_t* xq = L.m.xq ? reinterpret_cast<int8_t*>(b + L.m.xq) : nullptr;  // warp engine only
  float* xs = reinterpret_cast<float*>(b + L.m.xs);
  uint16_t* xq16 = L.m.xq16 ? reinterpret_cast<uint16_t*>(b + L.m.xq16) : nullptr;
  uint16_t* yr = reinterpret_cast<uint16_t*>(b + L.y_routed);
  if (w8a8_status e = cuda_status(launch_route(topk_ids, R, static_cast<int>(E), reinterpret_cast<int32_t*>(b + L.counts),
                                               gl, pos, status, st)))
    return e;
  // the routed codes go where the chain's engine reads them: fp16 for the tensor-core engines, else int8
  const int out = xq16 != nullptr ? 1 : 0;
  const cudaError_t ep = x_scale == nullptr
      ? launch_quant_scatter(static_cast<const uint16_t*>(x), T, H, pos, kk, xq, xq16, xs, out, st, sms)
      : launch_scatter_rows_i8(static_cast<const int8_t*>(x), x_scale, T, H, pos, kk, xq, xq16, xs, out, st, sms);
  if (ep != cudaSuccess) return W8A8_ERR_CUDA;
  if (w8a8_status e = moe_chain(xq, xs, true, gl, E, R, H, I, w13_packed, w13_scale, w2_packed, w2_scale, ws, yr,
                                st, sms))
    return e;
  return cuda_status(launch_combine(yr, pos, topk_weights, T, kk, H, y, status, st, sms));
}

w8a8_status w8a8_read_device_status(void* ws, w8a8_stream_t stream) {
  if (!ws) return W8A8_ERR_NULL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return W8A8_ERR_CUDA;
  DeviceStatus s;
  if (cudaMemcpy(&s, ws, sizeof(s), cudaMemcpyDeviceToHost) != cudaSuccess) return W8A8_ERR_CUDA;
  if (s.code != 0u) {
    if (cudaMemset(ws, 0, sizeof(s)) != cudaSuccess) return W8A8_ERR_CUDA;
  }
  return static_cast<w8a8_status>(s.code);
}

int w8a8_last_engine(void) { return t_last_engine; }

}  // extern "C"
