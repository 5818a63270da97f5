// kernels.cuh -- launchers of the kernels in libw8a8.so (internal interface).
#pragma once

#include <algorithm>

#include "common.cuh"

namespace w8a8 {

struct PackLayout {
  uint64_t i8_offset;
  uint64_t f16_offset;  // 0 when the fp16 copy is absent
  uint64_t total;
};
PackLayout pack_layout(int64_t E, int64_t N, int64_t K, uint32_t flags);

cudaError_t launch_prepack(const int8_t* w, int64_t E, int64_t N, int64_t K, uint32_t flags, void* packed,
                           cudaStream_t stream, int num_sms);
// The header of a packed buffer whose payload a kernel before it on the stream wrote.
cudaError_t launch_pack_header(int64_t E, int64_t N, int64_t K, uint32_t flags, void* packed, cudaStream_t stream);
// Offline weight quantisation straight into a packed buffer: channel (e, c) of w [E,N,K] bf16 quantised
// per channel over K, codes (and their fp16 copy if flags ask) to its packed row, scale to scale[e*N + c].
cudaError_t launch_quant_pack(const uint16_t* w, int64_t E, int64_t N, int64_t K, uint32_t flags, void* packed,
                              float* scale, cudaStream_t stream, int num_sms);

cudaError_t launch_dynamic_quant(const uint16_t* x, int64_t M, int64_t K, int8_t* q, float* scale,
                                 cudaStream_t stream, int num_sms);
// the codes as integer-valued fp16 only (the operand the tcgen05 engines read)
cudaError_t launch_dynamic_quant_f16(const uint16_t* x, int64_t M, int64_t K, uint16_t* q_f16, float* scale,
                                     cudaStream_t stream, int num_sms);

// MoE routing permute: token row m of x [T,H] quantised once, its codes and scale written to the
// routed rows dst[m*k + j] (j < k; an index < 0 is skipped).  out: 0 int8 into q, 1 fp16 into q_f16,
// 2 both.
cudaError_t launch_quant_scatter(const uint16_t* x, int64_t T, int64_t H, const int32_t* dst, int k, int8_t* q,
                                 uint16_t* q_f16, float* scale, int out, cudaStream_t stream, int num_sms);

// MoE routing (route.cu).  Stable counting sort of the T*k (token, slot) pairs by expert.
// counts: int32 scratch of route_scratch_ints(T*k, E) entries.
int64_t route_scratch_ints(int64_t n, int64_t E);
cudaError_t launch_route(const int64_t* topk_ids, int64_t n, int E, int32_t* counts, int64_t* group_list,
                         int32_t* pos, DeviceStatus* status, cudaStream_t stream);
// Routed copies of already-quantised token rows: xq_tok [T,H] int8 + xs_tok [T] -> rows dst[t*k + j].
cudaError_t launch_scatter_rows_i8(const int8_t* xq_tok, const float* xs_tok, int64_t T, int64_t H,
                                   const int32_t* dst, int k, int8_t* q, uint16_t* q_f16, float* scale, int out,
                                   cudaStream_t stream, int num_sms);
// Top-k weighted combine of the routed rows back into token rows.
cudaError_t launch_combine(const uint16_t* y_routed, const int32_t* pos, const float* w, int64_t T, int k,
                           int64_t H, uint16_t* y, DeviceStatus* status, cudaStream_t stream, int num_sms);

// Static W8A8 (static.cu): q = clamp(rint(x / s) + o, -128, 127); load-time deq_scale / quant_bias.
cudaError_t launch_static_quant(const uint16_t* x, int64_t M, int64_t K, float s, int o, int8_t* q,
                                cudaStream_t stream, int num_sms);
cudaError_t launch_static_prepare(const int8_t* w, int64_t N, int64_t K, const float* w_scale, float s, int o,
                                  const uint16_t* bias, float* deq, int32_t* qb, cudaStream_t stream, int num_sms);

// MXFP8 quantisation (mx.cu): x [M,K] bf16 -> E4M3 q [M,K] + E8M0 scale [M,K/32].
cudaError_t launch_mx_quant(const uint16_t* x, int64_t M, int64_t K, uint8_t* q, uint8_t* scale, cudaStream_t stream,
                            int num_sms);

// MXFP8 contraction (mx.cu): E4M3 a [M,K] + E8M0 [M,K/32], E4M3 w [N,K] + E8M0 [N,K/32] -> bf16 y [M,N],
// on the warp-level FP8 instruction.
cudaError_t launch_mx_matmul(const uint8_t* qa, const uint8_t* sa, int64_t M, int64_t K, const uint8_t* qw,
                             const uint8_t* sw, int64_t N, uint16_t* y, cudaStream_t stream);
// The same on the block-scaled tensor cores (mx_tc.cu, CTA pairs, tcgen05 kind::mxf8f6f4) for the shapes
// mx_tc_supported() accepts (K % 512 == 0, N % 8 == 0).  status may be nullptr.
bool mx_tc_supported(int64_t M, int64_t N, int64_t K);
cudaError_t launch_mx_tc(const uint8_t* qa, const uint8_t* sa, int64_t M, int64_t K, const uint8_t* qw,
                         const uint8_t* sw, int64_t N, uint16_t* y, DeviceStatus* status, int num_sms,
                         cudaStream_t stream);

// Epilogue of the contraction.
enum EpiMode : int {
  EPI_BF16 = 0,    // y[r,n] = bf16(((float)acc * sx[r]) * sw[e,n] (+ bias[n]))
  EPI_ACC = 1,     // acc[r,n] = exact int32
  EPI_SWIGLU = 2,  // W13 with gate/up interleave: h[r,j] = swiglu(bf16 gate, bf16 up)
};

// One grouped (or dense: group_list == nullptr, one group of R rows) contraction.
struct GemmArgs {
  const int8_t* q = nullptr;          // [R,K] int8 activations
  const float* x_scale = nullptr;     // [R]
  const int64_t* group_list = nullptr;  // [E] counts, or nullptr for one group of R rows
  int64_t E = 1, R = 0, K = 0, N = 0; // N = rows per expert of the packed weight
  const void* packed = nullptr;       // packed weight buffer (header first)
  uint32_t pack_flags = 0;            // flags the call expects in the header
  int pack_known = 0;                 // 1: this process packed the buffer with these E, N, K (host record)
  const float* w_scale = nullptr;     // [E,N] in ORIGINAL channel order
  const uint16_t* bias = nullptr;     // [N] bf16 or nullptr (dense only)
  const int32_t* qbias = nullptr;     // [N] int32 added to the accumulator before dequant, or nullptr (dense,
                                      // static W8A8; x_scale is then nullptr and reads as 1)
  void* out = nullptr;                // bf16 [R,N] | int32 [R,N] | bf16 h [R,N/2]
  int mode = EPI_BF16;
  DeviceStatus* status = nullptr;
  int32_t* ws_acc = nullptr;          // split-K partial sums [R,N] (zero on entry and exit)
  uint32_t* ws_count = nullptr;       // split-K arrival counters (zero on entry and exit)
  int64_t ws_count_len = 0;
};

struct GemmPlan {
  int variant;   // tile shape id
  int ksplit;
  int grid;
  size_t smem;
};

// Host: choose the tile shape and split for the register-path engine.
GemmPlan plan_reg_gemm(const GemmArgs& a, int num_sms);
// Workspace (split-K partials + counters) the plan needs, in bytes.
size_t reg_gemm_ws_bytes(int64_t E, int64_t R, int64_t N, int64_t K, int num_sms);
cudaError_t launch_reg_gemm(const GemmArgs& a, const GemmPlan& p, cudaStream_t stream);

// tcgen05 engine (large M): both operands as integer-valued fp16, K-major.
// a_f16: [R,K] activations; b_f16: [E*N,K] packed weights (fp16 copy).
cudaError_t launch_tc_gemm(const GemmArgs& a, const void* a_f16, const void* b_f16, int num_sms, cudaStream_t stream);
// tcgen05 engine on CTA pairs for large M, dense or grouped: int8 weights (the packed payload) widened in
// TMEM as the M = 256 side, a_f16: [R,K] activations as fp16 (the N side, up to 192 tokens per tile).
cudaError_t launch_tcp_gemm(const GemmArgs& a, const void* a_f16, int num_sms, cudaStream_t stream);
cudaError_t launch_s8_to_f16(const int8_t* src, uint16_t* dst, int64_t n, cudaStream_t stream, int num_sms);

// tcgen05 decode engine (dense, M <= 64): int8 weights widened into TMEM, K
// split over CTAs whose exact int32 partials are added into a per-row-block
// sum tile in the workspace (bulk reduce-add); the last CTA to arrive applies
// the epilogue.  dec_plan returns ksplit 0 when the shape does not suit it.
struct DecPlan {
  int ksplit = 0;  // K splits per 128-row weight block
};
size_t dec_ws_bytes(int64_t N);
DecPlan dec_plan(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_dec_gemm(const GemmArgs& a, const DecPlan& plan, void* dec_ws, cudaStream_t stream);

}  // namespace w8a8
