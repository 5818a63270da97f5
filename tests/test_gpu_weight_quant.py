"""GPU parity of the offline per-channel weight quantisation (through the C ABI):
INT8 codes and FP32 scales bit-exact against the oracle, the packed buffer
written in one pass from BF16 byte-identical to packing the oracle's INT8
weight, and contractions on those packs equal to the oracle's."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_dynamic_quant_gb300 as W
from w8a8_dynamic_quant_gb300 import synthetic as S

from gpu_helpers import dev, dev_bf16, f32_bits, host_bits

pytestmark = pytest.mark.gpu


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("E,N,K", [(1, 1, 16), (1, 130, 80), (3, 64, 4096), (2, 200, 7168), (5, 128, 64),
                                   (1, 256, 8192)])
def test_quantize_weight_exact(E, N, K):
    w = S.make_bf16_weight(E, N, K, seed=E + N + K, device="cuda")
    w[0, 0] = 0  # an all-zero channel
    q, s = W.w8a8_quantize_weight(w)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_weight(bits(w))
    assert np.array_equal(f32_bits(s.cpu().numpy()), f32_bits(s_ref))
    assert np.array_equal(q.cpu().numpy(), q_ref)


@pytest.mark.parametrize("E,N,K", [(1, 384, 272), (4, 256, 1024), (2, 128, 4096)])
@pytest.mark.parametrize("flags", [0, W.PACK_F16, W.PACK_GATE_UP, W.PACK_GATE_UP | W.PACK_F16])
def test_quantize_prepack_equals_prepack_of_oracle_codes(E, N, K, flags):
    w = S.make_bf16_weight(E, N, K, seed=N + K + flags, device="cuda")
    packed, s = W.w8a8_quantize_prepack_weight(w, flags)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_weight(bits(w))
    want = W.w8a8_prepack_weight(dev(q_ref), flags)
    torch.cuda.synchronize()
    assert np.array_equal(f32_bits(s.cpu().numpy()), f32_bits(s_ref))
    # the header's fields (56 bytes), the int8 payload and the fp16 copy; the rest of the 256-byte header
    # block and the alignment padding are written by neither packer
    n = E * N * K
    f16_off = (256 + n + 255) // 256 * 256
    regions = [(0, 56), (256, 256 + n)] + ([(f16_off, f16_off + 2 * n)] if flags & W.PACK_F16 else [])
    for a, b in regions:
        assert torch.equal(packed[a:b], want[a:b]), f"packed bytes [{a},{b}) differ"


def test_quantize_prepack_dense_then_decode_contraction():
    """A contraction enqueued right after the packing (the decode engine streams the packed weights
    before it waits for the kernels ahead of it) sees the finished pack."""
    M, N, K = 64, 2048, 7168
    w = S.make_bf16_weight(1, N, K, seed=7, device="cuda")[0]
    d = S.make_dense(M, K, N, n_outlier=72, outlier_mult=30.0, seed=3)
    xq, xs = oracle.dynamic_quant(d.x)
    ws = W.workspace(W.quant_matmul_workspace_bytes(M, N, K))
    ys = []
    for rep in range(3):
        packed, s = W.w8a8_quantize_prepack_weight(w, W.PACK_F16)
        ys.append(W.w8a8_quant_matmul(dev(xq), dev(xs), packed, s, N, ws=ws))
    torch.cuda.synchronize()
    assert W.last_engine() == W.ENGINE_DECODE
    q_ref, s_ref = oracle.quantize_weight(bits(w))
    y_ref = oracle.quant_matmul(xq, xs, q_ref, s_ref, None)
    for y in ys:
        assert np.array_equal(host_bits(y), y_ref)


def test_quantize_prepack_moe_layer_from_bf16_weights():
    """W13 and W2 quantised and packed from BF16 on the device feed the MoE chain; the result equals the
    oracle's chain on the oracle's quantised weights."""
    m = S.make_moe(T=300, H=256, I=128, E=4, topk=2, routing="zipf", zipf_s=1.1, n_dead=0, seed=31)
    w13 = S.make_bf16_weight(m.E, 2 * m.I, m.H, seed=1, device="cuda")
    w2 = S.make_bf16_weight(m.E, m.H, m.I, seed=2, device="cuda")
    w13p, s13 = W.w8a8_quantize_prepack_weight(w13, W.PACK_GATE_UP | W.PACK_F16)
    w2p, s2 = W.w8a8_quantize_prepack_weight(w2, W.PACK_F16)
    y = W.moe_w13_swiglu_requant_w2(dev_bf16(m.x), None, dev(m.group_list), w13p, s13, w2p, s2)
    torch.cuda.synchronize()
    q13, r13 = oracle.quantize_weight(bits(w13))
    q2, r2 = oracle.quantize_weight(bits(w2))
    y_ref = oracle.moe_w13_swiglu_requant_w2(m.x, None, m.group_list, q13, r13, q2, r2)
    assert np.array_equal(host_bits(y), y_ref)
