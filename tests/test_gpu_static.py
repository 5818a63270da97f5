"""GPU parity of the static W8A8 variant (through the C ABI): the INT8 codes of
the fixed-scale quantiser, the load-time deq_scale / quant_bias, and the BF16
outputs of the matmul on every dense engine, all bit-exact against the
oracle."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_dynamic_quant_gb300 as W
from w8a8_dynamic_quant_gb300 import synthetic as S

from gpu_helpers import dev, dev_bf16, f32_bits, host_bits, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K,s,o", [(1, 16, 0.03, 0), (7, 96, 0.0625, 5), (300, 4096, 0.021, -8),
                                     (64, 7168, 0.5, 127), (33, 272, 1e-3, -128)])
def test_static_quant_exact(M, K, s, o):
    rng = np.random.default_rng(M + K)
    x = (rng.standard_normal((M, K)) * 2).astype(np.float32)
    x[0, :4] = [np.float32(s) * 2.5, -np.float32(s) * 3.5, 1e30, -1e30]  # ties and the clamps
    xb = S.to_bf16_bits(x)
    q = W.w8a8_static_quant(dev_bf16(xb), s, o)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), oracle.static_quant(xb, np.float32(s), o))


@pytest.mark.parametrize("N,K,bias", [(1, 16, True), (200, 96, False), (2048, 7168, True), (130, 4096, True)])
def test_static_prepare_exact(N, K, bias):
    rng = np.random.default_rng(N + K)
    w = rng.integers(-128, 128, (N, K), dtype=np.int8)
    ws = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    w[0] = 0
    ws[0] = 0.0  # an all-zero channel: deq_scale 0, the bias dropped
    b = S.to_bf16_bits(rng.normal(0, 0.5, N).astype(np.float32)) if bias else None
    s, o = np.float32(0.031), -5
    deq, qb = W.w8a8_static_prepare(dev(w), dev(ws), s, o, None if b is None else dev_bf16(b))
    torch.cuda.synchronize()
    deq_ref, qb_ref = oracle.static_prepare(w, ws, s, o, b)
    assert np.array_equal(f32_bits(deq.cpu().numpy()), f32_bits(deq_ref))
    assert np.array_equal(qb.cpu().numpy(), qb_ref)


def static_case(M, N, K, f16, bias, seed):
    d = S.make_dense(M, K, N, n_outlier=min(4, K), outlier_mult=20.0, bias=bias, seed=seed)
    s, o = np.float32(0.03), 3
    q = oracle.static_quant(d.x, s, o)
    deq, qb = oracle.static_prepare(d.w, d.w_scale, s, o, d.bias)
    wp = W.w8a8_prepack_weight(dev(d.w), W.PACK_F16 if f16 else 0)
    y = W.w8a8_static_quant_matmul(dev(q), wp, dev(deq), dev(qb))
    torch.cuda.synchronize()
    return d, q, deq, qb, host_bits(y)


@pytest.mark.parametrize("M,N,K,f16,engine", [(1, 256, 512, False, "decode"), (64, 2048, 7168, False, "decode"),
                                              (17, 200, 80, False, "decode"), (100, 384, 1040, False, "warp"),
                                              (300, 384, 1040, False, "tc_i8"), (130, 200, 64, False, "tc_i8"),
                                              (512, 512, 2048, True, "tc"), (1000, 768, 2064, True, "tc")])
@pytest.mark.parametrize("bias", [False, True])
def test_static_quant_matmul_exact(M, N, K, f16, engine, bias):
    d, q, deq, qb, y = static_case(M, N, K, f16, bias, seed=M + N)
    want = {"decode": W.ENGINE_DECODE, "warp": W.ENGINE_WARP, "tc": W.ENGINE_TC, "tc_i8": W.ENGINE_TC_I8}[engine]
    assert W.last_engine() == want
    assert np.array_equal(y, oracle.static_quant_matmul(q, d.w, deq, qb))


@pytest.mark.parametrize("cfg", [2, 3])
def test_static_full_config_sampled_rows(cfg):
    d = S.dense_config(cfg)
    s, o = S.static_params(cfg)
    xq = W.w8a8_static_quant(dev_bf16(d.x), s, o)
    wd = dev(d.w)
    deq, qb = W.w8a8_static_prepare(wd, dev(d.w_scale), s, o, None)
    wp = W.w8a8_prepack_weight(wd, W.PACK_F16 if d.M >= 128 else 0)
    y = W.w8a8_static_quant_matmul(xq, wp, deq, qb)
    torch.cuda.synchronize()
    q_ref = oracle.static_quant(d.x, np.float32(s), o)
    assert np.array_equal(xq.cpu().numpy(), q_ref)
    deq_ref, qb_ref = oracle.static_prepare(d.w, d.w_scale, np.float32(s), o, None)
    assert np.array_equal(qb.cpu().numpy(), qb_ref)
    rows = sample_rows(d.M, 24, seed=cfg)
    idx = torch.as_tensor(rows, device="cuda")
    assert np.array_equal(host_bits(y[idx]), oracle.static_quant_matmul(q_ref[rows], d.w, deq_ref, qb_ref))


@pytest.mark.parametrize("s,o", [(0.03, 0), (0.0625, 7), (1.0 / 3.0, -3), (0.0071, 100)])
def test_static_quant_every_bf16_value_in_range(s, o):
    """Every BF16 value of magnitude below 64 (both signs): the exact-tie and near-tie quotients that the
    reciprocal path must hand to the division, and the clamps."""
    mags = np.arange(0x0000, 0x4280, dtype=np.uint32)       # +0 .. 64 in bf16 bit patterns
    vals = np.concatenate([mags, mags | 0x8000]).astype(np.uint16)
    pad = (-vals.size) % 16
    xb = np.concatenate([vals, np.zeros(pad, np.uint16)]).reshape(-1, 16)
    q = W.w8a8_static_quant(dev_bf16(xb), s, o)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), oracle.static_quant(xb, np.float32(s), o))


@pytest.mark.parametrize("M,f16,engine", [(1, False, W.ENGINE_DECODE), (100, False, W.ENGINE_WARP),
                                          (130, False, W.ENGINE_TC_I8), (256, True, W.ENGINE_TC)])
def test_static_matmul_sum_past_int32(M, f16, engine):
    """acc + quant_bias beyond the int32 range (codes of +-127 against weights of 127, so |acc| is about
    1.2e8, and a quant_bias within 100 of +-2^31): the epilogue takes the exact 64-bit sum."""
    N, K = 256, 7168
    q = np.full((M, K), 127, np.int8)
    q[M // 2:] = -127
    w = np.full((N, K), 127, np.int8)
    qb = np.where(np.arange(N) % 2 == 0, 2 ** 31 - 100, -(2 ** 31) + 7).astype(np.int32)
    deq = np.full(N, 1e-9, np.float32)
    wp = W.w8a8_prepack_weight(dev(w), W.PACK_F16 if f16 else 0)
    y = W.w8a8_static_quant_matmul(dev(q), wp, dev(deq), dev(qb))
    torch.cuda.synchronize()
    assert W.last_engine() == engine
    assert np.array_equal(host_bits(y), oracle.static_quant_matmul(q, w, deq, qb))
