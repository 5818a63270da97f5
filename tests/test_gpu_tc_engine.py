"""GPU parity of the tcgen05 engines (large-M shapes; weights packed with their
fp16 copy, and without it, when the CTA-pair engine widens the INT8 weights
in tensor memory): INT32 accumulators, BF16 outputs and the MoE
intermediates must be bit-exact against the oracle.  Each test also checks
that the expected tcgen05 engine really ran (the host's engine record and the
fp16 activation copy it leaves in the workspace)."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_dynamic_quant_gb300 as W
from w8a8_dynamic_quant_gb300 import synthetic as S

from gpu_helpers import dev, dev_bf16, f32_bits, host_bits, moe_subset_oracle, sample_rows

pytestmark = pytest.mark.gpu
F16 = W.PACK_F16


def a16_region(ws, rows, K):
    """The fp16 activation copy the tcgen05 engine writes: the last 256-aligned block of rows*K*2 bytes."""
    nbytes = rows * K * 2
    start = ws.numel() - (nbytes + 255) // 256 * 256
    return ws[start:start + nbytes].view(torch.float16).view(rows, K)


def tc_dense(q, xs, w, wsc, bias=None, f16_copy=True):
    """Dense contraction on a tcgen05 engine: the fp16-copy engine, or without the copy the CTA-pair
    engine on the INT8 weights."""
    M, K = q.shape
    N = w.shape[0]
    wp = W.w8a8_prepack_weight(dev(w), F16 if f16_copy else 0)
    ws = W.workspace(W.quant_matmul_workspace_bytes(M, N, K))
    y = W.w8a8_quant_matmul(dev(q), dev(xs), wp, dev(wsc), N, None if bias is None else dev_bf16(bias), ws=ws)
    assert W.last_engine() == (W.ENGINE_TC if f16_copy else W.ENGINE_TC_I8)
    ws2 = W.workspace(W.quant_matmul_workspace_bytes(M, N, K))
    acc = W.w8a8_int8_matmul_acc(dev(q), wp, N, ws=ws2)
    assert W.last_engine() == (W.ENGINE_TC if f16_copy else W.ENGINE_TC_I8)
    torch.cuda.synchronize()
    # the tcgen05 engine widens q to fp16 at the end of the workspace
    assert torch.equal(a16_region(ws, M, K).cpu(), torch.from_numpy(q.astype(np.float16))), \
        "tcgen05 engine did not run"
    return host_bits(y), acc.cpu().numpy()


@pytest.mark.parametrize("M,N,K,bias", [(128, 256, 64, False), (130, 200, 80, True), (300, 512, 1040, True),
                                        (256, 384, 4096, False), (1000, 768, 2064, True), (129, 2048, 7168, False),
                                        (600, 1280, 576, True), (385, 300, 144, False)])
@pytest.mark.parametrize("f16_copy", [True, False])
def test_tc_dense_exact(M, N, K, bias, f16_copy):
    d = S.make_dense(M, K, N, n_outlier=min(4, K), outlier_mult=20.0, bias=bias, seed=M * 3 + N + K)
    q, xs = oracle.dynamic_quant(d.x)
    y, acc = tc_dense(q, xs, d.w, d.w_scale, d.bias, f16_copy)
    assert np.array_equal(acc, oracle.int8_gemm_acc(q, d.w))
    assert np.array_equal(y, oracle.quant_matmul(q, xs, d.w, d.w_scale, d.bias))


@pytest.mark.parametrize("f16_copy", [True, False])
def test_tc_accumulation_exact_at_extremes(f16_copy):
    K = 65536
    M = 128
    q = np.full((M, K), 127, np.int8)
    q[1] = -127
    q[2] = -128
    q[3, ::2] = -127
    q[4:] = np.random.default_rng(0).integers(-127, 128, (M - 4, K), dtype=np.int8)
    w = np.full((256, K), 127, np.int8)
    w[1] = -128
    w[2, : K // 2] = 1
    w[3, ::3] = -127
    w[4:] = np.random.default_rng(1).integers(-128, 128, (252, K), dtype=np.int8)
    _, acc = tc_dense(q, np.ones(M, np.float32), w, np.ones(256, np.float32), f16_copy=f16_copy)
    ref = q.astype(np.int64) @ w.astype(np.int64).T
    assert np.array_equal(acc.astype(np.int64), ref)


@pytest.mark.parametrize("f16_copy", [True, False])
def test_tc_dense_prefill_config_sampled_rows(f16_copy):
    d = S.dense_config(3)
    q, xs = oracle.dynamic_quant(d.x)
    wp = W.w8a8_prepack_weight(dev(d.w), F16 if f16_copy else 0)
    qd = dev(q)
    ws = W.workspace(W.quant_matmul_workspace_bytes(d.M, d.N, d.K))
    y = W.w8a8_quant_matmul(qd, dev(xs), wp, dev(d.w_scale), d.N, ws=ws)
    assert W.last_engine() == (W.ENGINE_TC if f16_copy else W.ENGINE_TC_I8)
    acc = W.w8a8_int8_matmul_acc(qd, wp, d.N)
    rows = sample_rows(d.M, 40, seed=5)
    idx = torch.as_tensor(rows, device="cuda")
    assert np.array_equal(acc[idx].cpu().numpy(), oracle.int8_gemm_acc(q[rows], d.w))
    assert np.array_equal(host_bits(y[idx]), oracle.quant_matmul(q[rows], xs[rows], d.w, d.w_scale, None))
    assert torch.equal(a16_region(ws, d.M, d.K).cpu(), torch.from_numpy(q.astype(np.float16)))


@pytest.mark.parametrize("gl,K,N", [([300, 0, 129, 77, 0, 200], 512, 256), ([64] * 8, 1024, 512),
                                    ([0, 0, 1000, 24], 2064, 384), ([385, 0, 129, 1], 576, 768),
                                    ([150, 0, 70], 80, 200),
                                    ([70 + (e * 37) % 90 if e % 7 else 0 for e in range(300)], 64, 128)])
@pytest.mark.parametrize("f16_copy", [True, False])
def test_tc_grouped_exact(gl, K, N, f16_copy):
    """Grouped contraction on the tensor cores, with the packed fp16 weight copy (fp16 weights by TMA)
    and without it (int8 weights widened in tensor memory)."""
    rng = np.random.default_rng(sum(gl) + K)
    R, E = int(sum(gl)), len(gl)
    x = S.to_bf16_bits(rng.standard_normal((R, K)).astype(np.float32))
    q, xs = oracle.dynamic_quant(x)
    w = rng.integers(-127, 128, (E, N, K), dtype=np.int8)
    wsc = rng.uniform(1e-3, 1e-2, (E, N)).astype(np.float32)
    glnp = np.asarray(gl, np.int64)
    wp = W.w8a8_prepack_weight(dev(w), F16 if f16_copy else 0)
    ws = W.workspace(W.grouped_matmul_workspace_bytes(E, R, N, K))
    y = torch.full((R, N), 3.0, dtype=torch.bfloat16, device="cuda")
    y = W.w8a8_grouped_matmul(dev(q), dev(xs), dev(glnp), wp, dev(wsc), ws=ws, y=y)
    assert W.last_engine() == (W.ENGINE_TC if f16_copy else W.ENGINE_TC_I8)
    acc = W.w8a8_grouped_matmul_acc(dev(q), dev(glnp), wp, N)
    torch.cuda.synchronize()
    assert torch.equal(a16_region(ws, R, K).cpu(), torch.from_numpy(q.astype(np.float16))), \
        "tcgen05 engine did not run"
    y_ref, acc_ref = oracle.grouped_matmul(q, xs, glnp, w, wsc, want_acc=True)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert np.array_equal(host_bits(y), y_ref)


def tc_moe(m, f16_copy=True):
    extra = F16 if f16_copy else 0
    w13p = W.w8a8_prepack_weight(m.w13.cuda(), W.PACK_GATE_UP | extra)
    w2p = W.w8a8_prepack_weight(m.w2.cuda(), extra)
    x, xs = (dev_bf16(m.x), None) if m.x_scale is None else (dev(m.x), dev(m.x_scale))
    ws = W.workspace(W.moe_workspace_bytes(m.R, m.H, m.I, m.E))
    y = W.moe_w13_swiglu_requant_w2(x, xs, dev(m.group_list), w13p, dev(m.s13), w2p, dev(m.s2), ws=ws)
    assert W.last_engine() == (W.ENGINE_TC if f16_copy else W.ENGINE_TC_I8)
    torch.cuda.synchronize()
    off16 = W.moe_workspace_offset(m.R, m.H, m.I, m.E, 5)
    assert off16 > 0
    xq16 = ws[off16: off16 + m.R * m.H * 2].view(torch.float16)
    assert bool((xq16 != 0).any()), "tcgen05 engine did not run"
    return host_bits(y), ws


def ws_slice(ws, m, which, dtype, shape):
    off = W.moe_workspace_offset(m.R, m.H, m.I, m.E, which)
    assert off >= 0, f"workspace item {which} is not kept for this shape"
    n = int(np.prod(shape)) * np.dtype(dtype).itemsize
    return ws[off:off + n].cpu().numpy().view(dtype).reshape(shape)


def hq_codes(ws, m):
    """The requantised h: on tensor-core shapes the workspace keeps only its integer-valued fp16 copy."""
    assert W.moe_workspace_offset(m.R, m.H, m.I, m.E, 3) == -1
    return ws_slice(ws, m, 6, np.float16, (m.R, m.I)).astype(np.int8)


@pytest.mark.parametrize("prequant", [False, True])
@pytest.mark.parametrize("f16_copy", [True, False])
def test_tc_moe_small_full(prequant, f16_copy):
    m = S.make_moe(T=256, H=256, I=128, E=4, topk=2, routing="zipf", zipf_s=1.1, n_dead=0,
                   prequant=prequant, seed=21)
    y, ws = tc_moe(m, f16_copy)
    y_ref, it = oracle.moe_w13_swiglu_requant_w2(m.x, m.x_scale, m.group_list, m.w13.numpy(), m.s13,
                                                 m.w2.numpy(), m.s2, intermediates=True)
    assert np.array_equal(ws_slice(ws, m, 2, np.uint16, (m.R, m.I)), it["h"])
    assert np.array_equal(hq_codes(ws, m), it["hq"])
    assert np.array_equal(f32_bits(ws_slice(ws, m, 4, np.float32, (m.R,))), f32_bits(it["hs"]))
    if m.x_scale is None:  # the routed rows' codes, quantised once
        assert W.moe_workspace_offset(m.R, m.H, m.I, m.E, 0) == -1
        assert np.array_equal(ws_slice(ws, m, 5, np.float16, (m.R, m.H)).astype(np.int8), it["xq"])
    assert np.array_equal(y, y_ref)


@pytest.mark.parametrize("f16_copy", [True, False])
def test_tc_moe_prefill_config_sampled_rows(f16_copy):
    m = S.moe_config(4, device="cuda")
    y, ws = tc_moe(m, f16_copy)
    rows = sample_rows(m.R, 24, seed=9)
    y_ref, it = moe_subset_oracle(m, rows)
    assert np.array_equal(ws_slice(ws, m, 2, np.uint16, (m.R, m.I))[rows], it["h"])
    assert np.array_equal(hq_codes(ws, m)[rows], it["hq"])
    assert np.array_equal(y[rows], y_ref)
