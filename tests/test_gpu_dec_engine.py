"""GPU parity of the decode engine (dense, M <= 64 tokens): int8 weights
widened into tensor memory, K split over CTAs whose exact int32 partials are
added into a sum tile in the workspace; the last CTA to arrive applies the
epilogue and leaves the sums and counters zero.  Bit-exact against the
oracle."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_dynamic_quant_gb300 as W
from w8a8_dynamic_quant_gb300 import synthetic as S

from gpu_helpers import dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


def run(q, xs, w, wsc, bias=None):
    M, K = q.shape
    N = w.shape[0]
    wp = W.w8a8_prepack_weight(dev(w))
    ws = W.workspace(W.quant_matmul_workspace_bytes(M, N, K))
    y = W.w8a8_quant_matmul(dev(q), dev(xs), wp, dev(wsc), N, None if bias is None else dev_bf16(bias), ws=ws)
    assert W.last_engine() == W.ENGINE_DECODE, "decode engine did not run"
    ws2 = W.workspace(W.quant_matmul_workspace_bytes(M, N, K))
    acc = W.w8a8_int8_matmul_acc(dev(q), wp, N, ws=ws2)
    assert W.last_engine() == W.ENGINE_DECODE
    torch.cuda.synchronize()
    # the sum tiles and arrival counters are left zero for the next call: past the 256-byte status word,
    # the workspace is all zero again
    assert int(ws[256:].count_nonzero()) == 0 and int(ws2[256:].count_nonzero()) == 0
    assert W.read_device_status(ws) == 0
    return host_bits(y), acc.cpu().numpy()


@pytest.mark.parametrize("M", [1, 7, 33, 64])
@pytest.mark.parametrize("N,K", [(128, 16), (200, 80), (2048, 1024), (384, 4096), (256, 7168), (130, 8192),
                                 (2048, 7168)])
def test_dec_shapes_exact(M, N, K):
    d = S.make_dense(M, K, N, n_outlier=min(5, K), outlier_mult=25.0, bias=(N % 2 == 0), seed=M * 7 + N + K)
    q, xs = oracle.dynamic_quant(d.x)
    y, acc = run(q, xs, d.w, d.w_scale, d.bias)
    assert np.array_equal(acc, oracle.int8_gemm_acc(q, d.w))
    assert np.array_equal(y, oracle.quant_matmul(q, xs, d.w, d.w_scale, d.bias))


def test_dec_partial_sums_at_the_extremes():
    """Every product 128*128 (the largest magnitude int8 allows): a CTA's fp32
    partial over its <= 896 of K stays an exact integer below 2^24, and the
    int32 sums over the whole K reach K * 2^14."""
    M, N, K = 64, 256, 8192
    q = np.full((M, K), -128, np.int8)
    q[1] = 127
    q[2, ::2] = -127
    q[3:] = np.random.default_rng(3).integers(-128, 128, (M - 3, K), dtype=np.int8)
    w = np.full((N, K), -128, np.int8)
    w[1] = 127
    w[2, : K // 2] = 1
    w[3:] = np.random.default_rng(4).integers(-128, 128, (N - 3, K), dtype=np.int8)
    _, acc = run(q, np.ones(M, np.float32), w, np.ones(N, np.float32))
    ref = q.astype(np.int64) @ w.astype(np.int64).T
    assert ref[0, 0] == K * 16384
    assert np.array_equal(acc.astype(np.int64), ref)


def test_dec_repeated_calls_reuse_the_workspace():
    d = S.dense_config(2)
    q, xs = oracle.dynamic_quant(d.x)
    wp = W.w8a8_prepack_weight(dev(d.w))
    ws = W.workspace(W.quant_matmul_workspace_bytes(d.M, d.N, d.K))
    ref = oracle.quant_matmul(q, xs, d.w, d.w_scale, None)
    for _ in range(5):
        y = W.w8a8_quant_matmul(dev(q), dev(xs), wp, dev(d.w_scale), d.N, ws=ws)
        assert np.array_equal(host_bits(y), ref)
    assert W.read_device_status(ws) == 0


def test_dec_chained_calls_share_buffers():
    """Quantisation and decode contraction enqueued back to back, every call
    reusing one code buffer, one scale buffer and one workspace: the launches
    overlap (each may start while the previous one still runs), yet no kernel
    touches those buffers before the kernel it depends on has finished, so
    every output matches the oracle."""
    M, N, K = 64, 1024, 3584
    rng = np.random.default_rng(11)
    w = rng.integers(-127, 128, (N, K), dtype=np.int8)
    wsc = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    xs = [S.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32) * (1.0 + i)) for i in range(6)]
    wp = W.w8a8_prepack_weight(dev(w))
    wsc_d = dev(wsc)
    xd = [dev_bf16(x) for x in xs]
    q = torch.empty((M, K), dtype=torch.int8, device="cuda")
    s = torch.empty(M, dtype=torch.float32, device="cuda")
    ws = W.workspace(W.quant_matmul_workspace_bytes(M, N, K))
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in xs]
    torch.cuda.synchronize()
    for x, y in zip(xd, ys):
        W.w8a8_dynamic_quant(x, q=q, scale=s)
        W.w8a8_quant_matmul(q, s, wp, wsc_d, N, ws=ws, y=y)
        assert W.last_engine() == W.ENGINE_DECODE
    torch.cuda.synchronize()
    assert W.read_device_status(ws) == 0
    for x, y in zip(xs, ys):
        qo, so = oracle.dynamic_quant(x)
        assert np.array_equal(host_bits(y), oracle.quant_matmul(qo, so, w, wsc, None))


def test_dec_small_m_with_fp16_pack_stays_in_workspace():
    """A dense call with at most 64 rows on weights packed WITH the fp16 copy runs the decode engine
    and writes nothing past the workspace it was given (its workspace holds no fp16 code copy)."""
    M, N, K = 64, 256, 7168
    rng = np.random.default_rng(5)
    q = rng.integers(-127, 128, (M, K), dtype=np.int8)
    xs = rng.uniform(1e-3, 1e-2, M).astype(np.float32)
    w = rng.integers(-127, 128, (N, K), dtype=np.int8)
    wsc = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    wp = W.w8a8_prepack_weight(dev(w), W.PACK_F16)
    nbytes = W.quant_matmul_workspace_bytes(M, N, K)
    guard = 1 << 20
    buf = torch.zeros(nbytes + guard, dtype=torch.uint8, device="cuda")
    buf[nbytes:] = 0xA5
    y = W.w8a8_quant_matmul(dev(q), dev(xs), wp, dev(wsc), N, ws=buf[:nbytes])
    assert W.last_engine() == W.ENGINE_DECODE
    torch.cuda.synchronize()
    assert bool((buf[nbytes:] == 0xA5).all()), "write past the workspace"
    assert np.array_equal(host_bits(y), oracle.quant_matmul(q, xs, w, wsc, None))
