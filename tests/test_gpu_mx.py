"""GPU parity of the MXFP8 path (through the C ABI): the quantiser's E4M3 codes
and E8M0 scales bit-exact against the oracle, over wide dynamic ranges, zero
groups, BF16 subnormals, saturating groups and every finite BF16 value; the
contraction, on the block-scaled tensor cores and on the warp-level FP8
instruction, within the binary32 accumulation bound of the exact result."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_dynamic_quant_gb300 as W
from w8a8_dynamic_quant_gb300 import synthetic as S

from gpu_helpers import dev_bf16

pytestmark = pytest.mark.gpu


def check(xb):
    q, s = W.w8a8_mx_quant(dev_bf16(xb))
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.mx_quant(xb)
    assert np.array_equal(s.cpu().numpy(), s_ref), "E8M0 scales differ"
    bad = np.argwhere(q.cpu().numpy() != q_ref)
    assert bad.size == 0, f"{len(bad)} E4M3 codes differ, first {bad[:4]}"


@pytest.mark.parametrize("M,K", [(1, 32), (37, 512), (64, 7168), (300, 96)])
def test_mx_quant_exact(M, K):
    rng = np.random.default_rng(M + K)
    x = rng.standard_normal((M, K)) * 2.0 ** rng.integers(-40, 40, (M, 1))
    x = x.astype(np.float32)
    x[0, :32] = 0.0                                            # a group of zeros
    if K >= 64:
        x[0, 32:64] = np.float32(1.8) * 2.0 ** np.arange(-3, 29)[:32].astype(np.float32)  # saturating top
    if M > 1:
        x[1, :32] = (rng.integers(1, 128, 32) * 2.0 ** -133).astype(np.float32)  # BF16 subnormals
    check(S.to_bf16_bits(x))


def test_mx_quant_every_finite_bf16_value():
    bits = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    v = S.bf16_bits_to_f32(bits)
    vals = bits[np.isfinite(v)]
    vals = vals[: vals.size // 1024 * 1024]
    check(vals.reshape(-1, 1024))


def test_mx_quant_dense_decode_input():
    d = S.dense_config(2)
    check(d.x)


def mx_bound(qa, sa, qw, sw, y_ref):
    """1 bf16 ulp of the exact result plus the binary32 accumulation: (32 + K/32) roundings of at most
    2^-24 of the running magnitude, bounded by the sum of |terms|."""
    dec = np.vectorize(oracle.e4m3_to_f32, otypes=[np.float32])
    A = np.abs(dec(qa).astype(np.float64)) * np.repeat(2.0 ** (sa.astype(np.float64) - 127), 32, axis=1)
    B = np.abs(dec(qw).astype(np.float64)) * np.repeat(2.0 ** (sw.astype(np.float64) - 127), 32, axis=1)
    mag = A @ B.T
    K = qa.shape[1]
    ref = S.bf16_bits_to_f32(y_ref).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
    return ref, ulp + (32 + K // 32) * 2.0 ** -24 * mag


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (37, 200, 512), (128, 256, 1024), (300, 130, 384),
                                   (64, 2048, 7168), (300, 520, 1024), (193, 264, 2048), (16, 8, 512)])
def test_mx_matmul_within_bound(M, N, K):
    """Both engines: the block-scaled tensor cores for K % 512 == 0 and N % 8 == 0, else the warp-level
    FP8 instruction."""
    rng = np.random.default_rng(M + N + K)
    xa = S.to_bf16_bits((rng.standard_normal((M, K)) * 2.0 ** rng.integers(-6, 6, (M, 1))).astype(np.float32))
    xw = S.to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    qa, sa = oracle.mx_quant(xa)
    qw, sw = oracle.mx_quant(xw)
    from gpu_helpers import dev
    y = W.w8a8_mx_matmul(dev(qa), dev(sa), dev(qw), dev(sw))
    assert W.last_engine() == (W.ENGINE_TC if K % 512 == 0 and N % 8 == 0 else W.ENGINE_WARP)
    torch.cuda.synchronize()
    got = S.bf16_bits_to_f32(y.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    y_ref = oracle.mx_matmul(qa, sa, qw, sw)
    ref, bound = mx_bound(qa, sa, qw, sw, y_ref)
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"max excess {np.max(err - bound)}"
    assert np.mean(err == 0) > 0.9  # nearly all outputs are the exactly rounded ones
