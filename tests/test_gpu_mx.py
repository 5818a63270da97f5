"""GPU parity of the MXFP8 quantiser (through the C ABI): E4M3 codes and E8M0
scales bit-exact against the oracle, over wide dynamic ranges, zero groups,
BF16 subnormals, saturating groups and every finite BF16 value."""
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
