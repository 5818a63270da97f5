"""w8a8_quant_matmul_noalloc: the dense quantised matmul for callers that
cannot allocate device memory (no allocator in their plugin interface, all
HBM reserved by the host for its own pools, or cudaMalloc not allowed where
they run).  Its scratch is a fixed array inside the library, so this test
checks that two calls in a row through the C ABI give the same output as the
workspace entry point w8a8_quant_matmul, and that a problem too large for the
array is refused before launch.  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import w8a8_dynamic_quant_gb300 as W
from w8a8_dynamic_quant_gb300 import _capi
from w8a8_dynamic_quant_gb300 import synthetic as S

from gpu_helpers import bf16_ulp_diff, dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", [2, 1])
def test_noalloc_matches_workspace_entry_on_two_calls(cfg):
    d = S.dense_config(cfg)
    q, xs = oracle.dynamic_quant(d.x)
    qd, xsd = dev(q), dev(xs)
    wp = W.w8a8_prepack_weight(dev(d.w))
    swd = dev(d.w_scale)
    bias = None if d.bias is None else dev_bf16(d.bias)
    ref = host_bits(W.w8a8_quant_matmul(qd, xsd, wp, swd, d.N, bias))
    lib = _capi.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        y = torch.full((d.M, d.N), -1.0, dtype=torch.bfloat16, device="cuda")
        rc = lib.w8a8_quant_matmul_noalloc(qd.data_ptr(), xsd.data_ptr(), d.M, d.K, wp.data_ptr(), swd.data_ptr(),
                                           d.N, None if bias is None else bias.data_ptr(), y.data_ptr(), stream)
        assert rc == 0, _capi.W8A8Error("w8a8_quant_matmul_noalloc", rc)
        torch.cuda.synchronize()
        got = host_bits(y)
        assert bf16_ulp_diff(got, ref).max() <= 1, f"call {call}"
        assert np.array_equal(got, ref), f"call {call}"


def test_noalloc_refuses_problems_larger_than_its_scratch():
    lib = _capi.lib()
    fake = ctypes.c_void_p(256)
    # 4096 x 4096 int32 partial sums need 64 MiB: more than the built-in array
    rc = lib.w8a8_quant_matmul_noalloc(fake, fake, 4096, 64, fake, fake, 4096, None, fake, None)
    assert rc == 4
