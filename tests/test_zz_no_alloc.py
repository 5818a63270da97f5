"""w8a8_quant_matmul_noalloc: the dense quantised matmul for callers that
cannot allocate device memory (no allocator in their plugin interface, all
HBM reserved by the host for its own pools, or cudaMalloc not allowed where
they run).  Its scratch is a fixed array inside the library, so these tests
check, through the C ABI, that two calls in a row give the oracle's output
bit for bit and the same output as the workspace entry point
w8a8_quant_matmul, that a device-side error (a packed weight whose header
does not match the call) reaches the caller through
w8a8_quant_matmul_noalloc_status, that a problem whose partial sums do not fit
the array runs without splitting K, and that one whose counters do not fit is
refused before launch.  Collected last on purpose."""
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


def _call(lib, qd, xsd, M, K, wp, swd, N, bias, y):
    return lib.w8a8_quant_matmul_noalloc(qd.data_ptr(), xsd.data_ptr(), M, K, wp.data_ptr(), swd.data_ptr(), N,
                                         None if bias is None else bias.data_ptr(), y.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("cfg", [2, 1])
def test_noalloc_matches_oracle_and_workspace_entry_on_two_calls(cfg):
    d = S.dense_config(cfg)
    q, xs = oracle.dynamic_quant(d.x)
    y_oracle = oracle.quant_matmul(q, xs, d.w, d.w_scale, d.bias)
    qd, xsd = dev(q), dev(xs)
    wp = W.w8a8_prepack_weight(dev(d.w))
    swd = dev(d.w_scale)
    bias = None if d.bias is None else dev_bf16(d.bias)
    ref = host_bits(W.w8a8_quant_matmul(qd, xsd, wp, swd, d.N, bias))
    lib = _capi.lib()
    for call in range(2):
        y = torch.full((d.M, d.N), -1.0, dtype=torch.bfloat16, device="cuda")
        rc = _call(lib, qd, xsd, d.M, d.K, wp, swd, d.N, bias, y)
        assert rc == 0, _capi.W8A8Error("w8a8_quant_matmul_noalloc", rc)
        assert lib.w8a8_quant_matmul_noalloc_status(torch.cuda.current_stream().cuda_stream) == 0
        got = host_bits(y)
        assert bf16_ulp_diff(got, y_oracle).max() <= 1, f"call {call}"
        assert np.array_equal(got, y_oracle), f"call {call}: differs from the oracle"
        assert np.array_equal(got, ref), f"call {call}: differs from w8a8_quant_matmul"


def test_noalloc_reports_a_mismatched_pack_through_its_status_call():
    d = S.dense_config(1)  # N = 256
    q, xs = oracle.dynamic_quant(d.x)
    qd, xsd = dev(q), dev(xs)
    wp = W.w8a8_prepack_weight(dev(d.w))
    swd = dev(d.w_scale)
    lib = _capi.lib()
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.w8a8_quant_matmul_noalloc_status(stream) == 0
    n_wrong = d.N // 2  # the header records N = 256
    y = torch.full((d.M, n_wrong), 3.0, dtype=torch.bfloat16, device="cuda")
    assert _call(lib, qd, xsd, d.M, d.K, wp, swd, n_wrong, None, y) == 0  # host checks pass; the device refuses
    assert lib.w8a8_quant_matmul_noalloc_status(stream) == _capi.W8A8_ERR_PACKED
    assert bool((y == 3.0).all()), "a refused call must leave y unwritten"
    assert lib.w8a8_quant_matmul_noalloc_status(stream) == 0, "reading the status clears it"
    # the array is usable again at once
    y2 = torch.empty((d.M, d.N), dtype=torch.bfloat16, device="cuda")
    assert _call(lib, qd, xsd, d.M, d.K, wp, swd, d.N, dev_bf16(d.bias), y2) == 0
    assert lib.w8a8_quant_matmul_noalloc_status(stream) == 0
    assert np.array_equal(host_bits(y2), oracle.quant_matmul(q, xs, d.w, d.w_scale, d.bias))


def test_noalloc_runs_problems_whose_partial_sums_do_not_fit():
    """4096 x 4096 outputs: their int32 partial sums (64 MiB) do not fit the built-in array, so the call
    runs without splitting K and must still give the oracle's output bit for bit."""
    lib = _capi.lib()
    d = S.make_dense(4096, 64, 4096, n_outlier=2, outlier_mult=10.0, bias=True, seed=11)
    q, xs = oracle.dynamic_quant(d.x)
    qd, xsd, swd = dev(q), dev(xs), dev(d.w_scale)
    wp = W.w8a8_prepack_weight(dev(d.w))
    y = torch.empty((d.M, d.N), dtype=torch.bfloat16, device="cuda")
    assert _call(lib, qd, xsd, d.M, d.K, wp, swd, d.N, dev_bf16(d.bias), y) == 0
    assert lib.w8a8_quant_matmul_noalloc_status(torch.cuda.current_stream().cuda_stream) == 0
    assert np.array_equal(host_bits(y), oracle.quant_matmul(q, xs, d.w, d.w_scale, d.bias))


def test_noalloc_refuses_problems_whose_counters_do_not_fit():
    lib = _capi.lib()
    fake = ctypes.c_void_p(256)
    # 65536 x 65536 outputs need 4 Mi arrival counters (16 MiB): more than the built-in array; refused
    # before anything is read or launched
    rc = lib.w8a8_quant_matmul_noalloc(fake, fake, 65536, 64, fake, fake, 65536, None, fake, None)
    assert rc == _capi.W8A8_ERR_WORKSPACE
