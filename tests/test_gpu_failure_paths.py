"""Device-side failure paths, exercised without a fault or a hang.

A bounded mbarrier wait that runs out must leave W8A8_ERR_DEVICE_TIMEOUT in
the workspace's status word and return, with the CUDA context still usable:
the library's self-check kernel waits, with the helper every tensor-core
kernel uses, on an mbarrier that nobody arrives on and no copy completes on,
under a 50 ms limit.  Data-dependent errors (a group list whose counts do not
sum to R, a packed weight whose header does not match the call) must come
back through the status word with nothing written."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_dynamic_quant_gb300 as W
from w8a8_dynamic_quant_gb300 import _capi
from w8a8_dynamic_quant_gb300 import synthetic as S

from gpu_helpers import dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_with_timeout_status_and_context_stays_usable():
    ws = W.workspace(_capi.STATUS_BYTES, "cuda")
    lib = _capi.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        assert lib.w8a8_selftest_bounded_wait(ws.data_ptr(), 50000, stream) == 0
        assert W.read_device_status(ws) == _capi.W8A8_ERR_DEVICE_TIMEOUT
        assert W.read_device_status(ws) == 0, "reading the status clears it"
    # the context still runs work correctly
    d = S.dense_config(1)
    q, s = W.w8a8_dynamic_quant(dev_bf16(d.x))
    torch.cuda.synchronize()
    q_ref, _ = oracle.dynamic_quant(d.x)
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_bounded_wait_rejects_out_of_range_limits():
    lib = _capi.lib()
    ws = W.workspace(_capi.STATUS_BYTES, "cuda")
    assert lib.w8a8_selftest_bounded_wait(ws.data_ptr(), 0, None) == 2
    assert lib.w8a8_selftest_bounded_wait(ws.data_ptr(), 2000001, None) == 2
    assert lib.w8a8_selftest_bounded_wait(None, 1000, None) == _capi.W8A8_ERR_WORKSPACE


def test_mismatched_pack_is_reported_and_nothing_written():
    d = S.dense_config(1)
    q, xs = oracle.dynamic_quant(d.x)
    wp = W.w8a8_prepack_weight(dev(d.w))  # header: N = 256
    n_wrong = d.N // 2
    ws = W.workspace(W.quant_matmul_workspace_bytes(d.M, n_wrong, d.K), "cuda")
    y = torch.full((d.M, n_wrong), 5.0, dtype=torch.bfloat16, device="cuda")
    W.w8a8_quant_matmul(dev(q), dev(xs), wp, dev(d.w_scale)[:n_wrong].contiguous(), n_wrong, None, ws=ws, y=y)
    assert W.read_device_status(ws) == _capi.W8A8_ERR_PACKED
    assert bool((y == 5.0).all())
    assert host_bits(y).shape == (d.M, n_wrong)
