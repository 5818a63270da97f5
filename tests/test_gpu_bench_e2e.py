"""The bench's end-to-end leg: host inputs copied in, the public calls, the result copied back, with the
copies of one step overlapping the compute of its neighbours (two buffer slots, three streams).  These
tests check that the overlap does not corrupt anything.  Every step's host result must equal the oracle's
output for the same inputs, bit for bit, at the dense tiny and decode configs and on a small MoE layer.
The reduced MoE case that profiler captures use must build and run."""
import os
import sys

import numpy as np
import pytest
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu


def _host_bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("cfg", [1, 2])
def test_pipelined_e2e_dense_results_match_the_oracle(cfg):
    import bench
    dev = torch.device("cuda")
    wl = bench.make_workload(cfg, dev)
    wl.e2e_setup(dev)
    steps = 5  # more than the two slots: every slot is reused while the other one is in flight
    for slot in range(bench.E2E_SLOTS):
        wl.e2e_slots[slot]["hy"].fill_(0)
    bench.run_e2e(torch, wl, steps)
    d = wl.d
    q, xs = oracle.dynamic_quant(d.x)
    ref = oracle.quant_matmul(q, xs, d.w, d.w_scale, d.bias)
    for slot in range(bench.E2E_SLOTS):
        assert np.array_equal(_host_bits(wl.e2e_slots[slot]["hy"]), ref), f"slot {slot}"


def test_pipelined_e2e_moe_results_match_the_direct_call():
    """A quarter-size MoE prefill layer (the reduced case): the pipelined host results equal one direct
    call of the same layer, which the parity tests pin to the oracle."""
    import bench
    import w8a8_dynamic_quant_gb300 as W
    dev = torch.device("cuda")
    wl = bench.make_workload(4, dev, moe_scale=16)
    assert wl.m.E == 4 and wl.m.T == 256
    y = W.moe_w13_swiglu_requant_w2(wl.x, wl.xs, wl.gl, wl.w13p, wl.s13, wl.w2p, wl.s2, wl.ws)
    torch.cuda.synchronize()
    ref = _host_bits(y.cpu())
    wl.e2e_setup(dev)
    bench.run_e2e(torch, wl, 5)
    for slot in range(bench.E2E_SLOTS):
        assert np.array_equal(_host_bits(wl.e2e_slots[slot]["hy"]), ref), f"slot {slot}"
