"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs.  INT8 payloads, FP32 scales and INT32 accumulators must
be bit-exact; BF16 outputs must be within 1 bf16 ulp (the contract) and are in
fact checked bitwise, because both sides evaluate the same binary32 steps.
Full-size workloads are checked on sampled rows."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import w8a8_dynamic_quant_gb300 as W
from w8a8_dynamic_quant_gb300 import synthetic as S

from gpu_helpers import (bf16_ulp_diff, dev, dev_bf16, f32_bits, host_bits, moe_subset_oracle,
                         sample_rows)

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def gpu_quant(x_bits):
    q, s = W.w8a8_dynamic_quant(dev_bf16(x_bits))
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def assert_quant_equal(x_bits):
    q, s = gpu_quant(x_bits)
    qr, sr = oracle.dynamic_quant(x_bits)
    assert np.array_equal(f32_bits(s), f32_bits(sr)), "scales differ"
    bad = np.argwhere(q != qr)
    assert bad.size == 0, f"{len(bad)} int8 codes differ, first {bad[:4]}"


# ------------------------------------------------------------------ quant ----

@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_quant_dense_configs(cfg):
    assert_quant_equal(S.dense_config(cfg).x)


def test_quant_moe_prefill_routed_rows():
    c = S.CONFIGS[4]
    rng = S.rng_for(0)
    x = S.to_bf16_bits(rng.standard_normal((c["T"], c["H"]), dtype=np.float32))
    ids, _ = S.route(rng, c["T"], c["E"], c["topk"], c["routing"], c["zipf_s"], c["n_dead"])
    ti, _ = S.expert_sorted_rows(ids, c["E"])
    assert_quant_equal(x[ti])


@pytest.mark.parametrize("M,K", [(1, 16), (37, 48), (5, 2048), (9, 2064), (3, 20000), (300, 128)])
def test_quant_shapes(M, K):
    rng = np.random.default_rng(M * 7 + K)
    x = rng.standard_normal((M, K)).astype(np.float32) * np.float32(4)
    assert_quant_equal(S.to_bf16_bits(x))


def test_quant_edge_rows():
    K = 256
    rows = [np.zeros(K, np.float32), np.full(K, 0.3, np.float32), np.full(K, -7.0, np.float32),
            np.resize(np.float32([127, 62.5, 2.5, -0.5, 0.5, -2.5, 1.5, -3.5, 126.5, -125.5]), K),
            np.float32(np.random.default_rng(0).standard_normal(K)) * np.float32(1e-38),
            np.float32(np.random.default_rng(1).standard_normal(K)) * np.float32(1e36)]
    oh = np.zeros(K, np.float32)
    oh[100] = -3.0
    rows.append(oh)
    assert_quant_equal(S.to_bf16_bits(np.stack(rows)))


def test_quant_quotients_at_and_near_half_integers():
    """Rows whose quotients x / s sit exactly on, or within a few binary32 ulps
    of, the half-integers where rounding changes: the kernels take their
    exact-division path there and must still agree bit for bit."""
    K = 256
    ks = np.arange(-127, 127, dtype=np.float32)
    rows = []
    for e in (-20, -3, 0, 5, 40):  # s = 2^e exactly when the row's absmax is 127 * 2^e
        base = np.float32(2.0 ** e)
        ties = (ks + np.float32(0.5)) * base
        row = np.resize(ties, K)
        row[0] = np.float32(127) * base
        rows.append(row)
    # absmax not a multiple of 127: s is inexact and the quotients land near, not on, the ties
    rng = np.random.default_rng(5)
    for amax in (np.float32(126.9), np.float32(100.25), np.float32(3.0e-3), np.float32(7.77e20)):
        s = np.float32(amax / np.float32(127))
        near = (rng.integers(-127, 127, K).astype(np.float32) + np.float32(0.5)) * s
        near = near * (np.float32(1) + rng.integers(-4, 5, K).astype(np.float32) * np.float32(2.0 ** -20))
        near[0] = amax
        rows.append(near)
    x = np.stack(rows).astype(np.float32)
    assert_quant_equal(S.to_bf16_bits(x))
    # the rows do hold many exact ties after rounding to bf16
    xb = S.bf16_bits_to_f32(S.to_bf16_bits(x))
    q, s = oracle.dynamic_quant(S.to_bf16_bits(x))
    quot = xb / s[:, None]
    assert np.count_nonzero(np.abs(quot - np.rint(quot)) == 0.5) > 500


@pytest.mark.parametrize("M,K", [(2437, 16), (4096, 256), (2500, 2064), (3001, 4096), (2433, 8192),
                                 (2440, 8208)])
def test_quant_many_rows(M, K):
    """Row sets that fill every SM several times over, rows of 32 B to 16 KB, row counts that leave the
    last CTAs with one row fewer; the rows mix random values, exact ties, zeros and extremes."""
    rng = np.random.default_rng(M + K)
    x = rng.standard_normal((M, K)).astype(np.float32) * np.float32(3)
    ks = np.arange(-127, 127, dtype=np.float32)
    for i in range(0, M, 7):  # every 7th row: quotients exactly on half-integers (s = 2^e)
        base = np.float32(2.0 ** int(rng.integers(-20, 20)))
        x[i] = np.resize((ks + np.float32(0.5)) * base, K)
        x[i, int(rng.integers(0, K))] = np.float32(127) * base
    x[3] = 0.0
    x[5] *= np.float32(1e-38)
    x[M - 1] *= np.float32(1e36)
    assert_quant_equal(S.to_bf16_bits(x))


def test_quant_every_scale_near_half_integers():
    """One row for every positive finite bf16 absmax (32639 rows, so every scale s = amax / 127 the
    quantiser can meet): the row holds its absmax and, for each half-integer h = k + 0.5 (k = 0 .. 126),
    the four bf16 values bracketing h * s, with alternating signs.  These are the quotients where a
    reciprocal product can round to the wrong side; the codes must still be those of the binary32
    quotient, for the tiny scales (exact path) as for the rest."""
    amax_bits = np.arange(1, 0x7F80, dtype=np.uint32)  # 0x0001 .. 0x7F7F
    amax = (amax_bits << 16).view(np.float32)
    s = (amax / np.float32(127)).astype(np.float32)
    h = np.arange(127, dtype=np.float64) + 0.5
    t = h[None, :] * s[:, None].astype(np.float64)  # exact in binary64
    lo = (t.astype(np.float32).view(np.uint32) >> 16).astype(np.int64)  # bf16 at or below h * s
    cand = np.stack([lo - 1, lo, lo + 1, lo + 2], axis=2).reshape(len(amax_bits), -1)
    cand = np.clip(cand, 0, amax_bits[:, None].astype(np.int64))  # |x| <= amax
    sign = np.where((np.arange(cand.shape[1]) // 4) % 2 == 1, 0x8000, 0)[None, :]
    K = 512
    x = np.zeros((len(amax_bits), K), dtype=np.uint16)
    x[:, 0] = amax_bits
    x[:, 1:1 + cand.shape[1]] = (cand | sign).astype(np.uint16)
    assert_quant_equal(x)


def test_quant_empty_is_noop():
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    q, s = W.w8a8_dynamic_quant(x)
    assert q.shape == (0, 64) and s.shape == (0,)


# ------------------------------------------------------------ dense GEMM ----

def gpu_dense(d, want_acc=True, flags=0):
    q, xs = oracle.dynamic_quant(d.x)
    wp = W.w8a8_prepack_weight(dev(d.w), flags)
    y = W.w8a8_quant_matmul(dev(q), dev(xs), wp, dev(d.w_scale), d.N,
                            None if d.bias is None else dev_bf16(d.bias))
    acc = W.w8a8_int8_matmul_acc(dev(q), wp, d.N) if want_acc else None
    torch.cuda.synchronize()
    return q, xs, host_bits(y), (acc.cpu().numpy() if want_acc else None)


@pytest.mark.parametrize("cfg", [1, 2])
def test_dense_configs_exact(cfg):
    d = S.dense_config(cfg)
    q, xs, y, acc = gpu_dense(d)
    acc_ref = oracle.int8_gemm_acc(q, d.w)
    assert np.array_equal(acc, acc_ref)
    y_ref = oracle.quant_matmul(q, xs, d.w, d.w_scale, d.bias)
    assert bf16_ulp_diff(y, y_ref).max() <= 1
    assert np.array_equal(y, y_ref)


def test_dense_prefill_config_sampled_rows():
    d = S.dense_config(3)
    q, xs = oracle.dynamic_quant(d.x)
    wp = W.w8a8_prepack_weight(dev(d.w))
    qd = dev(q)
    y = W.w8a8_quant_matmul(qd, dev(xs), wp, dev(d.w_scale), d.N)
    acc = W.w8a8_int8_matmul_acc(qd, wp, d.N)
    rows = sample_rows(d.M, 40)
    y_s = host_bits(y[torch.as_tensor(rows, device="cuda")])
    acc_s = acc[torch.as_tensor(rows, device="cuda")].cpu().numpy()
    assert np.array_equal(acc_s, oracle.int8_gemm_acc(q[rows], d.w))
    assert np.array_equal(y_s, oracle.quant_matmul(q[rows], xs[rows], d.w, d.w_scale, None))


@pytest.mark.parametrize("M,N,K,bias", [(37, 200, 80, True), (1, 1, 16, False), (130, 129, 1040, True),
                                        (64, 384, 2064, False), (200, 256, 7168, True)])
def test_dense_ragged_shapes(M, N, K, bias):
    d = S.make_dense(M, K, N, n_outlier=min(3, K), outlier_mult=10.0, bias=bias, seed=M + N + K)
    q, xs, y, acc = gpu_dense(d)
    assert np.array_equal(acc, oracle.int8_gemm_acc(q, d.w))
    assert np.array_equal(y, oracle.quant_matmul(q, xs, d.w, d.w_scale, d.bias))


def test_accumulation_exact_at_extremes():
    """Sums far beyond 2^24 (the fp32 integer range) stay exact: the fp32
    partial sums are drained to int32 every 1024 products."""
    K = 65536
    q = np.full((4, K), 127, np.int8)
    q[1] = -127
    q[2] = -128
    q[3, ::2] = -127
    w = np.full((8, K), 127, np.int8)
    w[1] = -128
    w[2, : K // 2] = 1          # large then small: low bits of a big partial sum
    w[3, ::3] = -127
    wp = W.w8a8_prepack_weight(dev(w))
    acc = W.w8a8_int8_matmul_acc(dev(q), wp, 8).cpu().numpy()
    ref = q.astype(np.int64) @ w.astype(np.int64).T
    assert np.array_equal(acc.astype(np.int64), ref)
    assert ref.max() >= 2 ** 30


def test_dense_workspace_left_zeroed_and_reusable():
    d = S.dense_config(2)
    q, xs = oracle.dynamic_quant(d.x)
    wp = W.w8a8_prepack_weight(dev(d.w))
    ws = W.workspace(W.quant_matmul_workspace_bytes(d.M, d.N, d.K))
    outs = []
    for _ in range(3):
        outs.append(host_bits(W.w8a8_quant_matmul(dev(q), dev(xs), wp, dev(d.w_scale), d.N, ws=ws)))
    torch.cuda.synchronize()
    assert W.read_device_status(ws) == 0
    # what must start at zero is zero again: the arrival counters at the end
    nblk = (d.N + 127) // 128
    assert int(ws[-256:].count_nonzero()) == 0 and nblk * 8 <= 256
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    assert np.array_equal(outs[0], oracle.quant_matmul(q, xs, d.w, d.w_scale, None))


def test_packed_header_mismatch_reports_status():
    d = S.dense_config(1)
    q, xs = oracle.dynamic_quant(d.x)
    wp = W.w8a8_prepack_weight(dev(d.w))
    ws = W.workspace(W.quant_matmul_workspace_bytes(d.M, d.N - 128, d.K))
    y = torch.full((d.M, d.N - 128), 7.0, dtype=torch.bfloat16, device="cuda")
    W.w8a8_quant_matmul(dev(q), dev(xs), wp, dev(d.w_scale[:128]), d.N - 128, ws=ws, y=y)
    assert W.read_device_status(ws) == 9
    assert bool((y == 7.0).all())
    assert W.read_device_status(ws) == 0  # cleared by the read


# ---------------------------------------------------------- grouped GEMM ----

def grouped_case(gl, K, N, seed):
    rng = np.random.default_rng(seed)
    R = int(np.sum(gl))
    E = len(gl)
    x = S.to_bf16_bits(rng.standard_normal((R, K)).astype(np.float32))
    q, xs = oracle.dynamic_quant(x)
    w = rng.integers(-127, 128, (E, N, K), dtype=np.int8)
    ws_ = rng.uniform(1e-3, 1e-2, (E, N)).astype(np.float32)
    return q, xs, np.asarray(gl, np.int64), w, ws_


def check_grouped(q, xs, gl, w, wsc):
    E, N, K = w.shape
    wp = W.w8a8_prepack_weight(dev(w))
    R = q.shape[0]
    y = torch.full((R, N), 3.0, dtype=torch.bfloat16, device="cuda")
    y = W.w8a8_grouped_matmul(dev(q), dev(xs), dev(gl), wp, dev(wsc), y=y)
    acc = W.w8a8_grouped_matmul_acc(dev(q), dev(gl), wp, N)
    torch.cuda.synchronize()
    y_ref, acc_ref = oracle.grouped_matmul(q, xs, gl, w, wsc, want_acc=True)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert np.array_equal(host_bits(y), y_ref)


def test_grouped_golden_example():
    with open(os.path.join(GOLDEN, "group_list_example.json")) as f:
        gl = json.load(f)["group_list"]
    check_grouped(*grouped_case(gl, 512, 256, 1))


@pytest.mark.parametrize("gl,K,N", [([0, 5, 0, 0, 77, 1, 0, 40, 0], 272, 320),
                                    ([300], 128, 128), ([0, 0, 64, 0], 64, 200),
                                    ([3, 9, 1, 17, 2, 0, 4, 8] * 4, 1024, 256)])
def test_grouped_ragged(gl, K, N):
    check_grouped(*grouped_case(gl, K, N, len(gl) + K))


def test_grouped_bad_group_list_sets_status_and_writes_nothing():
    q, xs, gl, w, wsc = grouped_case([10, 0, 6], 64, 128, 3)
    wp = W.w8a8_prepack_weight(dev(w))
    for bad in ([10, 0, 7], [17, -1, 0]):
        ws = W.workspace(W.grouped_matmul_workspace_bytes(3, 16, 128, 64))
        y = torch.full((16, 128), 5.0, dtype=torch.bfloat16, device="cuda")
        W.w8a8_grouped_matmul(dev(q), dev(xs), dev(np.array(bad, np.int64)), wp, dev(wsc), ws=ws, y=y)
        assert W.read_device_status(ws) == 5
        assert bool((y == 5.0).all())


# -------------------------------------------------------------- MoE chain ----

def moe_gpu(m, ws=None, flags13=W.PACK_GATE_UP, flags2=0):
    w13p = W.w8a8_prepack_weight(m.w13.cuda(), flags13)
    w2p = W.w8a8_prepack_weight(m.w2.cuda(), flags2)
    if m.x_scale is None:
        x, xs = dev_bf16(m.x), None
    else:
        x, xs = dev(m.x), dev(m.x_scale)
    ws = W.workspace(W.moe_workspace_bytes(m.R, m.H, m.I, m.E)) if ws is None else ws
    y = W.moe_w13_swiglu_requant_w2(x, xs, dev(m.group_list), w13p, dev(m.s13), w2p, dev(m.s2), ws=ws)
    torch.cuda.synchronize()
    return host_bits(y), ws


def ws_slice(ws, m, which, dtype, shape):
    off = W.moe_workspace_offset(m.R, m.H, m.I, m.E, which)
    n = int(np.prod(shape)) * np.dtype(dtype).itemsize
    return ws[off:off + n].cpu().numpy().view(dtype).reshape(shape)


@pytest.mark.parametrize("prequant", [False, True])
def test_moe_small_full_with_intermediates(prequant):
    m = S.make_moe(T=70, H=256, I=128, E=8, topk=2, routing="zipf", zipf_s=1.1, n_dead=2,
                   prequant=prequant, seed=11)
    y, ws = moe_gpu(m)
    x_in = m.x
    y_ref, it = oracle.moe_w13_swiglu_requant_w2(x_in, m.x_scale, m.group_list, m.w13.numpy(), m.s13,
                                                 m.w2.numpy(), m.s2, intermediates=True)
    if not prequant:
        assert np.array_equal(ws_slice(ws, m, 0, np.int8, (m.R, m.H)), it["xq"])
        assert np.array_equal(f32_bits(ws_slice(ws, m, 1, np.float32, (m.R,))), f32_bits(it["xs"]))
    assert np.array_equal(ws_slice(ws, m, 2, np.uint16, (m.R, m.I)), it["h"])
    assert np.array_equal(ws_slice(ws, m, 3, np.int8, (m.R, m.I)), it["hq"])
    assert np.array_equal(f32_bits(ws_slice(ws, m, 4, np.float32, (m.R,))), f32_bits(it["hs"]))
    assert np.array_equal(y, y_ref)


def test_moe_prequantised_input_is_not_quantised_again():
    m = S.make_moe(T=50, H=192, I=64, E=5, topk=2, routing="uniform", seed=4)
    y_bf16_path, ws = moe_gpu(m)
    xq = ws_slice(ws, m, 0, np.int8, (m.R, m.H)).copy()
    xs = ws_slice(ws, m, 1, np.float32, (m.R,)).copy()
    m.x, m.x_scale = xq, xs
    y_int8_path, _ = moe_gpu(m)
    assert np.array_equal(y_bf16_path, y_int8_path)


def test_moe_bad_group_list():
    m = S.make_moe(T=20, H=64, I=64, E=4, topk=2, seed=2)
    m.group_list = m.group_list.copy()
    m.group_list[1] += 3
    w13p = W.w8a8_prepack_weight(m.w13.cuda(), W.PACK_GATE_UP)
    w2p = W.w8a8_prepack_weight(m.w2.cuda())
    ws = W.workspace(W.moe_workspace_bytes(m.R, m.H, m.I, m.E))
    y = torch.full((m.R, m.H), 9.0, dtype=torch.bfloat16, device="cuda")
    W.moe_w13_swiglu_requant_w2(dev_bf16(m.x), None, dev(m.group_list), w13p, dev(m.s13), w2p, dev(m.s2),
                                ws=ws, y=y)
    assert W.read_device_status(ws) == 5
    assert bool((y == 9.0).all())


@pytest.mark.parametrize("cfg,n_rows", [(4, 24), (5, 32)])
def test_moe_configs_sampled_rows(cfg, n_rows):
    m = S.moe_config(cfg, device="cuda")
    y, ws = moe_gpu(m)
    rows = sample_rows(m.R, n_rows, seed=cfg)
    y_ref, it = moe_subset_oracle(m, rows)
    assert np.array_equal(ws_slice(ws, m, 2, np.uint16, (m.R, m.I))[rows], it["h"])
    if W.moe_workspace_offset(m.R, m.H, m.I, m.E, 3) >= 0:
        hq = ws_slice(ws, m, 3, np.int8, (m.R, m.I))
    else:  # tensor-core shapes keep the codes as integer-valued fp16 only
        hq = ws_slice(ws, m, 6, np.float16, (m.R, m.I)).astype(np.int8)
    assert np.array_equal(hq[rows], it["hq"])
    assert np.array_equal(y[rows], y_ref)
    # every routed row was written (no row left at the workspace's initial state)
    assert int(np.count_nonzero(np.all(y == 0, axis=1))) == 0
