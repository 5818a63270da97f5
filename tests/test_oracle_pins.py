"""Pins for the CPU oracle against facts that do not come from the oracle itself.

Each check uses a library routine, brute force, a closed form or an invariant
of the method, so that a plausible slip in the oracle (a dropped term, a wrong
divisor, a transposed operand, a swapped gate/up half, an off-by-one group
offset) fails at least one of them.  CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from w8a8_dynamic_quant_gb300 import synthetic as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(b):
    return S.bf16_bits_to_f32(b)


def bf16_ulp(v):
    """Spacing of bf16 numbers at |v| (normal range)."""
    v = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return 2.0 ** (e - 7)


# ------------------------------------------------------------------ bf16 ----

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    vals = rng.standard_normal(4000).astype(np.float32) * np.float32(37.0)
    bits = vals.view(np.uint32)
    # exact ties (low half == 0x8000) with both parities of the kept bit
    ties = ((bits & 0xFFFF0000) | 0x8000).view(np.float32)
    allv = np.concatenate([vals, ties, np.float32([0.0, -0.0, 1e-40, -3.0e38, 3.3895e38])])
    ref = torch.from_numpy(allv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(float(v)) for v in allv], np.uint16)
    assert np.array_equal(got, ref)
    back = np.array([oracle.bf16_to_f32(int(b)) for b in ref[:200]], np.float32)
    assert np.array_equal(back, f32(ref[:200]))


# ------------------------------------------------------------------- exp ----

def _ulp32(v):
    return np.spacing(np.float32(abs(v))).astype(np.float64)


def test_exp_spec_accuracy_and_special_values():
    rng = np.random.default_rng(2)
    xs = np.concatenate([np.linspace(-87.0, 88.5, 20001), rng.uniform(-20, 20, 20000),
                         rng.uniform(-1, 1, 5000)]).astype(np.float32)
    worst = 0.0
    for x in xs:
        got = oracle.exp_f32(float(x))
        ref = math.exp(float(x))
        err = abs(got - ref) / float(_ulp32(ref))
        worst = max(worst, err)
    assert worst <= 2.0, worst
    assert oracle.exp_f32(0.0) == 1.0
    assert oracle.exp_f32(-0.0) == 1.0
    assert math.isinf(oracle.exp_f32(89.5))
    assert oracle.exp_f32(-105.0) == 0.0
    assert math.isnan(oracle.exp_f32(float("nan")))
    # subnormal results stay within one subnormal step of the truth
    for x in np.linspace(-103.9, -87.4, 500).astype(np.float32):
        got = oracle.exp_f32(float(x))
        assert abs(got - math.exp(float(x))) <= 2.0 ** -149 * 1.01 + abs(math.exp(float(x))) * 2 ** -22


# ----------------------------------------------------------------- quant ----

def _rand_bf16_rows(rng, M, K, scale=1.0):
    x = rng.standard_normal((M, K)).astype(np.float32) * np.float32(scale)
    return S.to_bf16_bits(x)


def test_quant_matches_torch_round_half_even():
    """q equals torch's divide-then-round(half-to-even)-then-clamp with the oracle's scale."""
    rng = np.random.default_rng(3)
    x = _rand_bf16_rows(rng, 64, 200, 3.0)
    x[5, :] = S.to_bf16_bits(np.float32(rng.integers(-4, 5, 200)))  # many exact .5 quotients
    # amax 127 gives s == 1 exactly, so these are exact ties at odd and even halves
    ties = np.float32([127, 62.5, 2.5, -0.5, 0.5, -2.5, 1.5, -3.5, 126.5, -125.5])
    x[6, :] = S.to_bf16_bits(np.resize(ties, 200))
    q, s = oracle.dynamic_quant(x)
    xt = torch.from_numpy(f32(x))
    st = torch.from_numpy(s)[:, None]
    ref = torch.round(xt / st).clamp(-127, 127).to(torch.int8).numpy()
    assert np.array_equal(q, ref)


def test_quant_brute_force_argmin():
    """q is the nearest integer multiple of s to x (ties to even) except at fp32 near-ties."""
    rng = np.random.default_rng(4)
    x = _rand_bf16_rows(rng, 40, 33, 2.0)
    q, s = oracle.dynamic_quant(x)
    xf = f32(x).astype(np.float64)
    cand = np.arange(-127, 128, dtype=np.float64)
    mism = 0
    for m in range(x.shape[0]):
        for k in range(x.shape[1]):
            d = np.abs(xf[m, k] - cand * float(s[m]))
            best = np.flatnonzero(d <= d.min() * (1 + 1e-15) + 1e-300)
            pick = best[np.argmin(np.abs(cand[best]) % 2)] if best.size > 1 else best[0]
            if int(cand[pick]) != int(q[m, k]):
                mism += 1
                t = xf[m, k] / float(s[m])
                assert abs(abs(t - math.floor(t)) - 0.5) < 2e-6, (m, k, t, q[m, k])
    assert mism <= 2


def test_quant_invariants_and_closed_forms():
    rng = np.random.default_rng(5)
    x = _rand_bf16_rows(rng, 50, 300, 5.0)
    x[0, :] = S.to_bf16_bits(np.full(300, 0.3, np.float32))          # constant row
    x[1, :] = 0                                                        # zero row
    oh = np.zeros(300, np.float32)
    oh[17] = -2.5
    x[2, :] = S.to_bf16_bits(oh)                                       # one-hot negative
    q, s = oracle.dynamic_quant(x)
    xf = f32(x).astype(np.float64)
    amax = np.abs(xf).max(axis=1)
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    assert not np.any(q == -128)
    nz = amax > 0
    # the scale reproduces amax after one multiply by the level count (within 1 ulp)
    assert np.all(np.abs(s[nz].astype(np.float64) * 127.0 - amax[nz]) <= np.spacing(amax[nz].astype(np.float32)))
    # the element of largest magnitude maps to +-127
    am = np.argmax(np.abs(xf), axis=1)
    assert np.all(np.abs(q[nz, am[nz]]) == 127)
    # reconstruction error at most half a step, plus the binary32 rounding of
    # the quotient x/s (|x/s| <= 127, so at most 127 * 2^-24 of a step)
    err = np.abs(xf - q * s[:, None].astype(np.float64))
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 127 * 2.0 ** -24) + 1e-45)
    # closed forms
    assert np.all(q[0] == 127) and s[0] == np.float32(f32(x[0:1, 0:1])[0, 0]) / np.float32(127)
    assert s[1] == 0.0 and np.all(q[1] == 0)
    assert q[2, 17] == -127 and np.count_nonzero(q[2]) == 1


def test_quant_sign_and_power_of_two_invariance():
    rng = np.random.default_rng(6)
    x = _rand_bf16_rows(rng, 20, 128, 1.5)
    q, s = oracle.dynamic_quant(x)
    qn, sn = oracle.dynamic_quant(x ^ np.uint16(0x8000))
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)
    x8 = S.to_bf16_bits(f32(x) * np.float32(8.0))
    q8, s8 = oracle.dynamic_quant(x8)
    assert np.array_equal(q8, q) and np.array_equal(s8, s * np.float32(8.0))


# ------------------------------------------------------------------ GEMM ----

@pytest.mark.parametrize("M,K,N", [(7, 96, 13), (1, 32, 1), (33, 512, 40)])
def test_gemm_acc_matches_int64_matmul(M, K, N):
    rng = np.random.default_rng(M * 1000 + N)
    q = rng.integers(-127, 128, (M, K), dtype=np.int8)
    w = rng.integers(-128, 128, (N, K), dtype=np.int8)
    acc = oracle.int8_gemm_acc(q, w)
    ref = q.astype(np.int64) @ w.astype(np.int64).T
    assert acc.dtype == np.int32 and np.array_equal(acc.astype(np.int64), ref)


def test_gemm_acc_identity_and_extreme():
    rng = np.random.default_rng(7)
    q = rng.integers(-127, 128, (5, 64), dtype=np.int8)
    w = (np.eye(64, dtype=np.int64) * 127).astype(np.int8)
    assert np.array_equal(oracle.int8_gemm_acc(q, w), q.astype(np.int32) * 127)
    K = 4096
    q = np.full((2, K), 127, np.int8)
    q[1] = -127
    w = np.full((3, K), 127, np.int8)
    acc = oracle.int8_gemm_acc(q, w)
    assert acc[0, 0] == K * 16129 and acc[1, 2] == -K * 16129


def test_epilogue_against_float64():
    rng = np.random.default_rng(8)
    M, N = 40, 70
    acc = rng.integers(-(2 ** 27), 2 ** 27, (M, N), dtype=np.int64).astype(np.int32)
    xs = rng.uniform(1e-3, 0.5, M).astype(np.float32)
    ws = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    bias = S.to_bf16_bits(rng.standard_normal(N).astype(np.float32) * np.float32(30))
    for b in (None, bias):
        y = f32(oracle.epilogue(acc, xs, ws, b)).astype(np.float64)
        ref = acc.astype(np.float64) * xs[:, None] * ws[None, :]
        if b is not None:
            ref = ref + f32(b)[None, :]
        assert np.all(np.abs(y - ref) <= bf16_ulp(ref) * 0.5 * 1.01 + 1e-30)


def test_epilogue_closed_forms():
    M, N = 3, 5
    bias = S.to_bf16_bits(np.float32([1.5, -2.0, 0.25, 7.0, -0.125]))
    y = oracle.epilogue(np.zeros((M, N), np.int32), np.ones(M, np.float32), np.ones(N, np.float32), bias)
    assert np.array_equal(y, np.broadcast_to(bias, (M, N)))
    acc = np.arange(-7, 8, dtype=np.int32).reshape(3, 5) * 17
    y = oracle.epilogue(acc, np.ones(M, np.float32), np.ones(N, np.float32), None)
    assert np.array_equal(f32(y), acc.astype(np.float32))


def test_quant_matmul_non_square_against_numpy():
    rng = np.random.default_rng(9)
    M, K, N = 9, 160, 21
    q = rng.integers(-127, 128, (M, K), dtype=np.int8)
    w = rng.integers(-127, 128, (N, K), dtype=np.int8)
    xs = rng.uniform(1e-2, 1e-1, M).astype(np.float32)
    ws = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    bias = S.to_bf16_bits(rng.standard_normal(N).astype(np.float32))
    y = f32(oracle.quant_matmul(q, xs, w, ws, bias)).astype(np.float64)
    ref = (q.astype(np.float64) @ w.astype(np.float64).T) * xs[:, None] * ws[None, :] + f32(bias)[None, :]
    assert np.all(np.abs(y - ref) <= bf16_ulp(ref) * 0.5 * 1.01 + 1e-30)


# --------------------------------------------------------------- grouped ----

def _golden_groups():
    with open(os.path.join(GOLDEN, "group_list_example.json")) as f:
        g = json.load(f)
    return np.array(g["group_list"], np.int64), int(g["R"])


def test_grouped_golden_example_against_numpy():
    gl, R = _golden_groups()
    assert gl.sum() == R
    E, K, N = gl.shape[0], 64, 24
    rng = np.random.default_rng(10)
    q = rng.integers(-127, 128, (R, K), dtype=np.int8)
    xs = rng.uniform(1e-2, 1e-1, R).astype(np.float32)
    w = rng.integers(-127, 128, (E, N, K), dtype=np.int8)
    w[2] = 127  # the empty expert: any use of it would show
    ws = rng.uniform(1e-3, 1e-2, (E, N)).astype(np.float32)
    y, acc = oracle.grouped_matmul(q, xs, gl, w, ws, want_acc=True)
    off = np.concatenate([[0], np.cumsum(gl)])
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        ref_acc = q[rows].astype(np.int64) @ w[e].astype(np.int64).T
        assert np.array_equal(acc[rows].astype(np.int64), ref_acc)
        ref = ref_acc * xs[rows, None].astype(np.float64) * ws[e][None, :]
        got = f32(y[rows]).astype(np.float64)
        assert np.all(np.abs(got - ref) <= bf16_ulp(ref) * 0.5 * 1.01 + 1e-30)


def test_grouped_rejects_bad_group_lists():
    q = np.zeros((10, 32), np.int8)
    xs = np.ones(10, np.float32)
    w = np.zeros((3, 8, 32), np.int8)
    ws = np.ones((3, 8), np.float32)
    for bad in ([5, 4, 0], [5, 6, 0], [11, -1, 0]):
        assert oracle.check_group_list(np.array(bad), 10) != 0
        with pytest.raises(oracle.OracleError) as ei:
            oracle.grouped_matmul(q, xs, np.array(bad, np.int64), w, ws)
        assert ei.value.code == 5
    assert oracle.check_group_list(np.array([10, 0, 0]), 10) == 0


def test_synthetic_routing_rows_sum_to_tokens_times_topk():
    for cfg in (4, 5):
        c = S.CONFIGS[cfg]
        rng = S.rng_for(0)
        ids, p = S.route(rng, c["T"], c["E"], c["topk"], c["routing"], c.get("zipf_s", 1.1), c.get("n_dead", 0))
        assert all(len(set(r)) == c["topk"] for r in ids[:200])
        ti, cnt = S.expert_sorted_rows(ids, c["E"])
        assert cnt.sum() == c["T"] * c["topk"] == ti.shape[0]
        if cfg == 4:
            assert (cnt == 0).sum() >= 1
        assert oracle.check_group_list(cnt, cnt.sum()) == 0


# ---------------------------------------------------------------- SwiGLU ----

def test_swiglu_against_float64_and_closed_forms():
    rng = np.random.default_rng(11)
    R, I = 30, 64
    y13 = S.to_bf16_bits(rng.standard_normal((R, 2 * I)).astype(np.float32) * np.float32(6))
    y13[0, :I] = 0                                              # gate 0 -> h 0
    y13[1, :I] = S.to_bf16_bits(np.full(I, 60.0, np.float32))   # saturated gate: h = g*u
    y13[2, :I] = S.to_bf16_bits(np.full(I, -120.0, np.float32)) # exp overflow: h = -0
    h = oracle.swiglu(y13, I)
    g = f32(y13[:, :I]).astype(np.float64)
    u = f32(y13[:, I:]).astype(np.float64)
    ref = g / (1.0 + np.exp(-g)) * u
    got = f32(h).astype(np.float64)
    assert np.all(np.abs(got - ref) <= bf16_ulp(ref) * 0.5 * 1.02 + 1e-30)
    assert np.all(got[0] == 0)
    assert np.array_equal(h[1], S.to_bf16_bits((np.float32(60.0) * f32(y13[1, I:]))))
    assert np.all(got[2] == 0)


def test_swiglu_gate_is_first_half():
    I = 8
    y13 = np.zeros((1, 2 * I), np.uint16)
    y13[0, :I] = S.to_bf16_bits(np.full(I, 40.0, np.float32))  # gate
    y13[0, I:] = S.to_bf16_bits(np.full(I, 1.0, np.float32))   # up
    h = f32(oracle.swiglu(y13, I))
    assert np.allclose(h, 40.0)  # the other order would give silu(1)*40 ~ 29.2


# ------------------------------------------------------------- MoE chain ----

def _small_moe(prequant=False, seed=0):
    return S.make_moe(T=40, H=96, I=48, E=6, topk=2, routing="zipf", zipf_s=1.1, n_dead=1,
                      prequant=prequant, seed=seed)


def test_moe_chain_composition_and_no_double_quant():
    m = _small_moe()
    w13, w2 = m.w13.numpy(), m.w2.numpy()
    y, it = oracle.moe_w13_swiglu_requant_w2(m.x, None, m.group_list, w13, m.s13, w2, m.s2,
                                             intermediates=True)
    q, s = oracle.dynamic_quant(m.x)
    assert np.array_equal(it["xq"], q) and np.array_equal(it["xs"], s)
    assert np.array_equal(it["y13"], oracle.grouped_matmul(q, s, m.group_list, w13, m.s13))
    assert np.array_equal(it["h"], oracle.swiglu(it["y13"], m.I))
    hq, hs = oracle.dynamic_quant(it["h"])
    assert np.array_equal(it["hq"], hq) and np.array_equal(it["hs"], hs)
    assert np.array_equal(y, oracle.grouped_matmul(hq, hs, m.group_list, w2, m.s2))
    # already-quantised input with its scale is used as is: bit-identical output
    y2 = oracle.moe_w13_swiglu_requant_w2(it["xq"], it["xs"], m.group_list, w13, m.s13, w2, m.s2)
    assert np.array_equal(y, y2)


def test_moe_chain_close_to_float64_reference():
    m = _small_moe(seed=3)
    w13 = m.w13.numpy().astype(np.float64)
    w2 = m.w2.numpy().astype(np.float64)
    y = f32(oracle.moe_w13_swiglu_requant_w2(m.x, None, m.group_list, m.w13.numpy(), m.s13,
                                             m.w2.numpy(), m.s2)).astype(np.float64)
    x = f32(m.x).astype(np.float64)
    off = np.concatenate([[0], np.cumsum(m.group_list)])
    ref = np.zeros_like(y)
    for e in range(m.E):
        rows = slice(off[e], off[e + 1])
        if off[e] == off[e + 1]:
            continue
        y13 = (x[rows] @ w13[e].T) * m.s13[e][None, :]
        g, u = y13[:, :m.I], y13[:, m.I:]
        h = g / (1 + np.exp(-g)) * u
        ref[rows] = (h @ w2[e].T) * m.s2[e][None, :]
    # both sides quantise activations twice with 8-bit codes: allow a few percent of the row scale
    scale = np.abs(ref).max(axis=1, keepdims=True) + 1e-30
    assert np.max(np.abs(y - ref) / scale) < 0.06
    assert np.corrcoef(y.ravel(), ref.ravel())[0, 1] > 0.999


def test_moe_prequant_case_runs_and_rejects_bad_groups():
    m = _small_moe(prequant=True, seed=5)
    assert m.x.dtype == np.int8 and m.x_scale is not None
    y = oracle.moe_w13_swiglu_requant_w2(m.x, m.x_scale, m.group_list, m.w13.numpy(), m.s13,
                                         m.w2.numpy(), m.s2)
    assert y.shape == (m.R, m.H)
    bad = m.group_list.copy()
    bad[0] += 1
    with pytest.raises(oracle.OracleError):
        oracle.moe_w13_swiglu_requant_w2(m.x, m.x_scale, bad, m.w13.numpy(), m.s13, m.w2.numpy(), m.s2)


# ------------------------------------------------- route, permute, combine ----

def _ids(T, k, E, seed, distinct=True):
    rng = np.random.default_rng(seed)
    if distinct and T == 0:
        return np.zeros((0, k), np.int64)
    if distinct:
        return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int64)
    return rng.integers(0, E, size=(T, k), dtype=np.int64)


@pytest.mark.parametrize("T,k,E,distinct", [(50, 4, 9, True), (31, 3, 5, False), (17, 1, 4, True),
                                            (0, 2, 3, True), (64, 8, 300, True)])
def test_route_is_a_stable_sort_by_expert(T, k, E, distinct):
    ids = _ids(T, k, E, seed=T + k + E, distinct=distinct)
    g, pos = oracle.moe_route(ids, E)
    flat = ids.ravel()
    # library pins: counts are a histogram; the routed order is numpy's stable sort of the ids
    assert np.array_equal(g, np.bincount(flat, minlength=E))
    order = np.argsort(flat, kind="stable")
    want = np.empty(T * k, np.int64)
    want[order] = np.arange(T * k)
    assert np.array_equal(pos.ravel().astype(np.int64), want)
    # rows of expert e are the block [sum_{e'<e} g, + g[e]) of the routed order
    off = np.concatenate([[0], np.cumsum(g)])
    assert np.all((pos.ravel() >= off[flat]) & (pos.ravel() < off[flat + 1]))


def test_route_matches_synthetic_expert_rows():
    m = _small_moe(seed=7)
    g, pos = oracle.moe_route(m.topk_ids, m.E)
    assert np.array_equal(g, m.group_list)
    token_of_row = np.empty(m.R, np.int64)
    token_of_row[pos.ravel()] = np.repeat(np.arange(m.T), m.topk)
    assert np.array_equal(token_of_row, m.token_index)


def test_route_rejects_ids_outside_the_experts():
    ids = _ids(5, 2, 4, seed=1)
    for bad in (4, -1):
        ids2 = ids.copy()
        ids2[3, 1] = bad
        try:
            oracle.moe_route(ids2, 4)
            code = 0
        except oracle.OracleError as e:
            code = e.code
        assert code == 10


@pytest.mark.parametrize("prequant", [False, True])
def test_permute_quant_is_quant_of_the_gathered_rows(prequant):
    m = _small_moe(prequant=prequant, seed=11)
    xq, xs, g, pos = oracle.moe_permute_quant(m.x_tok, m.x_tok_scale, m.topk_ids, m.E)
    assert np.array_equal(g, m.group_list)
    if prequant:  # already INT8 with a per-token scale: copied, not quantised again
        assert np.array_equal(xq, m.x_tok[m.token_index])
        assert np.array_equal(xs.view(np.uint32), m.x_tok_scale[m.token_index].view(np.uint32))
    else:         # quantising a token once and copying it = quantising each routed copy
        q, s = oracle.dynamic_quant(m.x)
        assert np.array_equal(xq, q) and np.array_equal(xs.view(np.uint32), s.view(np.uint32))


def test_combine_against_float64():
    rng = np.random.default_rng(5)
    T, k, H = 23, 6, 40
    ids = _ids(T, k, 11, seed=2)
    _, pos = oracle.moe_route(ids, 11)
    yr = S.to_bf16_bits(rng.standard_normal((T * k, H)).astype(np.float32) * np.float32(3))
    w = rng.uniform(-1, 1, (T, k)).astype(np.float32)
    y = f32(oracle.moe_unpermute_combine(yr, pos, w)).astype(np.float64)
    v = f32(yr).astype(np.float64)[pos.astype(np.int64)]          # [T,k,H]
    terms = w.astype(np.float64)[:, :, None] * v
    exact = terms.sum(axis=1)
    # k binary32 products and sums (error <= k * 2^-24 * sum|terms|), then one bf16 rounding
    bound = bf16_ulp(exact) * 0.5 * 1.01 + k * 2.0 ** -24 * np.abs(terms).sum(axis=1) * 1.01
    assert np.all(np.abs(y - exact) <= bound)


def test_combine_closed_forms_and_order():
    rng = np.random.default_rng(6)
    T, H = 9, 24
    yr = S.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    pos = rng.permutation(T).astype(np.int32).reshape(T, 1)
    # one choice with weight 1: the routed row comes back unchanged
    assert np.array_equal(oracle.moe_unpermute_combine(yr, pos, np.ones((T, 1), np.float32)),
                          yr[pos[:, 0]])
    # weights 0: +0 everywhere
    assert np.all(oracle.moe_unpermute_combine(yr, pos, np.zeros((T, 1), np.float32)) == 0)
    # two equal halves of one row give the row back exactly
    yr2 = np.concatenate([yr, yr])
    pos2 = np.stack([np.arange(T), np.arange(T) + T], axis=1).astype(np.int32)
    assert np.array_equal(oracle.moe_unpermute_combine(yr2, pos2, np.full((T, 2), 0.5, np.float32)), yr)
    # slot order, binary32 sums, one final rounding: terms 1+2^-8 then four of 2^-25.  In slot
    # order each small term is lost (a quarter ulp of binary32 at 1) and the bf16 rounding of the
    # tie 1+2^-8 goes to even, 1.0; summed in reverse (or exactly) they reach 1+2^-8+2^-23, which
    # rounds up to 1+2^-7.
    one = S.to_bf16_bits(np.ones((5, 1), np.float32))
    w5 = np.array([[1 + 2.0 ** -8] + [2.0 ** -25] * 4], np.float32)
    p5 = np.arange(5, dtype=np.int32).reshape(1, 5)
    assert oracle.moe_unpermute_combine(one, p5, w5)[0, 0] == 0x3F80
    assert oracle.moe_unpermute_combine(one, p5[:, ::-1].copy(), w5[:, ::-1].copy())[0, 0] == 0x3F81


def test_moe_layer_reduces_to_the_expert_chain():
    """With one choice per token and weight 1, the layer is the expert chain on the
    expert-sorted token rows, put back in token order."""
    m = S.make_moe(T=40, H=96, I=48, E=6, topk=1, routing="zipf", zipf_s=1.1, n_dead=1, seed=13)
    w13, w2 = m.w13.numpy(), m.w2.numpy()
    y = oracle.moe_layer(m.x_tok, None, m.topk_ids, np.ones((m.T, 1), np.float32), w13, m.s13, w2, m.s2)
    y_rows = oracle.moe_w13_swiglu_requant_w2(m.x, None, m.group_list, w13, m.s13, w2, m.s2)
    want = np.empty_like(y)
    want[m.token_index] = y_rows
    assert np.array_equal(y, want)


@pytest.mark.parametrize("prequant", [False, True])
def test_moe_layer_routed_output_and_float64_combine(prequant):
    m = _small_moe(prequant=prequant, seed=17)
    w13, w2 = m.w13.numpy(), m.w2.numpy()
    y, yr = oracle.moe_layer(m.x_tok, m.x_tok_scale, m.topk_ids, m.topk_weights, w13, m.s13, w2, m.s2,
                             want_routed=True)
    # the routed rows are the expert chain's output on the expert-sorted rows
    assert np.array_equal(yr, oracle.moe_w13_swiglu_requant_w2(m.x, m.x_scale, m.group_list, w13, m.s13,
                                                                w2, m.s2))
    # token t's output is the weighted sum of its k routed rows (rows found by the synthetic order)
    row_of = {}
    for r, t in enumerate(m.token_index):
        row_of.setdefault(int(t), []).append(r)
    v = f32(yr).astype(np.float64)
    for t in range(m.T):
        rows = [row_of[t][sorted(m.topk_ids[t]).index(e)] for e in m.topk_ids[t]]
        exact = sum(float(m.topk_weights[t, j]) * v[rows[j]] for j in range(m.topk))
        got = f32(y[t]).astype(np.float64)
        assert np.all(np.abs(got - exact) <= bf16_ulp(exact) * 0.51 + 1e-6 * np.abs(v[rows]).sum(0))


# ------------------------------------------------- per-channel weight quant ----

def test_weight_quant_is_per_output_channel():
    """Channels (rows of W [N,K]) with very different ranges get their own scales: s[n] = max_k |W[n,k]| / 127
    (a per-tensor or per-input-column scale would give other values), the codes reproduce W within s/2, and
    each channel's largest element maps to +-127."""
    rng = np.random.default_rng(21)
    E, N, K = 3, 40, 96
    mags = (2.0 ** rng.integers(-6, 6, (E, N, 1))).astype(np.float32)
    w = S.to_bf16_bits(rng.standard_normal((E, N, K)).astype(np.float32) * mags)
    w[1, 5] = 0  # an all-zero channel: scale 0, codes 0
    q, s = oracle.quantize_weight(w)
    wf = f32(w).astype(np.float64)
    amax = np.abs(wf).max(axis=2)
    assert np.array_equal(s, (amax / 127.0).astype(np.float32))  # exact: binary32 divide of an exact amax
    assert np.all(q[1, 5] == 0) and s[1, 5] == 0
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    err = np.abs(wf - q.astype(np.float64) * s[..., None].astype(np.float64))
    assert np.all(err <= s[..., None].astype(np.float64) * (0.5 + 127 * 2.0 ** -24) + 1e-30)
    big = np.argmax(np.abs(wf), axis=2)
    top = np.take_along_axis(q, big[..., None], axis=2)[..., 0]
    live = amax > 0
    assert np.all(np.abs(top[live]) == 127)
    # a 2-D weight is one expert
    q2, s2 = oracle.quantize_weight(w[2])
    assert np.array_equal(q2, q[2]) and np.array_equal(s2, s[2])


# ------------------------------------------------------------- static W8A8 ----

def test_static_quant_brute_force_and_closed_forms():
    """q = clamp(rint(x/s) + o, -128, 127): against the nearest code of the affine grid s*(c - o) found by
    brute force (ties to the even rint(x/s)), exact grid points, and both clamps."""
    rng = np.random.default_rng(31)
    s, o = np.float32(0.0625), 5
    x = S.to_bf16_bits((rng.standard_normal((6, 64)) * 4).astype(np.float32))
    q = oracle.static_quant(x, s, o).astype(np.int64)
    xf = f32(x).astype(np.float64)
    grid = np.arange(-128, 128)
    dist = np.abs(xf[..., None] - float(s) * (grid - o))          # [6,64,256]
    best = dist.min(axis=-1)
    # the chosen code is a nearest one, and where two are equally near it is the one with rint(x/s) even
    chosen = np.take_along_axis(dist, (q + 128)[..., None], axis=-1)[..., 0]
    assert np.all(chosen <= best + 1e-12)
    tie = (np.sum(dist <= best[..., None] + 1e-12, axis=-1) > 1)
    assert np.all(((q[tie] - o) % 2) == 0)
    # exact grid points, and the clamps
    pts = S.to_bf16_bits((np.float32(s) * np.array([[-3, 0, 7, 100, 5000, -5000]], np.float32)))
    assert oracle.static_quant(pts, s, o).tolist() == [[2, 5, 12, 105, 127, -128]]


def test_static_prepare_against_float64():
    rng = np.random.default_rng(32)
    N, K = 50, 96
    w = rng.integers(-127, 128, (N, K), dtype=np.int8)
    ws = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    bias = S.to_bf16_bits(rng.normal(0, 0.5, N).astype(np.float32))
    s, o = np.float32(0.03), -7
    deq, qb = oracle.static_prepare(w, ws, s, o, bias)
    assert np.array_equal(deq.view(np.uint32), (np.float32(s) * ws).view(np.uint32))
    exact = f32(bias).astype(np.float64) / deq.astype(np.float64) - w.astype(np.int64).sum(axis=1) * o
    assert np.all(np.abs(qb - exact) <= 0.5 + 1e-3 * np.abs(exact) / 2 ** 10 + 1e-6)
    # no bias: just minus the correction, an exact integer
    _, qb0 = oracle.static_prepare(w, ws, s, o, None)
    assert np.array_equal(qb0.astype(np.int64), -w.astype(np.int64).sum(axis=1) * o)


@pytest.mark.parametrize("o", [0, 9, -20])
def test_static_path_approximates_the_float_layer(o):
    """Static quant -> matmul with the prepared deq_scale / quant_bias approximates x @ W_deq^T + bias in
    float64 within the input grid's rounding: the offset correction cancels the zero point (a sign slip
    in it would leave an error of about s * o * sum|W|)."""
    rng = np.random.default_rng(33 + o)
    M, N, K = 12, 40, 256
    s = np.float32(0.02)
    x = S.to_bf16_bits((rng.standard_normal((M, K)) * 0.6).astype(np.float32))
    w = rng.integers(-127, 128, (N, K), dtype=np.int8)
    ws = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    bias = S.to_bf16_bits(rng.normal(0, 0.3, N).astype(np.float32))
    q = oracle.static_quant(x, s, o)
    deq, qb = oracle.static_prepare(w, ws, s, o, bias)
    y = f32(oracle.static_quant_matmul(q, w, deq, qb)).astype(np.float64)
    wd = w.astype(np.float64) * ws[:, None].astype(np.float64)
    ref = f32(x).astype(np.float64) @ wd.T + f32(bias).astype(np.float64)[None, :]
    # per element: K input rounding errors of at most s/2 each times |W_deq|, the bias rounding, bf16
    bound = 0.5 * float(s) * np.abs(wd).sum(axis=1)[None, :] + 0.5 * deq[None, :] + np.abs(ref) * 2.0 ** -8
    assert np.all(np.abs(y - ref) <= bound)
    # exact on the code grid: the same layer on the dequantised input is matched to the output rounding
    xd = float(s) * (q.astype(np.float64) - o)
    ref_q = xd @ wd.T + f32(bias).astype(np.float64)[None, :]
    assert np.all(np.abs(y - ref_q) <= 0.5 * deq[None, :] + np.abs(ref_q) * 2.0 ** -8 * 1.01 + 1e-9)


# -------------------------------------------------------------------- MXFP8 ----

def test_e4m3_encode_decode_against_torch():
    """The E4M3 codes of every BF16 value up to 448 in magnitude equal torch's float8_e4m3fn conversion
    (round to nearest even); every code decodes as torch decodes it; beyond 448 the codes saturate."""
    bits = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    v = f32(bits)
    fin = np.isfinite(v) & (np.abs(v) <= 448)
    vals = v[fin][::7]  # a spread subset keeps the test quick
    ours = np.array([oracle.e4m3_from_f32(x) for x in vals], np.uint8)
    ref = torch.from_numpy(vals.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    codes = np.arange(256, dtype=np.uint8)
    dec = np.array([oracle.e4m3_to_f32(int(c)) for c in codes], np.float32)
    tdec = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    same = (dec == tdec) | (np.isnan(dec) & np.isnan(tdec))
    assert same.all()
    for x, b in [(448.0, 0x7E), (449.0, 0x7E), (1e30, 0x7E), (-600.0, 0xFE), (2.0 ** -10, 0x00),
                 (3 * 2.0 ** -10, 0x02), (2.0 ** -6, 0x08)]:
        assert oracle.e4m3_from_f32(x) == b, x


def test_mx_quant_closed_forms_and_bounds():
    rng = np.random.default_rng(41)
    M, K = 6, 128
    x = (rng.standard_normal((M, K)) * 2.0 ** rng.integers(-20, 20, (M, 1))).astype(np.float32)
    x[0, :32] = 1.0                  # all ones: shared exponent 0 - 8, codes 256 = 2^8
    x[1, 32:64] = 0.0                # zeros: scale byte 0, codes 0
    x[2, 64:96] = 0.0
    x[2, 70] = -3.0                  # one value: 3 = 1.5 * 2^1 -> shared -7, element 384
    xb = S.to_bf16_bits(x)
    q, s = oracle.mx_quant(xb)
    assert s[0, 0] == 127 - 8 and np.all(q[0, :32] == 0x78)
    assert s[1, 1] == 0 and np.all(q[1, 32:64] == 0)
    assert s[2, 2] == 127 - 7 and q[2, 70] == oracle.e4m3_from_f32(-384.0)
    # shared = floor(log2 amax) - 8 for every group
    xf = f32(xb).astype(np.float64).reshape(M, K // 32, 32)
    amax = np.abs(xf).max(axis=2)
    live = amax > 0
    want = np.floor(np.log2(amax[live])) - 8 + 127
    assert np.array_equal(s[live].astype(np.float64), want)
    # reconstruction: within half a step of the 3-bit mantissa, or the saturation at 448 for the top values
    dec = np.vectorize(oracle.e4m3_to_f32)(q).astype(np.float64).reshape(M, K // 32, 32)
    scale = 2.0 ** (s.astype(np.float64) - 127)[..., None]
    rec = dec * scale
    y = xf / scale
    step = np.where(np.abs(y) >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6))) - 3), 2.0 ** -9)
    ok = np.abs(rec - xf) <= 0.5 * step * scale + 1e-300
    sat = np.abs(y) > 448
    assert np.all(ok | sat)
    assert np.all(np.abs(dec[sat]) == 448)


def test_mx_matmul_against_float64():
    rng = np.random.default_rng(42)
    M, N, K = 9, 13, 96
    xa = S.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    xw = S.to_bf16_bits((rng.standard_normal((N, K)) * 0.05).astype(np.float32))
    qa, sa = oracle.mx_quant(xa)
    qw, sw = oracle.mx_quant(xw)
    y = f32(oracle.mx_matmul(qa, sa, qw, sw)).astype(np.float64)
    dec = np.vectorize(oracle.e4m3_to_f32)
    A = dec(qa).astype(np.float64) * np.repeat(2.0 ** (sa.astype(np.float64) - 127), 32, axis=1)
    B = dec(qw).astype(np.float64) * np.repeat(2.0 ** (sw.astype(np.float64) - 127), 32, axis=1)
    ref = A @ B.T
    assert np.all(np.abs(y - ref) <= bf16_ulp(ref) * 0.5 * 1.001 + 1e-30)
    # and the MX product approximates the BF16 product within the E4M3 rounding of both operands
    full = f32(xa).astype(np.float64) @ f32(xw).astype(np.float64).T
    mag = np.abs(f32(xa)).astype(np.float64) @ np.abs(f32(xw)).astype(np.float64).T
    assert np.all(np.abs(y - full) <= 2 * 2.0 ** -4 * mag + bf16_ulp(full))
