"""GPU parity of the MoE routing around the expert chain (through the C ABI):
the permute + quantisation of token rows into expert-grouped routed rows, the
top-k weighted combine, and the whole layer from token rows.  Group lists,
routed row indices, INT8 codes and FP32 scales are compared bit-exactly with
the oracle, and so are the BF16 outputs (both sides take the same binary32
steps).  Full-size layers are checked on sampled tokens: a token's output
depends on its own row and its experts only."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_dynamic_quant_gb300 as W
from w8a8_dynamic_quant_gb300 import synthetic as S

from gpu_helpers import dev, dev_bf16, f32_bits, host_bits, sample_rows

pytestmark = pytest.mark.gpu


def ids_for(T, k, E, seed, distinct=True):
    rng = np.random.default_rng(seed)
    if distinct and k <= E:
        keys = rng.random((T, E))
        return np.argsort(keys, axis=1)[:, :k].astype(np.int64)
    return rng.integers(0, E, size=(T, k), dtype=np.int64)


def tokens(T, H, seed, prequant):
    rng = np.random.default_rng(seed)
    if prequant:
        return (rng.integers(-127, 128, (T, H), dtype=np.int8),
                rng.uniform(1e-3, 5e-2, T).astype(np.float32))
    x = rng.standard_normal((T, H)).astype(np.float32)
    x[:, rng.choice(H, size=max(1, H // 100), replace=False)] *= np.float32(25.0)
    if T > 3:
        x[3] = 0.0  # an all-zero token: scale 0, codes 0
    return S.to_bf16_bits(x), None


def gpu_permute(x, xs, ids, E):
    xd = dev(x) if xs is not None else dev_bf16(x)
    out = W.moe_permute_quant(xd, None if xs is None else dev(xs), dev(ids), E)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in out]


@pytest.mark.parametrize("T,k,E,H,distinct", [(1, 1, 1, 16, True), (7, 2, 3, 64, True),
                                              (300, 8, 64, 512, True), (1000, 3, 5, 96, False),
                                              (171, 4, 1024, 272, True), (2500, 1, 7, 128, True),
                                              (33, 6, 6, 4096, True),
                                              # past the one-CTA sort: more than 65536 pairs, or 1024 experts
                                              # with 40000 pairs (its shared memory would pass 200 KB)
                                              (20000, 4, 64, 64, True), (10000, 4, 1024, 16, True)])
@pytest.mark.parametrize("prequant", [False, True])
def test_permute_quant_exact(T, k, E, H, distinct, prequant):
    ids = ids_for(T, k, E, seed=T * 7 + E, distinct=distinct)
    x, xs = tokens(T, H, seed=T + H, prequant=prequant)
    xq, xsr, gl, pos = gpu_permute(x, xs, ids, E)
    xq_ref, xs_ref, gl_ref, pos_ref = oracle.moe_permute_quant(x, xs, ids, E)
    assert np.array_equal(gl, gl_ref)
    assert np.array_equal(pos, pos_ref)
    assert np.array_equal(f32_bits(xsr), f32_bits(xs_ref))
    assert np.array_equal(xq, xq_ref)


def test_permute_quant_no_tokens():
    gl = torch.full((5,), 7, dtype=torch.int64, device="cuda")
    ws = W.workspace(W.moe_route_workspace_bytes(0, 4, 5))
    rc = W._capi.lib().moe_permute_quant(None, None, None, 0, 4, 5, 64, None, None, gl.data_ptr(), None,
                                         ws.data_ptr(), ws.numel(), None)
    assert rc == 0
    torch.cuda.synchronize()
    assert gl.cpu().tolist() == [0] * 5


@pytest.mark.parametrize("T", [600, 40000])
def test_permute_quant_bad_id_is_reported(T):
    k, E, H = 2, 8, 64
    ids = ids_for(T, k, E, seed=3)
    ids[555, 1] = E       # past the last expert
    ids[20, 0] = -4       # negative
    x, _ = tokens(T, H, seed=4, prequant=False)
    ws = W.workspace(W.moe_route_workspace_bytes(T, k, E))
    xq, xs, gl, pos = W.moe_permute_quant(dev_bf16(x), None, dev(ids), E, ws=ws)
    assert W.read_device_status(ws) == 10
    assert W.read_device_status(ws) == 0  # read clears it
    pos = pos.cpu().numpy()
    assert pos[555, 1] == -1 and pos[20, 0] == -1
    assert int(gl.sum()) == T * k - 2
    # the good pairs keep their rank: the oracle on the same ids with the bad pairs removed
    good = np.ones((T, k), bool)
    good[555, 1] = good[20, 0] = False
    assert np.array_equal(np.sort(pos[good]), np.arange(T * k - 2))


@pytest.mark.parametrize("T,k,H", [(1, 1, 8), (5, 9, 1040), (300, 8, 4096), (129, 3, 2056), (64, 8, 7168),
                                   (2, 17, 24), (3000, 2, 1024)])
def test_combine_exact(T, k, H):
    rng = np.random.default_rng(T + k + H)
    ids = ids_for(T, k, max(k, 11), seed=T)
    _, pos = oracle.moe_route(ids, max(k, 11))
    yr = S.to_bf16_bits(rng.standard_normal((T * k, H)).astype(np.float32) * np.float32(4))
    w = rng.uniform(-0.2, 1.0, (T, k)).astype(np.float32)
    y = W.moe_unpermute_combine(dev_bf16(yr), dev(pos), dev(w))
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(y), oracle.moe_unpermute_combine(yr, pos, w))


def test_combine_summation_order():
    """Terms 1+2^-8 then four of 2^-25: in slot order in binary32 the small terms are lost and the bf16
    rounding of the tie gives 1.0 (0x3F80); any other order or a wider sum gives 0x3F81."""
    one = S.to_bf16_bits(np.ones((5, 8), np.float32))
    w = np.array([[1 + 2.0 ** -8] + [2.0 ** -25] * 4], np.float32)
    pos = np.arange(5, dtype=np.int32).reshape(1, 5)
    y = host_bits(W.moe_unpermute_combine(dev_bf16(one), dev(pos), dev(w)))
    assert np.all(y == 0x3F80)
    y2 = host_bits(W.moe_unpermute_combine(dev_bf16(one), dev(pos[:, ::-1].copy()), dev(w[:, ::-1].copy())))
    assert np.all(y2 == 0x3F81)


def test_combine_bad_pos_is_reported():
    T, k, H = 40, 2, 64
    rng = np.random.default_rng(8)
    _, pos = oracle.moe_route(ids_for(T, k, 4, seed=9), 4)
    yr = S.to_bf16_bits(rng.standard_normal((T * k, H)).astype(np.float32))
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    bad = pos.copy()
    bad[7, 1] = T * k      # one past the routed rows
    bad[9, 0] = -1
    ws = W.workspace(256)
    y = host_bits(W.moe_unpermute_combine(dev_bf16(yr), dev(bad), dev(w), ws=ws))
    assert W.read_device_status(ws) == 10
    # the other tokens are unaffected; a bad term is left out of its token's sum
    ref = oracle.moe_unpermute_combine(yr, pos, w)
    keep = np.ones(T, bool)
    keep[[7, 9]] = False
    assert np.array_equal(y[keep], ref[keep])
    w7 = w.copy()
    w7[7, 1] = 0.0
    only0 = oracle.moe_unpermute_combine(yr, pos, w7)
    assert np.array_equal(y[7], only0[7])


def layer_case(T, H, I, E, k, prequant, seed, f16_copy):
    m = S.make_moe(T=T, H=H, I=I, E=E, topk=k, routing="zipf", zipf_s=1.1, n_dead=1, prequant=prequant,
                   seed=seed)
    extra = W.PACK_F16 if f16_copy else 0
    w13p = W.w8a8_prepack_weight(m.w13.cuda(), W.PACK_GATE_UP | extra)
    w2p = W.w8a8_prepack_weight(m.w2.cuda(), extra)
    x = dev(m.x_tok) if prequant else dev_bf16(m.x_tok)
    xs = None if m.x_tok_scale is None else dev(m.x_tok_scale)
    ws = W.workspace(W.moe_layer_workspace_bytes(T, k, H, I, E))
    y = W.moe_layer(x, xs, dev(m.topk_ids), dev(m.topk_weights), w13p, dev(m.s13), w2p, dev(m.s2), ws=ws)
    torch.cuda.synchronize()
    return m, host_bits(y), ws


@pytest.mark.parametrize("T,H,I,E,k", [(40, 96, 64, 6, 2), (512, 256, 128, 4, 2), (300, 512, 192, 8, 3)])
@pytest.mark.parametrize("prequant", [False, True])
@pytest.mark.parametrize("f16_copy", [True, False])
def test_moe_layer_exact(T, H, I, E, k, prequant, f16_copy):
    m, y, ws = layer_case(T, H, I, E, k, prequant, seed=T + E, f16_copy=f16_copy)
    y_ref, yr_ref = oracle.moe_layer(m.x_tok, m.x_tok_scale, m.topk_ids, m.topk_weights, m.w13.numpy(), m.s13,
                                     m.w2.numpy(), m.s2, want_routed=True)
    off = W.moe_layer_workspace_offset(T, k, H, I, E, 9)
    yr = ws[off:off + T * k * H * 2].cpu().numpy().view(np.uint16).reshape(T * k, H)
    assert np.array_equal(yr, yr_ref)
    assert np.array_equal(y, y_ref)
    if T * k >= 64 * E:  # shapes the tensor-core engines take: the routed codes are kept as fp16
        assert W.last_engine() == (W.ENGINE_TC if f16_copy else W.ENGINE_TC_I8)
        o16 = W.moe_layer_workspace_offset(T, k, H, I, E, 5)
        xq16 = ws[o16:o16 + T * k * H * 2].view(torch.float16).cpu().numpy().reshape(T * k, H)
        xq_ref, _, _, _ = oracle.moe_permute_quant(m.x_tok, m.x_tok_scale, m.topk_ids, E)
        assert np.array_equal(xq16, xq_ref.astype(np.float16))


def layer_subset_oracle(m, toks):
    """Oracle layer output for tokens `toks` only, over the experts they chose (renumbered)."""
    ids = m.topk_ids[toks]
    experts = np.unique(ids)
    remap = np.searchsorted(experts, ids).astype(np.int64)
    idx = torch.as_tensor(experts, device=m.w13.device)
    w13 = m.w13.index_select(0, idx).cpu().numpy()
    w2 = m.w2.index_select(0, idx).cpu().numpy()
    xs = None if m.x_tok_scale is None else m.x_tok_scale[toks]
    return oracle.moe_layer(m.x_tok[toks], xs, remap, m.topk_weights[toks], w13, m.s13[experts], w2,
                            m.s2[experts])


@pytest.mark.parametrize("cfg", [4, 5])
def test_moe_layer_full_config_sampled_tokens(cfg):
    m = S.moe_config(cfg, device="cuda")
    w13p = W.w8a8_prepack_weight(m.w13, W.PACK_GATE_UP | W.PACK_F16)
    w2p = W.w8a8_prepack_weight(m.w2, W.PACK_F16)
    x = dev(m.x_tok) if m.x_tok_scale is not None else dev_bf16(m.x_tok)
    xs = None if m.x_tok_scale is None else dev(m.x_tok_scale)
    ids = dev(m.topk_ids)
    ws = W.workspace(W.moe_layer_workspace_bytes(m.T, m.topk, m.H, m.I, m.E))
    y = W.moe_layer(x, xs, ids, dev(m.topk_weights), w13p, dev(m.s13), w2p, dev(m.s2), ws=ws)
    torch.cuda.synchronize()
    assert W.read_device_status(ws) == 0
    # routing metadata in full
    gl_off = W.moe_layer_workspace_offset(m.T, m.topk, m.H, m.I, m.E, 7)
    gl = ws[gl_off:gl_off + m.E * 8].cpu().numpy().view(np.int64)
    assert np.array_equal(gl, m.group_list)
    toks = sample_rows(m.T, 12, seed=cfg)
    y_ref = layer_subset_oracle(m, toks)
    assert np.array_equal(host_bits(y)[toks], y_ref)
