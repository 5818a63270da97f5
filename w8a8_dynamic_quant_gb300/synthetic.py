"""Seeded synthetic inputs for the W8A8_DYNAMIC linear and MoE-expert path.

This module only draws random inputs; it holds none of the method's
arithmetic, so the oracle and the CUDA path can both consume its output.

Recipe (one generator per case, seed 0 unless stated; draw order fixed):
  dense  X ~ N(0,1) fp32 [M,K] -> a fixed set of outlier columns (chosen
         without replacement) multiplied by a factor -> rounded to BF16;
         W uniform integers in [-127,127] [N,K]; w_scale U[1e-3,1e-2] [N];
         bias ~ N(0, 0.1) rounded to BF16 [N] when the case has one.
  moe    X ~ N(0,1) BF16 [T,H]; routing: every token picks top-k DISTINCT
         experts by Gumbel-top-k over expert probabilities p_e (Zipf: p of
         popularity rank r proportional to (r+1)^-s, ranks mapped to experts
         by a seeded permutation, the lowest-popularity `n_dead` ranks get
         p = 0 so some experts receive no rows; uniform: equal p);
         routed rows are token copies sorted by expert (token order inside an
         expert), group_list = rows per expert; w13/w2 uniform integers in
         [-127,127] drawn with torch's seeded generator on the target device
         (the weights of the big cases are GBs); scales U[1e-3,1e-2].
         Pre-quantised cases draw an INT8 payload uniform in [-127,127] and a
         per-token fp32 scale U[1e-3,5e-2] per TOKEN, and routed rows carry
         their token's payload and scale.  Token rows are kept too, with
         router weights drawn last: U[0.05,1] per chosen expert, divided by
         the token's sum, fp32.
  bf16 weights (the source of the offline per-channel quantisation):
         N(0,1) * 0.02 * 2^c per output channel, c uniform in {-4..2}, and one
         element in every 64th channel multiplied by 8 (an outlier); drawn on
         the target device with torch's seeded generator, rounded to BF16.
  static W8A8: per-tensor input scale U[0.02, 0.04] (binary32) and input
         offset uniform in {-8..8}, stand-ins for calibrated values, drawn
         per workload from their own generator.
BF16 rounding of the drawn fp32 values uses torch's conversion.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

# The five workloads.  Sizes, distributions and outlier recipes as stated per case.
CONFIGS = {
    1: dict(kind="dense", name="dense_tiny_M16_N256_K512", M=16, K=512, N=256,
            n_outlier=2, outlier_mult=20.0, bias=True),
    2: dict(kind="dense", name="dense_decode_M64_N2048_K7168", M=64, K=7168, N=2048,
            n_outlier=72, outlier_mult=30.0, bias=False),
    3: dict(kind="dense", name="dense_prefill_M8192_N14336_K4096", M=8192, K=4096, N=14336,
            n_outlier=20, outlier_mult=20.0, bias=False),
    4: dict(kind="moe", name="moe_prefill_T4096_H4096_I2048_E64_top8_zipf1.1", T=4096, H=4096,
            I=2048, E=64, topk=8, routing="zipf", zipf_s=1.1, n_dead=4, prequant=False),
    5: dict(kind="moe", name="moe_decode_T128_H7168_I2048_E256_top8_prequant", T=128, H=7168,
            I=2048, E=256, topk=8, routing="uniform", prequant=True),
}


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 array -> BF16 bit patterns (uint16), via torch's RNE conversion."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> fp32 values (exact widening)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class DenseInputs:
    name: str
    x: np.ndarray            # uint16 BF16 bits [M,K]
    w: np.ndarray            # int8 [N,K]
    w_scale: np.ndarray      # fp32 [N]
    bias: Optional[np.ndarray]  # uint16 BF16 bits [N] or None
    outlier_cols: np.ndarray

    @property
    def M(self):
        return self.x.shape[0]

    @property
    def K(self):
        return self.x.shape[1]

    @property
    def N(self):
        return self.w.shape[0]


def make_dense(M: int, K: int, N: int, n_outlier: int = 0, outlier_mult: float = 1.0,
               bias: bool = False, seed: int = 0, name: str = "dense") -> DenseInputs:
    rng = rng_for(seed)
    x = rng.standard_normal((M, K), dtype=np.float32)
    cols = np.sort(rng.choice(K, size=n_outlier, replace=False)) if n_outlier else np.zeros(0, np.int64)
    if n_outlier:
        x[:, cols] *= np.float32(outlier_mult)
    w = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    w_scale = rng.uniform(1e-3, 1e-2, size=N).astype(np.float32)
    b = None
    if bias:
        b = to_bf16_bits(rng.standard_normal(N, dtype=np.float32) * np.float32(0.1))
    return DenseInputs(name=name, x=to_bf16_bits(x), w=w, w_scale=w_scale, bias=b, outlier_cols=cols)


def dense_config(cfg_id: int, seed: int = 0) -> DenseInputs:
    c = CONFIGS[cfg_id]
    assert c["kind"] == "dense"
    return make_dense(c["M"], c["K"], c["N"], c["n_outlier"], c["outlier_mult"], c["bias"], seed,
                      name=c["name"])


@dataclass
class MoEInputs:
    name: str
    T: int
    H: int
    I: int
    E: int
    topk: int
    topk_ids: np.ndarray       # int64 [T, topk] chosen experts per token
    token_index: np.ndarray    # int64 [R] source token of each routed row
    group_list: np.ndarray     # int64 [E] rows per expert
    x: np.ndarray              # routed rows: uint16 BF16 [R,H] or int8 [R,H] (prequant)
    x_scale: Optional[np.ndarray]  # fp32 [R] when pre-quantised, else None
    w13: torch.Tensor          # int8 [E,2I,H] (on `device`)
    s13: np.ndarray            # fp32 [E,2I]
    w2: torch.Tensor           # int8 [E,H,I]
    s2: np.ndarray             # fp32 [E,H]
    extra: dict = field(default_factory=dict)
    x_tok: Optional[np.ndarray] = None        # token rows: uint16 BF16 [T,H] or int8 [T,H] (prequant)
    x_tok_scale: Optional[np.ndarray] = None  # fp32 [T] when pre-quantised, else None
    topk_weights: Optional[np.ndarray] = None  # fp32 [T, topk] router weights, each row sums to ~1

    @property
    def R(self):
        return int(self.token_index.shape[0])


def route(rng: np.random.Generator, T: int, E: int, topk: int, routing: str,
          zipf_s: float = 1.1, n_dead: int = 0):
    """Top-k distinct experts per token by Gumbel-top-k; returns (topk_ids [T,k], p [E])."""
    if routing == "zipf":
        perm = rng.permutation(E)
        live = E - n_dead
        p = np.zeros(E, np.float64)
        p[perm[:live]] = (np.arange(live, dtype=np.float64) + 1.0) ** (-zipf_s)
        p /= p.sum()
    elif routing == "uniform":
        p = np.full(E, 1.0 / E)
    else:
        raise ValueError(routing)
    with np.errstate(divide="ignore"):
        logp = np.log(p)
    keys = logp[None, :] + rng.gumbel(size=(T, E))
    topk_ids = np.argsort(-keys, axis=1, kind="stable")[:, :topk].astype(np.int64)
    return topk_ids, p


def expert_sorted_rows(topk_ids: np.ndarray, E: int):
    """Routed row order: expert-major, token order inside an expert."""
    T, k = topk_ids.shape
    rows = []
    counts = np.zeros(E, np.int64)
    for e in range(E):
        toks = np.nonzero((topk_ids == e).any(axis=1))[0]
        rows.append(toks)
        counts[e] = toks.shape[0]
    token_index = np.concatenate(rows).astype(np.int64) if rows else np.zeros(0, np.int64)
    return token_index, counts


def make_moe(T: int, H: int, I: int, E: int, topk: int, routing: str = "uniform",
             zipf_s: float = 1.1, n_dead: int = 0, prequant: bool = False, seed: int = 0,
             device: str = "cpu", name: str = "moe") -> MoEInputs:
    rng = rng_for(seed)
    x_tok = None
    if not prequant:
        x_tok = to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1000003 + 17)
    w13 = torch.randint(-127, 128, (E, 2 * I, H), dtype=torch.int8, device=device, generator=gen)
    s13 = rng.uniform(1e-3, 1e-2, size=(E, 2 * I)).astype(np.float32)
    w2 = torch.randint(-127, 128, (E, H, I), dtype=torch.int8, device=device, generator=gen)
    s2 = rng.uniform(1e-3, 1e-2, size=(E, H)).astype(np.float32)
    topk_ids, p = route(rng, T, E, topk, routing, zipf_s, n_dead)
    token_index, counts = expert_sorted_rows(topk_ids, E)
    s_tok = None
    if prequant:
        x_tok = rng.integers(-127, 128, size=(T, H), dtype=np.int8)
        s_tok = rng.uniform(1e-3, 5e-2, size=T).astype(np.float32)
        x = x_tok[token_index]
        x_scale = s_tok[token_index]
    else:
        x = x_tok[token_index]
        x_scale = None
    # router weights of the chosen experts: positive, normalised per token
    u = rng.uniform(0.05, 1.0, size=(T, topk))
    topk_weights = (u / u.sum(axis=1, keepdims=True)).astype(np.float32)
    return MoEInputs(name=name, T=T, H=H, I=I, E=E, topk=topk, topk_ids=topk_ids,
                     token_index=token_index, group_list=counts, x=np.ascontiguousarray(x),
                     x_scale=x_scale, w13=w13, s13=s13, w2=w2, s2=s2, extra=dict(p=p),
                     x_tok=x_tok, x_tok_scale=s_tok, topk_weights=topk_weights)


def static_params(cfg_id: int, seed: int = 0):
    """(input_scale, input_offset) of the static variant for a workload."""
    rng = rng_for(seed * 31 + cfg_id + 1000)
    return float(np.float32(rng.uniform(0.02, 0.04))), int(rng.integers(-8, 9))


def make_bf16_weight(E: int, N: int, K: int, seed: int = 0, device: str = "cpu") -> torch.Tensor:
    """A BF16 weight stack [E,N,K] with per-channel ranges spread over 2^-4 .. 2^2 (and some outliers)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 7919 + 3)
    w = torch.randn((E, N, K), generator=gen, device=device)
    c = torch.randint(-4, 3, (E, N, 1), generator=gen, device=device).float()
    w.mul_(torch.exp2(c) * 0.02)
    rows = torch.arange(0, N, 64, device=device)  # every 64th channel gets one outlier
    col = torch.randint(0, K, (E, rows.numel()), generator=gen, device=device)
    e_idx = torch.arange(E, device=device)[:, None].expand_as(col)
    w[e_idx, rows[None, :].expand_as(col), col] *= 8.0
    return w.to(torch.bfloat16)


def moe_config(cfg_id: int, seed: int = 0, device: str = "cpu") -> MoEInputs:
    c = CONFIGS[cfg_id]
    assert c["kind"] == "moe"
    return make_moe(c["T"], c["H"], c["I"], c["E"], c["topk"], c["routing"], c.get("zipf_s", 1.1),
                    c.get("n_dead", 0), c["prequant"], seed, device, name=c["name"])
