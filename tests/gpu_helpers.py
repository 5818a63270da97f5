"""Helpers shared by the GPU parity tests: moving seeded host inputs to the
device, and oracle evaluations on row subsets of full-size problems."""
import numpy as np
import torch

import oracle


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def f32_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def bf16_ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """|difference| in units of bf16 representable steps (same-sign ordering)."""
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    return np.abs(key(a_bits) - key(b_bits))


def sample_rows(n_rows: int, k: int, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = rng.choice(n_rows, size=min(k, n_rows), replace=False)
    return np.unique(np.concatenate([pick, [0, n_rows - 1]]))


def moe_subset_oracle(m, rows: np.ndarray):
    """Oracle MoE output for the routed rows `rows` only (each row's chain is
    independent of the other rows), built as a compact problem over the
    experts those rows belong to."""
    rows = np.sort(rows)
    off = np.concatenate([[0], np.cumsum(m.group_list)])
    exp_of_row = np.searchsorted(off, rows, side="right") - 1
    experts = np.unique(exp_of_row)
    gl = np.array([int(np.sum(exp_of_row == e)) for e in experts], np.int64)
    idx = torch.as_tensor(experts, device=m.w13.device)
    w13 = m.w13.index_select(0, idx).cpu().numpy()
    w2 = m.w2.index_select(0, idx).cpu().numpy()
    xs = None if m.x_scale is None else m.x_scale[rows]
    return oracle.moe_w13_swiglu_requant_w2(m.x[rows], xs, gl, w13, m.s13[experts], w2, m.s2[experts],
                                            intermediates=True)
