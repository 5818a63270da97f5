"""GB300 (sm_103a) W8A8_DYNAMIC linear layer and MoE-expert path.

A thin torch binding over the C ABI of libw8a8.so (include/w8a8.h): every
function below only checks tensor shapes/dtypes/devices, takes data pointers
and the current CUDA stream, and calls the library.  All arithmetic runs in
the library's CUDA kernels; nothing here computes, and there is no fallback.

BF16 tensors are torch.bfloat16; INT8 tensors torch.int8; scales float32;
group lists int64 (on the device).  Workspaces are zero-filled uint8 device
tensors that can be reused across calls on one stream.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _capi
from ._capi import PACK_F16, PACK_GATE_UP, W8A8Error

__all__ = [
    "PACK_F16", "PACK_GATE_UP", "W8A8Error", "prepacked_bytes", "w8a8_prepack_weight",
    "w8a8_dynamic_quant", "quant_matmul_workspace_bytes", "w8a8_quant_matmul",
    "w8a8_int8_matmul_acc", "grouped_matmul_workspace_bytes", "w8a8_grouped_matmul",
    "w8a8_grouped_matmul_acc", "moe_workspace_bytes", "moe_workspace_offset",
    "moe_w13_swiglu_requant_w2", "read_device_status", "workspace", "w8a8_quant_matmul_noalloc",
    "last_engine", "ENGINE_NONE", "ENGINE_WARP", "ENGINE_DECODE", "ENGINE_TC", "ENGINE_TC_I8",
    "w8a8_quantize_weight", "w8a8_quantize_prepack_weight", "w8a8_static_quant", "w8a8_static_prepare",
    "w8a8_static_quant_matmul", "w8a8_mx_quant", "w8a8_mx_matmul", "moe_route_workspace_bytes", "moe_permute_quant", "moe_unpermute_combine", "moe_layer_workspace_bytes",
    "moe_layer_workspace_offset", "moe_layer",
]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(device: torch.device):
    return torch.cuda.current_stream(device).cuda_stream


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zero-filled device workspace of `nbytes` bytes (256-byte aligned by the caching allocator)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def prepacked_bytes(E: int, N: int, K: int, flags: int = 0) -> int:
    return int(_capi.lib().w8a8_prepacked_bytes(E, N, K, flags))


def w8a8_prepack_weight(w: torch.Tensor, flags: int = 0) -> torch.Tensor:
    """INT8 weight [N,K] or expert stack [E,N,K] -> packed device buffer (uint8)."""
    w3 = w.unsqueeze(0) if w.dim() == 2 else w
    if w3.dim() != 3:
        raise ValueError("w must be [N,K] or [E,N,K]")
    _need(w3, "w", torch.int8)
    E, N, K = w3.shape
    nbytes = prepacked_bytes(E, N, K, flags)
    if nbytes == 0:
        raise ValueError("bad weight shape")
    packed = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    with torch.cuda.device(w.device):
        _capi.check("w8a8_prepack_weight", _capi.lib().w8a8_prepack_weight(
            w3.data_ptr(), E, N, K, flags, packed.data_ptr(), _stream(w.device)))
    return packed


def _weight3(w: torch.Tensor):
    w3 = w.unsqueeze(0) if w.dim() == 2 else w
    if w3.dim() != 3:
        raise ValueError("w must be [N,K] or [E,N,K]")
    _need(w3, "w", torch.bfloat16)
    return w3


def w8a8_quantize_weight(w: torch.Tensor):
    """BF16 weight [N,K] or [E,N,K] -> (int8 q of the same shape, float32 per-channel scales [N] / [E,N])."""
    w3 = _weight3(w)
    E, N, K = w3.shape
    q = torch.empty((E, N, K), dtype=torch.int8, device=w.device)
    scale = torch.empty((E, N), dtype=torch.float32, device=w.device)
    with torch.cuda.device(w.device):
        _capi.check("w8a8_quantize_weight", _capi.lib().w8a8_quantize_weight(
            w3.data_ptr(), E, N, K, q.data_ptr(), scale.data_ptr(), _stream(w.device)))
    return (q[0], scale[0]) if w.dim() == 2 else (q, scale)


def w8a8_quantize_prepack_weight(w: torch.Tensor, flags: int = 0, packed: Optional[torch.Tensor] = None,
                                 scale: Optional[torch.Tensor] = None):
    """BF16 weight [N,K] or [E,N,K] -> (packed device buffer, float32 per-channel scales [N] / [E,N]),
    quantised per channel and packed in one pass."""
    w3 = _weight3(w)
    E, N, K = w3.shape
    nbytes = prepacked_bytes(E, N, K, flags)
    if nbytes == 0:
        raise ValueError("bad weight shape")
    packed = torch.empty(nbytes, dtype=torch.uint8, device=w.device) if packed is None else packed
    _need(packed, "packed", torch.uint8, (nbytes,), w.device)
    scale = torch.empty((E, N), dtype=torch.float32, device=w.device) if scale is None else scale.view(E, N)
    _need(scale, "scale", torch.float32, (E, N), w.device)
    with torch.cuda.device(w.device):
        _capi.check("w8a8_quantize_prepack_weight", _capi.lib().w8a8_quantize_prepack_weight(
            w3.data_ptr(), E, N, K, flags, packed.data_ptr(), scale.data_ptr(), _stream(w.device)))
    return packed, (scale[0] if w.dim() == 2 else scale)


def w8a8_dynamic_quant(x: torch.Tensor, q: Optional[torch.Tensor] = None,
                       scale: Optional[torch.Tensor] = None):
    """BF16 x [M,K] -> (int8 q [M,K], float32 scale [M])."""
    _need(x, "x", torch.bfloat16)
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.int8, device=x.device) if q is None else q
    scale = torch.empty((M,), dtype=torch.float32, device=x.device) if scale is None else scale
    _need(q, "q", torch.int8, (M, K), x.device)
    _need(scale, "scale", torch.float32, (M,), x.device)
    with torch.cuda.device(x.device):
        _capi.check("w8a8_dynamic_quant", _capi.lib().w8a8_dynamic_quant(
            x.data_ptr(), M, K, q.data_ptr(), scale.data_ptr(), _stream(x.device)))
    return q, scale


def w8a8_mx_quant(x: torch.Tensor, q: Optional[torch.Tensor] = None, scale: Optional[torch.Tensor] = None):
    """MXFP8: bf16 x [M,K] (K % 32 == 0) -> (uint8 E4M3 codes [M,K], uint8 E8M0 scales [M,K/32])."""
    _need(x, "x", torch.bfloat16)
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device) if q is None else q
    scale = torch.empty((M, K // 32), dtype=torch.uint8, device=x.device) if scale is None else scale
    _need(q, "q", torch.uint8, (M, K), x.device)
    _need(scale, "scale", torch.uint8, (M, K // 32), x.device)
    with torch.cuda.device(x.device):
        _capi.check("w8a8_mx_quant", _capi.lib().w8a8_mx_quant(
            x.data_ptr(), M, K, q.data_ptr(), scale.data_ptr(), _stream(x.device)))
    return q, scale


def w8a8_mx_matmul(qa: torch.Tensor, sa: torch.Tensor, qw: torch.Tensor, sw: torch.Tensor,
                   y: Optional[torch.Tensor] = None):
    """MXFP8 contraction: E4M3 qa [M,K] + E8M0 sa [M,K/32], E4M3 qw [N,K] + E8M0 sw [N,K/32] -> bf16 y [M,N]."""
    _need(qa, "qa", torch.uint8)
    M, K = qa.shape
    dev = qa.device
    _need(sa, "sa", torch.uint8, (M, K // 32), dev)
    _need(qw, "qw", torch.uint8, None, dev)
    N = qw.shape[0]
    _need(sw, "sw", torch.uint8, (N, K // 32), dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev) if y is None else y
    _need(y, "y", torch.bfloat16, (M, N), dev)
    with torch.cuda.device(dev):
        _capi.check("w8a8_mx_matmul", _capi.lib().w8a8_mx_matmul(
            qa.data_ptr(), sa.data_ptr(), M, K, qw.data_ptr(), sw.data_ptr(), N, y.data_ptr(), _stream(dev)))
    return y


def w8a8_static_quant(x: torch.Tensor, input_scale: float, input_offset: int, q: Optional[torch.Tensor] = None):
    """Static W8A8 quantisation: bf16 x [M,K] -> int8 q = clamp(rint(x / s) + o, -128, 127)."""
    _need(x, "x", torch.bfloat16)
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.int8, device=x.device) if q is None else q
    _need(q, "q", torch.int8, (M, K), x.device)
    with torch.cuda.device(x.device):
        _capi.check("w8a8_static_quant", _capi.lib().w8a8_static_quant(
            x.data_ptr(), M, K, float(input_scale), int(input_offset), q.data_ptr(), _stream(x.device)))
    return q


def w8a8_static_prepare(w: torch.Tensor, weight_scale: torch.Tensor, input_scale: float, input_offset: int,
                        bias: Optional[torch.Tensor] = None):
    """Load time: int8 W [N,K], float32 weight scales [N] (+ bf16 bias [N]) -> (float32 deq_scale [N],
    int32 quant_bias [N])."""
    _need(w, "w", torch.int8)
    N, K = w.shape
    dev = w.device
    _need(weight_scale, "weight_scale", torch.float32, (N,), dev)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, (N,), dev)
    deq = torch.empty((N,), dtype=torch.float32, device=dev)
    qb = torch.empty((N,), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _capi.check("w8a8_static_prepare", _capi.lib().w8a8_static_prepare(
            w.data_ptr(), N, K, weight_scale.data_ptr(), float(input_scale), int(input_offset), _ptr(bias),
            deq.data_ptr(), qb.data_ptr(), _stream(dev)))
    return deq, qb


def w8a8_static_quant_matmul(q: torch.Tensor, w_packed: torch.Tensor, deq_scale: torch.Tensor,
                             quant_bias: torch.Tensor, ws: Optional[torch.Tensor] = None,
                             y: Optional[torch.Tensor] = None):
    """Static W8A8 matmul: int8 q [M,K] x packed W [N,K] -> bf16 y = bf16(float(acc + quant_bias) * deq_scale)."""
    _need(q, "q", torch.int8)
    M, K = q.shape
    dev = q.device
    _need(deq_scale, "deq_scale", torch.float32, None, dev)
    N = deq_scale.shape[0]
    _need(quant_bias, "quant_bias", torch.int32, (N,), dev)
    _need(w_packed, "w_packed", torch.uint8, None, dev)
    ws = workspace(quant_matmul_workspace_bytes(M, N, K), dev) if ws is None else ws
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev) if y is None else y
    _need(y, "y", torch.bfloat16, (M, N), dev)
    with torch.cuda.device(dev):
        _capi.check("w8a8_static_quant_matmul", _capi.lib().w8a8_static_quant_matmul(
            q.data_ptr(), M, K, w_packed.data_ptr(), deq_scale.data_ptr(), quant_bias.data_ptr(), N, y.data_ptr(),
            ws.data_ptr(), ws.numel(), _stream(dev)))
    return y


def quant_matmul_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(_capi.lib().w8a8_quant_matmul_workspace_bytes(M, N, K))


def w8a8_quant_matmul(q: torch.Tensor, x_scale: torch.Tensor, w_packed: torch.Tensor,
                      w_scale: torch.Tensor, N: int, bias: Optional[torch.Tensor] = None,
                      ws: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None):
    """int8 q [M,K] x packed W [N,K] -> bf16 y [M,N] = ((acc * x_scale) * w_scale) + bias."""
    _need(q, "q", torch.int8)
    M, K = q.shape
    dev = q.device
    _need(x_scale, "x_scale", torch.float32, (M,), dev)
    _need(w_packed, "w_packed", torch.uint8, None, dev)
    _need(w_scale, "w_scale", torch.float32, (N,), dev)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, (N,), dev)
    ws = workspace(quant_matmul_workspace_bytes(M, N, K), dev) if ws is None else ws
    _need(ws, "ws", torch.uint8, None, dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev) if y is None else y
    _need(y, "y", torch.bfloat16, (M, N), dev)
    with torch.cuda.device(dev):
        _capi.check("w8a8_quant_matmul", _capi.lib().w8a8_quant_matmul(
            q.data_ptr(), x_scale.data_ptr(), M, K, w_packed.data_ptr(), w_scale.data_ptr(), N,
            _ptr(bias), y.data_ptr(), ws.data_ptr(), ws.numel(), _stream(dev)))
    return y


def w8a8_quant_matmul_noalloc(q: torch.Tensor, x_scale: torch.Tensor, w_packed: torch.Tensor,
                              w_scale: torch.Tensor, N: int, bias: Optional[torch.Tensor] = None,
                              y: Optional[torch.Tensor] = None):
    """w8a8_quant_matmul for callers that cannot allocate device memory: the
    library's built-in scratch array replaces the workspace (y must be given by
    such callers; it is allocated here only for convenience)."""
    _need(q, "q", torch.int8)
    M, K = q.shape
    dev = q.device
    _need(x_scale, "x_scale", torch.float32, (M,), dev)
    _need(w_packed, "w_packed", torch.uint8, None, dev)
    _need(w_scale, "w_scale", torch.float32, (N,), dev)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, (N,), dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev) if y is None else y
    _need(y, "y", torch.bfloat16, (M, N), dev)
    with torch.cuda.device(dev):
        _capi.check("w8a8_quant_matmul_noalloc", _capi.lib().w8a8_quant_matmul_noalloc(
            q.data_ptr(), x_scale.data_ptr(), M, K, w_packed.data_ptr(), w_scale.data_ptr(), N,
            _ptr(bias), y.data_ptr(), _stream(dev)))
    return y


def w8a8_int8_matmul_acc(q: torch.Tensor, w_packed: torch.Tensor, N: int,
                         ws: Optional[torch.Tensor] = None):
    """Exact INT32 accumulators acc [M,N] = q [M,K] x W[N,K]^T (validation entry)."""
    _need(q, "q", torch.int8)
    M, K = q.shape
    dev = q.device
    ws = workspace(quant_matmul_workspace_bytes(M, N, K), dev) if ws is None else ws
    acc = torch.empty((M, N), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _capi.check("w8a8_int8_matmul_acc", _capi.lib().w8a8_int8_matmul_acc(
            q.data_ptr(), M, K, w_packed.data_ptr(), N, acc.data_ptr(), ws.data_ptr(), ws.numel(),
            _stream(dev)))
    return acc


def grouped_matmul_workspace_bytes(E: int, R: int, N: int, K: int) -> int:
    return int(_capi.lib().w8a8_grouped_matmul_workspace_bytes(E, R, N, K))


def w8a8_grouped_matmul(q: torch.Tensor, x_scale: torch.Tensor, group_list: torch.Tensor,
                        w_packed: torch.Tensor, w_scale: torch.Tensor,
                        ws: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None):
    """int8 q [R,K] (rows grouped by expert) x packed W [E,N,K] -> bf16 [R,N]."""
    _need(q, "q", torch.int8)
    R, K = q.shape
    dev = q.device
    _need(group_list, "group_list", torch.int64, None, dev)
    E = group_list.numel()
    _need(w_scale, "w_scale", torch.float32, None, dev)
    N = w_scale.shape[-1]
    _need(x_scale, "x_scale", torch.float32, (R,), dev)
    ws = workspace(grouped_matmul_workspace_bytes(E, R, N, K), dev) if ws is None else ws
    y = torch.empty((R, N), dtype=torch.bfloat16, device=dev) if y is None else y
    with torch.cuda.device(dev):
        _capi.check("w8a8_grouped_matmul", _capi.lib().w8a8_grouped_matmul(
            q.data_ptr(), x_scale.data_ptr(), group_list.data_ptr(), E, R, K, w_packed.data_ptr(),
            w_scale.data_ptr(), N, y.data_ptr(), ws.data_ptr(), ws.numel(), _stream(dev)))
    return y


def w8a8_grouped_matmul_acc(q: torch.Tensor, group_list: torch.Tensor, w_packed: torch.Tensor,
                            N: int, ws: Optional[torch.Tensor] = None):
    _need(q, "q", torch.int8)
    R, K = q.shape
    dev = q.device
    _need(group_list, "group_list", torch.int64, None, dev)
    E = group_list.numel()
    ws = workspace(grouped_matmul_workspace_bytes(E, R, N, K), dev) if ws is None else ws
    acc = torch.empty((R, N), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _capi.check("w8a8_grouped_matmul_acc", _capi.lib().w8a8_grouped_matmul_acc(
            q.data_ptr(), group_list.data_ptr(), E, R, K, w_packed.data_ptr(), N, acc.data_ptr(),
            ws.data_ptr(), ws.numel(), _stream(dev)))
    return acc


def moe_workspace_bytes(R: int, H: int, I: int, E: int) -> int:
    return int(_capi.lib().moe_workspace_bytes(R, H, I, E))


def moe_workspace_offset(R: int, H: int, I: int, E: int, which: int) -> int:
    return int(_capi.lib().moe_workspace_offset(R, H, I, E, which))


def moe_w13_swiglu_requant_w2(x: torch.Tensor, x_scale: Optional[torch.Tensor],
                              group_list: torch.Tensor, w13_packed: torch.Tensor,
                              w13_scale: torch.Tensor, w2_packed: torch.Tensor,
                              w2_scale: torch.Tensor, ws: Optional[torch.Tensor] = None,
                              y: Optional[torch.Tensor] = None):
    """MoE expert FFN: x bf16 [R,H] (x_scale None) or int8 [R,H] with x_scale [R] -> bf16 [R,H]."""
    R, H = x.shape
    dev = x.device
    if x_scale is None:
        _need(x, "x", torch.bfloat16)
    else:
        _need(x, "x", torch.int8)
        _need(x_scale, "x_scale", torch.float32, (R,), dev)
    _need(group_list, "group_list", torch.int64, None, dev)
    E = group_list.numel()
    _need(w13_scale, "w13_scale", torch.float32, None, dev)
    I = w13_scale.shape[-1] // 2
    _need(w2_scale, "w2_scale", torch.float32, (E, H), dev)
    ws = workspace(moe_workspace_bytes(R, H, I, E), dev) if ws is None else ws
    y = torch.empty((R, H), dtype=torch.bfloat16, device=dev) if y is None else y
    with torch.cuda.device(dev):
        _capi.check("moe_w13_swiglu_requant_w2", _capi.lib().moe_w13_swiglu_requant_w2(
            x.data_ptr(), _ptr(x_scale), group_list.data_ptr(), E, R, H, I, w13_packed.data_ptr(),
            w13_scale.data_ptr(), w2_packed.data_ptr(), w2_scale.data_ptr(), ws.data_ptr(),
            ws.numel(), y.data_ptr(), _stream(dev)))
    return y


def moe_route_workspace_bytes(T: int, k: int, E: int) -> int:
    return int(_capi.lib().moe_route_workspace_bytes(T, k, E))


def moe_permute_quant(x: torch.Tensor, x_scale: Optional[torch.Tensor], topk_ids: torch.Tensor, E: int,
                      ws: Optional[torch.Tensor] = None, out=None):
    """Token rows -> routed rows grouped by expert.  x bf16 [T,H] (x_scale None: each token quantised
    once) or int8 [T,H] with x_scale [T]; topk_ids int64 [T,k].  Returns (int8 xq [T*k,H],
    float32 xs [T*k], int64 group_list [E], int32 pos [T,k]), written into `out` when given."""
    T, H = x.shape
    dev = x.device
    if x_scale is None:
        _need(x, "x", torch.bfloat16)
    else:
        _need(x, "x", torch.int8)
        _need(x_scale, "x_scale", torch.float32, (T,), dev)
    _need(topk_ids, "topk_ids", torch.int64, None, dev)
    if topk_ids.dim() != 2 or topk_ids.shape[0] != T:
        raise ValueError("topk_ids must be [T,k]")
    k = topk_ids.shape[1]
    ws = workspace(moe_route_workspace_bytes(T, k, E), dev) if ws is None else ws
    _need(ws, "ws", torch.uint8, None, dev)
    if out is None:
        out = (torch.empty((T * k, H), dtype=torch.int8, device=dev),
               torch.empty((T * k,), dtype=torch.float32, device=dev),
               torch.empty((E,), dtype=torch.int64, device=dev),
               torch.empty((T, k), dtype=torch.int32, device=dev))
    xq, xs, group_list, pos = out
    _need(xq, "xq", torch.int8, (T * k, H), dev)
    _need(xs, "xs", torch.float32, (T * k,), dev)
    _need(group_list, "group_list", torch.int64, (E,), dev)
    _need(pos, "pos", torch.int32, (T, k), dev)
    with torch.cuda.device(dev):
        _capi.check("moe_permute_quant", _capi.lib().moe_permute_quant(
            x.data_ptr(), _ptr(x_scale), topk_ids.data_ptr(), T, k, E, H, xq.data_ptr(), xs.data_ptr(),
            group_list.data_ptr(), pos.data_ptr(), ws.data_ptr(), ws.numel(), _stream(dev)))
    return xq, xs, group_list, pos


def moe_unpermute_combine(y_routed: torch.Tensor, pos: torch.Tensor, topk_weights: torch.Tensor,
                          ws: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None):
    """bf16 y_routed [T*k,H], int32 pos [T,k], float32 topk_weights [T,k] -> bf16 y [T,H]."""
    _need(y_routed, "y_routed", torch.bfloat16)
    dev = y_routed.device
    _need(pos, "pos", torch.int32, None, dev)
    if pos.dim() != 2:
        raise ValueError("pos must be [T,k]")
    T, k = pos.shape
    H = y_routed.shape[1]
    if y_routed.shape[0] != T * k:
        raise ValueError("y_routed must have T*k rows")
    _need(topk_weights, "topk_weights", torch.float32, (T, k), dev)
    ws = workspace(_capi.STATUS_BYTES, dev) if ws is None else ws
    _need(ws, "ws", torch.uint8, None, dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if y is None else y
    _need(y, "y", torch.bfloat16, (T, H), dev)
    with torch.cuda.device(dev):
        _capi.check("moe_unpermute_combine", _capi.lib().moe_unpermute_combine(
            y_routed.data_ptr(), pos.data_ptr(), topk_weights.data_ptr(), T, k, H, y.data_ptr(),
            ws.data_ptr(), ws.numel(), _stream(dev)))
    return y


def moe_layer_workspace_bytes(T: int, k: int, H: int, I: int, E: int) -> int:
    return int(_capi.lib().moe_layer_workspace_bytes(T, k, H, I, E))


def moe_layer_workspace_offset(T: int, k: int, H: int, I: int, E: int, which: int) -> int:
    return int(_capi.lib().moe_layer_workspace_offset(T, k, H, I, E, which))


def moe_layer(x: torch.Tensor, x_scale: Optional[torch.Tensor], topk_ids: torch.Tensor,
              topk_weights: torch.Tensor, w13_packed: torch.Tensor, w13_scale: torch.Tensor,
              w2_packed: torch.Tensor, w2_scale: torch.Tensor, ws: Optional[torch.Tensor] = None,
              y: Optional[torch.Tensor] = None):
    """MoE layer from token rows and router output: x bf16 [T,H] (or int8 with x_scale [T]),
    topk_ids int64 [T,k], topk_weights float32 [T,k] -> bf16 y [T,H]."""
    T, H = x.shape
    dev = x.device
    if x_scale is None:
        _need(x, "x", torch.bfloat16)
    else:
        _need(x, "x", torch.int8)
        _need(x_scale, "x_scale", torch.float32, (T,), dev)
    _need(topk_ids, "topk_ids", torch.int64, None, dev)
    if topk_ids.dim() != 2 or topk_ids.shape[0] != T:
        raise ValueError("topk_ids must be [T,k]")
    k = topk_ids.shape[1]
    _need(topk_weights, "topk_weights", torch.float32, (T, k), dev)
    _need(w13_scale, "w13_scale", torch.float32, None, dev)
    E = w13_scale.shape[0]
    I = w13_scale.shape[-1] // 2
    _need(w2_scale, "w2_scale", torch.float32, (E, H), dev)
    ws = workspace(moe_layer_workspace_bytes(T, k, H, I, E), dev) if ws is None else ws
    _need(ws, "ws", torch.uint8, None, dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if y is None else y
    _need(y, "y", torch.bfloat16, (T, H), dev)
    with torch.cuda.device(dev):
        _capi.check("moe_layer", _capi.lib().moe_layer(
            x.data_ptr(), _ptr(x_scale), topk_ids.data_ptr(), topk_weights.data_ptr(), T, k, E, H, I,
            w13_packed.data_ptr(), w13_scale.data_ptr(), w2_packed.data_ptr(), w2_scale.data_ptr(),
            ws.data_ptr(), ws.numel(), y.data_ptr(), _stream(dev)))
    return y


def read_device_status(ws: torch.Tensor) -> int:
    """Synchronise the current stream and return (and clear) the device status word of `ws`."""
    with torch.cuda.device(ws.device):
        return int(_capi.lib().w8a8_read_device_status(ws.data_ptr(), _stream(ws.device)))


ENGINE_NONE, ENGINE_WARP, ENGINE_DECODE, ENGINE_TC, ENGINE_TC_I8 = 0, 1, 2, 3, 4


def last_engine() -> int:
    """Engine the calling thread's last contraction ran on (ENGINE_WARP / ENGINE_DECODE / ENGINE_TC /
    ENGINE_TC_I8)."""
    return int(_capi.lib().w8a8_last_engine())
