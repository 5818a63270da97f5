"""CPU oracle for the W8A8_DYNAMIC linear layer and MoE-expert chain.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only users.  The product path (the CUDA
library under ``w8a8_dynamic_quant_gb300``) never imports this package, and
this package never imports the product.

Every function is a thin numpy <-> C marshalling layer over
``w8a8_oracle.c``; the arithmetic and its page citations live in that file.
BF16 tensors travel as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import threading

import numpy as np

from . import build as _build

_lib = None
_lock = threading.Lock()

_c_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(_build.build())
    return _lib


def use_library(path: str):
    """Point this wrapper at another build of the oracle source (the mutation
    tests load deliberately broken copies this way); returns the previous one."""
    global _lib
    with _lock:
        prev = _lib
        _lib = _load(path)
    return prev


def restore_library(prev):
    global _lib
    with _lock:
        _lib = prev


def _load(path: str) -> ctypes.CDLL:
    L = ctypes.CDLL(path)
    L.oracle_num_threads.restype = ctypes.c_int
    L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_f32.restype = ctypes.c_float
    L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    L.oracle_f32_to_bf16.restype = ctypes.c_uint16
    L.oracle_exp_f32.argtypes = [ctypes.c_float]
    L.oracle_exp_f32.restype = ctypes.c_float
    L.oracle_dynamic_quant.argtypes = [_vp, _c_i64, _c_i64, _vp, _vp]
    L.oracle_int8_gemm_acc.argtypes = [_vp, _c_i64, _c_i64, _vp, _c_i64, _vp]
    L.oracle_epilogue.argtypes = [_vp, _c_i64, _c_i64, _vp, _vp, _vp, _vp]
    L.oracle_quant_matmul.argtypes = [_vp, _vp, _c_i64, _c_i64, _vp, _vp, _c_i64, _vp, _vp]
    L.oracle_check_group_list.argtypes = [_vp, _c_i64, _c_i64]
    L.oracle_grouped_matmul.argtypes = [_vp, _vp, _vp, _c_i64, _c_i64, _c_i64, _vp, _vp,
                                        _c_i64, _vp, _vp]
    L.oracle_swiglu.argtypes = [_vp, _c_i64, _c_i64, _vp]
    L.oracle_moe_w13_swiglu_requant_w2.argtypes = [
        _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, _c_i64, _vp, _vp, _vp, _vp, _vp,
        _vp, _vp, _vp, _vp, _vp, _vp]
    L.oracle_static_quant.argtypes = [_vp, _c_i64, _c_i64, ctypes.c_float, ctypes.c_int32, _vp]
    L.oracle_static_prepare.argtypes = [_vp, _c_i64, _c_i64, _vp, ctypes.c_float, ctypes.c_int32, _vp, _vp, _vp]
    L.oracle_static_quant_matmul.argtypes = [_vp, _c_i64, _c_i64, _vp, _c_i64, _vp, _vp, _vp]
    L.oracle_e4m3_from_f32.argtypes = [ctypes.c_float]
    L.oracle_e4m3_from_f32.restype = ctypes.c_uint8
    L.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_to_f32.restype = ctypes.c_float
    L.oracle_mx_quant.argtypes = [_vp, _c_i64, _c_i64, _vp, _vp]
    L.oracle_mx_matmul.argtypes = [_vp, _vp, _c_i64, _c_i64, _vp, _vp, _c_i64, _vp]
    L.oracle_quantize_weight.argtypes = [_vp, _c_i64, _c_i64, _c_i64, _vp, _vp]
    L.oracle_moe_route.argtypes = [_vp, _c_i64, _c_i64, _c_i64, _vp, _vp]
    L.oracle_moe_permute_quant.argtypes = [_vp, _vp, _vp, _c_i64, _c_i64, _c_i64, _c_i64, _vp, _vp,
                                           _vp, _vp]
    L.oracle_moe_unpermute_combine.argtypes = [_vp, _vp, _vp, _c_i64, _c_i64, _c_i64, _vp]
    L.oracle_moe_layer.argtypes = [_vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _vp,
                                   _vp, _vp, _vp, _vp, _vp]
    return L


class OracleError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned status {code}")
        self.code = code


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _check(fn: str, rc: int):
    if rc != 0:
        raise OracleError(fn, rc)


def num_threads() -> int:
    return lib().oracle_num_threads()


def bf16_to_f32(b: int) -> float:
    return lib().oracle_bf16_to_f32(int(b))


def f32_to_bf16(f: float) -> int:
    return lib().oracle_f32_to_bf16(float(f))


def exp_f32(x: float) -> float:
    """The binary32 exp specification used by SwiGLU (scalar)."""
    return lib().oracle_exp_f32(float(x))


def dynamic_quant(x_bf16: np.ndarray):
    """BF16 bits [M,K] -> (int8 q [M,K], fp32 scale [M])."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    s = np.empty((M,), np.float32)
    _check("oracle_dynamic_quant", lib().oracle_dynamic_quant(_p(x), M, K, _p(q), _p(s)))
    return q, s


def int8_gemm_acc(q: np.ndarray, w: np.ndarray) -> np.ndarray:
    """int8 q [M,K] x int8 W [N,K] -> exact int32 acc [M,N]."""
    q = _c(q, np.int8)
    w = _c(w, np.int8)
    M, K = q.shape
    N = w.shape[0]
    assert w.shape[1] == K
    acc = np.empty((M, N), np.int32)
    _check("oracle_int8_gemm_acc", lib().oracle_int8_gemm_acc(_p(q), M, K, _p(w), N, _p(acc)))
    return acc


def epilogue(acc, x_scale, w_scale, bias=None) -> np.ndarray:
    acc = _c(acc, np.int32)
    M, N = acc.shape
    xs = _c(x_scale, np.float32)
    ws = _c(w_scale, np.float32)
    b = None if bias is None else _c(bias, np.uint16)
    y = np.empty((M, N), np.uint16)
    _check("oracle_epilogue", lib().oracle_epilogue(_p(acc), M, N, _p(xs), _p(ws), _p(b), _p(y)))
    return y


def quant_matmul(q, x_scale, w, w_scale, bias=None) -> np.ndarray:
    """int8 q [M,K], fp32 x_scale [M], int8 W [N,K], fp32 w_scale [N], bf16 bias [N]|None -> bf16 [M,N]."""
    q = _c(q, np.int8)
    xs = _c(x_scale, np.float32)
    w = _c(w, np.int8)
    ws = _c(w_scale, np.float32)
    b = None if bias is None else _c(bias, np.uint16)
    M, K = q.shape
    N = w.shape[0]
    y = np.empty((M, N), np.uint16)
    _check("oracle_quant_matmul",
           lib().oracle_quant_matmul(_p(q), _p(xs), M, K, _p(w), _p(ws), N, _p(b), _p(y)))
    return y


def check_group_list(group_list, R) -> int:
    g = _c(group_list, np.int64)
    return lib().oracle_check_group_list(_p(g), g.shape[0], int(R))


def grouped_matmul(q, x_scale, group_list, w, w_scale, want_acc=False):
    """int8 q [R,K], fp32 x_scale [R], int64 counts [E], int8 W [E,N,K], fp32 w_scale [E,N] -> bf16 [R,N] (, int32 acc)."""
    q = _c(q, np.int8)
    xs = _c(x_scale, np.float32)
    g = _c(group_list, np.int64)
    w = _c(w, np.int8)
    ws = _c(w_scale, np.float32)
    R, K = q.shape
    E, N, K2 = w.shape
    assert K2 == K and g.shape[0] == E
    y = np.empty((R, N), np.uint16)
    acc = np.empty((R, N), np.int32) if want_acc else None
    _check("oracle_grouped_matmul",
           lib().oracle_grouped_matmul(_p(q), _p(xs), _p(g), E, R, K, _p(w), _p(ws), N, _p(y), _p(acc)))
    return (y, acc) if want_acc else y


def swiglu(y13: np.ndarray, I: int) -> np.ndarray:
    y13 = _c(y13, np.uint16)
    R = y13.shape[0]
    assert y13.shape[1] == 2 * I
    h = np.empty((R, I), np.uint16)
    _check("oracle_swiglu", lib().oracle_swiglu(_p(y13), R, I, _p(h)))
    return h


def moe_w13_swiglu_requant_w2(x, x_scale, group_list, w13, s13, w2, s2, intermediates=False):
    """MoE expert FFN.  x: bf16 bits [R,H] if x_scale is None, else int8 [R,H]."""
    g = _c(group_list, np.int64)
    w13 = _c(w13, np.int8)
    s13 = _c(s13, np.float32)
    w2 = _c(w2, np.int8)
    s2 = _c(s2, np.float32)
    E, twoI, H = w13.shape
    I = twoI // 2
    assert w2.shape == (E, H, I) and s13.shape == (E, twoI) and s2.shape == (E, H)
    if x_scale is None:
        x = _c(x, np.uint16)
        xs_in = None
    else:
        x = _c(x, np.int8)
        xs_in = _c(x_scale, np.float32)
    R = x.shape[0]
    assert x.shape[1] == H
    y = np.empty((R, H), np.uint16)
    inter = {}
    if intermediates:
        inter = dict(xq=np.empty((R, H), np.int8), xs=np.empty((R,), np.float32),
                     y13=np.empty((R, twoI), np.uint16), h=np.empty((R, I), np.uint16),
                     hq=np.empty((R, I), np.int8), hs=np.empty((R,), np.float32))
    _check("oracle_moe_w13_swiglu_requant_w2",
           lib().oracle_moe_w13_swiglu_requant_w2(
               _p(x), _p(xs_in), _p(g), E, R, H, I, _p(w13), _p(s13), _p(w2), _p(s2), _p(y),
               _p(inter.get("xq")), _p(inter.get("xs")), _p(inter.get("y13")),
               _p(inter.get("h")), _p(inter.get("hq")), _p(inter.get("hs"))))
    return (y, inter) if intermediates else y


def static_quant(x, input_scale: float, input_offset: int):
    """bf16 bits x [M,K] -> int8 q = clamp(rint(x / s) + o, -128, 127) (static, per-tensor s and o)."""
    x = _c(x, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    _check("oracle_static_quant", lib().oracle_static_quant(_p(x), M, K, float(input_scale), int(input_offset),
                                                            _p(q)))
    return q


def static_prepare(w, w_scale, input_scale: float, input_offset: int, bias=None):
    """int8 W [N,K], fp32 weight scales [N] (+ bf16 bits bias [N]) -> (fp32 deq_scale [N], int32 quant_bias [N])."""
    w = _c(w, np.int8)
    ws = _c(w_scale, np.float32)
    b = None if bias is None else _c(bias, np.uint16)
    N, K = w.shape
    deq = np.empty((N,), np.float32)
    qb = np.empty((N,), np.int32)
    _check("oracle_static_prepare", lib().oracle_static_prepare(_p(w), N, K, _p(ws), float(input_scale),
                                                                int(input_offset), _p(b), _p(deq), _p(qb)))
    return deq, qb


def static_quant_matmul(q, w, deq_scale, quant_bias):
    """int8 q [M,K] x int8 W [N,K] -> bf16 bits y = bf16(float(acc + quant_bias[n]) * deq_scale[n])."""
    q = _c(q, np.int8)
    w = _c(w, np.int8)
    deq = _c(deq_scale, np.float32)
    qb = _c(quant_bias, np.int32)
    M, K = q.shape
    N = w.shape[0]
    y = np.empty((M, N), np.uint16)
    _check("oracle_static_quant_matmul", lib().oracle_static_quant_matmul(_p(q), M, K, _p(w), N, _p(deq), _p(qb),
                                                                          _p(y)))
    return y


def quantize_weight(w):
    """bf16 bits W [N,K] or [E,N,K] -> (int8 q of the same shape, fp32 per-channel scales [N] or [E,N])."""
    w = _c(w, np.uint16)
    w3 = w.reshape((1,) + w.shape) if w.ndim == 2 else w
    E, N, K = w3.shape
    q = np.empty((E, N, K), np.int8)
    s = np.empty((E, N), np.float32)
    _check("oracle_quantize_weight", lib().oracle_quantize_weight(_p(w3), E, N, K, _p(q), _p(s)))
    return (q[0], s[0]) if w.ndim == 2 else (q, s)


def moe_route(topk_ids, E: int):
    """int64 topk_ids [T,k] -> (int64 group_list [E], int32 pos [T,k]): routed rows ordered by
    (expert, token, slot); pos[t,j] is the routed row of token t's j-th choice."""
    ids = _c(topk_ids, np.int64)
    T, k = ids.shape
    g = np.empty((E,), np.int64)
    pos = np.empty((T, k), np.int32)
    _check("oracle_moe_route", lib().oracle_moe_route(_p(ids), T, k, E, _p(g), _p(pos)))
    return g, pos


def moe_permute_quant(x, x_scale, topk_ids, E: int):
    """Token rows -> routed rows.  x: bf16 bits [T,H] (x_scale None) or int8 [T,H] with fp32
    x_scale [T].  Returns (int8 xq [T*k,H], fp32 xs [T*k], int64 group_list [E], int32 pos [T,k])."""
    ids = _c(topk_ids, np.int64)
    T, k = ids.shape
    if x_scale is None:
        x = _c(x, np.uint16)
        xs_in = None
    else:
        x = _c(x, np.int8)
        xs_in = _c(x_scale, np.float32)
    assert x.shape[0] == T
    H = x.shape[1]
    xq = np.empty((T * k, H), np.int8)
    xs = np.empty((T * k,), np.float32)
    g = np.empty((E,), np.int64)
    pos = np.empty((T, k), np.int32)
    _check("oracle_moe_permute_quant", lib().oracle_moe_permute_quant(
        _p(x), _p(xs_in), _p(ids), T, k, E, H, _p(xq), _p(xs), _p(g), _p(pos)))
    return xq, xs, g, pos


def moe_unpermute_combine(y_routed, pos, topk_weights):
    """bf16 bits y_routed [T*k,H], int32 pos [T,k], fp32 weights [T,k] -> bf16 bits y [T,H]."""
    yr = _c(y_routed, np.uint16)
    pos = _c(pos, np.int32)
    w = _c(topk_weights, np.float32)
    T, k = pos.shape
    assert w.shape == (T, k) and yr.shape[0] == T * k
    H = yr.shape[1]
    y = np.empty((T, H), np.uint16)
    _check("oracle_moe_unpermute_combine",
           lib().oracle_moe_unpermute_combine(_p(yr), _p(pos), _p(w), T, k, H, _p(y)))
    return y


def moe_layer(x, x_scale, topk_ids, topk_weights, w13, s13, w2, s2, want_routed=False):
    """Whole MoE layer from token rows: permute + quant -> W13 -> SwiGLU -> requant -> W2 ->
    weighted combine.  Returns bf16 bits y [T,H] (and the routed W2 output [T*k,H])."""
    ids = _c(topk_ids, np.int64)
    w = _c(topk_weights, np.float32)
    w13 = _c(w13, np.int8)
    s13 = _c(s13, np.float32)
    w2 = _c(w2, np.int8)
    s2 = _c(s2, np.float32)
    E, twoI, H = w13.shape
    I = twoI // 2
    T, k = ids.shape
    assert w.shape == (T, k) and w2.shape == (E, H, I)
    if x_scale is None:
        x = _c(x, np.uint16)
        xs_in = None
    else:
        x = _c(x, np.int8)
        xs_in = _c(x_scale, np.float32)
    assert x.shape == (T, H)
    y = np.empty((T, H), np.uint16)
    yr = np.empty((T * k, H), np.uint16) if want_routed else None
    _check("oracle_moe_layer", lib().oracle_moe_layer(
        _p(x), _p(xs_in), _p(ids), _p(w), T, k, E, H, I, _p(w13), _p(s13), _p(w2), _p(s2), _p(y),
        _p(yr)))
    return (y, yr) if want_routed else y


def e4m3_from_f32(v: float) -> int:
    return int(lib().oracle_e4m3_from_f32(float(v)))


def e4m3_to_f32(b: int) -> float:
    return float(lib().oracle_e4m3_to_f32(int(b)))


def mx_quant(x):
    """bf16 bits x [M,K] (K % 32 == 0) -> (uint8 E4M3 codes [M,K], uint8 E8M0 scales [M,K/32])."""
    x = _c(x, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((M, K // 32), np.uint8)
    _check("oracle_mx_quant", lib().oracle_mx_quant(_p(x), M, K, _p(q), _p(s)))
    return q, s


def mx_matmul(qa, sa, qw, sw):
    """MXFP8 operands (E4M3 codes + E8M0 scales per 32 along K) -> bf16 bits y [M,N] (float64 sum)."""
    qa, sa, qw, sw = (_c(t, np.uint8) for t in (qa, sa, qw, sw))
    M, K = qa.shape
    N = qw.shape[0]
    y = np.empty((M, N), np.uint16)
    _check("oracle_mx_matmul", lib().oracle_mx_matmul(_p(qa), _p(sa), M, K, _p(qw), _p(sw), N, _p(y)))
    return y
