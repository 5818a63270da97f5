"""ctypes declarations of the C ABI in include/w8a8.h (libw8a8.so).

Loading fails loudly: there is no Python or CPU fallback for any operation.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw8a8.so")

_i64 = ctypes.c_int64
_u32 = ctypes.c_uint32
_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_int = ctypes.c_int

# name -> (restype, argtypes); every symbol declared in include/w8a8.h
SIGNATURES = {
    "w8a8_status_string": (ctypes.c_char_p, [_int]),
    "w8a8_version": (_int, []),
    "w8a8_prepacked_bytes": (_sz, [_i64, _i64, _i64, _u32]),
    "w8a8_prepack_weight": (_int, [_vp, _i64, _i64, _i64, _u32, _vp, _vp]),
    "w8a8_quantize_weight": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "w8a8_quantize_prepack_weight": (_int, [_vp, _i64, _i64, _i64, _u32, _vp, _vp, _vp]),
    "w8a8_dynamic_quant": (_int, [_vp, _i64, _i64, _vp, _vp, _vp]),
    "w8a8_mx_quant": (_int, [_vp, _i64, _i64, _vp, _vp, _vp]),
    "w8a8_mx_matmul": (_int, [_vp, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _vp]),
    "w8a8_static_quant": (_int, [_vp, _i64, _i64, ctypes.c_float, ctypes.c_int32, _vp, _vp]),
    "w8a8_static_prepare": (_int, [_vp, _i64, _i64, _vp, ctypes.c_float, ctypes.c_int32, _vp, _vp, _vp, _vp]),
    "w8a8_static_quant_matmul": (_int, [_vp, _i64, _i64, _vp, _vp, _vp, _i64, _vp, _vp, _sz, _vp]),
    "w8a8_quant_matmul_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "w8a8_quant_matmul": (_int, [_vp, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _vp, _vp, _sz, _vp]),
    "w8a8_int8_matmul_acc": (_int, [_vp, _i64, _i64, _vp, _i64, _vp, _vp, _sz, _vp]),
    "w8a8_grouped_matmul_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64]),
    "w8a8_grouped_matmul": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _i64, _vp, _vp, _sz, _vp]),
    "w8a8_grouped_matmul_acc": (_int, [_vp, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _sz, _vp]),
    "moe_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64]),
    "moe_workspace_offset": (_i64, [_i64, _i64, _i64, _i64, _int]),
    "moe_w13_swiglu_requant_w2": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _sz,
                                         _vp, _vp]),
    "moe_route_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "moe_permute_quant": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_unpermute_combine": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _sz, _vp]),
    "moe_layer_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64, _i64]),
    "moe_layer": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _sz, _vp,
                         _vp]),
    "moe_layer_workspace_offset": (_i64, [_i64, _i64, _i64, _i64, _i64, _int]),
    "w8a8_quant_matmul_noalloc": (_int, [_vp, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _vp, _vp]),
    "w8a8_quant_matmul_noalloc_status": (_int, [_vp]),
    "w8a8_read_device_status": (_int, [_vp, _vp]),
    "w8a8_selftest_bounded_wait": (_int, [_vp, _u32, _vp]),
    "w8a8_last_engine": (_int, []),
}

STATUS = {0: "W8A8_OK", 1: "W8A8_ERR_NULL", 2: "W8A8_ERR_SHAPE", 3: "W8A8_ERR_ALIGN",
          4: "W8A8_ERR_WORKSPACE", 5: "W8A8_ERR_GROUP_LIST", 6: "W8A8_ERR_DEVICE_TIMEOUT",
          7: "W8A8_ERR_CUDA", 8: "W8A8_ERR_UNSUPPORTED", 9: "W8A8_ERR_PACKED", 10: "W8A8_ERR_TOPK_IDS"}
STATUS_BYTES = 256
W8A8_OK, W8A8_ERR_WORKSPACE, W8A8_ERR_DEVICE_TIMEOUT, W8A8_ERR_PACKED = 0, 4, 6, 9
PACK_GATE_UP = 1
PACK_F16 = 2

_lib = None
_lock = threading.Lock()


class W8A8Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = STATUS.get(code, f"status {code}")
        try:
            msg = lib().w8a8_status_string(code).decode()
        except Exception:
            pass
        super().__init__(f"{fn}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded libw8a8.so.  Raises if the CUDA library has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            import torch  # noqa: F401  (brings the shared CUDA runtime into the process)
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def check(fn: str, code: int):
    if code != 0:
        raise W8A8Error(fn, code)
