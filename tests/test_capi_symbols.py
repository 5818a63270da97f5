"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
function include/w8a8.h declares, and rejects bad arguments on the host before
touching the device.  No compute calls: CPU only."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w8a8.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:W8A8_API\s+)?(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\**\s+\**([a-z][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from w8a8_dynamic_quant_gb300 import build, _capi
    build.build()
    return _capi.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("w8a8_prepack_weight", "w8a8_dynamic_quant", "w8a8_quant_matmul",
                 "w8a8_grouped_matmul", "moe_w13_swiglu_requant_w2", "w8a8_read_device_status"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    from w8a8_dynamic_quant_gb300 import _capi
    names = declared_functions()
    assert set(names) == set(_capi.SIGNATURES), set(names) ^ set(_capi.SIGNATURES)
    for n in names:
        assert hasattr(lib, n), n


def test_only_the_boundary_is_exported(lib):
    import subprocess
    from w8a8_dynamic_quant_gb300 import _capi
    out = subprocess.run(["nm", "-D", "--defined-only", _capi.LIB_PATH], capture_output=True, text=True).stdout
    ours = {ln.split()[-1] for ln in out.splitlines() if ln.split() and ln.split()[-1].startswith(("w8a8_", "moe_"))}
    assert ours == set(declared_functions())


def test_status_strings_and_sizes(lib):
    assert lib.w8a8_status_string(0) == b"W8A8_OK"
    assert b"group_list" in lib.w8a8_status_string(5)
    assert lib.w8a8_version() >= 100
    assert lib.w8a8_prepacked_bytes(1, 256, 512, 0) >= 256 * 512 + 256
    assert lib.w8a8_prepacked_bytes(2, 256, 512, 2) >= 3 * 2 * 256 * 512
    assert lib.w8a8_prepacked_bytes(0, 256, 512, 0) == 0
    assert lib.moe_workspace_bytes(1024, 7168, 2048, 256) > 1024 * (7168 + 3 * 2048)
    offs = [lib.moe_workspace_offset(100, 256, 128, 8, i) for i in range(5)]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lib.moe_workspace_offset(100, 256, 128, 8, 9) == -1
    assert lib.w8a8_status_string(10).startswith(b"W8A8_ERR_TOPK_IDS")
    assert lib.moe_route_workspace_bytes(4096, 8, 64) >= 256 + 64 * 4 * (4096 * 8 // 512)
    assert lib.moe_route_workspace_bytes(4, 0, 8) == 0
    T, k, H, I, E = 100, 3, 256, 128, 8
    lo = [lib.moe_layer_workspace_offset(T, k, H, I, E, i) for i in (0, 1, 2, 3, 4, 7, 8, 9)]
    assert lo == sorted(lo) and all(o % 256 == 0 for o in lo)
    assert lo[:5] == [lib.moe_workspace_offset(T * k, H, I, E, i) for i in range(5)]
    assert lib.moe_layer_workspace_bytes(T, k, H, I, E) >= lo[-1] + T * k * H * 2


def test_host_validation_rejects_before_launch(lib):
    # K % 16 != 0 -> ALIGN; negative M -> SHAPE; NULL pointers -> NULL; none reach the device
    fake = ctypes.c_void_p(16)
    assert lib.w8a8_dynamic_quant(fake, 4, 24, fake, fake, None) == 3
    assert lib.w8a8_dynamic_quant(fake, -1, 32, fake, fake, None) == 2
    assert lib.w8a8_dynamic_quant(None, 4, 32, fake, fake, None) == 1
    assert lib.w8a8_dynamic_quant(fake, 0, 32, fake, fake, None) == 0  # empty: nothing to do
    assert lib.w8a8_quant_matmul(fake, fake, 4, 70000 * 16, fake, fake, 8, None, fake, fake, 1 << 20, None) == 2
    assert lib.w8a8_quant_matmul(fake, fake, 4, 64, ctypes.c_void_p(256), fake, 8, None, fake, None, 0, None) == 4
    assert lib.w8a8_quant_matmul(fake, fake, 4, 64, ctypes.c_void_p(256), fake, 8, None, fake, fake, 16, None) == 4
    assert lib.w8a8_grouped_matmul(fake, fake, fake, 2000, 8, 64, fake, fake, 8, fake, fake, 1 << 20, None) == 2
    assert lib.moe_w13_swiglu_requant_w2(fake, None, fake, 4, 8, 64, 96, fake, fake, fake, fake, fake, 1 << 30,
                                         fake, None) == 2  # I % 64 != 0
    assert lib.w8a8_prepack_weight(fake, 1, 130, 64, 1, ctypes.c_void_p(256), None) == 2  # gate/up needs I % 64 == 0
    assert lib.w8a8_prepack_weight(fake, 1, 128, 64, 8, ctypes.c_void_p(256), None) == 2  # unknown flag
    # MXFP8: K % 32, negative M; contraction K % 128
    assert lib.w8a8_mx_matmul(fake, fake, 4, 96, fake, fake, 8, fake, None) == 3
    assert lib.w8a8_mx_quant(fake, 4, 48, fake, fake, None) == 3
    assert lib.w8a8_mx_quant(fake, -1, 64, fake, fake, None) == 2
    # static W8A8: scale <= 0, offset out of int8, K % 16, missing quant_bias
    assert lib.w8a8_static_quant(fake, 4, 32, 0.0, 0, fake, None) == 2
    assert lib.w8a8_static_quant(fake, 4, 32, 0.1, 200, fake, None) == 2
    assert lib.w8a8_static_quant(fake, 4, 24, 0.1, 0, fake, None) == 3
    assert lib.w8a8_static_prepare(fake, 8, 32, fake, 0.1, 0, None, None, fake, None) == 1
    assert lib.w8a8_static_quant_matmul(fake, 4, 64, ctypes.c_void_p(256), fake, None, 8, fake, fake, 1 << 20,
                                        None) == 1
    # weight quantisation: K % 16, E out of range, unknown flag, gate/up needs (N/2) % 64, packed alignment
    assert lib.w8a8_quantize_weight(fake, 1, 8, 24, fake, fake, None) == 3
    assert lib.w8a8_quantize_weight(fake, 2000, 8, 32, fake, fake, None) == 2
    assert lib.w8a8_quantize_weight(None, 1, 8, 32, fake, fake, None) == 1
    assert lib.w8a8_quantize_prepack_weight(fake, 1, 128, 64, 8, ctypes.c_void_p(256), fake, None) == 2
    assert lib.w8a8_quantize_prepack_weight(fake, 1, 130, 64, 1, ctypes.c_void_p(256), fake, None) == 2
    assert lib.w8a8_quantize_prepack_weight(fake, 1, 128, 64, 0, ctypes.c_void_p(272), fake, None) == 3
    # routing: k < 1, E out of range, H % 16, T*k past int32, missing workspace
    big = 1 << 20
    assert lib.moe_permute_quant(fake, None, fake, 4, 0, 8, 64, fake, fake, fake, fake, fake, big, None) == 2
    assert lib.moe_permute_quant(fake, None, fake, 4, 2, 2000, 64, fake, fake, fake, fake, fake, big, None) == 2
    assert lib.moe_permute_quant(fake, None, fake, 4, 2, 8, 72, fake, fake, fake, fake, fake, big, None) == 3
    assert lib.moe_permute_quant(fake, None, fake, 1 << 30, 4, 8, 64, fake, fake, fake, fake, fake, big, None) == 2
    assert lib.moe_permute_quant(fake, None, fake, 4, 2, 8, 64, fake, fake, fake, fake, None, big, None) == 4
    assert lib.moe_permute_quant(fake, None, fake, 4, 2, 8, 64, fake, fake, fake, fake, fake, 16, None) == 4
    assert lib.moe_unpermute_combine(fake, fake, fake, 4, 2, 60, fake, fake, big, None) == 3
    assert lib.moe_unpermute_combine(fake, fake, fake, 4, 2, 64, fake, fake, 16, None) == 4
    assert lib.moe_unpermute_combine(fake, None, fake, 4, 2, 64, fake, fake, big, None) == 1
    assert lib.moe_unpermute_combine(fake, fake, fake, 0, 2, 64, fake, fake, big, None) == 0
    assert lib.moe_layer(fake, None, fake, fake, 4, 2, 8, 64, 96, fake, fake, fake, fake, fake, 1 << 30,
                         fake, None) == 2  # I % 64 != 0
    p256 = ctypes.c_void_p(256)
    assert lib.moe_layer(fake, None, fake, fake, 4, 2, 8, 64, 128, p256, fake, p256, fake, fake, 16,
                         fake, None) == 4
    assert lib.moe_layer(fake, None, fake, fake, 0, 2, 8, 64, 128, fake, fake, fake, fake, fake, 16,
                         fake, None) == 0  # no tokens: nothing to do
