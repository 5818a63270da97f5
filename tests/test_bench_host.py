"""Host-side helpers of bench.py (no GPU).

- The recorded DRAM traffic is keyed by call, workload and packed layout.
- A row is used only while the call's CUDA sources hash to the digest recorded with it.
- The pipelined end-to-end leg is described in the bench line.
- The host CPU model is reported beside the oracle baseline."""
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _Wl:
    def __init__(self, name, pack=None):
        self.name = name
        self.pack = pack


def test_traffic_key_names_the_packed_layout():
    assert bench.traffic_key(_Wl("moe_prefill_x", "i8+f16")) == "moe_prefill_x [i8+f16]"
    assert bench.traffic_key(_Wl("dense_decode_x", "i8")) == "dense_decode_x [i8]"
    assert bench.traffic_key(_Wl("weight_quant_x")) == "weight_quant_x"


def test_the_traffic_table_has_a_row_for_the_default_workload():
    key = bench.traffic_key(_Wl("moe_prefill_T4096_H4096_I2048_E64_top8_zipf1.1", "i8+f16"))
    rows = [[c.strip() for c in ln.strip().strip("|").split("|")]
            for ln in open(os.path.join(ROOT, "profiles", "ncu_traffic.md")) if ln.startswith("| moe_layer")]
    assert any(r[1] == key and float(r[2]) > 1e9 and len(r[3]) == 16 for r in rows)
    assert bench.recorded_traffic("moe_layer", key + "x") is None
    assert bench.recorded_traffic("no_such_call", key) is None


def test_recorded_traffic_needs_the_recorded_source_digest(tmp_path, monkeypatch):
    """A row whose digest no longer matches the sources is not used."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    digest = bench.source_digest("moe_layer")
    (prof / "ncu_traffic.md").write_text(
        "| kernel | workload | dram_bytes_per_launch | source_digest |\n|---|---|---|---|\n"
        f"| moe_layer | w [i8] | 123 | {digest} |\n"
        "| moe_layer | v [i8] | 456 | 0000000000000000 |\n")
    shutil.copytree(os.path.join(ROOT, "w8a8_dynamic_quant_gb300", "csrc"),
                    tmp_path / "w8a8_dynamic_quant_gb300" / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("moe_layer", "w [i8]") == 123.0
    assert bench.recorded_traffic("moe_layer", "v [i8]") is None
    # a changed source file invalidates the row
    f = tmp_path / "w8a8_dynamic_quant_gb300" / "csrc" / "quant.cu"
    f.write_text(f.read_text() + "\n// changed\n")
    assert bench.recorded_traffic("moe_layer", "w [i8]") is None


def test_source_digest_covers_the_files_each_call_is_built_from():
    for call in ("dynamic_quant", "quant_matmul", "moe_layer", "mx_matmul"):
        for f in bench.KERNEL_SOURCES[call]:
            assert os.path.exists(os.path.join(ROOT, "w8a8_dynamic_quant_gb300", "csrc", f)), (call, f)
        assert len(bench.source_digest(call)) == 16


def test_e2e_pipeline_shape():
    assert bench.E2E_SLOTS >= 2
    assert "streams" in bench.E2E_PIPELINE and str(bench.E2E_SLOTS) in bench.E2E_PIPELINE


def test_cpu_model_is_reported():
    m = bench.cpu_model()
    assert isinstance(m, str) and m
