#!/usr/bin/env python3
"""Benchmark of the W8A8_DYNAMIC hot path on GB300 (one JSON line on stdout).

Default workload: the MoE prefill layer, T=4096 tokens, H=4096, I=2048,
E=64 experts, top-8 routing with Zipf(1.1) popularity (R = 32768 routed rows,
4 experts empty); one step = per-token INT8 quant of the routed BF16 rows ->
W13 grouped GEMM with SwiGLU fused into its epilogue -> per-token INT8
requant -> W2 grouped GEMM -> BF16.  `--workload N` selects one of the five
workloads (1 tiny dense, 2 dense decode, 3 dense prefill, 4 MoE prefill,
5 MoE decode with pre-quantised input).

Timing: W warm-up steps, then exactly K steps between a barrier +
synchronize on both sides.  The step (every kernel of the path, in order, on
one input set) is captured into CUDA graphs over rotating input sets whose
total size exceeds the 129 MB L2 (or a single set when one set already
exceeds it): one graph of a step on each set and one of a whole rotation, so
that exactly W and K steps run; the K steps are timed with CUDA events on
the stream they run on.  Kernels of a step may overlap where the library
lets them (the decode contraction starts its weight stream while the
quantisation still runs).  Each kernel type is
also captured on its own over the same sets for the per-kernel breakdown and
the roofline of the dominant kernel.  The
`e2e` leg runs the same step through the public Python API with the inputs
copied from pinned host memory and the result copied back every step, the
copies of one step overlapping the compute of its neighbours (two buffer
slots, three streams).
`cpu_baseline` times the CPU oracle on the host cores on a bounded sample.
`--impl reference` runs that oracle as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W8A8 GEMM TOPS & % INT8 peak; grouped-MoE layer tokens/s; quant GB/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- helpers --

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        d = dict(FALLBACK_PEAKS)
        d["source"] = "fallback"
        return d


def weight_read_bound_ms(active_params: float, bytes_per_param: float, n_gpus: int, hbm_bytes_per_s: float):
    """Decode lower bound: every active weight byte is read once per token, spread over n_gpus."""
    return active_params * bytes_per_param / (n_gpus * hbm_bytes_per_s) * 1e3


# CUDA sources each timed kernel is built from (a recorded ncu figure is valid
# only while these files are unchanged)
KERNEL_SOURCES = {
    "dynamic_quant": ["quant.cu", "common.cuh", "kernels.cuh"],
    "quant_matmul": ["gemm_reg.cu", "gemm_dec.cu", "gemm_tc.cu", "gemm_tcp.cu", "tc_common.cuh", "capi.cu",
                     "common.cuh", "kernels.cuh"],
    "moe_layer": ["gemm_reg.cu", "gemm_tc.cu", "gemm_tcp.cu", "tc_common.cuh", "quant.cu", "route.cu", "capi.cu",
                  "common.cuh", "kernels.cuh"],
    "mx_matmul": ["mx.cu", "mx_tc.cu", "tc_common.cuh", "capi.cu", "common.cuh", "kernels.cuh"],
}


def source_digest(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "w8a8_dynamic_quant_gb300", "csrc")
    for f in KERNEL_SOURCES.get(kernel, sorted(os.listdir(csrc))):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def traffic_key(wl) -> str:
    """The workload a recorded DRAM figure belongs to: its name and, where the workload has one, the packed
    weight layout (the contractions read different bytes with and without the fp16 weight copy)."""
    pack = getattr(wl, "pack", None)
    return f"{wl.name} [{pack}]" if pack else wl.name


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch recorded from an ncu capture (profiles/ncu_traffic.md), if the
    kernel sources are unchanged since; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.md")
    if not os.path.exists(path):
        return None
    digest = source_digest(kernel)
    for ln in open(path):
        parts = [p.strip() for p in ln.strip().strip("|").split("|")]
        if len(parts) >= 4 and parts[0] == kernel and parts[1] == workload and parts[3] == digest:
            try:
                return float(parts[2])
            except ValueError:
                return None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in open(self.path):
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def aggregate(units: float, seconds: float, group=None):
    """Whole-job figures across ranks: total units and the slowest rank's time."""
    import torch
    import torch.distributed as dist
    if group is None and not (dist.is_available() and dist.is_initialized()):
        return units, seconds
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend(group) == "nccl" else torch.device("cpu")
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    s = torch.tensor([seconds], dtype=torch.float64, device=dev)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(s, op=dist.ReduceOp.MAX, group=group)
    return float(u.item()), float(s.item())


E2E_SLOTS = 2
E2E_PIPELINE = (f"{E2E_SLOTS} buffer slots; host->device copies, the API calls and the device->host read "
                "on three streams, so that step i's copies overlap the compute of its neighbours")


def run_e2e(torch, wl, steps: int):
    """`steps` end-to-end steps of a workload through its public API calls, pipelined over E2E_SLOTS
    device input/output slots: the copy-in of step i waits until step i - E2E_SLOTS has computed (its
    slot's inputs are free), the compute waits for its inputs and for the read-back of the slot's
    previous output, the read-back waits for the compute.  Returns after a device synchronize."""
    s_comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(E2E_SLOTS)]
    ev_comp = [torch.cuda.Event() for _ in range(E2E_SLOTS)]
    ev_out = [torch.cuda.Event() for _ in range(E2E_SLOTS)]
    s_in.wait_stream(s_comp)
    s_out.wait_stream(s_comp)
    for i in range(steps):
        slot = i % E2E_SLOTS
        if i >= E2E_SLOTS:
            s_in.wait_event(ev_comp[slot])
        with torch.cuda.stream(s_in):
            wl.e2e_in(slot)
        ev_in[slot].record(s_in)
        s_comp.wait_event(ev_in[slot])
        if i >= E2E_SLOTS:
            s_comp.wait_event(ev_out[slot])
        wl.e2e_compute(slot)
        ev_comp[slot].record(s_comp)
        s_out.wait_event(ev_comp[slot])
        with torch.cuda.stream(s_out):
            wl.e2e_out(slot)
        ev_out[slot].record(s_out)
    torch.cuda.synchronize()


# --------------------------------------------------------------- workloads --

class Dense:
    """Dense W8A8_DYNAMIC linear: quant + quantised matmul."""

    def __init__(self, cfg_id: int, device, pack: str = "auto"):
        import torch
        import w8a8_dynamic_quant_gb300 as W
        from w8a8_dynamic_quant_gb300 import synthetic as S
        self.W, self.torch = W, torch
        d = S.dense_config(cfg_id)
        self.d = d
        self.name = d.name
        M, N, K = d.M, d.N, d.K
        self.M, self.N, self.K = M, N, K
        if pack == "auto":
            pack = "i8+f16" if M >= 128 else "i8"
        self.pack = pack
        set_bytes = 2 * M * K + M * K + N * K * (3 if pack == "i8+f16" else 1) + 2 * M * N
        self.n_sets = max(1, -(-int(1.2 * L2_BYTES) // set_bytes))
        self.n_sets = min(self.n_sets, 16)
        xd = torch.from_numpy(d.x.view("int16")).to(device).view(torch.bfloat16)
        wd = torch.from_numpy(d.w).to(device)
        # large M runs on a tcgen05 engine: on the fp16 copy of the weight when the pack holds it
        self.pack_flags = W.PACK_F16 if pack == "i8+f16" else 0
        sw = torch.from_numpy(d.w_scale).to(device)
        bias = None if d.bias is None else torch.from_numpy(d.bias.view("int16")).to(device).view(torch.bfloat16)
        self.sets = []
        for i in range(self.n_sets):
            self.sets.append(dict(
                x=xd.clone(), wp=W.w8a8_prepack_weight(wd, self.pack_flags), sw=sw.clone(),
                bias=None if bias is None else bias.clone(),
                q=torch.empty((M, K), dtype=torch.int8, device=device),
                s=torch.empty((M,), dtype=torch.float32, device=device),
                y=torch.empty((M, N), dtype=torch.bfloat16, device=device),
                ws=W.workspace(W.quant_matmul_workspace_bytes(M, N, K), device)))
        self.units_per_step = 2.0 * M * N * K  # GEMM ops
        self.unit = "TOPS"
        self.kernels = ["dynamic_quant", "quant_matmul"]
        # algorithmic bytes per launch
        self.alg_bytes = {"dynamic_quant": 2 * M * K + M * K + 4 * M,
                          "quant_matmul": M * K + N * K + 4 * M + 4 * N + 2 * M * N + (2 * N if bias is not None else 0)}
        self.alg_flops = {"quant_matmul": 2.0 * M * N * K}
        self.bound = "hbm" if M <= 256 else "tensor"
        self.launches_per_step = 2
        self.input_note = (f"{self.n_sets} rotating input sets of {set_bytes / 1e6:.1f} MB "
                           f"({self.n_sets * set_bytes / 1e6:.0f} MB > 129 MB L2)" if self.n_sets > 1
                           else f"one input set of {set_bytes / 1e6:.0f} MB > 129 MB L2")

    def launch(self, kernel: str, i: int):
        st = self.sets[i]
        if kernel == "dynamic_quant":
            self.W.w8a8_dynamic_quant(st["x"], st["q"], st["s"])
        else:
            self.W.w8a8_quant_matmul(st["q"], st["s"], st["wp"], st["sw"], self.N, st["bias"], st["ws"], st["y"])

    def config(self):
        return {"workload": self.name, "M": self.M, "N": self.N, "K": self.K, "bias": self.d.bias is not None,
                "packed_weights": {"i8": "int8 only", "i8+f16": "int8 + integer-valued fp16 copy"}[self.pack],
                "seed": 0, "inputs": self.input_note}

    def value(self, units, seconds):
        return units / seconds / 1e12

    # end to end through the public API, host buffers: per pipeline slot a device input and output and a
    # pinned host output (the step's compute buffers are shared: the steps compute one after the other)
    def e2e_setup(self, device):
        torch = self.torch
        self.hx = torch.from_numpy(self.d.x.view("int16")).view(torch.bfloat16).pin_memory()
        self.e2e_slots = [dict(x=torch.empty((self.M, self.K), dtype=torch.bfloat16, device=device),
                               y=torch.empty((self.M, self.N), dtype=torch.bfloat16, device=device),
                               hy=torch.empty((self.M, self.N), dtype=torch.bfloat16).pin_memory())
                          for _ in range(E2E_SLOTS)]
        self.h2d = self.hx.numel() * 2
        self.d2h = self.M * self.N * 2

    def e2e_in(self, slot):
        self.e2e_slots[slot]["x"].copy_(self.hx, non_blocking=True)

    def e2e_compute(self, slot):
        st, sl = self.sets[0], self.e2e_slots[slot]
        q, s = self.W.w8a8_dynamic_quant(sl["x"], st["q"], st["s"])
        self.W.w8a8_quant_matmul(q, s, st["wp"], st["sw"], self.N, st["bias"], st["ws"], sl["y"])

    def e2e_out(self, slot):
        sl = self.e2e_slots[slot]
        sl["hy"].copy_(sl["y"], non_blocking=True)

    # CPU oracle on `rows` rows of the same workload
    def oracle_units(self, rows):
        return 2.0 * rows * self.N * self.K

    def oracle_step(self, rows):
        import oracle
        x = self.d.x[:rows]
        q, s = oracle.dynamic_quant(x)
        oracle.quant_matmul(q, s, self.d.w, self.d.w_scale, self.d.bias)

    @property
    def oracle_full_rows(self):
        return self.M


class DenseStatic(Dense):
    """The static W8A8 variant of a dense workload: quantisation with a fixed per-tensor input scale and
    offset, then the matmul whose epilogue adds the load-time quant_bias and scales by deq_scale."""

    def __init__(self, cfg_id: int, device):
        super().__init__(cfg_id, device)
        from w8a8_dynamic_quant_gb300 import synthetic as S
        W, torch, d = self.W, self.torch, self.d
        self.s_in, self.o_in = S.static_params(cfg_id)
        self.name = d.name + "_static"
        wd = torch.from_numpy(d.w).to(device)
        for st in self.sets:  # load time, outside the timed step
            st["deq"], st["qb"] = W.w8a8_static_prepare(wd, st["sw"], self.s_in, self.o_in, st["bias"])
        M, N, K = self.M, self.N, self.K
        self.kernels = ["static_quant", "static_quant_matmul"]
        self.alg_bytes = {"static_quant": 2 * M * K + M * K,
                          "static_quant_matmul": M * K + N * K + 8 * N + 2 * M * N}
        self.alg_flops = {"static_quant_matmul": 2.0 * M * N * K}

    def launch(self, kernel: str, i: int):
        st = self.sets[i]
        if kernel == "static_quant":
            self.W.w8a8_static_quant(st["x"], self.s_in, self.o_in, st["q"])
        else:
            self.W.w8a8_static_quant_matmul(st["q"], st["wp"], st["deq"], st["qb"], st["ws"], st["y"])

    def config(self):
        c = super().config()
        c.update(workload=self.name, input_scale=self.s_in, input_offset=self.o_in)
        return c

    def e2e_compute(self, slot):
        st, sl = self.sets[0], self.e2e_slots[slot]
        q = self.W.w8a8_static_quant(sl["x"], self.s_in, self.o_in, st["q"])
        self.W.w8a8_static_quant_matmul(q, st["wp"], st["deq"], st["qb"], st["ws"], sl["y"])

    def oracle_step(self, rows):
        import oracle
        if not hasattr(self, "_prep"):
            self._prep = oracle.static_prepare(self.d.w, self.d.w_scale, self.s_in, self.o_in, self.d.bias)
        q = oracle.static_quant(self.d.x[:rows], self.s_in, self.o_in)
        oracle.static_quant_matmul(q, self.d.w, *self._prep)


class DenseMX(Dense):
    """The MXFP8 variant of a dense workload: the activations quantised to E4M3 + one E8M0 scale per 32
    along K, then the MXFP8 contraction against weights quantised the same way at load (TOPS)."""

    def __init__(self, cfg_id: int, device):
        super().__init__(cfg_id, device)
        torch, M, K = self.torch, self.M, self.K
        self.name = self.d.name + "_mxfp8"
        N = self.N
        # load time: the weights (the workload's INT8 weight times its channel scale, as BF16) to MXFP8
        wbf = (torch.from_numpy(self.d.w).to(device).float() * torch.from_numpy(self.d.w_scale).to(device)[:, None])
        wq, wsc = self.W.w8a8_mx_quant(wbf.to(torch.bfloat16))
        for st in self.sets:
            st["mq"] = torch.empty((M, K), dtype=torch.uint8, device=device)
            st["ms"] = torch.empty((M, K // 32), dtype=torch.uint8, device=device)
            st["wq"], st["wsc"] = wq.clone(), wsc.clone()
        self.kernels = ["mx_quant", "mx_matmul"]
        self.alg_bytes = {"mx_quant": 2 * M * K + M * K + M * K // 32,
                          "mx_matmul": M * K + N * K + (M + N) * K // 32 + 2 * M * N}
        self.alg_flops = {"mx_matmul": 2.0 * M * N * K}
        self.launches_per_step = 2
        self.tensor_peak_ratio = 2.0  # FP8 tensor rate: the measured bf16 peak x the nominal 2x

    def launch(self, kernel: str, i: int):
        st = self.sets[i]
        if kernel == "mx_quant":
            self.W.w8a8_mx_quant(st["x"], st["mq"], st["ms"])
        else:
            self.W.w8a8_mx_matmul(st["mq"], st["ms"], st["wq"], st["wsc"], st["y"])

    def e2e_compute(self, slot):
        st, sl = self.sets[0], self.e2e_slots[slot]
        q, s = self.W.w8a8_mx_quant(sl["x"], st["mq"], st["ms"])
        self.W.w8a8_mx_matmul(q, s, st["wq"], st["wsc"], sl["y"])

    def oracle_step(self, rows):
        import oracle
        if not hasattr(self, "_wmx"):
            wbf = (self.d.w.astype("float32") * self.d.w_scale[:, None])
            from w8a8_dynamic_quant_gb300 import synthetic as S
            self._wmx = oracle.mx_quant(S.to_bf16_bits(wbf))
        qa, sa = oracle.mx_quant(self.d.x[:rows])
        oracle.mx_matmul(qa, sa, *self._wmx)


class MoE:
    """MoE expert FFN: (quant) -> W13 grouped GEMM + SwiGLU -> requant -> W2 grouped GEMM."""

    def __init__(self, cfg_id: int, device, pack_weights: bool = True, pack: str = "auto", scale: int = 1):
        import numpy as np
        import torch
        import w8a8_dynamic_quant_gb300 as W
        from w8a8_dynamic_quant_gb300 import synthetic as S
        self.W, self.torch, self.np = W, torch, np
        if scale == 1:
            m = S.moe_config(cfg_id, device=str(device))
        else:  # a small case of the same layer: T and E divided by `scale` (profiler captures)
            c = S.CONFIGS[cfg_id]
            T, E = c["T"] // scale, c["E"] // scale
            m = S.make_moe(T, c["H"], c["I"], E, c["topk"], c["routing"], c.get("zipf_s", 1.1),
                           c.get("n_dead", 0) // scale, c["prequant"], 0, str(device),
                           name=f"{c['name']}_reduced_T{T}_E{E}")
        self.m = m
        self.name = m.name
        self.n_sets = 1
        # prefill-sized groups run on a tcgen05 engine: with the packed FP16 weight copy ("i8+f16") or
        # on the INT8 payload widened in tensor memory ("i8")
        if pack == "auto":
            pack = "i8+f16" if m.R >= 64 * m.E else "i8"
        f16 = W.PACK_F16 if pack == "i8+f16" else 0
        self.pack = pack
        self.w13p = W.w8a8_prepack_weight(m.w13, W.PACK_GATE_UP | f16) if pack_weights else None
        self.w2p = W.w8a8_prepack_weight(m.w2, f16) if pack_weights else None
        self.gl = torch.from_numpy(m.group_list).to(device)
        self.s13 = torch.from_numpy(m.s13).to(device)
        self.s2 = torch.from_numpy(m.s2).to(device)
        if m.x_scale is None:
            self.x = torch.from_numpy(m.x.view("int16")).to(device).view(torch.bfloat16)
            self.xs = None
        else:
            self.x = torch.from_numpy(m.x).to(device)
            self.xs = torch.from_numpy(m.x_scale).to(device)
        self.ws = W.workspace(W.moe_workspace_bytes(m.R, m.H, m.I, m.E), device)
        self.y = torch.empty((m.R, m.H), dtype=torch.bfloat16, device=device)
        self.units_per_step = float(m.T)  # tokens
        self.unit = "tokens/s"
        self.kernels = ["moe_layer"]
        active = int((m.group_list > 0).sum())
        R, H, I = m.R, m.H, m.I
        wbytes = active * (2 * I * H + H * I) + 4 * active * (2 * I + H)
        xbytes = R * H * (1 if m.x_scale is not None else 2 + 1 + 1)  # x read (+ quant write/read)
        hbytes = R * I * (2 + 2 + 1 + 1)  # h write+read, hq write+read
        self.alg_bytes = {"moe_layer": wbytes + xbytes + hbytes + 2 * R * H + 8 * R}
        self.alg_flops = {"moe_layer": 2.0 * R * (2 * I * H + H * I)}
        self.bound = "hbm" if m.x_scale is not None else "tensor"
        self.launches_per_step = 3 if m.x_scale is not None else 4
        self.input_note = f"weights {wbytes / 1e9:.2f} GB active > 129 MB L2 (single set)"

    def launch(self, kernel: str, i: int):
        m = self.m
        self.W.moe_w13_swiglu_requant_w2(self.x, self.xs, self.gl, self.w13p, self.s13, self.w2p, self.s2,
                                         self.ws, self.y)

    def config(self):
        m = self.m
        return {"workload": self.name, "T": m.T, "R": m.R, "H": m.H, "I": m.I, "E": m.E, "topk": m.topk,
                "active_experts": int((m.group_list > 0).sum()), "prequantised_input": m.x_scale is not None,
                "packed_weights": {"i8": "int8 only", "i8+f16": "int8 + integer-valued fp16 copy"}[self.pack],
                "seed": 0, "inputs": self.input_note}

    def value(self, units, seconds):
        return units / seconds

    def e2e_setup(self, device):
        torch = self.torch
        m = self.m
        if m.x_scale is None:
            self.hx = torch.from_numpy(m.x.view("int16")).view(torch.bfloat16).pin_memory()
            self.hxs = None
        else:
            self.hx = torch.from_numpy(m.x).pin_memory()
            self.hxs = torch.from_numpy(m.x_scale).pin_memory()
        self.hgl = torch.from_numpy(m.group_list).pin_memory()
        self.e2e_slots = [dict(x=torch.empty_like(self.x), xs=None if self.xs is None else torch.empty_like(self.xs),
                               gl=torch.empty_like(self.gl), y=torch.empty_like(self.y),
                               hy=torch.empty((m.R, m.H), dtype=torch.bfloat16).pin_memory())
                          for _ in range(E2E_SLOTS)]
        self.h2d = self.hx.numel() * self.hx.element_size() + (0 if self.hxs is None else self.hxs.numel() * 4) + \
            self.hgl.numel() * 8
        self.d2h = m.R * m.H * 2

    def e2e_in(self, slot):
        sl = self.e2e_slots[slot]
        sl["x"].copy_(self.hx, non_blocking=True)
        if self.hxs is not None:
            sl["xs"].copy_(self.hxs, non_blocking=True)
        sl["gl"].copy_(self.hgl, non_blocking=True)

    def e2e_compute(self, slot):
        sl = self.e2e_slots[slot]
        self.W.moe_w13_swiglu_requant_w2(sl["x"], sl["xs"], sl["gl"], self.w13p, self.s13, self.w2p, self.s2,
                                         self.ws, sl["y"])

    def e2e_out(self, slot):
        sl = self.e2e_slots[slot]
        sl["hy"].copy_(sl["y"], non_blocking=True)

    # CPU oracle on a subset of routed rows (tokens = rows / topk)
    def oracle_units(self, rows):
        return rows / self.m.topk

    def _subset(self, rows):
        """Host inputs of the compact problem made of `rows` evenly spaced routed rows."""
        cache = getattr(self, "_subset_cache", {})
        self._subset_cache = cache
        if rows not in cache:
            np = self.np
            m = self.m
            sel = np.unique(np.linspace(0, m.R - 1, rows).astype(np.int64))
            off = np.concatenate([[0], np.cumsum(m.group_list)])
            eor = np.searchsorted(off, sel, side="right") - 1
            experts = np.unique(eor)
            gl = np.array([int(np.sum(eor == e)) for e in experts], np.int64)
            idx = self.torch.as_tensor(experts, device=m.w13.device)
            cache[rows] = (m.x[sel], None if m.x_scale is None else m.x_scale[sel], gl,
                           m.w13.index_select(0, idx).cpu().numpy(), m.s13[experts],
                           m.w2.index_select(0, idx).cpu().numpy(), m.s2[experts])
        return cache[rows]

    def oracle_step(self, rows):
        import oracle
        oracle.moe_w13_swiglu_requant_w2(*self._subset(rows))

    @property
    def oracle_full_rows(self):
        return self.m.R


class MoETokens(MoE):
    """The MoE layer from token rows and router output: routing permute + quant -> the expert chain ->
    top-k weighted combine (one moe_layer call).  The permute and the combine are also timed alone,
    through their own calls, for their HBM rooflines."""

    def __init__(self, cfg_id: int, device, kernels=None, pack: str = "auto", scale: int = 1):
        # the routing kernels alone (profiling) need no packed weights
        super().__init__(cfg_id, device, pack_weights=kernels is None or "moe_layer" in kernels, pack=pack,
                         scale=scale)
        W, torch, m = self.W, self.torch, self.m
        T, k, H, I, E, R = m.T, m.topk, m.H, m.I, m.E, m.R
        self.name = m.name + "_from_tokens"
        if m.x_tok_scale is None:
            self.xt = torch.from_numpy(m.x_tok.view("int16")).to(device).view(torch.bfloat16)
            self.xts = None
        else:
            self.xt = torch.from_numpy(m.x_tok).to(device)
            self.xts = torch.from_numpy(m.x_tok_scale).to(device)
        self.ids = torch.from_numpy(m.topk_ids).to(device)
        self.tw = torch.from_numpy(m.topk_weights).to(device)
        self.lws = W.workspace(W.moe_layer_workspace_bytes(T, k, H, I, E), device)
        self.yt = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        # buffers of the permute and combine timed alone
        self.rws = W.workspace(W.moe_route_workspace_bytes(T, k, E), device)
        self.pq_out = (torch.empty((R, H), dtype=torch.int8, device=device),
                       torch.empty((R,), dtype=torch.float32, device=device),
                       torch.empty((E,), dtype=torch.int64, device=device),
                       torch.empty((T, k), dtype=torch.int32, device=device))
        self.cws = W.workspace(256, device)
        # inputs of the combine timed alone: seeded routed rows and the permute's row indices
        gen = torch.Generator(device=device)
        gen.manual_seed(cfg_id * 7919 + 1)
        self.yr = torch.randn((R, H), generator=gen, device=device).to(torch.bfloat16)
        self.yc = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        W.moe_permute_quant(self.xt, self.xts, self.ids, m.E, self.rws, out=self.pq_out)
        self.kernels = ["moe_layer", "moe_permute_quant", "moe_unpermute_combine"]
        self.step_kernels = ["moe_layer"]
        self.breakdown_reps = {"moe_permute_quant": 20, "moe_unpermute_combine": 20}
        if kernels is not None:  # profiling: only the named calls, each one a step
            self.kernels = [k for k in self.kernels if k in kernels]
            self.step_kernels = list(self.kernels)
        xin = T * H * (1 if m.x_tok_scale is not None else 2) + (4 * T if m.x_tok_scale is not None else 0)
        route = 8 * R + 4 * R + 8 * E  # ids read, routed row index written, group list
        permute = xin + route + R * H + 4 * R  # token rows in, int8 routed rows + scales out
        combine = 2 * R * H + 8 * R + 2 * T * H  # routed rows, weights and indices in, token rows out
        chain = self.alg_bytes["moe_layer"] - R * H * (1 if m.x_scale is not None else 2 + 1 + 1)
        # the layer: token rows in, routed codes written once and read by W13, chain, combine
        self.alg_bytes = {"moe_layer": xin + route + 2 * R * H + 4 * R + chain + combine,
                          "moe_permute_quant": permute, "moe_unpermute_combine": combine}
        route = 1 if R <= 8192 else 3  # one-CTA sort for decode-sized batches, else count / scan / assign
        per_call = {"moe_layer": route + 1 + 3 + 1,  # route, permute, W13 + requant + W2, combine
                    "moe_permute_quant": route + 1, "moe_unpermute_combine": 1}
        self.launches_per_step = sum(per_call[k] for k in self.step_kernels)
        if "moe_layer" not in self.step_kernels:
            self.bound = "hbm"

    def _call(self, kernel, xt, xts, ids, tw, y):
        W = self.W
        if kernel == "moe_layer":
            W.moe_layer(xt, xts, ids, tw, self.w13p, self.s13, self.w2p, self.s2, self.lws, y)
        elif kernel == "moe_permute_quant":
            W.moe_permute_quant(xt, xts, ids, self.m.E, self.rws, out=self.pq_out)
        else:
            W.moe_unpermute_combine(self.yr, self.pq_out[3], tw, self.cws, y)

    def launch(self, kernel: str, i: int):
        self._call(kernel, self.xt, self.xts, self.ids, self.tw, self.yt if kernel == "moe_layer" else self.yc)

    def config(self):
        c = super().config()
        c["workload"] = self.name
        c["input"] = "token rows [T,H] + top-k ids and weights [T,topk]"
        return c

    def e2e_setup(self, device):
        torch, m = self.torch, self.m
        if m.x_tok_scale is None:
            self.hx = torch.from_numpy(m.x_tok.view("int16")).view(torch.bfloat16).pin_memory()
            self.hxs = None
        else:
            self.hx = torch.from_numpy(m.x_tok).pin_memory()
            self.hxs = torch.from_numpy(m.x_tok_scale).pin_memory()
        self.hids = torch.from_numpy(m.topk_ids).pin_memory()
        self.htw = torch.from_numpy(m.topk_weights).pin_memory()
        self.e2e_slots = [dict(xt=torch.empty_like(self.xt), xts=None if self.xts is None else torch.empty_like(self.xts),
                               ids=torch.empty_like(self.ids), tw=torch.empty_like(self.tw),
                               y=torch.empty_like(self.yt),
                               hy=torch.empty((m.T, m.H), dtype=torch.bfloat16).pin_memory())
                          for _ in range(E2E_SLOTS)]
        self.h2d = self.hx.numel() * self.hx.element_size() + (0 if self.hxs is None else self.hxs.numel() * 4) + \
            self.hids.numel() * 8 + self.htw.numel() * 4
        self.d2h = m.T * m.H * 2

    def e2e_in(self, slot):
        sl = self.e2e_slots[slot]
        sl["xt"].copy_(self.hx, non_blocking=True)
        if self.hxs is not None:
            sl["xts"].copy_(self.hxs, non_blocking=True)
        sl["ids"].copy_(self.hids, non_blocking=True)
        sl["tw"].copy_(self.htw, non_blocking=True)

    def e2e_compute(self, slot):
        sl = self.e2e_slots[slot]
        for k in self.step_kernels:  # the layer, or the routing calls alone in profiling runs
            self._call(k, sl["xt"], sl["xts"], sl["ids"], sl["tw"], sl["y"])

    def e2e_out(self, slot):
        sl = self.e2e_slots[slot]
        sl["hy"].copy_(sl["y"], non_blocking=True)

    # CPU oracle on a subset of tokens (units = tokens)
    def oracle_units(self, rows):
        return rows

    def _token_subset(self, n):
        cache = getattr(self, "_tok_cache", {})
        self._tok_cache = cache
        if n not in cache:
            np, m = self.np, self.m
            toks = np.unique(np.linspace(0, m.T - 1, n).astype(np.int64))
            ids = m.topk_ids[toks]
            experts = np.unique(ids)
            idx = self.torch.as_tensor(experts, device=m.w13.device)
            cache[n] = (m.x_tok[toks], None if m.x_tok_scale is None else m.x_tok_scale[toks],
                        np.searchsorted(experts, ids).astype(np.int64), m.topk_weights[toks],
                        m.w13.index_select(0, idx).cpu().numpy(), m.s13[experts],
                        m.w2.index_select(0, idx).cpu().numpy(), m.s2[experts])
        return cache[n]

    def oracle_step(self, rows):
        import oracle
        oracle.moe_layer(*self._token_subset(rows))

    @property
    def oracle_full_rows(self):
        return self.m.T


class WeightPrep:
    """Offline weight quantisation (per output channel, symmetric INT8) from BF16, written straight into
    the packed buffers the contractions read: the workload's dense weight, or its W13 and W2 stacks."""

    def __init__(self, cfg_id: int, device, host_only: bool = False):
        import numpy as np
        import torch
        import w8a8_dynamic_quant_gb300 as W
        from w8a8_dynamic_quant_gb300 import synthetic as S
        self.W, self.torch, self.np = W, torch, np
        c = S.CONFIGS[cfg_id]
        if c["kind"] == "dense":
            f16 = W.PACK_F16 if c["M"] >= 128 else 0
            self.shapes = [(1, c["N"], c["K"], f16)]
        else:
            R, E, H, I = c["T"] * c["topk"], c["E"], c["H"], c["I"]
            f16 = W.PACK_F16 if R >= 64 * E else 0
            self.shapes = [(E, 2 * I, H, W.PACK_GATE_UP | f16), (E, H, I, f16)]
        self.name = "weight_quant_" + c["name"]
        self.n_sets = 1
        self.unit = "GB/s"
        self.bound = "hbm"
        self.kernels = ["quantize_prepack_weight"]
        nbytes = sum(E * N * K * (2 + 1 + (2 if f & W.PACK_F16 else 0)) + 4 * E * N for E, N, K, f in self.shapes)
        self.alg_bytes = {"quantize_prepack_weight": nbytes}
        self.alg_flops = {}
        self.units_per_step = float(nbytes)
        self.launches_per_step = 2 * len(self.shapes)  # quantise-and-pack, header
        self.channels = sum(E * N for E, N, _, _ in self.shapes)
        total_bf16 = sum(2 * E * N * K for E, N, K, _ in self.shapes)
        self.input_note = f"bf16 weights {total_bf16 / 1e9:.2f} GB > 129 MB L2 (single set)"
        self.step_rows = 256
        if host_only:
            return
        self.w = [S.make_bf16_weight(E, N, K, seed=i, device=str(device)) for i, (E, N, K, _) in enumerate(self.shapes)]
        self.packed = [torch.empty(W.prepacked_bytes(E, N, K, f), dtype=torch.uint8, device=device)
                       for E, N, K, f in self.shapes]
        self.scales = [torch.empty((E, N), dtype=torch.float32, device=device) for E, N, _, _ in self.shapes]

    def launch(self, kernel: str, i: int):
        for w, (_, _, _, f), p, sc in zip(self.w, self.shapes, self.packed, self.scales):
            self.W.w8a8_quantize_prepack_weight(w, f, p, sc)

    def config(self):
        return {"workload": self.name, "weights": [list(x[:3]) for x in self.shapes],
                "flags": [x[3] for x in self.shapes], "source": "bf16", "seed": 0, "inputs": self.input_note}

    def value(self, units, seconds):
        return units / seconds / 1e9

    # the packed weights stay on the device (where the contractions read them); the scales come back
    def e2e_setup(self, device):
        torch = self.torch
        self.hw = [w.cpu().pin_memory() for w in self.w]
        self.e2e_slots = [dict(w=[torch.empty_like(w) for w in self.w], sc=[torch.empty_like(x) for x in self.scales],
                               hs=[torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in self.scales])
                          for _ in range(E2E_SLOTS)]
        self.h2d = sum(w.numel() * 2 for w in self.hw)
        self.d2h = sum(x.numel() * 4 for x in self.scales)

    def e2e_in(self, slot):
        for w, hw in zip(self.e2e_slots[slot]["w"], self.hw):
            w.copy_(hw, non_blocking=True)

    def e2e_compute(self, slot):
        sl = self.e2e_slots[slot]
        for w, (_, _, _, f), p, sc in zip(sl["w"], self.shapes, self.packed, sl["sc"]):
            self.W.w8a8_quantize_prepack_weight(w, f, p, sc)

    def e2e_out(self, slot):
        sl = self.e2e_slots[slot]
        for sc, hs in zip(sl["sc"], sl["hs"]):
            hs.copy_(sc, non_blocking=True)

    # CPU oracle on `rows` output channels of the first weight (units: algorithmic bytes of those channels)
    def oracle_units(self, rows):
        E, N, K, f = self.shapes[0]
        return rows * (K * (2 + 1 + (2 if f & self.W.PACK_F16 else 0)) + 4)

    def oracle_step(self, rows):
        import oracle
        cache = getattr(self, "_host_cache", {})
        self._host_cache = cache
        if rows not in cache:
            from w8a8_dynamic_quant_gb300 import synthetic as S
            K = self.shapes[0][2]
            w = S.make_bf16_weight(1, rows, K, seed=0, device="cpu")
            cache[rows] = w.view(self.torch.int16).numpy().view(self.np.uint16)
        oracle.quantize_weight(cache[rows])

    @property
    def oracle_full_rows(self):
        return self.channels


def make_workload(cfg_id, device, from_tokens=False, kernels=None, prepare=False, static=False, mx=False,
                  pack="auto", moe_scale=1):
    from w8a8_dynamic_quant_gb300 import synthetic as S
    if prepare:
        return WeightPrep(cfg_id, device)
    if mx:
        return DenseMX(cfg_id, device)
    if S.CONFIGS[cfg_id]["kind"] == "dense":
        return DenseStatic(cfg_id, device) if static else Dense(cfg_id, device, pack)
    return (MoETokens(cfg_id, device, kernels, pack, moe_scale) if from_tokens
            else MoE(cfg_id, device, pack=pack, scale=moe_scale))


# -------------------------------------------------------------- the arms --

def cpu_model() -> str:
    """The host CPU's model as the kernel reports it (x86: "model name"; Arm: implementer and part)."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    fields = {}
    for ln in info.splitlines():
        if ":" in ln:
            k, v = ln.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    arm_parts = {"0xd4f": "Neoverse V2", "0xd40": "Neoverse V1", "0xd0c": "Neoverse N1", "0xd49": "Neoverse N2"}
    part = fields.get("CPU part", "")
    if part:
        return f"{arm_parts.get(part, 'Arm')} (implementer {fields.get('CPU implementer', '?')}, part {part})"
    return "unknown"


def time_oracle(wl, budget_s: float, max_rows=None):
    """Time the CPU oracle on row samples of the workload for about budget_s seconds."""
    import oracle
    rows = wl.oracle_full_rows if max_rows is None else min(max_rows, wl.oracle_full_rows)
    t0 = time.perf_counter()
    wl.oracle_step(rows)
    t1 = time.perf_counter() - t0
    # shrink the sample if one full step is longer than the budget
    while t1 > budget_s and rows > 1:
        rows = max(1, rows // 4)
        t0 = time.perf_counter()
        wl.oracle_step(rows)
        t1 = time.perf_counter() - t0
    reps, total = 1, t1
    while total < budget_s:
        t0 = time.perf_counter()
        wl.oracle_step(rows)
        total += time.perf_counter() - t0
        reps += 1
    units = wl.oracle_units(rows) * reps
    return {"value": wl.value(units, total), "unit": wl.unit, "cores": oracle.num_threads(), "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"{reps} run(s) of {rows} of {wl.oracle_full_rows} rows, {total:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch  # noqa: F401
    import oracle  # noqa: F401
    from w8a8_dynamic_quant_gb300 import synthetic as S
    # the oracle arm needs only host data: build the workload's host side on the CPU
    if args.prepare:
        wl = WeightPrep(args.workload, "cpu", host_only=True)
    elif S.CONFIGS[args.workload]["kind"] == "dense":
        wl = (_HostDenseStatic(args.workload) if args.static else
              _HostDenseMX(args.workload) if args.mx else _HostDense(args.workload))
    else:
        wl = _HostMoETokens(args.workload) if args.from_tokens else _HostMoE(args.workload)
    for _ in range(args.warmup):
        wl.oracle_step(wl.step_rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        wl.oracle_step(wl.step_rows)
    dt = time.perf_counter() - t0
    units = wl.oracle_units(wl.step_rows) * args.steps
    value = wl.value(units, dt)
    cores = oracle.num_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": wl.unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic", "config": wl.config(),
            "cpu_baseline": {"value": value, "unit": wl.unit, "cores": cores, "kind": "oracle", "cpu": cpu_model(),
                             "sample": f"{wl.step_rows} of {wl.oracle_full_rows} rows per step"},
            "e2e": {"value": value, "unit": wl.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


class _HostDense(Dense):
    def __init__(self, cfg_id):
        from w8a8_dynamic_quant_gb300 import synthetic as S
        self.d = S.dense_config(cfg_id)
        self.name = self.d.name
        self.M, self.N, self.K = self.d.M, self.d.N, self.d.K
        self.pack = "i8+f16" if self.M >= 128 else "i8"  # the GPU arm's default layout, named in config
        self.unit = "TOPS"
        self.input_note = "host arrays (CPU oracle)"
        # about 0.1-0.5 s of CPU per step on 16 cores
        self.step_rows = max(1, min(self.M, int(2e9 // (2 * self.N * self.K))))


class _HostDenseStatic(DenseStatic):
    def __init__(self, cfg_id):
        from w8a8_dynamic_quant_gb300 import synthetic as S
        _HostDense.__init__(self, cfg_id)
        self.s_in, self.o_in = S.static_params(cfg_id)
        self.name = self.d.name + "_static"


class _HostDenseMX(DenseMX):
    def __init__(self, cfg_id):
        _HostDense.__init__(self, cfg_id)
        self.name = self.d.name + "_mxfp8"
        self.step_rows = max(1, self.step_rows // 8)  # the float64 MX oracle is slower per row


class _HostMoE(MoE):
    def __init__(self, cfg_id):
        import numpy as np
        import torch
        from w8a8_dynamic_quant_gb300 import synthetic as S
        self.np, self.torch = np, torch
        self.m = S.moe_config(cfg_id, device="cpu")
        self.name = self.m.name
        self.pack = "i8+f16" if self.m.R >= 64 * self.m.E else "i8"  # the GPU arm's default layout
        self.unit = "tokens/s"
        self.input_note = "host arrays (CPU oracle)"
        self.step_rows = 8


class _HostMoETokens(MoETokens):
    def __init__(self, cfg_id):
        import numpy as np
        import torch
        from w8a8_dynamic_quant_gb300 import synthetic as S
        self.np, self.torch = np, torch
        self.m = S.moe_config(cfg_id, device="cpu")
        self.name = self.m.name + "_from_tokens"
        self.pack = "i8+f16" if self.m.R >= 64 * self.m.E else "i8"  # the GPU arm's default layout
        self.unit = "tokens/s"
        self.input_note = "host arrays (CPU oracle)"
        self.step_rows = 1  # tokens (each with topk routed rows)


def int8_tensor_reference(torch, device, n: int = 8192, reps: int = 5):
    """Throughput of the INT8 tensor-core path the libraries expose (torch._int_mm: cuBLASLt INT8 x INT8 ->
    INT32) on an n^3 GEMM, best of `reps`, in TOPS.  The library's exact engines feed integer-valued FP16 to
    the FP16 tensor instruction instead (sm_103a has no integer tcgen05 kind), so this is the INT8 rate the
    metric's "% INT8 peak" refers to, not the roof of those engines."""
    try:
        a = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=device)
        b = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=device).t()
        torch._int_mm(a, b)
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._int_mm(a, b)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        del a, b
        return {"tops": 2.0 * n ** 3 / (best / 1e3) / 1e12, "how": f"torch._int_mm int8 {n}^3, best of {reps}"}
    except Exception as e:  # an INT8 library path the installed torch lacks
        return {"tops": None, "how": f"unavailable: {type(e).__name__}"}


def run_gpu(args):
    import torch
    import torch.distributed as dist

    rank, world, local_rank = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    import __graft_entry__
    __graft_entry__.build()
    peaks = load_peaks()
    kernels = args.kernels.split(",") if args.kernels else None
    wl = make_workload(args.workload, device, args.from_tokens, kernels, args.prepare, args.static, args.mx,
                       args.pack, args.moe_scale)
    step_kernels = getattr(wl, "step_kernels", wl.kernels)
    stream = torch.cuda.current_stream(device)

    # one CUDA graph per kernel type over all rotating input sets
    graphs = {}
    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for k in wl.kernels:
            for i in range(wl.n_sets):
                wl.launch(k, i)  # warm the launch path before capture
    stream.wait_stream(side)
    torch.cuda.synchronize()
    # a short kernel is captured several times per breakdown graph, so the graph's own launch cost
    # is spread over the launches
    reps = {k: getattr(wl, "breakdown_reps", {}).get(k, 1) for k in wl.kernels}
    for k in wl.kernels:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps[k]):
                for i in range(wl.n_sets):
                    wl.launch(k, i)
        graphs[k] = g
    # a whole rotation over the input sets in one graph, and one graph per set for a single step
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph):
        for i in range(wl.n_sets):
            for k in step_kernels:
                wl.launch(k, i)
    one_graphs = []
    if wl.n_sets > 1:
        for i in range(wl.n_sets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for k in step_kernels:
                    wl.launch(k, i)
            one_graphs.append(g)
    torch.cuda.synchronize()

    def run_steps(n):
        """Exactly n steps: whole rotations, then single steps on the next sets."""
        for _ in range(n // wl.n_sets):
            step_graph.replay()
        for i in range(n % wl.n_sets):
            one_graphs[i].replay()

    run_steps(args.warmup)
    steps = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t_wall0 = time.perf_counter()
        ev0.record(stream)
        run_steps(steps)
        ev1.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
        # keep the GPU loaded long enough for the clock sampler to see it
        extra = 0
        while not args.quick and time.perf_counter() - t_wall0 < 1.0 and extra < 100000:
            step_graph.replay()
            extra += 1
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = clk.summary()
    step_ms = ev0.elapsed_time(ev1) / steps
    rounds = max(1, -(-steps // wl.n_sets))

    # per-kernel breakdown: each kernel type alone over the same sets (outside the timed region)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(wl.kernels) + 1)] for _ in range(rounds)]
    for r in range(rounds):
        for j, k in enumerate(wl.kernels):
            kev[r][j].record(stream)
            graphs[k].replay()
        kev[r][-1].record(stream)
    torch.cuda.synchronize()
    per_kernel_ms = {k: sum(kev[r][j].elapsed_time(kev[r][j + 1]) for r in range(rounds)) / (steps * reps[k])
                     for j, k in enumerate(wl.kernels)}
    units, seconds = aggregate(wl.units_per_step * steps, step_ms * steps / 1e3)
    value = wl.value(units, seconds)

    # e2e through the public API with host buffers
    wl.e2e_setup(device)
    run_e2e(torch, wl, 3)
    e2e_steps = 3 if args.quick else max(3, min(args.steps, 200))
    t0 = time.perf_counter()
    run_e2e(torch, wl, e2e_steps)
    e2e_s = time.perf_counter() - t0
    e_units, e_seconds = aggregate(wl.units_per_step * e2e_steps, e2e_s)

    # dominant kernel roofline
    dom = max(step_kernels, key=per_kernel_ms.get)
    dur_s = per_kernel_ms[dom] / 1e3
    if wl.bound == "hbm":
        achieved = wl.alg_bytes[dom] / dur_s / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
    else:
        achieved = wl.alg_flops[dom] / dur_s / 1e12
        peak, unit = peaks["bf16_tflops"] * getattr(wl, "tensor_peak_ratio", 1.0), "TFLOP/s"
    traffic = recorded_traffic(dom, traffic_key(wl))
    roofline = {"bound": wl.bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                "traffic": traffic, "kernel": dom, "peak_source": (f"{peaks['source']} (MEASURED_PEAKS.json)"
                if peaks["source"] == "measured" else "fallback") +
                (f" x {wl.tensor_peak_ratio:g} (nominal FP8/BF16 ratio)" if getattr(wl, "tensor_peak_ratio", 1.0) != 1.0
                 and wl.bound == "tensor" else ""),
                "alg_bytes_per_launch": wl.alg_bytes[dom],
                "per_kernel_us": {k: v * 1e3 for k, v in per_kernel_ms.items()},
                "sum_of_kernels_us": sum(per_kernel_ms[k] for k in step_kernels) * 1e3}
    if wl.bound == "tensor" and not args.quick:
        # the metric's "% INT8 peak": the INT8 tensor-core path of the libraries on this GPU, measured here
        int8 = int8_tensor_reference(torch, device)
        roofline["int8_reference"] = int8
        if int8.get("tops"):
            roofline["frac_of_int8_reference"] = achieved / int8["tops"]
    if "dynamic_quant" in per_kernel_ms:
        roofline["quant_gbs"] = wl.alg_bytes["dynamic_quant"] / (per_kernel_ms["dynamic_quant"] / 1e3) / 1e9
    if dom in wl.alg_flops:
        roofline["tops_dominant"] = wl.alg_flops[dom] / dur_s / 1e12
    # the routing kernels timed alone (HBM-bound)
    for k in wl.kernels:
        if k in step_kernels:
            continue
        gbs = wl.alg_bytes[k] / (per_kernel_ms[k] / 1e3) / 1e9
        roofline.setdefault("others", {})[k] = {"us": per_kernel_ms[k] * 1e3, "alg_bytes": wl.alg_bytes[k],
                                                "achieved_gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"]}

    line = {"metric": METRIC, "value": value, "unit": wl.unit, "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8", "data": "synthetic", "config": wl.config(),
            "roofline": roofline, "clocks": clocks, "gpu_launches": steps * wl.launches_per_step,
            "e2e": {"value": wl.value(e_units, e_seconds), "unit": wl.unit, "h2d_bytes_per_step": wl.h2d,
                    "d2h_bytes_per_step": wl.d2h, "steps": e2e_steps, "pipeline": E2E_PIPELINE},
            "wall_s_timed_region": t_wall}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle(wl, args.cpu_budget)
    elif rank == 0:
        line["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", type=int, default=4, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--pack", default="auto", choices=["auto", "i8", "i8+f16"],
                    help="packed weight layout: INT8 only, or INT8 plus the integer-valued FP16 copy the fastest "
                         "large-M engines read (auto: the copy for prefill-sized shapes)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of CPU oracle timing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--from-tokens", action="store_true",
                    help="MoE workloads: the layer from token rows and router output (routing permute + quant, "
                         "expert chain, top-k weighted combine) instead of expert-sorted routed rows")
    ap.add_argument("--static", action="store_true",
                    help="dense workloads: the static W8A8 variant (fixed input scale and offset, load-time "
                         "deq_scale and quant_bias)")
    ap.add_argument("--mx", action="store_true",
                    help="dense workloads: the MXFP8 variant (E4M3 + E8M0 per 32 along K, weights converted at load)")
    ap.add_argument("--prepare", action="store_true",
                    help="time the load-time weight preparation instead: the workload's weights quantised per "
                         "channel from BF16 and packed in one pass (GB/s)")
    ap.add_argument("--kernels", default=None,
                    help="with --from-tokens: time only these calls (comma list of moe_layer, moe_permute_quant, "
                         "moe_unpermute_combine), for profiler captures")
    ap.add_argument("--quick", action="store_true",
                    help="short run for profiler captures: no clock-sampling hold, 3 e2e steps")
    ap.add_argument("--moe-scale", type=int, default=1,
                    help="MoE workloads: T and E divided by this, a small case of the same kernels for "
                         "profiler captures that collect many metrics (not a bench line)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
