"""Benchmark of the FP8 / MXFP8 quantization hot path on one node.

Default workload (the largest single-GPU configuration): MoE expert
activations, 65536 x 7168 BF16 (Student-t, nu = 4), rows split over 64
experts by multinomial token counts.  One step quantizes that tensor, per
expert, in both ways the path has:
  * mxfp8_quantize, grouped, E4M3, rowwise + columnwise
                         (2 + 1 + 1 + 1/32 B/element + the column scales)
  * fp8q_cast_per_tensor, grouped current scaling, E4M3
                         (5 B/element: amax read, cast read + write)
Both ops read the same device tensor.

value: bytes read + written by the step's kernels, summed over all ranks,
divided by the max over ranks of the device time of K steps (GB/s).
roofline: the step's dominant kernel (the grouped MXFP8 kernel) timed alone
in a loop of at least 100 back-to-back launches, CUDA events around the
loop, against the measured HBM copy bandwidth.  Every op of the step is
timed the same way (`ops`).
per_config: the other four configurations, each measured the same way
(per-tensor current scaling of 1024 x 1024; MXFP8 of a 4096 x 4096
activation; 32 drifting steps of an 8192 x 8192 tensor under delayed
scaling, both formats, Interval 1 and 5, next to current scaling, with a
per-step table of scale, amax, saturation, SQNR and zero-rate; one 8B-class
linear layer's A, W and E in MXFP8).

--workload selects another workload as the headline (same line format):
  moe (default), per_tensor_1024, mx_4096, delayed_8192, linear_layer,
  activation (MXFP8 + current + delayed on one 4096 x 4096 activation),
  mx_8192, dequant_8192, mx_rules_4096, blockwise_8192, nvfp4_8192,
  qstats_8192, mxfp4_fp6_8192, mma_scales_8192.
--impl reference: the CPU oracle on this host (a bounded sample per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "quantize GB/s (bytes read+written) and % of GB300 HBM peak, bit-exact"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20
ROOFLINE_MIN_LAUNCHES = 100
E4M3, E5M2 = 0, 1
WORKLOADS = ["moe", "moe_16384", "per_tensor_1024", "mx_4096", "delayed_8192", "linear_layer", "activation", "mx_8192",
             "mx_mma_8192",
             "dequant_8192", "mx_rules_4096", "blockwise_8192", "nvfp4_8192", "qstats_8192", "mxfp4_fp6_8192",
             "mma_scales_8192"]
# the configurations measured beside the headline, by name
PER_CONFIG = (("c1", "per_tensor_1024"), ("c2", "mx_4096"), ("c3", "delayed_8192"), ("c4", "linear_layer"))
C3_STEPS = 32


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="moe", choices=WORKLOADS)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-config", action="store_true", help="measure the headline workload only")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--cpu-leg", default=None, help=argparse.SUPPRESS)  # internal: one oracle timing leg
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# workloads: shapes, algorithmic bytes, inputs
# ---------------------------------------------------------------------------
def mx_bytes(rows, cols, ncolblocks=None):
    ncb = (rows + 31) // 32 if ncolblocks is None else ncolblocks
    return rows * cols * 2 + rows * cols + rows * (cols // 32) + cols * rows + cols * ncb


def workload_spec(name):
    """(config dict, list of ops).  An op is a dict with its 'kind', tensor
    shape, format, algorithmic bytes per call and the input it reads
    ('gen': ops with the same gen read the same device tensor)."""
    if name == "moe":
        r, c = 65536, 7168
        ops = [{"kind": "mx_grouped", "shape": (r, c), "fmt": E4M3, "bytes": None, "gen": ("c5", 0)},
               {"kind": "current_grouped", "shape": (r, c), "fmt": E4M3, "bytes": 5 * r * c, "gen": ("c5", 0)}]
        return {"workload": "moe_64_experts_65536x7168_bf16", "rows": r, "cols": c, "experts": 64,
                "ops": ["grouped mxfp8 e4m3 row+col", "grouped current scaling e4m3"]}, ops
    if name == "moe_16384":
        r, c = 16384, 7168
        ops = [{"kind": "mx_grouped", "shape": (r, c), "fmt": E4M3, "bytes": None, "gen": ("c5", 0)},
               {"kind": "current_grouped", "shape": (r, c), "fmt": E4M3, "bytes": 5 * r * c, "gen": ("c5", 0)}]
        return {"workload": "moe_16_experts_16384x7168_bf16", "rows": r, "cols": c, "experts": 16,
                "ops": ["grouped mxfp8 e4m3 row+col", "grouped current scaling e4m3"]}, ops
    if name == "per_tensor_1024":
        ops = [{"kind": "current", "shape": (1024, 1024), "fmt": E4M3, "bytes": 5 * 1024 * 1024, "gen": ("c1", 0)}]
        return {"workload": "per_tensor_current_1024x1024_bf16", "rows": 1024, "cols": 1024,
                "ops": ["current scaling e4m3"]}, ops
    if name == "mx_4096":
        r = c = 4096
        ops = [{"kind": "mx", "shape": (r, c), "fmt": E4M3, "bytes": mx_bytes(r, c), "gen": ("c2", 0)}]
        return {"workload": "mxfp8_activation_4096x4096_bf16", "rows": r, "cols": c,
                "ops": ["mxfp8 e4m3 row+col"]}, ops
    if name == "delayed_8192":
        r = c = 8192
        ops = []
        for fmt in (E4M3, E5M2):
            for interval in (1, 5):
                ops.append({"kind": "delayed", "interval": interval, "shape": (r, c), "fmt": fmt,
                            "bytes": 3 * r * c + 4 * 16, "gen": ("c3seq", 0)})
        for fmt in (E4M3, E5M2):
            ops.append({"kind": "current", "shape": (r, c), "fmt": fmt, "bytes": 5 * r * c, "gen": ("c3seq", 0)})
        return {"workload": "delayed_drift_32x8192x8192_bf16", "rows": r, "cols": c, "sequence_steps": C3_STEPS,
                "ops": ["delayed e4m3 H16 margin3 interval1", "delayed e4m3 H16 margin3 interval5",
                        "delayed e5m2 H16 margin3 interval1", "delayed e5m2 H16 margin3 interval5",
                        "current scaling e4m3", "current scaling e5m2"],
                "input": "step i reads x_t, t = i mod 32, sigma_{t+1} = sigma_t * U(0.8, 1.25)"}, ops
    if name == "linear_layer":
        shapes = {"A": (16384, 4096), "W": (14336, 4096), "E": (16384, 14336)}
        ops = [{"kind": "mx", "shape": shapes[k], "fmt": E5M2 if k == "E" else E4M3,
                "bytes": mx_bytes(*shapes[k]), "gen": ("c4", k)} for k in ("A", "W", "E")]
        return {"workload": "linear_layer_8b_mxfp8", "A": "16384x4096", "W": "14336x4096",
                "E": "16384x14336", "ops": ["A mxfp8 e4m3 row+col", "W mxfp8 e4m3 row+col",
                                            "E mxfp8 e5m2 row+col"]}, ops
    if name == "activation":
        r = c = 4096
        ops = [{"kind": "mx", "shape": (r, c), "fmt": E4M3, "bytes": mx_bytes(r, c), "gen": ("c2", 0)},
               {"kind": "current", "shape": (r, c), "fmt": E4M3, "bytes": 5 * r * c, "gen": ("c2", 1)},
               {"kind": "delayed", "interval": 1, "shape": (r, c), "fmt": E4M3, "bytes": 3 * r * c + 4 * 16,
                "gen": ("c2", 2)}]
        cfg = {"workload": "activation_4096x4096_bf16", "rows": r, "cols": c,
               "ops": ["mxfp8 e4m3 row+col", "current scaling e4m3", "delayed e4m3 H16 margin3 interval1"]}
        return cfg, ops
    if name == "mx_8192":
        r = c = 8192
        ops = [{"kind": "mx", "shape": (r, c), "fmt": E4M3, "bytes": mx_bytes(r, c), "gen": ("c2", 0)}]
        return {"workload": "mxfp8_8192x8192_bf16", "rows": r, "cols": c, "ops": ["mxfp8 e4m3 row+col"]}, ops
    if name == "mx_mma_8192":
        r = c = 8192
        ops = [{"kind": "mx_mma", "shape": (r, c), "fmt": E4M3, "bytes": mx_bytes(r, c), "gen": ("c2", 0)}]
        return {"workload": "mxfp8_mma_scales_8192x8192_bf16", "rows": r, "cols": c,
                "ops": ["mxfp8 e4m3 row+col, scales written in the 128x4 MMA block layout"]}, ops
    if name == "mx_rules_4096":
        r = c = 4096
        ops = [{"kind": "mx_rule", "rule": 0, "shape": (r, c), "fmt": E4M3, "bytes": mx_bytes(r, c), "gen": ("c2", 0)},
               {"kind": "mx_rule", "rule": 1, "shape": (r, c), "fmt": E4M3, "bytes": mx_bytes(r, c), "gen": ("c2", 0)}]
        return {"workload": "mxfp8_scale_rules_4096x4096_bf16", "rows": r, "cols": c,
                "ops": ["mxfp8 e4m3 row+col, round-up rule, saturation counted",
                        "mxfp8 e4m3 row+col, OCP rule, saturation counted"]}, ops
    if name == "blockwise_8192":
        r = c = 8192
        ops = [{"kind": "bw", "block": 1, "shape": (r, c), "fmt": E4M3,
                "bytes": 4 * r * c + 4 * (r * (c // 128) + c * (r // 128)), "gen": ("c2", 0)},
               {"kind": "bw", "block": 128, "shape": (r, c), "fmt": E4M3, "bytes": 4 * r * c + 8 * (r // 128) * (c // 128),
                "gen": ("c4", "W")}]
        return {"workload": "blockwise_fp8_8192x8192_bf16", "rows": r, "cols": c,
                "ops": ["1x128 + 128x1 groups (activation), both copies", "128x128 blocks (weight), both copies"]}, ops
    if name == "nvfp4_8192":
        r = c = 8192
        ops = [{"kind": "nvfp4", "shape": (r, c), "fmt": E4M3, "bytes": 4 * r * c + r * c // 2 + r * c // 16 + 8,
                "gen": ("c2", 0)}]
        return {"workload": "nvfp4_8192x8192_bf16", "rows": r, "cols": c,
                "ops": ["nvfp4: tensor amax, then E2M1 codes and E4M3 scales per 16"]}, ops
    if name == "mma_scales_8192":
        r = c = 8192
        nb = r * (c // 32)  # scale bytes of one MX copy; 8192 is a multiple of 128 rows and 4 columns
        ops = [{"kind": "mmascale", "copy": "s_row", "shape": (r, c), "fmt": E4M3, "bytes": 2 * nb, "gen": ("c2", 0)},
               {"kind": "mmascale", "copy": "s_col", "shape": (r, c), "fmt": E4M3, "bytes": 2 * nb, "gen": ("c2", 0)}]
        return {"workload": "mma_scale_layout_8192x8192", "rows": r, "cols": c,
                "ops": ["rowwise mx scales [8192][256] -> 128x4 blocks",
                        "columnwise mx scales [8192][256] -> 128x4 blocks"]}, ops
    if name == "mxfp4_fp6_8192":
        r = c = 8192
        ops = [{"kind": "mxlow", "elem": 2, "shape": (r, c), "fmt": E4M3, "bytes": 3 * r * c + r * c // 16,
                "gen": ("c2", 0)},
               {"kind": "mxlow", "elem": 3, "shape": (r, c), "fmt": E4M3, "bytes": 4 * r * c + r * c // 16,
                "gen": ("c2", 0)}]
        return {"workload": "mxfp4_mxfp6_8192x8192_bf16", "rows": r, "cols": c,
                "ops": ["mxfp4 (e2m1) row+col, round-up rule", "mxfp6 (e2m3) row+col, round-up rule"]}, ops
    if name == "qstats_8192":
        r = c = 8192
        ops = [{"kind": "qs_mx_row", "shape": (r, c), "fmt": E4M3, "bytes": 3 * r * c + r * c // 32 + 64,
                "gen": ("c2", 0)},
               {"kind": "qs_mx_col", "shape": (r, c), "fmt": E4M3, "bytes": 3 * r * c + c * (r // 32) + 64,
                "gen": ("c2", 0)},
               {"kind": "qs_tensor", "shape": (r, c), "fmt": E4M3, "bytes": 3 * r * c + 4 + 64, "gen": ("c2", 0)}]
        return {"workload": "qstats_8192x8192_bf16", "rows": r, "cols": c,
                "ops": ["sqnr/zero-rate of the mxfp8 e4m3 rowwise copy", "... of the columnwise copy",
                        "... of the per-tensor e4m3 copy"]}, ops
    if name == "dequant_8192":
        r = c = 8192
        ops = [{"kind": "dq_mx_row", "shape": (r, c), "fmt": E4M3, "bytes": 3 * r * c + r * c // 32, "gen": ("c2", 0)},
               {"kind": "dq_mx_col", "shape": (r, c), "fmt": E4M3, "bytes": 3 * r * c + c * (r // 32), "gen": ("c2", 0)},
               {"kind": "dq_tensor", "shape": (r, c), "fmt": E4M3, "bytes": 3 * r * c + 4, "gen": ("c2", 1)}]
        return {"workload": "dequantize_8192x8192_to_bf16", "rows": r, "cols": c,
                "ops": ["mxfp8 e4m3 rowwise copy -> bf16", "mxfp8 e4m3 columnwise copy -> bf16",
                        "per-tensor e4m3 -> bf16"]}, ops
    raise ValueError(name)


DQ_KINDS = ("dq_mx_row", "dq_mx_col", "dq_tensor")
QS_KINDS = ("qs_mx_row", "qs_mx_col", "qs_tensor")
ROOFLINE_KINDS = ("mx", "mx_grouped", "mx_mma", "dq_mx_row", "mx_rule", "bw", "nvfp4", "qs_mx_row", "mxlow", "mmascale",
                  "delayed")
LOW_NAMES = {2: "e2m1", 3: "e2m3", 4: "e3m2"}


def host_input(gen, shape, t=0):
    """The seeded BF16 input of `gen` (numpy uint16 bits); t selects the
    step of a drifting sequence."""
    import synth
    kind, idx = gen
    if kind == "c2":
        return synth.config2(*shape, seed=2 + 100 * idx)
    if kind == "c1":
        return synth.config1(*shape, seed=1)
    if kind == "c3seq":
        return synth.config3_step(t, *shape, seed=3, steps=C3_STEPS)
    if kind == "c4":
        t = {"A": lambda: synth.normal_outliers(*shape, seed=4, std=0.02, p=0.0005, factor=50.0, tensor=1),
             "W": lambda: synth.normal_outliers(*shape, seed=4, std=0.02, p=0.0005, factor=50.0, tensor=2),
             "E": lambda: synth.student_t(*shape, 3.0, seed=4, scale=1e-4, tensor=3)}
        return t[idx]()
    if kind == "c5":
        return synth.student_t(*shape, 4.0, seed=5)
    raise ValueError(kind)


def current_label(op, fmt_name):
    """The kernel(s) of an ungrouped current-scaling call on a BF16 tensor of
    op's shape: one cluster up to 2 MB, one launch up to the single-launch
    limit, else the amax and the cast kernel."""
    r, c = op["shape"]
    if 2 * r * c <= 16 * 128 * 1024:
        return f"current_cluster_kernel<bf16,{fmt_name}>"
    if r * c <= current_one_launch_elems():
        return f"current_fused_kernel<bf16,{fmt_name}>"
    return f"amax_kernel + cast_kernel<bf16,{fmt_name}>"


def kernel_label(op):
    fmt_name = "e4m3" if op["fmt"] == E4M3 else "e5m2"
    if op["kind"] == "current":
        return current_label(op, fmt_name)
    return {"dq_mx_row": f"dequant_kernel<mx_row,{fmt_name},bf16>",
            "dq_mx_col": f"dequant_kernel<mx_col,{fmt_name},bf16>",
            "dq_tensor": f"dequant_kernel<tensor,{fmt_name},bf16>",
            "mx_rule": f"mx_lean_kernel<bf16,{fmt_name},both,rule+counts>",
            "mx_mma": f"mx_tma_kernel<bf16,{fmt_name},both> (MMA scale layout)",
            "mx_grouped": f"mx_band_kernel<bf16,{fmt_name},both> ({op.get('G')} groups)",
            "bw": f"blockwise_kernel<{fmt_name},{'1x128' if op.get('block') == 1 else '128x128'},both>",
            "nvfp4": "amax_kernel + nvfp4_kernel<bf16>",
            "qs_mx_row": f"qstats_lin_kernel<bf16,{fmt_name},mx_row>",
            "qs_mx_col": f"qstats_col_tma_kernel<bf16,{fmt_name}>",
            "qs_tensor": f"qstats_lin_kernel<bf16,{fmt_name},tensor>",
            "mxlow": f"mxlow_tma_kernel<{LOW_NAMES.get(op.get('elem'), '')},both>",
            "mmascale": "mma_scale_kernel",
            "current": f"amax_kernel + cast_kernel<bf16,{fmt_name}>",
            "current_grouped": f"amax_kernel + cast_kernel<bf16,{fmt_name}> ({op.get('G')} groups)",
            "delayed": f"cast_kernel<bf16,{fmt_name},history> (interval {op.get('interval')})",
            }.get(op["kind"], f"mx_lean_kernel<bf16,{fmt_name},both>")


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# the files whose text compiles into the MXFP8 kernel (internal.h holds only
# host-side declarations of all launchers and is left out)
MX_SOURCES = ("mxfp8_quantization_amax_gb300/csrc/mxfp8.cu", "mxfp8_quantization_amax_gb300/csrc/fp8q_device.cuh",
              "mxfp8_quantization_amax_gb300/csrc/tma.cuh")


def sources_sha(paths=MX_SOURCES):
    """First 16 hex digits of the sha256 of the kernel's source files, in order."""
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_traffic(workload):
    """DRAM bytes per launch of the workload's roofline kernel from the
    committed ncu summary (profiles/traffic.txt: one `key=value ...` line per
    workload; `sources=a,b,...` names the files whose hash keys it, the
    MXFP8 kernel's by default), or None if there is none or those sources
    changed since.  Returns (bytes, the line's other fields)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            lines = [ln.split() for ln in f if ln.startswith("workload=")]
        for toks in lines:
            d = dict(t.split("=", 1) for t in toks if "=" in t)
            if d.get("workload") != workload:
                continue
            paths = tuple(d["sources"].split(",")) if "sources" in d else MX_SOURCES
            if d.get("sha") == sources_sha(paths):
                return int(d["bytes_per_launch"]), d
    except OSError:
        return None, None
    return None, None


def max_over_ranks(value, world, device=None):
    """The largest of every rank's `value` (a float); itself when world == 1."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_step, world, ms_per_step):
    """Whole-job GB/s: every rank moves bytes_per_step each step; the job's
    step time is the slowest rank's."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# our arm: one workload prepared on the device
# ---------------------------------------------------------------------------
class Prepared:
    """A workload's device buffers and its ops' C-ABI calls, argument tuples
    built once so that the host enqueues a step in a few microseconds.

    Input sets rotate (so an input is out of L2 when it is read again), and
    so do output sets; a drifting sequence has one input set per step."""

    def __init__(self, name, dev, min_sets=1):
        import torch

        import mxfp8_quantization_amax_gb300 as fq
        import synth
        self.name, self.dev, self.fq = name, dev, fq
        self.cfg, self.ops = workload_spec(name)
        ops = self.ops
        self.offsets_host = None
        if name in ("moe", "moe_16384"):
            rows, self.G = self.ops[0]["shape"][0], self.cfg["experts"]
            self.offsets_host = synth.moe_offsets(rows, self.G, seed=5)
            o = self.offsets_host
            self.ncb = int(sum((int(o[g + 1] - o[g]) + 31) // 32 for g in range(self.G)))
            for op in ops:
                op["G"] = self.G
                if op["kind"] == "mx_grouped":
                    op["bytes"] = mx_bytes(*op["shape"], ncolblocks=self.ncb)
        self.bytes_per_step = sum(op["bytes"] for op in ops)
        gens = []
        for op in ops:
            if (op["gen"], op["shape"]) not in gens:
                gens.append((op["gen"], op["shape"]))
        seq = any(g[0][0] == "c3seq" for g in gens)
        in_bytes = sum(2 * int(np.prod(s)) for _, s in gens)
        out_bytes = sum(op["bytes"] - 2 * int(np.prod(op["shape"])) for op in ops)
        per_set = in_bytes + max(out_bytes, 0)
        n_rot = max(min_sets, min(64, -(-4 * L2_BYTES // per_set)))
        self.n_in = C3_STEPS if seq else n_rot
        self.n_out = n_rot
        self.nsets = max(self.n_in, self.n_out)
        self.l2_note = (f"{self.n_in} input set(s) and {self.n_out} output set(s) rotating; "
                        f"{per_set / 2 ** 20:.0f} MiB per set (> 4x L2 in total, or inputs larger than L2)")

        # inputs: input set s holds every distinct gen (a drifting sequence
        # draws x_t for set t; otherwise the sets are copies of set 0)
        self.in_sets = []
        for s in range(self.n_in):
            d = {}
            for gen, shape in gens:
                if s == 0 or seq:
                    h = host_input(gen, shape, t=s)
                    d[gen] = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev)
                else:
                    d[gen] = self.in_sets[0][gen].clone()
            self.in_sets.append(d)
        self.off_dev = None if self.offsets_host is None else torch.from_numpy(self.offsets_host).to(dev)

        lib = fq.lib()
        self.lib = lib
        stream = torch.cuda.current_stream().cuda_stream
        off_ptr = None if self.off_dev is None else self.off_dev.data_ptr()
        self.states = [fq.DelayedScaling(16, op["interval"], 3, op["fmt"]) if op["kind"] == "delayed" else None
                       for op in ops]
        derived = any(op["kind"] in DQ_KINDS or op["kind"] in QS_KINDS or op["kind"] == "mmascale" for op in ops)
        assert not (seq and derived), "a drifting sequence feeds quantizers only"
        # set s reads input set s % n_in and writes output set s % n_out
        out_sets = []
        self.sets = []
        for s in range(self.nsets):
            ins = self.in_sets[s % self.n_in]
            if s < self.n_out:
                out_sets.append([self._outputs(op, ins[op["gen"]]) for op in ops])
            bufs = []
            for j, op in enumerate(ops):
                b = dict(out_sets[s % self.n_out][j])
                if "in" not in b:  # a quantizer: it reads this set's input tensor
                    b["x"] = ins[op["gen"]]
                    b["in"] = [b["x"]]
                b["call"], b["launches"] = self._call(op, b, lib, stream, off_ptr, self.states[j])
                bufs.append(b)
            self.sets.append(bufs)
        torch.cuda.synchronize()

    def _derived(self, op, x):
        """Inputs a row consumes, made by the library's own quantizers before
        timing: codes to dequantize or measure, scales to rearrange."""
        fq = self.fq
        k = op["kind"]
        if k == "mmascale":
            return {"in": [fq.mxfp8_quantize(x, op["fmt"], 3)[op["copy"]]], "x": None}
        if k in QS_KINDS:
            if k == "qs_tensor":
                qr = fq.fp8q_cast_per_tensor(x, op["fmt"])
                return {"in": [x, qr["q"], qr["scale_inv"]], "x": x}
            qr = fq.mxfp8_quantize(x, op["fmt"], 3)
            return {"in": [x, qr["q_row"], qr["s_row"]] if k == "qs_mx_row" else [x, qr["q_col"], qr["s_col"]],
                    "x": x}
        if k in DQ_KINDS:
            if k == "dq_tensor":
                qr = fq.fp8q_cast_per_tensor(x, op["fmt"])
                return {"in": [qr["q"], qr["scale_inv"]], "x": None}
            qr = fq.mxfp8_quantize(x, op["fmt"], 3)
            return {"in": [qr["q_row"], qr["s_row"]] if k == "dq_mx_row" else [qr["q_col"], qr["s_col"]], "x": None}
        return {}

    def _outputs(self, op, x):
        import torch
        fq, dev = self.fq, self.dev
        r, c = op["shape"]
        k = op["kind"]
        b = {}
        if k == "mx_mma":
            ld = fq.mxfp8_col_blocks(r, None)
            b["out"] = {"q_row": torch.empty((r, c), dtype=torch.uint8, device=dev),
                        "s_row": torch.empty(fq.mxfp8_mma_scale_bytes(r, c // 32), dtype=torch.uint8, device=dev),
                        "q_col": torch.empty((c, r), dtype=torch.uint8, device=dev),
                        "s_col": torch.empty(fq.mxfp8_mma_scale_bytes(c, ld), dtype=torch.uint8, device=dev)}
            b["ld"] = ld
        elif k in ("mx", "mx_grouped", "mx_rule"):
            ld = fq.mxfp8_col_blocks(r, None if k != "mx_grouped" else list(self.offsets_host))
            if k == "mx_grouped":
                ld = (ld + 15) // 16 * 16  # the library's default layout for grouped scales
            b["out"] = {"q_row": torch.empty((r, c), dtype=torch.uint8, device=dev),
                        "s_row": torch.empty((r, c // 32), dtype=torch.uint8, device=dev),
                        "q_col": torch.empty((c, r), dtype=torch.uint8, device=dev),
                        "s_col": torch.empty((c, ld), dtype=torch.uint8, device=dev)}
            b["ld"] = ld
            if k == "mx_rule":
                b["sat"] = torch.zeros(2, dtype=torch.int64, device=dev)
        elif k == "mxlow":
            fp4 = op["elem"] == 2
            b["lo"] = {"q_row": torch.empty((r, c // 2 if fp4 else c), dtype=torch.uint8, device=dev),
                       "s_row": torch.empty((r, c // 32), dtype=torch.uint8, device=dev),
                       "q_col": torch.empty((c, r // 2 if fp4 else r), dtype=torch.uint8, device=dev),
                       "s_col": torch.empty((c, (r + 31) // 32), dtype=torch.uint8, device=dev)}
        elif k == "nvfp4":
            b["nv"] = {"q": torch.empty((r, c // 2), dtype=torch.uint8, device=dev),
                       "s": torch.empty((r, c // 16), dtype=torch.uint8, device=dev),
                       "amax": torch.empty(1, dtype=torch.float32, device=dev),
                       "scale": torch.empty(1, dtype=torch.float32, device=dev)}
        elif k == "bw":
            tr, tc = (r + 127) // 128, (c + 127) // 128
            b["bw"] = {"q": torch.empty((r, c), dtype=torch.uint8, device=dev),
                       "s": torch.empty((r, tc) if op["block"] == 1 else (tr, tc), dtype=torch.float32, device=dev),
                       "q_t": torch.empty((c, r), dtype=torch.uint8, device=dev),
                       "s_t": torch.empty((c, tr) if op["block"] == 1 else (tc, tr), dtype=torch.float32, device=dev)}
        elif k == "mmascale":
            b.update(self._derived(op, x))
            sr, sc = b["in"][0].shape
            b["y"] = torch.empty(((sr + 127) // 128 * 128) * ((sc + 3) // 4 * 4), dtype=torch.uint8, device=dev)
        elif k in QS_KINDS:
            b.update(self._derived(op, x))
            b["st"] = torch.empty(fq.QSTATS_BYTES // 8, dtype=torch.float64, device=dev)
            b["ws"] = torch.zeros(fq.fp8q_qstats_workspace_bytes(), dtype=torch.uint8, device=dev)
        elif k in DQ_KINDS:
            b.update(self._derived(op, x))
            b["y"] = torch.empty(b["in"][0].shape, dtype=torch.bfloat16, device=dev)
        elif k == "delayed":
            b["q"] = torch.empty((r, c), dtype=torch.uint8, device=dev)
            b["dl"] = {n: torch.empty(1, dtype=torch.float32, device=dev) for n in ("scale", "scale_inv", "amax")}
        else:  # current, current_grouped
            b["q"] = torch.empty((r, c), dtype=torch.uint8, device=dev)
            G = op.get("G", 1)
            b["pt"] = {n: torch.empty(G, dtype=torch.float32, device=dev) for n in ("amax", "scale", "scale_inv")}
            b["ws"] = torch.zeros(fq.fp8q_cast_workspace_bytes(G), dtype=torch.uint8, device=dev)
        return b

    @staticmethod
    def _call(op, b, lib, stream, off_ptr, st):
        """(C-ABI function, argument tuple) of one op, and its kernel launches."""
        r, c = op["shape"]
        k = op["kind"]
        if k in ("mx", "mx_grouped"):
            o = b["out"]
            g = k == "mx_grouped"
            return (lib.mxfp8_quantize, (
                b["x"].data_ptr(), 0, r, c, off_ptr if g else None, op.get("G", 1), op["fmt"], 3,
                o["q_row"].data_ptr(), o["s_row"].data_ptr(), o["q_col"].data_ptr(), o["s_col"].data_ptr(), b["ld"],
                stream)), 1
        if k in ("current", "current_grouped"):
            pt = b["pt"]
            g = k == "current_grouped"
            return (lib.fp8q_cast_per_tensor, (
                b["x"].data_ptr(), 0, r, c, off_ptr if g else None, op.get("G", 1), op["fmt"], 0, None,
                b["q"].data_ptr(), pt["amax"].data_ptr(), pt["scale"].data_ptr(), pt["scale_inv"].data_ptr(), None,
                b["ws"].data_ptr(), b["ws"].numel(), stream)), 1 if not g and r * c <= current_one_launch_elems() else 2
        if k == "mx_mma":
            o = b["out"]
            return (lib.mxfp8_quantize_ex, (
                b["x"].data_ptr(), 0, r, c, None, 1, op["fmt"], 3, 0, 1, o["q_row"].data_ptr(), o["s_row"].data_ptr(),
                o["q_col"].data_ptr(), o["s_col"].data_ptr(), b["ld"], None, stream)), 1
        if k == "mx_rule":
            o = b["out"]
            return (lib.mxfp8_quantize_rule, (
                b["x"].data_ptr(), 0, r, c, None, 1, op["fmt"], 3, op["rule"], o["q_row"].data_ptr(),
                o["s_row"].data_ptr(), o["q_col"].data_ptr(), o["s_col"].data_ptr(), b["ld"], b["sat"].data_ptr(),
                stream)), 2  # the counters' zeroing kernel, then the quantizer
        if k == "mxlow":
            o = b["lo"]
            return (lib.mx_quantize_fp4_fp6, (
                b["x"].data_ptr(), 0, r, c, op["elem"], 3, 0, o["q_row"].data_ptr(), o["s_row"].data_ptr(),
                o["q_col"].data_ptr(), o["s_col"].data_ptr(), None, stream)), 1
        if k == "nvfp4":
            o = b["nv"]
            return (lib.fp8q_quantize_nvfp4, (
                b["x"].data_ptr(), 0, r, c, o["q"].data_ptr(), o["s"].data_ptr(), o["amax"].data_ptr(),
                o["scale"].data_ptr(), stream)), 3  # zeroing of the amax, amax, then the quantization
        if k == "bw":
            o = b["bw"]
            return (lib.fp8q_quantize_blockwise, (
                b["x"].data_ptr(), 0, r, c, op["fmt"], op["block"], 0, 3, o["q"].data_ptr(), o["s"].data_ptr(),
                o["q_t"].data_ptr(), o["s_t"].data_ptr(), stream)), 1
        if k == "dq_tensor":
            return (lib.fp8q_dequantize_per_tensor, (
                b["in"][0].data_ptr(), r, c, None, 1, op["fmt"], b["in"][1].data_ptr(), 0, b["y"].data_ptr(),
                stream)), 1
        if k == "mmascale":
            sr, sc = b["in"][0].shape
            return (lib.mx_scales_to_mma_layout, (b["in"][0].data_ptr(), sr, sc, sc, b["y"].data_ptr(), stream)), 1
        if k == "qs_tensor":
            return (lib.fp8q_qstats_per_tensor, (
                b["x"].data_ptr(), 0, r, c, None, 1, op["fmt"], b["in"][1].data_ptr(), b["in"][2].data_ptr(),
                b["st"].data_ptr(), b["ws"].data_ptr(), b["ws"].numel(), stream)), 1
        if k in ("qs_mx_row", "qs_mx_col"):
            return (lib.mxfp8_qstats, (
                b["x"].data_ptr(), 0, r, c, None, 1, op["fmt"], 1 if k == "qs_mx_row" else 2,
                b["in"][1].data_ptr(), b["in"][2].data_ptr(), b["in"][2].shape[1], b["st"].data_ptr(),
                b["ws"].data_ptr(), b["ws"].numel(), stream)), 1
        if k in ("dq_mx_row", "dq_mx_col"):
            return (lib.mxfp8_dequantize, (
                b["in"][0].data_ptr(), b["in"][1].data_ptr(), r, c, None, 1, op["fmt"],
                1 if k == "dq_mx_row" else 2, b["in"][1].shape[1], 0, b["y"].data_ptr(), stream)), 1
        dl = b["dl"]  # delayed
        return (lib.fp8q_delayed_step, (
            st._h, b["x"].data_ptr(), 0, r * c, b["q"].data_ptr(), dl["scale"].data_ptr(),
            dl["scale_inv"].data_ptr(), dl["amax"].data_ptr(), None, stream)), 1

    def call(self, j, i):
        fn, a = self.sets[i % self.nsets][j]["call"]
        if fn(*a) != 0:
            raise RuntimeError(self.lib.fp8q_last_error_string().decode())
        return self.sets[i % self.nsets][j]["launches"]

    def step(self, i):
        n = 0
        for j in range(len(self.ops)):
            n += self.call(j, i)
        return n

    def outputs(self, j, i=0):
        op, b = self.ops[j], self.sets[i % self.nsets][j]
        k = op["kind"]
        if k in ("mx", "mx_grouped", "mx_rule", "mx_mma"):
            o = b["out"]
            return [o["q_row"], o["s_row"], o["q_col"], o["s_col"]]
        if k == "bw":
            return [b["bw"][n] for n in ("q", "s", "q_t", "s_t")]
        if k == "nvfp4":
            return [b["nv"][n] for n in ("q", "s", "scale")]
        if k == "mxlow":
            return [b["lo"][n] for n in ("q_row", "s_row", "q_col", "s_col")]
        if k in QS_KINDS:
            return [b["st"]]
        if k == "delayed":
            return [b["q"], b["dl"]["scale_inv"]]
        if k in ("current", "current_grouped"):
            return [b["q"], b["pt"]["scale_inv"]]
        return [b["y"]]

    def step_inputs(self, j, i=0):
        """The tensors an op reads in set i that come from the host in an
        end-to-end step (a quantizer's BF16 input; a dequantizer's codes)."""
        b = self.sets[i % self.nsets][j]
        return b["in"]

    def close(self):
        for st in self.states:
            if st is not None:
                st.close()


def current_one_launch_elems():
    """Largest BF16 tensor whose ungrouped current scaling is one launch: 8
    times the on-chip capacity of two 16384-element slices per resident CTA,
    4 CTAs per SM (larger tensors take the amax and the cast kernel)."""
    import torch
    return 8 * 2 * 4 * torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count * 16384


def time_graph(P, k):
    """Milliseconds per step with the steps replayed from one CUDA graph, so
    that no host launch cost is in the way: steps 0..m-1 (m = min(k, 256),
    rotating over the buffer sets as the loop does) captured once on the
    current stream, the graph replayed until at least k steps ran, CUDA
    events around the replays."""
    import torch
    m = max(1, min(k, 256))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.current_stream()):
        for i in range(m):
            P.step(i)
    reps = max(1, -(-k // m))
    g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    P.fq.check_device()
    del g
    return e0.elapsed_time(e1) / (reps * m)


def time_loop(fn, n):
    """Milliseconds per iteration of fn(i) for i in range(n), CUDA events
    around the whole loop on the current stream."""
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def time_op(P, j, min_launches=ROOFLINE_MIN_LAUNCHES, target_s=0.15):
    """Average device time of op j's call in a loop of back-to-back calls
    (at least min_launches, about target_s seconds), rotating over the
    buffer sets as the step does."""
    import torch
    for i in range(5):
        P.call(j, i)
    torch.cuda.synchronize()
    est = time_loop(lambda i: P.call(j, i), 10)
    n = int(min(5000, max(min_launches, target_s / max(est * 1e-3, 1e-7))))
    return time_loop(lambda i: P.call(j, i), n), n


def measure(P, steps, warmup, world, dev, want_clocks, local=0):
    """The step timed over exactly `steps` steps (events around the loop),
    then per-step event pairs for the median and minimum."""
    import torch
    import torch.distributed as dist
    for i in range(warmup):
        P.step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(local) if want_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = [0]

    def one(i):
        launches[0] += P.step(i)

    elapsed_ms = time_loop(one, steps) * steps
    P.fq.check_device()  # raises if a bounded device-side wait gave up
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    # per-step times: an event between two steps (never inside one)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record()
    for i in range(steps):
        P.step(i)
        ev[i + 1].record()
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return elapsed_ms, launches[0], clocks, per


def roofline_entry(P, op, avg_ms, n, peak, peak_src, traffic_key):
    achieved = op["bytes"] / (avg_ms * 1e-3) / 1e9
    traffic, tinfo = kernel_traffic(traffic_key)
    e = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
         "frac": round(achieved / peak, 4), "peak_source": peak_src, "kernel": kernel_label(op),
         "algorithmic_bytes_per_launch": op["bytes"], "avg_launch_us": round(avg_ms * 1e3, 3),
         "launches_timed": n, "timing": "back-to-back launches, CUDA events around the loop",
         "traffic": traffic}
    if traffic is not None:
        e["traffic_over_algorithmic"] = round(traffic / op["bytes"], 4)
        if tinfo and "capture" in tinfo:
            e["traffic_capture"] = tinfo["capture"]
    return e


def op_table(P, peak):
    """Every op of the workload timed alone (back-to-back calls)."""
    rows = []
    for j, op in enumerate(P.ops):
        ms, n = time_op(P, j)
        gbs = op["bytes"] / (ms * 1e-3) / 1e9
        row = {"op": P.cfg["ops"][j] if "ops" in P.cfg else op["kind"], "kernels": kernel_label(op),
               "us_per_call": round(ms * 1e3, 3), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
               "calls_timed": n, "bytes_per_call": op["bytes"]}
        if op["kind"] in ("current", "current_grouped"):
            # the method reads x twice (amax before any cast, 5 B per BF16
            # element); against the compulsory floor of one read and one
            # write (3 B per element) the same time reads lower
            r, c = op["shape"]
            floor = 3 * r * c
            row["floor_bytes_per_call"] = floor
            row["floor_frac"] = round(floor / (ms * 1e-3) / 1e9 / peak, 4)
        rows.append(row)
    return rows


def roofline_op(P):
    return next((j for j, op in enumerate(P.ops) if op["kind"] in ROOFLINE_KINDS), 0)


def delayed_vs_current(P):
    """Config 3 as the pages compare it: 32 drifting steps of one 8192 x 8192
    tensor under delayed scaling (history 16, margin 3; E4M3 and E5M2;
    Interval 1 and 5), next to current scaling of the same tensors.  Per step:
    the scale used, the tensor's true amax, the saturated elements, and the
    SQNR and zero-rate of each copy, all computed on the device."""
    import torch
    fq = P.fq
    seqs = {}
    states = {(fmt, iv): fq.DelayedScaling(16, iv, 3, fmt) for fmt in (E4M3, E5M2) for iv in (1, 5)}
    gen = P.ops[0]["gen"]
    rec = {("current", fmt): {"scale": [], "sat": [], "sqnr_db": [], "zero_rate": []} for fmt in (E4M3, E5M2)}
    for key in states:
        rec[("delayed",) + key] = {"scale": [], "sat": [], "sqnr_db": [], "zero_rate": []}
    amax = []
    for t in range(C3_STEPS):
        x = P.in_sets[t][gen]
        for fmt in (E4M3, E5M2):
            cur = fq.fp8q_cast_per_tensor(x, fmt, want_sat=True)
            st = fq.qstats_dict(fq.fp8q_qstats_per_tensor(x, cur["q"], cur["scale_inv"], fmt))
            r = rec[("current", fmt)]
            r["scale"].append(float(cur["scale"].item()))
            r["sat"].append(int(cur["sat"].item()))
            r["sqnr_db"].append(round(st["sqnr_db"], 3))
            r["zero_rate"].append(st["zero_rate"])
            if fmt == E4M3:
                amax.append(float(cur["amax"].item()))
        for (fmt, iv), s in states.items():
            d = s.step(x, want_sat=True)
            st = fq.qstats_dict(fq.fp8q_qstats_per_tensor(x, d["q"], d["scale_inv"], fmt))
            r = rec[("delayed", fmt, iv)]
            r["scale"].append(float(d["scale"].item()))
            r["sat"].append(int(d["sat"].item()))
            r["sqnr_db"].append(round(st["sqnr_db"], 3))
            r["zero_rate"].append(st["zero_rate"])
    torch.cuda.synchronize()
    for s in states.values():
        s.close()
    fmt_name = {E4M3: "e4m3", E5M2: "e5m2"}
    for k, r in rec.items():
        name = f"current_{fmt_name[k[1]]}" if k[0] == "current" else f"delayed_{fmt_name[k[1]]}_interval{k[2]}"
        r["saturated_steps"] = sum(1 for v in r["sat"] if v)
        seqs[name] = r
    import synth
    sig = synth.config3_sigmas(C3_STEPS, 3)
    return {"tensor": "8192x8192 bf16, x_t = sigma_t z_t, sigma_{t+1} = sigma_t U(0.8, 1.25)",
            "history": 16, "margin": 3, "steps": C3_STEPS, "sigma": [round(float(v), 5) for v in sig],
            "true_amax": amax, "copies": seqs,
            "columns": "per step: scale used, saturated elements, SQNR (dB) and zero-rate of the FP8 copy"}


def e2e_leg(P, steps, world, dev):
    """The same step through the public C-ABI with host buffers: every step's
    inputs copied in from pinned host memory and every output copied back,
    inside the timed region.  The copies are pipelined as a user would: the
    upload of step i + 1 and the download of step i run on their own streams
    while the kernels run on the library's stream; events keep a buffer from
    being overwritten before the step that reads it, or the download of it,
    has finished."""
    import torch
    import torch.distributed as dist
    ins_host = []   # (device tensor getter, pinned host tensor)
    seen = set()
    for j, op in enumerate(P.ops):
        for t in P.step_inputs(j, 0):
            key = t.data_ptr()
            if key in seen:
                continue
            seen.add(key)
            ins_host.append((j, len(ins_host), t.detach().cpu().pin_memory()))
    outs_host = [[torch.empty(t.numel() * t.element_size(), dtype=torch.uint8).pin_memory() for t in P.outputs(j)]
                 for j in range(len(P.ops))]
    bi = sum(h.numel() * h.element_size() for _, _, h in ins_host)
    bo = sum(t.numel() for lst in outs_host for t in lst)
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    last_read, last_d2h = {}, {}  # device buffer -> event after its last reader / download

    def step_ins(i):
        res, seen2 = [], set()
        for j in range(len(P.ops)):
            for t in P.step_inputs(j, i):
                if t.data_ptr() not in seen2:
                    seen2.add(t.data_ptr())
                    res.append(t)
        return res

    def e2e_step(i):
        ins = step_ins(i)
        with torch.cuda.stream(s_in):
            for t in ins:
                if t.data_ptr() in last_read:
                    s_in.wait_event(last_read[t.data_ptr()])
            for dst, (_, _, src) in zip(ins, ins_host):
                dst.copy_(src, non_blocking=True)
            loaded = torch.cuda.Event()
            loaded.record(s_in)
        outs = [t for j in range(len(P.ops)) for t in P.outputs(j, i)]
        comp.wait_event(loaded)
        for t in outs:
            if t.data_ptr() in last_d2h:
                comp.wait_event(last_d2h[t.data_ptr()])
        P.step(i)
        done = torch.cuda.Event()
        done.record(comp)
        for t in ins:
            last_read[t.data_ptr()] = done
        with torch.cuda.stream(s_out):
            s_out.wait_event(done)
            for j in range(len(P.ops)):
                for dst, src in zip(outs_host[j], P.outputs(j, i)):
                    dst.copy_(src.reshape(-1).view(torch.uint8), non_blocking=True)
            fetched = torch.cuda.Event()
            fetched.record(s_out)
        for t in outs:
            last_d2h[t.data_ptr()] = fetched

    def run(n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        s_in.wait_stream(comp)
        s_out.wait_stream(comp)
        for i in range(n):
            e2e_step(i)
        comp.wait_stream(s_in)
        comp.wait_stream(s_out)
        e1.record(comp)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    run(3)
    # three timed runs of `steps` steps; the median is reported (the host
    # link is shared with whatever else runs on the host)
    runs = []
    for _ in range(3):
        if world > 1:
            dist.barrier()
        runs.append(max_over_ranks(run(steps), world, dev))
    ms = statistics.median(runs)
    return {"value": round(job_gbs(P.bytes_per_step, world, ms), 2), "unit": "GB/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": round(ms, 4),
            "runs_ms_per_step": [round(r, 4) for r in runs], "statistic": "median of 3 runs",
            "copies": "upload of step i + 1 and download of step i on their own streams, overlapping the kernels",
            "buffer_sets": P.nsets}


def measure_config(name, dev, peak, peak_src, steps, warmup):
    """One of the other configurations, measured as the headline is (device
    time of whole steps; each op timed alone in back-to-back loops)."""
    import torch
    side = torch.cuda.Stream(dev)  # a graph cannot capture the legacy stream
    with torch.cuda.stream(side):
        return _measure_config(name, dev, peak, peak_src, steps, warmup)


def _measure_config(name, dev, peak, peak_src, steps, warmup):
    import torch
    P = Prepared(name, dev)
    try:
        est = time_loop(lambda i: P.step(i), 3)
        k = int(min(2000, max(steps, 0.05 / max(est * 1e-3, 1e-7))))
        elapsed, launches, _, per = measure(P, k, warmup, 1, dev, False)
        ms = elapsed / k
        gbs = P.bytes_per_step / (ms * 1e-3) / 1e9
        ops = op_table(P, peak)
        j = roofline_op(P)
        rf = dict(ops[j])
        rf.update({"bound": "hbm", "peak": peak, "unit": "GB/s", "peak_source": peak_src,
                   "achieved": rf.pop("gbs")})
        res = {"workload": P.cfg, "steps": k, "ms_per_step": round(ms, 5),
               "step_ms_median": round(statistics.median(per), 5), "step_ms_min": round(min(per), 5),
               "value": round(gbs, 2), "unit": "GB/s", "frac_of_hbm_peak": round(gbs / peak, 4),
               "bytes_per_step": P.bytes_per_step, "gpu_launches": launches, "ops": ops, "roofline": rf,
               "l2": P.l2_note}
        try:
            gms = time_graph(P, k)
            ggbs = P.bytes_per_step / (gms * 1e-3) / 1e9
            res["graph"] = {"ms_per_step": round(gms, 5), "value": round(ggbs, 2), "unit": "GB/s",
                            "frac_of_hbm_peak": round(ggbs / peak, 4),
                            "timing": "the same steps replayed from one CUDA graph (no host launch cost)"}
        except Exception as e:  # a capture the runtime refuses: report the loop only
            res["graph"] = {"unavailable": repr(e)[:200]}
        if name == "delayed_8192":
            res["delayed_vs_current"] = delayed_vs_current(P)
        return res
    finally:
        P.close()
        del P
        torch.cuda.empty_cache()


def run_ours(args):
    import torch
    import torch.distributed as dist

    import mxfp8_quantization_amax_gb300 as fq

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fq.build()
    peak, peak_src = hbm_peak()

    P = Prepared(args.workload, dev)
    elapsed_ms, launches, clocks, per = measure(P, args.steps, args.warmup, world, dev, True, local)
    ms_per_step = elapsed_ms / args.steps
    jr = roofline_op(P)
    rl_ms, rl_n = time_op(P, jr)
    ops = op_table(P, peak)
    extra = {}
    if any(op["kind"] == "mx_rule" for op in P.ops):
        extra["saturated_elements"] = {("round_up" if op["rule"] == 0 else "ocp"): P.sets[0][j]["sat"].cpu().tolist()
                                       for j, op in enumerate(P.ops) if op["kind"] == "mx_rule"}
    if any(op["kind"] in QS_KINDS for op in P.ops):
        extra["qstats"] = {}
        for j, op in enumerate(P.ops):
            if op["kind"] in QS_KINDS:
                d = fq.qstats_dict(P.sets[0][j]["st"])
                extra["qstats"][op["kind"]] = {"sqnr_db": round(d["sqnr_db"], 4), "zero_rate": d["zero_rate"],
                                               "n_flushed": d["n_flushed"], "n_zero": d["n_zero"]}
    if args.workload == "delayed_8192" and rank == 0:
        extra["delayed_vs_current"] = delayed_vs_current(P)
    # last: the end-to-end leg overwrites the device inputs with host copies.
    # It double-buffers, as a pipelined caller does: with a single buffer set
    # the next step's kernels would wait for this step's download.
    e2e = None
    if not args.no_e2e:
        PE = P if min(P.n_in, P.n_out) >= 2 else Prepared(args.workload, dev, min_sets=2)
        e2e = e2e_leg(PE, args.e2e_steps, world, dev)
        if PE is not P:
            PE.close()
            del PE
    fq.check_device()
    roofline = roofline_entry(P, P.ops[jr], rl_ms, rl_n, peak, peak_src, args.workload)
    cfg = dict(P.cfg)
    cfg["l2"] = P.l2_note
    bytes_per_step = P.bytes_per_step
    P.close()
    del P
    torch.cuda.empty_cache()

    per_config = None
    if rank == 0 and world == 1 and args.workload == "moe" and not args.no_per_config:
        per_config = {cid: measure_config(name, dev, peak, peak_src, args.steps, args.warmup)
                      for cid, name in PER_CONFIG}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    value = job_gbs(bytes_per_step, world, ms_per_step)
    line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": cfg, "frac_of_hbm_peak": round(value / world / peak, 4), "roofline": roofline,
            "e2e": e2e, "gpu_launches": launches, "clocks": clocks, "bytes_per_step": bytes_per_step,
            "step_ms_median": round(statistics.median(per), 5), "step_ms_min": round(min(per), 5),
            "ops": ops}
    line.update(extra)
    if per_config is not None:
        line["per_config"] = per_config
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.workload)
    if world > 1:
        dist.destroy_process_group()
    return line


# ---------------------------------------------------------------------------
# the oracle on this host: cpu_baseline and the reference arm
# ---------------------------------------------------------------------------
def oracle_sample_step(workload, sample_rows, inputs, states):
    """The oracle on the first `sample_rows` rows of each op's tensor;
    returns the algorithmic bytes it processed."""
    import oracle
    cfg, ops = workload_spec(workload)
    total = 0
    for op, x, st in zip(ops, inputs, states):
        k = op["kind"]
        r, c = x["shape"] if k in DQ_KINDS or k in QS_KINDS or k == "mmascale" else x.shape
        if k in ("mx", "mx_grouped"):
            oracle.mx_quantize(x, op["fmt"], 3)
            total += mx_bytes(r, c)
        elif k == "mx_mma":
            m = oracle.mx_quantize(x, op["fmt"], 3)
            oracle.mma_scale_layout(m["s_row"])
            oracle.mma_scale_layout(m["s_col"])
            total += mx_bytes(r, c)
        elif k == "mx_rule":
            oracle.mx_quantize_rule(x, op["fmt"], 3, op["rule"])
            total += mx_bytes(r, c)
        elif k == "mmascale":
            oracle.mma_scale_layout(x["s"])
            total += 2 * x["s"].size
        elif k == "mxlow":
            oracle.mxlp_quantize(x, op["elem"], 3, 0)
            total += (3 if op["elem"] == 2 else 4) * r * c + r * c // 16
        elif k == "nvfp4":
            oracle.nvfp4(x)
            total += 4 * r * c + r * c // 2 + r * c // 16
        elif k == "bw":
            g = (1, 128) if op["block"] == 1 else (128, 128)
            oracle.blockwise(x, op["fmt"], g)
            oracle.blockwise(x, op["fmt"], (128, 1) if op["block"] == 1 else g)
            total += 4 * r * c
        elif k in ("current", "current_grouped"):
            oracle.current_scaling(x, op["fmt"])
            total += 5 * r * c
        elif k == "dq_tensor":
            oracle.dequant_per_tensor(x["q"], op["fmt"], x["scale_inv"])
            total += 3 * r * c
        elif k in ("dq_mx_row", "dq_mx_col"):
            d = 1 if k == "dq_mx_row" else 2
            oracle.mx_dequantize(x["q"], x["s"], op["fmt"], d, r, c)
            total += 3 * r * c + x["s"].size
        elif k == "qs_tensor":
            oracle.qstats_per_tensor(x["x"], x["q"], op["fmt"], x["scale_inv"])
            total += 3 * r * c + 4 + 48
        elif k in ("qs_mx_row", "qs_mx_col"):
            oracle.qstats_mx(x["x"], x["q"], x["s"], op["fmt"], 1 if k == "qs_mx_row" else 2)
            total += 3 * r * c + x["s"].size + 48
        else:
            st.step(x)
            total += 3 * r * c
    return total


def oracle_inputs(workload, sample_rows):
    import oracle
    cfg, ops = workload_spec(workload)
    xs, states = [], []
    cache = {}
    for op in ops:
        r, c = op["shape"]
        rr = min(r, sample_rows)
        key = (op["gen"], rr, c)
        if key not in cache:
            cache[key] = np.ascontiguousarray(host_input(op["gen"], (rr, c)))
        x = cache[key]
        if op["kind"] == "dq_tensor":  # the codes to dequantize, made by the oracle before timing
            cs = oracle.current_scaling(x, op["fmt"])
            x = {"q": cs["q"].reshape(rr, c), "scale_inv": cs["scale_inv"], "shape": (rr, c)}
        elif op["kind"] in ("dq_mx_row", "dq_mx_col"):
            m = oracle.mx_quantize(x, op["fmt"], 3)
            x = ({"q": m["q_row"], "s": m["s_row"], "shape": (rr, c)} if op["kind"] == "dq_mx_row"
                 else {"q": m["q_col"], "s": m["s_col"], "shape": (rr, c)})
        elif op["kind"] == "mmascale":  # the scales to rearrange, made by the oracle before timing
            m = oracle.mx_quantize(x, op["fmt"], 3)
            x = {"s": m[op["copy"]], "shape": (rr, c)}
        elif op["kind"] == "qs_tensor":  # the copy to measure, made by the oracle before timing
            cs = oracle.current_scaling(x, op["fmt"])
            x = {"x": x, "q": cs["q"].reshape(rr, c), "scale_inv": cs["scale_inv"], "shape": (rr, c)}
        elif op["kind"] in ("qs_mx_row", "qs_mx_col"):
            m = oracle.mx_quantize(x, op["fmt"], 3)
            x = ({"x": x, "q": m["q_row"], "s": m["s_row"], "shape": (rr, c)} if op["kind"] == "qs_mx_row"
                 else {"x": x, "q": m["q_col"], "s": m["s_col"], "shape": (rr, c)})
        xs.append(x)
        states.append(oracle.DelayedScaling(16, op["interval"], 3, op["fmt"]) if op["kind"] == "delayed" else None)
    return xs, states


def sample_rows_for(workload):
    return {"activation": 256, "mx_4096": 256, "mx_8192": 128, "per_tensor_1024": 1024, "delayed_8192": 64,
            "linear_layer": 64, "moe": 1024, "moe_16384": 1024, "mx_mma_8192": 128, "dequant_8192": 128, "mx_rules_4096": 256, "blockwise_8192": 128,
            "nvfp4_8192": 128, "qstats_8192": 128, "mxfp4_fp6_8192": 128, "mma_scales_8192": 1024}[workload]


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                low = ln.lower()
                if low.startswith("model name") or low.startswith("cpu part") or low.startswith("hardware"):
                    return ln.split(":", 1)[1].strip() + f" ({platform.machine()})"
    except OSError:
        pass
    return platform.machine() or "unknown"


def cpu_leg(workload, budget_s):
    """Repeated oracle sample steps for about budget_s seconds: mean, median
    and best GB/s over the repetitions, and the threads the oracle used."""
    import oracle
    rows = sample_rows_for(workload)
    xs, states = oracle_inputs(workload, rows)
    oracle_sample_step(workload, rows, xs, states)  # warm
    reps = []
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s or len(reps) < 3:
        a = time.perf_counter()
        b = oracle_sample_step(workload, rows, xs, states)
        reps.append((b, time.perf_counter() - a))
    total_b = sum(b for b, _ in reps)
    total_t = sum(t for _, t in reps)
    rates = [b / t / 1e9 for b, t in reps]
    return {"value": round(total_b / total_t / 1e9, 4), "median": round(statistics.median(rates), 4),
            "best": round(max(rates), 4), "reps": len(reps), "seconds": round(total_t, 2),
            "cores": oracle.max_threads(), "sample_rows": rows}


def cpu_baseline(workload, budget_s=10.0, single_budget_s=5.0):
    """The oracle, as it stands, timed on this host: all cores (OpenMP) and,
    in a child process with OMP_NUM_THREADS=1, single-threaded."""
    leg = cpu_leg(workload, budget_s)
    single = None
    try:
        env = dict(os.environ, OMP_NUM_THREADS="1")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-leg", f"{workload}:{single_budget_s}"],
                           env=env, capture_output=True, text=True, timeout=300)
        single = json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else None
    except (OSError, ValueError, IndexError, subprocess.TimeoutExpired):
        single = None
    return {"value": leg["value"], "unit": "GB/s", "cores": leg["cores"], "kind": "oracle",
            "sample": f"first {leg['sample_rows']} rows of each op's tensor, {leg['reps']} repetitions in "
                      f"{leg['seconds']} s (value: total bytes / total time)",
            "median": leg["median"], "best": leg["best"], "cpu": cpu_model(),
            "single_thread": None if single is None else {"value": single["value"], "median": single["median"],
                                                          "best": single["best"], "cores": single["cores"],
                                                          "reps": single["reps"]}}


def run_reference(args):
    import oracle
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    cfg, _ = workload_spec(args.workload)
    rows = sample_rows_for(args.workload)
    xs, states = oracle_inputs(args.workload, rows)
    for _ in range(args.warmup):
        oracle_sample_step(args.workload, rows, xs, states)
    # bound the timed run to about two minutes of oracle work
    t0 = time.perf_counter()
    total, n = 0, 0
    for _ in range(args.steps):
        total += oracle_sample_step(args.workload, rows, xs, states)
        n += 1
        if time.perf_counter() - t0 > 120:
            break
    dt = time.perf_counter() - t0
    value = total / dt / 1e9
    cores = oracle.max_threads()
    sample = f"first {rows} rows of each op's tensor per step, {n} of {args.steps} steps timed"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": n, "warmup": args.warmup, "ms_per_step": round(dt / n * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample, "cpu": cpu_model()},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_leg:
        name, budget = args.cpu_leg.split(":")
        print(json.dumps(cpu_leg(name, float(budget))), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
