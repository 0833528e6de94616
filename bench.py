"""Benchmark of the FP8 / MXFP8 quantization hot path on one node.

One step = one pass of the whole path over one batch of the activation
workload (4096x4096 BF16: N(0,1) times a per-row lognormal(0,2) factor,
0.1% of entries x1000, 1% of the 1x32 blocks zero):
  * mxfp8_quantize, E4M3, rowwise + columnwise        (4.0625 B/element)
  * fp8q_cast_per_tensor, current scaling, E4M3       (5 B/element: amax read,
                                                       cast read + write)
  * fp8q_delayed_step, E4M3, history 16, margin 3,
    Interval 1 (amax fused into the cast)             (3 B/element + history)
Each op gets its own input tensor, and the step cycles over enough buffer
sets that no input is still in L2 when it is read again.

value: bytes read + written by the step's kernels, summed over all ranks,
divided by the max over ranks of the device time of K steps (GB/s).
roofline: the MXFP8 kernel alone, timed with CUDA events around its launch
in every 8th timed step, against the measured HBM copy bandwidth.

--workload selects another workload for the same line format:
  activation (default), mx_8192 (MXFP8 on 8192x8192, for profiling),
  per_tensor_1024 (1024x1024 current scaling),
  delayed_8192 (8192x8192 delayed steps), linear_layer (A, W, E of an
  8B-class layer, MXFP8 both directions), moe (65536x7168, 64 experts:
  grouped MXFP8 and grouped current scaling), dequant_8192 (both MXFP8
  copies and a per-tensor code array of 8192x8192 back to BF16),
  mx_rules_4096 (MXFP8 of the activation under the round-up and the OCP
  scale rule, saturated elements counted and reported), blockwise_8192
  (blockwise FP8 of an activation in 1x128/128x1 groups and of a weight in
  128x128 blocks, both copies each), nvfp4_8192 (NVFP4 of the activation:
  tensor amax, then E2M1 codes with E4M3 scales per 16).
--impl reference: the CPU oracle on this host (a bounded sample per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "quantize GB/s (bytes read+written) and % of GB300 HBM peak, bit-exact"
FALLBACK_HBM_GBS = 6800.0
MX_SAMPLE = 8  # the MXFP8 launch of every 8th timed step is bracketed by events
E4M3, E5M2 = 0, 1


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="activation",
                   choices=["activation", "mx_8192", "per_tensor_1024", "delayed_8192", "linear_layer", "moe",
                            "dequant_8192", "mx_rules_4096", "blockwise_8192", "nvfp4_8192",
                            "qstats_8192", "mxfp4_fp6_8192", "mma_scales_8192"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=20)
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# workloads: shapes, algorithmic bytes, host inputs
# ---------------------------------------------------------------------------
def mx_bytes(rows, cols, ncolblocks=None):
    ncb = (rows + 31) // 32 if ncolblocks is None else ncolblocks
    return rows * cols * 2 + rows * cols + rows * (cols // 32) + cols * rows + cols * ncb


def workload_spec(name):
    """(config dict, list of ops).  An op is a dict with 'kind', its tensor
    shape and its algorithmic bytes per call."""
    if name == "activation":
        r = c = 4096
        ops = [{"kind": "mx", "shape": (r, c), "fmt": E4M3, "bytes": mx_bytes(r, c), "gen": ("c2", 0)},
               {"kind": "current", "shape": (r, c), "fmt": E4M3, "bytes": 5 * r * c, "gen": ("c2", 1)},
               {"kind": "delayed", "shape": (r, c), "fmt": E4M3, "bytes": 3 * r * c + 4 * 16, "gen": ("c2", 2)}]
        cfg = {"workload": "activation_4096x4096_bf16", "rows": r, "cols": c,
               "ops": ["mxfp8 e4m3 row+col", "current scaling e4m3", "delayed e4m3 H16 margin3 interval1"]}
        return cfg, ops
    if name == "mx_8192":
        r = c = 8192
        ops = [{"kind": "mx", "shape": (r, c), "fmt": E4M3, "bytes": mx_bytes(r, c), "gen": ("c2", 0)}]
        return {"workload": "mxfp8_8192x8192_bf16", "rows": r, "cols": c, "ops": ["mxfp8 e4m3 row+col"]}, ops
    if name == "per_tensor_1024":
        ops = [{"kind": "current", "shape": (1024, 1024), "fmt": E4M3, "bytes": 5 * 1024 * 1024, "gen": ("c1", 0)}]
        return {"workload": "per_tensor_current_1024x1024_bf16", "rows": 1024, "cols": 1024}, ops
    if name == "delayed_8192":
        r = c = 8192
        ops = [{"kind": "delayed", "shape": (r, c), "fmt": E4M3, "bytes": 3 * r * c + 64, "gen": ("c3", 0)},
               {"kind": "delayed", "shape": (r, c), "fmt": E5M2, "bytes": 3 * r * c + 64, "gen": ("c3", 1)}]
        return {"workload": "delayed_8192x8192_bf16", "rows": r, "cols": c,
                "ops": ["delayed e4m3 H16 margin3 interval1", "delayed e5m2 H16 margin3 interval1"]}, ops
    if name == "linear_layer":
        shapes = {"A": (16384, 4096), "W": (14336, 4096), "E": (16384, 14336)}
        ops = [{"kind": "mx", "shape": shapes[k], "fmt": E5M2 if k == "E" else E4M3,
                "bytes": mx_bytes(*shapes[k]), "gen": ("c4", k)} for k in ("A", "W", "E")]
        return {"workload": "linear_layer_8b_mxfp8", "A": "16384x4096", "W": "14336x4096",
                "E": "16384x14336"}, ops
    if name == "moe":
        r, c = 65536, 7168
        ops = [{"kind": "mx_grouped", "shape": (r, c), "fmt": E4M3, "bytes": None, "gen": ("c5", 0)},
               {"kind": "current_grouped", "shape": (r, c), "fmt": E4M3, "bytes": 5 * r * c, "gen": ("c5", 0)}]
        return {"workload": "moe_64_experts_65536x7168_bf16", "rows": r, "cols": c, "experts": 64}, ops
    if name == "mx_rules_4096":
        r = c = 4096
        ops = [{"kind": "mx_rule", "rule": 0, "shape": (r, c), "fmt": E4M3, "bytes": mx_bytes(r, c), "gen": ("c2", 0)},
               {"kind": "mx_rule", "rule": 1, "shape": (r, c), "fmt": E4M3, "bytes": mx_bytes(r, c), "gen": ("c2", 0)}]
        return {"workload": "mxfp8_scale_rules_4096x4096_bf16", "rows": r, "cols": c,
                "ops": ["mxfp8 e4m3 row+col, round-up rule, saturation counted",
                        "mxfp8 e4m3 row+col, OCP rule, saturation counted"]}, ops
    if name == "blockwise_8192":
        r = c = 8192
        ops = [{"kind": "bw", "block": 1, "shape": (r, c), "fmt": E4M3, "bytes": 4 * r * c + 4 * (r * (c // 128) + c * (r // 128)),
                "gen": ("c2", 0)},
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
                "ops": ["rowwise mx scales [8192][256] -> 128x4 blocks", "columnwise mx scales [8192][256] -> 128x4 blocks"]}, ops
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
        ops = [{"kind": "qs_mx_row", "shape": (r, c), "fmt": E4M3, "bytes": 3 * r * c + r * c // 32 + 48, "gen": ("c2", 0)},
               {"kind": "qs_mx_col", "shape": (r, c), "fmt": E4M3, "bytes": 3 * r * c + c * (r // 32) + 48, "gen": ("c2", 0)},
               {"kind": "qs_tensor", "shape": (r, c), "fmt": E4M3, "bytes": 3 * r * c + 4 + 48, "gen": ("c2", 0)}]
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
ROOFLINE_KINDS = ("mx", "mx_grouped", "dq_mx_row", "mx_rule", "bw", "nvfp4", "qs_mx_row", "mxlow", "mmascale")
LOW_NAMES = {2: "e2m1", 3: "e2m3", 4: "e3m2"}


def host_input(gen, shape):
    import synth
    kind, idx = gen
    if kind == "c2":
        return synth.config2(*shape, seed=2 + 100 * idx)
    if kind == "c1":
        return synth.config1(*shape, seed=1)
    if kind == "c3":
        return synth.config3_step(0, *shape, seed=3 + idx)
    if kind == "c4":
        t = {"A": lambda: synth.normal_outliers(*shape, seed=4, std=0.02, p=0.0005, factor=50.0, tensor=1),
             "W": lambda: synth.normal_outliers(*shape, seed=4, std=0.02, p=0.0005, factor=50.0, tensor=2),
             "E": lambda: synth.student_t(*shape, 3.0, seed=4, scale=1e-4, tensor=3)}
        return t[idx]()
    if kind == "c5":
        return synth.student_t(*shape, 4.0, seed=5)
    raise ValueError(kind)


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
    """DRAM bytes per launch of the workload's first kernel from the
    committed ncu summary (profiles/traffic.txt: one `key=value ...` line per
    workload; `sources=a,b,...` names the files whose hash keys it, the
    MXFP8 kernel's by default), or None if there is none or those sources
    changed since."""
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
                return int(d["bytes_per_launch"])
    except OSError:
        return None
    return None


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
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist

    import mxfp8_quantization_amax_gb300 as fq
    import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world > 1:
        fq.build()
    cfg, ops = workload_spec(args.workload)

    # host inputs (pinned, for the end-to-end leg) and their device copies
    offsets_host = None
    if args.workload == "moe":
        offsets_host = synth.moe_offsets(65536, 64, seed=5)
        ncb = int(sum((int(offsets_host[g + 1] - offsets_host[g]) + 31) // 32 for g in range(64)))
        for op in ops:
            if op["kind"] == "mx_grouped":
                op["bytes"] = mx_bytes(*op["shape"], ncolblocks=ncb)
    host = []
    for op in ops:
        h = host_input(op["gen"], op["shape"])
        host.append(torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).pin_memory())
    bytes_per_step = sum(op["bytes"] for op in ops)
    in_bytes = sum(h.numel() * 2 for h in host)
    # enough buffer sets that a set is out of L2 when it comes round again
    l2 = 129 * 2 ** 20
    per_set = in_bytes + sum(op["bytes"] - 2 * int(np.prod(op["shape"])) for op in ops)
    nsets = max(1, min(64, -(-4 * l2 // per_set)))
    off_dev = None if offsets_host is None else torch.from_numpy(offsets_host).to(dev)

    sets = []
    for s in range(nsets):
        bufs = []
        for op, h in zip(ops, host):
            r, c = op["shape"]
            x = h.to(dev, non_blocking=True)
            b = {"x": x, "in": [x]}
            if op["kind"] in ("mx", "mx_grouped", "mx_rule"):
                ld = fq.mxfp8_col_blocks(r, None if offsets_host is None else list(offsets_host))
                if offsets_host is not None:
                    ld = (ld + 15) // 16 * 16  # the library's default layout for grouped scales
                b["out"] = {"q_row": torch.empty((r, c), dtype=torch.uint8, device=dev),
                            "s_row": torch.empty((r, c // 32), dtype=torch.uint8, device=dev),
                            "q_col": torch.empty((c, r), dtype=torch.uint8, device=dev),
                            "s_col": torch.empty((c, ld), dtype=torch.uint8, device=dev)}
                b["ld"] = ld
                if op["kind"] == "mx_rule":
                    b["sat"] = torch.zeros(2, dtype=torch.int64, device=dev)
            elif op["kind"] == "mxlow":
                fp4 = op["elem"] == 2
                b["lo"] = {"q_row": torch.empty((r, c // 2 if fp4 else c), dtype=torch.uint8, device=dev),
                           "s_row": torch.empty((r, c // 32), dtype=torch.uint8, device=dev),
                           "q_col": torch.empty((c, r // 2 if fp4 else r), dtype=torch.uint8, device=dev),
                           "s_col": torch.empty((c, (r + 31) // 32), dtype=torch.uint8, device=dev)}
            elif op["kind"] == "nvfp4":
                b["nv"] = {"q": torch.empty((r, c // 2), dtype=torch.uint8, device=dev),
                           "s": torch.empty((r, c // 16), dtype=torch.uint8, device=dev),
                           "amax": torch.empty(1, dtype=torch.float32, device=dev),
                           "scale": torch.empty(1, dtype=torch.float32, device=dev)}
            elif op["kind"] == "bw":
                tr, tc = (r + 127) // 128, (c + 127) // 128
                b["bw"] = {"q": torch.empty((r, c), dtype=torch.uint8, device=dev),
                           "s": torch.empty((r, tc) if op["block"] == 1 else (tr, tc), dtype=torch.float32, device=dev),
                           "q_t": torch.empty((c, r), dtype=torch.uint8, device=dev),
                           "s_t": torch.empty((c, tr) if op["block"] == 1 else (tc, tr), dtype=torch.float32,
                                              device=dev)}
            elif op["kind"] == "mmascale":
                # the scales to rearrange, made by the library's MX quantizer before timing
                qr = fq.mxfp8_quantize(x, op["fmt"], 3)
                b["in"] = [qr[op["copy"]]]
                del qr
                sr, sc = b["in"][0].shape
                b["y"] = torch.empty(((sr + 127) // 128 * 128) * ((sc + 3) // 4 * 4), dtype=torch.uint8, device=dev)
                b["x"] = None
                del x
            elif op["kind"] in QS_KINDS:
                # the copy to measure, made by the library's own quantizers
                # before timing; x stays as the reference
                if op["kind"] == "qs_tensor":
                    qr = fq.fp8q_cast_per_tensor(x, op["fmt"])
                    b["in"] = [x, qr["q"], qr["scale_inv"]]
                else:
                    qr = fq.mxfp8_quantize(x, op["fmt"], 3)
                    b["in"] = [x, qr["q_row"], qr["s_row"]] if op["kind"] == "qs_mx_row" else \
                        [x, qr["q_col"], qr["s_col"]]
                b["st"] = torch.empty(6, dtype=torch.float64, device=dev)
                b["ws"] = torch.zeros(fq.fp8q_qstats_workspace_bytes(), dtype=torch.uint8, device=dev)
            elif op["kind"] in DQ_KINDS:
                # the codes to dequantize, made by the library's own quantizers
                # before timing; the BF16 input is not kept
                if op["kind"] == "dq_tensor":
                    qr = fq.fp8q_cast_per_tensor(x, op["fmt"])
                    b["in"] = [qr["q"], qr["scale_inv"]]
                else:
                    qr = fq.mxfp8_quantize(x, op["fmt"], 3)
                    b["in"] = [qr["q_row"], qr["s_row"]] if op["kind"] == "dq_mx_row" else [qr["q_col"], qr["s_col"]]
                b["y"] = torch.empty(b["in"][0].shape, dtype=torch.bfloat16, device=dev)
                b["x"] = None
                del x
            else:
                b["q"] = torch.empty((r, c), dtype=torch.uint8, device=dev)
                G = 64 if op["kind"] == "current_grouped" else 1
                b["pt"] = {k: torch.empty(G, dtype=torch.float32, device=dev) for k in ("amax", "scale", "scale_inv")}
                b["ws"] = torch.zeros(fq.fp8q_cast_workspace_bytes(G), dtype=torch.uint8, device=dev)
            bufs.append(b)
        sets.append(bufs)
    states = [fq.DelayedScaling(16, 1, 3, op["fmt"]) if op["kind"] == "delayed" else None for op in ops]
    for bufs in sets:
        for op, b in zip(ops, bufs):
            if op["kind"] == "delayed":
                b["dl"] = {k: torch.empty(1, dtype=torch.float32, device=dev) for k in ("scale", "scale_inv", "amax")}
    torch.cuda.synchronize()

    # Each op's C-ABI call with its arguments prepared once, so the host
    # enqueues a step in a few microseconds and never starves the GPU.
    lib = fq.lib()
    stream = torch.cuda.current_stream().cuda_stream
    off_ptr = None if off_dev is None else off_dev.data_ptr()
    for bufs in sets:
        for op, b, st in zip(ops, bufs, states):
            r, c = op["shape"]
            k = op["kind"]
            if k in ("mx", "mx_grouped"):
                o = b["out"]
                b["call"] = (lib.mxfp8_quantize, (
                    b["x"].data_ptr(), 0, r, c, off_ptr if k == "mx_grouped" else None,
                    64 if k == "mx_grouped" else 1, op["fmt"], 3, o["q_row"].data_ptr(), o["s_row"].data_ptr(),
                    o["q_col"].data_ptr(), o["s_col"].data_ptr(), b["ld"], stream))
                b["launches"] = 1
            elif k in ("current", "current_grouped"):
                pt = b["pt"]
                b["call"] = (lib.fp8q_cast_per_tensor, (
                    b["x"].data_ptr(), 0, r, c, off_ptr if k == "current_grouped" else None,
                    64 if k == "current_grouped" else 1, op["fmt"], 0, None, b["q"].data_ptr(),
                    pt["amax"].data_ptr(), pt["scale"].data_ptr(), pt["scale_inv"].data_ptr(), None,
                    b["ws"].data_ptr(), b["ws"].numel(), stream))
                b["launches"] = 2
            elif k == "mx_rule":
                o = b["out"]
                b["call"] = (lib.mxfp8_quantize_rule, (
                    b["x"].data_ptr(), 0, r, c, None, 1, op["fmt"], 3, op["rule"], o["q_row"].data_ptr(),
                    o["s_row"].data_ptr(), o["q_col"].data_ptr(), o["s_col"].data_ptr(), b["ld"],
                    b["sat"].data_ptr(), stream))
                b["launches"] = 1  # (plus the driver's memset of the two counters)
            elif k == "mxlow":
                o = b["lo"]
                b["call"] = (lib.mx_quantize_fp4_fp6, (
                    b["x"].data_ptr(), 0, r, c, op["elem"], 3, 0, o["q_row"].data_ptr(), o["s_row"].data_ptr(),
                    o["q_col"].data_ptr(), o["s_col"].data_ptr(), None, stream))
                b["launches"] = 1
            elif k == "nvfp4":
                o = b["nv"]
                b["call"] = (lib.fp8q_quantize_nvfp4, (
                    b["x"].data_ptr(), 0, r, c, o["q"].data_ptr(), o["s"].data_ptr(), o["amax"].data_ptr(),
                    o["scale"].data_ptr(), stream))
                b["launches"] = 2  # amax, then the quantization (plus the driver's memset of amax)
            elif k == "bw":
                o = b["bw"]
                b["call"] = (lib.fp8q_quantize_blockwise, (
                    b["x"].data_ptr(), 0, r, c, op["fmt"], op["block"], 0, 3, o["q"].data_ptr(), o["s"].data_ptr(),
                    o["q_t"].data_ptr(), o["s_t"].data_ptr(), stream))
                b["launches"] = 1
            elif k == "dq_tensor":
                b["call"] = (lib.fp8q_dequantize_per_tensor, (
                    b["in"][0].data_ptr(), r, c, None, 1, op["fmt"], b["in"][1].data_ptr(), 0, b["y"].data_ptr(),
                    stream))
                b["launches"] = 1
            elif k == "mmascale":
                sr, sc = b["in"][0].shape
                b["call"] = (lib.mx_scales_to_mma_layout, (b["in"][0].data_ptr(), sr, sc, sc, b["y"].data_ptr(), stream))
                b["launches"] = 1
            elif k == "qs_tensor":
                b["call"] = (lib.fp8q_qstats_per_tensor, (
                    b["x"].data_ptr(), 0, r, c, None, 1, op["fmt"], b["in"][1].data_ptr(), b["in"][2].data_ptr(),
                    b["st"].data_ptr(), b["ws"].data_ptr(), b["ws"].numel(), stream))
                b["launches"] = 1
            elif k in ("qs_mx_row", "qs_mx_col"):
                b["call"] = (lib.mxfp8_qstats, (
                    b["x"].data_ptr(), 0, r, c, None, 1, op["fmt"], 1 if k == "qs_mx_row" else 2,
                    b["in"][1].data_ptr(), b["in"][2].data_ptr(), b["in"][2].shape[1], b["st"].data_ptr(),
                    b["ws"].data_ptr(), b["ws"].numel(), stream))
                b["launches"] = 1
            elif k in ("dq_mx_row", "dq_mx_col"):
                b["call"] = (lib.mxfp8_dequantize, (
                    b["in"][0].data_ptr(), b["in"][1].data_ptr(), r, c, None, 1, op["fmt"],
                    1 if k == "dq_mx_row" else 2, b["in"][1].shape[1], 0, b["y"].data_ptr(), stream))
                b["launches"] = 1
            else:
                dl = b["dl"]
                b["call"] = (lib.fp8q_delayed_step, (
                    st._h, b["x"].data_ptr(), 0, r * c, b["q"].data_ptr(), dl["scale"].data_ptr(),
                    dl["scale_inv"].data_ptr(), dl["amax"].data_ptr(), None, stream))
                b["launches"] = 1

    mx_events = []
    launches = {"n": 0}

    mx_first = next((j for j, op in enumerate(ops) if op["kind"] in ROOFLINE_KINDS), None)

    def step(i, record_mx=False):
        bufs = sets[i % nsets]
        for j, (op, b) in enumerate(zip(ops, bufs)):
            fn, a = b["call"]
            timed = record_mx and j == mx_first
            if timed:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
            if fn(*a) != 0:
                raise RuntimeError(lib.fp8q_last_error_string().decode())
            if timed:
                e1.record()
                mx_events.append((e0, e1))
            launches["n"] += b["launches"]

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches["n"] = 0
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(args.steps):
        # events around the step's first MXFP8 launch on every MX_SAMPLE-th
        # step: an event between two kernels stops the second from launching
        # early, so bracketing every launch would slow the step being timed
        step(i, record_mx=i % MX_SAMPLE == 0)
    t1.record()
    torch.cuda.synchronize()
    fq.check_device()  # raises if a bounded device-side wait gave up
    elapsed_ms = t0.elapsed_time(t1)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    mx_ms = [a.elapsed_time(b) for a, b in mx_events]
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)

    # end-to-end: host inputs -> device, the step, device -> host outputs
    e2e = None
    if not args.no_e2e:
        # each op's step inputs as pinned host copies (the quantizers' BF16
        # input, or the dequantizers' codes and scales) and its outputs
        def outputs(op, b):
            if op["kind"] in ("mx", "mx_grouped", "mx_rule"):
                o = b["out"]
                return [o["q_row"], o["s_row"], o["q_col"], o["s_col"]]
            if op["kind"] == "bw":
                return [b["bw"][k] for k in ("q", "s", "q_t", "s_t")]
            if op["kind"] == "nvfp4":
                return [b["nv"][k] for k in ("q", "s", "scale")]
            if op["kind"] == "mxlow":
                return [b["lo"][k] for k in ("q_row", "s_row", "q_col", "s_col")]
            if op["kind"] in QS_KINDS:
                return [b["st"]]
            return [b["y"]] if op["kind"] in DQ_KINDS or op["kind"] == "mmascale" else [b["q"]]

        ins_host = [[t.cpu().pin_memory() for t in sets[0][j]["in"]] for j in range(len(ops))]
        outs_host = [[torch.empty(t.numel() * t.element_size(), dtype=torch.uint8).pin_memory()
                      for t in outputs(op, sets[0][j])] for j, op in enumerate(ops)]
        bi = sum(t.numel() * t.element_size() for lst in ins_host for t in lst)
        bo = sum(t.numel() for lst in outs_host for t in lst)

        def e2e_step(i):
            b = sets[i % nsets]
            for j in range(len(ops)):
                for dst, src in zip(b[j]["in"], ins_host[j]):
                    dst.copy_(src, non_blocking=True)
            step(i)
            for j, op in enumerate(ops):
                for dst, src in zip(outs_host[j], outputs(op, b[j])):
                    dst.copy_(src.reshape(-1).view(torch.uint8), non_blocking=True)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(args.e2e_steps):
            e2e_step(i)
        z.record()
        torch.cuda.synchronize()
        e2e_ms = a.elapsed_time(z) / args.e2e_steps
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        e2e = {"value": round(job_gbs(bytes_per_step, world, e2e_ms), 2), "unit": "GB/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": round(e2e_ms, 4)}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    ms_per_step = elapsed_ms / args.steps
    value = job_gbs(bytes_per_step, world, ms_per_step)
    peak, peak_src = hbm_peak()
    mx_op = next((op for op in ops if op["kind"] in ROOFLINE_KINDS), None)
    roofline = None
    if mx_op is not None and mx_ms:
        # average over the sampled launches of the step's first MXFP8 op
        avg_ms = sum(mx_ms) / len(mx_ms)
        achieved = mx_op["bytes"] / (avg_ms * 1e-3) / 1e9
        fmt_name = "e4m3" if mx_op["fmt"] == E4M3 else "e5m2"
        label = {"dq_mx_row": f"dequant_kernel<mx_row,{fmt_name},bf16>",
                 "mx_rule": f"mx_kernel<bf16,{fmt_name},both,rule+counts>",
                 "bw": f"blockwise_kernel<{fmt_name},1x128,both>",
                 "nvfp4": "amax_kernel+nvfp4_kernel<bf16>",
                 "qs_mx_row": f"qstats_lin_kernel<bf16,{fmt_name},mx_row>",
                 "mxlow": f"mxlow_kernel<bf16,{LOW_NAMES.get(mx_op.get('elem'), '')},both>",
                 "mmascale": "mma_scale_kernel (rowwise mx scales)"}.get(
                     mx_op["kind"], f"mx_kernel<bf16,{fmt_name},both>")
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "peak_source": peak_src, "kernel": label,
                    "algorithmic_bytes_per_launch": mx_op["bytes"], "avg_launch_us": round(avg_ms * 1e3, 3),
                    "launches_timed": len(mx_ms),
                    "traffic": kernel_traffic(args.workload)}
    cfg = dict(cfg)
    cfg["l2"] = f"{nsets} rotating buffer sets of {per_set / 2**20:.0f} MiB (> 4x L2 in total)"
    line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": cfg, "frac_of_hbm_peak": round(value / world / peak, 4), "roofline": roofline,
            "e2e": e2e, "gpu_launches": launches["n"], "clocks": clocks,
            "bytes_per_step": bytes_per_step}
    if any(op["kind"] == "mx_rule" for op in ops):
        line["saturated_elements"] = {("round_up" if op["rule"] == 0 else "ocp"): sets[0][j]["sat"].cpu().tolist()
                                      for j, op in enumerate(ops) if op["kind"] == "mx_rule"}
    if any(op["kind"] in QS_KINDS for op in ops):
        line["qstats"] = {}
        for j, op in enumerate(ops):
            if op["kind"] in QS_KINDS:
                d = fq.qstats_dict(sets[0][j]["st"])
                line["qstats"][op["kind"]] = {"sqnr_db": round(d["sqnr_db"], 4), "zero_rate": d["zero_rate"],
                                              "n_flushed": d["n_flushed"], "n_zero": d["n_zero"]}
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.workload)
    for st in states:
        if st is not None:
            st.close()
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
    for op in ops:
        r, c = op["shape"]
        rr = min(r, sample_rows)
        x = np.ascontiguousarray(host_input(op["gen"], (rr, c)))
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
        states.append(oracle.DelayedScaling(16, 1, 3, op["fmt"]) if op["kind"] == "delayed" else None)
    return xs, states


def sample_rows_for(workload):
    return {"activation": 256, "mx_8192": 128, "per_tensor_1024": 1024, "delayed_8192": 128, "linear_layer": 64,
            "moe": 32, "dequant_8192": 128, "mx_rules_4096": 256, "blockwise_8192": 128, "nvfp4_8192": 128,
            "qstats_8192": 128, "mxfp4_fp6_8192": 128, "mma_scales_8192": 1024}[workload]


def cpu_baseline(workload, budget_s=10.0):
    import oracle
    rows = sample_rows_for(workload)
    xs, states = oracle_inputs(workload, rows)
    oracle_sample_step(workload, rows, xs, states)  # warm
    t0 = time.perf_counter()
    n, total = 0, 0
    while time.perf_counter() - t0 < budget_s:
        total += oracle_sample_step(workload, rows, xs, states)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": round(total / dt / 1e9, 4), "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"first {rows} rows of each op's tensor, {n} repetitions in {dt:.1f} s"}


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
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
