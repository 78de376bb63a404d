#!/usr/bin/env python3
"""Throughput of one fused-MoE layer step on GB300 (tokens/s), with roofline.

A step is the whole hot path on one batch of synthetic input already resident
in HBM: moe_route -> moe_align -> moe_prepare -> moe_experts (+ the shared
expert when the layer has one) -> moe_finalize, all through the C ABI on one
stream.  Default workload: the DeepSeek-V3-like layer (T=4096, H=7168, I=2048,
E=256, top-8, fp8 G(128) experts + a bf16 shared expert), the largest
configuration that fits one GPU, whose 11.4 GB of expert weights stream from
HBM every step (far more than the 129 MB L2, so no flush is needed).  Workloads
whose step touches less than the L2 (the tiny layer, the finalize kernel alone)
rotate through copies of their inputs that together exceed 4x the L2, so no
step reads what an earlier step left in the L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

With N > 1 (launched by torch.distributed.run) every rank runs an independent
replica of the layer on its own GPU -- the layer has no exchange step on one
node -- and rank 0 prints the line: value = tokens of all ranks / max time.

`--impl reference` times the CPU oracle on the host cores instead (bounded
token samples per step); it is the slow, plain restatement of the method that
the GPU path is checked against, not a tuned baseline.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, make_inputs  # noqa: E402

METRIC = "MoE-layer tokens/s (fraction of GB300 HBM/tensor roofline in `roofline`), 1 GPU"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="deepseek", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-unit", action="store_true",
                    help="for ncu --profile-from-start off: warm up, run the dominant unit (the roofline's "
                         "kernel group) once between cudaProfilerStart and cudaProfilerStop, and exit")
    ap.add_argument("--profile-step", action="store_true", help="the same with one layer step")
    ap.add_argument("--no-graph", action="store_true", help="launch the step's calls one by one instead of "
                    "replaying them as one captured CUDA graph")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ roofline accounting
def experts_algorithmic(cfg, counts):
    """Bytes and FLOPs one expert pass must move/do: the weights of the experts
    that received tokens (+ fp8 block scales), the activations read once, the
    intermediate h written and read once, the output rows written once; FLOPs
    2 H I per weight matrix (3 gated, 2 for *_no_mul) per token slot (no padded rows).
    NVFP4: half a byte per code plus one scale byte per 16; h is stored in bf16,
    then as NVFP4 codes and scales, each written and read once."""
    mats = 2 if cfg.activation.endswith("_no_mul") else 3  # gate (+ up) and down projections
    S = cfg.T * cfg.top_k
    flops = 2.0 * mats * S * cfg.H * cfg.I
    if cfg.quant == "nvfp4":
        touched = int((counts > 0).sum())
        w = touched * mats * cfg.H * cfg.I * 9 // 16
        act = cfg.T * cfg.H * 9 // 16 + 2 * S * cfg.I * 2 + 2 * S * cfg.I * 9 // 16 + S * cfg.H * 2
        return w + act, flops
    fp8 = cfg.quant != "bf16"
    esz = 1 if fp8 else 2
    touched = int((counts > 0).sum())
    w = touched * mats * cfg.H * cfg.I * esz
    if fp8:
        w += touched * mats * (cfg.H // 128) * (cfg.I // 128) * 4
    S = cfg.T * cfg.top_k
    act = cfg.T * cfg.H * esz + 2 * S * cfg.I * esz + S * cfg.H * 2
    if cfg.quant == "fp8":
        act += cfg.T * (cfg.H // 128) * 4 + 2 * S * (cfg.I // 128) * 4
    elif fp8:  # per-token / per-tensor: per-row scales, and h also stored in bf16 and read back
        act += cfg.T * 4 + 2 * S * 4 + 2 * S * cfg.I * 2
    return w + act, flops


# nominal dense tensor rates relative to bf16 (2.25 / 4.5 / 13.5 PFLOP/s on a GB300)
TENSOR_RATIO = {"bf16": 1.0, "nvfp4": 6.0}


def tensor_ratio(quant):
    return TENSOR_RATIO.get(quant, 2.0)  # the fp8 formats: 2x


# kernel sources of each dominant unit (csrc/ files)
UNIT_SOURCES = {"experts": ["moe_experts.cu", "moe_common.cuh", "moe_route.cuh"],
                "fused": ["moe_experts.cu", "moe_common.cuh", "moe_route.cuh"],
                "finalize": ["moe_finalize.cu", "moe_common.cuh"]}


def graph_kernel_nodes(graph):
    """Kernel nodes of a captured step (the step calls only this library, so these
    are its launches), read from the graph through the CUDA runtime; None when
    the graph cannot be read."""
    try:
        import ctypes
        raw = graph.raw_cuda_graph()
        rt = ctypes.CDLL("libcudart.so.13")
        n = ctypes.c_size_t(0)
        if rt.cudaGraphGetNodes(ctypes.c_void_p(int(raw)), None, ctypes.byref(n)) != 0 or n.value == 0:
            return None
        nodes = (ctypes.c_void_p * n.value)()
        if rt.cudaGraphGetNodes(ctypes.c_void_p(int(raw)), nodes, ctypes.byref(n)) != 0:
            return None
        kernels = 0
        for node in nodes:
            t = ctypes.c_int(-1)
            if rt.cudaGraphNodeGetType(ctypes.c_void_p(node), ctypes.byref(t)) != 0:
                return None
            kernels += t.value == 0  # cudaGraphNodeTypeKernel
        return kernels
    except Exception:
        return None


_CODE_TOKENS = re.compile(r'"(?:\\.|[^"\\])*"|\'(?:\\.|[^\'\\])*\'|//[^\n]*|/\*.*?\*/', re.S)


def code_only(src: str) -> str:
    """C++/CUDA source without its comments and with whitespace runs collapsed: what
    a comment or formatting edit leaves unchanged."""
    kept = _CODE_TOKENS.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", src)
    return " ".join(kept.split())


def sources_digest(files) -> str:
    """sha256 over the code of the given csrc/ files (the unit's kernels and their
    helpers), comments and formatting excluded."""
    import hashlib
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "mixture_experts_layer_tokens_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(files):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + code_only(fh.read()).encode())
    return h.hexdigest()


def measured_traffic(workload: str, path: str = None):
    """DRAM bytes (read + write) of one dominant-unit call from the committed ncu
    capture (profiles/dram_traffic.json; for a workload too large to capture, the
    recorded scaling of a smaller case); None when there is none or the unit's
    kernel sources changed since."""
    path = path or os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            e = json.load(f)["workloads"][workload]
        if e["sources_sha256"] != sources_digest(UNIT_SOURCES[e["unit"]]):
            return None
        return int(e["bytes_per_call"])
    except Exception:
        return None


def finalize_algorithmic(cfg, nvfp4):
    T, H, k = cfg.T, cfg.H, cfg.top_k
    rd = T * k * H * 2 + 2 * T * H * 2 + H * 2 + T * k * 4
    wr = T * H // 2 + T * H // 16 if nvfp4 else T * H * 2
    return rd + wr


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Polls the SM clock and the clock-event reasons of one GPU through NVML
    (read-only queries) every ~2 ms from a thread, for the duration of a timed
    region."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index):
        import ctypes
        import threading
        self.samples, self.max_mhz, self.err = [], None, None
        self._stop = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(device_index)
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(h)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
                    raise RuntimeError("no NVML handle")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1 = SM clock
                self.max_mhz = mx.value
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nv, self.h, self.reasons_fn = nv, h, reasons_fn
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        except Exception as e:  # no NVML on this machine
            self.err, self.thread = str(e), None

    def _run(self):
        import ctypes
        c, r = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            ok = self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0
            okr = self.reasons_fn(self.h, ctypes.byref(r)) == 0
            if ok:
                self.samples.append((c.value, r.value if okr else 0))
            time.sleep(0.002)

    def stop(self):
        if self.thread is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": self.err}
        self._stop.set()
        self.thread.join()
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        mask = 0
        for _, r in self.samples:
            mask |= r
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASONS.items() if mask & b), "samples": len(self.samples)}


# ------------------------------------------------------------------ oracle baseline
def oracle_tokens_seconds(inp, tokens):
    """Time the plain CPU oracle on the given tokens of the workload (fp64)."""
    from oracle import moe_ref
    cfg = inp.cfg
    t0 = time.perf_counter()
    logits = inp.logits[tokens].cpu()
    if cfg.scoring == "sigmoid":
        ids, w = moe_ref.route_sigmoid_top1(logits)
    else:
        ids, w = moe_ref.route_softmax_renorm(logits, cfg.top_k)
    a1 = inp.a1[tokens].cpu()
    if cfg.quant == "nvfp4":
        x = inp.extra
        a1q, sc = moe_ref.prepare_nvfp4(a1, w, cfg.weight_on_input, x["a1_gscale"])
        y = moe_ref.experts_nvfp4(a1q, sc, x["a1_gscale"], inp.w13.cpu(), inp.w13_scale.cpu(), x["w13_gscale"].cpu(),
                                  inp.w2.cpu(), inp.w2_scale.cpu(), x["w2_gscale"].cpu(), x["h_gscale"],
                                  moe_ref.align(ids, cfg.E, 128), cfg.top_k, cfg.activation)
    elif cfg.quant == "fp8_tensor":  # one intermediate scale over every expert's rows of the sample
        a1q, sc = moe_ref.prepare(a1, w, cfg.weight_on_input, cfg.quant)
        y = moe_ref.experts(a1q, sc, inp.w13, inp.w13_scale, inp.w2, inp.w2_scale, moe_ref.align(ids, cfg.E, 128),
                            cfg.top_k, cfg.quant, cfg.activation)
    else:
        a1q, sc = moe_ref.prepare(a1, w, cfg.weight_on_input, cfg.quant)
        y = torch.cat([moe_ref.token_expert_rows(a1q, sc, inp.w13, inp.w13_scale, inp.w2, inp.w2_scale, ids, i,
                                                 cfg.quant, cfg.activation) for i in range(len(tokens))], 0)
    shared = moe_ref.dense_mlp(a1, inp.shared_w13[0], inp.shared_w2[0]) if cfg.shared_I else None
    res = inp.residual[tokens].cpu() if inp.residual is not None else None
    moe_ref.finalize(y, w, cfg.top_k, cfg.weight_on_input, shared=shared, residual=res,
                     rms_weight=None if inp.rms_weight is None else inp.rms_weight.cpu())
    return time.perf_counter() - t0


def set_cpu_threads():
    try:
        n = len(os.sched_getaffinity(0))
    except Exception:
        n = os.cpu_count() or 1
    torch.set_num_threads(n)
    return n


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


# ------------------------------------------------------------------ distributed plumbing
def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "gb300" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


L2_BYTES = 129e6  # GB300 L2 (the device attribute is used when a GPU is present)


def l2_bytes():
    try:
        if torch.cuda.is_available():
            return float(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        pass
    return L2_BYTES


def step_bytes_estimate(cfg):
    """Bytes one step touches, from the configuration alone (every expert counted as
    touched): what decides whether the timed steps need rotating input sets."""
    if cfg.finalize_only:
        return finalize_algorithmic(cfg, True) + cfg.T * cfg.H * 2
    mats = 2 if cfg.activation.endswith("_no_mul") else 3
    esz = {"bf16": 2.0, "nvfp4": 9 / 16}.get(cfg.quant, 1.0)
    w = cfg.E * mats * cfg.H * cfg.I * esz + 3 * cfg.H * cfg.shared_I * 2
    return w + cfg.T * cfg.H * 2 * 3 + cfg.T * cfg.top_k * cfg.H * 2


def rotation_sets(cfg):
    """1 when a step touches more than the L2; otherwise the number of input sets,
    each a copy of the step's inputs, weights and outputs, that together exceed 4x the
    L2 (the timed steps cycle through them)."""
    est = step_bytes_estimate(cfg)
    l2 = l2_bytes()
    return 1 if est > l2 else int(math.ceil(4.0 * l2 / est)) + 1


def l2_note(cfg, nsets):
    est = step_bytes_estimate(cfg)
    if nsets == 1:
        return f"no flush: each step touches ~{est / 1e9:.2f} GB (more than the {l2_bytes() / 1e6:.0f} MB L2)"
    return (f"rotating inputs: {nsets} copies of the step's inputs, weights and outputs (~{est / 1e6:.0f} MB "
            f"each, {nsets * est / 1e6:.0f} MB in all, > 4x the {l2_bytes() / 1e6:.0f} MB L2), one per step in turn")


def clone_inputs(inp):
    """A copy of every tensor of a workload's inputs (same values, other memory)."""
    from mixture_experts_layer_tokens_gb300.inputs import LayerInputs
    cl = lambda v: v.clone() if isinstance(v, torch.Tensor) else v
    d = {k: cl(v) for k, v in inp.__dict__.items() if k != "extra"}
    d["extra"] = {k: cl(v) for k, v in inp.extra.items()}
    return LayerInputs(**d)


def measure_fp8_peak(dev):
    """Dense fp8 (E4M3 x E4M3, fp32 accumulate, bf16 out) throughput of cuBLASLt through
    torch._scaled_mm at 8192^3 on this GPU, timed with CUDA events: best of 10 (burst)
    and back to back for about 2 s (sustained).  None when the call is unavailable."""
    try:
        N = 8192
        a = torch.randn(N, N, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(N, N, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.ones((), device=dev)
        mm = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(5):
            mm()
        torch.cuda.synchronize(dev)
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mm()
            e1.record()
            torch.cuda.synchronize(dev)
            best = min(best, e0.elapsed_time(e1))
        n, t0 = 0, time.time()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        while time.time() - t0 < 2.0:
            for _ in range(20):
                mm()
            n += 20
            torch.cuda.synchronize(dev)
        e1.record()
        torch.cuda.synchronize(dev)
        flop = 2.0 * N ** 3
        del a, b
        return {"burst_tflops": round(flop / (best * 1e-3) / 1e12, 1),
                "sustained_tflops": round(flop * n / (e0.elapsed_time(e1) * 1e-3) / 1e12, 1),
                "how": "torch._scaled_mm e4m3 x e4m3 -> bf16, 8192^3, CUDA events: best of 10; back to back ~2 s"}
    except Exception:
        return None


def common_config(cfg, ws, nsets):
    """The `config` object of both arms' lines (the workload, not how it ran)."""
    return {"workload": cfg.description, "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "top_k": cfg.top_k,
            "parallelism": f"replicas{ws}", "l2": l2_note(cfg, nsets)}


# ------------------------------------------------------------------ reference arm
def run_reference(args, ws, rank):
    if rank != 0:
        return
    cfg = CONFIGS[args.workload]
    cores = set_cpu_threads()
    inp = make_inputs(cfg, device="cpu")
    per_step = 1
    times = []
    for i in range(args.warmup + args.steps):
        tok = [(i * 7) % cfg.T]
        dt = oracle_tokens_seconds(inp, tok)
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = per_step * len(times) / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": common_config(cfg, args.gpus, rotation_sets(cfg)),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} token of the {cfg.name} workload per step (fp64 oracle), "
                                       f"CPU {cpu_model()}"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def run_gpu(args, ws, rank, local):
    from mixture_experts_layer_tokens_gb300 import build as _b
    from mixture_experts_layer_tokens_gb300 import moe
    from mixture_experts_layer_tokens_gb300.layer import FinalizeStep, MoELayer

    if rank == 0:
        _b.build()
    barrier(ws)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = CONFIGS[args.workload]
    inp = make_inputs(cfg, seed=rank, device=dev)
    # small working sets: copies of the inputs, one per step in turn (see rotation_sets)
    nsets = rotation_sets(cfg)
    sets = [inp] + [clone_inputs(inp) for _ in range(nsets - 1)]
    stream = torch.cuda.Stream(device=dev)
    hbm_peak, bf16_peak, peak_kind = peaks()

    with torch.cuda.stream(stream):
        if cfg.finalize_only:
            step_objs = [FinalizeStep(x) for x in sets]
            for so in step_objs:
                so.weights()

            def make_step(so):
                def step():
                    so.weights()
                    so.finalize(True)
                return step
            steps = [make_step(so) for so in step_objs]
            launches_per_step = 2  # estimate; replaced by the captured graph's kernel count
        else:
            layers = [MoELayer(x, stream=stream) for x in sets]
            layer = layers[0]

            def make_step(ly, x):
                def step():
                    ly.forward(x.logits, x.a1)
                return step
            steps = [make_step(ly, x) for ly, x in zip(layers, sets)]
            # estimate (route, align, prepare, plan + gather + 2 GEMMs, finalize); replaced by
            # the captured graph's kernel count when the graph can be read
            launches_per_step = 1 + 1 + (0 if layer.passthrough else 1) + 4 + 1
        for i in range(max(args.warmup, nsets)):
            steps[i % nsets]()
        torch.cuda.synchronize(dev)
        assert moe.moe_device_status() == moe.MOE_OK

        # the dominant unit: the kernel group the roofline reports (one call per input set)
        if cfg.finalize_only:
            dom_name = "moe_finalize (NVFP4 out)"
            nbytes = finalize_algorithmic(cfg, True)
            flops = 0.0
            for so in step_objs:
                so.weights()
            dom_calls = [(lambda so=so: so.finalize(True)) for so in step_objs]
        else:
            # the routed experts and, when the layer has one, the shared expert (one
            # moe_experts_multi call when they share launches, else two calls)
            dom_name = (f"moe_experts (plan + gather + GEMM1 {cfg.activation} + GEMM2 scatter)"
                        + ("" if not cfg.shared_I else
                           " + shared expert" + (" in the same launches" if layer.fused_shared else "")))
            for st in steps:
                st()  # route/align/prepare state for the experts calls
            if layer.single:
                counts = torch.bincount(layer.topk_ids.reshape(-1).long(), minlength=cfg.E).cpu().numpy()
            else:
                counts = torch.diff(layer.al.expert_offsets).cpu().numpy()
            nbytes, flops = experts_algorithmic(cfg, counts)
            if cfg.shared_I:
                nbytes += 3 * cfg.H * cfg.shared_I * 2 + 2 * cfg.T * cfg.H * 2 + 2 * cfg.T * cfg.shared_I * 2
                flops += 6.0 * cfg.T * cfg.H * cfg.shared_I

            def make_dom(ly, x):
                a1q = x.a1 if ly.passthrough else ly.a1q
                if ly.single:
                    return lambda: ly.forward(x.logits, x.a1)
                return lambda: ly.experts(a1q, ly.a1q_scale, x.a1)
            dom_calls = [make_dom(ly, x) for ly, x in zip(layers, sets)]
            if layer.single:
                # one launch is the whole step: the experts' bytes plus the router logits and the
                # finalize's reads (expert rows, shared row, residual) and its output
                dom_name = ("moe_layer_fused (route, align, prepare, experts"
                            + (" + shared expert" if cfg.shared_I else "") + ", finalize: one launch)")
                S = cfg.T * cfg.top_k
                nbytes += cfg.T * cfg.E * 4 + S * cfg.H * 2 + cfg.T * cfg.H * 2 * (
                    1 + (cfg.shared_I > 0) + (inp.residual is not None))
        if args.profile_unit or args.profile_step:
            # one call between profiler start and stop (ncu --profile-from-start off), then exit
            (dom_calls[0] if args.profile_unit else steps[0])()
            torch.cuda.synchronize(dev)
            torch.cuda.profiler.start()
            (dom_calls[0] if args.profile_unit else steps[0])()
            torch.cuda.synchronize(dev)
            torch.cuda.profiler.stop()
            assert moe.moe_device_status() == moe.MOE_OK
            if rank == 0:
                print(json.dumps({"profiled": "unit" if args.profile_unit else "step", "workload": cfg.name,
                                  "kernel": dom_name}), flush=True)
            return
        graphs = None
        launches_counted = False
        if not args.no_graph:
            # each set's step captured once and replayed: same kernels, no per-call host work
            graphs = []
            for st in steps:
                try:
                    g = torch.cuda.CUDAGraph(keep_graph=True)
                except TypeError:
                    g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    st()
                graphs.append(g)
            counted = graph_kernel_nodes(graphs[0])
            if counted:
                launches_per_step = counted
                launches_counted = True
            for g in graphs:
                if hasattr(g, "instantiate"):
                    g.instantiate()
            for _ in range(3):
                for g in graphs:
                    g.replay()
            torch.cuda.synchronize(dev)
            assert moe.moe_device_status() == moe.MOE_OK
        run_steps = [g.replay for g in graphs] if graphs is not None else steps

        # ---- timed region: K steps (input set i % nsets at step i), events on the launching stream
        clocks = ClockSampler(local) if rank == 0 else None
        barrier(ws)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            run_steps[i % nsets]()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(ws)
        clk = clocks.stop() if clocks else None
        ms = e0.elapsed_time(e1) / args.steps
        ms_max = max_over_ranks(ms, ws, dev)
        value = ws * cfg.T / (ms_max * 1e-3)

        # ---- dominant unit: R back-to-back calls (cycling through the input sets) captured in
        # one graph, replayed; CUDA events on the launching stream give the device time per call
        R = nsets * max(1, math.ceil(10 / nsets))
        for c in dom_calls:
            c()
        torch.cuda.synchronize(dev)
        reps = max(1, args.steps // R)
        if args.no_graph:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(reps * R):
                dom_calls[i % nsets]()
            b.record(stream)
        else:
            dom_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(dom_graph, stream=stream):
                for i in range(R):
                    dom_calls[i % nsets]()
            dom_graph.replay()
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                dom_graph.replay()
            b.record(stream)
        torch.cuda.synchronize(dev)
        dom_ms = a.elapsed_time(b) / (reps * R)
        # the binding roof: HBM bytes or tensor FLOPs.  fp8: the measured fp8 peak of this GPU
        # (torch._scaled_mm) when it can be taken, else the measured bf16 peak x the nominal 2x;
        # NVFP4: measured bf16 x the nominal 6x
        fp8_peak = measure_fp8_peak(dev) if cfg.quant.startswith("fp8") else None
        if fp8_peak:
            tensor_peak = fp8_peak["burst_tflops"]
            tensor_kind = "measured fp8 (this run, burst: " + fp8_peak["how"] + ")"
        else:
            tensor_peak = bf16_peak * tensor_ratio(cfg.quant)
            tensor_kind = peak_kind + ("" if cfg.quant == "bf16" else
                                       f" bf16 x{tensor_ratio(cfg.quant):g} (nominal {cfg.quant}:bf16)")
        t_hbm = nbytes / (hbm_peak * 1e9)
        t_tensor = flops / (tensor_peak * 1e12) if flops else 0.0
        if t_tensor > t_hbm:
            achieved = flops / (dom_ms * 1e-3) / 1e12
            roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(tensor_peak, 1),
                        "unit": "TFLOP/s", "frac": round(achieved / tensor_peak, 4),
                        "traffic": measured_traffic(cfg.name),
                        "kernel": dom_name, "algorithmic_flops": flops, "ms": round(dom_ms, 4),
                        "peak_kind": tensor_kind}
            roofline["hbm_gbs"] = round(nbytes / (dom_ms * 1e-3) / 1e9, 1)
        else:
            achieved = nbytes / (dom_ms * 1e-3) / 1e9
            roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                        "frac": round(achieved / hbm_peak, 4), "traffic": measured_traffic(cfg.name),
                        "kernel": dom_name,
                        "algorithmic_bytes": int(nbytes), "ms": round(dom_ms, 4), "peak_kind": peak_kind}
            if flops:
                roofline["tflops"] = round(flops / (dom_ms * 1e-3) / 1e12, 1)
                roofline["tensor_frac"] = round(flops / (dom_ms * 1e-3) / 1e12 / tensor_peak, 4)
                roofline["tensor_peak_kind"] = tensor_kind
        if fp8_peak:
            roofline["fp8_peak_sustained"] = fp8_peak["sustained_tflops"]
            roofline["fp8_peak_nominal_ratio"] = round(bf16_peak * tensor_ratio(cfg.quant), 1)

        # ---- end to end through the public API with host buffers
        if cfg.finalize_only:
            e2e = None
        else:
            # Every step copies its inputs from pinned host memory and reads its output
            # back, as a serving loop does; the loop is pipelined like one: inputs and
            # outputs are double-buffered and the copies run on their own streams, so step
            # i's upload and step i-1's download overlap the neighbouring steps' compute.
            h_logits = inp.logits.cpu().pin_memory()
            h_a1 = inp.a1.cpu().pin_memory()
            h_out = [torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
            d_logits = [torch.empty_like(inp.logits) for _ in range(2)]
            d_a1 = [torch.empty_like(inp.a1) for _ in range(2)]
            d_out = [torch.empty_like(layer.out) for _ in range(2)]
            up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
            ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer b uploaded
            ev_done = [torch.cuda.Event() for _ in range(2)]  # the step on buffer b computed
            ev_out = [torch.cuda.Event() for _ in range(2)]   # output of buffer b downloaded
            layer_out = layer.out
            e2e_graphs = [None, None]
            if not args.no_graph:
                for bb in range(2):
                    layer.out = d_out[bb]
                    e2e_graphs[bb] = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(e2e_graphs[bb], stream=stream):
                        layer.forward(d_logits[bb], d_a1[bb])
                layer.out = layer_out

            def e2e_step(i):
                bb = i % 2
                up.wait_event(ev_done[bb])                # step i-2 has read this buffer's inputs
                with torch.cuda.stream(up):
                    d_logits[bb].copy_(h_logits, non_blocking=True)
                    d_a1[bb].copy_(h_a1, non_blocking=True)
                ev_in[bb].record(up)
                stream.wait_event(ev_in[bb])
                stream.wait_event(ev_out[bb])             # step i-2's output has been read back
                if e2e_graphs[bb] is not None:
                    e2e_graphs[bb].replay()
                else:
                    layer.out = d_out[bb]
                    layer.forward(d_logits[bb], d_a1[bb])
                    layer.out = layer_out
                ev_done[bb].record(stream)
                down.wait_event(ev_done[bb])
                with torch.cuda.stream(down):
                    h_out[bb].copy_(d_out[bb], non_blocking=True)
                ev_out[bb].record(down)

            for i in range(args.warmup):
                e2e_step(i)
            torch.cuda.synchronize(dev)
            barrier(ws)
            t0 = time.perf_counter()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            up.wait_event(a)
            for i in range(args.steps):
                e2e_step(i)
            stream.wait_event(ev_out[(args.steps - 1) % 2])  # the last output is on the host
            b.record(stream)
            torch.cuda.synchronize(dev)
            wall = (time.perf_counter() - t0) / args.steps
            ems = max(a.elapsed_time(b) / args.steps, wall * 1e3)
            ems = max_over_ranks(ems, ws, dev)
            e2e = {"value": ws * cfg.T / (ems * 1e-3), "unit": "tokens/s",
                   "h2d_bytes_per_step": h_logits.numel() * 4 + h_a1.numel() * 2,
                   "d2h_bytes_per_step": h_out[0].numel() * 2, "copies": "pipelined (double-buffered, own streams)"}

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and ws == 1 and not cfg.finalize_only:
        cores = set_cpu_threads()
        # tokens one at a time until about 10 s of oracle work (at least 2 tokens)
        dt, n = 0.0, 0
        while (dt < 10.0 or n < 2) and n < cfg.T:
            dt += oracle_tokens_seconds(inp, [(n * 37) % cfg.T])
            n += 1
        cpu = {"value": n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} tokens of the {cfg.name} workload, one at a time, through the fp64 oracle "
                         f"({dt:.1f} s), CPU {cpu_model()}"}
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": {"bf16": "bf16", "nvfp4": "nvfp4"}.get(cfg.quant, "fp8"),
            "data": "synthetic",
            "config": common_config(cfg, ws, nsets),
            "launch": {"mode": "cuda_graph" if not args.no_graph else "eager",
                       "gpu_launches_per_step": launches_per_step,
                       "gpu_launches_from": "captured graph's kernel nodes" if launches_counted else "estimate"},
            "roofline": roofline, "cpu_baseline": cpu, "clocks": clk, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_gpu(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
