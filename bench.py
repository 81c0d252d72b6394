#!/usr/bin/env python
"""Throughput of the fused MoE-LoRA layer (route + forward) on GB300.

One step = one layer call on one batch: top-k routing, align, row gather,
the two grouped GEMMs with their adapter shrink/expand, SwiGLU and the
weighted combine, replayed from a CUDA graph with every input resident in
HBM.  L2 is flushed before every timed step (256 MiB written, then another
256 MiB read, so no dirty lines are left for the step); each step is
timed with CUDA events on the stream it runs on, and the per-stage events
recorded inside the graph give each kernel's duration.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on the host cores instead (a bounded token sample per step).

Multi-GPU: launched under torchrun, every rank runs its own replica of the
layer on its own batch (tokens are independent, no collective on the data
path); the step time is the max over ranks and the value counts the tokens
of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from moe_layer_lora_gb300 import workloads as wl  # noqa: E402

METRIC = "MoE-LoRA layer tokens/s; % HBM roofline (decode), % bf16 TC peak (prefill)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------------ helpers --

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("mlora", "reference"), default="mlora")
    ap.add_argument("--workload", choices=wl.WORKLOADS, default="decode")
    ap.add_argument("--M", type=int, default=None, help="override the token count")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU work of the oracle baseline")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of replaying a graph")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload breakdown that follows the headline measurement")
    ap.add_argument("--mxfp8", action="store_true", help="the layer with MXFP8 expert weights")
    return ap.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(value: float, world: int, device) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(step_ms, tokens_per_rank: int, world: int, device):
    """Whole-job throughput: the slowest rank's total time over the tokens
    every rank processed (weak scaling: each rank runs its own batch)."""
    total_ms = reduce_max(float(sum(step_ms)), world, device)
    steps = len(step_ms)
    ms_per_step = total_ms / steps
    return total_ms, ms_per_step, tokens_per_rank * world / (ms_per_step / 1e3)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def workload_config(s: wl.Spec) -> dict:
    d = {"workload": f"{s.name}: M={s.M} H={s.H} I={s.I} E={s.E}" + (f"+{s.n_shared} shared" if s.n_shared else "")
         + f" top_k={s.top_k} {'softmax' if s.scoring == 0 else 'sigmoid+bias'}"
         + (f" L={s.L} r={s.r} ({s.lora_mode})" if s.has_lora else " no adapters"),
         "M": s.M, "H": s.H, "I": s.I, "E_tot": s.E_tot, "top_k": s.top_k, "n_shared": s.n_shared,
         "L": s.L, "rank": s.r, "scaling": s.scaling}
    return d


def algorithmic(s: wl.Spec, ids: np.ndarray, idx, mx: bool = False) -> dict:
    """Bytes each stage must move and flops it must do, from the routed ids:
    every touched expert's weights once (bf16, or MXFP8: one byte an element
    plus one scale byte per 32), every touched (adapter, expert) pair's four
    LoRA matrices once, the activations once."""
    M, H, I, r = s.M, s.H, s.I, s.r
    S = ids.size
    experts = np.unique(ids)
    n_exp = int(experts.size)
    lora = s.has_lora and idx is not None
    if lora:
        l_slot = np.repeat(np.asarray(idx), ids.shape[1])
        has = l_slot >= 0
        pairs = np.unique(l_slot[has].astype(np.int64) * s.E_tot + ids.reshape(-1)[has])
        n_pairs, a_slots = int(pairs.size), int(has.sum())
    else:
        n_pairs = a_slots = 0
    b = 2  # bf16
    bw = 1 + 1 / 32 if mx else b  # bytes of an expert weight element
    st = {
        # the experts kernel: both projections, their adapter shrink and expand
        "experts": dict(bytes=n_exp * 3 * I * H * bw + n_pairs * r * (2 * H + 3 * I) * b + S * (2 * H + 2 * I) * b,
                        flops=2.0 * S * 3 * H * I + 2.0 * a_slots * r * (2 * H + 3 * I)),
        "gather": dict(bytes=S * H * b * 2, flops=0.0),
        "combine": dict(bytes=S * H * 4 + M * H * b, flops=2.0 * S * H),
        "align": dict(bytes=S * 4 * 3, flops=0.0),
    }
    layer_bytes = (n_exp * 3 * I * H * bw + n_pairs * r * (2 * H + 3 * I) * b + 2 * M * H * b
                   + M * s.E * 4 + S * 8)
    layer_flops = sum(v["flops"] for v in st.values())
    return {"stages": st, "layer_bytes": layer_bytes, "layer_flops": layer_flops, "experts": n_exp,
            "pairs": n_pairs, "adapter_slots": a_slots}


class L2Flush:
    """Evicts L2 between timed steps: writes a 256 MiB buffer (larger than
    L2), then reads a second one, so the write-backs of the first happen
    here and L2 is left holding clean, unrelated lines."""

    def __init__(self, device):
        self.a = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.b = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=device)
        self.out = torch.empty((), dtype=torch.int64, device=device)

    def __call__(self):
        self.a.fill_(1)
        torch.sum(self.b, (0,), dtype=torch.int64, out=self.out)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed
    region (absent tool: no record)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


STAGE_SOURCES = {
    "experts": ("gemm.cu", "ptx.cuh", "internal.cuh"),
}


def kernel_source_hash(stage: str) -> str:
    """Hash of the sources a stage's kernel is built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_layer_lora_gb300", "csrc")
    for name in STAGE_SOURCES.get(stage, sorted(os.listdir(csrc))):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(stage: str, workload: str):
    """DRAM bytes per launch of `stage` on the named workload (its default
    size) from a committed ncu summary, when that summary was taken on the
    current kernel sources (else None).  A summary covers one workload
    (profiles/<stage>_<workload>.md, "dram bytes per launch: `v`") or
    several (any profiles/<stage>_*.md, "dram bytes per launch (<workload>): `v`")."""
    pdir = os.path.join(ROOT, "profiles")
    own = f"{stage}_{workload}.md"
    names = [own] + sorted(n for n in os.listdir(pdir) if n.startswith(stage + "_") and n != own)
    for name in names:
        try:
            text = open(os.path.join(pdir, name)).read()
        except OSError:
            continue
        key = r"dram bytes per launch:" if name == own else r"dram bytes per launch \(" + re.escape(workload) + r"\):"
        m_val = re.search(key + r"[\s|`]*([0-9.eE+]+)", text)
        if not m_val:
            continue
        m_hash = re.search(r"kernel source hash:[\s|`]*([0-9a-f]{16})", text)
        if not m_hash or m_hash.group(1) != kernel_source_hash(stage):
            return None
        return float(m_val.group(1))
    return None


# --------------------------------------------------------------- CPU oracle --

def oracle_sample(inp, n_tokens: int, hb=None):
    """The oracle's route + forward of the first n_tokens tokens (the step
    the GPU arm times, on a bounded sample); returns (seconds, tokens)."""
    import oracle
    s = inp.spec
    rows = np.arange(min(n_tokens, s.M))
    hb = hb or host_bits(inp)
    lora = s.has_lora
    t0 = time.perf_counter()
    ids, w = oracle.moe_route(inp.logits.numpy()[rows], None if inp.bias is None else inp.bias.numpy(), s.top_k,
                              s.scoring, s.renormalize, s.n_shared, s.routed_scaling_factor)
    oracle.moe_forward(hb["x"][rows], hb["w13"], hb["w2"], hb["A13"], hb["B13"], hb["A2"], hb["B2"],
                       inp.token_lora_idx.numpy()[rows] if lora else None, ids, w.astype(np.float32), s.scaling,
                       s.out_scale)
    return time.perf_counter() - t0, len(rows)


def host_bits(inp):
    """Host bf16 bit arrays of the layer's tensors (copied once)."""
    b = wl.bits
    lora = inp.spec.has_lora
    return {"x": b(inp.x), "w13": b(inp.w13), "w2": b(inp.w2), "A13": b(inp.A13) if lora else None,
            "B13": b(inp.B13) if lora else None, "A2": b(inp.A2) if lora else None,
            "B2": b(inp.B2) if lora else None}


def cpu_baseline(inp, target_s: float):
    """The oracle as it stands on the host cores (route + forward), on a
    bounded token sample sized to roughly target_s seconds of work."""
    import oracle
    s = inp.spec
    oracle.load()
    hb = host_bits(inp)
    cores = os.cpu_count() or 1
    n = min(s.M, cores)
    dt, n = oracle_sample(inp, n, hb)
    if dt < target_s / 3 and n < s.M:
        n2 = int(min(s.M, max(n, n * target_s / max(dt, 1e-3))) // max(1, min(cores, n)) * min(cores, n))
        n2 = max(n, min(s.M, n2))
        if n2 > n:
            dt, n = oracle_sample(inp, n2, hb)
    # a whole batch that takes well under the target is timed over several
    # passes, so that the figure is not one short run
    passes = 1
    if dt < target_s / 3:
        passes = int(min(50, max(1, target_s / max(dt, 1e-3) - 1)))
        for _ in range(passes - 1):
            dt_i, _ = oracle_sample(inp, n, hb)
            dt += dt_i
    return {"value": n * passes / dt, "unit": "tokens/s", "cores": min(cores, n), "kind": "oracle",
            "sample": f"route + forward of the first {n} of the {s.M} tokens of the {s.name} batch, {passes} "
                      f"fp64 pass{'es' if passes > 1 else ''} ({dt:.1f} s)",
            "seconds": dt}


# ---------------------------------------------------------------- GPU path --

# The workloads timed after the headline (the default run reports all of
# them): label -> (workload name, spec overrides).  "stress_all_none" is
# the adapter-stress batch with every token's adapter id at -1, the early
# exit of a layer whose adapters are given but unused.
SWEEP = (
    ("tiny", "tiny", {}),
    ("decode", "decode", {}),
    ("prefill", "prefill", {}),
    ("shared_M1", "shared", {"M": 1}),
    ("shared_M32", "shared", {"M": 32}),
    ("shared_M128", "shared", {"M": 128}),
    ("stress", "stress", {}),
    ("stress_all_none", "stress", {"lora_mode": "all_none"}),
    # the same layers with MXFP8 expert weights (E4M3, one E8M0 scale per 32)
    ("decode_mxfp8", "decode", {"mx": True}),
    ("prefill_mxfp8", "prefill", {"mx": True}),
    ("shared_M1_mxfp8", "shared", {"M": 1, "mx": True}),
    ("shared_M128_mxfp8", "shared", {"M": 128, "mx": True}),
    ("stress_mxfp8", "stress", {"mx": True}),
)


class LayerRun:
    """One workload's layer on one device: its inputs resident in HBM, the
    step (route + forward on a side stream), and CUDA graphs of the step --
    a plain one and one with event nodes at the stage boundaries."""

    def __init__(self, s: wl.Spec, device, use_graph: bool, packed: bool = False, mx: bool = False):
        import moe_layer_lora_gb300 as ml
        self.ml = ml
        self.s = s
        self.mx = mx
        self.device = device
        inp = wl.make(s, device=device)
        self.inp = inp
        d = {k: (None if v is None else v.to(device)) for k, v in dict(
            logits=inp.logits, bias=inp.bias, x=inp.x, w13=inp.w13, w2=inp.w2, A13=inp.A13, B13=inp.B13,
            A2=inp.A2, B2=inp.B2, idx=inp.token_lora_idx).items()}
        self.in_bytes = 0
        if packed:
            # the per-step inputs (x, router logits, adapter ids) live in one
            # device buffer with a pinned host twin, so the end-to-end step
            # brings them over in one copy
            parts = [("x", inp.x), ("logits", inp.logits)] + ([("idx", inp.token_lora_idx)] if s.has_lora else [])
            offs = {}
            for name, t in parts:
                offs[name] = self.in_bytes
                self.in_bytes += (t.numel() * t.element_size() + 255) // 256 * 256
            self.h_in = torch.empty(self.in_bytes, dtype=torch.uint8).pin_memory()
            self.d_in = torch.empty(self.in_bytes, dtype=torch.uint8, device=device)
            for name, t in parts:
                nb = t.numel() * t.element_size()
                self.h_in[offs[name]:offs[name] + nb].copy_(t.contiguous().reshape(-1).view(torch.uint8))
                d[name] = self.d_in[offs[name]:offs[name] + nb].view(t.dtype).view(t.shape)
            self.d_in.copy_(self.h_in)
        self.d = d
        L, r = (s.L, s.r) if s.has_lora else (0, 0)
        self.ids = torch.empty((s.M, s.K_total), dtype=torch.int32, device=device)
        self.w = torch.empty((s.M, s.K_total), dtype=torch.float32, device=device)
        self.y = torch.empty((s.M, s.H), dtype=torch.bfloat16, device=device)
        if mx:
            # the weights are quantized once, outside every timed region
            self.q = ml.mlora_mxfp8_quantize_weights(d["w13"], d["w2"])
            torch.cuda.synchronize(device)
            d["w13"] = d["w2"] = None
            wsb = ml.mlora_moe_workspace_size_mxfp8(s.M, s.H, s.I, s.E_tot, s.K_total, L, r)
        else:
            wsb = ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, L, r)
        self.ws = torch.empty(wsb, dtype=torch.uint8, device=device)
        self.stream = torch.cuda.Stream(device=device)
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(ml.STAGE_EVENTS)]
        for e in self.ev:
            e.record(self.stream)  # creates the event handles
        ml.mlora_set_stage_events(None)
        with torch.cuda.stream(self.stream):
            self.step()
            self.stream.synchronize()
            status = ml.mlora_moe_read_status(self.ws, stream=self.stream)
            if status != 0:
                raise RuntimeError(f"{s.name}: device status {status:#x} after the first step")
            self.plain = self.inst = None
            if use_graph:
                self.plain = torch.cuda.CUDAGraph()
                with torch.cuda.graph(self.plain, stream=self.stream):
                    self.step()
                ml.mlora_set_stage_events(self.ev)
                try:
                    self.inst = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(self.inst, stream=self.stream):
                        self.step()
                finally:
                    ml.mlora_set_stage_events(None)

    def step(self):
        s, d, ml = self.s, self.d, self.ml
        ml.mlora_moe_route(d["logits"], d["bias"], s.top_k, s.scoring, s.renormalize, s.n_shared,
                           s.routed_scaling_factor, topk_ids=self.ids, topk_w=self.w, stream=self.stream)
        if self.mx:
            ml.mlora_moe_forward_mxfp8(d["x"], *self.q, d["A13"], d["B13"], d["A2"], d["B2"], d["idx"], self.ids,
                                       self.w, s.scaling, s.n_shared, s.out_scale, y=self.y, workspace=self.ws,
                                       stream=self.stream)
            return
        ml.mlora_moe_forward(d["x"], d["w13"], d["w2"], d["A13"], d["B13"], d["A2"], d["B2"], d["idx"], self.ids,
                             self.w, s.scaling, s.n_shared, s.out_scale, y=self.y, workspace=self.ws,
                             stream=self.stream)

    def run_plain(self):
        if self.plain is not None:
            self.plain.replay()
        else:
            self.step()

    def run_inst(self):
        if self.inst is not None:
            self.inst.replay()
        else:
            self.ml.mlora_set_stage_events(self.ev)
            try:
                self.step()
            finally:
                self.ml.mlora_set_stage_events(None)

    def alg(self):
        return algorithmic(self.s, self.ids.cpu().numpy(),
                           self.inp.token_lora_idx.numpy() if self.s.has_lora else None, self.mx)

    def time(self, flush, steps: int, warmup: int, world: int = 1, clocks=None):
        """W warm-up steps, then K timed steps of the plain graph and K of the
        instrumented one, each after an L2 flush and bracketed by events on
        the layer's stream."""
        ml = self.ml
        st0 = torch.cuda.Event(enable_timing=True)
        st1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            for _ in range(warmup):
                flush()
                self.run_plain()
                flush()
                self.run_inst()
            self.stream.synchronize()
            barrier(world)
            torch.cuda.synchronize(self.device)
            step_ms, inst_ms, stage_ms = [], [], {n: [] for n in ml.STAGE_NAMES}
            if clocks is not None:
                clocks.__enter__()
            try:
                for _ in range(steps):
                    flush()
                    st0.record(self.stream)
                    self.run_plain()
                    st1.record(self.stream)
                    self.stream.synchronize()
                    step_ms.append(st0.elapsed_time(st1))
                torch.cuda.synchronize(self.device)
                barrier(world)
                # per-kernel times: as many steps of the instrumented graph
                for _ in range(steps):
                    flush()
                    st0.record(self.stream)
                    self.run_inst()
                    st1.record(self.stream)
                    self.stream.synchronize()
                    inst_ms.append(st0.elapsed_time(st1))
                    for i, n in enumerate(ml.STAGE_NAMES):
                        stage_ms[n].append(self.ev[i].elapsed_time(self.ev[i + 1]))
            finally:
                if clocks is not None:
                    clocks.__exit__(None, None, None)
            torch.cuda.synchronize(self.device)
            barrier(world)
            status = ml.mlora_moe_read_status(self.ws, stream=self.stream)
            if status != 0:
                raise RuntimeError(f"{self.s.name}: device status {status:#x} after the timed steps")
        return dict(step_ms=step_ms, inst_ms=float(np.mean(inst_ms)),
                    stage_avg={n: float(np.mean(v)) for n, v in stage_ms.items()})

    def time_e2e(self, steps: int, warmup: int, world: int):
        """The same step end to end with host buffers: every step copies its
        inputs from pinned host memory (one H2D), runs the layer and reads y
        back (one D2H), captured with the layer in one CUDA graph; host clock,
        one stream synchronisation per step."""
        h_y = torch.empty((self.s.M, self.s.H), dtype=torch.bfloat16).pin_memory()

        def body():
            self.d_in.copy_(self.h_in, non_blocking=True)
            self.step()
            h_y.copy_(self.y, non_blocking=True)

        with torch.cuda.stream(self.stream):
            g = None
            if self.plain is not None:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    body()

            def e2e_step():
                if g is not None:
                    g.replay()
                else:
                    body()
                self.stream.synchronize()

            for _ in range(max(1, warmup)):
                e2e_step()
            barrier(world)
            t0 = time.perf_counter()
            for _ in range(steps):
                e2e_step()
            e2e_s = time.perf_counter() - t0
            status = self.ml.mlora_moe_read_status(self.ws, stream=self.stream)
            if status != 0:
                raise RuntimeError(f"device status {status:#x} after the end-to-end steps")
        return e2e_s, self.in_bytes, h_y.numel() * 2


def roofline_fields(s: wl.Spec, alg: dict, kernel_ms: float, layer_ms: float, peaks: dict, mx: bool = False) -> dict:
    """The experts kernel's and the whole layer's fraction of the roofline
    that bounds the workload: the tensor peak for prefill (bf16; MXFP8: the
    measured bf16 peak times the nominal fp8 / bf16 ratio of 2), HBM
    otherwise."""
    st = alg["stages"]["experts"]
    if s.name == "prefill":
        peak = peaks["bf16_tflops"] * (2.0 if mx else 1.0)
        kernel = st["flops"] / (kernel_ms / 1e3) / 1e12
        layer = alg["layer_flops"] / (layer_ms / 1e3) / 1e12
        return {"bound": "tensor", "unit": "TFLOP/s", "peak": peak, "experts_achieved": kernel,
                "experts_frac": kernel / peak, "layer_frac": layer / peak,
                "peak_kind": "measured bf16 x 2 (nominal fp8 ratio)" if mx else "measured bf16"}
    kernel = st["bytes"] / (kernel_ms / 1e3) / 1e9
    layer = alg["layer_bytes"] / (layer_ms / 1e3) / 1e9
    return {"bound": "hbm", "unit": "GB/s", "peak": peaks["hbm_gbs"], "experts_achieved": kernel,
            "experts_frac": kernel / peaks["hbm_gbs"], "layer_frac": layer / peaks["hbm_gbs"]}


def workload_entry(s: wl.Spec, t: dict, alg: dict, peaks: dict, mx: bool = False) -> dict:
    ms = float(np.mean(t["step_ms"]))
    kernel_ms = t["stage_avg"]["experts"]
    e = {"workload": workload_config(s)["workload"], "M": s.M, "us_per_layer": ms * 1e3,
         "tokens_per_s": s.M / (ms / 1e3), "experts_us": kernel_ms * 1e3,
         "stage_us": {k: v * 1e3 for k, v in t["stage_avg"].items()},
         "algorithmic_bytes": alg["layer_bytes"], "algorithmic_flops": alg["layer_flops"],
         "experts_touched": alg["experts"], "adapter_pairs_touched": alg["pairs"]}
    e["weights"] = "mxfp8" if mx else "bf16"
    e.update(roofline_fields(s, alg, kernel_ms, ms, peaks, mx))
    return e


def run_sweep(args, device, flush, peaks, skip_label=None, skip_entry=None):
    """Every workload of SWEEP on this device, one at a time (inputs freed in
    between), with the same timing as the headline."""
    out = {}
    sampler = ClockSampler(device.index or 0)
    for label, name, over in SWEEP:
        if label == skip_label and skip_entry is not None:
            out[label] = skip_entry
            continue
        over = dict(over)
        mx = over.pop("mx", False)
        s = wl.spec(name, **over)
        run = LayerRun(s, device, not args.no_graph, mx=mx)
        t = run.time(flush, steps=args.steps, warmup=max(3, min(args.warmup, 5)))
        out[label] = workload_entry(s, t, run.alg(), peaks, mx)
        del run
        torch.cuda.empty_cache()
    return out


def sweep_label(s: wl.Spec, overrides: dict):
    for label, name, over in SWEEP:
        if name == s.name and over == overrides:
            return label
    return None


def relaunch_replicas(args, argv) -> int:
    """`--gpus N` without a launcher: start N ranks of this script under
    torch.distributed.run on this node (one replica per GPU)."""
    import socket
    n_dev = torch.cuda.device_count()
    if n_dev < args.gpus:
        print(f"bench.py: --gpus {args.gpus} asks for more GPUs than this node has ({n_dev})", file=sys.stderr)
        return 2
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__),
           *(sys.argv[1:] if argv is None else argv)]
    return subprocess.call(cmd)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and args.impl == "mlora":
        return relaunch_replicas(args, argv)
    overrides = {} if args.M is None else {"M": args.M}
    s = wl.spec(args.workload, **overrides)
    if args.impl == "reference":
        return main_reference(args, s, rank, world)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    peaks, peak_src = load_peaks()
    flush = L2Flush(device)
    run = LayerRun(s, device, not args.no_graph, packed=True, mx=args.mxfp8)
    clocks = ClockSampler(local_rank)
    t = run.time(flush, args.steps, args.warmup, world, clocks=clocks)
    e2e_s, bi, bo = run.time_e2e(args.steps, args.warmup, world)
    alg = run.alg()
    total_ms, _, _ = aggregate(t["step_ms"], s.M, world, device)
    e2e_s = reduce_max(e2e_s, world, device)
    inp = run.inp
    headline_entry = workload_entry(s, t, alg, peaks, args.mxfp8)
    del run
    torch.cuda.empty_cache()
    workloads = None
    if not args.no_workloads and world == 1 and args.M is None:
        workloads = run_sweep(args, device, flush, peaks,
                              sweep_label(s, {**overrides, **({"mx": True} if args.mxfp8 else {})}), headline_entry)
    if rank == 0:
        ms_per_step = total_ms / args.steps
        tokens = s.M * world
        value = tokens / (ms_per_step / 1e3)
        dom_ms = t["stage_avg"]["experts"]
        rf = roofline_fields(s, alg, dom_ms, ms_per_step, peaks, args.mxfp8)
        cpu = None
        if not args.no_cpu_baseline and world == 1 and not args.mxfp8:
            cpu = cpu_baseline(inp, args.cpu_seconds)
            cpu.pop("seconds", None)
        cfg = workload_config(s)
        cfg.update({"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                    "l2": "flushed before every timed step: 256 MiB written, then another 256 MiB read",
                    "graph": not args.no_graph, "global_batch": tokens})
        out = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_layer": ms_per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "mxfp8 (e4m3, e8m0 scales) expert weights, bf16 activations and adapters" if args.mxfp8
            else "bf16",
            "data": "synthetic (seeded, random-init weights)", "config": cfg,
            "roofline": {"bound": rf["bound"], "kernel": "experts", "achieved": rf["experts_achieved"],
                         "peak": rf["peak"], "unit": rf["unit"], "frac": rf["experts_frac"],
                         "peak_source": peak_src,
                         "traffic": profiled_traffic("experts", s.name) if args.M is None else None,
                         "kernel_ms": dom_ms},
            "layer": {"frac": rf["layer_frac"], "ms_per_step_with_stage_events": t["inst_ms"],
                      "algorithmic_bytes": alg["layer_bytes"], "algorithmic_flops": alg["layer_flops"],
                      "experts_touched": alg["experts"], "adapter_pairs_touched": alg["pairs"],
                      "stage_us": {k: v * 1e3 for k, v in t["stage_avg"].items()}},
            "workloads": workloads,
            "cpu_baseline": cpu,
            "e2e": {"value": tokens * args.steps / e2e_s, "unit": "tokens/s",
                    "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo},
            "gpu_launches": 5 * args.steps,  # route, align, gather, experts, combine per step
            "clocks": clocks.summary(),
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main_reference(args, s: wl.Spec, rank: int, world: int):
    """The oracle timed on the host cores as the reference arm: each step is
    the route + forward of a bounded token sample of the batch; the per-step
    time is scaled to the whole batch."""
    if rank != 0:
        return 0
    import oracle
    inp = wl.make(s)
    oracle.load()
    hb = host_bits(inp)
    cores = os.cpu_count() or 1
    n = min(s.M, cores)
    for _ in range(args.warmup):
        oracle_sample(inp, n, hb)
    total, tokens = 0.0, 0
    for _ in range(args.steps):
        dt, k = oracle_sample(inp, n, hb)
        total += dt
        tokens += k
    value = tokens / total
    cfg = workload_config(s)
    sample = (f"route + forward of the first {n} of the {s.M} tokens of the {s.name} batch per step; "
              f"ms_per_step is that time scaled to the whole {s.M}-token batch")
    cfg.update({"parallelism": "host cores", "global_batch": s.M, "sample": sample})
    cpu = {"value": value, "unit": "tokens/s", "cores": min(cores, n), "kind": "oracle", "sample": sample}
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": s.M / value * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded, random-init weights)", "config": cfg, "cpu_baseline": cpu,
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
