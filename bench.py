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


def algorithmic(s: wl.Spec, ids: np.ndarray, idx) -> dict:
    """Bytes each stage must move and flops it must do, from the routed ids:
    every touched expert's weights once, every touched (adapter, expert)
    pair's four LoRA matrices once, the activations once."""
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
    st = {
        # the experts kernel: both projections, their adapter shrink and expand
        "experts": dict(bytes=n_exp * 3 * I * H * b + n_pairs * r * (2 * H + 3 * I) * b + S * (2 * H + 2 * I) * b,
                        flops=2.0 * S * 3 * H * I + 2.0 * a_slots * r * (2 * H + 3 * I)),
        "gather": dict(bytes=S * H * b * 2, flops=0.0),
        "combine": dict(bytes=S * H * b + M * H * b, flops=2.0 * S * H),
        "align": dict(bytes=S * 4 * 3, flops=0.0),
    }
    layer_bytes = (n_exp * 3 * I * H * b + n_pairs * r * (2 * H + 3 * I) * b + 2 * M * H * b
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

def oracle_sample(inp, ids, w, n_tokens: int):
    import oracle
    s = inp.spec
    rows = np.arange(min(n_tokens, s.M))
    b = wl.bits
    lora = s.has_lora
    t0 = time.perf_counter()
    oracle.moe_forward(b(inp.x)[rows], b(inp.w13), b(inp.w2), b(inp.A13) if lora else None,
                       b(inp.B13) if lora else None, b(inp.A2) if lora else None, b(inp.B2) if lora else None,
                       inp.token_lora_idx.numpy()[rows] if lora else None, ids[rows],
                       w[rows].astype(np.float32), s.scaling, s.out_scale)
    return time.perf_counter() - t0, len(rows)


def cpu_baseline(inp, target_s: float):
    """The oracle as it stands on the host cores, on a bounded token sample
    sized to roughly target_s seconds of work."""
    import oracle
    s = inp.spec
    oracle.load()
    ids, w = oracle.moe_route(inp.logits.numpy(), None if inp.bias is None else inp.bias.numpy(), s.top_k,
                              s.scoring, s.renormalize, s.n_shared, s.routed_scaling_factor)
    cores = os.cpu_count() or 1
    n = min(s.M, cores)
    dt, n = oracle_sample(inp, ids, w, n)
    if dt < target_s / 3 and n < s.M:
        n2 = int(min(s.M, max(n, n * target_s / max(dt, 1e-3))) // max(1, min(cores, n)) * min(cores, n))
        n2 = max(n, min(s.M, n2))
        if n2 > n:
            dt, n = oracle_sample(inp, ids, w, n2)
    # a whole batch that takes well under the target is timed over several
    # passes, so that the figure is not one short run
    passes = 1
    if dt < target_s / 3:
        passes = int(min(50, max(1, target_s / max(dt, 1e-3) - 1)))
        for _ in range(passes - 1):
            dt_i, _ = oracle_sample(inp, ids, w, n)
            dt += dt_i
    return {"value": n * passes / dt, "unit": "tokens/s", "cores": min(cores, n), "kind": "oracle",
            "sample": f"first {n} of the {s.M} tokens of the {s.name} batch, {passes} fp64 layer "
                      f"pass{'es' if passes > 1 else ''} ({dt:.1f} s)",
            "seconds": dt}


# ---------------------------------------------------------------- GPU path --

def run_gpu(args, s: wl.Spec, rank: int, world: int, local_rank: int):
    import moe_layer_lora_gb300 as ml

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    inp = wl.make(s, device=device)
    d = {k: (None if v is None else v.to(device)) for k, v in dict(
        logits=inp.logits, bias=inp.bias, x=inp.x, w13=inp.w13, w2=inp.w2, A13=inp.A13, B13=inp.B13, A2=inp.A2,
        B2=inp.B2, idx=inp.token_lora_idx).items()}
    # the per-step inputs (x, router logits, adapter ids) live in one device
    # buffer with a pinned host twin, so the end-to-end step brings them over
    # in one copy
    parts = [("x", inp.x), ("logits", inp.logits)] + ([("idx", inp.token_lora_idx)] if s.has_lora else [])
    offs, in_bytes = {}, 0
    for name, t in parts:
        offs[name] = in_bytes
        in_bytes += (t.numel() * t.element_size() + 255) // 256 * 256
    h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device=device)
    for name, t in parts:
        nb = t.numel() * t.element_size()
        h_in[offs[name]:offs[name] + nb].copy_(t.contiguous().reshape(-1).view(torch.uint8))
        d[name] = d_in[offs[name]:offs[name] + nb].view(t.dtype).view(t.shape)
    d_in.copy_(h_in)
    L, r = (s.L, s.r) if s.has_lora else (0, 0)
    ids = torch.empty((s.M, s.K_total), dtype=torch.int32, device=device)
    w = torch.empty((s.M, s.K_total), dtype=torch.float32, device=device)
    y = torch.empty((s.M, s.H), dtype=torch.bfloat16, device=device)
    ws = torch.empty(ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, L, r), dtype=torch.uint8,
                     device=device)
    flush = L2Flush(device)
    stream = torch.cuda.Stream(device=device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(ml.STAGE_EVENTS)]
    for e in ev:
        e.record(stream)  # creates the event handles
    ml.mlora_set_stage_events(None)
    step_start = torch.cuda.Event(enable_timing=True)
    step_end = torch.cuda.Event(enable_timing=True)

    def step():
        ml.mlora_moe_route(d["logits"], d["bias"], s.top_k, s.scoring, s.renormalize, s.n_shared,
                           s.routed_scaling_factor, topk_ids=ids, topk_w=w, stream=stream)
        ml.mlora_moe_forward(d["x"], d["w13"], d["w2"], d["A13"], d["B13"], d["A2"], d["B2"], d["idx"], ids, w,
                             s.scaling, s.n_shared, s.out_scale, y=y, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        step()
        stream.synchronize()
        status = ml.mlora_moe_read_status(ws, stream=stream)
        if status != 0:
            raise RuntimeError(f"device status {status:#x} after the first step")
        # two graphs of the same step: a plain one for the headline time and
        # one with event nodes at the stage boundaries for per-kernel times
        plain = inst = None
        if not args.no_graph:
            plain = torch.cuda.CUDAGraph()
            with torch.cuda.graph(plain, stream=stream):
                step()
            ml.mlora_set_stage_events(ev)
            inst = torch.cuda.CUDAGraph()
            with torch.cuda.graph(inst, stream=stream):
                step()
            ml.mlora_set_stage_events(None)
        run = plain.replay if plain is not None else step

        def run_inst():
            if inst is not None:
                inst.replay()
            else:
                ml.mlora_set_stage_events(ev)
                step()
                ml.mlora_set_stage_events(None)

        for _ in range(args.warmup):
            flush()
            run()
            flush()
            run_inst()
        stream.synchronize()
        ids_host = ids.cpu().numpy()
        alg = algorithmic(s, ids_host, inp.token_lora_idx.numpy() if s.has_lora else None)

        barrier(world)
        torch.cuda.synchronize(device)
        step_ms, inst_ms, stage_ms = [], [], {n: [] for n in ml.STAGE_NAMES}
        with ClockSampler(local_rank) as clocks:
            for _ in range(args.steps):
                flush()
                step_start.record(stream)
                run()
                step_end.record(stream)
                stream.synchronize()
                step_ms.append(step_start.elapsed_time(step_end))
            torch.cuda.synchronize(device)
            barrier(world)
            # per-kernel times: as many steps of the instrumented graph
            for _ in range(args.steps):
                flush()
                step_start.record(stream)
                run_inst()
                step_end.record(stream)
                stream.synchronize()
                inst_ms.append(step_start.elapsed_time(step_end))
                for i, n in enumerate(ml.STAGE_NAMES):
                    stage_ms[n].append(ev[i].elapsed_time(ev[i + 1]))
        torch.cuda.synchronize(device)
        barrier(world)
        launches_per_step = 5  # route, align, gather, experts, combine

        # end to end through the public API with host buffers: H2D of the
        # step's inputs from pinned memory (one copy), the layer, D2H of the
        # output, captured with the layer in one CUDA graph
        h_y = torch.empty((s.M, s.H), dtype=torch.bfloat16).pin_memory()
        bi = in_bytes
        bo = h_y.numel() * 2

        def e2e_body():
            d_in.copy_(h_in, non_blocking=True)
            step()
            h_y.copy_(y, non_blocking=True)

        e2e_graph = None
        if not args.no_graph:
            e2e_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(e2e_graph, stream=stream):
                e2e_body()

        def e2e_step():
            if e2e_graph is not None:
                e2e_graph.replay()
            else:
                e2e_body()
            stream.synchronize()

        for _ in range(max(1, args.warmup)):
            e2e_step()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        e2e_s = time.perf_counter() - t0
        status = ml.mlora_moe_read_status(ws, stream=stream)
        if status != 0:
            raise RuntimeError(f"device status {status:#x} after the timed steps")

    total_ms, _, _ = aggregate(step_ms, s.M, world, device)
    e2e_s = reduce_max(e2e_s, world, device)
    stage_avg = {n: float(np.mean(v)) for n, v in stage_ms.items()}
    return dict(inp=inp, alg=alg, total_ms=total_ms, step_ms=step_ms, inst_ms=float(np.mean(inst_ms)),
                stage_avg=stage_avg, e2e_s=e2e_s, bi=bi,
                bo=bo, clocks=clocks.summary(), launches=launches_per_step * args.steps)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    overrides = {} if args.M is None else {"M": args.M}
    s = wl.spec(args.workload, **overrides)
    if args.impl == "reference":
        return main_reference(args, s, rank, world)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_gpu(args, s, rank, world, local_rank)
    if rank == 0:
        peaks, peak_src = load_peaks()
        alg = res["alg"]
        ms_per_step = res["total_ms"] / args.steps
        tokens = s.M * world
        value = tokens / (ms_per_step / 1e3)
        # dominant kernel and its roofline
        dom = max(res["stage_avg"], key=lambda n: res["stage_avg"][n])
        dom_ms = res["stage_avg"][dom]
        st = alg["stages"].get(dom, {"bytes": 0, "flops": 0})
        bound = "tensor" if s.name == "prefill" else "hbm"
        if bound == "hbm":
            achieved = st["bytes"] / (dom_ms / 1e3) / 1e9
            peak, unit = peaks["hbm_gbs"], "GB/s"
        else:
            achieved = st["flops"] / (dom_ms / 1e3) / 1e12
            peak, unit = peaks["bf16_tflops"], "TFLOP/s"
        layer_hbm_frac = alg["layer_bytes"] / (ms_per_step / 1e3) / 1e9 / peaks["hbm_gbs"]
        layer_tc_frac = alg["layer_flops"] / (ms_per_step / 1e3) / 1e12 / peaks["bf16_tflops"]
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(res["inp"], args.cpu_seconds)
            cpu.pop("seconds", None)
        cfg = workload_config(s)
        cfg.update({"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                    "l2": "flushed before every timed step: 256 MiB written, then another 256 MiB read",
                    "graph": not args.no_graph, "global_batch": tokens})
        out = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_layer": ms_per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded, random-init weights)", "config": cfg,
            "roofline": {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak, "unit": unit,
                         "frac": achieved / peak, "peak_source": peak_src,
                         "traffic": profiled_traffic(dom, s.name) if args.M is None else None,
                         "kernel_ms": dom_ms},
            "layer": {"hbm_frac": layer_hbm_frac, "tensor_frac": layer_tc_frac,
                      "ms_per_step_with_stage_events": res["inst_ms"],
                      "algorithmic_bytes": alg["layer_bytes"], "algorithmic_flops": alg["layer_flops"],
                      "experts_touched": alg["experts"], "adapter_pairs_touched": alg["pairs"],
                      "stage_us": {k: v * 1e3 for k, v in res["stage_avg"].items()}},
            "cpu_baseline": cpu,
            "e2e": {"value": tokens * args.steps / res["e2e_s"], "unit": "tokens/s",
                    "h2d_bytes_per_step": res["bi"], "d2h_bytes_per_step": res["bo"]},
            "gpu_launches": res["launches"],
            "clocks": res["clocks"],
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main_reference(args, s: wl.Spec, rank: int, world: int):
    """The oracle timed on the host cores as the reference arm."""
    if rank != 0:
        return 0
    import oracle
    inp = wl.make(s)
    oracle.load()
    ids, w = oracle.moe_route(inp.logits.numpy(), None if inp.bias is None else inp.bias.numpy(), s.top_k,
                              s.scoring, s.renormalize, s.n_shared, s.routed_scaling_factor)
    cores = os.cpu_count() or 1
    n = min(s.M, cores)
    for _ in range(args.warmup):
        oracle_sample(inp, ids, w, n)
    total, tokens = 0.0, 0
    for _ in range(args.steps):
        dt, k = oracle_sample(inp, ids, w, n)
        total += dt
        tokens += k
    value = tokens / total
    cfg = workload_config(s)
    cfg.update({"parallelism": "host cores", "global_batch": s.M})
    cpu = {"value": value, "unit": "tokens/s", "cores": min(cores, n), "kind": "oracle",
           "sample": f"first {n} of the {s.M} tokens of the {s.name} batch per step"}
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded, random-init weights)", "config": cfg, "cpu_baseline": cpu,
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
