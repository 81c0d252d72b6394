"""Offline tuner of the experts kernel's tile configuration.

    python -m moe_layer_lora_gb300.autotune [--shapes decode,prefill,...] [--out PATH]

"Amazon SageMaker 및 Amazon Bedrock에서 vLLM을 활용한 MoE 모델 Multi-LoRA 서빙
최적화", section "섹션별 상세" paragraph 4: the block and split parameters
are found per deployment and loaded automatically.  Here that is: for each
layer shape and a sweep of batch sizes, the bf16 layer is timed with every
tile width forced (256, 192, 128 weight rows; mlora_set_tile_config), the
fastest width is kept per power-of-two bucket of the block count the batch
produces, then the fastest shrink group size (adapters per shrink tile) for
shapes with adapters; the result is written to csrc/tuned_tiles.inc, which
the next build compiles into libmlora.so, with a line saying where and how
it was measured.  Every forced configuration is checked to give the same
output bits as the library's choice (the width and the grouping never
change an output element's arithmetic).

Timing: CUDA events around graph replays of the forward on a side stream,
L2 flushed (a 256 MiB write, then a 256 MiB read) before every replay; the
median of --reps replays.
"""
from __future__ import annotations

import argparse
import datetime
import os
import statistics
import sys

import numpy as np
import torch

from . import _lib as ml
from . import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))
DEFAULT_OUT = os.path.join(HERE, "csrc", "tuned_tiles.inc")

# layer shapes (the five workloads') and the batch sizes swept for each
SHAPES = {
    "tiny": ("tiny", {}, [1, 4, 16, 64, 256, 1024]),
    "decode": ("decode", {}, [1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024]),
    "prefill": ("prefill", {}, [512, 1024, 2048, 4096, 8192]),
    "shared": ("shared", {}, [1, 2, 4, 8, 16, 32, 64, 128, 256, 512]),
    "stress": ("stress", {}, [1, 4, 16, 64, 128, 256, 512, 1024]),
}
BUCKETS = 16


def bucket(nblocks: int) -> int:
    b = 0
    while b + 1 < BUCKETS and (nblocks >> (b + 1)) > 0:
        b += 1
    return b


class Timer:
    def __init__(self, device, reps: int):
        self.reps = reps
        self.a = torch.empty(256 << 20, dtype=torch.uint8, device=device)
        self.b = torch.ones((256 << 20) // 4, dtype=torch.int32, device=device)
        self.o = torch.empty((), dtype=torch.int64, device=device)
        self.e0 = torch.cuda.Event(enable_timing=True)
        self.e1 = torch.cuda.Event(enable_timing=True)

    def flush(self):
        self.a.fill_(1)
        torch.sum(self.b, (0,), dtype=torch.int64, out=self.o)

    def time(self, graph: torch.cuda.CUDAGraph, stream) -> float:
        ts = []
        with torch.cuda.stream(stream):
            for i in range(self.reps + 2):
                self.flush()
                self.e0.record(stream)
                graph.replay()
                self.e1.record(stream)
                stream.synchronize()
                if i >= 2:
                    ts.append(self.e0.elapsed_time(self.e1))
        return statistics.median(ts)


class Layer:
    """One batch of a shape: inputs on the device, routed once, and a
    function that captures the forward as a CUDA graph under the thread's
    current tile configuration."""

    def __init__(self, spec: wl.Spec, device):
        self.s = spec
        inp = wl.make(spec, device=device)
        self.d = {k: (None if v is None else v.to(device)) for k, v in dict(
            logits=inp.logits, bias=inp.bias, x=inp.x, w13=inp.w13, w2=inp.w2, A13=inp.A13, B13=inp.B13, A2=inp.A2,
            B2=inp.B2, idx=inp.token_lora_idx).items()}
        s = spec
        self.ids, self.w = ml.mlora_moe_route(self.d["logits"], self.d["bias"], s.top_k, s.scoring, s.renormalize,
                                              s.n_shared, s.routed_scaling_factor)
        counts = np.bincount(self.ids.cpu().numpy().reshape(-1), minlength=s.E_tot)
        self.nblocks = int(sum((c + 127) // 128 for c in counts))
        L, r = (s.L, s.r) if s.has_lora else (0, 0)
        self.ws = torch.empty(ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, L, r),
                              dtype=torch.uint8, device=device)
        self.y = torch.empty((s.M, s.H), dtype=torch.bfloat16, device=device)
        self.stream = torch.cuda.Stream(device=device)

    def _forward(self):
        s, d = self.s, self.d
        ml.mlora_moe_forward(d["x"], d["w13"], d["w2"], d["A13"], d["B13"], d["A2"], d["B2"], d["idx"], self.ids,
                             self.w, s.scaling, s.n_shared, s.out_scale, y=self.y, workspace=self.ws,
                             stream=self.stream)

    def capture(self):
        with torch.cuda.stream(self.stream):
            self._forward()
            self.stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                self._forward()
        return g

    def output(self):
        with torch.cuda.stream(self.stream):
            self._forward()
        self.stream.synchronize()
        return self.y.clone()


def tune_shape(label: str, device, timer: Timer, log) -> dict:
    name, over, Ms = SHAPES[label]
    base = wl.spec(name, **over)
    rows = {}  # bucket -> list of (M, times per width class)
    ref_cfg = None
    for M in Ms:
        spec = wl.spec(name, **{**over, "M": M})
        layer = Layer(spec, device)
        ml.mlora_set_tile_config(-1, 0)
        y_ref = layer.output()
        times = []
        for wc in range(3):
            ml.mlora_set_tile_config(wc, 0)
            if not torch.equal(layer.output(), y_ref):
                raise RuntimeError(f"{label} M={M}: width class {wc} changed the output bits")
            times.append(timer.time(layer.capture(), layer.stream))
        ml.mlora_set_tile_config(-1, 0)
        rows.setdefault(bucket(layer.nblocks), []).append((M, times))
        log(f"{label} M={M} blocks={layer.nblocks} bucket={bucket(layer.nblocks)} "
            f"us: 256={times[0] * 1e3:.1f} 192={times[1] * 1e3:.1f} 128={times[2] * 1e3:.1f}")
        del layer
        torch.cuda.empty_cache()
    table = [-1] * BUCKETS
    for b, ms in rows.items():
        # the width with the smallest total time relative to each batch's best
        rel = [sum(t[wc] / min(t) for _, t in ms) for wc in range(3)]
        table[b] = int(np.argmin(rel))
    gsize = 0
    if base.has_lora:
        rp = (base.r + 15) // 16 * 16
        options = [g for g in (1, 2, 4) if g * rp <= 256]
        scores = {g: 0.0 for g in options}
        for M in Ms:
            spec = wl.spec(name, **{**over, "M": M})
            layer = Layer(spec, device)
            wc = table[bucket(layer.nblocks)]
            y_ref = layer.output()
            ts = {}
            for g in options:
                ml.mlora_set_tile_config(wc, g)
                if not torch.equal(layer.output(), y_ref):
                    raise RuntimeError(f"{label} M={M}: shrink group size {g} changed the output bits")
                ts[g] = timer.time(layer.capture(), layer.stream)
            ml.mlora_set_tile_config(-1, 0)
            best = min(ts.values())
            for g in options:
                scores[g] += ts[g] / best
            log(f"{label} M={M} shrink group size us: " + " ".join(f"{g}={ts[g] * 1e3:.1f}" for g in options))
            del layer
            torch.cuda.empty_cache()
        gsize = min(scores, key=scores.get)
    rank = base.r if base.has_lora else 0
    return {"label": label, "H": base.H, "I": base.I, "E_tot": base.E_tot, "K_total": base.K_total,
            "rank": rank, "table": table, "gsize": gsize}


def write_inc(path: str, results, provenance: str):
    lines = [
        "// tuned_tiles.inc -- the experts kernel's tuned tile widths and shrink group",
        "// sizes, written by moe_layer_lora_gb300/autotune.py (do not edit by hand).",
        "// One row per layer shape: {H, I, E_tot, K_total, rank (0: no adapters),",
        "// {tile width class per block-count bucket b = [2^b, 2^(b+1)) blocks:",
        "// 0 = 256, 1 = 192, 2 = 128 weight rows, -1 = the wave rule}, shrink group",
        "// size (0: the rule)}.  Shapes not listed use the rules.",
        f"// {provenance}",
    ]
    for r in results:
        tab = ", ".join(str(v) for v in r["table"])
        lines.append(f"{{{r['H']}, {r['I']}, {r['E_tot']}, {r['K_total']}, {r['rank']}, {{{tab}}}, {r['gsize']}}},"
                     f"  // {r['label']}")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--shapes", default=",".join(SHAPES))
    ap.add_argument("--out", default=DEFAULT_OUT)
    ap.add_argument("--reps", type=int, default=15)
    ap.add_argument("--log", default=None, help="also write the measurements to this file")
    args = ap.parse_args(argv)
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    timer = Timer(device, args.reps)
    logf = open(args.log, "w") if args.log else None

    def log(msg):
        print(msg, flush=True)
        if logf:
            logf.write(msg + "\n")

    results = [tune_shape(label, device, timer, log) for label in args.shapes.split(",")]
    when = datetime.datetime.now(datetime.timezone.utc).strftime("%Y-%m-%d %H:%M UTC")
    prov = (f"measured on {torch.cuda.get_device_name(device)} ({torch.cuda.get_device_properties(device).multi_processor_count}"
            f" SMs), {when}: python -m moe_layer_lora_gb300.autotune --shapes {args.shapes} --reps {args.reps}")
    write_inc(args.out, results, prov)
    log(f"wrote {args.out}")
    if logf:
        logf.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
