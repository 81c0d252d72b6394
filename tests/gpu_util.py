"""Helpers shared by the GPU parity tests: device copies of the seeded
inputs, the CUDA path through the C ABI, the oracle on the same host bytes,
and the tolerance check of the layer output."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import moe_layer_lora_gb300 as ml
from moe_layer_lora_gb300 import workloads as wl

# Layer-output tolerance: relative Frobenius error <= 1e-2 and max abs error
# <= 5e-2 * rms(reference) against the fp64 oracle.
REL_FRO = 1e-2
MAX_ABS_RMS = 5e-2
# Routing weights: fp32 exp/divide against fp64.
W_RTOL = 2e-6
W_ATOL = 1e-7


def dev(t, device="cuda"):
    return None if t is None else t.to(device, non_blocking=False).contiguous()


class DeviceInputs:
    def __init__(self, inp: wl.Inputs):
        self.inp = inp
        s = inp.spec
        self.logits = dev(inp.logits)
        self.bias = dev(inp.bias)
        self.x = dev(inp.x)
        self.w13 = dev(inp.w13)
        self.w2 = dev(inp.w2)
        self.A13, self.B13, self.A2, self.B2 = (dev(t) for t in (inp.A13, inp.B13, inp.A2, inp.B2))
        self.idx = dev(inp.token_lora_idx)
        self.spec = s


def gpu_route(d: DeviceInputs):
    s = d.spec
    return ml.mlora_moe_route(d.logits, d.bias, s.top_k, s.scoring, s.renormalize, s.n_shared,
                              s.routed_scaling_factor)


def gpu_forward(d: DeviceInputs, ids, w, idx="default", lora=True, workspace=None):
    s = d.spec
    use = lora and s.has_lora
    tli = d.idx if idx == "default" else idx
    return ml.mlora_moe_forward(d.x, d.w13, d.w2, d.A13 if use else None, d.B13 if use else None,
                                d.A2 if use else None, d.B2 if use else None, tli if use else None, ids, w,
                                s.scaling, s.n_shared, s.out_scale, workspace=workspace)


def oracle_route(inp: wl.Inputs):
    s = inp.spec
    return oracle.moe_route(inp.logits.numpy(), None if inp.bias is None else inp.bias.numpy(), s.top_k,
                            s.scoring, s.renormalize, s.n_shared, s.routed_scaling_factor)


def _hbits(t):
    """Host bit copy of a (possibly device) bf16 tensor."""
    return None if t is None else wl.bits(t)


def oracle_forward(inp: wl.Inputs, ids, w, rows=None, lora=True, idx=None):
    """fp64 layer output for the given token rows (all when rows is None);
    the layer acts on each token independently, so a row subset of the
    inputs gives exactly those rows of the output."""
    s = inp.spec
    use = lora and s.has_lora
    sel = slice(None) if rows is None else np.asarray(rows)
    x = wl.bits(inp.x)[sel]
    tli = None
    if use:
        tli = inp.token_lora_idx.numpy() if idx is None else np.asarray(idx, np.int32)
    b = _hbits
    return oracle.moe_forward(x, b(inp.w13), b(inp.w2), b(inp.A13) if use else None,
                              b(inp.B13) if use else None, b(inp.A2) if use else None,
                              b(inp.B2) if use else None, tli[sel] if use else None, ids[sel],
                              w[sel].astype(np.float32), s.scaling, s.out_scale)


def assert_unambiguous(inp: wl.Inputs):
    """Sigmoid+bias routing takes its integer decision on an fp32 key,
    sigmoid(l) + b, on both sides with each side's own expf.  The seeded
    inputs must keep every key that decides the order (the first top_k + 1
    of a token) more than 8 ulp from its neighbour, so that a 1-2 ulp expf
    difference cannot change the ids; a closer pair is an ambiguous input,
    reported as such rather than as an id mismatch."""
    s = inp.spec
    if s.scoring != wl.SCORE_SIGMOID_BIAS or s.M == 0:
        return
    l = inp.logits.numpy().astype(np.float32)
    b = np.zeros(s.E, np.float32) if inp.bias is None else inp.bias.numpy().astype(np.float32)
    key = (np.float32(1) / (np.float32(1) + np.exp(-l))) + b[None, :]
    srt = -np.sort(-key, axis=1)[:, : s.top_k + 1]
    gaps = srt[:, :-1] - srt[:, 1:]
    ulp = np.spacing(np.abs(srt[:, :-1])).astype(np.float64)
    close = np.argwhere(~(gaps > 8 * ulp))
    assert close.size == 0, f"ambiguous input: sigmoid+bias keys within 8 ulp at (token, rank) {close[:4].tolist()}"


def check_route(ids_gpu, w_gpu, ids_ref, w_ref):
    ids_g = ids_gpu.cpu().numpy()
    assert np.array_equal(ids_g, ids_ref), f"route ids differ at {np.argwhere(ids_g != ids_ref)[:8]}"
    np.testing.assert_allclose(w_gpu.cpu().numpy().astype(np.float64), w_ref, rtol=W_RTOL, atol=W_ATOL)


def y_errors(y_gpu, y_ref):
    yg = y_gpu.float().cpu().numpy().astype(np.float64)
    err = yg - y_ref
    rel_fro = float(np.linalg.norm(err) / max(np.linalg.norm(y_ref), 1e-300))
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    max_abs = float(np.abs(err).max()) if err.size else 0.0
    return rel_fro, max_abs, rms


def check_y(y_gpu, y_ref, label=""):
    rel_fro, max_abs, rms = y_errors(y_gpu, y_ref)
    assert np.isfinite(y_gpu.float().cpu().numpy()).all(), f"{label}: non-finite output"
    assert rel_fro <= REL_FRO, f"{label}: rel Frobenius error {rel_fro:.3e} > {REL_FRO}"
    assert max_abs <= MAX_ABS_RMS * rms, f"{label}: max abs error {max_abs:.3e} > {MAX_ABS_RMS}*rms ({rms:.3e})"
    return rel_fro, max_abs, rms


def sample_rows(M: int, n: int, seed: int, must=()):
    """n distinct token rows spread over [0, M) plus the listed ones."""
    rng = np.random.default_rng(seed)
    rows = set(int(r) for r in must)
    rows.update(int(r) for r in rng.choice(M, size=min(n, M), replace=False))
    return np.array(sorted(rows), dtype=np.int64)
