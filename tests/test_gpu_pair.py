"""The CTA-pair experts kernel (clusters of two CTAs sharing 256-row
tcgen05 MMAs over two blocks of one expert) against the single-CTA kernel
and the fp64 oracle.

Pair mode changes which SM computes which rows, the padding of the sorted
order (every expert's blocks padded to an even count) and the adapter
stages (the union of a pair's two adapter lists, zero rows for the block
that lacks one), but no output element's arithmetic: each output equals the
single-CTA kernel's bit for bit (torch.equal: an exact zero may differ in
sign).  The shapes cover partial and empty second blocks, ragged K chunks,
a last gate_up slab and a last down slab that run past I and H (the odd
CTA's half of the last down slab entirely out of range), K-chunk counts
that give every kind of two-chunk stage (both chunks whole, the second past
K, a partial last chunk, fewer than two whole chunks), shrink groups of
odd size (the odd CTA's zero adapter), many adapters per block, one token
(every pair's second block empty), the prefill layer and the adapter stress
layer.  Pair mode is opt-in (mlora_set_pair_mode)."""
import numpy as np
import pytest
import torch

import moe_layer_lora_gb300 as ml
from moe_layer_lora_gb300 import workloads as wl
import gpu_util as gu

pytestmark = pytest.mark.gpu


def _forward(d, ids, w, mode, lora=True):
    s = d.spec
    use = lora and s.has_lora
    ml.mlora_set_pair_mode(mode)
    try:
        ws = torch.empty(ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, s.L if use else 0,
                                                     s.r if use else 0), dtype=torch.uint8, device="cuda")
        y = gu.gpu_forward(d, ids, w, lora=lora, workspace=ws)
        torch.cuda.synchronize()
        assert ml.mlora_moe_read_status(ws) == 0
        return y
    finally:
        ml.mlora_set_pair_mode(False)


CASES = [
    dict(M=700, H=256, I=256, E=8, top_k=2, L=5, r=16, seed=501),  # adapters, rank 16 (groups of 4)
    dict(M=300, H=160, I=224, E=5, top_k=3, L=3, r=24, seed=502),  # ragged K chunk, partial last slabs
    dict(M=1000, H=320, I=192, E=12, top_k=2, L=9, r=64, seed=503),  # rank 64: groups of 1-4 adapters
    dict(M=513, H=288, I=136, E=6, top_k=4, L=0, r=0, lora_mode="none", seed=504),  # no adapters
    dict(M=64, H=256, I=128, E=16, top_k=2, L=4, r=8, seed=505),  # mostly one block per expert
    dict(M=1, H=512, I=384, E=8, top_k=4, L=2, r=16, seed=506),  # one token: every second block empty
    dict(M=900, H=512, I=512, E=4, top_k=1, L=6, r=32, n_shared=1, routed_scaling_factor=2.5,
         scoring=wl.SCORE_SIGMOID_BIAS, seed=507),  # shared slots, full blocks
    dict(M=500, H=96, I=64, E=4, top_k=2, L=2, r=8, seed=508),  # K below two chunks: chunk-by-chunk copies only
]


@pytest.mark.parametrize("over", CASES, ids=lambda o: f"M{o['M']}H{o['H']}I{o['I']}E{o['E']}L{o['L']}r{o['r']}")
def test_pair_equals_single_cta(over):
    s = wl.spec("tiny", **over)
    inp = wl.make(s, device="cuda")
    gu.assert_unambiguous(inp)
    d = gu.DeviceInputs(inp)
    ids, w = gu.gpu_route(d)
    y_single = _forward(d, ids, w, False)
    y_pair = _forward(d, ids, w, True)
    assert torch.equal(y_pair, y_single)
    ids_ref, w_ref = gu.oracle_route(inp)
    gu.check_route(ids, w, ids_ref, w_ref)
    rows = gu.sample_rows(s.M, 16, seed=over["seed"], must=(0, s.M - 1))
    gu.check_y(y_pair[torch.as_tensor(rows, device="cuda")], gu.oracle_forward(inp, ids_ref, w_ref, rows=rows),
               f"pair {over}")


def test_pair_poisoned_workspace_never_leaks():
    """Pair mode on a workspace filled with NaN bytes before each of eight
    calls (adapters, many small blocks): every call equals the single-CTA
    kernel on a clean workspace, so no CTA of either kind reads a block's
    act rows or LoRA tiles before all four epilogue warps wrote them."""
    s = wl.spec("tiny", M=700, H=256, I=256, E=8, top_k=2, L=5, r=16, seed=501)
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    ids, w = gu.gpu_route(d)
    y_single = _forward(d, ids, w, False)
    ml.mlora_set_pair_mode(True)
    try:
        ws = torch.empty(ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r),
                         dtype=torch.uint8, device="cuda")
        for call in range(8):
            ws.fill_(0xFF)
            y = gu.gpu_forward(d, ids, w, workspace=ws)
            torch.cuda.synchronize()
            assert ml.mlora_moe_read_status(ws) == 0, call
            assert torch.equal(y, y_single), call
    finally:
        ml.mlora_set_pair_mode(False)


def test_prefill_in_pairs_equals_single_cta():
    """The prefill layer (32 768 slots over 32 experts, adapters) in pair
    mode gives the single-CTA kernel's bits, which the full-row prefill test
    holds against the oracle; sampled rows against the oracle here too."""
    s = wl.spec("prefill")
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    ids, w = gu.gpu_route(d)
    y_pair = _forward(d, ids, w, True)
    y_single = _forward(d, ids, w, False)
    assert torch.equal(y_pair, y_single)
    ids_ref, w_ref = gu.oracle_route(inp)
    rows = gu.sample_rows(s.M, 24, seed=61, must=(0, s.M - 1))
    gu.check_y(y_pair[torch.as_tensor(rows, device="cuda")], gu.oracle_forward(inp, ids_ref, w_ref, rows=rows),
               "prefill pairs")


def test_stress_adapters_in_pairs():
    """64 adapters of rank 64, Zipf-distributed: long and different adapter
    lists in the two blocks of a pair."""
    s = wl.spec("stress")
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    ids, w = gu.gpu_route(d)
    y_single = _forward(d, ids, w, False)
    y_pair = _forward(d, ids, w, True)
    assert torch.equal(y_pair, y_single)
    y_base_pair = _forward(d, ids, w, True, lora=False)
    y_base = _forward(d, ids, w, False, lora=False)
    assert torch.equal(y_base_pair, y_base)


def test_pair_graph_replay_equals_eager():
    s = wl.spec("tiny", M=600, H=256, I=256, E=6, top_k=2, L=4, r=16, seed=510)
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    ml.mlora_set_pair_mode(True)
    try:
        ids = torch.empty((s.M, s.K_total), dtype=torch.int32, device="cuda")
        w = torch.empty((s.M, s.K_total), dtype=torch.float32, device="cuda")
        y = torch.empty((s.M, s.H), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r),
                         dtype=torch.uint8, device="cuda")
        stream = torch.cuda.Stream()

        def step():
            ml.mlora_moe_route(d.logits, d.bias, s.top_k, s.scoring, s.renormalize, s.n_shared,
                               s.routed_scaling_factor, topk_ids=ids, topk_w=w, stream=stream)
            ml.mlora_moe_forward(d.x, d.w13, d.w2, d.A13, d.B13, d.A2, d.B2, d.idx, ids, w, s.scaling, s.n_shared,
                                 s.out_scale, y=y, workspace=ws, stream=stream)

        with torch.cuda.stream(stream):
            step()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        for seed in (511, 512):
            new = wl.make(wl.spec("tiny", M=600, H=256, I=256, E=6, top_k=2, L=4, r=16, seed=seed),
                          with_weights=False)
            d.logits.copy_(new.logits)
            d.x.copy_(new.x)
            d.idx.copy_(new.token_lora_idx)
            g.replay()
            torch.cuda.synchronize()
            y_graph = y.clone()
            ids_e, w_e = gu.gpu_route(d)
            y_eager = gu.gpu_forward(d, ids_e, w_e)
            torch.cuda.synchronize()
            assert torch.equal(y_graph, y_eager)
    finally:
        ml.mlora_set_pair_mode(False)


def test_pair_wait_timeout_is_reported_and_the_context_recovers():
    """A wait that runs out inside the pair kernel (every CTA first waits on
    a flag nothing sets) ends in MLORA_DEV_TIMEOUT, both CTAs of each pair
    unwind, and the next forward is correct."""
    s = wl.spec("tiny", M=400, H=256, I=128, E=4, top_k=2, L=3, r=16, seed=520)
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    ids, w = gu.gpu_route(d)
    ml.mlora_set_pair_mode(True)
    try:
        ws = torch.empty(ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r),
                         dtype=torch.uint8, device="cuda")
        ml.mlora_set_wait_test(2_000_000, True)
        try:
            gu.gpu_forward(d, ids, w, workspace=ws)
            st = ml.mlora_moe_read_status(ws)
        finally:
            ml.mlora_set_wait_test(0, False)
        assert st & ml.DEV_TIMEOUT, st
        y = gu.gpu_forward(d, ids, w, workspace=ws)
        torch.cuda.synchronize()
        assert ml.mlora_moe_read_status(ws) == 0
    finally:
        ml.mlora_set_pair_mode(False)
    ids_ref, w_ref = gu.oracle_route(inp)
    gu.check_y(y, gu.oracle_forward(inp, ids_ref, w_ref), "pair after timeout")
