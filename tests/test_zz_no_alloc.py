"""The allocation-free entry point (mlora_moe_forward_static) against the
fp64 oracle and against the regular entry point.

mlora_moe_forward_static serves callers that cannot allocate device memory
where they run the layer (their memory belongs to another allocator, they
may not allocate after start-up, or they only hold tensor pointers): its
scratch is a fixed device array inside the library.  Two calls in a row,
with different inputs, must each match the oracle on sampled tokens and
mlora_moe_forward (own workspace) on every token, within the layer
tolerance; the array keeps the previous call's contents, so the second call
also shows that nothing stale leaks through.  The array's status word is
read through mlora_moe_read_status_static, clean after each call, and a
wait that runs out inside a static call is reported there.  This file sorts
last so that a run stopping at the first failure has run the rest.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_layer_lora_gb300 as ml
from moe_layer_lora_gb300 import _lib
from moe_layer_lora_gb300 import workloads as wl
import gpu_util as gu

pytestmark = pytest.mark.gpu


def _regular(d, ids, w, s):
    return ml.mlora_moe_forward(d.x, d.w13, d.w2, d.A13, d.B13, d.A2, d.B2, d.idx, ids, w, s.scaling,
                                s.n_shared, s.out_scale)


def _static(d, ids, w, s):
    return ml.mlora_moe_forward_static(d.x, d.w13, d.w2, d.A13, d.B13, d.A2, d.B2, d.idx, ids, w, s.scaling,
                                       s.n_shared, s.out_scale)


def test_static_matches_oracle_and_regular_two_calls():
    s = wl.spec("decode")
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    for call, seed in enumerate((s.seed, s.seed + 1000)):
        if call:
            new = wl.make(wl.spec("decode", seed=seed), with_weights=False)
            d.logits.copy_(new.logits)
            d.x.copy_(new.x)
            d.idx.copy_(new.token_lora_idx)
            inp.logits, inp.x, inp.token_lora_idx = new.logits, new.x, new.token_lora_idx
        ids, w = gu.gpu_route(d)
        y_sta = _static(d, ids, w, s)
        assert ml.mlora_moe_read_status_static() == 0, f"call {call + 1}"
        y_reg = _regular(d, ids, w, s)
        torch.cuda.synchronize()
        ids_ref, w_ref = gu.oracle_route(inp)
        gu.check_route(ids, w, ids_ref, w_ref)
        rows = gu.sample_rows(s.M, 16, seed=31 + call, must=(0, s.M - 1))
        y_ref = gu.oracle_forward(inp, ids_ref, w_ref, rows=rows)
        gu.check_y(y_sta[torch.as_tensor(rows, device="cuda")], y_ref, f"static call {call + 1} vs oracle")
        gu.check_y(y_sta, y_reg.double().cpu().numpy(), f"static call {call + 1} vs regular")


def test_static_reports_a_wait_timeout():
    """A static call whose waits run out (test hook: a first wait on a flag
    nothing sets, ~1 ms limit) reports MLORA_DEV_TIMEOUT through the static
    status reader; the next static call is clean and correct."""
    s = wl.spec("tiny")
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    ids, w = gu.gpu_route(d)
    ml.mlora_set_wait_test(2_000_000, True)
    try:
        _static(d, ids, w, s)
        st = ml.mlora_moe_read_status_static()
    finally:
        ml.mlora_set_wait_test(0, False)
    assert st & ml.DEV_TIMEOUT, st
    y = _static(d, ids, w, s)
    assert ml.mlora_moe_read_status_static() == 0
    ids_ref, w_ref = gu.oracle_route(inp)
    gu.check_y(y, gu.oracle_forward(inp, ids_ref, w_ref), "static call after a timed-out one")


def test_static_rejects_too_large():
    s = wl.spec("prefill")  # its workspace is far above the array
    need = ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r)
    assert need > _lib.STATIC_WORKSPACE_BYTES
    fn = _lib.load().mlora_moe_forward_static
    # NULL tensors: the size check answers first; were it ever moved behind
    # the pointer checks, the call would return INVALID_ARG, never launch
    st = fn(None, None, None, None, None, None, None, None, None, None, s.M, s.H, s.I, s.E_tot, s.K_total, s.L,
            s.r, 2.0, 0, 1.0, None, None)
    assert st == 4  # MLORA_ERR_WORKSPACE
    # and a size that fits with NULL tensors is refused as an argument error
    t = wl.spec("tiny")
    st = fn(None, None, None, None, None, None, None, None, None, None, t.M, t.H, t.I, t.E_tot, t.K_total, t.L,
            t.r, 2.0, 0, 1.0, None, None)
    assert st == 1  # MLORA_ERR_INVALID_ARG


def test_static_status_reader_rejects_null():
    assert _lib.load().mlora_moe_read_status_static(None, None) == 1
