"""The allocation-free entry point (mlora_moe_forward_static) against the
regular one.

mlora_moe_forward_static serves callers that cannot allocate device memory
where they run the layer (their memory belongs to another allocator, they
may not allocate after start-up, or they only hold tensor pointers): its
scratch is a fixed device array inside the library.  Two calls in a row,
with different inputs, must each match mlora_moe_forward (own workspace)
within the layer tolerance; the array keeps the previous call's contents,
so the second call also shows that nothing stale leaks through.  This file
sorts last so that a run stopping at the first failure has run the rest.
"""
import ctypes

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


def test_static_matches_regular_two_calls():
    s = wl.spec("decode")
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    for call, seed in enumerate((s.seed, s.seed + 1000)):
        if call:
            new = wl.make(wl.spec("decode", seed=seed), with_weights=False)
            d.logits.copy_(new.logits)
            d.x.copy_(new.x)
            d.idx.copy_(new.token_lora_idx)
        ids, w = gu.gpu_route(d)
        y_reg = _regular(d, ids, w, s)
        y_sta = ml.mlora_moe_forward_static(d.x, d.w13, d.w2, d.A13, d.B13, d.A2, d.B2, d.idx, ids, w,
                                            s.scaling, s.n_shared, s.out_scale)
        torch.cuda.synchronize()
        ref = y_reg.double().cpu().numpy()
        gu.check_y(y_sta, ref, f"static call {call + 1} vs regular")


def test_static_rejects_too_large():
    s = wl.spec("prefill")  # its workspace is far above the array
    need = ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r)
    assert need > _lib.STATIC_WORKSPACE_BYTES
    lib = _lib.load()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    fn = lib.mlora_moe_forward_static
    P, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [P] * 10 + [i] * 7 + [f, i, f, P, P]
    fn.restype = i
    st = fn(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, s.M, s.H, s.I, s.E_tot, s.K_total, s.L,
            s.r, 2.0, 0, 1.0, fake, None)
    assert st == 4  # MLORA_ERR_WORKSPACE
