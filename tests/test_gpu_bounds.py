"""The bounds-checked debug build (libmlora_checked.so, -DMLORA_CHECK_BOUNDS).

Every computed index into a workspace or output buffer is checked before the
store; a bad one would set MLORA_DEV_BOUNDS in the device status word and
skip the store instead of faulting.  These tests run the layer through that
build on shapes that exercise every tile kind, the narrow and wide tiles,
both align methods, ragged edges, the CTA-pair kernel and the MXFP8 layer:
the status word must stay clean and
the outputs must still match the oracle.  (A stand-in for a memory checker,
which this GPU pool does not offer.)"""
import numpy as np
import pytest
import torch

import moe_layer_lora_gb300 as ml
from moe_layer_lora_gb300 import _lib
from moe_layer_lora_gb300 import workloads as wl
import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def checked_library():
    _lib.use_library(_lib.LIB_CHECKED_PATH)
    yield
    _lib.use_library(_lib.LIB_PATH)


def _run(spec, rows=None):
    inp = wl.make(spec, device="cuda")
    gu.assert_unambiguous(inp)
    d = gu.DeviceInputs(inp)
    ids, w = gu.gpu_route(d)
    L, r = (spec.L, spec.r) if spec.has_lora else (0, 0)
    ws = torch.empty(ml.mlora_moe_workspace_size(spec.M, spec.H, spec.I, spec.E_tot, spec.K_total, L, r),
                     dtype=torch.uint8, device="cuda")
    y = gu.gpu_forward(d, ids, w, workspace=ws)
    torch.cuda.synchronize()
    status = ml.mlora_moe_read_status(ws)
    assert not status & ml.DEV_BOUNDS, f"{spec.name}: an index left its buffer (status {status:#x})"
    assert status == 0
    ids_ref, w_ref = gu.oracle_route(inp)
    y_ref = gu.oracle_forward(inp, ids_ref, w_ref, rows=rows)
    yg = y if rows is None else y[torch.as_tensor(rows, device="cuda")]
    gu.check_y(yg, y_ref, f"{spec.name} (bounds-checked build)")


def test_checked_build_is_loaded():
    assert _lib.load()._name.endswith("libmlora_checked.so")


@pytest.mark.parametrize("over", [
    dict(),                                                                   # tiny: narrow tiles
    dict(M=37, H=136, I=72, E=5, top_k=3, L=3, r=24, seed=101),               # ragged K, N, rank
    dict(M=9, H=8, I=8, E=4, top_k=4, L=5, r=64, seed=104),                   # tiny H/I, top_k = E
    dict(M=300, H=200, I=328, E=16, top_k=2, L=70, r=8, seed=105),            # L > 64 adapters
    dict(M=1100, H=136, I=72, E=5, top_k=4, L=3, r=24, seed=109),             # per-thread runs in align
    dict(M=1100, H=64, I=64, E=96, top_k=4, L=3, r=8, seed=112),              # runs, not staged
])
def test_small_layers(over):
    _run(wl.spec("tiny", **over))


def test_decode():
    _run(wl.spec("decode"))


def test_prefill_sampled():
    s = wl.spec("prefill")
    _run(s, rows=np.linspace(0, s.M - 1, 16).round().astype(np.int64))


def test_decode_two_tokens():
    _run(wl.spec("decode", M=2))                                              # 192-row tiles with adapters


def test_mid_width_ragged():
    _run(wl.spec("decode", M=8, H=2888, I=1448, E=8, top_k=2, L=4, r=16, seed=150))  # partial 192-row slabs


def test_shared_one_token():
    _run(wl.spec("shared", M=1))


def _run_pair(spec, rows=None):
    ml.mlora_set_pair_mode(True)
    try:
        _run(spec, rows)
    finally:
        ml.mlora_set_pair_mode(False)


@pytest.mark.parametrize("over", [
    dict(M=700, H=256, I=256, E=8, top_k=2, L=5, r=16, seed=501),             # pairs with adapters
    dict(M=300, H=160, I=224, E=5, top_k=3, L=3, r=24, seed=502),             # partial chunks and slabs
    dict(M=1, H=512, I=384, E=8, top_k=4, L=2, r=16, seed=506),               # every second block empty
    dict(M=500, H=96, I=64, E=4, top_k=2, L=2, r=8, seed=508),                # chunk-by-chunk copies only
])
def test_pair_small_layers(over):
    """The CTA-pair kernel (clusters of two, 256-row MMAs) through the
    bounds-checked build."""
    _run_pair(wl.spec("tiny", **over))


def test_pair_prefill_sampled():
    s = wl.spec("prefill")
    _run_pair(s, rows=np.linspace(0, s.M - 1, 16).round().astype(np.int64))


@pytest.mark.parametrize("name,over", [
    ("tiny", dict(M=37, H=160, I=224, E=5, top_k=3, L=3, r=24, seed=401)),    # ragged slabs and K-chunks
    ("decode", dict()),
    ("shared", dict(M=1)),
])
def test_mxfp8_layers(name, over):
    """The MXFP8 layer (E4M3 weights and rows, E8M0 scales) through the
    bounds-checked build, against the oracle's MXFP8 layer."""
    from test_gpu_mxfp8 import MxLayer
    s = wl.spec(name, **over)
    L = MxLayer(s)
    ids, w = gu.gpu_route(L.d)
    ws = torch.empty(ml.mlora_moe_workspace_size_mxfp8(s.M, s.H, s.I, s.E_tot, s.K_total,
                                                       s.L if s.has_lora else 0, s.r if s.has_lora else 0),
                     dtype=torch.uint8, device="cuda")
    y = L.forward(ids, w, workspace=ws)
    torch.cuda.synchronize()
    status = ml.mlora_moe_read_status(ws)
    assert not status & ml.DEV_BOUNDS, f"{name}: an index left its buffer (status {status:#x})"
    assert status == 0
    ids_ref, w_ref = gu.oracle_route(L.inp)
    gu.check_y(y, L.oracle(ids_ref, w_ref), f"mxfp8 {name} (bounds-checked build)")
