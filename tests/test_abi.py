"""The C-ABI library loads on a machine without a GPU, exports every symbol
include/mlora.h declares, and rejects bad arguments on the host before any
CUDA call (only calls that fail validation or are no-ops run here)."""
import ctypes
import os

import pytest

import moe_layer_lora_gb300 as ml
from moe_layer_lora_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    from moe_layer_lora_gb300 import build
    build.build()
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    names = _lib.declared_functions()
    for core in ("mlora_moe_route", "mlora_moe_align", "mlora_moe_align_max_padded", "mlora_moe_workspace_size",
                 "mlora_moe_forward", "mlora_moe_read_status", "mlora_set_stage_events", "mlora_status_string",
                 "mlora_set_wait_test"):
        assert core in names, core
    raw = ctypes.CDLL(_lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_stage_event_hook_validation(lib):
    assert lib.mlora_set_stage_events(None, 0) == 0
    arr = (ctypes.c_void_p * 3)(None, None, None)
    assert lib.mlora_set_stage_events(arr, 3) == 1


def test_wait_test_hook_validation(lib):
    assert lib.mlora_set_wait_test(-1, 0) == 1
    assert lib.mlora_set_wait_test(0, 0) == 0


def test_status_strings(lib):
    assert ml.mlora_status_string(0) == "ok"
    assert "shape" in ml.mlora_status_string(2)
    assert ml.mlora_status_string(99) == "unknown status"


def test_route_validation(lib):
    P = None
    f = lib.mlora_moe_route
    assert f(P, P, 4, 0, 1, 0, 1, 0, 1.0, P, P, P) == 2            # E = 0
    assert f(P, P, 4, 8, 9, 0, 1, 0, 1.0, P, P, P) == 2            # top_k > E
    assert f(P, P, 4, 8, 2, 7, 1, 0, 1.0, P, P, P) == 1            # bad scoring enum
    assert f(P, P, 4, 8, 2, 1, 1, 1, 0.0, P, P, P) == 1            # rsf <= 0 with shared slots
    assert f(P, P, 4, 2000, 2, 0, 1, 0, 1.0, P, P, P) == 2         # E > max
    assert f(P, P, 4, 128, 60, 0, 1, 8, 1.0, P, P, P) == 2         # K' > max
    assert f(P, P, 4, 8, 2, 0, 1, 0, 1.0, P, P, P) == 1            # NULL tensors
    assert f(P, P, 0, 8, 2, 0, 1, 0, 1.0, P, P, P) == 0            # M = 0: nothing to do


def test_align_validation(lib):
    P = None
    f = lib.mlora_moe_align
    assert f(P, 4, 2, 8, 0, P, P, P, P) == 2                       # block_m = 0
    assert f(P, 4, 2, 0, 16, P, P, P, P) == 2                      # E_tot = 0
    assert f(P, 4, 2, 8, 2048, P, P, P, P) == 2                    # block_m > max
    assert f(P, 4, 2, 8, 16, P, P, P, P) == 1                      # NULL buffers
    assert lib.mlora_moe_align_max_padded(3, 2, 3, 4) == 16
    assert lib.mlora_moe_align_max_padded(0, 2, 3, 4) == 0
    assert lib.mlora_moe_align_max_padded(3, 2, 3, 0) == 0


def test_align_max_padded_matches_oracle(lib):
    import oracle
    for args in [(3, 2, 3, 4), (16, 2, 8, 128), (64, 4, 32, 16), (8192, 4, 32, 128), (1, 9, 129, 128), (0, 1, 1, 1)]:
        assert lib.mlora_moe_align_max_padded(*args) == oracle.moe_align_max_padded(*args)


def _fwd(lib, M=4, H=64, I=64, E=4, K=2, L=0, r=0, n_shared=0, ptrs=True, ws=None, wsb=1 << 30, A13=None):
    P = ctypes.c_void_p(4096) if ptrs else None
    return lib.mlora_moe_forward(P, P, P, A13, A13, A13, A13, A13, P, P, M, H, I, E, K, L, r, 1.0, n_shared, 1.0,
                                 P, ws if ws is not None else ctypes.c_void_p(1 << 20), wsb, None)


def test_forward_validation(lib):
    assert _fwd(lib, H=60) == 2                                    # H % 8
    assert _fwd(lib, I=4) == 2                                     # I < 8
    assert _fwd(lib, E=2000) == 2                                  # E_tot > max
    assert _fwd(lib, K=0) == 2                                     # K' = 0
    assert _fwd(lib, n_shared=2) == 2                              # n_shared >= K'
    good = ctypes.c_void_p(4096)
    assert _fwd(lib, L=2, r=12, A13=good) == 3                     # rank not a multiple of 8
    assert _fwd(lib, L=2, r=128, A13=good) == 3                    # rank > 64
    assert _fwd(lib, ptrs=False) == 1                              # NULL tensors
    assert _fwd(lib, ws=ctypes.c_void_p(4096 + 16)) == 4           # misaligned workspace
    assert _fwd(lib, wsb=16) == 4                                  # too small
    assert _fwd(lib, M=0) == 0                                     # empty batch: no-op


def test_forward_misaligned_pointer(lib):
    bad = ctypes.c_void_p(4096 + 8)
    P = ctypes.c_void_p(4096)
    st = lib.mlora_moe_forward(bad, P, P, None, None, None, None, None, P, P, 4, 64, 64, 4, 2, 0, 0, 1.0, 0, 1.0,
                               P, ctypes.c_void_p(1 << 20), 1 << 30, None)
    assert st == 1


def test_workspace_size(lib):
    base = ml.mlora_moe_workspace_size(64, 2880, 2880, 32, 4, 0, 0)
    with_lora = ml.mlora_moe_workspace_size(64, 2880, 2880, 32, 4, 8, 16)
    assert 0 < base < with_lora
    assert base % 256 == 0 and with_lora % 256 == 0
    assert ml.mlora_moe_workspace_size(64, 2881, 2880, 32, 4, 0, 0) == 0
    assert ml.mlora_moe_workspace_size(8192, 2880, 2880, 32, 4, 8, 32) < 2 << 30


def test_mxfp8_sizes(lib):
    """MXFP8 needs H and I multiples of 32; sizes of the packed scales."""
    assert lib.mlora_mxfp8_scales_size(4, 72, 64, 0) == 0         # H not a multiple of 32
    assert lib.mlora_mxfp8_scales_size(4, 64, 64, 2) == 0         # which is 0 or 1
    assert lib.mlora_moe_workspace_size_mxfp8(4, 64, 40, 4, 2, 0, 0) == 0
    # gate_up: 32 experts x ceil(2880/96) slabs x ceil(2880/128) chunks x 1024 bytes
    assert lib.mlora_mxfp8_scales_size(32, 2880, 2880, 0) == 32 * 30 * 23 * 1024
    assert lib.mlora_mxfp8_scales_size(32, 2880, 2880, 1) == 32 * 15 * 23 * 1024
    assert ml.mlora_moe_workspace_size_mxfp8(64, 2880, 2880, 32, 4, 8, 16) > 0


def test_mxfp8_forward_validation(lib):
    P = ctypes.c_void_p(4096)
    f = lib.mlora_moe_forward_mxfp8
    args = [P] * 5 + [None] * 5 + [P, P]
    assert f(*args, 4, 72, 64, 4, 2, 0, 0, 1.0, 0, 1.0, P, ctypes.c_void_p(1 << 20), 1 << 30, None) == 2
    null_scales = [P, P, None, P, None] + [None] * 5 + [P, P]
    assert f(*null_scales, 4, 64, 64, 4, 2, 0, 0, 1.0, 0, 1.0, P, ctypes.c_void_p(1 << 20), 1 << 30, None) == 1


def test_tile_config_rule_and_hook(lib):
    """Without a tuned row the wave rule picks the width: narrow tiles for
    few blocks, 256 once the gate_up tiles fill two waves; the shrink group
    holds at most 4 adapters and 256 stacked rank rows.  The tuner's hook
    forces both and rejects values out of range."""
    H, I, E, K = 2880, 2880, 32, 4
    assert ml.mlora_tile_config(H, I, E, K, 16, 1, 152)[:2] == (2, 4)
    assert ml.mlora_tile_config(H, I, E, K, 16, 64, 152)[:2] == (0, 4)
    assert ml.mlora_tile_config(H, I, E, K, 64, 64, 152)[1] == 4
    assert ml.mlora_tile_config(H, I, E, K, 0, 64, 152)[1] == 1
    try:
        ml.mlora_set_tile_config(1, 2)
        assert ml.mlora_tile_config(H, I, E, K, 16, 64, 152)[:2] == (1, 2)
        ml.mlora_set_tile_config(2, 4)
        # rank 64: four adapters would stack 256 rows, within the limit
        assert ml.mlora_tile_config(H, I, E, K, 64, 3, 152)[:2] == (2, 4)
    finally:
        ml.mlora_set_tile_config(-1, 0)
    assert lib.mlora_set_tile_config(3, 0) == 1
    assert lib.mlora_set_tile_config(-2, 0) == 1
    assert lib.mlora_set_tile_config(0, 5) == 1


def test_pair_mode_switch_and_workspace(lib):
    """Pair mode is off unless the thread turns it on; while on, the bf16
    workspace holds padding up to two blocks per expert (the MXFP8 layer
    never pairs)."""
    assert not ml.mlora_pair_mode()
    args = (64, 2880, 2880, 32, 4, 8, 16)
    plain = ml.mlora_moe_workspace_size(*args)
    mx = ml.mlora_moe_workspace_size_mxfp8(*args)
    try:
        ml.mlora_set_pair_mode(True)
        assert ml.mlora_pair_mode()
        # up to 255 padding rows per expert instead of 127
        assert ml.mlora_moe_workspace_size(*args) > plain
        assert ml.mlora_moe_workspace_size_mxfp8(*args) == mx
    finally:
        ml.mlora_set_pair_mode(False)
    assert not ml.mlora_pair_mode()
    assert ml.mlora_moe_workspace_size(*args) == plain
    assert lib.mlora_set_pair_mode(2) == 1
    assert lib.mlora_set_pair_mode(-1) == 1


def test_tuned_table_rows_are_valid():
    """Every row of the compiled-in tuned table names width classes in
    range (or -1) and a group size the rank allows; the library reports the
    row as applied for its shape."""
    import re
    path = os.path.join(os.path.dirname(_lib.LIB_PATH), "csrc", "tuned_tiles.inc")
    rows = re.findall(r"^\{(\d+), (\d+), (\d+), (\d+), (\d+), \{([-\d, ]+)\}, (\d+)\},", open(path).read(), re.M)
    for H, I, E, K, r, tab, g in rows:
        H, I, E, K, r, g = map(int, (H, I, E, K, r, g))
        wcs = [int(v) for v in tab.split(",")]
        assert len(wcs) == 16 and all(-1 <= v <= 2 for v in wcs)
        rp = (r + 15) // 16 * 16
        assert g == 0 or (1 <= g <= 4 and (r == 0 or g * rp <= 256))
        for b, v in enumerate(wcs):
            wc, gs, tuned = ml.mlora_tile_config(H, I, E, K, r, 1 << b, 152)
            assert tuned
            if v >= 0:
                assert wc == v
