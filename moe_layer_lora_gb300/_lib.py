"""ctypes binding of libmlora.so (include/mlora.h), same names as the C ABI.

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (PyTorch provides device
memory and streams); outputs not passed in are allocated with torch before
the call.  A missing library raises at import of the first call: there is
no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmlora.so")
LIB_CHECKED_PATH = os.path.join(HERE, "libmlora_checked.so")  # bounds-checked debug build
HEADER = os.path.join(os.path.dirname(HERE), "include", "mlora.h")

MLORA_OK = 0
STATUS_NAMES = {0: "MLORA_OK", 1: "MLORA_ERR_INVALID_ARG", 2: "MLORA_ERR_SHAPE", 3: "MLORA_ERR_UNSUPPORTED",
                4: "MLORA_ERR_WORKSPACE", 5: "MLORA_ERR_CUDA"}
SCORE_SOFTMAX = 0
SCORE_SIGMOID_BIAS = 1
DEV_TIMEOUT = 1
DEV_BAD_EXPERT_ID = 2
DEV_BAD_LORA_IDX = 4
DEV_BOUNDS = 8  # bounds-checked debug build only
FORWARD_BLOCK_M = 128


class MloraError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


_lib = None


def use_library(path: str = LIB_PATH):
    """Switch the binding to another build of the library, e.g. the
    bounds-checked debug build LIB_CHECKED_PATH; LIB_PATH is the default."""
    global _lib
    _lib = None
    return load(path)


def load(path: str = LIB_PATH):
    """Load libmlora.so and declare its C signatures.  Raises if not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m moe_layer_lora_gb300.build` "
                           "(the layer has no fallback implementation)")
    lib = ctypes.CDLL(path)
    P, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.mlora_moe_route.argtypes = [P, P, i, i, i, i, i, i, f, P, P, P]
    lib.mlora_moe_route.restype = i
    lib.mlora_moe_align_max_padded.argtypes = [i, i, i, i]
    lib.mlora_moe_align_max_padded.restype = sz
    lib.mlora_moe_align.argtypes = [P, i, i, i, i, P, P, P, P]
    lib.mlora_moe_align.restype = i
    lib.mlora_moe_workspace_size.argtypes = [i] * 7
    lib.mlora_moe_workspace_size.restype = sz
    lib.mlora_moe_forward.argtypes = [P] * 10 + [i] * 7 + [f, i, f, P, P, sz, P]
    lib.mlora_moe_forward.restype = i
    lib.mlora_moe_read_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
    lib.mlora_moe_read_status.restype = i
    lib.mlora_set_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i]
    lib.mlora_set_stage_events.restype = i
    lib.mlora_set_wait_test.argtypes = [ctypes.c_longlong, i]
    lib.mlora_set_wait_test.restype = i
    lib.mlora_status_string.argtypes = [i]
    lib.mlora_status_string.restype = ctypes.c_char_p
    lib.mlora_moe_forward_static.argtypes = [P] * 10 + [i] * 7 + [f, i, f, P, P]
    lib.mlora_moe_forward_static.restype = i
    lib.mlora_moe_read_status_static.argtypes = [ctypes.POINTER(ctypes.c_uint32), P]
    lib.mlora_moe_read_status_static.restype = i
    lib.mlora_mxfp8_scales_size.argtypes = [i] * 4
    lib.mlora_mxfp8_scales_size.restype = sz
    lib.mlora_mxfp8_quantize_weights.argtypes = [P, P, i, i, i, P, P, P, P, P]
    lib.mlora_mxfp8_quantize_weights.restype = i
    lib.mlora_moe_workspace_size_mxfp8.argtypes = [i] * 7
    lib.mlora_moe_workspace_size_mxfp8.restype = sz
    lib.mlora_moe_forward_mxfp8.argtypes = [P] * 12 + [i] * 7 + [f, i, f, P, P, sz, P]
    lib.mlora_moe_forward_mxfp8.restype = i
    lib.mlora_set_tile_config.argtypes = [i, i]
    lib.mlora_set_tile_config.restype = i
    ip = ctypes.POINTER(ctypes.c_int)
    lib.mlora_tile_config.argtypes = [i] * 7 + [ip, ip, ip]
    lib.mlora_tile_config.restype = i
    lib.mlora_set_pair_mode.argtypes = [i]
    lib.mlora_set_pair_mode.restype = i
    lib.mlora_pair_mode.argtypes = []
    lib.mlora_pair_mode.restype = i
    _lib = lib
    return lib


def declared_functions(header: str = HEADER):
    """Names of the functions include/mlora.h declares."""
    with open(header) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mlora_[a-z_]+)\s*\(", text)))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, device=None) -> ctypes.c_void_p:
    """The stream handle to enqueue on: `stream`, else the current stream of
    `device`.  A stream of another device than the tensors' is refused (the
    library launches on the current device, which the callers below set to
    the tensors' device)."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif device is not None and stream.device != torch.device(device):
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, status: int):
    if status != MLORA_OK:
        raise MloraError(fn, status)


def _need_shape(t, dtype, name: str, shape=None):
    """The library reads every tensor as a dense row-major array of the given
    shape (its tensor maps are built from those sizes, not from the
    allocation), so a mismatch is refused here, before any device work."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _need_place(t: torch.Tensor, name: str, device=None):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {t.dtype} tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the layer's inputs on {device}")


def _need(t, dtype, name: str, shape=None, device=None):
    _need_shape(t, dtype, name, shape)
    _need_place(t, name, device)


def _layer_args(x, w13, w2, A13, B13, A2, B2, token_lora_idx, topk_ids, topk_w, y, weight_dtype=torch.bfloat16,
                extra=()):
    """Checks the layer's tensors against each other; returns
    (M, H, I, E_tot, K', L, rank, lora).  `extra`: more (tensor, dtype,
    name, shape) checks (shape may be a callable of (E_tot, H, I))."""
    if not isinstance(x, torch.Tensor) or x.dim() != 2 or not isinstance(w13, torch.Tensor) or w13.dim() != 3:
        raise ValueError("x must be [M, H] and w13 [E_tot, 2I, H]")
    M, H = x.shape
    E_tot, twoI = w13.shape[0], w13.shape[1]
    if twoI % 2:
        raise ValueError(f"w13 must have an even row count 2I, got {twoI}")
    I = twoI // 2
    if not isinstance(topk_ids, torch.Tensor) or topk_ids.dim() != 2:
        raise ValueError("topk_ids must be [M, K']")
    KT = topk_ids.shape[1]
    checks = [(x, torch.bfloat16, "x", (M, H)), (w13, weight_dtype, "w13", (E_tot, 2 * I, H)),
              (w2, weight_dtype, "w2", (E_tot, H, I)), (topk_ids, torch.int32, "topk_ids", (M, KT)),
              (topk_w, torch.float32, "topk_w", (M, KT))]
    checks += [(t, dt, name, shape(E_tot, H, I) if callable(shape) else shape) for t, dt, name, shape in extra]
    if y is not None:
        checks.append((y, torch.bfloat16, "y", (M, H)))
    given = [t is not None for t in (A13, B13, A2, B2, token_lora_idx)]
    if any(given) and not all(given):
        raise ValueError("A13, B13, A2, B2 and token_lora_idx are given together (adapters) or all None "
                         "(no adapters)")
    lora = all(given)
    L = r = 0
    if lora:
        if not isinstance(A13, torch.Tensor) or A13.dim() != 4:
            raise ValueError("A13 must be [L, E_tot, rank, H]")
        L, r = A13.shape[0], A13.shape[2]
        checks += [(A13, torch.bfloat16, "A13", (L, E_tot, r, H)), (B13, torch.bfloat16, "B13", (L, E_tot, 2 * I, r)),
                   (A2, torch.bfloat16, "A2", (L, E_tot, r, I)), (B2, torch.bfloat16, "B2", (L, E_tot, H, r)),
                   (token_lora_idx, torch.int32, "token_lora_idx", (M,))]
    # every shape and dtype first, then where the tensors live
    for t, dtype, name, shape in checks:
        _need_shape(t, dtype, name, shape)
    for t, _, name, _ in checks:
        _need_place(t, name, x.device)
    return M, H, I, E_tot, KT, L, r, lora


def mlora_moe_route(logits: torch.Tensor, bias: Optional[torch.Tensor], top_k: int, scoring: int,
                    renormalize: int = 1, n_shared: int = 0, routed_scaling_factor: float = 1.0,
                    topk_ids: Optional[torch.Tensor] = None, topk_w: Optional[torch.Tensor] = None,
                    stream=None):
    if not isinstance(logits, torch.Tensor) or logits.dim() != 2:
        raise ValueError("logits must be [M, E]")
    M, E = logits.shape
    KT = top_k + n_shared
    dev = logits.device
    checks = [(logits, torch.float32, "logits", (M, E))]
    if topk_ids is not None:
        checks.append((topk_ids, torch.int32, "topk_ids", (M, KT)))
    if topk_w is not None:
        checks.append((topk_w, torch.float32, "topk_w", (M, KT)))
    if bias is not None:
        checks.append((bias, torch.float32, "bias", (E,)))
    for t, dtype, name, shape in checks:
        _need_shape(t, dtype, name, shape)
    for t, _, name, _ in checks:
        _need_place(t, name, dev)
    if topk_ids is None:
        topk_ids = torch.empty((M, KT), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((M, KT), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = load().mlora_moe_route(_ptr(logits), _ptr(bias), M, E, top_k, scoring, renormalize, n_shared,
                                    float(routed_scaling_factor), _ptr(topk_ids), _ptr(topk_w),
                                    _stream(stream, dev))
    _check("mlora_moe_route", st)
    return topk_ids, topk_w


def mlora_moe_align_max_padded(M: int, K_total: int, E_tot: int, block_m: int) -> int:
    return int(load().mlora_moe_align_max_padded(M, K_total, E_tot, block_m))


def mlora_moe_align(topk_ids: torch.Tensor, E_tot: int, block_m: int, stream=None):
    """Returns (sorted_ids, expert_ids, num_post_padded[1]) as CUDA tensors."""
    if not isinstance(topk_ids, torch.Tensor) or topk_ids.dim() != 2:
        raise ValueError("topk_ids must be [M, K']")
    M, KT = topk_ids.shape
    _need(topk_ids, torch.int32, "topk_ids", (M, KT))
    mp = mlora_moe_align_max_padded(M, KT, E_tot, block_m)
    dev = topk_ids.device
    sorted_ids = torch.empty(mp, dtype=torch.int32, device=dev)
    expert_ids = torch.empty(mp // block_m, dtype=torch.int32, device=dev)
    npp = torch.empty(1, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        st = load().mlora_moe_align(_ptr(topk_ids), M, KT, E_tot, block_m, _ptr(sorted_ids), _ptr(expert_ids),
                                    _ptr(npp), _stream(stream, dev))
    _check("mlora_moe_align", st)
    return sorted_ids, expert_ids, npp


def mlora_moe_workspace_size(M: int, H: int, I: int, E_tot: int, K_total: int, L: int, rank: int) -> int:
    return int(load().mlora_moe_workspace_size(M, H, I, E_tot, K_total, L, rank))


def mlora_moe_forward(x, w13, w2, A13, B13, A2, B2, token_lora_idx, topk_ids, topk_w, scaling: float,
                      n_shared: int = 0, out_scale: float = 1.0, y: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None):
    """The fused MoE-LoRA layer; returns y [M, H] bf16 (see include/mlora.h)."""
    M, H, I, E_tot, KT, L, r, lora = _layer_args(x, w13, w2, A13, B13, A2, B2, token_lora_idx, topk_ids, topk_w, y)
    if y is None:
        y = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    need = mlora_moe_workspace_size(M, H, I, E_tot, KT, L, r)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    _need(workspace, torch.uint8, "workspace", None, x.device)
    with torch.cuda.device(x.device):
        st = load().mlora_moe_forward(
            _ptr(x), _ptr(w13), _ptr(w2), _ptr(A13) if lora else None, _ptr(B13) if lora else None,
            _ptr(A2) if lora else None, _ptr(B2) if lora else None, _ptr(token_lora_idx) if lora else None,
            _ptr(topk_ids), _ptr(topk_w), M, H, I, E_tot, KT, L, r, float(scaling), int(n_shared),
            float(out_scale), _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream, x.device))
    _check("mlora_moe_forward", st)
    return y


def mlora_mxfp8_scales_size(E_tot: int, H: int, I: int, which: int) -> int:
    return int(load().mlora_mxfp8_scales_size(E_tot, H, I, which))


def mlora_mxfp8_quantize_weights(w13: torch.Tensor, w2: torch.Tensor, stream=None):
    """bf16 expert weights to MXFP8 on their device: returns (w13_q, w13_s,
    w2_q, w2_s), E4M3 codes in the weights' layout and packed E8M0 scales
    (see include/mlora.h)."""
    if not isinstance(w13, torch.Tensor) or w13.dim() != 3 or not isinstance(w2, torch.Tensor) or w2.dim() != 3:
        raise ValueError("w13 must be [E_tot, 2I, H] and w2 [E_tot, H, I]")
    E_tot, twoI, H = w13.shape
    I = twoI // 2
    _need(w13, torch.bfloat16, "w13", (E_tot, 2 * I, H))
    _need(w2, torch.bfloat16, "w2", (E_tot, H, I), w13.device)
    n13, n2 = mlora_mxfp8_scales_size(E_tot, H, I, 0), mlora_mxfp8_scales_size(E_tot, H, I, 1)
    if not n13 or not n2:
        raise ValueError(f"MXFP8 needs H and I multiples of 32 (H={H}, I={I})")
    dev = w13.device
    w13_q = torch.empty((E_tot, 2 * I, H), dtype=torch.uint8, device=dev)
    w2_q = torch.empty((E_tot, H, I), dtype=torch.uint8, device=dev)
    w13_s = torch.empty(n13, dtype=torch.uint8, device=dev)
    w2_s = torch.empty(n2, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = load().mlora_mxfp8_quantize_weights(_ptr(w13), _ptr(w2), E_tot, H, I, _ptr(w13_q), _ptr(w13_s),
                                                 _ptr(w2_q), _ptr(w2_s), _stream(stream, dev))
    _check("mlora_mxfp8_quantize_weights", st)
    return w13_q, w13_s, w2_q, w2_s


def mlora_moe_workspace_size_mxfp8(M: int, H: int, I: int, E_tot: int, K_total: int, L: int, rank: int) -> int:
    return int(load().mlora_moe_workspace_size_mxfp8(M, H, I, E_tot, K_total, L, rank))


def mlora_moe_forward_mxfp8(x, w13_q, w13_s, w2_q, w2_s, A13, B13, A2, B2, token_lora_idx, topk_ids, topk_w,
                            scaling: float, n_shared: int = 0, out_scale: float = 1.0,
                            y: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                            stream=None):
    """The fused MoE-LoRA layer with MXFP8 expert weights (from
    mlora_mxfp8_quantize_weights); returns y [M, H] bf16."""
    extra = [(w13_s, torch.uint8, "w13_s", lambda E, H, I: (mlora_mxfp8_scales_size(E, H, I, 0),)),
             (w2_s, torch.uint8, "w2_s", lambda E, H, I: (mlora_mxfp8_scales_size(E, H, I, 1),))]
    M, H, I, E_tot, KT, L, r, lora = _layer_args(x, w13_q, w2_q, A13, B13, A2, B2, token_lora_idx, topk_ids,
                                                 topk_w, y, weight_dtype=torch.uint8, extra=extra)
    if y is None:
        y = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    need = mlora_moe_workspace_size_mxfp8(M, H, I, E_tot, KT, L, r)
    if need == 0:
        raise ValueError(f"invalid MXFP8 layer sizes (H={H}, I={I} must be multiples of 32)")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _need(workspace, torch.uint8, "workspace", None, x.device)
    with torch.cuda.device(x.device):
        st = load().mlora_moe_forward_mxfp8(
            _ptr(x), _ptr(w13_q), _ptr(w13_s), _ptr(w2_q), _ptr(w2_s), _ptr(A13) if lora else None,
            _ptr(B13) if lora else None, _ptr(A2) if lora else None, _ptr(B2) if lora else None,
            _ptr(token_lora_idx) if lora else None, _ptr(topk_ids), _ptr(topk_w), M, H, I, E_tot, KT, L, r,
            float(scaling), int(n_shared), float(out_scale), _ptr(y), _ptr(workspace), workspace.numel(),
            _stream(stream, x.device))
    _check("mlora_moe_forward_mxfp8", st)
    return y


STATIC_WORKSPACE_BYTES = 64 << 20


def mlora_moe_forward_static(x, w13, w2, A13, B13, A2, B2, token_lora_idx, topk_ids, topk_w, scaling: float,
                             n_shared: int = 0, out_scale: float = 1.0, y: Optional[torch.Tensor] = None,
                             stream=None):
    """The layer with the library's fixed scratch array instead of a
    workspace: for callers that cannot allocate device memory where they
    run it.  Only y is allocated here (by torch) when not passed in."""
    M, H, I, E_tot, KT, L, r, lora = _layer_args(x, w13, w2, A13, B13, A2, B2, token_lora_idx, topk_ids, topk_w, y)
    if y is None:
        y = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    with torch.cuda.device(x.device):
        st = load().mlora_moe_forward_static(
            _ptr(x), _ptr(w13), _ptr(w2), _ptr(A13) if lora else None, _ptr(B13) if lora else None,
            _ptr(A2) if lora else None, _ptr(B2) if lora else None, _ptr(token_lora_idx) if lora else None,
            _ptr(topk_ids), _ptr(topk_w), M, H, I, E_tot, KT, L, r, float(scaling), int(n_shared),
            float(out_scale), _ptr(y), _stream(stream, x.device))
    _check("mlora_moe_forward_static", st)
    return y


def mlora_moe_read_status_static(device=None, stream=None) -> int:
    """Device status word of the last mlora_moe_forward_static on `device`
    (default: the current device); waits for the stream."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    out = ctypes.c_uint32(0)
    with torch.cuda.device(dev):
        st = load().mlora_moe_read_status_static(ctypes.byref(out), _stream(stream, dev))
    _check("mlora_moe_read_status_static", st)
    return int(out.value)


def mlora_moe_read_status(workspace: torch.Tensor, stream=None) -> int:
    out = ctypes.c_uint32(0)
    with torch.cuda.device(workspace.device):
        st = load().mlora_moe_read_status(_ptr(workspace), ctypes.byref(out), _stream(stream, workspace.device))
    _check("mlora_moe_read_status", st)
    return int(out.value)


STAGE_EVENTS = 5
STAGE_NAMES = ("align", "gather", "experts", "combine")


def mlora_set_stage_events(events) -> None:
    """Record the given torch.cuda.Event objects (STAGE_EVENTS of them, made
    with enable_timing=True) at the forward's stage boundaries on this
    thread; None switches the hook off."""
    if events is None:
        _check("mlora_set_stage_events", load().mlora_set_stage_events(None, 0))
        return
    handles = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check("mlora_set_stage_events", load().mlora_set_stage_events(handles, len(events)))


def mlora_set_wait_test(wait_limit_cycles: int, stall: bool) -> None:
    """Test hook (see include/mlora.h): a shorter limit for the experts
    kernel's waits and, with stall, a first wait on a flag nothing sets.
    (0, False) restores the defaults."""
    _check("mlora_set_wait_test", load().mlora_set_wait_test(int(wait_limit_cycles), 1 if stall else 0))


def mlora_set_tile_config(width_class: int = -1, gsize: int = 0) -> None:
    """Force, for this thread's later forwards, the experts kernel's tile
    width class (0: 256, 1: 192, 2: 128 weight rows; -1: tuned table or
    rule) and shrink group size (0: table or rule) -- the tuner's hook."""
    _check("mlora_set_tile_config", load().mlora_set_tile_config(int(width_class), int(gsize)))


def mlora_tile_config(H: int, I: int, E_tot: int, K_total: int, rank: int, nblocks: int, grid: int):
    """(width class, shrink group size, tuned) a bf16 layer of this shape
    uses for nblocks blocks on a grid of `grid` CTAs."""
    wc, g, t = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check("mlora_tile_config", load().mlora_tile_config(H, I, E_tot, K_total, rank, nblocks, grid,
                                                         ctypes.byref(wc), ctypes.byref(g), ctypes.byref(t)))
    return wc.value, g.value, bool(t.value)


def mlora_set_pair_mode(on: bool) -> None:
    """For this thread's later bf16 forwards: run the experts kernel as CTA
    pairs (True) or one CTA per SM (False, the default).  Query workspace
    sizes after setting it."""
    _check("mlora_set_pair_mode", load().mlora_set_pair_mode(1 if on else 0))


def mlora_pair_mode() -> bool:
    """Whether this thread's bf16 forwards run as CTA pairs."""
    return bool(load().mlora_pair_mode())


def mlora_status_string(status: int) -> str:
    return load().mlora_status_string(status).decode()
