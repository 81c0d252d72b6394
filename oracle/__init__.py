"""fp64 CPU oracle for the fused MoE-LoRA layer (ctypes wrapper over oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``; the product path never touches
it.  It shares no code with the CUDA library.  See oracle.c for the pages
and passages each function follows.

Functions with no external pin are named in ``UNPINNED`` (empty: every
function is pinned by the tests under ``tests/test_oracle_*.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

UNPINNED: tuple = ()

_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile oracle.c into a shared library with gcc (plain -O2, OpenMP)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def load(path: str = _LIB_PATH):
    """Load (building first if needed) and declare the oracle's C ABI."""
    global _lib
    if _lib is not None and path == _LIB_PATH:
        return _lib
    if not os.path.exists(path) or (path == _LIB_PATH and os.path.getmtime(path) < os.path.getmtime(_SRC)):
        build(out=path)
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i = ctypes.c_int
    f = ctypes.c_float
    lib.oracle_moe_route.argtypes = [P, P, i, i, i, i, i, i, f, P, P]
    lib.oracle_moe_route.restype = i
    lib.oracle_moe_align_max_padded.argtypes = [i, i, i, i]
    lib.oracle_moe_align_max_padded.restype = ctypes.c_long
    lib.oracle_moe_align.argtypes = [P, i, i, i, i, P, P, P]
    lib.oracle_moe_align.restype = i
    lib.oracle_moe_forward.argtypes = [P] * 10 + [i] * 7 + [f, f, P]
    lib.oracle_moe_forward.restype = i
    lib.oracle_mx_quantize.argtypes = [P, ctypes.c_long, i, P, P]
    lib.oracle_mx_quantize.restype = i
    lib.oracle_mx_dequantize.argtypes = [P, P, ctypes.c_long, i, P]
    lib.oracle_mx_dequantize.restype = i
    lib.oracle_moe_forward_mx.argtypes = [P] * 12 + [i] * 7 + [f, f, P]
    lib.oracle_moe_forward_mx.restype = i
    if path == _LIB_PATH:
        _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


def moe_route(logits, bias, top_k, scoring, renormalize=1, n_shared=0,
              routed_scaling_factor=1.0, lib=None):
    """Returns (topk_ids int32 [M,K'], topk_w float64 [M,K'])."""
    lib = lib or load()
    logits = _c(logits, np.float32)
    bias = _c(bias, np.float32)
    M, E = logits.shape
    KT = top_k + n_shared
    ids = np.zeros((M, KT), np.int32)
    w = np.zeros((M, KT), np.float64)
    rc = lib.oracle_moe_route(_ptr(logits), _ptr(bias), M, E, top_k, scoring, renormalize,
                              n_shared, float(routed_scaling_factor), _ptr(ids), _ptr(w))
    if rc != 0:
        raise ValueError(f"oracle_moe_route rejected its arguments ({rc})")
    return ids, w


def moe_align_max_padded(M, K_total, E_tot, block_m, lib=None):
    lib = lib or load()
    return int(lib.oracle_moe_align_max_padded(M, K_total, E_tot, block_m))


def moe_align(topk_ids, E_tot, block_m, lib=None):
    """Returns (sorted_ids, expert_ids, num_post_padded)."""
    lib = lib or load()
    topk_ids = _c(topk_ids, np.int32)
    M, KT = topk_ids.shape
    mp = moe_align_max_padded(M, KT, E_tot, block_m, lib)
    sorted_ids = np.zeros(mp, np.int32)
    expert_ids = np.zeros(mp // block_m, np.int32)
    npp = np.zeros(1, np.int32)
    rc = lib.oracle_moe_align(_ptr(topk_ids), M, KT, E_tot, block_m, _ptr(sorted_ids),
                              _ptr(expert_ids), _ptr(npp))
    if rc != 0:
        raise ValueError(f"oracle_moe_align rejected its arguments ({rc})")
    return sorted_ids, expert_ids, int(npp[0])


def moe_forward(x, w13, w2, A13, B13, A2, B2, token_lora_idx, topk_ids, topk_w,
                scaling, out_scale=1.0, lib=None):
    """fp64 layer output [M, H].  Bf16 tensors are passed as uint16 bit arrays;
    A13/B13/A2/B2/token_lora_idx may be None (no adapters)."""
    lib = lib or load()
    x = _c(x, np.uint16)
    w13 = _c(w13, np.uint16)
    w2 = _c(w2, np.uint16)
    A13, B13, A2, B2 = (_c(t, np.uint16) for t in (A13, B13, A2, B2))
    token_lora_idx = _c(token_lora_idx, np.int32)
    topk_ids = _c(topk_ids, np.int32)
    topk_w = _c(topk_w, np.float32)
    M, H = x.shape
    E_tot, twoI, H2 = w13.shape
    assert H2 == H and twoI % 2 == 0
    I = twoI // 2
    KT = topk_ids.shape[1]
    if A13 is not None:
        L, _, r, _ = A13.shape
    else:
        L, r = 0, 0
    y = np.zeros((M, H), np.float64)
    rc = lib.oracle_moe_forward(_ptr(x), _ptr(w13), _ptr(w2), _ptr(A13), _ptr(B13), _ptr(A2),
                                _ptr(B2), _ptr(token_lora_idx), _ptr(topk_ids), _ptr(topk_w),
                                M, H, I, E_tot, KT, L, r, float(scaling), float(out_scale), _ptr(y))
    if rc != 0:
        raise ValueError(f"oracle_moe_forward rejected its arguments ({rc})")
    return y


def mx_quantize(w_bits, lib=None):
    """MXFP8 (E4M3 elements, one E8M0 scale per 32 along the last axis) of a
    bf16 bit array [..., K]: returns (codes uint8 [..., K], scales uint8
    [..., K/32])."""
    lib = lib or load()
    w = _c(w_bits, np.uint16)
    K = w.shape[-1]
    rows = w.size // K
    codes = np.zeros(w.shape, np.uint8)
    scales = np.zeros(w.shape[:-1] + (K // 32,), np.uint8)
    rc = lib.oracle_mx_quantize(_ptr(w), rows, K, _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError(f"oracle_mx_quantize rejected its arguments ({rc})")
    return codes, scales


def mx_dequantize(codes, scales, lib=None):
    """The float64 values an MXFP8 array stands for."""
    lib = lib or load()
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    K = codes.shape[-1]
    out = np.zeros(codes.shape, np.float64)
    rc = lib.oracle_mx_dequantize(_ptr(codes), _ptr(scales), codes.size // K, K, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_mx_dequantize rejected its arguments ({rc})")
    return out


def moe_forward_mx(x, w13q, w13s, w2q, w2s, A13, B13, A2, B2, token_lora_idx, topk_ids, topk_w,
                   scaling, out_scale=1.0, lib=None):
    """fp64 layer output [M, H] with MXFP8 expert weights (codes and scales
    as mx_quantize returns them); x and the LoRA tensors as bf16 bits."""
    lib = lib or load()
    x = _c(x, np.uint16)
    w13q, w13s, w2q, w2s = (_c(t, np.uint8) for t in (w13q, w13s, w2q, w2s))
    A13, B13, A2, B2 = (_c(t, np.uint16) for t in (A13, B13, A2, B2))
    token_lora_idx = _c(token_lora_idx, np.int32)
    topk_ids = _c(topk_ids, np.int32)
    topk_w = _c(topk_w, np.float32)
    M, H = x.shape
    E_tot, twoI, H2 = w13q.shape
    assert H2 == H and twoI % 2 == 0
    I = twoI // 2
    KT = topk_ids.shape[1]
    L, r = (A13.shape[0], A13.shape[2]) if A13 is not None else (0, 0)
    y = np.zeros((M, H), np.float64)
    rc = lib.oracle_moe_forward_mx(_ptr(x), _ptr(w13q), _ptr(w13s), _ptr(w2q), _ptr(w2s), _ptr(A13), _ptr(B13),
                                   _ptr(A2), _ptr(B2), _ptr(token_lora_idx), _ptr(topk_ids), _ptr(topk_w),
                                   M, H, I, E_tot, KT, L, r, float(scaling), float(out_scale), _ptr(y))
    if rc != 0:
        raise ValueError(f"oracle_moe_forward_mx rejected its arguments ({rc})")
    return y
