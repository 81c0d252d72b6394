"""Independent pins for the fp64 oracle.

Each ``pin_*`` function raises AssertionError when the oracle library it is
given disagrees with something the pages or plain mathematics fix: closed
forms, brute force on tiny inputs, special cases that reduce to a library
routine, and invariants.  None of them re-types the oracle's loops: the
forward pins use a dense, vectorised formulation with the adapter folded
into the weights (W + s*B*A) and a dense gate matrix, which associates the
arithmetic differently from the oracle's per-token loops.

The functions take the loaded oracle library as an argument so that
``test_oracle_mutants.py`` can run the same pins against copies of the
oracle with planted mistakes and check that every mistake is caught.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import scipy.special
import torch

import oracle
from moe_layer_lora_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- routing --

def pin_route_softmax_closed_form(lib):
    """logits (0,1,2,3), k=2: ids (3,2); renormalised weights e/(1+e), 1/(1+e);
    full-softmax weights e^3/S, e^2/S with S = 1+e+e^2+e^3."""
    logits = np.array([[0.0, 1.0, 2.0, 3.0]], np.float32)
    ids, w = oracle.moe_route(logits, None, 2, wl.SCORE_SOFTMAX, 1, lib=lib)
    assert ids.tolist() == [[3, 2]], ids
    e = math.e
    np.testing.assert_allclose(w[0], [e / (1 + e), 1 / (1 + e)], rtol=1e-14)
    ids, w = oracle.moe_route(logits, None, 2, wl.SCORE_SOFTMAX, 0, lib=lib)
    S = 1 + e + e * e + e ** 3
    assert ids.tolist() == [[3, 2]]
    np.testing.assert_allclose(w[0], [e ** 3 / S, e * e / S], rtol=1e-14)


def pin_route_ties_lower_id(lib):
    """Equal keys rank by the lower expert id (the order fixes slot numbering)."""
    logits = np.array([[1.0, 2.0, 2.0, 0.5, 2.0]], np.float32)
    ids, w = oracle.moe_route(logits, None, 3, wl.SCORE_SOFTMAX, 1, lib=lib)
    assert ids.tolist() == [[1, 2, 4]], ids
    np.testing.assert_allclose(w[0], [1 / 3] * 3, rtol=1e-14)


def _brute_topk(keys, k):
    """The unique k-subset whose every member outranks every non-member
    (descending key, ties to lower id), found by enumerating all subsets."""
    E = len(keys)
    found = []
    for S in itertools.combinations(range(E), k):
        inside = set(S)
        ok = all((keys[a] > keys[b]) or (keys[a] == keys[b] and a < b)
                 for a in inside for b in range(E) if b not in inside)
        if ok:
            found.append(S)
    assert len(found) == 1
    return sorted(found[0], key=lambda e: (-keys[e], e))


def pin_route_softmax_brute_force(lib):
    rng = np.random.default_rng(7)
    M, E, k = 12, 7, 3
    logits = rng.standard_normal((M, E)).astype(np.float32)
    for renorm in (1, 0):
        ids, w = oracle.moe_route(logits, None, k, wl.SCORE_SOFTMAX, renorm, lib=lib)
        full = scipy.special.softmax(logits.astype(np.float64), axis=1)
        for m in range(M):
            assert list(ids[m]) == _brute_topk(list(logits[m]), k)
            sel = full[m, ids[m]]
            want = sel / sel.sum() if renorm else sel
            np.testing.assert_allclose(w[m], want, rtol=1e-12)


def pin_route_sigmoid_bias_shared(lib):
    """Sigmoid+bias selection on sigmoid(l)+b, weights sigmoid(l) renormalised
    over routed slots; shared slots E..E+n-1 at weight 1/rsf."""
    rng = np.random.default_rng(11)
    M, E, k, n_sh, rsf = 10, 9, 3, 2, 2.5
    logits = rng.standard_normal((M, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.7).astype(np.float32)
    ids, w = oracle.moe_route(logits, bias, k, wl.SCORE_SIGMOID_BIAS, 1, n_sh, rsf, lib=lib)
    assert ids.shape == (M, k + n_sh)
    sig = scipy.special.expit(logits.astype(np.float64))
    for m in range(M):
        keys = list(sig[m] + bias.astype(np.float64))
        assert list(ids[m, :k]) == _brute_topk(keys, k)
        assert list(ids[m, k:]) == [E, E + 1]
        np.testing.assert_allclose(w[m, k:], [0.4, 0.4], rtol=1e-15)
        s = sig[m, ids[m, :k]]
        np.testing.assert_allclose(w[m, :k], s / s.sum(), rtol=1e-12)
    ids, w = oracle.moe_route(logits, bias, k, wl.SCORE_SIGMOID_BIAS, 0, 0, 1.0, lib=lib)
    for m in range(M):
        np.testing.assert_allclose(w[m], sig[m, ids[m]], rtol=1e-12)


def pin_route_golden_shared(lib):
    g = _golden("route_shared_tiny.json")
    logits = np.array(g["logits"], np.float32)
    ids, w = oracle.moe_route(logits, None, g["top_k"], wl.SCORE_SOFTMAX, 1, g["n_shared"],
                              g["routed_scaling_factor"], lib=lib)
    assert ids.tolist() == g["expected_ids"]
    np.testing.assert_allclose(w[:, g["top_k"]:], g["expected_shared_weight"], rtol=1e-15)


# ------------------------------------------------------------------- align --

def brute_align(topk_ids, E_tot, BM):
    """Stable sort of flat slots by expert, each expert padded to BM with the
    sentinel M*K'; built with Python's sorted() rather than counting."""
    flat = np.asarray(topk_ids).reshape(-1)
    S = len(flat)
    order = sorted(range(S), key=lambda f: (int(flat[f]), f))
    out, experts = [], []
    for e, grp in itertools.groupby(order, key=lambda f: int(flat[f])):
        grp = list(grp)
        nb = -(-len(grp) // BM)
        out += grp + [S] * (nb * BM - len(grp))
        experts += [e] * nb
    return out, experts


def pin_align_brute_force(lib):
    rng = np.random.default_rng(3)
    for (M, KT, Et, BM) in [(5, 2, 4, 4), (13, 3, 6, 8), (1, 1, 3, 16), (40, 4, 9, 16), (7, 5, 5, 1)]:
        ids = np.stack([rng.permutation(Et)[:KT] for _ in range(M)]).astype(np.int32)
        s_ids, e_ids, npp = oracle.moe_align(ids, Et, BM, lib=lib)
        want, want_e = brute_align(ids, Et, BM)
        assert npp == len(want)
        assert s_ids[:npp].tolist() == want
        assert e_ids[: npp // BM].tolist() == want_e
        assert (s_ids[npp:] == M * KT).all() and (e_ids[npp // BM:] == -1).all()
        # invariants: every slot exactly once, blocks hold one expert each
        real = s_ids[s_ids < M * KT]
        assert sorted(real.tolist()) == list(range(M * KT))
        flat = ids.reshape(-1)
        for b in range(npp // BM):
            blk = s_ids[b * BM:(b + 1) * BM]
            assert all(flat[f] == e_ids[b] for f in blk if f < M * KT)
        assert npp % BM == 0
        assert len(s_ids) == oracle.moe_align_max_padded(M, KT, Et, BM, lib=lib) >= npp


def pin_align_golden(lib):
    g = _golden("align_tiny.json")
    ids = np.array(g["topk_ids"], np.int32)
    s_ids, e_ids, npp = oracle.moe_align(ids, g["E_tot"], g["block_m"], lib=lib)
    assert npp == g["expected_num_post_padded"]
    assert s_ids.tolist() == g["expected_sorted_ids"]
    assert e_ids.tolist() == g["expected_expert_ids"]


# ----------------------------------------------------------------- forward --

def dense_forward(x, w13, w2, A13, B13, A2, B2, idx, ids, w, s, out_scale):
    """y = out_scale * sum_e G[:, e] * FFN_{e,l}(x) with the dense gate matrix
    G and each (adapter, expert) weight materialised as W + s*B@A."""
    M, H = x.shape
    Et, twoI, _ = w13.shape
    I = twoI // 2
    G = np.zeros((M, Et))
    np.add.at(G, (np.repeat(np.arange(M), ids.shape[1]), ids.reshape(-1)), w.reshape(-1))
    if idx is None:
        idx = np.full(M, -1)
    y = np.zeros((M, H))
    for l in np.unique(idx):
        rows = idx == l
        for e in range(Et):
            W13 = w13[e] + (s * B13[l, e] @ A13[l, e] if l >= 0 else 0.0)
            W2 = w2[e] + (s * B2[l, e] @ A2[l, e] if l >= 0 else 0.0)
            h = x[rows] @ W13.T
            a = h[:, :I] * scipy.special.expit(h[:, :I]) * h[:, I:]
            y[rows] += G[rows, e][:, None] * (a @ W2.T)
    return out_scale * y


def _tiny_inputs(seed=5, M=9, H=24, I=16, E=5, k=2, L=3, r=4, n_shared=0, rsf=1.0,
                 scoring=wl.SCORE_SOFTMAX):
    s = wl.spec("tiny", M=M, H=H, I=I, E=E, top_k=k, L=L, r=r, n_shared=n_shared,
                routed_scaling_factor=rsf, scoring=scoring, seed=seed,
                lora_mode="uniform" if L else "none")
    return s, wl.make(s)


def _f64(t):
    return None if t is None else wl.to_f64(t)


def _oracle_y(lib, inp, ids, w, scaling, out_scale=1.0, lora=True, idx=None):
    b = wl.bits
    use = lora and inp.A13 is not None
    return oracle.moe_forward(
        b(inp.x), b(inp.w13), b(inp.w2),
        b(inp.A13) if use else None, b(inp.B13) if use else None,
        b(inp.A2) if use else None, b(inp.B2) if use else None,
        (idx if idx is not None else inp.token_lora_idx.numpy()) if use else None,
        ids, w.astype(np.float32), scaling, out_scale, lib=lib)


def pin_forward_dense_brute_force(lib):
    for seed, (H, I, E, k, L, r) in [(5, (24, 16, 5, 2, 3, 4)), (6, (16, 40, 3, 3, 2, 8))]:
        s, inp = _tiny_inputs(seed=seed, H=H, I=I, E=E, k=k, L=L, r=r)
        ids, w = oracle.moe_route(inp.logits.numpy(), None, k, 0, 1, lib=lib)
        y = _oracle_y(lib, inp, ids, w, s.scaling)
        f = _f64
        ref = dense_forward(f(inp.x), f(inp.w13), f(inp.w2), f(inp.A13), f(inp.B13), f(inp.A2),
                            f(inp.B2), inp.token_lora_idx.numpy(), ids,
                            w.astype(np.float32).astype(np.float64), s.scaling, 1.0)
        np.testing.assert_allclose(y, ref, rtol=1e-9, atol=1e-9 * np.abs(ref).max())


def pin_forward_dense_mlp(lib):
    """E=1, top_k=1 is a plain SwiGLU MLP: y = (silu(x W1^T) * (x W3^T)) W2^T."""
    s, inp = _tiny_inputs(seed=8, M=6, H=32, I=24, E=1, k=1, L=0, r=0)
    ids, w = oracle.moe_route(inp.logits.numpy(), None, 1, 0, 1, lib=lib)
    assert (ids == 0).all() and np.allclose(w, 1.0)
    y = _oracle_y(lib, inp, ids, w, 0.0)
    x = torch.from_numpy(_f64(inp.x))
    W = torch.from_numpy(_f64(inp.w13[0]))
    W1, W3 = W[:24], W[24:]
    W2 = torch.from_numpy(_f64(inp.w2[0]))
    ref = torch.nn.functional.linear(
        torch.nn.functional.silu(torch.nn.functional.linear(x, W1)) * torch.nn.functional.linear(x, W3), W2)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-10, atol=1e-12)


def pin_forward_lora_b_zero_is_base(lib):
    """All B = 0: the adapters contribute exactly nothing, so the output is the
    base MoE, identical to the call without adapters and to all-(-1)."""
    s, inp = _tiny_inputs(seed=9)
    ids, w = oracle.moe_route(inp.logits.numpy(), None, s.top_k, 0, 1, lib=lib)
    base = _oracle_y(lib, inp, ids, w, s.scaling, lora=False)
    inp.B13 = torch.zeros_like(inp.B13)
    inp.B2 = torch.zeros_like(inp.B2)
    y0 = _oracle_y(lib, inp, ids, w, s.scaling)
    assert np.array_equal(y0, base)
    allnone = _oracle_y(lib, inp, ids, w, s.scaling, idx=np.full(s.M, -1, np.int32))
    assert np.array_equal(allnone, base)


def pin_forward_no_adapter_tokens_equal_base(lib):
    s, inp = _tiny_inputs(seed=10, M=16)
    ids, w = oracle.moe_route(inp.logits.numpy(), None, s.top_k, 0, 1, lib=lib)
    base = _oracle_y(lib, inp, ids, w, s.scaling, lora=False)
    y = _oracle_y(lib, inp, ids, w, s.scaling)
    none = inp.token_lora_idx.numpy() == -1
    some = ~none
    assert none.any() and some.any()
    assert np.array_equal(y[none], base[none])
    assert np.abs(y[some] - base[some]).max() > 1e-3


def pin_forward_linear_in_scaling(lib):
    """With only the down adapter non-zero, y(s) = y(0) + s*(y(1) - y(0))."""
    s, inp = _tiny_inputs(seed=12)
    inp.B13 = torch.zeros_like(inp.B13)
    ids, w = oracle.moe_route(inp.logits.numpy(), None, s.top_k, 0, 1, lib=lib)
    y0 = _oracle_y(lib, inp, ids, w, 0.0)
    y1 = _oracle_y(lib, inp, ids, w, 1.0)
    y3 = _oracle_y(lib, inp, ids, w, 3.0)
    np.testing.assert_allclose(y3, y0 + 3.0 * (y1 - y0), rtol=1e-10, atol=1e-12)
    assert np.abs(y1 - y0).max() > 1e-3


def pin_forward_token_permutation(lib):
    s, inp = _tiny_inputs(seed=13, M=11)
    ids, w = oracle.moe_route(inp.logits.numpy(), None, s.top_k, 0, 1, lib=lib)
    y = _oracle_y(lib, inp, ids, w, s.scaling)
    perm = np.random.default_rng(0).permutation(s.M)
    inp.x = inp.x[perm].contiguous()
    idx = inp.token_lora_idx.numpy()[perm]
    yp = _oracle_y(lib, inp, ids[perm], w[perm], s.scaling, idx=np.ascontiguousarray(idx))
    np.testing.assert_allclose(yp, y[perm], rtol=1e-13, atol=1e-15)


def shared_mlp_dense(x, W13, W2):
    """The separate shared-expert MLP of the unfused form, via torch (fp64)."""
    I = W13.shape[0] // 2
    xt, W, W2t = (torch.from_numpy(a) for a in (x, W13, W2))
    F = torch.nn.functional
    return F.linear(F.silu(F.linear(xt, W[:I])) * F.linear(xt, W[I:]), W2t).numpy()


def pin_forward_shared_fusion_equals_unfused(lib):
    """Fused: shared expert appended as a slot of weight 1/rsf, layer output
    scaled by rsf.  Unfused: rsf * routed MoE + separate shared MLP."""
    rsf = 2.5
    s, inp = _tiny_inputs(seed=14, M=7, H=32, I=16, E=6, k=3, L=0, r=0, n_shared=1, rsf=rsf,
                          scoring=wl.SCORE_SIGMOID_BIAS)
    logits, bias = inp.logits.numpy(), inp.bias.numpy()
    ids, w = oracle.moe_route(logits, bias, 3, 1, 1, 1, rsf, lib=lib)
    fused = _oracle_y(lib, inp, ids, w, 0.0, out_scale=rsf)
    routed = _oracle_y(lib, inp, np.ascontiguousarray(ids[:, :3]), np.ascontiguousarray(w[:, :3]),
                       0.0, out_scale=1.0)
    shared = shared_mlp_dense(_f64(inp.x), _f64(inp.w13[6]), _f64(inp.w2[6]))
    np.testing.assert_allclose(fused, rsf * routed + shared, rtol=1e-6,
                               atol=1e-6 * np.abs(shared).max())


def pin_forward_lora_on_shared_slot(lib):
    """Shared slots take the token's adapter like any expert (brute force)."""
    s, inp = _tiny_inputs(seed=15, M=8, H=16, I=8, E=4, k=2, L=2, r=4, n_shared=1, rsf=2.0,
                          scoring=wl.SCORE_SIGMOID_BIAS)
    ids, w = oracle.moe_route(inp.logits.numpy(), inp.bias.numpy(), 2, 1, 1, 1, 2.0, lib=lib)
    y = _oracle_y(lib, inp, ids, w, s.scaling, out_scale=2.0)
    f = _f64
    ref = dense_forward(f(inp.x), f(inp.w13), f(inp.w2), f(inp.A13), f(inp.B13), f(inp.A2),
                        f(inp.B2), inp.token_lora_idx.numpy(), ids,
                        w.astype(np.float32).astype(np.float64), s.scaling, 2.0)
    np.testing.assert_allclose(y, ref, rtol=1e-9, atol=1e-9 * np.abs(ref).max())


ALL_PINS = [
    pin_route_softmax_closed_form, pin_route_ties_lower_id, pin_route_softmax_brute_force,
    pin_route_sigmoid_bias_shared, pin_route_golden_shared,
    pin_align_brute_force, pin_align_golden,
    pin_forward_dense_brute_force, pin_forward_dense_mlp, pin_forward_lora_b_zero_is_base,
    pin_forward_no_adapter_tokens_equal_base, pin_forward_linear_in_scaling,
    pin_forward_token_permutation, pin_forward_shared_fusion_equals_unfused,
    pin_forward_lora_on_shared_slot,
]
