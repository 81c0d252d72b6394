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


# ------------------------------------------------------------------ MXFP8 --
# The MXFP8 oracle follows the OCP Microscaling Formats Specification v1.0
# (blocks of 32 elements, E8M0 scale, E4M3 elements; conversion: shared
# exponent floor(log2(max|v|)) - 8, elements rounded to nearest-even and
# saturated).  The pins below check it against torch's own float8_e4m3fn
# codec, against a brute-force nearest-value search over the 256 codes,
# against hand-derived blocks, and (the layer) against a dense vectorised
# formulation.

def e4m3_table():
    """Value of every E4M3 code, from torch's float8_e4m3fn (an implementation
    of the same format that shares nothing with the oracle)."""
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def brute_mx_block(v):
    """One block of 32 values: (codes, scale byte) by exhaustive search for
    the nearest finite E4M3 value of v / 2^shared, ties to the even code."""
    v = np.asarray(v, np.float64)
    amax = float(np.abs(v).max())
    se = -127 if amax == 0.0 else min(127, max(-127, math.frexp(amax)[1] - 1 - 8))
    x = v * 2.0 ** -se
    pos = e4m3_table()[:0x7F]          # codes 0x00 .. 0x7E: 0 .. 448
    codes = np.zeros(32, np.uint8)
    for i, xi in enumerate(x):
        a = abs(xi)
        if a >= 448.0:
            c = 0x7E
        else:
            d = np.abs(pos - a)
            cand = np.flatnonzero(d == d.min())
            c = int(cand[0]) if len(cand) == 1 else int(cand[cand % 2 == 0][0])
        codes[i] = c | (0x80 if math.copysign(1.0, xi) < 0 else 0)
    return codes, se + 127


def brute_mx_round_trip(a):
    """Rows of values through MXFP8 and back (blocks of 32 along the last
    axis), with the brute-force quantizer."""
    a = np.asarray(a, np.float64)
    out = np.empty_like(a)
    tab = e4m3_table()
    for idx in np.ndindex(a.shape[:-1]):
        for b in range(a.shape[-1] // 32):
            c, sc = brute_mx_block(a[idx][b * 32:(b + 1) * 32])
            out[idx][b * 32:(b + 1) * 32] = tab[c] * 2.0 ** (sc - 127)
    return out


def _bf16_bits(v):
    return torch.tensor(np.asarray(v, np.float64), dtype=torch.float32).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def pin_mx_e4m3_values_match_torch(lib):
    """Every code's value (scale byte 127 = 2^0), the sign of zero included,
    and the scale bytes as powers of two."""
    t = e4m3_table()
    v = oracle.mx_dequantize(np.arange(256, dtype=np.uint8).reshape(8, 32), np.full((8, 1), 127, np.uint8),
                             lib=lib).reshape(-1)
    nan = np.isnan(t)
    assert nan.sum() == 2 and np.array_equal(np.isnan(v), nan)
    assert np.array_equal(v[~nan], t[~nan])
    assert np.array_equal(np.signbit(v[~nan]), np.signbit(t[~nan]))
    one = np.full((1, 32), 0x38, np.uint8)  # 1.0
    for sc in (0, 1, 100, 127, 200, 254):
        got = oracle.mx_dequantize(one, np.array([[sc]], np.uint8), lib=lib)
        assert (got == 2.0 ** (sc - 127)).all()


def pin_mx_quantize_golden(lib):
    """Blocks worked out by hand from the specification's conversion.  The
    first holds 1.0, so max|v| = 1, the shared exponent is 0 - 8 and the
    scale byte 119; every element is then scaled by 2^8:
      1.0          -> 256   = 2^8 * 1.000: code 0x78
      9.5/256      -> 9.5, halfway between 9 and 10: even mantissa, 10 = 0x52
      10.5/256     -> 10.5, halfway between 10 and 11: 10 again, 0x52
      -0.0         -> negative zero, 0x80
      2^-17        -> 2^-9, the smallest subnormal, 0x01
      2^-18        -> 2^-10, halfway between 0 and 2^-9: 0, 0x00
      1.5 * 2^-18  -> 0.75 * 2^-9: 2^-9, 0x01
      1.9 (bf16 1.8984375) -> 486, above 448: saturated, 0x7E
    and a block of zeros takes the smallest scale byte, 0."""
    v = np.zeros((2, 32))
    v[0, :8] = [1.0, 9.5 / 256, 10.5 / 256, -0.0, 2.0 ** -17, 2.0 ** -18, 1.5 * 2.0 ** -18, 1.9]
    codes, scales = oracle.mx_quantize(_bf16_bits(v), lib=lib)
    assert scales.tolist() == [[119], [0]]
    assert codes[0, :8].tolist() == [0x78, 0x52, 0x52, 0x80, 0x01, 0x00, 0x01, 0x7E]
    assert (codes[1] == 0).all()


def pin_mx_quantize_brute_force(lib):
    """Random bf16 blocks over many magnitudes, zeros and outliers included,
    against the exhaustive nearest-value search."""
    rng = np.random.default_rng(31)
    rows = []
    for mag in (1e-30, 1e-6, 3e-3, 1.0, 7.0, 1e4, 1e30):
        rows.append(rng.standard_normal(32) * mag)
    r = rng.standard_normal(32)
    r[rng.integers(0, 32)] = 200.0  # one outlier: the rest fall towards the subnormals
    rows.append(r)
    r = rng.standard_normal(32)
    r[::3] = 0.0
    rows.append(r)
    rows.append(rng.choice([-1.0, 1.0], 32) * 2.0 ** rng.integers(-20, 5, 32))
    bits = _bf16_bits(np.array(rows))
    codes, scales = oracle.mx_quantize(bits, lib=lib)
    vals = wl.to_f64(wl.from_bits(bits))
    for i, row in enumerate(vals):
        c, sc = brute_mx_block(row)
        assert scales[i, 0] == sc, (i, scales[i, 0], sc)
        assert np.array_equal(codes[i], c), (i, codes[i], c)


def _to_bf16(a):
    """Round to bf16 through fp32 (torch's conversions, nearest even)."""
    return torch.from_numpy(np.asarray(a, np.float64)).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def dense_forward_mx(x, w13q, w13s, w2q, w2s, A13, B13, A2, B2, idx, ids, w, s, out_scale):
    """The MXFP8 layer as dense vectorised algebra: quantized x and SwiGLU
    output (brute-force quantizer), weights decoded with torch's E4M3 codec,
    adapters on the unquantized activations (the gate_up shrink result
    s * x A13^T rounded to bf16 by torch), a dense gate matrix."""
    tab = e4m3_table()
    W13 = tab[w13q] * np.repeat(2.0 ** (w13s.astype(np.float64) - 127), 32, axis=-1)
    W2 = tab[w2q] * np.repeat(2.0 ** (w2s.astype(np.float64) - 127), 32, axis=-1)
    M, H = x.shape
    Et, twoI, _ = W13.shape
    I = twoI // 2
    G = np.zeros((M, Et))
    np.add.at(G, (np.repeat(np.arange(M), ids.shape[1]), ids.reshape(-1)), w.reshape(-1))
    idx = np.full(M, -1) if idx is None else idx
    xq = brute_mx_round_trip(x)
    y = np.zeros((M, H))
    for l in np.unique(idx):
        rows = idx == l
        for e in range(Et):
            if not G[rows, e].any():
                continue
            h = xq[rows] @ W13[e].T
            if l >= 0:
                h = h + _to_bf16(s * (x[rows] @ A13[l, e].T)) @ B13[l, e].T
            a = h[:, :I] * scipy.special.expit(h[:, :I]) * h[:, I:]
            d = brute_mx_round_trip(a) @ W2[e].T
            if l >= 0:
                d = d + s * (a @ A2[l, e].T) @ B2[l, e].T
            y[rows] += G[rows, e][:, None] * d
    return out_scale * y


def _mx_inputs(seed, M=6, H=64, I=32, E=4, k=2, L=2, r=8):
    s, inp = _tiny_inputs(seed=seed, M=M, H=H, I=I, E=E, k=k, L=L, r=r)
    w13q, w13s = oracle.mx_quantize(wl.bits(inp.w13))
    w2q, w2s = oracle.mx_quantize(wl.bits(inp.w2))
    return s, inp, (w13q, w13s, w2q, w2s)


def _oracle_y_mx(lib, inp, q, ids, w, scaling, lora=True, out_scale=1.0):
    b = wl.bits
    use = lora and inp.A13 is not None
    return oracle.moe_forward_mx(b(inp.x), *q, b(inp.A13) if use else None, b(inp.B13) if use else None,
                                 b(inp.A2) if use else None, b(inp.B2) if use else None,
                                 inp.token_lora_idx.numpy() if use else None, ids, w.astype(np.float32),
                                 scaling, out_scale, lib=lib)


def pin_mx_forward_dense(lib):
    for seed, (H, I, E, k, L, r) in [(41, (64, 32, 4, 2, 2, 8)), (42, (32, 96, 3, 3, 3, 16))]:
        s, inp, q = _mx_inputs(seed, H=H, I=I, E=E, k=k, L=L, r=r)
        ids, w = oracle.moe_route(inp.logits.numpy(), None, k, 0, 1, lib=lib)
        y = _oracle_y_mx(lib, inp, q, ids, w, s.scaling)
        f = _f64
        ref = dense_forward_mx(f(inp.x), *q, f(inp.A13), f(inp.B13), f(inp.A2), f(inp.B2),
                               inp.token_lora_idx.numpy(), ids, w.astype(np.float32).astype(np.float64),
                               s.scaling, 1.0)
        np.testing.assert_allclose(y, ref, rtol=1e-9, atol=1e-9 * np.abs(ref).max())


def pin_mx_forward_b_zero_is_base(lib):
    """All adapter B = 0: the MXFP8 layer equals itself without adapters."""
    s, inp, q = _mx_inputs(43)
    ids, w = oracle.moe_route(inp.logits.numpy(), None, s.top_k, 0, 1, lib=lib)
    base = _oracle_y_mx(lib, inp, q, ids, w, s.scaling, lora=False)
    inp.B13 = torch.zeros_like(inp.B13)
    inp.B2 = torch.zeros_like(inp.B2)
    assert np.array_equal(_oracle_y_mx(lib, inp, q, ids, w, s.scaling), base)


ALL_PINS = [
    pin_route_softmax_closed_form, pin_route_ties_lower_id, pin_route_softmax_brute_force,
    pin_route_sigmoid_bias_shared, pin_route_golden_shared,
    pin_align_brute_force, pin_align_golden,
    pin_forward_dense_brute_force, pin_forward_dense_mlp, pin_forward_lora_b_zero_is_base,
    pin_forward_no_adapter_tokens_equal_base, pin_forward_linear_in_scaling,
    pin_forward_token_permutation, pin_forward_shared_fusion_equals_unfused,
    pin_forward_lora_on_shared_slot,
    pin_mx_e4m3_values_match_torch, pin_mx_quantize_golden, pin_mx_quantize_brute_force,
    pin_mx_forward_dense, pin_mx_forward_b_zero_is_base,
]
