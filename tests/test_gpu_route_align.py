"""GPU routing and align against the oracle: ids and the sorted, padded
permutation bit-exact, routing weights within fp32 rounding."""
import numpy as np
import pytest
import torch

import oracle
import moe_layer_lora_gb300 as ml
from moe_layer_lora_gb300 import workloads as wl
import gpu_util as gu

pytestmark = pytest.mark.gpu


def _route_case(spec):
    inp = wl.make(spec, with_weights=False)
    d_logits = gu.dev(inp.logits)
    d_bias = gu.dev(inp.bias)
    ids_ref, w_ref = gu.oracle_route(inp)
    gu.assert_unambiguous(inp)
    ids, w = ml.mlora_moe_route(d_logits, d_bias, spec.top_k, spec.scoring, spec.renormalize, spec.n_shared,
                                spec.routed_scaling_factor)
    torch.cuda.synchronize()
    gu.check_route(ids, w, ids_ref, w_ref)
    return ids_ref


@pytest.mark.parametrize("name", wl.WORKLOADS)
def test_route_workloads(name):
    _route_case(wl.spec(name))


@pytest.mark.parametrize("M", [1, 32, 128])
def test_route_shared_sweep(M):
    _route_case(wl.spec("shared", M=M))


@pytest.mark.parametrize("over", [
    dict(renormalize=0),
    dict(scoring=wl.SCORE_SIGMOID_BIAS, renormalize=0, E=64, top_k=6),
    dict(E=1024, top_k=8, M=33),
    dict(E=3, top_k=3, M=5),
    dict(E=40, top_k=5, n_shared=2, routed_scaling_factor=2.0, M=17),
    dict(E=1, top_k=1, M=9),
    dict(E=200, top_k=64, M=3),
])
def test_route_edges(over):
    _route_case(wl.spec("tiny", **over))


def test_route_ties_lower_id():
    logits = torch.tensor([[1.0, 2.0, 2.0, 0.5, 2.0, 2.0]] * 3, dtype=torch.float32)
    ids, w = ml.mlora_moe_route(logits.cuda(), None, 4, wl.SCORE_SOFTMAX)
    assert ids.cpu().tolist() == [[1, 2, 4, 5]] * 3
    ids_ref, w_ref = oracle.moe_route(logits.numpy(), None, 4, 0, 1)
    gu.check_route(ids, w, ids_ref, w_ref)


def _align_case(ids_np, E_tot, BM):
    s_ref, e_ref, n_ref = oracle.moe_align(ids_np, E_tot, BM)
    s, e, n = ml.mlora_moe_align(torch.from_numpy(ids_np).cuda(), E_tot, BM)
    torch.cuda.synchronize()
    assert int(n.item()) == n_ref
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(e.cpu().numpy(), e_ref)


@pytest.mark.parametrize("name", wl.WORKLOADS)
@pytest.mark.parametrize("BM", [16, 32, 64, 128])
def test_align_workloads(name, BM):
    spec = wl.spec(name)
    ids_ref, _ = gu.oracle_route(wl.make(spec, with_weights=False))
    _align_case(ids_ref, spec.E_tot, BM)


def test_align_edges():
    rng = np.random.default_rng(0)
    # one expert takes every slot: many blocks of the same expert
    _align_case(np.full((300, 1), 2, np.int32), 4, 16)
    # block_m = 1 (no padding) and a large block
    ids = np.stack([rng.permutation(7)[:3] for _ in range(50)]).astype(np.int32)
    _align_case(ids, 7, 1)
    _align_case(ids, 7, 1024)
    # the largest expert count
    ids = rng.integers(0, 1024, size=(700, 4), dtype=np.int32)
    _align_case(ids, 1024, 8)
    # more slots than one pass of the scatter, ragged tail (per-thread runs,
    # staged in shared memory)
    ids = rng.integers(0, 5, size=(3001, 3), dtype=np.int32)
    _align_case(ids, 5, 64)
    # runs whose padded list does not fit in shared memory (96 experts)
    ids = rng.integers(0, 96, size=(4000, 8), dtype=np.int32)
    _align_case(ids, 96, 16)
    # several passes: one expert too many for runs, and more than 65535 slots
    ids = rng.integers(0, 97, size=(1500, 3), dtype=np.int32)
    _align_case(ids, 97, 32)
    ids = rng.integers(0, 8, size=(16500, 4), dtype=np.int32)
    _align_case(ids, 8, 128)


def test_align_unaligned_ids():
    # ids that start 4 bytes past a 16-byte boundary: the runs read them
    # one by one
    rng = np.random.default_rng(1)
    ids_np = rng.integers(0, 6, size=(2001, 3), dtype=np.int32)
    buf = torch.empty(ids_np.size + 1, dtype=torch.int32, device="cuda")
    buf[1:] = torch.from_numpy(ids_np.reshape(-1)).cuda()
    view = buf[1:].view(2001, 3)
    assert view.data_ptr() % 16 == 4
    s_ref, e_ref, n_ref = oracle.moe_align(ids_np, 6, 16)
    s, e, n = ml.mlora_moe_align(view, 6, 16)
    torch.cuda.synchronize()
    assert int(n.item()) == n_ref
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(e.cpu().numpy(), e_ref)


def test_align_empty():
    s, e, n = ml.mlora_moe_align(torch.zeros((0, 4), dtype=torch.int32, device="cuda"), 8, 16)
    torch.cuda.synchronize()
    assert int(n.item()) == 0 and s.numel() == 0 and e.numel() == 0


def _random_align_cases(n: int, seed: int = 77):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.choice([1, 3, 8, 32, 96, 97, 129, 500, 1024]))
        K = int(rng.integers(1, 9))
        M = int(rng.choice([1, 7, 100, 255, 256, 257, 1000, 3000, 9000]))
        BM = int(rng.choice([1, 16, 64, 128, 256]))
        skew = bool(rng.random() < 0.5)
        out.append((i, E, K, M, BM, skew))
    return out


@pytest.mark.parametrize("case", _random_align_cases(20), ids=lambda c: f"E{c[1]}K{c[2]}M{c[3]}BM{c[4]}")
def test_align_random(case):
    """Seeded random expert counts, slot counts (one pass, several passes,
    per-thread runs), block sizes and skewed loads: bit-exact vs the oracle."""
    i, E, K, M, BM, skew = case
    rng = np.random.default_rng(1000 + i)
    if skew:
        p = rng.dirichlet(np.full(E, 0.3))
        ids = rng.choice(E, size=(M, K), p=p).astype(np.int32)
    else:
        ids = rng.integers(0, E, size=(M, K), dtype=np.int32)
    _align_case(ids, E, BM)


@pytest.mark.parametrize("scoring", [wl.SCORE_SOFTMAX, wl.SCORE_SIGMOID_BIAS])
def test_route_nan_keys_rank_last(scoring):
    """A NaN key ranks below every number (ties among NaN keys to the lower
    id), so ids stay in range: a row of NaN logits takes experts 0..k-1, and
    a row with some NaN logits takes the top-k of its finite ones."""
    E, k = 40, 4
    logits = torch.randn(4, E, generator=torch.Generator().manual_seed(3), dtype=torch.float32)
    logits[0] = float("nan")
    logits[1, :5] = float("nan")
    bias = (torch.randn(E, generator=torch.Generator().manual_seed(4)) * 0.5).float() if scoring else None
    ids, _ = ml.mlora_moe_route(logits.cuda(), None if bias is None else bias.cuda(), k, scoring)
    ids = ids.cpu().numpy()
    assert ((ids >= 0) & (ids < E)).all()
    assert ids[0].tolist() == [0, 1, 2, 3]
    part_ids, _ = oracle.moe_route(logits[1:2, 5:].numpy(), None if bias is None else bias[5:].numpy(), k, scoring, 1)
    assert ids[1].tolist() == (part_ids[0] + 5).tolist()
    full_ids, _ = oracle.moe_route(logits[2:].numpy(), None if bias is None else bias.numpy(), k, scoring, 1)
    assert np.array_equal(ids[2:], full_ids)
