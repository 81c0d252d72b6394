"""The fused MoE-LoRA layer on the GPU against the fp64 oracle.

Every output of the five workloads at full size is compared (decode,
prefill, the shared-expert sweep, adapter stress), as is every output of the
small and edge cases; the random wide layers and the 65 536-token layer
compare sampled token rows (the oracle computes one token at a time, so a
row subset of its inputs gives exactly those rows).  The benchmark's launch
configuration (a replayed CUDA graph after an L2 flush) is checked to equal
an eager call bit for bit.  Tolerance: relative Frobenius error <= 1e-2 and
max abs error <= 5e-2 * rms(oracle).  Sigmoid+bias cases first check that
their seeded keys hold no near-tie (an ambiguous input)."""
import numpy as np
import pytest
import torch

import oracle
import pins
import moe_layer_lora_gb300 as ml
from moe_layer_lora_gb300 import workloads as wl
import gpu_util as gu

pytestmark = pytest.mark.gpu


def _layer(spec, rows=None, label=""):
    inp = wl.make(spec, device="cuda")
    gu.assert_unambiguous(inp)
    d = gu.DeviceInputs(inp)
    ids, w = gu.gpu_route(d)
    ws = torch.empty(ml.mlora_moe_workspace_size(spec.M, spec.H, spec.I, spec.E_tot, spec.K_total,
                                                 spec.L if spec.has_lora else 0, spec.r if spec.has_lora else 0),
                     dtype=torch.uint8, device="cuda")
    y = gu.gpu_forward(d, ids, w, workspace=ws)
    torch.cuda.synchronize()
    assert ml.mlora_moe_read_status(ws) == 0
    ids_ref, w_ref = gu.oracle_route(inp)
    gu.check_route(ids, w, ids_ref, w_ref)
    y_ref = gu.oracle_forward(inp, ids_ref, w_ref, rows=rows)
    yg = y if rows is None else y[torch.as_tensor(rows, device="cuda")]
    errs = gu.check_y(yg, y_ref, label or spec.name)
    return inp, d, ids, w, y, ids_ref, w_ref, errs


def test_tiny():
    _layer(wl.spec("tiny"))


def test_mid_width_tiles_ragged():
    """Eight tokens over eight experts on a layer whose I and H are not
    multiples of the 192-row tile (the width a launch of 7 or 8 blocks
    takes here): the last gate_up slab holds 8 valid rows of each half and
    the last down slab 8 (MMA N trimmed to 16), with adapters."""
    _layer(wl.spec("decode", M=8, H=2888, I=1448, E=8, top_k=2, L=4, r=16, seed=150), label="192-row ragged")


@pytest.mark.parametrize("M", [1, 2, 5])
def test_decode_few_tokens(M):
    """Decode-shaped layers with a handful of tokens: the launches whose tile
    width is 192 or 128 rows instead of 256, with adapters."""
    _layer(wl.spec("decode", M=M), label=f"decode M={M}")


def test_decode_full():
    _layer(wl.spec("decode"))


def test_prefill_full():
    """All 8192 tokens of the prefill layer (16 sequences of 512, one
    adapter each, two without) against the oracle."""
    _layer(wl.spec("prefill"))


@pytest.mark.parametrize("M", [1, 32, 128])
def test_shared_fusion_matches_unfused(M):
    """Fused shared slot (weight 1/rsf, output scaled by rsf) against the
    unfused form: rsf * routed MoE (oracle) + separate shared MLP."""
    s = wl.spec("shared", M=M)
    inp, d, ids, w, y, ids_ref, w_ref, _ = _layer(s)
    k = s.top_k
    routed = oracle.moe_forward(wl.bits(inp.x), gu._hbits(inp.w13), gu._hbits(inp.w2), None, None, None, None,
                                None, np.ascontiguousarray(ids_ref[:, :k]),
                                np.ascontiguousarray(w_ref[:, :k]).astype(np.float32), 0.0, 1.0)
    shared = pins.shared_mlp_dense(wl.to_f64(inp.x), wl.to_f64(inp.w13[s.E]), wl.to_f64(inp.w2[s.E]))
    unfused = s.routed_scaling_factor * routed + shared
    gu.check_y(y, unfused, f"shared M={M} vs unfused")


def test_stress_full_and_early_exit():
    """All 512 tokens of the adapter-stress layer (64 adapters of rank 64,
    Zipf, a quarter without), then the same batch with every token at -1."""
    s = wl.spec("stress")
    inp, d, ids, w, y, ids_ref, w_ref, _ = _layer(s)
    # every token without an adapter: the LoRA work exits on the device and
    # the output equals the adapter-free layer bit for bit
    none = torch.full((s.M,), -1, dtype=torch.int32, device="cuda")
    y_none = gu.gpu_forward(d, ids, w, idx=none)
    y_base = gu.gpu_forward(d, ids, w, lora=False)
    torch.cuda.synchronize()
    assert torch.equal(y_none, y_base)
    y_ref = gu.oracle_forward(inp, ids_ref, w_ref, lora=False)
    gu.check_y(y_base, y_ref, "stress all -1")


@pytest.mark.parametrize("over", [
    dict(M=37, H=136, I=72, E=5, top_k=3, L=3, r=24, seed=101),             # ragged K, N, rank
    dict(M=5, H=64, I=64, E=6, top_k=2, L=2, r=48, seed=102),               # rank 48
    dict(M=130, H=256, I=128, E=3, top_k=1, L=1, r=16, seed=103),           # >128 slots of one expert
    dict(M=9, H=8, I=8, E=4, top_k=4, L=5, r=64, seed=104),                 # tiny H/I, top_k = E
    dict(M=300, H=200, I=328, E=16, top_k=2, L=70, r=8, seed=105),          # L > 64 adapters
    dict(M=64, H=512, I=256, E=8, top_k=2, n_shared=2, routed_scaling_factor=2.0,
         scoring=wl.SCORE_SIGMOID_BIAS, L=4, r=16, seed=106),               # shared slots with adapters
    dict(M=16, H=256, I=128, E=8, top_k=2, L=0, r=0, lora_mode="none", seed=107),  # no adapters
    dict(M=24, H=384, I=136, E=8, top_k=2, renormalize=0, L=4, r=32, seed=108),
    # more than 4096 slots: the tensor-core shrink on ragged K and rank
    dict(M=1100, H=136, I=72, E=5, top_k=4, L=3, r=24, seed=109),
    dict(M=1030, H=64, I=200, E=6, top_k=4, L=9, r=8, seed=110),
    dict(M=1100, H=64, I=64, E=96, top_k=4, L=3, r=8, seed=112),           # runs align, not staged
])
def test_edges(over):
    _layer(wl.spec("tiny", **over), label=str(over))


def test_empty_batch():
    s = wl.spec("tiny")
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    e = torch.empty((0, s.H), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((0, s.K_total), dtype=torch.int32, device="cuda")
    w = torch.empty((0, s.K_total), dtype=torch.float32, device="cuda")
    y = ml.mlora_moe_forward(e, d.w13, d.w2, d.A13, d.B13, d.A2, d.B2,
                             torch.empty(0, dtype=torch.int32, device="cuda"), ids, w, 2.0)
    assert y.shape == (0, s.H)


def test_wait_timeout_is_reported_and_the_context_recovers():
    """Every CTA first waits on a workspace flag that nothing sets, with a
    ~1 ms limit: the kernel must give up, report MLORA_DEV_TIMEOUT in the
    status word and exit cleanly; the next forward on the same workspace is
    clean and matches the oracle."""
    s = wl.spec("tiny")
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    ids, w = gu.gpu_route(d)
    ws = torch.empty(ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r), dtype=torch.uint8,
                     device="cuda")
    ml.mlora_set_wait_test(2_000_000, True)
    try:
        gu.gpu_forward(d, ids, w, workspace=ws)
        st = ml.mlora_moe_read_status(ws)
    finally:
        ml.mlora_set_wait_test(0, False)
    assert st & ml.DEV_TIMEOUT, st
    y = gu.gpu_forward(d, ids, w, workspace=ws)
    assert ml.mlora_moe_read_status(ws) == 0
    ids_ref, w_ref = gu.oracle_route(inp)
    gu.check_y(y, gu.oracle_forward(inp, ids_ref, w_ref), "after a timed-out forward")


@pytest.mark.parametrize("L", [64, 65])
def test_block_adapter_sets_word_edges(L):
    """Blocks holding adapters on both sides of the 32-adapter word boundary
    and the last adapter id, with tokens without an adapter between them:
    a block's adapter list comes from a 64-bit set when there are at most 64
    adapters, and from one warp minimum per adapter beyond."""
    s = wl.spec("tiny", M=40, H=64, I=64, E=2, top_k=1, L=L, r=8, seed=611 + L)
    inp = wl.make(s, device="cuda")
    gu.assert_unambiguous(inp)
    idx = np.array([(0, 31, 32, L - 1, -1, 1, 30, 33)[i % 8] for i in range(s.M)], np.int32)
    d = gu.DeviceInputs(inp)
    ids, w = gu.gpu_route(d)
    y = gu.gpu_forward(d, ids, w, idx=torch.from_numpy(idx).cuda())
    torch.cuda.synchronize()
    ids_ref, w_ref = gu.oracle_route(inp)
    gu.check_y(y, gu.oracle_forward(inp, ids_ref, w_ref, idx=idx), f"adapter sets L={L}")


def test_bad_device_values_are_flagged():
    """Out-of-range adapter ids act as 'no adapter', out-of-range expert ids
    drop their slot; both set a bit of the device status word."""
    s = wl.spec("tiny")
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    ids, w = gu.gpu_route(d)
    ws = torch.empty(ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r), dtype=torch.uint8,
                     device="cuda")
    bad_idx = d.idx.clone()
    bad_idx[3] = s.L + 7
    y = gu.gpu_forward(d, ids, w, idx=bad_idx, workspace=ws)
    assert ml.mlora_moe_read_status(ws) == ml.DEV_BAD_LORA_IDX
    fixed = inp.token_lora_idx.numpy().copy()
    fixed[3] = -1
    ids_ref, w_ref = gu.oracle_route(inp)
    gu.check_y(y, gu.oracle_forward(inp, ids_ref, w_ref, idx=fixed), "bad adapter id")
    bad_ids = ids.clone()
    bad_ids[5, 1] = s.E_tot + 3
    y2 = gu.gpu_forward(d, bad_ids, w, workspace=ws)
    assert ml.mlora_moe_read_status(ws) == ml.DEV_BAD_EXPERT_ID
    w_drop = w_ref.copy()
    w_drop[5, 1] = 0.0
    gu.check_y(y2, gu.oracle_forward(inp, ids_ref, w_drop), "dropped slot")


def test_graph_capture_replay():
    """Route + forward captured once, replayed on new inputs written into the
    same buffers; each replay matches an eager call."""
    s = wl.spec("tiny", M=48, seed=111)
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    ids = torch.empty((s.M, s.K_total), dtype=torch.int32, device="cuda")
    w = torch.empty((s.M, s.K_total), dtype=torch.float32, device="cuda")
    y = torch.empty((s.M, s.H), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r), dtype=torch.uint8,
                     device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        ml.mlora_moe_route(d.logits, None, s.top_k, s.scoring, topk_ids=ids, topk_w=w, stream=stream)
        ml.mlora_moe_forward(d.x, d.w13, d.w2, d.A13, d.B13, d.A2, d.B2, d.idx, ids, w, s.scaling, y=y,
                             workspace=ws, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        ml.mlora_moe_route(d.logits, None, s.top_k, s.scoring, topk_ids=ids, topk_w=w, stream=stream)
        ml.mlora_moe_forward(d.x, d.w13, d.w2, d.A13, d.B13, d.A2, d.B2, d.idx, ids, w, s.scaling, y=y,
                             workspace=ws, stream=stream)
    for seed in (5, 6):
        new = wl.make(wl.spec("tiny", M=48, seed=seed), with_weights=False)
        d.logits.copy_(new.logits)
        d.x.copy_(new.x)
        d.idx.copy_(new.token_lora_idx)
        g.replay()
        torch.cuda.synchronize()
        y_graph = y.clone()
        ids_e, w_e = ml.mlora_moe_route(d.logits, None, s.top_k, s.scoring)
        y_eager = ml.mlora_moe_forward(d.x, d.w13, d.w2, d.A13, d.B13, d.A2, d.B2, d.idx, ids_e, w_e, s.scaling)
        torch.cuda.synchronize()
        assert torch.equal(y_graph, y_eager)
        inp.logits, inp.x, inp.token_lora_idx = new.logits, new.x, new.token_lora_idx
        ids_ref, w_ref = gu.oracle_route(inp)
        gu.check_y(y_graph, gu.oracle_forward(inp, ids_ref, w_ref), f"graph replay seed {seed}")


def _graph_step(d: gu.DeviceInputs, ids, w, y, ws, stream):
    s = d.spec
    lora = s.has_lora
    ml.mlora_moe_route(d.logits, d.bias, s.top_k, s.scoring, s.renormalize, s.n_shared, s.routed_scaling_factor,
                       topk_ids=ids, topk_w=w, stream=stream)
    ml.mlora_moe_forward(d.x, d.w13, d.w2, d.A13 if lora else None, d.B13 if lora else None,
                         d.A2 if lora else None, d.B2 if lora else None, d.idx if lora else None, ids, w,
                         s.scaling, s.n_shared, s.out_scale, y=y, workspace=ws, stream=stream)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "shared", "stress"])
def test_benchmark_launch_configuration(name):
    """The step as the benchmark times it: route + forward captured in a CUDA
    graph on a side stream, replayed after an L2 flush, plain and with the
    stage events recorded inside the graph.  Both replays equal an eager call
    bit for bit; the output matches the oracle on sampled tokens."""
    s = wl.spec(name)
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    L, r = (s.L, s.r) if s.has_lora else (0, 0)
    ids = torch.empty((s.M, s.K_total), dtype=torch.int32, device="cuda")
    w = torch.empty((s.M, s.K_total), dtype=torch.float32, device="cuda")
    y = torch.empty((s.M, s.H), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, L, r), dtype=torch.uint8,
                     device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        _graph_step(d, ids, w, y, ws, stream)
    stream.synchronize()
    y_eager = y.clone()
    graphs = []
    events = [torch.cuda.Event(enable_timing=True) for _ in range(ml.STAGE_EVENTS)]
    for e in events:  # torch creates the CUDA event on first record
        e.record(stream)
    for instrumented in (False, True):
        g = torch.cuda.CUDAGraph()
        if instrumented:
            ml.mlora_set_stage_events(events)
        try:
            with torch.cuda.graph(g, stream=stream):
                _graph_step(d, ids, w, y, ws, stream)
        finally:
            ml.mlora_set_stage_events(None)
        graphs.append(g)
    for g in graphs:
        for _ in range(2):
            y.zero_()
            flush.fill_(1)
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(y, y_eager)
            assert ml.mlora_moe_read_status(ws) == 0
    rows = None if s.M <= 128 else np.linspace(0, s.M - 1, 24).round().astype(np.int64)
    ids_ref, w_ref = gu.oracle_route(inp)
    y_ref = gu.oracle_forward(inp, ids_ref, w_ref, rows=rows)
    yg = y if rows is None else y[torch.as_tensor(rows, device="cuda")]
    gu.check_y(yg, y_ref, f"{name} graph replay")


def _random_specs(n: int, seed: int = 2024):
    """Seeded random small layers: shapes (multiples of 8), expert counts,
    top-k, shared slots, both scorings, renormalisation, ranks 8..64,
    adapter counts and modes."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.integers(1, 40))
        n_shared = int(rng.integers(0, 3)) if E > 1 else 0
        top_k = int(rng.integers(1, min(E, 8) + 1))
        scoring = int(rng.integers(0, 2))
        lora = bool(rng.random() < 0.75)
        over = dict(
            M=int(rng.integers(1, 300)),
            H=8 * int(rng.integers(1, 48)),
            I=8 * int(rng.integers(1, 48)),
            E=E, top_k=top_k, n_shared=n_shared,
            routed_scaling_factor=float(rng.choice([1.0, 2.5])) if n_shared else 1.0,
            scoring=scoring, renormalize=int(rng.integers(0, 2)),
            L=int(rng.integers(1, 12)) if lora else 0,
            r=8 * int(rng.integers(1, 9)) if lora else 0,
            lora_mode=str(rng.choice(["uniform", "zipf", "all_none"])) if lora else "none",
            seed=500 + i,
        )
        out.append(over)
    return out


@pytest.mark.parametrize("over", _random_specs(24), ids=lambda o: f"M{o['M']}H{o['H']}I{o['I']}E{o['E']}k{o['top_k']}")
def test_random_small_layers(over):
    """Random small configurations against the oracle (every output)."""
    _layer(wl.spec("tiny", **over), label=str(over))


def _hot_expert_ids(M, E, k, n_hot, seed):
    """Hand-made routing in which expert 0 gets exactly n_hot slots and the
    others share the rest evenly (fewer than n_hot each), with distinct
    experts within every row; positive weights that sum to 1 per row."""
    ids = np.empty((M, k), np.int32)
    for t in range(M):
        if t < n_hot:
            ids[t, 0] = 0
            ids[t, 1:] = 1 + (t * (k - 1) + np.arange(k - 1)) % (E - 1)
        else:
            ids[t] = 1 + (t * k + np.arange(k)) % (E - 1)
    assert all(len(set(r)) == k for r in ids.tolist())
    counts = np.bincount(ids.ravel(), minlength=E)
    assert counts[0] == n_hot and counts[1:].max() < n_hot
    w = np.random.default_rng(seed).uniform(0.1, 1.0, (M, k)).astype(np.float32)
    return ids, (w / w.sum(1, keepdims=True)).astype(np.float32)


@pytest.mark.parametrize("M,E,n_hot", [(40, 4, 32), (40, 4, 33), (1024, 128, 32), (1024, 128, 33)])
def test_ring_geometry_boundary(M, E, n_hot):
    """The experts kernel shrinks its A stages when no expert has more than
    32 slots; the busiest expert at exactly 32 and at 33 slots, with a
    one-CTA align (80 slots) and a cluster align (2048 slots)."""
    s = wl.spec("tiny", M=M, H=64, I=72, E=E, top_k=2, L=3, r=16, seed=120 + n_hot)
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    ids, w = _hot_expert_ids(M, E, 2, n_hot, seed=7)
    ws = torch.empty(ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r), dtype=torch.uint8,
                     device="cuda")
    y = gu.gpu_forward(d, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), workspace=ws)
    assert ml.mlora_moe_read_status(ws) == 0
    gu.check_y(y, gu.oracle_forward(inp, ids, w), f"busiest expert {n_hot} slots")


def test_poisoned_workspace_never_leaks():
    """Every forward writes whatever it reads: with the workspace filled
    with NaN bytes before each of eight calls, every output matches the
    oracle.  A block whose rows another CTA consumes (the act rows of the
    down projection, the LoRA tiles of the expands) is published only once
    all four epilogue warps wrote their rows, whichever warp runs ahead."""
    M, E, k = 1024, 128, 2
    s = wl.spec("tiny", M=M, H=64, I=136, E=E, top_k=k, L=3, r=16, seed=131)
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    ids_h, w_h = _hot_expert_ids(M, E, k, 32, seed=1)
    ids, w = torch.from_numpy(ids_h).cuda(), torch.from_numpy(w_h).cuda()
    y_ref = gu.oracle_forward(inp, ids_h, w_h)
    ws = torch.empty(ml.mlora_moe_workspace_size(M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r), dtype=torch.uint8,
                     device="cuda")
    for call in range(8):
        ws.fill_(0xFF)
        y = gu.gpu_forward(d, ids, w, workspace=ws)
        torch.cuda.synchronize()
        assert ml.mlora_moe_read_status(ws) == 0, call
        gu.check_y(y, y_ref, f"poisoned workspace, call {call}")


def test_graph_replay_switches_tile_geometry():
    """One captured forward, replayed on routings that move the kernel
    between its tile widths (wide/narrow, chosen from the padded block
    count) and ring geometries (chosen from the busiest expert), all decided
    on the device at each replay; every replay equals an eager call and the
    oracle."""
    M, E, k = 1024, 128, 2
    s = wl.spec("tiny", M=M, H=64, I=136, E=E, top_k=k, L=3, r=16, seed=131)
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)

    def spread_over(n_e):
        ids = ((np.arange(M)[:, None] * k + np.arange(k)[None, :]) % n_e).astype(np.int32)
        return ids, np.full((M, k), 1.0 / k, np.float32)

    routings = {
        "wide, 4 KiB A stages": _hot_expert_ids(M, E, k, 32, seed=1),   # 128 blocks x 2 slabs, max 32 slots
        "wide, 16 KiB A stages": _hot_expert_ids(M, E, k, 33, seed=2),  # max 33 slots
        "narrow, 16 KiB A stages": spread_over(40),                     # 40 blocks, ~52 slots each
        "narrow, 4 KiB A stages": spread_over(64),                      # 64 blocks, 32 slots each
    }
    ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
    w = torch.empty((M, k), dtype=torch.float32, device="cuda")
    y = torch.empty((M, s.H), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(ml.mlora_moe_workspace_size(M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r), dtype=torch.uint8,
                     device="cuda")
    first_ids, first_w = routings["wide, 4 KiB A stages"]
    ids.copy_(torch.from_numpy(first_ids))
    w.copy_(torch.from_numpy(first_w))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        ml.mlora_moe_forward(d.x, d.w13, d.w2, d.A13, d.B13, d.A2, d.B2, d.idx, ids, w, s.scaling, y=y,
                             workspace=ws, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        ml.mlora_moe_forward(d.x, d.w13, d.w2, d.A13, d.B13, d.A2, d.B2, d.idx, ids, w, s.scaling, y=y,
                             workspace=ws, stream=stream)
    for label, (ids_h, w_h) in routings.items():
        ids.copy_(torch.from_numpy(ids_h))
        w.copy_(torch.from_numpy(w_h))
        g.replay()
        torch.cuda.synchronize()
        assert ml.mlora_moe_read_status(ws) == 0, label
        y_graph = y.clone()
        y_eager = ml.mlora_moe_forward(d.x, d.w13, d.w2, d.A13, d.B13, d.A2, d.B2, d.idx, ids, w, s.scaling)
        torch.cuda.synchronize()
        assert torch.equal(y_graph, y_eager), label
        gu.check_y(y_graph, gu.oracle_forward(inp, ids_h, w_h), label)


def test_concurrent_forwards_on_two_streams():
    """Two layers launched on two streams without synchronisation: their
    persistent experts grids compete for the SMs, so each may start with only
    part of its CTAs resident.  Every tile, a CTA's first included, is
    claimed by a running CTA, so both finish with a clean status and the
    same bytes as one at a time."""
    specs = [wl.spec("decode", M=24, seed=140), wl.spec("decode", M=40, seed=141)]
    layers = []
    for s in specs:
        inp = wl.make(s, device="cuda")
        d = gu.DeviceInputs(inp)
        ids, w = gu.gpu_route(d)
        ws = torch.empty(ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r),
                         dtype=torch.uint8, device="cuda")
        y_ref = gu.gpu_forward(d, ids, w, workspace=ws)
        layers.append((d, ids, w, ws, y_ref))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(4):
        outs = []
        for (d, ids, w, ws, _), st in zip(layers, streams):
            s = d.spec
            y = torch.empty((s.M, s.H), dtype=torch.bfloat16, device="cuda")
            with torch.cuda.stream(st):
                ml.mlora_moe_forward(d.x, d.w13, d.w2, d.A13, d.B13, d.A2, d.B2, d.idx, ids, w, s.scaling, y=y,
                                     workspace=ws, stream=st)
            outs.append(y)
        torch.cuda.synchronize()
        for (d, ids, w, ws, y_ref), y in zip(layers, outs):
            assert ml.mlora_moe_read_status(ws) == 0
            assert torch.equal(y, y_ref)


def test_largest_batch():
    """A prefill-shaped layer with 65536 tokens (262144 routed slots, 32 768
    per CTA of the align cluster, ~2100 blocks): routing and the sorted,
    padded permutation bit-exact against the oracle over the whole batch,
    the layer output on sampled tokens."""
    s = wl.spec("prefill", M=65536)
    inp = wl.make(s, device="cuda")
    d = gu.DeviceInputs(inp)
    ids, w = gu.gpu_route(d)
    ids_ref, w_ref = gu.oracle_route(inp)
    gu.check_route(ids, w, ids_ref, w_ref)
    s_ref, e_ref, n_ref = oracle.moe_align(ids_ref, s.E_tot, 128)
    srt, eid, npad = ml.mlora_moe_align(ids, s.E_tot, 128)
    torch.cuda.synchronize()
    assert int(npad.item()) == n_ref
    assert np.array_equal(srt.cpu().numpy(), s_ref)
    assert np.array_equal(eid.cpu().numpy(), e_ref)
    ws = torch.empty(ml.mlora_moe_workspace_size(s.M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r), dtype=torch.uint8,
                     device="cuda")
    y = gu.gpu_forward(d, ids, w, workspace=ws)
    torch.cuda.synchronize()
    assert ml.mlora_moe_read_status(ws) == 0
    rows = gu.sample_rows(s.M, 12, seed=9, must=(0, s.M - 1))
    gu.check_y(y[torch.as_tensor(rows, device="cuda")], gu.oracle_forward(inp, ids_ref, w_ref, rows=rows),
               "65536 tokens")


def _random_wide_specs(n: int, seed: int = 77):
    """Seeded random layers over wider shapes than the small ones above: H and
    I up to 4096 (slabs of every tile width, ragged last slabs), up to 128
    experts, batches from one token to 600, with and without adapters."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.integers(1, 129))
        n_shared = int(rng.integers(0, 2)) if E > 1 else 0
        top_k = int(rng.integers(1, min(E, 8) + 1))
        lora = bool(rng.random() < 0.7)
        out.append(dict(
            M=int(rng.choice([1, 2, 3, 5, 8, 13, 32, 64, 100, 257, 600])),
            H=8 * int(rng.integers(1, 513)), I=8 * int(rng.integers(1, 513)),
            E=E, top_k=top_k, n_shared=n_shared,
            routed_scaling_factor=float(rng.choice([1.0, 2.5])) if n_shared else 1.0,
            scoring=int(rng.integers(0, 2)), renormalize=int(rng.integers(0, 2)),
            L=int(rng.integers(1, 20)) if lora else 0, r=8 * int(rng.integers(1, 9)) if lora else 0,
            lora_mode=str(rng.choice(["uniform", "zipf", "all_none"])) if lora else "none",
            seed=9000 + i,
        ))
    return out


@pytest.mark.parametrize("over", _random_wide_specs(40),
                         ids=lambda o: f"M{o['M']}H{o['H']}I{o['I']}E{o['E']}k{o['top_k']}L{o['L']}")
def test_random_wide_layers(over):
    """Random wider layers against the oracle on sampled tokens (the first,
    the last and six more)."""
    s = wl.spec("tiny", **over)
    rows = gu.sample_rows(s.M, 6, seed=over["seed"], must=(0, s.M - 1))
    _layer(s, rows=rows, label=str(over))


@pytest.mark.parametrize("name,M", [("decode", 4), ("decode", 64), ("stress", 96), ("shared", 32)])
def test_tile_configurations_change_no_bit(name, M):
    """The tuner's choices (tile width, shrink group size) never change an
    output bit: every forced configuration equals the library's own choice,
    which matches the oracle."""
    s = wl.spec(name, M=M)
    inp, d, ids, w, y, ids_ref, w_ref, _ = _layer(s)
    rp = (s.r + 15) // 16 * 16 if s.has_lora else 0
    groups = [g for g in (1, 2, 4) if g * rp <= 256] if s.has_lora else [0]
    try:
        for wc in range(3):
            for g in groups:
                ml.mlora_set_tile_config(wc, g)
                yf = gu.gpu_forward(d, ids, w)
                torch.cuda.synchronize()
                assert torch.equal(yf, y), (wc, g)
    finally:
        ml.mlora_set_tile_config(-1, 0)
