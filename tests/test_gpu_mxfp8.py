"""The MXFP8 expert path on the GPU against the fp64 oracle.

The weight quantizer is byte-exact (codes and scales) against the oracle's
MXFP8 conversion; the packed scales are unpacked by the layout include/mlora.h
documents.  The layer (x and the SwiGLU output quantized on the device,
adapters in bf16) matches the oracle's MXFP8 layer within the layer
tolerance on every output of the decode, shared-expert and adapter-stress
workloads, on sampled rows of prefill, and on ragged and edge shapes; a
replayed CUDA graph equals an eager call bit for bit, and a batch whose
tokens use no adapter equals the adapter-free layer bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
import moe_layer_lora_gb300 as ml
from moe_layer_lora_gb300 import workloads as wl
import gpu_util as gu

pytestmark = pytest.mark.gpu


def unpack_scales(packed, E, H, I, which):
    """Natural [rows, K/32] scales from the packed layout of include/mlora.h;
    also returns the mask of packed bytes no weight row maps to."""
    nslab = math.ceil(I / 96) if which == 0 else math.ceil(H / 192)
    nchunk = math.ceil(H / 128) if which == 0 else math.ceil(I / 128)
    rows, K = (2 * I, H) if which == 0 else (H, I)
    P = packed.reshape(E, nslab, nchunk, 2, 512)
    out = np.zeros((E, rows, K // 32), np.uint8)
    used = np.zeros(P.shape, bool)
    for cb in range(nslab):
        for t in range(192):
            if which == 0:
                j = cb * 96 + (t if t < 96 else t - 96)
                if j >= I:
                    continue
                row = j if t < 96 else I + j
            else:
                row = cb * 192 + t
                if row >= H:
                    continue
            atom, r = t // 128, t % 128
            for kc in range(nchunk):
                for kb in range(4):
                    blk = kc * 4 + kb
                    if blk >= K // 32:
                        continue
                    byte = (r % 32) * 16 + (r // 32) * 4 + kb
                    out[:, row, blk] = P[:, cb, kc, atom, byte]
                    used[:, cb, kc, atom, byte] = True
    return out, ~used, P


@pytest.mark.parametrize("E,H,I", [(3, 64, 96), (2, 160, 224), (4, 2880, 2880)])
def test_quantize_weights_byte_exact(E, H, I):
    s = wl.spec("tiny", E=E, H=H, I=I, L=0, r=0, lora_mode="none", seed=300 + H)
    inp = wl.make(s, device="cuda")
    w13, w2 = inp.w13.cuda(), inp.w2.cuda()
    w13_q, w13_s, w2_q, w2_s = ml.mlora_mxfp8_quantize_weights(w13, w2)
    torch.cuda.synchronize()
    for w, q, sc, which in ((w13, w13_q, w13_s, 0), (w2, w2_q, w2_s, 1)):
        codes_ref, scales_ref = oracle.mx_quantize(wl.bits(w))
        assert np.array_equal(q.cpu().numpy(), codes_ref)
        nat, unused, P = unpack_scales(sc.cpu().numpy(), E, H, I, which)
        assert np.array_equal(nat, scales_ref)
        assert (P[unused] == 0).all()


class MxLayer:
    def __init__(self, spec):
        self.spec = spec
        self.inp = wl.make(spec, device="cuda")
        gu.assert_unambiguous(self.inp)
        self.d = gu.DeviceInputs(self.inp)
        self.q = ml.mlora_mxfp8_quantize_weights(self.d.w13, self.d.w2)
        # the oracle's MXFP8 weights, from the oracle's own quantizer (the
        # byte-exact test above ties the two)
        self.q_ref = oracle.mx_quantize(wl.bits(self.inp.w13)) + oracle.mx_quantize(wl.bits(self.inp.w2))

    def forward(self, ids, w, lora=True, idx="default", workspace=None, y=None, stream=None):
        s, d = self.spec, self.d
        use = lora and s.has_lora
        tli = d.idx if idx == "default" else idx
        return ml.mlora_moe_forward_mxfp8(d.x, *self.q, d.A13 if use else None, d.B13 if use else None,
                                          d.A2 if use else None, d.B2 if use else None, tli if use else None,
                                          ids, w, s.scaling, s.n_shared, s.out_scale, y=y, workspace=workspace,
                                          stream=stream)

    def oracle(self, ids, w, rows=None, lora=True, idx=None):
        s, inp = self.spec, self.inp
        use = lora and s.has_lora
        sel = slice(None) if rows is None else np.asarray(rows)
        b = gu._hbits
        tli = None
        if use:
            tli = (inp.token_lora_idx.numpy() if idx is None else np.asarray(idx, np.int32))[sel]
        return oracle.moe_forward_mx(wl.bits(inp.x)[sel], *self.q_ref, b(inp.A13) if use else None,
                                     b(inp.B13) if use else None, b(inp.A2) if use else None,
                                     b(inp.B2) if use else None, tli, ids[sel], w[sel].astype(np.float32),
                                     s.scaling, s.out_scale)


def _check_layer(spec, rows=None, label=""):
    L = MxLayer(spec)
    ids, w = gu.gpu_route(L.d)
    ws = torch.empty(ml.mlora_moe_workspace_size_mxfp8(spec.M, spec.H, spec.I, spec.E_tot, spec.K_total,
                                                       spec.L if spec.has_lora else 0,
                                                       spec.r if spec.has_lora else 0),
                     dtype=torch.uint8, device="cuda")
    y = L.forward(ids, w, workspace=ws)
    torch.cuda.synchronize()
    assert ml.mlora_moe_read_status(ws) == 0
    ids_ref, w_ref = gu.oracle_route(L.inp)
    gu.check_route(ids, w, ids_ref, w_ref)
    y_ref = L.oracle(ids_ref, w_ref, rows=rows)
    yg = y if rows is None else y[torch.as_tensor(rows, device="cuda")]
    gu.check_y(yg, y_ref, label or f"mxfp8 {spec.name}")
    return L, ids, w, y, ids_ref, w_ref


@pytest.mark.parametrize("over", [
    dict(),                                                                   # tiny, adapters rank 8
    dict(M=37, H=160, I=224, E=5, top_k=3, L=3, r=24, seed=401),             # ragged slabs and K-chunks
    dict(M=9, H=32, I=32, E=4, top_k=4, L=5, r=64, seed=402),                # one K-block, rank 64
    dict(M=300, H=256, I=96, E=16, top_k=2, L=70, r=8, seed=403),            # many adapters
    dict(M=16, H=256, I=128, E=8, top_k=2, L=0, r=0, lora_mode="none", seed=404),  # no adapters
    dict(M=64, H=512, I=256, E=8, top_k=2, n_shared=2, routed_scaling_factor=2.0,
         scoring=wl.SCORE_SIGMOID_BIAS, L=4, r=16, seed=405),               # shared slots with adapters
    dict(M=130, H=128, I=128, E=3, top_k=1, L=1, r=16, seed=406),           # full blocks
    dict(M=1100, H=96, I=64, E=6, top_k=4, L=9, r=8, seed=407),             # > 4096 slots
])
def test_mxfp8_small_layers(over):
    _check_layer(wl.spec("tiny", **over), label=f"mxfp8 {over}")


def test_mxfp8_decode_full():
    _check_layer(wl.spec("decode"))


def test_mxfp8_poisoned_workspace_never_leaks():
    """The MXFP8 layer on a workspace filled with NaN bytes before each of
    eight calls (128 experts, the busiest with 32 slots): every output
    matches the oracle, so no call reads a row before it is published."""
    M, E, k = 1024, 128, 2
    L = MxLayer(wl.spec("tiny", M=M, H=128, I=160, E=E, top_k=k, L=3, r=16, seed=132))
    ids_h = ((np.arange(M)[:, None] * k + np.arange(k)[None, :]) % 64).astype(np.int32)
    w_h = np.full((M, k), 1.0 / k, np.float32)
    ids, w = torch.from_numpy(ids_h).cuda(), torch.from_numpy(w_h).cuda()
    y_ref = L.oracle(ids_h, w_h)
    s = L.spec
    ws = torch.empty(ml.mlora_moe_workspace_size_mxfp8(M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r),
                     dtype=torch.uint8, device="cuda")
    for call in range(8):
        ws.fill_(0xFF)
        y = L.forward(ids, w, workspace=ws)
        torch.cuda.synchronize()
        assert ml.mlora_moe_read_status(ws) == 0, call
        gu.check_y(y, y_ref, f"mxfp8 poisoned workspace, call {call}")


@pytest.mark.parametrize("M", [2, 7])
def test_mxfp8_decode_few_tokens(M):
    """A handful of tokens on the decode layer: blocks of one or two rows,
    a 192-row tile per slab, adapters on most slots."""
    _check_layer(wl.spec("decode", M=M), label=f"mxfp8 decode M={M}")


@pytest.mark.parametrize("M", [1, 32, 128])
def test_mxfp8_shared_full(M):
    _check_layer(wl.spec("shared", M=M))


def test_mxfp8_stress_full_and_early_exit():
    L, ids, w, y, ids_ref, w_ref = _check_layer(wl.spec("stress"))
    s = L.spec
    none = torch.full((s.M,), -1, dtype=torch.int32, device="cuda")
    y_none = L.forward(ids, w, idx=none)
    y_base = L.forward(ids, w, lora=False)
    torch.cuda.synchronize()
    assert torch.equal(y_none, y_base)
    gu.check_y(y_base, L.oracle(ids_ref, w_ref, lora=False), "mxfp8 stress all -1")


def test_mxfp8_prefill_sampled():
    s = wl.spec("prefill")
    rows = gu.sample_rows(s.M, 48, seed=17, must=(0, s.M - 1))
    _check_layer(s, rows=rows)


def test_mxfp8_graph_replay_equals_eager():
    s = wl.spec("decode", M=24, seed=410)
    L = MxLayer(s)
    ids = torch.empty((s.M, s.K_total), dtype=torch.int32, device="cuda")
    w = torch.empty((s.M, s.K_total), dtype=torch.float32, device="cuda")
    y = torch.empty((s.M, s.H), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(ml.mlora_moe_workspace_size_mxfp8(s.M, s.H, s.I, s.E_tot, s.K_total, s.L, s.r),
                     dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def step():
        ml.mlora_moe_route(L.d.logits, None, s.top_k, s.scoring, topk_ids=ids, topk_w=w, stream=stream)
        L.forward(ids, w, y=y, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    for seed in (411, 412):
        new = wl.make(wl.spec("decode", M=24, seed=seed), with_weights=False)
        L.d.logits.copy_(new.logits)
        L.d.x.copy_(new.x)
        L.d.idx.copy_(new.token_lora_idx)
        g.replay()
        torch.cuda.synchronize()
        y_graph = y.clone()
        ids_e, w_e = ml.mlora_moe_route(L.d.logits, None, s.top_k, s.scoring)
        y_eager = L.forward(ids_e, w_e)
        torch.cuda.synchronize()
        assert torch.equal(y_graph, y_eager)
        L.inp.logits, L.inp.x, L.inp.token_lora_idx = new.logits, new.x, new.token_lora_idx
        ids_ref, w_ref = gu.oracle_route(L.inp)
        gu.check_y(y_graph, L.oracle(ids_ref, w_ref), f"mxfp8 graph replay seed {seed}")
