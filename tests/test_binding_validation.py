"""The Python binding refuses tensors whose shape, dtype or placement does
not match the layer before any device work: the library builds its tensor
maps from the sizes it is given, not from the allocations, so a mismatch
would otherwise read past a buffer.  CPU only (the checks run before any
CUDA call; a tensor that passes every shape check is then refused for not
being on a CUDA device)."""
import pytest
import torch

import moe_layer_lora_gb300 as ml

M, H, I, E, K, L, R = 4, 64, 48, 3, 2, 2, 8


def _layer(**bad):
    t = dict(
        x=torch.zeros(M, H, dtype=torch.bfloat16),
        w13=torch.zeros(E, 2 * I, H, dtype=torch.bfloat16),
        w2=torch.zeros(E, H, I, dtype=torch.bfloat16),
        A13=torch.zeros(L, E, R, H, dtype=torch.bfloat16),
        B13=torch.zeros(L, E, 2 * I, R, dtype=torch.bfloat16),
        A2=torch.zeros(L, E, R, I, dtype=torch.bfloat16),
        B2=torch.zeros(L, E, H, R, dtype=torch.bfloat16),
        token_lora_idx=torch.zeros(M, dtype=torch.int32),
        topk_ids=torch.zeros(M, K, dtype=torch.int32),
        topk_w=torch.zeros(M, K, dtype=torch.float32),
    )
    t.update(bad)
    return t


def _forward(t, **kw):
    return ml.mlora_moe_forward(t["x"], t["w13"], t["w2"], t["A13"], t["B13"], t["A2"], t["B2"],
                                t["token_lora_idx"], t["topk_ids"], t["topk_w"], 2.0, **kw)


@pytest.mark.parametrize("name,bad", [
    ("w2", torch.zeros(E, H, I // 2, dtype=torch.bfloat16)),          # I read from w13 disagrees
    ("w2", torch.zeros(E + 1, H, I, dtype=torch.bfloat16)),           # expert count
    ("w13", torch.zeros(E, 2 * I, H, dtype=torch.float32)),           # dtype
    ("B13", torch.zeros(L, E, I, R, dtype=torch.bfloat16)),           # gate+up rows
    ("A2", torch.zeros(L, E, R, H, dtype=torch.bfloat16)),            # K of the down shrink
    ("B2", torch.zeros(L - 1, E, H, R, dtype=torch.bfloat16)),        # adapter count
    ("token_lora_idx", torch.zeros(M + 1, dtype=torch.int32)),        # one id per token
    ("token_lora_idx", torch.zeros(M, dtype=torch.int64)),            # int32 ids
    ("topk_w", torch.zeros(M, K + 1, dtype=torch.float32)),           # one weight per slot
    ("topk_w", torch.zeros(M, K, dtype=torch.float64)),
])
def test_forward_refuses_mismatched_tensor(name, bad):
    with pytest.raises(ValueError, match=name):
        _forward(_layer(**{name: bad}))


def test_forward_refuses_wrong_output():
    with pytest.raises(ValueError, match="y"):
        _forward(_layer(), y=torch.zeros(M, H + 8, dtype=torch.bfloat16))


def test_forward_refuses_non_contiguous():
    x = torch.zeros(H, M, dtype=torch.bfloat16).t()  # [M, H] view, not row-major
    with pytest.raises(ValueError, match="contiguous CUDA"):
        _forward(_layer(x=x))


def test_forward_refuses_host_tensors():
    with pytest.raises(ValueError, match="CUDA"):
        _forward(_layer())


def test_route_refuses_mismatched_tensors():
    logits = torch.zeros(M, E, dtype=torch.float32)
    with pytest.raises(ValueError, match="bias"):
        ml.mlora_moe_route(logits, torch.zeros(E + 1, dtype=torch.float32), 2, ml.SCORE_SIGMOID_BIAS)
    with pytest.raises(ValueError, match="topk_ids"):
        ml.mlora_moe_route(logits, None, 2, ml.SCORE_SOFTMAX, topk_ids=torch.zeros(M, 3, dtype=torch.int32),
                           topk_w=torch.zeros(M, 2, dtype=torch.float32))
    with pytest.raises(ValueError, match="logits"):
        ml.mlora_moe_route(logits.double(), None, 2, ml.SCORE_SOFTMAX)


def test_align_refuses_wrong_ids():
    with pytest.raises(ValueError, match="topk_ids"):
        ml.mlora_moe_align(torch.zeros(M, K, dtype=torch.int64), E, 16)


@pytest.mark.parametrize("missing", ["A13", "B13", "A2", "B2", "token_lora_idx"])
def test_forward_refuses_a_partial_adapter_set(missing):
    """Four of the five adapter tensors would otherwise run the layer
    silently without adapters: all five or none."""
    with pytest.raises(ValueError, match="all None"):
        _forward(_layer(**{missing: None}))


def test_stream_of_another_device_is_refused():
    """The library launches on the current device, which the binding sets
    to the tensors' device; a stream of another device is refused."""
    from moe_layer_lora_gb300 import _lib

    class FakeStream:
        device = torch.device("cuda", 1)
        cuda_stream = 0

    with pytest.raises(ValueError, match="stream is on cuda:1"):
        _lib._stream(FakeStream(), torch.device("cuda", 0))
    assert _lib._stream(FakeStream(), torch.device("cuda", 1)).value is None
