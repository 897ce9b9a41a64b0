"""Guard bands around the caller's output buffers: every path and expert format
writes exactly its [T][H] output rows (and the routing outputs exactly their
[T][K] / [T] / [T][E] entries), nothing before or after them.

Each output is a view into a larger buffer whose leading and trailing rows hold
a sentinel bit pattern; after the call the sentinels must be intact and the
output itself finite. Every compute call goes through the C ABI.
"""
import numpy as np
import pytest
import torch

import quantized_moe_expert_gb300 as ds4
import synth
from gpu_util import to_dev, x_to_dev

pytestmark = pytest.mark.gpu

GUARD = 4                 # rows before and after each output
SENTINEL = 0x7FA5A5A5     # a NaN payload no kernel writes


def guarded(rows, cols, dtype):
    full = torch.empty((rows + 2 * GUARD, cols), dtype=torch.int32, device="cuda")
    full.fill_(SENTINEL)
    view = full[GUARD:GUARD + rows]
    return full, view.view(dtype) if dtype != torch.int32 else view


def intact(full, rows):
    f = full.cpu().numpy()
    return (f[:GUARD] == SENTINEL).all() and (f[GUARD + rows:] == SENTINEL).all()


LAYERS = {
    "q2": ({}, 0),
    "mx4": ({"routed_format": "mx4"}, ds4.FLAG_MXFP4),
    "vq12": ({"routed_format": "vq", "vq_bits": 12}, ds4.FLAG_VQ12),
}


@pytest.fixture(scope="module", params=sorted(LAYERS))
def layer(request):
    kw, flags = LAYERS[request.param]
    wl = synth.WORKLOADS["tiny"]
    lay = synth.make_layer(wl.shape, wl.layer_seeds[0], **kw)
    moe = ds4.MoELayer(wl.shape, to_dev(lay), max_tokens=80, flags=flags)
    yield wl.shape, moe
    moe.close()


@pytest.mark.parametrize("path", [ds4.PATH_AUTO, ds4.PATH_DECODE, ds4.PATH_BATCH, ds4.PATH_PREFILL])
@pytest.mark.parametrize("T", [1, 5, 9, 64, 80])
def test_forward_writes_only_its_rows(layer, path, T):
    shape, moe = layer
    if path == ds4.PATH_BATCH and T > ds4.BATCH_MAX_T:
        pytest.skip("above the batch path's token limit")
    x = synth.normal_bf16(T * shape.hidden, 7000 + T, synth.S_X).reshape(T, shape.hidden)
    full, y = guarded(T, shape.hidden, torch.float32)
    ds4.ds4moe_forward_path(moe.handle, x_to_dev(x), T, path, y)
    torch.cuda.synchronize()
    assert intact(full, T)
    assert torch.isfinite(y).all()
    assert moe.status() == 0


@pytest.mark.parametrize("T", [1, 8, 80])
def test_routing_outputs_write_only_their_entries(layer, T):
    shape, moe = layer
    K, E = shape.top_k, shape.n_experts
    x = synth.normal_bf16(T * shape.hidden, 7100 + T, synth.S_X).reshape(T, shape.hidden)
    fi, idx = guarded(T, K, torch.int32)
    fw, w = guarded(T, K, torch.float32)
    fg, gap = guarded(T, 1, torch.float32)
    fs, sel = guarded(T, E, torch.float32)
    ds4.ds4moe_route_detail(moe.handle, x_to_dev(x), T, idx, w, gap.view(T), sel)
    torch.cuda.synchronize()
    assert intact(fi, T) and intact(fw, T) and intact(fg, T) and intact(fs, T)
    assert ((idx >= 0) & (idx < E)).all() and torch.isfinite(w).all()
    assert moe.status() == 0
