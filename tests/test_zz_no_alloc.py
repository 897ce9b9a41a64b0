"""ds4moe_route_noalloc: routing that allocates no device memory.

Some callers cannot allocate at call time: an engine that has reserved all of
HBM for its own pools at start-up, or a latency-critical path that must not
pay for cudaMalloc's device-wide synchronisation. For them the library routes
from the caller's router weights using a fixed, statically allocated scratch
array instead of a handle's scratch. This test calls it through the C ABI and
checks it against the handle-based ds4moe_route on two calls in a row.
"""
import numpy as np
import pytest
import torch

import quantized_moe_expert_gb300 as ds4
import synth
from gpu_util import TOL_WEIGHTS, to_dev, x_to_dev

pytestmark = pytest.mark.gpu


def test_route_noalloc_matches_route_on_two_calls():
    wl = synth.WORKLOADS["tiny"]
    shape = wl.shape
    layer = synth.make_layer(shape, wl.layer_seeds[0])
    layer["router_bias"] = (0.3 * synth.zipf_profile(shape.n_experts, wl.layer_seeds[0])).astype(np.float32)
    dev = to_dev(layer)
    moe = ds4.MoELayer(shape, dev, max_tokens=64)
    H, E, K = shape.hidden, shape.n_experts, shape.top_k
    for call, T in enumerate((37, 5)):  # two calls in a row; the second reuses the scratch
        x = x_to_dev(synth.normal_bf16(T * H, 4242 + call, synth.S_X).reshape(T, H))
        idx_ref, w_ref, _, _ = moe.route(x)
        idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
        w = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
        ds4.ds4moe_route_noalloc(dev["router_w"], dev["router_bias"], x, T, H, E, K, idx, w)
        torch.cuda.synchronize()
        assert (idx.cpu().numpy() == idx_ref.cpu().numpy()).all()
        assert np.abs(w.cpu().numpy() - w_ref.cpu().numpy()).max() <= TOL_WEIGHTS
    assert moe.status() == 0
    moe.close()


def test_route_noalloc_rejects_requests_beyond_its_scratch():
    H, E, K = 4096, 384, 6
    T = ds4.DS4MOE_NOALLOC_SCRATCH // (4 * (H + H // 16 + E)) + 1
    router = torch.zeros((E, H), dtype=torch.float32, device="cuda")
    x = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    idx = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, K), dtype=torch.float32, device="cuda")
    with pytest.raises(ds4.DS4MoEError) as e:
        ds4.ds4moe_route_noalloc(router, None, x, T, H, E, K, idx, w)
    assert e.value.code == ds4.DS4MOE_ESCRATCH
    assert (idx == 0).all().item()  # nothing was launched
