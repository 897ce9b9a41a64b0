"""ds4moe_route_noalloc: routing that allocates no device memory.

Some callers cannot allocate at call time: an engine that has reserved all of
HBM for its own pools at start-up, or a latency-critical path that must not
pay for cudaMalloc's device-wide synchronisation. For them the library routes
from the caller's router weights using a fixed, statically allocated scratch
array instead of a handle's scratch. These tests call it through the C ABI
and check it against the oracle's routing (tokens whose K-th and (K+1)-th
scores are closer than the near-tie threshold may pick either expert) and
against the handle-based ds4moe_route, on two calls in a row, and at the
largest request its scratch holds for the H=4096, E=384 layer.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_gb300 as ds4
import synth
from gpu_util import TOL_WEIGHTS, check_routing, to_dev, x_to_dev

pytestmark = pytest.mark.gpu


def noalloc_route(router_w, router_bias, x, H, E, K):
    T = x.shape[0]
    idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
    ds4.ds4moe_route_noalloc(router_w, router_bias, x, T, H, E, K, idx, w)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def test_route_noalloc_matches_oracle_and_route_on_two_calls():
    wl = synth.WORKLOADS["tiny"]
    shape = wl.shape
    layer = synth.make_layer(shape, wl.layer_seeds[0])
    layer["router_bias"] = (0.3 * synth.zipf_profile(shape.n_experts, wl.layer_seeds[0])).astype(np.float32)
    dev = to_dev(layer)
    moe = ds4.MoELayer(shape, dev, max_tokens=64)
    H, E, K = shape.hidden, shape.n_experts, shape.top_k
    for call, T in enumerate((37, 5)):  # two calls in a row; the second reuses the scratch
        xh = synth.normal_bf16(T * H, 4242 + call, synth.S_X).reshape(T, H)
        x = x_to_dev(xh)
        idx, w = noalloc_route(dev["router_w"], dev["router_bias"], x, H, E, K)
        ref = oracle.route(shape, layer["router_w"], layer["router_bias"], xh)
        check_routing(idx, w, None, ref, K)
        # the same fp32 router arithmetic as the handle's path for T < 16
        if T < 16:
            idx_h, w_h, _, _ = moe.route(x)
            assert (idx == idx_h.cpu().numpy()).all()
            assert np.abs(w - w_h.cpu().numpy()).max() <= TOL_WEIGHTS
    assert moe.status() == 0
    moe.close()


def test_route_noalloc_at_its_largest_request():
    """H=4096, E=384, K=6: T=221 fits the scratch after its three 256-byte
    roundings and routes like the oracle; T=222 does not fit and is refused."""
    shape = synth.V4F_SHAPE
    H, E, K = shape.hidden, shape.n_experts, shape.top_k
    seed = synth.WORKLOADS["decode_t1"].layer_seeds[0]
    rw = synth.normal_f32(E * H, seed, synth.S_ROUTER, 0.02).reshape(E, H)
    rwd = torch.from_numpy(rw).cuda()
    T = 221
    assert 4 * T * (H + H // 16 + E) <= ds4.DS4MOE_NOALLOC_SCRATCH < 4 * (T + 1) * (H + H // 16 + E)
    xh = synth.normal_bf16(T * H, 4300, synth.S_X).reshape(T, H)
    idx, w = noalloc_route(rwd, None, x_to_dev(xh), H, E, K)
    ref = oracle.route(shape, rw, None, xh)
    check_routing(idx, w, None, ref, K)
    x2 = torch.zeros((T + 1, H), dtype=torch.int16, device="cuda")
    idx2 = torch.zeros((T + 1, K), dtype=torch.int32, device="cuda")
    w2 = torch.zeros((T + 1, K), dtype=torch.float32, device="cuda")
    with pytest.raises(ds4.DS4MoEError) as e:
        ds4.ds4moe_route_noalloc(rwd, None, x2, T + 1, H, E, K, idx2, w2)
    assert e.value.code == ds4.DS4MOE_ESCRATCH
    assert (idx2 == 0).all().item()  # nothing was launched


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


def test_route_noalloc_rejects_host_buffers():
    H, E, K, T = 512, 32, 6, 4
    router = torch.zeros((E, H), dtype=torch.float32, device="cuda")
    x = torch.zeros((T, H), dtype=torch.int16)  # host memory
    idx = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, K), dtype=torch.float32, device="cuda")
    with pytest.raises(ds4.DS4MoEError) as e:
        ds4.ds4moe_route_noalloc(router, None, x, T, H, E, K, idx, w)
    assert e.value.code == ds4.DS4MOE_EINVAL
