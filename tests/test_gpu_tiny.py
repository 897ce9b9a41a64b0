"""GPU parity on small layers the oracle finishes in seconds, with edge cases.

Every compute call goes through the C ABI; the oracle is the reference.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_gb300 as ds4
import synth
from gpu_util import assert_close, TOL_DECODE, TOL_PREFILL, check_routing, rel_l2, to_dev, x_to_dev

pytestmark = pytest.mark.gpu


def tokens(shape, T, seed):
    return synth.normal_bf16(T * shape.hidden, seed, synth.S_X).reshape(T, shape.hidden)


@pytest.fixture(scope="module")
def tiny():
    wl = synth.WORKLOADS["tiny"]
    layer = synth.make_layer(wl.shape, wl.layer_seeds[0])
    moe = ds4.MoELayer(wl.shape, to_dev(layer), max_tokens=80)
    yield wl.shape, layer, moe
    moe.close()


def test_route_matches_oracle(tiny):
    shape, layer, moe = tiny
    x = tokens(shape, 80, 101)
    idx, w, gap, sel = moe.route(x_to_dev(x), want_sel=True)
    ref = oracle.route(shape, layer["router_w"], None, x)
    check_routing(idx.cpu().numpy(), w.cpu().numpy(), gap.cpu().numpy(), ref, shape.top_k)
    assert np.allclose(sel.cpu().numpy(), ref["sel"], rtol=0, atol=2e-6)
    assert moe.status() == 0


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8, 12, 16])
def test_decode_path(tiny, T):
    shape, layer, moe = tiny
    x = tokens(shape, T, 200 + T)
    y = moe.forward(x_to_dev(x), path=ds4.PATH_DECODE).cpu().numpy()
    y_ref, _ = oracle.forward(shape, layer, x)
    assert_close(y, y_ref, TOL_DECODE)
    assert moe.status() == 0


@pytest.mark.parametrize("T", [9, 16, 37, 80])
def test_prefill_path(tiny, T):
    shape, layer, moe = tiny
    x = tokens(shape, T, 300 + T)
    y = moe.forward(x_to_dev(x), path=ds4.PATH_PREFILL).cpu().numpy()
    y_ref, r = oracle.forward(shape, layer, x)
    assert_close(y, y_ref, TOL_PREFILL)
    assert moe.status() == 0


def test_auto_path_and_stats(tiny):
    shape, layer, moe = tiny
    x = tokens(shape, ds4.AUTO_BATCH_MAX_T + 1, 401)
    moe.forward(x_to_dev(x[:4]))
    s = moe.stats()
    assert s.path == ds4.PATH_BATCH and s.tokens == 4 and s.kernel_count > 0
    r = oracle.route(shape, layer["router_w"], None, x[:4])
    assert s.n_unique == len(np.unique(r["idx"]))
    assert s.max_load == np.bincount(r["idx"].ravel()).max()
    moe.forward(x_to_dev(x[:ds4.AUTO_DECODE_MAX_T]))
    assert moe.stats().path == ds4.PATH_DECODE
    moe.forward(x_to_dev(x[:ds4.AUTO_DECODE_MAX_T + 1]))
    assert moe.stats().path == ds4.PATH_BATCH
    moe.forward(x_to_dev(x[:ds4.AUTO_BATCH_MAX_T]))
    assert moe.stats().path == ds4.PATH_BATCH
    moe.forward(x_to_dev(x[:ds4.AUTO_BATCH_MAX_T + 1]))
    assert moe.stats().path == ds4.PATH_PREFILL


def test_forward_routed_uses_given_routing(tiny):
    shape, layer, moe = tiny
    x = tokens(shape, 6, 501)
    rng = np.random.default_rng(5)
    idx = np.stack([rng.choice(shape.n_experts, shape.top_k, replace=False) for _ in range(6)]).astype(np.int32)
    w = rng.random((6, shape.top_k))
    w /= w.sum(axis=1, keepdims=True)
    for path, tol in ((ds4.PATH_DECODE, TOL_DECODE), (ds4.PATH_PREFILL, TOL_PREFILL)):
        y = moe.forward_routed(x_to_dev(x), torch.from_numpy(idx).cuda(),
                               torch.from_numpy(w.astype(np.float32)).cuda(), path=path).cpu().numpy()
        y_ref = oracle.forward_routed(shape, layer, x, idx, w.astype(np.float32).astype(np.float64))
        assert_close(y, y_ref, tol)
    assert moe.status() == 0


def test_token_independence_and_determinism(tiny):
    shape, layer, moe = tiny
    x = tokens(shape, 8, 601)
    xd = x_to_dev(x)
    y8 = moe.forward(xd, path=ds4.PATH_DECODE).cpu().numpy()
    y8b = moe.forward(xd, path=ds4.PATH_DECODE).cpu().numpy()
    assert (y8 == y8b).all()
    for t in range(8):
        # a token's output does not depend on the other tokens of the batch (up to
        # the summation order of the tensor-core packing, which depends on T)
        y1 = moe.forward(xd[t:t + 1].contiguous(), path=ds4.PATH_DECODE).cpu().numpy()
        assert rel_l2(y1[0], y8[t]) <= 1e-5


def test_forward_host_matches_device(tiny):
    shape, layer, moe = tiny
    x = tokens(shape, 5, 701)
    y_dev = moe.forward(x_to_dev(x)).cpu().numpy()
    x_host = torch.from_numpy(x.view(np.int16)).pin_memory()
    y_host = torch.empty((5, shape.hidden), dtype=torch.float32).pin_memory()
    ds4.ds4moe_forward_host(moe.handle, x_host.data_ptr(), 5, y_host.data_ptr())
    assert (y_host.numpy() == y_dev).all()


def test_zero_tokens_is_a_noop(tiny):
    shape, layer, moe = tiny
    y = torch.full((1, shape.hidden), 7.0, device="cuda")
    x = x_to_dev(tokens(shape, 1, 801))
    ds4.ds4moe_forward(moe.handle, x, 0, y)
    assert (y == 7.0).all().item()


def test_argument_errors(tiny):
    shape, layer, moe = tiny
    x = x_to_dev(tokens(shape, 4, 901))
    y = torch.empty((4, shape.hidden), device="cuda")
    with pytest.raises(ds4.DS4MoEError) as e:
        ds4.ds4moe_forward(moe.handle, x, moe.max_tokens + 1, y)
    assert e.value.code == ds4.DS4MOE_EINVAL
    with pytest.raises(ds4.DS4MoEError):
        ds4.ds4moe_forward(moe.handle, x, -1, y)
    host_y = torch.empty((4, shape.hidden))
    with pytest.raises(ds4.DS4MoEError):
        ds4.ds4moe_forward(moe.handle, x, 4, host_y)
    with pytest.raises(ds4.DS4MoEError):
        ds4.ds4moe_forward(moe.handle, x.cpu(), 4, y)
    with pytest.raises(ds4.DS4MoEError):
        ds4.ds4moe_forward_path(moe.handle, x, 4, 7, y)
    assert moe.status() == 0


def test_out_of_range_routed_index_is_reported(tiny):
    shape, layer, moe = tiny
    x = x_to_dev(tokens(shape, 1, 902))
    idx = torch.tensor([[0, 1, 2, 3, 4, shape.n_experts + 5]], dtype=torch.int32, device="cuda")
    w = torch.full((1, shape.top_k), 1.0 / shape.top_k, device="cuda")
    moe.forward_routed(x, idx, w)
    assert moe.status() == ds4.DS4MOE_EDEVICE
    assert moe.status() == 0  # the sticky error was cleared


def test_repeated_given_expert(tiny):
    """A token whose given experts repeat: the decode path replaces each repeat (in k
    order) by the smallest expert index the token's row does not hold and reports
    DS4MOE_EDEVICE; the prefill path applies the expert once per occurrence."""
    shape, layer, moe = tiny
    K = shape.top_k
    x = tokens(shape, 2, 777)
    idx = np.array([[3, 3, 9, 3, 12, 20], [1, 2, 4, 8, 16, 31]], dtype=np.int32)[:, :K]
    w = np.full((2, K), 1.0 / K, dtype=np.float32)
    replaced = idx.copy()
    for r in range(1, K):
        if replaced[0, r] in replaced[0, :r]:
            c = 0
            while c in replaced[0]:
                c += 1
            replaced[0, r] = c
    assert replaced[0].tolist() == [3, 0, 9, 1, 12, 20][:K]
    y = moe.forward_routed(x_to_dev(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                           path=ds4.PATH_DECODE).cpu().numpy()
    assert moe.status() == ds4.DS4MOE_EDEVICE
    y_ref = oracle.forward_routed(shape, layer, x, replaced, w.astype(np.float64))
    assert_close(y, y_ref, TOL_DECODE)
    y = moe.forward_routed(x_to_dev(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                           path=ds4.PATH_PREFILL).cpu().numpy()
    assert moe.status() == 0
    y_ref = oracle.forward_routed(shape, layer, x, idx, w.astype(np.float64))
    assert_close(y, y_ref, TOL_PREFILL)


def test_create_rejects_host_weights():
    shape = synth.Shape(256, 256, 4, 2, 0)
    layer = synth.make_layer(shape, 1234)
    w = to_dev(layer)
    w["gate"] = torch.from_numpy(layer["gate"])  # host memory
    with pytest.raises(ds4.DS4MoEError) as e:
        ds4.MoELayer(shape, w, 4)
    assert e.value.code == ds4.DS4MOE_EINVAL


@pytest.mark.parametrize("shape", [
    synth.Shape(256, 256, 1, 1, 0),        # one expert, no shared expert
    synth.Shape(256, 512, 6, 6, 256),      # K == E: every expert chosen
    synth.Shape(768, 256, 40, 8, 0),       # K at its maximum, H of 3 blocks
    synth.Shape(1024, 768, 64, 4, 512),    # ragged multiples of the block size
])
def test_shape_variants(shape):
    layer = synth.make_layer(shape, 4321)
    moe = ds4.MoELayer(shape, to_dev(layer), max_tokens=24)
    for T, path, tol in ((3, ds4.PATH_DECODE, TOL_DECODE), (24, ds4.PATH_PREFILL, TOL_PREFILL)):
        x = tokens(shape, T, 1000 + T)
        y = moe.forward(x_to_dev(x), path=path).cpu().numpy()
        y_ref, r = oracle.forward(shape, layer, x)
        idx, w, gap, _ = moe.route(x_to_dev(x))
        check_routing(idx.cpu().numpy(), w.cpu().numpy(), None, r, shape.top_k)
        assert_close(y, y_ref, tol)
    assert moe.status() == 0
    moe.close()


def test_router_bias_changes_selection_only():
    shape = synth.Shape(512, 256, 32, 6, 256)
    layer = synth.make_layer(shape, 777)
    layer["router_bias"] = (0.3 * synth.zipf_profile(32, 777)).astype(np.float32)
    moe = ds4.MoELayer(shape, to_dev(layer), max_tokens=16)
    x = tokens(shape, 16, 778)
    idx, w, gap, _ = moe.route(x_to_dev(x))
    ref = oracle.route(shape, layer["router_w"], layer["router_bias"], x)
    check_routing(idx.cpu().numpy(), w.cpu().numpy(), gap.cpu().numpy(), ref, shape.top_k)
    y = moe.forward(x_to_dev(x), path=ds4.PATH_DECODE).cpu().numpy()
    y_ref = oracle.forward_routed(shape, layer, x, ref["idx"], ref["weights"])
    assert_close(y, y_ref, TOL_DECODE)
    moe.close()


def test_memory_counts_every_resident_layout(tiny):
    """ds4moe_memory's weight bytes: the router (fp32 rows, their three bf16 parts
    padded to 128 rows, the bias), the routed experts in both resident layouts
    (84 B per 256 weights each) and the shared expert in both (34 B per 32
    weights each), plus at most the pieces' 256-byte alignment."""
    shape, layer, moe = tiny
    H, I, E, Ish = shape.hidden, shape.inter, shape.n_experts, shape.shared_inter
    router = E * H * 4 + -(-E // 128) * 128 * 3 * H * 2 + E * 4
    routed = 3 * E * I * H * 84 // 256
    shared = 3 * Ish * H * 34 // 32
    expected = router + 2 * routed + 2 * shared
    wb, sb = ds4.ds4moe_memory(moe.handle)
    assert expected <= wb <= expected + 64 * 1024, (wb, expected)
    assert sb > 0
