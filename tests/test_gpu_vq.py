"""GPU parity of layers with VQ-12/13 routed experts (DS4MOE_FLAG_VQ12/VQ13).

Every 8 weights of a row are a codeword of the layer's E4M3 codebook times a
binary16 row gain; activations are not quantised. Two forms: CUDA-core
products (the decode bound) and the grouped GEMMs on the tensor cores, which
round x and the SwiGLU rows to binary16 (the prefill bound). Every compute call
goes through the C ABI.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_gb300 as ds4
import synth
from gpu_util import TOL_DECODE, TOL_PREFILL, assert_close, check_routing, to_dev, x_to_dev

pytestmark = pytest.mark.gpu

FLAGS = {12: ds4.FLAG_VQ12, 13: ds4.FLAG_VQ13}


def tokens(shape, T, seed):
    return synth.normal_bf16(T * shape.hidden, seed, synth.S_X).reshape(T, shape.hidden)


@pytest.fixture(scope="module", params=[12, 13])
def tiny(request):
    bits = request.param
    wl = synth.WORKLOADS["tiny"]
    layer = synth.make_layer(wl.shape, wl.layer_seeds[0], routed_format="vq", vq_bits=bits)
    moe = ds4.MoELayer(wl.shape, to_dev(layer), max_tokens=80, flags=FLAGS[bits])
    yield wl.shape, layer, moe
    moe.close()


@pytest.mark.parametrize("T", [1, 3, 8, 13, 80])
def test_forward_matches_oracle(tiny, T):
    shape, layer, moe = tiny
    x = tokens(shape, T, 1500 + T)
    xd = x_to_dev(x)
    y = moe.forward(xd, path=ds4.PATH_DECODE).cpu().numpy()
    s = moe.stats()
    idx, w, gap, _ = moe.route(xd)
    assert s.tokens == T and s.n_unique == len(np.unique(idx.cpu().numpy()))
    y_ref, r = oracle.forward(shape, layer, x)
    near = check_routing(idx.cpu().numpy(), w.cpu().numpy(), gap.cpu().numpy(), r, shape.top_k)
    if near.any():
        y_ref = oracle.forward_routed(shape, layer, x, idx.cpu().numpy(), w.cpu().numpy().astype(np.float64))
    assert_close(y, y_ref, TOL_DECODE)
    assert moe.status() == 0


def test_forward_routed_with_gains(tiny):
    shape, layer, _ = tiny
    L = dict(layer)
    L["down_gain"] = synth.gain_table(shape.n_experts, shape.hidden, 13, synth.S_GAIN1, 127 - 2)
    bits = layer["vq_bits"]
    moe = ds4.MoELayer(shape, to_dev(L), max_tokens=16, flags=FLAGS[bits])
    try:
        rng = np.random.default_rng(10)
        T = 6
        x = tokens(shape, T, 1601)
        idx = np.stack([rng.choice(shape.n_experts, shape.top_k, replace=False) for _ in range(T)]).astype(np.int32)
        w = rng.random((T, shape.top_k)).astype(np.float32)
        y_ref = oracle.forward_routed(shape, L, x, idx, w.astype(np.float64))
        for path, tol in ((ds4.PATH_DECODE, TOL_DECODE), (ds4.PATH_PREFILL, TOL_PREFILL)):
            y = moe.forward_routed(x_to_dev(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                                   path=path).cpu().numpy()
            assert_close(y, y_ref, tol)
        assert moe.status() == 0
    finally:
        moe.close()


@pytest.mark.parametrize("T", [1, 5, 16, 80])
def test_tensor_form_matches_oracle(tiny, T):
    shape, layer, moe = tiny
    x = tokens(shape, T, 1700 + T)
    y = moe.forward(x_to_dev(x), path=ds4.PATH_PREFILL).cpu().numpy()
    assert moe.stats().path == ds4.PATH_PREFILL
    r = moe.inspect(T, grouping=False)
    y_ref, ref = oracle.forward(shape, layer, x)
    near = check_routing(r["idx"], r["w"], r["gap"], ref, shape.top_k)
    if near.any():
        y_ref = oracle.forward_routed(shape, layer, x, r["idx"], r["w"].astype(np.float64))
    assert_close(y, y_ref, TOL_PREFILL)
    assert moe.status() == 0


def test_automatic_form_by_token_count(tiny):
    shape, layer, moe = tiny
    T = max(ds4.AUTO_VQ_PREFILL_MIN_T, 2)
    x = x_to_dev(tokens(shape, T, 1801))
    if ds4.AUTO_VQ_PREFILL_MIN_T > 1:
        moe.forward(x[:ds4.AUTO_VQ_PREFILL_MIN_T - 1])
        assert moe.stats().path == ds4.PATH_DECODE
    moe.forward(x[:ds4.AUTO_VQ_PREFILL_MIN_T])
    assert moe.stats().path == ds4.PATH_PREFILL
    moe.forward(x, path=ds4.PATH_DECODE)  # the CUDA-core form on request
    assert moe.stats().path == ds4.PATH_DECODE
    moe.forward(x, path=ds4.PATH_BATCH)
    assert moe.stats().path == ds4.PATH_DECODE
    assert moe.status() == 0


def test_create_checks_the_vq_fields():
    wl = synth.WORKLOADS["tiny"]
    layer = synth.make_layer(wl.shape, wl.layer_seeds[0], routed_format="vq", vq_bits=12)
    dev = to_dev(layer)
    missing = dict(dev)
    missing.pop("gate_rowgain")
    with pytest.raises(ds4.DS4MoEError):
        ds4.MoELayer(wl.shape, missing, max_tokens=8, flags=ds4.FLAG_VQ12)
    with pytest.raises(ds4.DS4MoEError):  # a 12-bit layer given as 13-bit: no planes
        ds4.MoELayer(wl.shape, dev, max_tokens=8, flags=ds4.FLAG_VQ13)


@pytest.fixture(scope="module")
def big():
    wl = synth.WORKLOADS["decode_t1"]
    layer = synth.make_layer(wl.shape, wl.layer_seeds[0], routed_format="vq", vq_bits=12)
    dev = to_dev(layer)
    moe = ds4.MoELayer(wl.shape, dev, max_tokens=256, flags=ds4.FLAG_VQ12)
    del dev
    torch.cuda.empty_cache()
    yield wl.shape, layer, moe
    moe.close()


def test_full_size_t1_and_t8(big):
    shape, layer, moe = big
    for x in (synth.make_tokens("decode_t1", T=1), synth.make_tokens("decode_t8")):
        xd = x_to_dev(x)
        y = moe.forward(xd, path=ds4.PATH_DECODE).cpu().numpy()
        idx, w, gap, _ = moe.route(xd)
        idx, w = idx.cpu().numpy(), w.cpu().numpy()
        y_ref = oracle.forward_routed(shape, layer, x, idx, w.astype(np.float64))
        assert_close(y, y_ref, TOL_DECODE)
    assert moe.status() == 0


def test_full_size_tensor_form(big):
    """H=4096, E=384 VQ-12 layer, 256 tokens on the tensor-core form; sampled rows."""
    shape, layer, moe = big
    T = 256
    x = synth.normal_bf16(T * shape.hidden, synth.SEED_BASE + 0x400, synth.S_X).reshape(T, shape.hidden)
    y = moe.forward(x_to_dev(x)).cpu().numpy()
    assert moe.stats().path == ds4.PATH_PREFILL
    r = moe.inspect(T, grouping=False)
    ref = oracle.route(shape, layer["router_w"], None, x)
    near = check_routing(r["idx"], r["w"], r["gap"], ref, shape.top_k)
    rows = np.array(sorted(set([0, 1, 127, 128, 255] + np.random.default_rng(8).choice(T, 5, replace=False).tolist())))
    ridx = np.where(near[rows][:, None], r["idx"][rows], ref["idx"][rows])
    rw = np.where(near[rows][:, None], r["w"][rows].astype(np.float64), ref["weights"][rows])
    y_ref = oracle.forward_routed(shape, layer, np.ascontiguousarray(x[rows]), ridx, rw)
    assert_close(y[rows], y_ref, TOL_PREFILL)
    assert np.isfinite(y).all()
    assert moe.status() == 0


def test_full_size_automatic_form_t1_and_t8(big):
    """H=4096, E=384 VQ-12 layer on the automatic path (the tensor-core form at
    every T): the decode pool's first token and the eight-token batch, on the
    library's routing, at the tensor-core form's bound."""
    shape, layer, moe = big
    for x in (synth.make_tokens("decode_t1", T=1), synth.make_tokens("decode_t8")):
        T = x.shape[0]
        y = moe.forward(x_to_dev(x)).cpu().numpy()
        assert moe.stats().path == ds4.PATH_PREFILL
        r = moe.inspect(T, grouping=False)
        check_routing(r["idx"], r["w"], r["gap"], oracle.route(shape, layer["router_w"], None, x), shape.top_k)
        y_ref = oracle.forward_routed(shape, layer, x, r["idx"], r["w"].astype(np.float64))
        assert_close(y, y_ref, TOL_PREFILL)
    assert moe.status() == 0


def test_full_size_vq13_both_forms():
    """H=4096, E=384 VQ-13 layer (the 12-bit stream plus the bit plane): the
    eight-token batch on the tensor-core form (the automatic one) and on the
    CUDA-core form, each at its bound, on the library's routing."""
    wl = synth.WORKLOADS["decode_t1"]
    layer = synth.make_layer(wl.shape, wl.layer_seeds[0], routed_format="vq", vq_bits=13)
    dev = to_dev(layer)
    moe = ds4.MoELayer(wl.shape, dev, max_tokens=8, flags=ds4.FLAG_VQ13)
    del dev
    torch.cuda.empty_cache()
    try:
        shape = wl.shape
        x = synth.make_tokens("decode_t8")
        for path, tol in ((ds4.PATH_AUTO, TOL_PREFILL), (ds4.PATH_DECODE, TOL_DECODE)):
            y = moe.forward(x_to_dev(x), path=path).cpu().numpy()
            r = moe.inspect(8, grouping=False)
            check_routing(r["idx"], r["w"], r["gap"], oracle.route(shape, layer["router_w"], None, x), shape.top_k)
            y_ref = oracle.forward_routed(shape, layer, x, r["idx"], r["w"].astype(np.float64))
            assert_close(y, y_ref, tol)
        assert moe.status() == 0
    finally:
        moe.close()
