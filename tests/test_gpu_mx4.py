"""GPU parity of layers with MXFP4 routed experts (DS4MOE_FLAG_MXFP4).

Two forms: decode, whose expert products run on Q8-quantised activations (the
oracle's "q8" arithmetic), and prefill, the grouped GEMMs on the tensor cores
with FP4-quantised activations (the oracle's "mx4" arithmetic; held to the
prefill bound). Routing, shared expert, down gains and combine are the ones of
the 2-bit layer. Every compute call goes through the C ABI.
"""
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
    layer = synth.make_layer(wl.shape, wl.layer_seeds[0], routed_format="mx4")
    moe = ds4.MoELayer(wl.shape, to_dev(layer), max_tokens=80, flags=ds4.FLAG_MXFP4)
    yield wl.shape, layer, moe
    moe.close()


@pytest.mark.parametrize("T", [1, 3, 8, 13, 80])
def test_forward_matches_oracle(tiny, T):
    shape, layer, moe = tiny
    x = tokens(shape, T, 1100 + T)
    xd = x_to_dev(x)
    y = moe.forward(xd, path=ds4.PATH_DECODE).cpu().numpy()
    s = moe.stats()  # of the forward call (route() below replaces them)
    idx, w, gap, _ = moe.route(xd)
    assert s.tokens == T and s.n_unique == len(np.unique(idx.cpu().numpy()))
    y_ref, r = oracle.forward(shape, layer, x, act="q8")
    near = check_routing(idx.cpu().numpy(), w.cpu().numpy(), gap.cpu().numpy(), r, shape.top_k)
    if near.any():
        y_ref = oracle.forward_routed(shape, layer, x, idx.cpu().numpy(), w.cpu().numpy().astype(np.float64),
                                      act="q8")
    assert_close(y, y_ref, TOL_DECODE)
    assert moe.status() == 0


def test_decode_and_batch_arguments_give_the_decode_form(tiny):
    shape, layer, moe = tiny
    xd = x_to_dev(tokens(shape, 5, 1201))
    a = moe.forward(xd, path=ds4.PATH_DECODE)
    b = moe.forward(xd, path=ds4.PATH_BATCH)
    assert torch.equal(a, b) and moe.stats().path == ds4.PATH_DECODE
    assert moe.status() == 0


@pytest.mark.parametrize("T", [1, 16, 64, 80])
def test_prefill_form_matches_oracle(tiny, T):
    """FP4 activations on the tensor cores against the oracle's MXFP4 arithmetic."""
    shape, layer, moe = tiny
    x = tokens(shape, T, 1250 + T)
    xd = x_to_dev(x)
    y = moe.forward(xd, path=ds4.PATH_PREFILL).cpu().numpy()
    assert moe.stats().path == ds4.PATH_PREFILL
    r = moe.inspect(T, grouping=False)
    y_ref, ref = oracle.forward(shape, layer, x, act="mx4")
    near = check_routing(r["idx"], r["w"], r["gap"], ref, shape.top_k)
    if near.any():
        y_ref = oracle.forward_routed(shape, layer, x, r["idx"], r["w"].astype(np.float64), act="mx4")
    assert_close(y, y_ref, TOL_PREFILL)
    assert moe.status() == 0


def test_fp4_activations_are_what_the_prefill_form_uses(tiny):
    """The prefill form is far from the oracle with exact or Q8 activations
    (FP4 moves the output by about a fifth) and close to the oracle's FP4."""
    shape, layer, moe = tiny
    T = 40
    x = tokens(shape, T, 1451)
    r = oracle.route(shape, layer["router_w"], None, x)
    w32 = r["weights"].astype(np.float32)
    y = moe.forward_routed(x_to_dev(x), torch.from_numpy(r["idx"]).cuda(), torch.from_numpy(w32).cuda(),
                           path=ds4.PATH_PREFILL).cpu().numpy()
    yf = oracle.forward_routed(shape, layer, x, r["idx"], w32.astype(np.float64), act="mx4")
    yq = oracle.forward_routed(shape, layer, x, r["idx"], w32.astype(np.float64), act="q8")
    ye = oracle.forward_routed(shape, layer, x, r["idx"], w32.astype(np.float64), act="exact")
    assert rel_l2(y, yf) <= TOL_PREFILL
    assert rel_l2(y, yq) > 5 * TOL_PREFILL and rel_l2(y, ye) > 5 * TOL_PREFILL


def test_automatic_form_by_token_count(tiny):
    shape, layer, moe = tiny
    x = tokens(shape, ds4.AUTO_MX4_PREFILL_MIN_T, 1501)
    moe.forward(x_to_dev(x[:ds4.AUTO_MX4_PREFILL_MIN_T - 1]))
    assert moe.stats().path == ds4.PATH_DECODE
    moe.forward(x_to_dev(x))
    assert moe.stats().path == ds4.PATH_PREFILL
    assert moe.status() == 0


def test_forward_routed_and_gains(tiny):
    shape, layer, _ = tiny
    L = dict(layer)
    L["down_gain"] = synth.gain_table(shape.n_experts, shape.hidden, 12, synth.S_GAIN1, 127 - 2)
    moe = ds4.MoELayer(shape, to_dev(L), max_tokens=16, flags=ds4.FLAG_MXFP4)
    try:
        rng = np.random.default_rng(9)
        T = 6
        x = tokens(shape, T, 1301)
        idx = np.stack([rng.choice(shape.n_experts, shape.top_k, replace=False) for _ in range(T)]).astype(np.int32)
        w = rng.random((T, shape.top_k)).astype(np.float32)
        y = moe.forward_routed(x_to_dev(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                               path=ds4.PATH_DECODE).cpu().numpy()
        y_ref = oracle.forward_routed(shape, L, x, idx, w.astype(np.float64), act="q8")
        y_plain = oracle.forward_routed(shape, layer, x, idx, w.astype(np.float64), act="q8")
        assert rel_l2(y_plain, y_ref) > 0.1
        assert_close(y, y_ref, TOL_DECODE)
        # the prefill form applies the same gains in its combine
        y4 = moe.forward_routed(x_to_dev(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                                path=ds4.PATH_PREFILL).cpu().numpy()
        assert_close(y4, oracle.forward_routed(shape, L, x, idx, w.astype(np.float64), act="mx4"), TOL_PREFILL)
        assert moe.status() == 0
    finally:
        moe.close()


def test_q8_activations_are_what_the_layer_uses(tiny):
    """The oracle with exact activations is measurably farther from the kernels
    than the oracle with Q8 activations (the quantisation is really applied)."""
    shape, layer, moe = tiny
    T = 8
    x = tokens(shape, T, 1401)
    r = oracle.route(shape, layer["router_w"], None, x)
    w32 = r["weights"].astype(np.float32)
    y = moe.forward_routed(x_to_dev(x), torch.from_numpy(r["idx"]).cuda(), torch.from_numpy(w32).cuda(),
                           path=ds4.PATH_DECODE).cpu().numpy()
    yq = oracle.forward_routed(shape, layer, x, r["idx"], w32.astype(np.float64), act="q8")
    ye = oracle.forward_routed(shape, layer, x, r["idx"], w32.astype(np.float64), act="exact")
    assert rel_l2(y, yq) <= TOL_DECODE < rel_l2(y, ye)


@pytest.fixture(scope="module")
def big():
    wl = synth.WORKLOADS["decode_t1"]
    layer = synth.make_layer(wl.shape, wl.layer_seeds[0], routed_format="mx4")
    dev = to_dev(layer)
    moe = ds4.MoELayer(wl.shape, dev, max_tokens=256, flags=ds4.FLAG_MXFP4)
    del dev
    torch.cuda.empty_cache()
    yield wl.shape, layer, moe
    moe.close()


def test_full_size_t1_and_t8(big):
    """H=4096, E=384 MXFP4 layer: the decode token pool's first token and the
    eight-token batch, each on the library's own routing (checked too)."""
    shape, layer, moe = big
    for x in (synth.make_tokens("decode_t1", T=1), synth.make_tokens("decode_t8")):
        xd = x_to_dev(x)
        y = moe.forward(xd, path=ds4.PATH_DECODE).cpu().numpy()
        idx, w, gap, _ = moe.route(xd)
        idx, w = idx.cpu().numpy(), w.cpu().numpy()
        r = oracle.route(shape, layer["router_w"], None, x)
        check_routing(idx, w, gap.cpu().numpy(), r, shape.top_k)
        y_ref = oracle.forward_routed(shape, layer, x, idx, w.astype(np.float64), act="q8")
        assert_close(y, y_ref, TOL_DECODE)
    assert moe.status() == 0


def test_full_size_prefill_form(big):
    """H=4096, E=384 MXFP4 layer, 256 tokens on the tensor-core form: routing on
    every token, the output on a sample of rows against the oracle's FP4
    arithmetic."""
    shape, layer, moe = big
    T = 256
    x = synth.normal_bf16(T * shape.hidden, synth.SEED_BASE + 0x300, synth.S_X).reshape(T, shape.hidden)
    xd = x_to_dev(x)
    y = moe.forward(xd).cpu().numpy()
    assert moe.stats().path == ds4.PATH_PREFILL
    r = moe.inspect(T, grouping=False)
    ref = oracle.route(shape, layer["router_w"], None, x)
    near = check_routing(r["idx"], r["w"], r["gap"], ref, shape.top_k)
    rows = np.array(sorted(set([0, 1, 127, 128, 255] + np.random.default_rng(7).choice(T, 5, replace=False).tolist())))
    ridx = np.where(near[rows][:, None], r["idx"][rows], ref["idx"][rows])
    rw = np.where(near[rows][:, None], r["w"][rows].astype(np.float64), ref["weights"][rows])
    y_ref = oracle.forward_routed(shape, layer, np.ascontiguousarray(x[rows]), ridx, rw, act="mx4")
    assert_close(y[rows], y_ref, TOL_PREFILL)
    assert np.isfinite(y).all()
    assert moe.status() == 0


def test_full_size_automatic_form(big):
    """H=4096, E=384 MXFP4 layer on the automatic path: 2 tokens on the decode
    form (Q8 activations) and the eight-token batch on the prefill form (FP4
    activations, tensor cores), each against the oracle's arithmetic of that
    form on the library's routing."""
    shape, layer, moe = big
    pool = synth.make_tokens("decode_t8")
    for T, path, act, tol in ((2, ds4.PATH_DECODE, "q8", TOL_DECODE), (8, ds4.PATH_PREFILL, "mx4", TOL_PREFILL)):
        x = np.ascontiguousarray(pool[:T])
        y = moe.forward(x_to_dev(x)).cpu().numpy()
        assert moe.stats().path == path
        r = moe.inspect(T, grouping=False)
        check_routing(r["idx"], r["w"], r["gap"], oracle.route(shape, layer["router_w"], None, x), shape.top_k)
        y_ref = oracle.forward_routed(shape, layer, x, r["idx"], r["w"].astype(np.float64), act=act)
        assert_close(y, y_ref, tol)
    assert moe.status() == 0
