"""GPU parity of the per-expert down gains (sidecar and post-training tables).

The gains of "YoungAi - DeepSeek V4.1 Flash on one DGX Spark" (sections 3 and
4.2) rescale each output channel of an expert's down projection: y = sum_k
w_k (s1_e * s2_e ⊙ ye_k) + ysh. Both paths run through the C ABI on the
oracle's routing (routing parity is covered elsewhere), with gain scales large
enough that a wrong channel, nibble or expert moves the output far beyond the
tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_gb300 as ds4
import synth
from gpu_util import assert_close, TOL_DECODE, TOL_PREFILL, rel_l2, to_dev, x_to_dev

pytestmark = pytest.mark.gpu

SCALE_BYTE = 127 - 2  # X = 1/4: gains 1 + e2m1/4 in [-0.5, 2.5]


def tokens(shape, T, seed):
    return synth.normal_bf16(T * shape.hidden, seed, synth.S_X).reshape(T, shape.hidden)


def gain_layer(layer, shape, seed, tables):
    L = dict(layer)
    if tables & 1:
        L["down_gain"] = synth.gain_table(shape.n_experts, shape.hidden, seed, synth.S_GAIN1, SCALE_BYTE)
    if tables & 2:
        L["down_gain2"] = synth.gain_table(shape.n_experts, shape.hidden, seed, synth.S_GAIN2, SCALE_BYTE)
    return L


def routed(moe, x, idx, w, path):
    return moe.forward_routed(x_to_dev(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                              path=path).cpu().numpy()


@pytest.fixture(scope="module")
def tiny():
    wl = synth.WORKLOADS["tiny"]
    layer = synth.make_layer(wl.shape, wl.layer_seeds[0])
    handles = {}
    for tables in (1, 2, 3):
        handles[tables] = ds4.MoELayer(wl.shape, to_dev(gain_layer(layer, wl.shape, 11, tables)), max_tokens=80)
    yield wl.shape, layer, handles
    for m in handles.values():
        m.close()


@pytest.mark.parametrize("tables", [1, 2, 3])
@pytest.mark.parametrize("path,T", [(ds4.PATH_DECODE, 1), (ds4.PATH_DECODE, 3), (ds4.PATH_DECODE, 8),
                                    (ds4.PATH_PREFILL, 9), (ds4.PATH_PREFILL, 80), (ds4.PATH_BATCH, 9),
                                    (ds4.PATH_BATCH, 64)])
def test_gains_match_oracle(tiny, tables, path, T):
    shape, layer, handles = tiny
    moe = handles[tables]
    x = tokens(shape, T, 700 + T)
    r = oracle.route(shape, layer["router_w"], None, x)
    w32 = r["weights"].astype(np.float32)
    y = routed(moe, x, r["idx"], w32, path)
    L = gain_layer(layer, shape, 11, tables)
    y_ref = oracle.forward_routed(shape, L, x, r["idx"], w32.astype(np.float64))
    y_plain = oracle.forward_routed(shape, layer, x, r["idx"], w32.astype(np.float64))
    # the gains move the output by far more than the tolerance
    assert rel_l2(y_plain, y_ref) > 20 * TOL_PREFILL
    assert_close(y, y_ref, (TOL_PREFILL if path == ds4.PATH_PREFILL else TOL_DECODE))
    assert moe.status() == 0


def test_unit_gains_are_bit_identical(tiny):
    """All codes 0 (and codes 8, -0) make every gain exactly 1: same bits as no table."""
    shape, layer, _ = tiny
    nb = shape.hidden // 32
    L = dict(layer)
    L["down_gain"] = np.tile(np.array([0] * 16 + [SCALE_BYTE], np.uint8), (shape.n_experts, nb, 1))
    L["down_gain2"] = np.tile(np.array([0x88] * 16 + [127], np.uint8), (shape.n_experts, nb, 1))
    plain = ds4.MoELayer(shape, to_dev(layer), max_tokens=40)
    unit = ds4.MoELayer(shape, to_dev(L), max_tokens=40)
    try:
        for T, path in ((1, ds4.PATH_DECODE), (8, ds4.PATH_DECODE), (40, ds4.PATH_PREFILL), (20, ds4.PATH_BATCH)):
            xd = x_to_dev(tokens(shape, T, 800 + T))
            a = plain.forward(xd, path=path)
            b = unit.forward(xd, path=path)
            assert torch.equal(a, b)
        assert plain.status() == 0 and unit.status() == 0
    finally:
        plain.close()
        unit.close()


def test_gains_follow_the_expert_not_the_slot(tiny):
    """The same experts in another order (weights permuted with them) give the same output."""
    shape, layer, handles = tiny
    moe = handles[3]
    T = 4
    x = tokens(shape, T, 901)
    r = oracle.route(shape, layer["router_w"], None, x)
    w32 = r["weights"].astype(np.float32)
    perm = np.array([5, 3, 0, 4, 1, 2])
    for path, tol in ((ds4.PATH_DECODE, TOL_DECODE), (ds4.PATH_PREFILL, TOL_PREFILL), (ds4.PATH_BATCH, TOL_DECODE)):
        a = routed(moe, x, r["idx"], w32, path)
        b = routed(moe, x, np.ascontiguousarray(r["idx"][:, perm]), np.ascontiguousarray(w32[:, perm]), path)
        assert_close(b, a, tol)


@pytest.fixture(scope="module")
def big():
    wl = synth.WORKLOADS["decode_t1"]
    layer = synth.make_layer(wl.shape, wl.layer_seeds[0], gains=2)
    dev = to_dev(layer)
    moe = ds4.MoELayer(wl.shape, dev, max_tokens=1024)
    del dev
    torch.cuda.empty_cache()
    yield wl.shape, layer, moe
    moe.close()


def test_full_size_decode_t8_and_prefill_rows(big):
    """H=4096, E=384 with both gain tables: decode T=8 on every token, prefill
    T=1024 on sampled rows, each on the library's own routing."""
    shape, layer, moe = big
    x = synth.make_tokens("decode_t8")
    xd = x_to_dev(x)
    y = moe.forward(xd).cpu().numpy()
    idx, w, _, _ = moe.route(xd)
    idx, w = idx.cpu().numpy(), w.cpu().numpy().astype(np.float64)
    y_ref = oracle.forward_routed(shape, layer, x, idx, w)
    assert_close(y, y_ref, TOL_DECODE)
    xp = synth.make_tokens("prefill_t1024")
    xpd = x_to_dev(xp)
    yp = moe.forward(xpd).cpu().numpy()
    idx, w, _, _ = moe.route(xpd)
    rows = [0, 1, 127, 128, 511, 1023]
    idx, w = idx.cpu().numpy()[rows], w.cpu().numpy()[rows].astype(np.float64)
    y_ref = oracle.forward_routed(shape, layer, xp[rows], idx, w)
    assert_close(yp[rows], y_ref, TOL_PREFILL)
    assert moe.status() == 0
