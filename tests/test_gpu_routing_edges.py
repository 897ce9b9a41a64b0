"""GPU parity on the routing contract's edge cases, for all three selection
implementations: the fused decode kernel (T <= 8 per launch), the fp32
router with its selection kernel (T < 16) and the tensor-core router with
exact refinement (T >= 16), and the outputs of the decode, batch and prefill
paths on those routings.

* Exact ties at the K-th boundary: two identical router rows with the same
  bias always tie for the K-th place; the lower expert index must win on
  every token and the reported gap must be exactly 0.
* Forced near-ties: a router row perturbed by a tiny amount puts a gap below
  1e-5 at the boundary of every token; the token must be flagged on both
  sides, and the output must equal the oracle's for the routing the GPU took
  (and for the oracle's routing through ds4moe_forward_routed).
* NaN scores rank below every number: an expert whose router row holds a NaN
  is never chosen while K others have numbers, and a token whose every score
  is NaN takes the K lowest expert indices with equal weights.
* The token-to-expert grouping (counts, positions, distinct experts) equals a
  stable counting sort of the GPU's own routing, bit for bit.

Every compute call goes through the C ABI; the oracle is the reference.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_gb300 as ds4
import synth
from gpu_util import NEAR_TIE, TOL_DECODE, TOL_PREFILL, TOL_WEIGHTS, assert_close, check_routing, to_dev, x_to_dev

pytestmark = pytest.mark.gpu

TOP = [1, 2, 3, 4, 7]  # always the top five (selection bias +2)
TIE = (5, 17)          # identical rows, bias +1: tie for sixth place on every token
NEAR = (5, 29)         # row 29 = row 5 with one weight nudged: a sub-1e-5 gap on every token
NAN_EXPERT = 9


def edge_layer(kind: str) -> dict:
    shape = synth.TINY_SHAPE
    layer = synth.make_layer(shape, synth.SEED_BASE)
    rw = layer["router_w"].copy()
    bias = np.zeros(shape.n_experts, dtype=np.float32)
    if kind in ("tie", "near"):
        bias[TOP] = 2.0
        a, b = TIE if kind == "tie" else NEAR
        rw[b] = rw[a]
        if kind == "near":
            rw[b, 0] += np.float32(1e-5)
        bias[[a, b]] = 1.0
    elif kind == "nan":
        rw[NAN_EXPERT, 100] = np.nan
        bias[NAN_EXPERT] = 2.0
    layer["router_w"] = rw
    layer["router_bias"] = bias
    return layer


def tokens(T, seed):
    H = synth.TINY_SHAPE.hidden
    return synth.normal_bf16(T * H, seed, synth.S_X).reshape(T, H)


@pytest.fixture(scope="module", params=["tie", "near", "nan"])
def edge(request):
    layer = edge_layer(request.param)
    moe = ds4.MoELayer(synth.TINY_SHAPE, to_dev(layer), max_tokens=64)
    yield request.param, layer, moe
    moe.close()


# (how the routing is produced, T): the decode kernel's own selection, the fp32
# router, the tensor-core router (route and the prefill forward)
CASES = [("decode", 1), ("decode", 5), ("decode", 8), ("route", 5), ("route", 12), ("route", 40),
         ("prefill", 40), ("batch", 13), ("batch", 64)]
PATHS = {"decode": ds4.PATH_DECODE, "prefill": ds4.PATH_PREFILL, "batch": ds4.PATH_BATCH}
TOLS = {"decode": TOL_DECODE, "batch": TOL_DECODE, "prefill": TOL_PREFILL}


def gpu_routing(moe, x, how):
    """(idx, w, gap, y or None) from the requested selection implementation."""
    T = x.shape[0]
    xd = x_to_dev(x)
    if how == "route":
        idx, w, gap, _ = moe.route(xd)
        return idx.cpu().numpy(), w.cpu().numpy(), gap.cpu().numpy(), None
    y = moe.forward(xd, path=PATHS[how]).cpu().numpy()
    r = moe.inspect(T, grouping=False)
    return r["idx"], r["w"], r["gap"], y


def oracle_weights(layer, x, idx):
    """Renormalised sigmoid scores of the given experts, from the oracle's exact logits."""
    L = oracle.logits(synth.TINY_SHAPE, layer["router_w"], x)
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(L, idx.astype(np.int64), axis=1)))
    return s / s.sum(axis=1, keepdims=True)


@pytest.mark.parametrize("how,T", CASES)
def test_selection_edges(edge, how, T):
    kind, layer, moe = edge
    shape = synth.TINY_SHAPE
    x = tokens(T, 900 + T + 31 * len(how))
    idx, w, gap, y = gpu_routing(moe, x, how)
    r = oracle.route(shape, layer["router_w"], layer["router_bias"], x)
    if kind == "tie":
        # the tie is exact on both sides: identical routing, lower index first, gap exactly 0
        assert (idx == r["idx"]).all()
        assert (idx[:, 5] == TIE[0]).all() and not (idx == TIE[1]).any()
        assert (gap == 0).all() and (r["gap"] == 0).all()
        assert np.abs(w - r["weights"]).max() <= TOL_WEIGHTS
    elif kind == "near":
        # flagged on both sides; the first five agree, the sixth is one of the pair
        assert (r["gap"] < NEAR_TIE).all() and (gap < NEAR_TIE).all()
        assert (idx[:, :5] == r["idx"][:, :5]).all()
        assert np.isin(idx[:, 5], NEAR).all()
        assert np.abs(w - oracle_weights(layer, x, idx)).max() <= TOL_WEIGHTS
    else:
        assert not (idx == NAN_EXPERT).any()
        check_routing(idx, w, gap, r, shape.top_k)
    if y is not None:
        tol = TOLS[how]
        y_ref = oracle.forward_routed(shape, layer, x, idx, w.astype(np.float64))
        assert_close(y, y_ref, tol)
    assert moe.status() == 0


@pytest.mark.parametrize("path,T", [(ds4.PATH_DECODE, 5), (ds4.PATH_PREFILL, 40), (ds4.PATH_BATCH, 40)])
def test_near_tie_output_on_the_oracles_routing(edge, path, T):
    kind, layer, moe = edge
    if kind != "near":
        pytest.skip("near-tie layer only")
    shape = synth.TINY_SHAPE
    x = tokens(T, 1300 + T)
    y_ref, r = oracle.forward(shape, layer, x)
    y = moe.forward_routed(x_to_dev(x), torch.from_numpy(r["idx"]).cuda(),
                           torch.from_numpy(r["weights"].astype(np.float32)).cuda(), path=path).cpu().numpy()
    assert_close(y, y_ref, TOL_PREFILL if path == ds4.PATH_PREFILL else TOL_DECODE)
    assert moe.status() == 0


@pytest.mark.parametrize("how,T", [("decode", 1), ("decode", 4), ("route", 6), ("route", 20), ("prefill", 20),
                                   ("batch", 20)])
def test_all_nan_token_takes_the_lowest_indices(how, T):
    shape = synth.TINY_SHAPE
    layer = synth.make_layer(shape, synth.SEED_BASE)
    moe = ds4.MoELayer(shape, to_dev(layer), max_tokens=64)
    try:
        x = tokens(T, 1500 + T)
        bad = T // 2
        x[bad, 3] = 0x7FC0  # bf16 NaN: every logit of this token is NaN
        idx, w, gap, y = gpu_routing(moe, x, how)
        assert list(idx[bad]) == list(range(shape.top_k))
        assert np.all(w[bad] == np.float32(1.0 / shape.top_k))
        good = np.arange(T) != bad
        r = oracle.route(shape, layer["router_w"], None, x)
        assert list(r["idx"][bad]) == list(range(shape.top_k))
        if good.any():
            check_routing(idx[good], w[good], gap[good], {k: v[good] for k, v in r.items()}, shape.top_k)
        if y is not None and good.any():
            y_ref = oracle.forward_routed(shape, layer, x[good], idx[good], w[good].astype(np.float64))
            assert_close(y[good], y_ref, TOLS[how])
        assert moe.status() == 0
    finally:
        moe.close()


@pytest.mark.parametrize("T", [40, 130, 2400])
def test_grouping_at_the_largest_expert_count(T):
    """E = 1024 and top-8: the widest per-warp histograms (128 KB of shared
    memory) and the scans at their full width; at T=2400 (19200 pairs) the
    indices no longer fit beside the histograms and the walks read them from
    global memory."""
    shape = synth.Shape(256, 256, 1024, 8, 256)
    layer = synth.make_layer(shape, 4242)
    moe = ds4.MoELayer(shape, to_dev(layer), max_tokens=T)
    try:
        moe.forward(x_to_dev(synth.normal_bf16(T * shape.hidden, 1900 + T, synth.S_X).reshape(T, shape.hidden)),
                    path=ds4.PATH_PREFILL)
        check_grouping(moe, T, shape.n_experts)
        assert moe.status() == 0
    finally:
        moe.close()


def counting_sort(idx, E):
    """Stable counting sort of the (token, k) pairs by expert: counts, the
    grouped position of every pair, the distinct experts and their starts."""
    flat = idx.ravel().astype(np.int64)
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    order = np.argsort(flat, kind="stable")
    inv = np.empty_like(order)
    inv[order] = np.arange(flat.size)
    uexp = np.nonzero(counts)[0]
    return counts, inv, uexp, np.append(offsets[uexp], flat.size)


def check_grouping(moe, T, E):
    g = moe.inspect(T)
    counts, inv, uexp, ustart = counting_sort(g["idx"], E)
    assert (g["counts"] == counts).all()
    assert (g["inv"] == inv).all()
    assert g["n_unique"] == uexp.size
    assert (g["uexp"] == uexp).all()
    assert (g["ustart"] == ustart).all()


@pytest.mark.parametrize("path,T", [(ds4.PATH_DECODE, 1), (ds4.PATH_DECODE, 3), (ds4.PATH_DECODE, 8),
                                    (ds4.PATH_PREFILL, 16), (ds4.PATH_PREFILL, 64), (ds4.PATH_BATCH, 9),
                                    (ds4.PATH_BATCH, 64), (ds4.PATH_PREFILL, 65), (ds4.PATH_PREFILL, 1000)])
def test_grouping_is_a_stable_counting_sort(path, T):
    """Up to 64 tokens the one-launch grouping of the batch path (or the decode
    kernel's own), above it the one-block grouping over per-warp histograms
    (T=1000: 6000 pairs, about 190 per expert, chunks of 188 pairs per warp)."""
    shape = synth.TINY_SHAPE
    layer = synth.make_layer(shape, synth.SEED_BASE)
    moe = ds4.MoELayer(shape, to_dev(layer), max_tokens=max(64, T))
    try:
        moe.forward(x_to_dev(tokens(T, 1700 + T)), path=path)
        check_grouping(moe, T, shape.n_experts)
        # a caller-given routing with heavy sharing: many pairs on few experts
        rng = np.random.default_rng(T)
        idx = np.stack([rng.choice(8, shape.top_k, replace=False) for _ in range(T)]).astype(np.int32)
        w = np.full((T, shape.top_k), 1.0 / shape.top_k, dtype=np.float32)
        moe.forward_routed(x_to_dev(tokens(T, 1800 + T)), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                           path=path)
        check_grouping(moe, T, shape.n_experts)
        assert moe.status() == 0
    finally:
        moe.close()
