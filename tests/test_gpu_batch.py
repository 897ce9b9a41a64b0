"""GPU parity of the batch path (DS4MOE_PATH_BATCH): routing and grouping,
then two persistent tile-GEMV kernels over (distinct expert x up to 8 pairs,
row tile), every expert read once per group of its pairs.

The path computes what the decode path does (exact 2-bit and 8-bit products,
fp32 accumulation, SwiGLU rows as a hi + lo pair), so it is held to the
decode tolerance. Cases: the tiny layer at T = 1..64 (ragged slot counts, an
expert with more than 8 pairs needing several slots), a caller routing that
puts every pair on a few experts, a shape whose column blocks do not divide
evenly over the warps, the token limit, and the full H=4096, E=384 layer at
T = 16 and 64 (sampled rows). Every compute call goes through the C ABI.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_gb300 as ds4
import synth
from gpu_util import TOL_DECODE, TOL_PREFILL, assert_close, check_routing, to_dev, x_to_dev

pytestmark = pytest.mark.gpu


def tokens(shape, T, seed):
    return synth.normal_bf16(T * shape.hidden, seed, synth.S_X).reshape(T, shape.hidden)


def routed(moe, x, idx, w):
    return moe.forward_routed(x_to_dev(x), torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).cuda(),
                              torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).cuda(),
                              path=ds4.PATH_BATCH).cpu().numpy()


@pytest.fixture(scope="module")
def tiny():
    shape = synth.TINY_SHAPE
    layer = synth.make_layer(shape, synth.SEED_BASE)
    moe = ds4.MoELayer(shape, to_dev(layer), max_tokens=80)
    yield shape, layer, moe
    moe.close()


@pytest.mark.parametrize("T", [1, 5, 9, 16, 33, 63, 64])
def test_batch_matches_oracle(tiny, T):
    shape, layer, moe = tiny
    x = tokens(shape, T, 2100 + T)
    y = moe.forward(x_to_dev(x), path=ds4.PATH_BATCH).cpu().numpy()
    s = moe.stats()
    assert s.path == ds4.PATH_BATCH
    r = moe.inspect(T, grouping=False)
    y_ref, ref = oracle.forward(shape, layer, x)
    near = check_routing(r["idx"], r["w"], r["gap"], ref, shape.top_k)
    if near.any():
        y_ref = oracle.forward_routed(shape, layer, x, r["idx"], r["w"].astype(np.float64))
    assert_close(y, y_ref, TOL_DECODE)
    assert moe.status() == 0


@pytest.mark.parametrize("T,n_hot", [(9, 1), (16, 2), (64, 6), (64, 32)])
def test_batch_on_shared_experts(tiny, T, n_hot):
    """A routing on n_hot experts: up to T pairs per expert, i.e. up to eight
    slots of one expert, partly filled last slots."""
    shape, layer, moe = tiny
    rng = np.random.default_rng(3000 + T + n_hot)
    K = min(shape.top_k, n_hot)
    idx = np.full((T, shape.top_k), -1, dtype=np.int32)
    for t in range(T):
        idx[t, :K] = rng.choice(n_hot, K, replace=False)
        # the rest of the row: distinct experts outside the hot set
        idx[t, K:] = rng.choice(np.arange(n_hot, shape.n_experts), shape.top_k - K, replace=False)
    w = rng.random((T, shape.top_k)).astype(np.float32) + 0.1
    w /= w.sum(axis=1, keepdims=True)
    x = tokens(shape, T, 3100 + T)
    y = routed(moe, x, idx, w)
    y_ref = oracle.forward_routed(shape, layer, x, idx, w.astype(np.float64))
    assert_close(y, y_ref, TOL_DECODE)
    g = moe.inspect(T)
    assert g["counts"].max() == np.bincount(idx.ravel(), minlength=shape.n_experts).max()
    assert moe.status() == 0


def test_batch_equals_decode_numerics(tiny):
    """The batch and decode paths take the same exact products and the same
    SwiGLU rounding: their outputs agree far inside the tolerance."""
    shape, layer, moe = tiny
    x = tokens(shape, 8, 3300)
    xd = x_to_dev(x)
    yb = moe.forward(xd, path=ds4.PATH_BATCH).cpu().numpy()
    yd = moe.forward(xd, path=ds4.PATH_DECODE).cpu().numpy()
    d = np.linalg.norm(yb.astype(np.float64) - yd) / np.linalg.norm(yd.astype(np.float64))
    assert d < 1e-5, d


def test_batch_token_limit(tiny):
    shape, layer, moe = tiny
    x = x_to_dev(tokens(shape, ds4.BATCH_MAX_T + 1, 3400))
    y = torch.empty((ds4.BATCH_MAX_T + 1, shape.hidden), dtype=torch.float32, device="cuda")
    with pytest.raises(ds4.DS4MoEError) as e:
        ds4.ds4moe_forward_path(moe.handle, x, ds4.BATCH_MAX_T + 1, ds4.PATH_BATCH, y)
    assert e.value.code == ds4.DS4MOE_EINVAL
    # the automatic path hands the same call to the prefill path
    moe.forward(x)
    assert moe.stats().path == ds4.PATH_PREFILL
    assert moe.status() == 0


def test_batch_small_max_tokens():
    """A layer created for fewer than 64 tokens takes batch calls up to its own limit."""
    shape = synth.TINY_SHAPE
    layer = synth.make_layer(shape, synth.SEED_BASE)
    moe = ds4.MoELayer(shape, to_dev(layer), max_tokens=20)
    try:
        x = tokens(shape, 20, 3500)
        y = moe.forward(x_to_dev(x), path=ds4.PATH_BATCH).cpu().numpy()
        r = moe.inspect(20, grouping=False)
        y_ref = oracle.forward_routed(shape, layer, x, r["idx"], r["w"].astype(np.float64))
        assert_close(y, y_ref, TOL_DECODE)
        assert moe.status() == 0
    finally:
        moe.close()


@pytest.mark.parametrize("ish", [768, 0])
def test_batch_uneven_blocks(ish):
    """H=1280 (5 column blocks over 16 warps), I=768 (3 blocks over 8 warps); the
    shared expert's 8-bit stages of 1280 and 384 columns (40 and 12 blocks), or
    no shared expert."""
    shape = synth.Shape(1280, 768, 16, 4, ish)
    layer = synth.make_layer(shape, synth.SEED_BASE + 40)
    moe = ds4.MoELayer(shape, to_dev(layer), max_tokens=64)
    try:
        for T in (3, 40):
            x = tokens(shape, T, 3600 + T)
            y = moe.forward(x_to_dev(x), path=ds4.PATH_BATCH).cpu().numpy()
            r = moe.inspect(T, grouping=False)
            y_ref = oracle.forward_routed(shape, layer, x, r["idx"], r["w"].astype(np.float64))
            assert_close(y, y_ref, TOL_DECODE)
        assert moe.status() == 0
    finally:
        moe.close()


# Full-size rows checked against the oracle: both ends and a seeded sample.
def full_sample(T):
    return sorted(set([0, T - 1] + np.random.default_rng(T).choice(T, min(T, 6), replace=False).tolist()))


@pytest.fixture(scope="module")
def big():
    wl = synth.WORKLOADS["decode_t1"]
    layer = synth.make_layer(wl.shape, wl.layer_seeds[0])
    dev = to_dev(layer)
    moe = ds4.MoELayer(wl.shape, dev, max_tokens=64)
    del dev
    torch.cuda.empty_cache()
    yield wl.shape, layer, moe
    moe.close()


@pytest.mark.parametrize("T", [16, 64])
def test_batch_full_layer(big, T):
    shape, layer, moe = big
    x = synth.normal_bf16(T * shape.hidden, synth.SEED_BASE + 0x100 + T, synth.S_X).reshape(T, shape.hidden)
    xd = x_to_dev(x)
    y = moe.forward(xd).cpu().numpy()
    s = moe.stats()
    assert s.path == (ds4.PATH_BATCH if T > ds4.AUTO_DECODE_MAX_T else ds4.PATH_DECODE)
    r = moe.inspect(T, grouping=False)
    ref = oracle.route(shape, layer["router_w"], None, x)
    near = check_routing(r["idx"], r["w"], r["gap"], ref, shape.top_k)
    rows = np.array(full_sample(T))
    ridx = np.where(near[rows][:, None], r["idx"][rows], ref["idx"][rows])
    rw = np.where(near[rows][:, None], r["w"][rows].astype(np.float64), ref["weights"][rows])
    y_ref = oracle.forward_routed(shape, layer, np.ascontiguousarray(x[rows]), ridx, rw)
    assert_close(y[rows], y_ref, TOL_DECODE)
    assert np.isfinite(y).all()
    assert s.n_unique == len(np.unique(r["idx"]))
    assert moe.status() == 0


def test_a_bounded_wait_that_runs_out_is_reported(tiny):
    """Failure detection without a GPU fault: a test hook makes CTA 0 of the next
    batch product launch issue nothing for its first stage. Its waits give up
    after about a second, every role of the CTA stops and drains its own copies,
    ds4moe_status returns DS4MOE_ETIMEOUT, and the next call on the same handle
    is right again."""
    shape, layer, moe = tiny
    x = tokens(shape, 8, 3700)
    xd = x_to_dev(x)
    ds4.ds4moe_debug_skip_signal(moe.handle, 1)
    moe.forward(xd, path=ds4.PATH_BATCH)
    assert moe.status() == ds4.DS4MOE_ETIMEOUT
    y = moe.forward(xd, path=ds4.PATH_BATCH).cpu().numpy()
    r = moe.inspect(8, grouping=False)
    y_ref = oracle.forward_routed(shape, layer, x, r["idx"], r["w"].astype(np.float64))
    assert_close(y, y_ref, TOL_DECODE)
    assert moe.status() == 0
    with pytest.raises(ds4.DS4MoEError):
        ds4.ds4moe_debug_skip_signal(moe.handle, -1)


def test_wide_layer_without_a_batch_plan():
    """H=8192: a 2-bit stage of the batch kernel (two 16-row tiles over the whole
    row) does not fit its shared memory, so the layer has no batch path: an
    explicit batch call is refused, the automatic path takes the prefill path
    (shared expert on its GEMMs), and the decode kernel streams the wide rows in
    K chunks; both match the oracle."""
    shape = synth.Shape(8192, 256, 8, 2, 256)
    layer = synth.make_layer(shape, synth.SEED_BASE + 50)
    moe = ds4.MoELayer(shape, to_dev(layer), max_tokens=16)
    try:
        T = 9
        x = tokens(shape, T, 3800)
        xd = x_to_dev(x)
        y = torch.empty((T, shape.hidden), dtype=torch.float32, device="cuda")
        with pytest.raises(ds4.DS4MoEError) as e:
            ds4.ds4moe_forward_path(moe.handle, xd, T, ds4.PATH_BATCH, y)
        assert e.value.code == ds4.DS4MOE_EINVAL
        for path, want, tol in ((ds4.PATH_AUTO, ds4.PATH_PREFILL, TOL_PREFILL),
                                (ds4.PATH_DECODE, ds4.PATH_DECODE, TOL_DECODE)):
            yy = moe.forward(xd, path=path).cpu().numpy()
            assert moe.stats().path == want
            r = moe.inspect(T, grouping=False)
            y_ref = oracle.forward_routed(shape, layer, x, r["idx"], r["w"].astype(np.float64))
            assert_close(yy, y_ref, tol)
        assert moe.status() == 0
    finally:
        moe.close()
