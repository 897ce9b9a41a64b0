"""GPU parity at the edges of the prefill path: the token counts where the
router switches from the fp32 dot-product kernel to the tensor-core GEMM
(with its K split and exact refinement), token counts that leave ragged
tiles, and the largest expert count and top-k the library accepts.
"""
import numpy as np
import pytest

import oracle
import quantized_moe_expert_gb300 as ds4
import synth
from gpu_util import assert_close, TOL_DECODE, TOL_PREFILL, check_routing, rel_l2, to_dev, x_to_dev

pytestmark = pytest.mark.gpu


def tokens(shape, T, seed):
    return synth.normal_bf16(T * shape.hidden, seed, synth.S_X).reshape(T, shape.hidden)


def run_and_check(moe, shape, layer, x, path, tol):
    xd = x_to_dev(x)
    y = moe.forward(xd, path=path).cpu().numpy()
    idx, w, gap, _ = moe.route(xd)
    r = oracle.route(shape, layer["router_w"], layer.get("router_bias"), x)
    near = check_routing(idx.cpu().numpy(), w.cpu().numpy(), gap.cpu().numpy(), r, shape.top_k)
    if near.any():
        y_ref = oracle.forward_routed(shape, layer, x, idx.cpu().numpy(), w.cpu().numpy().astype(np.float64))
    else:
        y_ref, _ = oracle.forward(shape, layer, x)
    assert_close(y, y_ref, tol)
    assert np.isfinite(y).all()
    assert moe.status() == 0


@pytest.fixture(scope="module")
def mid():
    shape = synth.Shape(1024, 512, 48, 6, 256)
    layer = synth.make_layer(shape, 777)
    moe = ds4.MoELayer(shape, to_dev(layer), max_tokens=300)
    yield shape, layer, moe
    moe.close()


@pytest.mark.parametrize("T", [9, 15, 16, 17, 130, 257])
def test_prefill_token_counts(mid, T):
    shape, layer, moe = mid
    run_and_check(moe, shape, layer, tokens(shape, T, 5000 + T), ds4.PATH_PREFILL, TOL_PREFILL)


def test_paths_in_rotation(mid):
    """Each path's call right after another path's, over token counts around the
    group boundaries: every call's kernels chain on the stream behind the
    previous call's (programmatic dependent launches), so a kernel that read
    its inputs before its predecessors finished would see the previous call's
    routing or rows here. Each output is held to the routing the library took."""
    shape, layer, moe = mid
    paths = ((ds4.PATH_PREFILL, TOL_PREFILL), (ds4.PATH_BATCH, TOL_DECODE), (ds4.PATH_DECODE, TOL_DECODE))
    for T in (9, 16, 17, 18, 24, 33):
        x = tokens(shape, T, 5000 + T)
        xd = x_to_dev(x)
        for path, tol in paths:
            y = moe.forward(xd, path=path).cpu().numpy()
            r = moe.inspect(T, grouping=False)
            y_ref = oracle.forward_routed(shape, layer, x, r["idx"], r["w"].astype(np.float64))
            assert_close(y, y_ref, tol)
            assert moe.status() == 0


def test_binary16_saturation_in_the_shared_gemms(mid):
    """Above 64 tokens the shared expert's tensor-core GEMMs take x as binary16,
    saturating at +-65504: a token with bf16 values beyond that range gets a
    finite output, and every other token of the call still matches the oracle."""
    shape, layer, moe = mid
    T = 80
    x = tokens(shape, T, 5900).copy()
    x[7, :64] = np.uint16(0x4980) # bf16 bits of 2^20, far beyond binary16's range
    xd = x_to_dev(x)
    y = moe.forward(xd, path=ds4.PATH_PREFILL).cpu().numpy()
    assert np.isfinite(y).all()
    r = moe.inspect(T, grouping=False)
    others = np.array([t for t in range(T) if t != 7])
    y_ref = oracle.forward_routed(shape, layer, np.ascontiguousarray(x[others]), r["idx"][others],
                                  r["w"][others].astype(np.float64))
    assert_close(y[others], y_ref, TOL_PREFILL)
    assert moe.status() == 0


def test_largest_expert_count_and_top_k():
    shape = synth.Shape(256, 256, 1024, 8, 256)
    layer = synth.make_layer(shape, 4242)
    moe = ds4.MoELayer(shape, to_dev(layer), max_tokens=40)
    try:
        for T, path, tol in ((8, ds4.PATH_DECODE, TOL_DECODE), (40, ds4.PATH_PREFILL, TOL_PREFILL)):
            run_and_check(moe, shape, layer, tokens(shape, T, 6000 + T), path, tol)
    finally:
        moe.close()
