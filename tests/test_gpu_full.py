"""GPU parity at the full H=4096, E=384 layer (decode T=1; T=8 on the batch and
the decode path; prefill T=1024).

The oracle computes every decode token and a sample of prefill rows one by
one; routing is compared on every token. Runs in the launch configuration
the benchmark times (ds4moe_forward, auto path).
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_gb300 as ds4
import synth
from gpu_util import assert_close, TOL_DECODE, TOL_PREFILL, check_routing, rel_l2, to_dev, x_to_dev

pytestmark = pytest.mark.gpu

# Prefill rows checked against the oracle: both ends, tile edges and a seeded sample.
PREFILL_SAMPLE = sorted(set([0, 1, 127, 128, 129, 511, 512, 1023]
                            + np.random.default_rng(99).choice(1024, 8, replace=False).tolist()))


@pytest.fixture(scope="module")
def big():
    wl = synth.WORKLOADS["decode_t1"]
    layer = synth.make_layer(wl.shape, wl.layer_seeds[0])
    dev = to_dev(layer)
    moe = ds4.MoELayer(wl.shape, dev, max_tokens=1024)
    del dev
    torch.cuda.empty_cache()
    yield wl.shape, layer, moe
    moe.close()


def test_decode_t1(big):
    shape, layer, moe = big
    x = synth.make_tokens("decode_t1", T=4)  # parity token and three more of the timing pool
    for t in range(4):
        xt = x[t:t + 1]
        y = moe.forward(x_to_dev(xt)).cpu().numpy()
        idx, w, gap, _ = moe.route(x_to_dev(xt))
        y_ref, r = oracle.forward(shape, layer, xt)
        near = check_routing(idx.cpu().numpy(), w.cpu().numpy(), gap.cpu().numpy(), r, shape.top_k)
        if near.any():
            y_ref = oracle.forward_routed(shape, layer, xt, idx.cpu().numpy(),
                                          w.cpu().numpy().astype(np.float64))
        assert_close(y, y_ref, TOL_DECODE)
    assert moe.status() == 0


def test_decode_t8(big):
    shape, layer, moe = big
    x = synth.make_tokens("decode_t8")
    xd = x_to_dev(x)
    y = moe.forward(xd).cpu().numpy()  # the automatic path: the batch kernels
    s = moe.stats()  # statistics of the forward call (route() below replaces them)
    yd = moe.forward(xd, path=ds4.PATH_DECODE).cpu().numpy()  # the fused decode kernel
    sd = moe.stats()
    idx, w, gap, _ = moe.route(xd)
    y_ref, r = oracle.forward(shape, layer, x)
    check_routing(idx.cpu().numpy(), w.cpu().numpy(), gap.cpu().numpy(), r, shape.top_k)
    assert s.path == ds4.PATH_BATCH and s.n_unique == len(np.unique(r["idx"]))
    assert sd.path == ds4.PATH_DECODE and sd.n_unique == s.n_unique
    assert_close(y, y_ref, TOL_DECODE)
    assert_close(yd, y_ref, TOL_DECODE)
    assert moe.status() == 0


def test_prefill_t1024(big):
    shape, layer, moe = big
    x = synth.make_tokens("prefill_t1024")
    xd = x_to_dev(x)
    y = moe.forward(xd).cpu().numpy()
    assert moe.stats().path == ds4.PATH_PREFILL
    idx, w, gap, _ = moe.route(xd)
    r = oracle.route(shape, layer["router_w"], None, x)
    near = check_routing(idx.cpu().numpy(), w.cpu().numpy(), gap.cpu().numpy(), r, shape.top_k)
    counts = np.bincount(r["idx"].ravel(), minlength=shape.n_experts)
    assert counts.max() < 4 * counts.mean()  # near-uniform load, as the workload intends
    rows = np.array(PREFILL_SAMPLE)
    gi, gw = idx.cpu().numpy()[rows], w.cpu().numpy()[rows].astype(np.float64)
    use_gpu_routing = near[rows][:, None]
    ridx = np.where(use_gpu_routing, gi, r["idx"][rows])
    rw = np.where(use_gpu_routing, gw, r["weights"][rows])
    y_ref = oracle.forward_routed(shape, layer, np.ascontiguousarray(x[rows]), ridx, rw)
    assert_close(y[rows], y_ref, TOL_PREFILL)
    assert np.isfinite(y).all()
    assert moe.status() == 0
