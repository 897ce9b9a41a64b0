"""GPU parity on the long skewed prefill: four H=4096, E=384 layers with a
Zipf(1.1) router bias, T=4096 tokens, in the launch configuration the
benchmark times (ds4moe_forward, auto path).

Routing (expert indices, weights, gaps) is compared on every token of every
layer; outputs are compared with the oracle on sampled rows, including tokens
of the hottest expert, whose 128-row tiles exercise the wide-accumulator path.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_gb300 as ds4
import synth
from gpu_util import assert_close, TOL_PREFILL, check_routing, rel_l2, to_dev, x_to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layer_no", range(4))
def test_prefill_t4096_zipf_layer(layer_no):
    wl = synth.WORKLOADS["prefill_t4096_zipf4"]
    shape = wl.shape
    layer = synth.make_layer(shape, wl.layer_seeds[layer_no], zipf=True)
    dev = to_dev(layer)
    moe = ds4.MoELayer(shape, dev, max_tokens=wl.tokens)
    del dev
    torch.cuda.empty_cache()
    try:
        x = synth.make_tokens("prefill_t4096_zipf4")
        xd = x_to_dev(x)
        y = moe.forward(xd).cpu().numpy()
        assert moe.stats().path == ds4.PATH_PREFILL
        idx, w, gap, _ = moe.route(xd)
        idx, w = idx.cpu().numpy(), w.cpu().numpy()
        r = oracle.route(shape, layer["router_w"], layer["router_bias"], x)
        near = check_routing(idx, w, gap.cpu().numpy(), r, shape.top_k)
        counts = np.bincount(r["idx"].ravel(), minlength=shape.n_experts)
        assert counts.max() >= 15 * counts.mean()  # the skew the workload asks for (~20x)
        hot = int(np.argmax(counts))
        hot_tokens = np.nonzero((r["idx"] == hot).any(axis=1))[0]
        rng = np.random.default_rng(1000 + layer_no)
        rows = sorted(set([0, 1, wl.tokens - 1] + rng.choice(hot_tokens, 4, replace=False).tolist()
                          + rng.choice(wl.tokens, 4, replace=False).tolist()))
        rows = np.array(rows)
        use_gpu = near[rows][:, None]
        ridx = np.where(use_gpu, idx[rows], r["idx"][rows])
        rw = np.where(use_gpu, w[rows].astype(np.float64), r["weights"][rows])
        y_ref = oracle.forward_routed(shape, layer, np.ascontiguousarray(x[rows]), ridx, rw)
        assert_close(y[rows], y_ref, TOL_PREFILL)
        assert np.isfinite(y).all()
        assert moe.status() == 0
    finally:
        moe.close()
        torch.cuda.empty_cache()
