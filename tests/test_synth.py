"""The seeded input generator: encodings, determinism and distributions."""
import numpy as np
import torch

import synth


def test_f16_encoder_matches_numpy_round_to_nearest_even():
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.normal(0, 0.01, 20000), rng.normal(0, 1e-5, 20000),  # many subnormal halves
        rng.normal(0, 3e4, 2000), [0.0, -0.0, 65504.0, 65519.9, 65520.0, 1e6, 2 ** -25, 2 ** -24 * 1.5,
                                   2 ** -26, 6.1e-5, 2 ** -14 * (1 + 2 ** -11)]])
    vals32 = vals.astype(np.float32)
    want = vals32.astype(np.float16).view(np.uint16)
    got = np.array([synth.f32_to_f16_bits(float(v)) for v in vals32], dtype=np.uint16)
    assert (got == want).all()


def test_bf16_encoder_matches_torch():
    rng = np.random.default_rng(12)
    vals = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-30, 100), [0.0, 1.0 + 2 ** -8]])
    vals32 = vals.astype(np.float32)
    want = torch.from_numpy(vals32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([synth.f32_to_bf16_bits(float(v)) for v in vals32], dtype=np.uint16)
    assert (got == want).all()


def test_counter_based_streams_are_deterministic_and_prefix_stable():
    a = synth.q2_matrix(64, 512, 123, synth.S_GATE)
    b = synth.q2_matrix(64, 512, 123, synth.S_GATE)
    c = synth.q2_matrix(32, 512, 123, synth.S_GATE)
    d = synth.q2_matrix(64, 512, 123, synth.S_UP)
    assert (a == b).all()
    assert (a[:32] == c).all()
    assert (a != d).mean() > 0.9
    x1 = synth.normal_bf16(1001, 5, synth.S_X)
    x2 = synth.normal_bf16(2000, 5, synth.S_X)
    assert (x1[:1000] == x2[:1000]).all()


def test_q2_distributions():
    m = synth.q2_matrix(2048, 4096, 7, synth.S_DOWN).reshape(-1, 84)
    scales = m[:, :16]
    codes = np.stack([(m[:, 16:80] >> (2 * s)) & 3 for s in range(4)])
    for v in (scales & 15, scales >> 4, codes):
        frac = np.bincount(v.ravel()) / v.size
        assert np.allclose(frac, 1.0 / frac.size, rtol=0.02)
    d = m[:, 80:82].copy().view(np.float16).astype(np.float64)
    dmin = m[:, 82:84].copy().view(np.float16).astype(np.float64)
    for v in (d, dmin):
        assert (v >= 0).all()
        # |N(0, 0.01^2)| has mean 0.01 * sqrt(2/pi)
        assert abs(v.mean() - 0.01 * np.sqrt(2 / np.pi)) < 2e-4


def test_q8_distributions():
    m = synth.q8_matrix(2048, 2048, 8, synth.S_SH_DOWN).reshape(-1, 34)
    q = m[:, 2:].view(np.int8).astype(np.int64)
    assert q.min() == -127 and q.max() == 127
    assert abs(q.mean()) < 0.2
    d = m[:, :2].copy().view(np.float16).astype(np.float64)
    assert (d >= 0).all() and abs(d.mean() - 0.001 * np.sqrt(2 / np.pi)) < 2e-5


def test_normals_and_rank_permutation():
    z = synth.normal_f32(1 << 20, 9, synth.S_ROUTER, 0.02).astype(np.float64)
    assert abs(z.mean()) < 1e-4 and abs(z.std() - 0.02) < 1e-4
    r = synth.rank_permutation(384, 10)
    assert sorted(r.tolist()) == list(range(1, 385))
    assert (r != synth.rank_permutation(384, 11)).any()


def test_workload_tokens_shapes_and_seeds():
    x = synth.make_tokens("decode_t8")
    assert x.shape == (8, 4096) and x.dtype == np.uint16
    assert (synth.make_tokens("decode_t8", T=1) == x[:1]).all()
    pool = synth.make_tokens("decode_t1", T=3, first=0)
    assert (pool[0] == synth.make_tokens("decode_t1")[0]).all()
    assert (pool[1] != pool[0]).any()
    xf = synth.bf16_bits_to_f32(synth.make_tokens("tiny")).astype(np.float64)
    assert abs(xf.std() - 1.0) < 0.05


def test_zipf_bias_profile():
    wl = synth.WORKLOADS["prefill_t4096_zipf4"]
    for seed in wl.layer_seeds:
        beta = synth.zipf_beta(seed)
        assert 0.05 < beta < 4.0
        p = synth.zipf_profile(384, seed)
        assert np.isclose(p.max(), 1.0) and np.isclose(np.sort(p)[-2], 2.0 ** -1.1)


def test_gain_and_mx4_distributions():
    g = synth.gain_table(8, 512, 3, synth.S_GAIN1)
    assert g.shape == (8, 16, 17) and (g[..., 16] == synth.GAIN_SCALE_BYTE).all()
    nib = np.concatenate([g[..., :16] & 15, g[..., :16] >> 4]).ravel()
    assert set(np.unique(nib)) == set(range(16))
    assert np.array_equal(g, synth.gain_table(8, 512, 3, synth.S_GAIN1))
    m = synth.mx4_matrix(64, 512, 5, synth.S_GATE)
    assert m.shape == (64, 16, 17)
    sc = m[..., 16].ravel()
    assert set(np.unique(sc)) == {synth.MX4_SCALE_BYTE - 2, synth.MX4_SCALE_BYTE - 1, synth.MX4_SCALE_BYTE}
    nib = np.concatenate([m[..., :16] & 15, m[..., :16] >> 4]).ravel()
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * nib.size / 16 and counts.max() < 1.1 * nib.size / 16
    # a prefix of the blocks does not depend on how many are drawn
    assert np.array_equal(synth.mx4_matrix(8, 512, 5, synth.S_GATE), m[:8])


def test_vq_generators():
    cb = synth.e4m3_codebook(4096, 3)
    ex = (cb >> 3) & 15
    assert cb.shape == (4096, 8) and ex.min() == 5 and ex.max() == 9  # magnitudes 2^-2 .. 2^2 * 1.875, no NaN
    assert abs((cb >> 7).mean() - 0.5) < 0.02
    layer = synth.make_layer(synth.Shape(512, 256, 2, 2, 0), 4, routed_format="vq", vq_bits=13)
    assert layer["gate"].shape == (2, 256 * 64 * 3 // 2) and layer["gate_plane"].shape == (2, 256 * 64 // 8)
    assert layer["down"].shape == (2, 512 * 32 * 3 // 2) and layer["down_rowgain"].shape == (2, 512)
    g = layer["up_rowgain"].view(np.float16).astype(np.float64)
    assert (g >= 0).all() and abs(g.mean() - synth.VQ_ROWGAIN_SIGMA * np.sqrt(2 / np.pi)) < 0.01
    again = synth.make_layer(synth.Shape(512, 256, 2, 2, 0), 4, routed_format="vq", vq_bits=13)
    assert all(np.array_equal(layer[k], again[k]) for k in ("vq_codebook", "gate", "gate_plane", "down_rowgain"))
    assert synth.make_layer(synth.Shape(512, 256, 2, 2, 0), 4, routed_format="vq")["gate_plane"] is None
