"""Pins of the CPU oracle against facts independent of it.

Each test fixes a value the format definition, a closed form, a library
routine or brute force determines, chosen so that a plausible slip in the
oracle (a swapped nibble or field, a transposed matrix, gate and up
exchanged, bias leaking into the weights, a dropped shared term, wrong block
order) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth
from handmade import as_u8, bf16_bits, f16_bits, gain_block, q2_block, q8_block

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "blocks.json")

Q2_CLOSED = {
    "unit_scale_ramp": lambda i: i % 4,
    "scale_min_ramp": lambda i: 1.75 * (i // 16) - 3.75,
    "zero": lambda i: 0.0,
    "subnormal_d": lambda i: 45 * 2.0 ** -24,
    "negative_d": lambda i: -(i % 4),
    "byte_position": lambda i: ((i // 4) % 4) - ((i // 16) % 2),
}
Q8_CLOSED = {
    "half_scale_ramp": lambda i: 0.5 * (i if i < 16 else 15 - i),
    "neg_two_extremes": lambda i: -2 * (-127 if i % 2 == 0 else 127),
}


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ---- number formats ---------------------------------------------------------

def test_f16_decode_exhaustive_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    # signed zeros keep their sign
    assert math.copysign(1.0, oracle.f16(0x8000)) == -1.0


def test_bf16_decode_exhaustive_matches_bit_shift():
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()


def test_sigmoid_silu_closed_forms():
    assert oracle.sigmoid(0.0) == 0.5
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.sigmoid(math.log(3.0)) - 0.75) < 1e-15
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    assert oracle.silu(-800.0) == 0.0
    assert oracle.silu(50.0) == pytest.approx(50.0, rel=1e-20)


# ---- block dequantisation ---------------------------------------------------

@pytest.mark.parametrize("case", [c["name"] for c in json.load(open(GOLDEN))["q2"]])
def test_q2_golden_blocks(case):
    c = next(c for c in _golden()["q2"] if c["name"] == case)
    blk = (bytes.fromhex(c["scales"][0]) * c["scales"][1] + bytes.fromhex(c["qs"][0]) * c["qs"][1]
           + int(c["d"], 16).to_bytes(2, "little") + int(c["dmin"], 16).to_bytes(2, "little"))
    assert len(blk) == 84
    got = oracle.dequant_q2(np.frombuffer(blk, dtype=np.uint8))
    want = np.array([Q2_CLOSED[case](i) for i in range(256)], dtype=np.float64)
    assert (got == want).all()


@pytest.mark.parametrize("case", [c["name"] for c in json.load(open(GOLDEN))["q8"]])
def test_q8_golden_blocks(case):
    c = next(c for c in _golden()["q8"] if c["name"] == case)
    blk = int(c["d"], 16).to_bytes(2, "little") + bytes.fromhex(c["qs"][0]) * c["qs"][1]
    assert len(blk) == 34
    got = oracle.dequant_q8(np.frombuffer(blk, dtype=np.uint8))
    want = np.array([Q8_CLOSED[case](i) for i in range(32)], dtype=np.float64)
    assert (got == want).all()


def test_q2_round_trip_from_fields():
    """Random fields -> bytes (independent encoder) -> oracle decode == field formula."""
    rng = np.random.default_rng(1)
    for _ in range(50):
        d = float(np.float16(rng.normal(0, 0.02)))
        dmin = float(np.float16(abs(rng.normal(0, 0.02))))
        sc = rng.integers(0, 16, 16)
        m = rng.integers(0, 16, 16)
        q = rng.integers(0, 4, 256)
        got = oracle.dequant_q2(np.frombuffer(q2_block(d, dmin, sc, m, q), dtype=np.uint8))
        j = np.arange(256) // 16
        want = d * sc[j] * q - dmin * m[j]
        assert (got == want).all()


def test_q8_round_trip_from_fields():
    rng = np.random.default_rng(2)
    for _ in range(50):
        d = float(np.float16(rng.normal(0, 0.01)))
        q = rng.integers(-127, 128, 32)
        got = oracle.dequant_q8(np.frombuffer(q8_block(d, q), dtype=np.uint8))
        assert (got == d * q).all()


def test_row_dequant_block_order():
    """Block b of a row covers weights 256b..256b+255."""
    blocks = [q2_block(float(b + 1), 0.0, 1, 0, 1) for b in range(4)]
    row = np.frombuffer(b"".join(blocks), dtype=np.uint8)
    w = oracle.dequant_q2_matrix(row.reshape(1, 4, 84))[0]
    assert (w == np.repeat(np.arange(1, 5, dtype=np.float64), 256)).all()


# ---- routing ----------------------------------------------------------------

def _identity_router(E, H):
    w = np.zeros((E, H), dtype=np.float32)
    w[np.arange(E), np.arange(E)] = 1.0
    return w


def _route_logits(logits_rows, K, bias=None, H=None):
    """Route tokens whose logits are given exactly (identity router, x = logits)."""
    logits_rows = np.asarray(logits_rows, dtype=np.float32)
    T, E = logits_rows.shape
    H = H or max(E, 8)
    x = np.zeros((T, H), dtype=np.float32)
    x[:, :E] = logits_rows
    shape = synth.Shape(H, 256, E, K, 0)
    return oracle.route(shape, _identity_router(E, H), bias, bf16_bits(x), want_logits=True)


def _expected_topk(sel32, K):
    order = np.lexsort((np.arange(sel32.size), -sel32.astype(np.float64)))
    return order[:K]


def test_route_logits_are_exact_dot_products():
    rng = np.random.default_rng(3)
    H, E = 64, 5
    x = rng.normal(size=(3, H)).astype(np.float32)
    x = (bf16_bits(np.float32(np.round(x * 8) / 8)))  # small dyadic values, exact in bf16
    W = (np.round(rng.normal(size=(E, H)) * 16) / 16).astype(np.float32)
    r = oracle.route(synth.Shape(H, 256, E, 2, 0), W, None, x, want_logits=True)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    assert (r["logits"] == xf @ W.astype(np.float64).T).all()  # dyadic -> every sum exact


def test_topk_matches_sort_and_brute_force():
    rng = np.random.default_rng(4)
    E, K = 9, 3
    for _ in range(200):
        logits = np.clip(rng.normal(size=(1, E)) * 2, -7.5, 7.5)
        logits = np.float32(np.round(logits * 16) / 16)  # <= 7 significant bits: exact in bf16
        r = _route_logits(logits, K)
        sel = r["sel"][0]
        assert list(r["idx"][0]) == list(_expected_topk(sel, K))
        # brute force: the chosen set is the unique K-subset that beats every outsider
        best = [S for S in itertools.combinations(range(E), K)
                if all((sel[a], -a) > (sel[b], -b) for a in S for b in range(E) if b not in S)]
        assert len(best) == 1 and set(best[0]) == set(r["idx"][0])


def test_topk_large_random_vs_sort():
    rng = np.random.default_rng(5)
    E, K = 384, 6
    logits = np.float32(np.round(np.clip(rng.normal(size=(64, E)), -7.5, 7.5) * 16) / 16)
    r = _route_logits(logits, K, H=512)
    for t in range(64):
        assert list(r["idx"][t]) == list(_expected_topk(r["sel"][t], K))
        s = np.sort(r["sel"][t].astype(np.float64))[::-1]
        assert r["gap"][t] == s[K - 1] - s[K]


def test_topk_ties_prefer_lower_index():
    r = _route_logits([[1.0, 2.0, 2.0, 2.0, 0.5, 2.0]], 3)
    assert list(r["idx"][0]) == [1, 2, 3]
    assert r["gap"][0] == 0.0
    r = _route_logits([[0.25] * 8], 4)
    assert list(r["idx"][0]) == [0, 1, 2, 3]
    assert np.allclose(r["weights"][0], 0.25, rtol=0, atol=1e-15)


def _policy_topk(sel32, K):
    """Brute-force ranking under the selection policy: numbers by descending
    score then ascending index, every NaN after them by ascending index."""
    num = [e for e in range(sel32.size) if not np.isnan(sel32[e])]
    nan = [e for e in range(sel32.size) if np.isnan(sel32[e])]
    num.sort(key=lambda e: (-float(sel32[e]), e))
    return (num + nan)[:K]


def test_topk_nan_scores_rank_below_every_number():
    rng = np.random.default_rng(11)
    E, K = 24, 6
    shape = synth.Shape(256, 256, E, K, 0)
    for trial in range(300):
        L = rng.integers(-3, 4, size=(1, E)).astype(np.float64) / 4.0  # many exact ties
        L[0, rng.random(E) < rng.random()] = np.nan
        if trial % 7 == 0:
            L[0, rng.integers(E)] = -np.inf
        r = oracle.select(shape, L, None)
        assert list(r["idx"][0]) == _policy_topk(r["sel"][0], K), (trial, L)
    # a token with every score NaN takes the K lowest indices with equal weights
    r = oracle.select(shape, np.full((1, E), np.nan), None)
    assert list(r["idx"][0]) == list(range(K))
    assert np.all(r["weights"][0] == 1.0 / K) and np.isnan(r["gap"][0])


def test_topk_degenerate_k_equals_e_and_single_expert():
    r = _route_logits([[0.5, -1.0, 3.0]], 3)
    assert list(r["idx"][0]) == [2, 0, 1]
    assert r["gap"][0] == math.inf
    r = _route_logits([[-4.0]], 1)
    assert list(r["idx"][0]) == [0] and r["weights"][0, 0] == 1.0


def test_weights_renormalised_sigmoid():
    logits = [0.0, math.log(3.0), -1.5, 0.75]
    r = _route_logits([np.float32(np.round(np.array(logits) * 128) / 128)], 2)
    L = r["logits"][0]
    s = 1.0 / (1.0 + np.exp(-L))
    sel = [int(i) for i in r["idx"][0]]
    assert sel == [1, 3]
    want = s[sel] / s[sel].sum()
    assert np.allclose(r["weights"][0], want, rtol=1e-15, atol=0)
    assert abs(r["weights"][0].sum() - 1.0) < 1e-15


def test_bias_changes_selection_only():
    logits = np.float32([[0.0, 1.0, 2.0, 3.0]])
    bias = np.float32([10.0, 0.0, 0.0, 0.0])
    r = _route_logits(logits, 2, bias=bias)
    assert list(r["idx"][0]) == [0, 3]
    s0, s3 = 0.5, 1.0 / (1.0 + math.exp(-3.0))
    assert np.allclose(r["weights"][0], [s0 / (s0 + s3), s3 / (s0 + s3)], rtol=1e-15, atol=0)
    assert r["sel"][0, 0] == np.float32(0.5 + 10.0)


# ---- expert FFN closed forms ------------------------------------------------

def _one_expert_layer(H=512, I=256):
    """E=K=1, no shared expert, x = 1 on the first 256 dims and 2 on the rest.

    gate row i: block b has all codes 1, sc=1, m=0, d = a[i, b]  -> g_i = 256 sum_b a[i,b] x_b
    up row i:   d = bb[i, b]                                      -> u_i likewise
    down row j: codes 1, sc=1, m=1, d=c[j], dmin=e[j]            -> y_j = (c_j - e_j) sum_i h_i
    """
    nb = H // 256
    a = np.array([[2.0 ** -10 * (1 + (i + 3 * b) % 4) for b in range(nb)] for i in range(I)])
    bb = np.array([[2.0 ** -11 * (1 + (i + b) % 8) for b in range(nb)] for i in range(I)])
    c = np.array([2.0 ** -6 * (1 + j % 3) for j in range(H)])
    e = np.array([2.0 ** -8 * (j % 2) for j in range(H)])
    gate = as_u8([[q2_block(a[i, b], 0.0, 1, 0, 1) for b in range(nb)] for i in range(I)])
    up = as_u8([[q2_block(bb[i, b], 0.0, 1, 0, 1) for b in range(nb)] for i in range(I)])
    down = as_u8([[q2_block(c[j], e[j], 1, 1, 1) for _ in range(I // 256)] for j in range(H)])
    xval = np.where(np.arange(H) < 256, 1.0, 2.0)
    xb = np.array([256.0 * (1.0 if b == 0 else 2.0) for b in range(nb)])
    g = a @ xb
    u = bb @ xb
    h = g / (1 + np.exp(-g)) * u
    y = (c - e) * h.sum()
    return gate, up, down, xval, y


def test_single_expert_closed_form():
    H, I = 512, 256
    gate, up, down, xval, y_want = _one_expert_layer(H, I)
    shape = synth.Shape(H, I, 1, 1, 0)
    layer = {"gate": gate.reshape(1, I, H // 256, 84), "up": up.reshape(1, I, H // 256, 84),
             "down": down.reshape(1, H, I // 256, 84), "router_w": np.zeros((1, H), np.float32),
             "router_bias": None, "sh_gate": None, "sh_up": None, "sh_down": None}
    x = bf16_bits(np.float32(xval)[None, :])
    y, r = oracle.forward(shape, layer, x)
    assert r["idx"][0, 0] == 0 and r["weights"][0, 0] == 1.0
    assert np.allclose(y[0], y_want, rtol=1e-13, atol=0)
    # the expert entry point agrees with the layer on this case
    ye = oracle.expert(shape, layer["gate"][0], layer["up"][0], layer["down"][0], xval)
    assert np.allclose(ye, y_want, rtol=1e-13, atol=0)


def test_shared_expert_closed_form():
    """Shared gate row i = alpha_i, up row i = beta_i, down row j = gamma_j * (+1/-1 by block)."""
    H, Ish = 256, 64
    alpha = np.array([2.0 ** -9 * (1 + i % 4) for i in range(Ish)])
    beta = np.array([2.0 ** -10 * (1 + i % 5) for i in range(Ish)])
    gamma = np.array([2.0 ** -7 * (1 + j % 7) for j in range(H)])
    sg = as_u8([[q8_block(alpha[i], 1) for _ in range(H // 32)] for i in range(Ish)])
    su = as_u8([[q8_block(beta[i], 1) for _ in range(H // 32)] for i in range(Ish)])
    # down row j: block 0 codes +1, block 1 codes -1 (Ish = 64 -> 2 blocks)
    sd = as_u8([[q8_block(gamma[j], 1), q8_block(gamma[j], -1)] for j in range(H)])
    x = np.ones(H)
    g = alpha * H
    u = beta * H
    h = g / (1 + np.exp(-g)) * u
    want = gamma * (h[:32].sum() - h[32:].sum())
    got = oracle.shared(synth.Shape(H, 256, 1, 1, Ish), sg, su, sd, x)
    assert np.allclose(got, want, rtol=1e-13, atol=0)


def test_combine_two_experts_closed_form():
    """E=2, K=2, one-hot router: y = w0 ye0 + w1 ye1 + ysh with w from the sigmoid scores.

    Every gate/up row of expert e is constant (a_e, b_e), so g = a_e sum(x) and
    u = b_e sum(x); down row j of expert e is the constant c_ej, so
    ye_j = c_ej * I * silu(g) * u. The shared expert is the same with 8-bit rows.
    """
    H, I, Ish = 256, 256, 32
    a = [2.0 ** -10 * (1 + e) for e in range(2)]
    b = [2.0 ** -11 * (2 + e) for e in range(2)]
    c = [[2.0 ** -6 * (1 + j % 2 + 2 * e) for j in range(H)] for e in range(2)]
    gates = [as_u8([[q2_block(a[e], 0.0, 1, 0, 1)] for _ in range(I)]) for e in range(2)]
    ups = [as_u8([[q2_block(b[e], 0.0, 1, 0, 1)] for _ in range(I)]) for e in range(2)]
    downs = [as_u8([[q2_block(c[e][j], 0.0, 1, 0, 1)] for j in range(H)]) for e in range(2)]
    sg = as_u8([[q8_block(2.0 ** -8, 1) for _ in range(H // 32)] for _ in range(Ish)])
    su = as_u8([[q8_block(2.0 ** -8, 2) for _ in range(H // 32)] for _ in range(Ish)])
    sd = as_u8([[q8_block(2.0 ** -5, -1)] for _ in range(H)])
    router = np.zeros((2, H), np.float32)
    router[0, 0] = 1.0
    router[1, 1] = 1.0
    x = np.ones(H, np.float32)
    x[0], x[1] = 0.5, -1.25
    layer = {"gate": np.stack(gates), "up": np.stack(ups), "down": np.stack(downs), "router_w": router,
             "router_bias": None, "sh_gate": sg, "sh_up": su, "sh_down": sd}
    y, r = oracle.forward(synth.Shape(H, I, 2, 2, Ish), layer, bf16_bits(x[None, :]))
    xs = float(x.astype(np.float64).sum())
    s = np.array([1 / (1 + math.exp(-0.5)), 1 / (1 + math.exp(1.25))])
    w = s / s.sum()
    ye = []
    for e in range(2):
        g, u = a[e] * xs, b[e] * xs
        ye.append(np.array(c[e]) * I * (g / (1 + math.exp(-g)) * u))
    gsh, ush = 2.0 ** -8 * xs, 2.0 ** -8 * 2 * xs
    ysh = -(2.0 ** -5) * Ish * (gsh / (1 + math.exp(-gsh)) * ush)
    want = w[0] * ye[0] + w[1] * ye[1] + ysh
    assert list(r["idx"][0]) == [0, 1]
    assert np.allclose(r["weights"][0], w, rtol=1e-15, atol=0)
    assert np.allclose(y[0], want, rtol=1e-13, atol=0)


# ---- invariants on random layers --------------------------------------------

@pytest.fixture(scope="module")
def tiny():
    wl = synth.WORKLOADS["tiny"]
    layer = synth.make_layer(wl.shape, wl.layer_seeds[0])
    x = synth.make_tokens("tiny")
    return wl.shape, layer, x


def test_identical_experts_equal_single_expert(tiny):
    shape, layer, x = tiny
    L = dict(layer)
    for k in ("gate", "up", "down"):
        L[k] = np.ascontiguousarray(np.broadcast_to(layer[k][:1], layer[k].shape))
    y, r = oracle.forward(shape, L, x)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    for t in range(x.shape[0]):
        single = oracle.expert(shape, L["gate"][0], L["up"][0], L["down"][0], xf[t])
        ysh = oracle.shared(shape, L["sh_gate"], L["sh_up"], L["sh_down"], xf[t])
        ref = single + ysh
        assert np.linalg.norm(y[t] - ref) <= 1e-12 * np.linalg.norm(ref)


def test_token_independence_and_thread_count(tiny):
    shape, layer, x = tiny
    y_all, _ = oracle.forward(shape, layer, x, nthreads=4)
    y_one, _ = oracle.forward(shape, layer, x, nthreads=1)
    y_rows, _ = oracle.forward(shape, layer, x, nthreads=16)  # fewer tokens than threads: rows shared
    assert (y_all == y_one).all() and (y_rows == y_one).all()
    for t in range(x.shape[0]):
        yt, _ = oracle.forward(shape, layer, x[t:t + 1])
        assert (yt[0] == y_all[t]).all()


def test_expert_permutation_invariance(tiny):
    shape, layer, x = tiny
    y, r = oracle.forward(shape, layer, x)
    assert (r["gap"] > 0).all()
    perm = np.random.default_rng(7).permutation(shape.n_experts)  # new expert p holds old perm[p]
    L = dict(layer)
    for k in ("gate", "up", "down", "router_w"):
        L[k] = np.ascontiguousarray(layer[k][perm])
    y2, r2 = oracle.forward(shape, L, x)
    assert (perm[r2["idx"]] == r["idx"]).all()
    assert (y2 == y).all()


def test_shared_term_is_added_unweighted(tiny):
    shape, layer, x = tiny
    y, r = oracle.forward(shape, layer, x)
    no_sh = dict(layer, sh_gate=None, sh_up=None, sh_down=None)
    y0 = oracle.forward_routed(shape, no_sh, x, r["idx"], r["weights"])
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    for t in range(x.shape[0]):
        ysh = oracle.shared(shape, layer["sh_gate"], layer["sh_up"], layer["sh_down"], xf[t])
        assert np.allclose(y[t] - y0[t], ysh, rtol=1e-9, atol=1e-9 * np.abs(ysh).max())


def _np_dequant_q2(m):
    """Vectorised decoder written from the layout (cross-check, not a pin)."""
    m = m.reshape(-1, 84)
    scales = m[:, :16].astype(np.int64)
    qs = m[:, 16:80].astype(np.int64)
    d = m[:, 80:82].copy().view(np.float16).astype(np.float64)[:, 0]
    dmin = m[:, 82:84].copy().view(np.float16).astype(np.float64)[:, 0]
    q = np.stack([(qs >> (2 * s)) & 3 for s in range(4)], axis=-1).reshape(-1, 256)
    sc = np.repeat(scales & 15, 16, axis=1)
    mn = np.repeat(scales >> 4, 16, axis=1)
    return d[:, None] * sc * q - dmin[:, None] * mn


def _np_dequant_q8(m):
    m = m.reshape(-1, 34)
    d = m[:, :2].copy().view(np.float16).astype(np.float64)[:, 0]
    return d[:, None] * m[:, 2:].view(np.int8).astype(np.float64)


def test_dense_cross_check(tiny):
    """All experts evaluated densely with numpy matmuls, masked by the routing."""
    shape, layer, x = tiny
    H, I, E = shape.hidden, shape.inter, shape.n_experts
    y, r = oracle.forward(shape, layer, x)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    Wg = _np_dequant_q2(layer["gate"]).reshape(E, I, H)
    Wu = _np_dequant_q2(layer["up"]).reshape(E, I, H)
    Wd = _np_dequant_q2(layer["down"]).reshape(E, H, I)
    g = np.einsum("eih,th->tei", Wg, xf)
    u = np.einsum("eih,th->tei", Wu, xf)
    h = g / (1 + np.exp(-g)) * u
    ye = np.einsum("ehi,tei->teh", Wd, h)
    gate_w = np.zeros((x.shape[0], E))
    for t in range(x.shape[0]):
        gate_w[t, r["idx"][t]] = r["weights"][t]
    Sg = _np_dequant_q8(layer["sh_gate"]).reshape(shape.shared_inter, H)
    Su = _np_dequant_q8(layer["sh_up"]).reshape(shape.shared_inter, H)
    Sd = _np_dequant_q8(layer["sh_down"]).reshape(H, shape.shared_inter)
    gs, us = xf @ Sg.T, xf @ Su.T
    ysh = (gs / (1 + np.exp(-gs)) * us) @ Sd.T
    dense = np.einsum("te,teh->th", gate_w, ye) + ysh
    assert np.linalg.norm(dense - y) <= 1e-12 * np.linalg.norm(dense)
    # routing by numpy over the oracle's own fp32 selection scores
    for t in range(x.shape[0]):
        assert list(r["idx"][t]) == list(_expected_topk(r["sel"][t], shape.top_k))


# ---- per-expert down gains ---------------------------------------------------
# "YoungAi - DeepSeek V4.1 Flash on one DGX Spark", section 4.2: the gains are
# FP4 E2M1 with one scale per 32 channels in 17-byte blocks, the stored lattice
# value is s - 1, and the block sum is y = sum_k rw_k (s_e ⊙ ye_k) + ysh;
# section 3: g_eff = g_base * s_sidecar * s_posttrain (two tables multiply).

# OCP microscaling E2M1: exponent bias 1, one mantissa bit, exponent 0 subnormal;
# the eight magnitudes of the format as the standard lists them.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_code_table():
    got = [oracle.e2m1(c) for c in range(16)]
    assert got[:8] == E2M1_MAGNITUDES
    assert got[8:] == [-v for v in E2M1_MAGNITUDES]
    assert math.copysign(1.0, got[8]) == -1.0  # code 8 is negative zero
    # "E2M1 has only 8 magnitudes"
    assert len({abs(v) for v in got}) == 8


def test_e8m0_scale():
    assert oracle.e8m0(127) == 1.0
    assert oracle.e8m0(127 - 5) == 2.0 ** -5
    assert oracle.e8m0(0) == 2.0 ** -127
    assert oracle.e8m0(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0(255))


def test_gain_block_fields():
    """Channel i reads nibble i % 2 of byte i // 2 (even channel low), scale byte last."""
    codes = [(5 * i + 3) % 16 for i in range(32)]
    blk = np.frombuffer(gain_block(codes, 127 - 3), np.uint8)
    want = [1.0 + 2.0 ** -3 * (E2M1_MAGNITUDES[c & 7] * (-1 if c & 8 else 1)) for c in codes]
    assert list(oracle.gain_block(blk)) == want
    # a single nonzero code lands on its own channel only
    for ch in (0, 1, 6, 31):
        c = [0] * 32
        c[ch] = 7  # +6
        s = oracle.gain_block(np.frombuffer(gain_block(c, 127 - 4), np.uint8))
        assert s[ch] == 1.0 + 6 * 2.0 ** -4 and np.count_nonzero(s != 1.0) == 1


def test_gain_table_sizes_match_the_pages():
    """17 bytes per 32 channels of each expert: with the pages' 5,120 channels,
    384 experts and top-6, about 40 MB for 39 layers and about 0.6 MB read per
    decoded token (sections 3 and 4.2)."""
    H, E, K, layers = 5120, 384, 6, 39
    t = synth.gain_table(2, H, 1, synth.S_GAIN1)
    assert t.shape == (2, H // 32, synth.GAIN_BLOCK_BYTES) and synth.GAIN_BLOCK_BYTES == 17
    per_expert = t[0].nbytes
    assert abs(E * per_expert * layers / 40e6 - 1) < 0.05
    assert abs(K * per_expert * layers / 0.6e6 - 1) < 0.1


def test_unit_gains_leave_the_layer_unchanged(tiny):
    shape, layer, x = tiny
    y0, r = oracle.forward(shape, layer, x)
    L = dict(layer)
    nb = shape.hidden // 32
    ones = as_u8([[gain_block(0, 127) for _ in range(nb)] for _ in range(shape.n_experts)])
    zeros_neg = as_u8([[gain_block(8, 3) for _ in range(nb)] for _ in range(shape.n_experts)])
    L["down_gain"], L["down_gain2"] = ones, zeros_neg
    y1 = oracle.forward_routed(shape, L, x, r["idx"], r["weights"])
    assert np.array_equal(y0, y1)


def test_gain_closed_form_one_expert():
    """E=K=1: y_j = s1_j s2_j (c_j - e_j) sum_i h_i, per output channel."""
    H, I = 512, 256
    gate, up, down, xval, y_plain = _one_expert_layer(H, I)
    nb = H // 32
    c1 = [[(j + 3 * b) % 16 for j in range(32)] for b in range(nb)]
    c2 = [[(7 * j + b) % 16 for j in range(32)] for b in range(nb)]
    g1 = as_u8([[gain_block(c1[b], 127 - 3) for b in range(nb)]])
    g2 = as_u8([[gain_block(c2[b], 127 - 4) for b in range(nb)]])

    def val(c):
        return E2M1_MAGNITUDES[c & 7] * (-1 if c & 8 else 1)
    s1 = np.array([1 + 2.0 ** -3 * val(c1[j // 32][j % 32]) for j in range(H)])
    s2 = np.array([1 + 2.0 ** -4 * val(c2[j // 32][j % 32]) for j in range(H)])
    shape = synth.Shape(H, I, 1, 1, 0)
    layer = {"gate": gate.reshape(1, I, H // 256, 84), "up": up.reshape(1, I, H // 256, 84),
             "down": down.reshape(1, H, I // 256, 84), "sh_gate": None, "sh_up": None, "sh_down": None,
             "down_gain": g1}
    x = bf16_bits(np.float32(xval)[None, :])
    idx, w = np.zeros((1, 1), np.int32), np.ones((1, 1))
    y1 = oracle.forward_routed(shape, layer, x, idx, w)
    assert np.allclose(y1[0], s1 * y_plain, rtol=1e-13, atol=0)
    layer["down_gain2"] = g2
    y2 = oracle.forward_routed(shape, layer, x, idx, w)
    assert np.allclose(y2[0], s1 * s2 * y_plain, rtol=1e-13, atol=0)
    del layer["down_gain"]
    y3 = oracle.forward_routed(shape, layer, x, idx, w)
    assert np.allclose(y3[0], s2 * y_plain, rtol=1e-13, atol=0)


def test_gain_correction_is_routed_per_expert(tiny):
    """Delta = sum_k rw_k (s_{e_k} - 1) ⊙ ye_k: the gains of the expert a token
    picked, never those of its k-th slot or of another expert."""
    shape, layer, x = tiny
    y0, r = oracle.forward(shape, layer, x)
    L = dict(layer)
    L["down_gain"] = synth.gain_table(shape.n_experts, shape.hidden, 7, synth.S_GAIN1, 127 - 2)
    y1 = oracle.forward_routed(shape, L, x, r["idx"], r["weights"])
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    for t in range(x.shape[0]):
        delta = np.zeros(shape.hidden)
        for k in range(shape.top_k):
            e = int(r["idx"][t, k])
            s = np.concatenate([oracle.gain_block(b) for b in L["down_gain"][e]])
            ye = oracle.expert(shape, layer["gate"][e], layer["up"][e], layer["down"][e], xf[t])
            delta += r["weights"][t, k] * (s - 1) * ye
        assert np.allclose(y1[t] - y0[t], delta, rtol=1e-9, atol=1e-12 * np.abs(y0[t]).max())


# ---- MXFP4 routed experts ----------------------------------------------------
# "Running DeepSeek V4 Flash on an RTX 5080 ...", model list: MXFP4 routed
# experts; batched expert work on FP4 activations, decode on Q8 activations.
# Element and scale types: OCP microscaling (E2M1, E8M0 per 32).

def _mx4_layer_one_expert(H=256, I=256, code_g=2, code_u=4, sc_gu=127 - 6, down_codes=None, sc_d=127 - 5):
    """E=K=1 MXFP4 layer: every gate row the constant e2m1(code_g) 2^(sc-127),
    up likewise, down row j the constant code down_codes[j]."""
    if down_codes is None:
        down_codes = [(j % 7) + 1 + 8 * (j % 2) for j in range(H)]
    gate = as_u8([[gain_block(code_g, sc_gu) for _ in range(H // 32)] for _ in range(I)])
    up = as_u8([[gain_block(code_u, sc_gu) for _ in range(H // 32)] for _ in range(I)])
    down = as_u8([[gain_block(down_codes[j], sc_d) for _ in range(I // 32)] for j in range(H)])
    layer = {"gate": gate.reshape(1, I, H // 32, 17), "up": up.reshape(1, I, H // 32, 17),
             "down": down.reshape(1, H, I // 32, 17), "sh_gate": None, "sh_up": None, "sh_down": None,
             "routed_format": "mx4"}
    return layer


def _e2m1(c):
    return E2M1_MAGNITUDES[c & 7] * (-1.0 if c & 8 else 1.0)


def _np_q8(v):
    """Q8 blocks in numpy float32 arithmetic (IEEE): d = amax/127, q = rint(v/d)."""
    v = np.asarray(v, dtype=np.float32).reshape(-1, 32)
    amax = np.abs(v).max(axis=1)
    d = amax / np.float32(127)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(d[:, None] > 0, np.rint(v / d[:, None]), 0).astype(np.int8)
    return d, q.reshape(-1)


def _np_mx4_code(r):
    """E2M1 code nearest to r: all 16 codes, least distance, ties to the code
    with mantissa bit 0; magnitudes above 6 go to 6; sign follows r."""
    mag = min(abs(r), 6.0)
    cands = sorted(range(8), key=lambda c: (abs(mag - E2M1_MAGNITUDES[c]), c & 1))
    return cands[0] | (8 if math.copysign(1.0, r) < 0 else 0)


def _np_mx4(v):
    v = np.asarray(v, dtype=np.float32).reshape(-1, 32).astype(np.float64)
    sc, codes = [], []
    for blk in v:
        amax = np.abs(blk).max()
        if amax == 0:
            b = 0
        else:
            m, e = np.frexp(amax)
            b = int(min(max(e - 1 - 2 + 127, 0), 254))
        X = 2.0 ** (b - 127)
        sc.append(b)
        codes += [_np_mx4_code(r / X) for r in blk]
    return np.array(sc, np.uint8), np.array(codes, np.uint8)


def test_mx4_block_fields():
    codes = [(5 * i + 3) % 16 for i in range(32)]
    blk = np.frombuffer(gain_block(codes, 127 - 6), np.uint8)
    assert list(oracle.dequant_mx4(blk)) == [2.0 ** -6 * _e2m1(c) for c in codes]
    for ch in (0, 1, 17, 31):
        c = [0] * 32
        c[ch] = 5  # +3
        w = oracle.dequant_mx4(np.frombuffer(gain_block(c, 127 + 2), np.uint8))
        assert w[ch] == 12.0 and np.count_nonzero(w) == 1


def test_act_q8_is_binary32_round_to_nearest_even():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(32 * 6).astype(np.float32), np.zeros(32, np.float32),
                        # amax 127: d = 1, ties x.5 go to the even integer
                        np.array([127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -126.5] + [0.0] * 24, np.float32)])
    d, q = oracle.act_q8(x)
    dw, qw = _np_q8(x)
    assert np.array_equal(d, dw) and np.array_equal(q, qw)
    assert list(q[-32:-24]) == [127, 2, 4, -2, -4, 0, 2, -126]
    assert d[6] == 0 and not q[192:224].any()


def test_act_mx4_is_the_ocp_conversion():
    # element rounding on the E2M1 grid (X = 1 when the block maximum is in [4, 8))
    vals = [6.0, 2.5, 3.5, 5.0, 0.25, 0.75, 1.25, 1.75, -2.6, -0.1, 4.9, 0.0]
    want = [7, 4, 6, 6, 0, 2, 2, 4, 13, 8, 6, 0]
    sc, c = oracle.act_mx4(np.array(vals + [0.0] * 20, np.float32))
    assert sc[0] == 127 and list(c[:12]) == want
    # the scale: 2^(floor(log2 amax) - 2); values above 6 X saturate
    for amax, byte in ((15.5, 128), (8.0, 128), (7.99, 127), (0.3, 123), (2.0 ** -130, 0)):
        sc, c = oracle.act_mx4(np.array([amax] + [0.0] * 31, np.float32))
        assert sc[0] == byte
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(32 * 8) * np.repeat(2.0 ** rng.integers(-6, 6, 8), 32)).astype(np.float32)
    sc, c = oracle.act_mx4(x)
    scw, cw = _np_mx4(x)
    assert np.array_equal(sc, scw) and np.array_equal(c, cw)


def test_mx4_expert_closed_form_q8_and_mx4_activations():
    """Constant gate/up rows: g = a * sum(a_x), u = b * sum(a_x) with a_x the
    quantised x; h quantised again; down row j constant c_j: ye_j = c_j sum(hq)."""
    H, I = 256, 256
    layer = _mx4_layer_one_expert(H, I)
    shape = synth.Shape(H, I, 1, 1, 0)
    a, b = 2.0 ** -6 * 1.0, 2.0 ** -6 * 2.0
    c = np.array([2.0 ** -5 * _e2m1((j % 7) + 1 + 8 * (j % 2)) for j in range(H)])
    rng = np.random.default_rng(5)
    x = rng.standard_normal(H).astype(np.float32)
    xb = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)  # exact in bf16
    for act in ("q8", "mx4"):
        if act == "q8":
            d, q = _np_q8(xb)
            ax = np.repeat(d.astype(np.float64), 32) * q
        else:
            sc, cc = _np_mx4(xb)
            ax = np.repeat(2.0 ** (sc.astype(np.float64) - 127), 32) * np.array([_e2m1(v) for v in cc])
        g, u = a * ax.sum(), b * ax.sum()
        h = np.full(I, np.float32(g / (1 + math.exp(-g)) * u))
        if act == "q8":
            d, q = _np_q8(h)
            hq = np.repeat(d.astype(np.float64), 32) * q
        else:
            sc, cc = _np_mx4(h)
            hq = np.repeat(2.0 ** (sc.astype(np.float64) - 127), 32) * np.array([_e2m1(v) for v in cc])
        want = c * hq.sum()
        y = oracle.forward_routed(shape, layer, bf16_bits(xb[None, :]), np.zeros((1, 1), np.int32),
                                  np.ones((1, 1)), act=act)
        assert np.allclose(y[0], want, rtol=1e-12, atol=0)
        ye = oracle.expert_mx4(shape, act, layer["gate"][0], layer["up"][0], layer["down"][0], xb)
        assert np.allclose(ye, want, rtol=1e-12, atol=0)


def test_mx4_exact_activations_match_dense_numpy():
    shape = synth.Shape(512, 256, 4, 2, 0)
    layer = synth.make_layer(shape, 77, routed_format="mx4")
    layer["sh_gate"] = layer["sh_up"] = layer["sh_down"] = None
    x = synth.normal_bf16(3 * 512, 78, synth.S_X).reshape(3, 512)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    tab = np.array([_e2m1(c) for c in range(16)])

    def dq(m):
        m = m.reshape(-1, 17)
        lo, hi = m[:, :16] & 15, m[:, :16] >> 4
        codes = np.stack([lo, hi], axis=2).reshape(-1, 32)
        return (tab[codes] * 2.0 ** (m[:, 16:17].astype(np.float64) - 127)).reshape(-1)
    Wg = dq(layer["gate"]).reshape(4, 256, 512)
    Wu = dq(layer["up"]).reshape(4, 256, 512)
    Wd = dq(layer["down"]).reshape(4, 512, 256)
    idx = np.array([[0, 3], [2, 1], [3, 0]], np.int32)
    w = np.array([[0.75, 0.25], [0.5, 0.5], [0.125, 0.875]])
    y = oracle.forward_routed(shape, layer, x, idx, w, act="exact")
    for t in range(3):
        want = np.zeros(512)
        for k in range(2):
            e = idx[t, k]
            g, u = Wg[e] @ xf[t], Wu[e] @ xf[t]
            want += w[t, k] * (Wd[e] @ (g / (1 + np.exp(-g)) * u))
        assert np.allclose(y[t], want, rtol=1e-12, atol=1e-15)
    # quantised activations stay close to exact ones: Q8 within a few 1e-2, FP4 within 0.3
    y8 = oracle.forward_routed(shape, layer, x, idx, w, act="q8")
    y4 = oracle.forward_routed(shape, layer, x, idx, w, act="mx4")
    e8 = np.linalg.norm(y8 - y) / np.linalg.norm(y)
    e4 = np.linalg.norm(y4 - y) / np.linalg.norm(y)
    assert 0 < e8 < 3e-2 and e8 < e4 < 0.3, (e8, e4)


# ---- VQ routed experts -------------------------------------------------------
# "YoungAi - DeepSeek V4.1 Flash on one DGX Spark", section 4.1: every 8 weights
# of a row are one 12- or 13-bit index into a per-layer E4M3 codebook, times one
# binary16 gain per row; 13-bit layers keep a 12-bit stream plus a bit plane.

def _pack12(indices):
    """Index k at bits 12k .. 12k+11, least significant bit first."""
    bits = np.zeros(len(indices) * 12, np.uint8)
    for k, v in enumerate(indices):
        for i in range(12):
            bits[12 * k + i] = (v >> i) & 1
    return np.packbits(bits, bitorder="little")


def _plane(indices):
    return np.packbits(np.array([(v >> 12) & 1 for v in indices], np.uint8), bitorder="little")


def _e4m3_torch(b):
    import torch
    return torch.from_numpy(np.asarray(b, np.uint8)).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def test_e4m3_matches_torch_for_every_byte():
    want = _e4m3_torch(np.arange(256))
    got = np.array([oracle.e4m3(b) for b in range(256)])
    nan = np.isnan(want)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF] and np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert oracle.e4m3(0x7E) == 448.0 and oracle.e4m3(0x01) == 2.0 ** -9 and oracle.e4m3(0x38) == 1.0


def test_vq_index_stream_and_bit_plane():
    rng = np.random.default_rng(8)
    idx13 = rng.integers(0, 8192, 600)
    stream, plane = _pack12(idx13 & 4095), _plane(idx13)
    assert stream.size == 900  # 256 indices fill 384 bytes
    for k in (0, 1, 2, 255, 256, 257, 511, 599):
        assert oracle.vq_index(stream, None, k) == idx13[k] & 4095
        assert oracle.vq_index(stream, plane, k) == idx13[k]
    # index 256 starts at byte 384, bit 0
    one = _pack12([0] * 256 + [1])
    assert one[384] == 1 and oracle.vq_index(one, None, 256) == 1


def test_vq_row_is_gain_times_codewords():
    cb = np.zeros((4096, 8), np.uint8)
    cb[5] = [0x38, 0x40, 0x30, 0xB8, 0x00, 0x01, 0x7E, 0x44]  # 1, 2, 0.5, -1, 0, 2^-9, 448, 3
    cb[4095] = 0x3C  # 1.5
    idx = [5, 4095, 5, 0]
    gains = np.array([f16_bits(0.75), f16_bits(-2.0)], np.uint16)
    stream = _pack12([0] * 4 + idx)  # row 0: indices 0..3, row 1: the ones above
    w = oracle.dequant_vq_row(cb, stream, None, gains, 1, 32)
    c5 = [1, 2, 0.5, -1, 0, 2.0 ** -9, 448, 3]
    want = -2.0 * np.array(c5 + [1.5] * 8 + c5 + [0.0] * 8)
    assert np.array_equal(w, want)


def _vq_one_expert(H=256, I=256):
    """E=K=1 VQ layer: gate row i = a_i (codeword of ones times gain a_i), up
    row i = b_i, down row j = c_j * (+1 on the first I/2 columns, -1 after)."""
    cb = np.zeros((4096, 8), np.uint8)
    cb[1] = 0x38  # all 1.0
    cb[2] = 0xB8  # all -1.0
    a = np.array([2.0 ** -9 * (1 + i % 5) for i in range(I)])
    b = np.array([2.0 ** -8 * (1 + i % 3) for i in range(I)])
    c = np.array([2.0 ** -6 * (1 + j % 7) for j in range(H)])
    gate = _pack12([1] * (I * H // 8))
    down_idx = [1 if 8 * j < I // 2 else 2 for _ in range(H) for j in range(I // 8)]
    layer = {"routed_format": "vq", "vq_codebook": cb,
             "gate": gate[None], "gate_plane": None, "gate_rowgain": np.array([[f16_bits(v) for v in a]], np.uint16),
             "up": gate[None], "up_plane": None, "up_rowgain": np.array([[f16_bits(v) for v in b]], np.uint16),
             "down": _pack12(down_idx)[None], "down_plane": None,
             "down_rowgain": np.array([[f16_bits(v) for v in c]], np.uint16),
             "sh_gate": None, "sh_up": None, "sh_down": None}
    return layer, a, b, c


def test_vq_expert_closed_form():
    H, I = 256, 256
    layer, a, b, c = _vq_one_expert(H, I)
    x = np.where(np.arange(H) % 3 == 0, 1.0, -0.5).astype(np.float32)
    xs = float(x.astype(np.float64).sum())
    g, u = a * xs, b * xs
    h = g / (1 + np.exp(-g)) * u
    want = c * (h[:I // 2].sum() - h[I // 2:].sum())
    shape = synth.Shape(H, I, 1, 1, 0)
    y = oracle.forward_routed(shape, layer, bf16_bits(x[None, :]), np.zeros((1, 1), np.int32), np.ones((1, 1)))
    assert np.allclose(y[0], want, rtol=1e-12, atol=0)
    assert np.allclose(oracle.expert_vq(shape, layer, 0, x), want, rtol=1e-12, atol=0)


@pytest.mark.parametrize("bits", [12, 13])
def test_vq_layer_matches_dense_numpy(bits):
    shape = synth.Shape(512, 256, 3, 2, 0)
    layer = synth.make_layer(shape, 91, routed_format="vq", vq_bits=bits)
    layer["sh_gate"] = layer["sh_up"] = layer["sh_down"] = None
    cbv = _e4m3_torch(layer["vq_codebook"].reshape(-1)).reshape(-1, 8)

    def dense(name, rows, k):
        out = []
        for e in range(shape.n_experts):
            bits_ = np.unpackbits(layer[name][e], bitorder="little").reshape(-1, 12).astype(np.int64)
            idx = (bits_ << np.arange(12)).sum(axis=1)
            if bits == 13:
                idx |= np.unpackbits(layer[name + "_plane"][e], bitorder="little").astype(np.int64) << 12
            g = layer[name + "_rowgain"][e].view(np.float16).astype(np.float64)
            out.append(cbv[idx].reshape(rows, k) * g[:, None])
        return out
    Wg, Wu, Wd = dense("gate", 256, 512), dense("up", 256, 512), dense("down", 512, 256)
    x = synth.normal_bf16(2 * 512, 92, synth.S_X).reshape(2, 512)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    idx = np.array([[2, 0], [1, 2]], np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5]])
    y = oracle.forward_routed(shape, layer, x, idx, w)
    for t in range(2):
        want = np.zeros(512)
        for k in range(2):
            e = idx[t, k]
            gg, uu = Wg[e] @ xf[t], Wu[e] @ xf[t]
            want += w[t, k] * (Wd[e] @ (gg / (1 + np.exp(-gg)) * uu))
        assert np.allclose(y[t], want, rtol=1e-12, atol=1e-12 * np.abs(want).max())
