"""Helpers shared by the GPU parity tests: upload, tolerances, comparisons."""
import numpy as np
import torch

# Tolerances of the layer output against the binary64 oracle, as relative L2
# error over the whole [T, H] output: fp32-accumulate decode path, and bf16
# tensor-core prefill path.
TOL_DECODE = 2e-3
TOL_PREFILL = 1e-2
# Routing weights: absolute difference of the fp32 renormalised sigmoid scores.
TOL_WEIGHTS = 1e-6
# Tokens whose oracle gap between the K-th and (K+1)-th fp32 selection score is
# below this are near-ties: their expert set may legitimately differ.
NEAR_TIE = 1e-5


def to_dev(layer: dict, dev="cuda") -> dict:
    """The layer's arrays as device tensors (other entries, e.g. "routed_format", are left out)."""
    return {k: (None if v is None else torch.from_numpy(np.ascontiguousarray(v)).to(dev)) for k, v in layer.items()
            if v is None or isinstance(v, np.ndarray)}


def x_to_dev(x: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev)


def rel_l2(y: np.ndarray, ref: np.ndarray) -> float:
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(y - ref) / np.linalg.norm(ref))


def rel_l2_rows(y: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Relative L2 error of each token (row) of a [T, H] output."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.linalg.norm(y - ref, axis=1) / np.linalg.norm(ref, axis=1)


def assert_close(y: np.ndarray, ref: np.ndarray, tol: float):
    """The output within tol of the oracle's, as relative L2 over the whole
    [T, H] array and over every token on its own (a wrong token cannot hide
    behind many right ones). Returns (whole-array error, worst token error)."""
    whole = rel_l2(y, ref)
    rows = rel_l2_rows(np.atleast_2d(y), np.atleast_2d(ref))
    worst = int(np.argmax(rows))
    assert whole <= tol, f"relative L2 {whole:.3e} above {tol:.0e}"
    assert rows[worst] <= tol, f"token {worst}: relative L2 {rows[worst]:.3e} above {tol:.0e}"
    return whole, float(rows[worst])


def check_routing(idx, w, gap, ref: dict, K: int):
    """idx/w/gap from the GPU vs the oracle's routing dict.

    Exact expert indices (in order) on every token that is not a near-tie;
    weights within TOL_WEIGHTS where the indices agree. Returns the boolean mask
    of near-tie tokens (their routing truth is the oracle's order).
    """
    idx = np.asarray(idx)
    w = np.asarray(w, dtype=np.float64)
    near = ref["gap"] < NEAR_TIE
    same = (idx == ref["idx"]).all(axis=1)
    bad = ~same & ~near
    assert not bad.any(), f"routing differs on {bad.sum()} tokens that are not near-ties: {np.nonzero(bad)[0][:10]}"
    if same.any():
        err = np.abs(w[same] - ref["weights"][same]).max()
        assert err <= TOL_WEIGHTS, f"routing weight error {err:.3e}"
    if gap is not None:
        g = np.asarray(gap, dtype=np.float64)
        fin = np.isfinite(ref["gap"]) & same
        assert np.allclose(g[fin], ref["gap"][fin], rtol=0, atol=2e-6)
    return near
