"""Pins of the gate/beta projection oracle (oracle/gate_proj.py) against values worked by
hand from the pages' formula, brute-force loops, and algebraic properties. Each planted
mistake (a transposed weight, the products in the other order, W_b applied to f) fails."""
import json
import os

import numpy as np
import pytest

from oracle.gate_proj import gate_proj

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "gate_proj_small.json")


def _cases():
    return json.load(open(GOLDEN))["cases"]


def test_hand_worked_values():
    for c in _cases():
        z, b = gate_proj(np.array(c["x"]), np.array(c["fa"]), np.array(c["fb"]), np.array(c["bp"]))
        assert np.array_equal(z, np.array(c["z"], dtype=np.float64)), c["note"]
        assert np.array_equal(b, np.array(c["b"], dtype=np.float64)), c["note"]


def test_brute_force_loops():
    rng = np.random.default_rng(3)
    T, hidden, hd, proj, heads = 3, 7, 4, 5, 2
    x, fa = rng.standard_normal((T, hidden)), rng.standard_normal((hd, hidden))
    fb, bp = rng.standard_normal((proj, hd)), rng.standard_normal((heads, hidden))
    z, b = gate_proj(x, fa, fb, bp)
    for t in range(T):
        f = [sum(fa[j][i] * x[t][i] for i in range(hidden)) for j in range(hd)]
        for c in range(proj):
            assert abs(z[t][c] - sum(fb[c][j] * f[j] for j in range(hd))) < 1e-12
        for h in range(heads):
            assert abs(b[t][h] - sum(bp[h][i] * x[t][i] for i in range(hidden))) < 1e-12


def test_low_rank_and_linearity():
    rng = np.random.default_rng(4)
    hidden, hd, proj, heads = 16, 4, 12, 3
    fa, fb, bp = rng.standard_normal((hd, hidden)), rng.standard_normal((proj, hd)), rng.standard_normal((heads, hidden))
    # x in the null space of W_fa: no decay-gate signal at all, whatever W_fb is
    _, _, vt = np.linalg.svd(fa)
    null = vt[hd:]
    z, b = gate_proj(null, fa, fb, bp)
    assert np.abs(z).max() < 1e-12 and np.abs(b).max() > 1e-3
    # z has rank <= hd over any batch of tokens
    z, _ = gate_proj(rng.standard_normal((40, hidden)), fa, fb, bp)
    assert np.linalg.matrix_rank(z, tol=1e-9) == hd
    # linear in x
    x1, x2 = rng.standard_normal((5, hidden)), rng.standard_normal((5, hidden))
    za, ba = gate_proj(2.0 * x1 - 3.0 * x2, fa, fb, bp)
    z1, b1 = gate_proj(x1, fa, fb, bp)
    z2, b2 = gate_proj(x2, fa, fb, bp)
    assert np.abs(za - (2 * z1 - 3 * z2)).max() < 1e-10 and np.abs(ba - (2 * b1 - 3 * b2)).max() < 1e-10


@pytest.mark.parametrize("mistake", ["fa_transposed", "fb_transposed", "order_swapped", "b_from_f"])
def test_planted_mistakes_fail_a_pin(mistake):
    def wrong(x, fa, fb, bp):
        x = np.asarray(x, dtype=np.float64)
        if mistake == "fa_transposed":
            return (x @ fa) @ fb.T, x @ bp.T
        if mistake == "fb_transposed":
            return (x @ fa.T) @ fb, x @ bp.T
        if mistake == "order_swapped":
            return (x @ fb.T) @ fa.T, x @ bp.T
        return (x @ fa.T) @ fb.T, (x @ fa.T) @ bp.T[: fa.shape[0]]

    c = _cases()[1]
    args = [np.array(c[n], dtype=np.float64) for n in ("x", "fa", "fb", "bp")]
    try:
        z, b = wrong(*args)
        caught = not (np.array_equal(z, np.array(c["z"], dtype=np.float64)) and
                      np.array_equal(b, np.array(c["b"], dtype=np.float64)))
    except ValueError:  # a shape mismatch catches it too
        caught = True
    assert caught
