"""Pins of the layer oracle (oracle/layer.py): the dense product against brute-force loops,
a whole layer's first token from a zero state against the page's formula written out with
numpy (so a swapped projection, a missing residual or W_o applied before the mixer fails),
and the prefill form against token-by-token decode steps."""
import math

import numpy as np

import kda_inputs as KI
from oracle import layer as OL


def test_linear_brute_force():
    rng = np.random.default_rng(5)
    M, N, K = 3, 4, 6
    x, w, r = rng.standard_normal((M, K)), rng.standard_normal((N, K)), rng.standard_normal((M, N))
    y = OL.linear(x, w, r)
    for m in range(M):
        for n in range(N):
            assert abs(y[m][n] - (sum(x[m][k] * w[n][k] for k in range(K)) + r[m][n])) < 1e-12
    assert np.allclose(OL.linear(x, w), y - r, rtol=0, atol=1e-12)


def test_layer_first_token_closed_form(oracle_mod):
    """hidden = D; W_q = I, W_k = 2I, W_v = 3I, W_g = -I, W_o = 5I (distinct, so a swap shows).
    From a zero state and history one token gives, per head (conv with only the newest tap):
    q = SiLU(w3q x), k = SiLU(w3k 2x), v = SiLU(w3v 3x), q^ k^ L2-normalised, q^ scaled,
    o = beta (k^.q^) v, mixed = sigmoid(-x) w_norm o / rms(o), x' = x + 5 mixed."""
    H, d = 2, 8
    D = H * d
    cfg = oracle_mod.OracleCfg(H=H, d=d)
    p = KI.make_params(H, d, 4, seed=17)
    rng = np.random.default_rng(17)
    x = rng.standard_normal((2, D))
    I = np.eye(D)
    w = {"w_qkvg": np.concatenate([I, 2 * I, 3 * I, -I]), "w_fa": rng.standard_normal((d, D)) / 4,
         "w_fb": rng.standard_normal((D, d)) / 3, "w_b": rng.standard_normal((H, D)) / 4, "w_o": 5 * I}
    S, tail = oracle_mod.new_state(cfg, 2)
    got = OL.layer_decode(cfg, p, w, S, tail, np.array([1, 0], dtype=np.int32), x)
    xf = x.astype(np.float32).astype(np.float64)  # the mixer takes float32 inputs
    sig = lambda t: 1.0 / (1.0 + np.exp(-t))
    b_all = (x @ w["w_b"].T).astype(np.float32).astype(np.float64)
    for r in range(2):
        mixed = np.zeros(D)
        for h in range(H):
            sl = slice(h * d, (h + 1) * d)
            feat = {}
            for i, (n, sc) in enumerate((("q", 1), ("k", 2), ("v", 3))):
                pre = p.conv_w[i, sl, 3].astype(np.float64) * (sc * xf[r, sl]).astype(np.float32)
                feat[n] = pre * sig(pre)
            qh = feat["q"] / math.sqrt(feat["q"] @ feat["q"] + 1e-6) * d ** -0.5
            kh = feat["k"] / math.sqrt(feat["k"] @ feat["k"] + 1e-6)
            o = sig(b_all[r, h]) * (kh @ qh) * feat["v"]
            g = (-xf[r, sl]).astype(np.float32).astype(np.float64)
            mixed[sl] = sig(g) * p.norm_w * o / math.sqrt(np.mean(o * o) + 1e-6)
        np.testing.assert_allclose(got[r], x[r] + 5 * mixed, rtol=1e-6, atol=1e-7)
    # the slots advanced: row 0 wrote slot 1, row 1 slot 0, both away from zero
    assert np.abs(S[0]).max() > 0 and np.abs(S[1]).max() > 0


def test_layer_prefill_equals_token_by_token_decode(oracle_mod):
    """The prefill form of the layer oracle over T tokens of two sequences equals T decode steps
    of the layer oracle (pinned above by its closed form) fed the same rows in order."""
    from oracle import layer as OL
    H, d, hidden = 2, 8, 24
    D = H * d
    rng = np.random.default_rng(5)
    p = KI.make_params(H, d, 4, 5)
    w = {"w_qkvg": rng.standard_normal((4 * D, hidden)) * 0.3, "w_fa": rng.standard_normal((d, hidden)) * 0.3,
         "w_fb": rng.standard_normal((D, d)) * 0.3, "w_b": rng.standard_normal((H, hidden)) * 0.3,
         "w_o": rng.standard_normal((hidden, D)) * 0.3}
    oc = oracle_mod.OracleCfg(H=H, d=d)
    lens = [5, 3]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = rng.standard_normal((cu[-1], hidden))
    slots = [1, 0]
    S0 = rng.standard_normal((2, H, d, d)) * 0.1
    T0 = rng.standard_normal((2, 3, 3, D))
    S_p, T_p = S0.copy(), T0.copy()
    got = OL.layer_prefill(oc, p, w, S_p, T_p, slots, cu, x)
    S_d, T_d = S0.copy(), T0.copy()
    ref = np.zeros_like(got)
    for i, slot in enumerate(slots):
        for t in range(cu[i], cu[i + 1]):
            ref[t] = OL.layer_decode(oc, p, w, S_d, T_d, np.array([slot]), x[t:t + 1])[0]
    assert np.abs(got - ref).max() <= 1e-9 * max(1.0, np.abs(ref).max())
    assert np.abs(S_p - S_d).max() <= 1e-9 * np.abs(S_d).max() and np.array_equal(T_p, T_d)

