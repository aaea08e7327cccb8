"""Pins of the FP64 oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself through a re-typed copy of its
own loop: every check is a hand-worked case, a closed form, an invariant of
the delta rule, a special case that reduces to a library routine, or a brute
force comparison with the chunked rewrite.
"""
import json
import math
import os

import numpy as np
import pytest

import kda_inputs as KI
from oracle import chunked

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _rand_unit(rng, d):
    x = rng.standard_normal(d)
    return x / np.linalg.norm(x)


# ---------------- delta rule (kimi_k3.c header, "KDA per-head recurrence") ----------------

def test_delta_step_hand_worked(oracle_mod):
    for case in _load("delta_step_d2.json")["cases"]:
        S = np.array(case["S"], dtype=np.float64)
        o = oracle_mod.delta_step(S, case["alpha"], case["beta"], case["k"], case["v"], case["q"])
        np.testing.assert_allclose(S, case["S_new"], rtol=0, atol=1e-14, err_msg=case["name"])
        np.testing.assert_allclose(o, case["o"], rtol=0, atol=1e-14, err_msg=case["name"])


def test_delta_step_matches_literal_matrix_product(oracle_mod):
    """(I - b k k^T) @ diag(a) @ S + b k v^T and S'^T q, with numpy's matmul."""
    rng = np.random.default_rng(5)
    for d in (1, 3, 16, 128):
        S = rng.standard_normal((d, d))
        a = rng.uniform(math.exp(-5), 1, d)
        b = rng.uniform()
        k = _rand_unit(rng, d)
        v = rng.standard_normal(d)
        q = rng.standard_normal(d)
        ref = (np.eye(d) - b * np.outer(k, k)) @ np.diag(a) @ S + b * np.outer(k, v)
        S1 = S.copy()
        o = oracle_mod.delta_step(S1, a, b, k, v, q)
        np.testing.assert_allclose(S1, ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(o, ref.T @ q, rtol=1e-12, atol=1e-12)


def test_retrieval_invariant(oracle_mod):
    """alpha = 1, beta = 1, unit k: the updated state returns v for k (S'^T k = v)."""
    rng = np.random.default_rng(1)
    for d in (2, 7, 128):
        S = rng.standard_normal((d, d))
        k = _rand_unit(rng, d)
        v = rng.standard_normal(d)
        oracle_mod.delta_step(S, np.ones(d), 1.0, k, v, np.zeros(d))
        np.testing.assert_allclose(S.T @ k, v, rtol=0, atol=1e-12)


def test_beta_zero_is_pure_row_decay(oracle_mod):
    """beta = 0 leaves Diag(alpha) S: rows (key index) scale, columns do not."""
    rng = np.random.default_rng(2)
    d = 16
    S0 = rng.standard_normal((d, d))
    S = S0.copy()
    prod = np.ones(d)
    for _ in range(5):
        a = rng.uniform(math.exp(-5), 1, d)
        prod *= a
        oracle_mod.delta_step(S, a, 0.0, _rand_unit(rng, d), rng.standard_normal(d), np.zeros(d))
    np.testing.assert_allclose(S, prod[:, None] * S0, rtol=1e-13, atol=0)
    # a column scaling would differ on this non-symmetric state
    assert not np.allclose(S, S0 * prod[None, :])


def test_orthonormal_keys_all_retrieved(oracle_mod):
    rng = np.random.default_rng(3)
    d = 32
    Q, _ = np.linalg.qr(rng.standard_normal((d, d)))
    keys = Q.T  # rows orthonormal
    vals = rng.standard_normal((d, d))
    S = np.zeros((d, d))
    for i in range(d):
        oracle_mod.delta_step(S, np.ones(d), 1.0, keys[i], vals[i], np.zeros(d))
    for i in range(d):
        np.testing.assert_allclose(S.T @ keys[i], vals[i], atol=1e-12)


def test_repeated_key_latest_value_wins(oracle_mod):
    rng = np.random.default_rng(4)
    d = 12
    S = rng.standard_normal((d, d))
    k = _rand_unit(rng, d)
    v1, v2 = rng.standard_normal(d), rng.standard_normal(d)
    oracle_mod.delta_step(S, np.ones(d), 1.0, k, v1, np.zeros(d))
    oracle_mod.delta_step(S, np.ones(d), 1.0, k, v2, np.zeros(d))
    np.testing.assert_allclose(S.T @ k, v2, atol=1e-12)


def test_scalar_recurrence_d1(oracle_mod):
    """d = 1: s' = (1 - b k^2) a s + b k v, o = s' q."""
    rng = np.random.default_rng(6)
    s = 0.7
    S = np.array([[s]])
    for _ in range(20):
        a, b, k, v, q = rng.uniform(0.01, 1), rng.uniform(), rng.standard_normal(), rng.standard_normal(), rng.standard_normal()
        o = oracle_mod.delta_step(S, [a], b, [k], [v], [q])
        s = (1 - b * k * k) * a * s + b * k * v
        assert S[0, 0] == pytest.approx(s, rel=1e-13, abs=1e-15)
        assert o[0] == pytest.approx(s * q, rel=1e-13, abs=1e-15)


def test_frobenius_growth_bound(oracle_mod):
    """||(I - b k k^T) D S|| <= ||S|| for b in [0,1], |k| <= 1, 0 < alpha <= 1, so
    ||S_t||_F <= ||S_0||_F + sum_i b_i |k_i| |v_i|."""
    rng = np.random.default_rng(7)
    d = 24
    S = rng.standard_normal((d, d))
    bound = np.linalg.norm(S)
    for _ in range(200):
        k = _rand_unit(rng, d) * rng.uniform(0.5, 1.0)
        v = rng.standard_normal(d) * 3
        b = rng.uniform()
        oracle_mod.delta_step(S, rng.uniform(math.exp(-5), 1, d), b, k, v, np.zeros(d))
        bound += b * np.linalg.norm(k) * np.linalg.norm(v)
        assert np.linalg.norm(S) <= bound * (1 + 1e-12)


# ---------------- gates ----------------

def test_gate_closed_forms(oracle_mod):
    g = _load("gate_closed_forms.json")

    def val(x):
        if isinstance(x, (int, float)):
            return float(x)
        return {"ln2": math.log(2), "ln3/2": math.log(3) / 2, "-ln3/2": -math.log(3) / 2}[x]

    for c in g["cases"]:
        a, gk = oracle_mod.gate_alpha(val(c["A_log"]), val(c["z"]), val(c["dt"]), g["gmin"])
        assert gk == pytest.approx(c["gk"], abs=1e-14)
        assert a == pytest.approx(math.exp(c["gk"]), rel=1e-14)


def test_gate_range_and_monotone(oracle_mod):
    zs = np.linspace(-6, 6, 241)
    for A_log in (0.0, 1.0, math.log(16)):
        al = [oracle_mod.gate_alpha(A_log, z, 0.1, -5.0)[0] for z in zs]
        for z, a in zip(zs, al):
            arg = math.exp(A_log) * (z + 0.1)
            if abs(arg) < 30:   # open interval while the sigmoid is not rounded to 0 or 1
                assert math.exp(-5) < a < 1
            else:
                assert math.exp(-5) <= a <= 1
        # decreasing in z (strictly while unsaturated)
        assert all(x >= y for x, y in zip(al, al[1:]))
        assert all(x > y for z, x, y in zip(zs, al, al[1:]) if abs(math.exp(A_log) * (z + 0.1)) < 30)
    # saturation limits of the sigmoid (closed interval once it rounds)
    assert oracle_mod.gate_alpha(0.0, 1e4, 0.0, -5.0)[0] == pytest.approx(math.exp(-5), rel=1e-15)
    assert oracle_mod.gate_alpha(0.0, -1e4, 0.0, -5.0)[0] == 1.0


def test_sigmoid_silu_textbook(oracle_mod):
    assert oracle_mod.sigmoid(0.0) == 0.5
    assert oracle_mod.sigmoid(math.log(3)) == pytest.approx(0.75, rel=1e-15)
    assert oracle_mod.silu(0.0) == 0.0
    # silu(x) - silu(-x) = x
    for x in (0.3, 1.0, 4.5):
        assert oracle_mod.silu(x) - oracle_mod.silu(-x) == pytest.approx(x, rel=1e-14)


# ---------------- L2 norm and q scale ----------------

def test_l2norm_closed_form(oracle_mod):
    rng = np.random.default_rng(8)
    for scale in (1.0, 128 ** -0.5):
        for mag in (1e-4, 1e-2, 1.0, 30.0):
            x = rng.standard_normal(128) * mag
            s = float(np.dot(x, x))
            y = oracle_mod.l2norm(x, 1e-6, scale)
            # norm: scale * sqrt(s / (s + eps)); direction unchanged
            assert np.linalg.norm(y) == pytest.approx(scale * math.sqrt(s / (s + 1e-6)), rel=1e-13)
            np.testing.assert_allclose(y / np.linalg.norm(y), x / np.linalg.norm(x), atol=1e-14)
    # eps sits inside the sqrt: a zero vector stays zero (no division by zero)
    assert np.all(oracle_mod.l2norm(np.zeros(8), 1e-6, 1.0) == 0)


# ---------------- conv ----------------

def test_conv_impulse_response(oracle_mod):
    g = _load("conv_impulse.json")
    taps = g["taps"]
    hist = [0.0, 0.0, 0.0]
    for x, c in zip(g["x"], g["pre_silu"]):
        y = oracle_mod.conv_silu(taps, hist, x)
        assert y == pytest.approx(c / (1 + math.exp(-c)), rel=1e-15, abs=0)
        hist = hist[1:] + [x]


def _tiny_setup(H=2, d=8, K=4, T=12, seed=11, bf16=False):
    p = KI.make_params(H, d, K, seed)
    tok = KI.make_tokens(T, H, d, seed, bf16)
    return p, tok


def test_conv_causality(oracle_mod):
    cfg = oracle_mod.OracleCfg(H=2, d=8)
    p, tok = _tiny_setup()
    S, tail = oracle_mod.new_state(cfg)
    out = oracle_mod.sequence(cfg, p, S, tail, tok)
    tok2 = {k: v.copy() for k, v in tok.items()}
    for n in ("q", "k", "v", "z", "g"):
        tok2[n][7:] += 3.0
    tok2["b"][7:] -= 1.0
    S2, tail2 = oracle_mod.new_state(cfg)
    out2 = oracle_mod.sequence(cfg, p, S2, tail2, tok2)
    assert np.array_equal(out[:7], out2[:7])
    assert not np.allclose(out[7:], out2[7:])


def test_split_invariance_and_tail_carry(oracle_mod):
    """Running [0,n) then [n,T) equals [0,T) bit for bit: the conv history and S carry."""
    cfg = oracle_mod.OracleCfg(H=2, d=8)
    p, tok = _tiny_setup(T=20)
    S, tail = oracle_mod.new_state(cfg)
    full = oracle_mod.sequence(cfg, p, S, tail, tok)
    for n in (1, 2, 3, 5, 19):
        S2, tail2 = oracle_mod.new_state(cfg)
        a = oracle_mod.sequence(cfg, p, S2, tail2, {k: v[:n] for k, v in tok.items()})
        b = oracle_mod.sequence(cfg, p, S2, tail2, {k: v[n:] for k, v in tok.items()})
        assert np.array_equal(np.concatenate([a, b]), full)
        assert np.array_equal(S2, S) and np.array_equal(tail2, tail)
    # the history holds the last K-1 raw inputs, oldest first
    for x, n in enumerate(("q", "k", "v")):
        assert np.array_equal(tail[x], tok[n][-3:].astype(np.float64))


# ---------------- whole pipeline closed form ----------------

def test_single_token_from_zero_state(oracle_mod):
    """From S = 0 and a zero conv history, one token gives o = beta (k.q) v, where
    q, k, v are SiLU(last tap * x), q,k L2-normalised and q scaled; then
    out = sigmoid(g) * w * o / rms(o). A readout taken before the update would give 0."""
    H, d = 3, 16
    cfg = oracle_mod.OracleCfg(H=H, d=d)
    p, tok = _tiny_setup(H=H, d=d, T=1, seed=12)
    S, tail = oracle_mod.new_state(cfg)
    out = oracle_mod.sequence(cfg, p, S, tail, tok)
    silu = lambda x: x / (1 + np.exp(-x))
    for h in range(H):
        sl = slice(h * d, (h + 1) * d)
        x = {n: silu(p.conv_w[i, sl, 3].astype(np.float64) * tok[n][0, sl]) for i, n in enumerate("qkv")}
        qh = x["q"] / np.sqrt(np.sum(x["q"] ** 2) + 1e-6) * d ** -0.5
        kh = x["k"] / np.sqrt(np.sum(x["k"] ** 2) + 1e-6)
        beta = 1 / (1 + np.exp(-float(tok["b"][0, h])))
        o = beta * np.dot(kh, qh) * x["v"]
        ref = (1 / (1 + np.exp(-tok["g"][0, sl].astype(np.float64)))) * p.norm_w * o / np.sqrt(np.mean(o ** 2) + 1e-6)
        np.testing.assert_allclose(out[0, sl], ref, rtol=1e-12, atol=1e-14)
        # the state is the rank-one beta k v^T
        np.testing.assert_allclose(S[h], beta * np.outer(kh, x["v"]), rtol=1e-12, atol=1e-15)


def test_rmsnorm_gate_textbook(oracle_mod):
    rng = np.random.default_rng(9)
    o = rng.standard_normal(128) * 3
    w = 1 + 0.3 * rng.standard_normal(128)
    g = rng.standard_normal(128)
    out = oracle_mod.rmsnorm_gate(o, w, g, 1e-6)
    rms = np.linalg.norm(o) / math.sqrt(128)
    ref = w * o / math.sqrt(rms ** 2 + 1e-6) / (1 + np.exp(-g))
    np.testing.assert_allclose(out, ref, rtol=1e-13)
    # scale invariance in o (up to eps)
    out2 = oracle_mod.rmsnorm_gate(o * 7.0, w, g, 1e-6)
    np.testing.assert_allclose(out2, out, rtol=1e-6)


# ---------------- chunked rewrite vs sequential recurrence ----------------

@pytest.mark.parametrize("d", [1, 2, 4, 8])
def test_chunked_equals_sequential(oracle_mod, d):
    rng = np.random.default_rng(100 + d)
    T = 40
    S0 = rng.standard_normal((d, d))
    k = np.stack([_rand_unit(rng, d) for _ in range(T)])
    q = rng.standard_normal((T, d)) * d ** -0.5
    v = rng.standard_normal((T, d))
    alpha = np.exp(-5 / (1 + np.exp(-rng.standard_normal((T, d)) * 3)))
    beta = rng.uniform(size=T)
    S = S0.copy()
    o_seq = np.stack([oracle_mod.delta_step(S, alpha[t], beta[t], k[t], v[t], q[t]) for t in range(T)])
    for C in (1, 2, 3, 4, 8, 16, 64):
        O, Sc = chunked.run_chunked(S0, q, k, v, alpha, beta, C)
        scale = max(1.0, np.abs(o_seq).max())
        assert np.abs(O - o_seq).max() <= 1e-12 * scale, C
        assert np.abs(Sc - S).max() <= 1e-12 * max(1.0, np.abs(S).max()), C


def test_chunked_full_head_strong_decay(oracle_mod):
    """d = 128, C = 64 with gates near the lower bound: the log decay spans ~-300 in a chunk."""
    rng = np.random.default_rng(21)
    d, T = 128, 70
    S0 = rng.standard_normal((d, d)) * 0.1
    k = np.stack([_rand_unit(rng, d) for _ in range(T)])
    q = rng.standard_normal((T, d)) * d ** -0.5
    v = rng.standard_normal((T, d))
    alpha = np.full((T, d), math.exp(-4.9))
    alpha[:, ::3] = 0.99
    beta = rng.uniform(size=T)
    S = S0.copy()
    o_seq = np.stack([oracle_mod.delta_step(S, alpha[t], beta[t], k[t], v[t], q[t]) for t in range(T)])
    O, Sc = chunked.run_chunked(S0, q, k, v, alpha, beta, 64)
    assert np.abs(O - o_seq).max() <= 1e-11 * np.abs(o_seq).max()
    assert np.abs(Sc - S).max() <= 1e-11 * np.abs(S).max()


# ---------------- state handling ----------------

def test_snapshot_restore_equivalence(oracle_mod):
    cfg = oracle_mod.OracleCfg(H=2, d=8)
    p, tok = _tiny_setup(T=16)
    S, tail = oracle_mod.new_state(cfg)
    oracle_mod.sequence(cfg, p, S, tail, {k: v[:9] for k, v in tok.items()})
    snapS, snapT = S.copy(), tail.copy()
    ref = oracle_mod.sequence(cfg, p, S, tail, {k: v[9:] for k, v in tok.items()})
    S2, tail2 = snapS.copy(), snapT.copy()
    again = oracle_mod.sequence(cfg, p, S2, tail2, {k: v[9:] for k, v in tok.items()})
    assert np.array_equal(ref, again) and np.array_equal(S, S2) and np.array_equal(tail, tail2)


def test_prefill_then_decode_equals_all_decode(oracle_mod):
    H, d = 2, 8
    cfg = oracle_mod.OracleCfg(H=H, d=d)
    p, tok = _tiny_setup(T=10)
    S, tail = oracle_mod.new_state(cfg)
    ref = oracle_mod.sequence(cfg, p, S, tail, tok)
    S_all, tail_all = oracle_mod.new_state(cfg, 3)
    slots = [2]
    oracle_mod.sequence(cfg, p, S_all[2], tail_all[2], {k: v[:4] for k, v in tok.items()})
    outs = [oracle_mod.decode_batch(cfg, p, S_all, tail_all, slots, {k: v[t:t + 1] for k, v in tok.items()})
            for t in range(4, 10)]
    got = np.concatenate(outs)
    assert np.array_equal(got, ref[4:])
    assert np.array_equal(S_all[2], S) and np.all(S_all[0] == 0) and np.all(S_all[1] == 0)


def test_decode_batch_rows_independent(oracle_mod):
    """A batch of sequences equals each sequence run alone (rows map to their slots)."""
    H, d, B = 2, 8, 4
    cfg = oracle_mod.OracleCfg(H=H, d=d)
    p = KI.make_params(H, d, 4, 13)
    tok = KI.make_tokens(B, H, d, 13, False)
    S_all = np.random.default_rng(0).standard_normal((5, H, d, d)) * 0.1
    tail_all = np.random.default_rng(1).standard_normal((5, 3, 3, H * d))
    slots = np.array([3, 0, 4, 1], dtype=np.int32)
    S_ref, t_ref = S_all.copy(), tail_all.copy()
    out = oracle_mod.decode_batch(cfg, p, S_all, tail_all, slots, tok)
    for r, s in enumerate(slots):
        Ss, ts = S_ref[s].copy(), t_ref[s].copy()
        o = oracle_mod.sequence(cfg, p, Ss, ts, {k: v[r:r + 1] for k, v in tok.items()})
        assert np.array_equal(o[0], out[r])
        assert np.array_equal(Ss, S_all[s])
    assert np.array_equal(S_all[2], S_ref[2])


def test_unit_equals_sequence_head(oracle_mod):
    H, d = 3, 8
    cfg = oracle_mod.OracleCfg(H=H, d=d)
    p, tok = _tiny_setup(H=H, d=d, T=6)
    S, tail = oracle_mod.new_state(cfg)
    out = oracle_mod.sequence(cfg, p, S, tail, tok)
    for h in range(H):
        S_h = np.zeros((d, d))
        tl = np.zeros((3, 3, H * d))
        o = oracle_mod.unit(cfg, h, p, S_h, tl, tok)
        assert np.array_equal(o, out[:, h * d:(h + 1) * d])
        assert np.array_equal(S_h, S[h])


def test_bf16_round_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-3], dtype=np.float32)
    y = KI.bf16_round(x)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even mantissa (1.0)
    assert y[0] == 1.0 and y[1] == 1.0 and y[2] == np.float32(1.015625)
    assert y[3] == -2.5
    assert np.all(np.abs(y - x) <= np.abs(x) * 2.0 ** -8)
    assert np.array_equal(KI.from_bf16_bits(KI.to_bf16_bits(y)), y)


# ---------------- per-head gate wiring through the whole pipeline ----------------

def test_gate_wiring_per_head_and_channel(oracle_mod):
    """Three tokens from a zero state and history, H = 3 heads whose A_log differ and whose
    dt_bias differ per channel. The expected values are the page's formula written with numpy
    matrix products: x_t = SiLU(sum of taps over the raw inputs seen so far), the gate
    alpha_t[c] = exp(-5 sigmoid(exp(A_log[h]) (z_t[c] + dt_bias[h d + c]))), and
    S_t = (I - b_t k_t k_t^T) Diag(alpha_t) S_{t-1} + b_t k_t v_t^T, o_t = S_t^T q_t.
    From the second token on the decay of S_1 enters o and S, so using another head's
    A_log, another head's dt_bias or another token's z changes the result
    (kimi_k3.c header comment, block "KDA per-head recurrence")."""
    H, d, T = 3, 16, 3
    cfg = oracle_mod.OracleCfg(H=H, d=d)
    p = KI.make_params(H, d, 4, seed=14)
    p.A_log[:] = np.array([0.05, 1.3, 2.6], dtype=np.float32)   # distinct per head
    tok = KI.make_tokens(T, H, d, 14, False)
    S, tail = oracle_mod.new_state(cfg)
    out = oracle_mod.sequence(cfg, p, S, tail, tok)

    sig = lambda x: 1.0 / (1.0 + np.exp(-x))
    for h in range(H):
        sl = slice(h * d, (h + 1) * d)
        W = p.conv_w[:, sl, :].astype(np.float64)            # [3, d, 4], oldest tap first
        raw = {n: tok[n][:, sl].astype(np.float64) for n in "qkv"}
        St = np.zeros((d, d))
        for t in range(T):
            feat = {}
            for i, n in enumerate("qkv"):
                window = np.zeros((4, d))                       # rows: x_{t-3} .. x_t
                for j in range(4):
                    s = t - 3 + j
                    if s >= 0:
                        window[j] = raw[n][s]
                pre = np.einsum("cj,jc->c", W[i], window)
                feat[n] = pre * sig(pre)
            qh = feat["q"] / np.sqrt(feat["q"] @ feat["q"] + 1e-6) * d ** -0.5
            kh = feat["k"] / np.sqrt(feat["k"] @ feat["k"] + 1e-6)
            arg = np.exp(float(p.A_log[h])) * (tok["z"][t, sl].astype(np.float64)
                                               + p.dt_bias[sl].astype(np.float64))
            alpha = np.exp(-5.0 * sig(arg))
            beta = sig(float(tok["b"][t, h]))
            St = (np.eye(d) - beta * np.outer(kh, kh)) @ np.diag(alpha) @ St + beta * np.outer(kh, feat["v"])
            o = St.T @ qh
            ref = sig(tok["g"][t, sl].astype(np.float64)) * p.norm_w * o / np.sqrt(np.mean(o * o) + 1e-6)
            np.testing.assert_allclose(out[t, sl], ref, rtol=1e-11, atol=1e-13, err_msg=f"h={h} t={t}")
        np.testing.assert_allclose(S[h], St, rtol=1e-11, atol=1e-14, err_msg=f"state h={h}")
    # the decay really acts here: with alpha = 1 forced the last state would differ
    assert np.abs(S[1]).max() > 0
