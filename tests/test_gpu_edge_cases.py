"""Parity at the method's degenerate settings, through the C ABI, against the FP64 oracle.

Each regime drives one part of the recurrence to its limit (kimi_k3.c header comment,
block "KDA per-head recurrence"):
  lower_gate   every decay gate at its lower bound: A_log = ln 16 and z = +8, so
               gk = -5 and alpha = e^-5 on every channel; the log decay reaches -320
               within one 64-token chunk
  keep_all     alpha -> 1 and beta -> 1 (z = -30, b = +30) with strongly correlated
               keys, the worst-conditioned (I + A) for the chunk's triangular solve
  no_write     beta -> 0 (b = -30): the update is a pure per-row decay
  zero_qk      runs of all-zero q and k rows, so that the conv output is exactly zero
               and the L2 eps alone sets the norm (q, k = 0, o = 0, out = 0)
Every regime runs the prefill (two sequences of 137 and 70 tokens: full chunks and a
ragged tail), 4 single-token decode steps and one 8-token decode call, each from a
filled state and conv history, with FP32 and with BF16 I/O.
"""
import math

import numpy as np
import pytest
import torch

import kda_inputs as KI
import linear_attention_mixer_gb300 as K
from tests.kda_testutil import (TOL_BF16, TOL_F32, dev_params, dev_tokens, download_state, rel_err, to_np,
                                upload_state)

pytestmark = pytest.mark.gpu

REGIMES = ["lower_gate", "keep_all", "no_write", "zero_qk"]
H, d = 4, 128
LENS = [137, 70]
N_DEC, N_MULTI = 4, 8


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_attention_mixer_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _setup(regime, T, bf16, seed):
    """Parameters, tokens [T] and a filled state/history of 2 slots for one regime."""
    p = KI.make_params(H, d, 4, seed)
    tok = KI.make_tokens(T, H, d, seed, bf16=bf16)
    S0 = KI.make_state(2, H, d, seed, std=0.05)
    T0 = KI.make_tail(2, H, d, 4, seed, bf16=bf16)
    if regime == "lower_gate":
        p.A_log[:] = np.float32(math.log(16.0))
        tok["z"][:] = 8.0
    elif regime == "keep_all":
        tok["z"][:] = -30.0
        tok["b"][:] = 30.0
        rng = np.random.default_rng(seed)
        common = rng.standard_normal(H * d).astype(np.float32)
        k = common[None, :] + 0.05 * tok["k"]
        tok["k"] = KI.bf16_round(k) if bf16 else k.astype(np.float32)
    elif regime == "no_write":
        tok["b"][:] = -30.0
    elif regime == "zero_qk":
        # q and k histories are zero; in a prefill, rows 40..59 of q and k are zero too, so from
        # row 43 on the conv window holds only zeros
        T0[:, :2] = 0.0
        if T > 60:
            for n in ("q", "k"):
                tok[n][40:60] = 0.0
    return p, tok, S0, T0


def _oracle_rows(oracle_mod, p, S0, T0, tok, groups):
    """Run the oracle on each group (slot, token rows); returns outputs per group and final S, tail."""
    oc = oracle_mod.OracleCfg(H=H, d=d)
    outs, Ss, tails = [], [], []
    for slot, rows in groups:
        S = S0[slot].astype(np.float64)
        tail = T0[slot].astype(np.float64)
        outs.append(oracle_mod.sequence(oc, p, S, tail, {n: a[rows] for n, a in tok.items()}))
        Ss.append(S)
        tails.append(tail)
    return outs, Ss, tails


def _check(tag, got_outs, ref_outs, Sg, tg, Ss, tails, tol):
    for i, (g, r) in enumerate(zip(got_outs, ref_outs)):
        e = rel_err(g, r)
        print(f"{tag} seq {i}: out {e:.2e} state {rel_err(Sg[i], Ss[i]):.2e}")
        assert np.all(np.isfinite(g)), tag
        assert e <= tol, (tag, i, e)
        assert rel_err(Sg[i], Ss[i]) <= tol, (tag, i)
        assert np.array_equal(tg[i], tails[i].astype(np.float32)), (tag, i)


@pytest.mark.parametrize("bf16", [False, True], ids=["fp32", "bf16"])
@pytest.mark.parametrize("regime", REGIMES)
def test_prefill_edge_regime(oracle_mod, regime, bf16):
    T = sum(LENS)
    p, tok, S0, T0 = _setup(regime, T, bf16, seed=90 + REGIMES.index(regime))
    cfg = K.kda_config(H, d, K.KDA_BF16 if bf16 else K.KDA_F32)
    st = K.kda_state_alloc(cfg, 2)
    cu_h = np.array([0, LENS[0], T], dtype=np.int32)
    try:
        upload_state(cfg, st, [0, 1], S0, T0)
        t = dev_tokens(tok, bf16)
        out = torch.empty(T, H * d, device="cuda", dtype=t["q"].dtype)
        K.kda_prefill(cfg, dev_params(p), st, torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                      torch.tensor(cu_h, device="cuda"), cu_h, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], out)
        got = to_np(out)
        Sg, tg = download_state(cfg, st, [0, 1])
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    groups = [(0, slice(0, LENS[0])), (1, slice(LENS[0], T))]
    ref, Ss, tails = _oracle_rows(oracle_mod, p, S0, T0, tok, groups)
    _check(f"prefill {regime} {'bf16' if bf16 else 'fp32'}", [got[r] for _, r in groups], ref, Sg, tg, Ss, tails,
           TOL_BF16 if bf16 else TOL_F32)
    if regime == "zero_qk":   # exactly zero where the conv window saw only zero q and k rows
        assert np.all(got[43:60] == 0.0)


@pytest.mark.parametrize("bf16", [False, True], ids=["fp32", "bf16"])
@pytest.mark.parametrize("regime", REGIMES)
def test_decode_edge_regime(oracle_mod, regime, bf16):
    """4 kda_decode_token steps and one kda_decode_tokens call of 8 tokens, 2 sequences each."""
    B = 2
    T = B * (N_DEC + N_MULTI)
    p, tok, S0, T0 = _setup(regime, T, bf16, seed=110 + REGIMES.index(regime))
    cfg = K.kda_config(H, d, K.KDA_BF16 if bf16 else K.KDA_F32)
    params = dev_params(p)
    st = K.kda_state_alloc(cfg, B)
    D = H * d
    slots = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    # token s of row r: single steps at r + B*s (s < N_DEC); the 8-token call at B*N_DEC + r*N_MULTI + j
    single_rows = [np.arange(N_DEC) * B + r for r in range(B)]
    multi_rows = [B * N_DEC + r * N_MULTI + np.arange(N_MULTI) for r in range(B)]
    if regime == "zero_qk":   # row 0's tokens are all zero in q and k; row 1's are not
        for n in ("q", "k"):
            tok[n][np.concatenate([single_rows[0], multi_rows[0]])] = 0.0
    try:
        upload_state(cfg, st, [0, 1], S0, T0)
        dec = []
        for s in range(N_DEC):
            t = dev_tokens(tok, bf16, rows=slice(B * s, B * (s + 1)))
            o = torch.empty(B, D, device="cuda", dtype=t["q"].dtype)
            K.kda_decode_token(cfg, params, st, slots, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], o)
            dec.append(to_np(o))
        dec = np.stack(dec, axis=1)  # [B][N_DEC][D]
        t = dev_tokens(tok, bf16, rows=slice(B * N_DEC, T))
        o = torch.empty(B * N_MULTI, D, device="cuda", dtype=t["q"].dtype)
        K.kda_decode_tokens(cfg, params, st, slots, N_MULTI, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], o)
        multi = to_np(o).reshape(B, N_MULTI, D)
        Sg, tg = download_state(cfg, st, [0, 1])
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    groups = [(r, np.concatenate([single_rows[r], multi_rows[r]])) for r in range(B)]
    ref, Ss, tails = _oracle_rows(oracle_mod, p, S0, T0, tok, groups)
    got = [np.concatenate([dec[r], multi[r]]) for r in range(B)]
    _check(f"decode {regime} {'bf16' if bf16 else 'fp32'}", got, ref, Sg, tg, Ss, tails,
           TOL_BF16 if bf16 else TOL_F32)
    if regime == "zero_qk":   # row 0: zero q and k history and inputs, so every output is zero
        assert np.all(got[0] == 0.0) and np.abs(got[1]).max() > 0
