"""Prefill parity: kda_prefill (chunked WY/UT form) through the C ABI against the
sequential FP64 oracle, including ragged chunk tails, varlen batches, carried
state and conv history, and the prefill/decode/snapshot equivalences."""
import numpy as np
import pytest
import torch

import kda_inputs as KI
import linear_attention_mixer_gb300 as K
from tests.kda_testutil import (TOL_BF16, TOL_F32, dev_params, dev_tokens, download_state, rel_err, to_np,
                                upload_state)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_attention_mixer_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _prefill(cfg, params, st, slots_np, lens, tok, bf16):
    cu_h = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu_h[-1])
    t = dev_tokens(tok, bf16, rows=slice(0, T))
    out = torch.empty(T, cfg.num_heads * cfg.head_dim, device="cuda", dtype=t["q"].dtype)
    K.kda_prefill(cfg, params, st, torch.tensor(slots_np, dtype=torch.int32, device="cuda"),
                  torch.tensor(cu_h, device="cuda"), cu_h, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], out)
    return to_np(out), cu_h


def test_tiny_fp32_prefill_then_decode(oracle_mod):
    """Tiny config (H=2, T=64, FP32): GPU prefill of 32 tokens then 32 GPU decode steps
    equals the all-sequential oracle."""
    c = KI.CONFIGS["tiny"]
    H, d, T, Tp = c["H"], c["d"], c["T"], c["T_prefill"]
    p = KI.make_params(H, d, 4, c["seed"])
    tok = KI.make_tokens(T, H, d, c["seed"], bf16=False)
    cfg = K.kda_config(H, d, K.KDA_F32)
    params = dev_params(p)
    st = K.kda_state_alloc(cfg, 1)
    try:
        pre, _ = _prefill(cfg, params, st, [0], [Tp], tok, False)
        slots = torch.tensor([0], dtype=torch.int32, device="cuda")
        dec = []
        for s in range(Tp, T):
            t = dev_tokens(tok, False, rows=slice(s, s + 1))
            o = torch.empty(1, H * d, device="cuda")
            K.kda_decode_token(cfg, params, st, slots, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], o)
            dec.append(to_np(o))
        Sg, tg = download_state(cfg, st, [0])
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    oc = oracle_mod.OracleCfg(H=H, d=d)
    S, tail = oracle_mod.new_state(oc)
    ref = oracle_mod.sequence(oc, p, S, tail, tok)
    got = np.concatenate([pre] + dec)
    print(f"tiny fp32 prefill+decode: prefill {rel_err(got[:Tp], ref[:Tp]):.2e} all {rel_err(got, ref):.2e} "
          f"state {rel_err(Sg[0], S):.2e}")
    assert rel_err(got[:Tp], ref[:Tp]) <= TOL_F32
    assert rel_err(got, ref) <= TOL_F32
    assert rel_err(Sg[0], S) <= TOL_F32
    assert np.array_equal(tg[0], tail.astype(np.float32))


@pytest.mark.parametrize("bf16", [False, True])
def test_varlen_ragged_chunks_with_carried_state(oracle_mod, bf16):
    """Lengths hit every chunk-boundary case (1, 2, 3, 63, 64, 65, ...), an empty
    sequence sits in the middle, and every slot starts from a filled state and history."""
    H, d = 3, 128
    lens = [1, 2, 3, 5, 0, 63, 64, 65, 127, 130, 200]
    N = len(lens)
    T = sum(lens)
    p = KI.make_params(H, d, 4, 31)
    tok = KI.make_tokens(T, H, d, 31, bf16=bf16)
    n_slots = N + 2
    S0 = KI.make_state(n_slots, H, d, 31, std=0.05)
    T0 = KI.make_tail(n_slots, H, d, 4, 31, bf16=bf16)
    slots = np.random.default_rng(31).permutation(n_slots)[:N].astype(np.int32)
    cfg = K.kda_config(H, d, K.KDA_BF16 if bf16 else K.KDA_F32)
    st = K.kda_state_alloc(cfg, n_slots)
    try:
        upload_state(cfg, st, list(range(n_slots)), S0, T0)
        got, cu = _prefill(cfg, dev_params(p), st, slots, lens, tok, bf16)
        Sg, tg = download_state(cfg, st, list(range(n_slots)))
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    oc = oracle_mod.OracleCfg(H=H, d=d)
    tol = TOL_BF16 if bf16 else TOL_F32
    worst_o, worst_s = 0.0, 0.0
    for i in range(N):
        s = slots[i]
        S = S0[s].astype(np.float64)
        tail = T0[s].astype(np.float64)
        rows = slice(cu[i], cu[i + 1])
        ref = oracle_mod.sequence(oc, p, S, tail, {n: a[rows] for n, a in tok.items()})
        if lens[i]:
            worst_o = max(worst_o, rel_err(got[rows], ref))
            assert rel_err(got[rows], ref) <= tol, (i, lens[i])
        worst_s = max(worst_s, rel_err(Sg[s], S))
        assert rel_err(Sg[s], S) <= tol, (i, lens[i])
        assert np.array_equal(tg[s], tail.astype(np.float32)), (i, lens[i])
    print(f"varlen ragged {'bf16' if bf16 else 'fp32'}: worst out {worst_o:.2e} worst state {worst_s:.2e}")
    for s in set(range(n_slots)) - set(slots.tolist()):
        assert np.array_equal(Sg[s], S0[s]) and np.array_equal(tg[s], T0[s])


def test_prefill_split_and_decode_equivalence():
    """GPU only: prefill [0,T) equals prefill [0,n) + prefill [n,T) and equals
    prefill [0,n) + decode of every later token (within the FP32 tolerance)."""
    H, d, T, n = 2, 128, 150, 70
    p = KI.make_params(H, d, 4, 41)
    tok = KI.make_tokens(T, H, d, 41, bf16=False)
    cfg = K.kda_config(H, d, K.KDA_F32)
    params = dev_params(p)
    st = K.kda_state_alloc(cfg, 3)
    try:
        full, _ = _prefill(cfg, params, st, [0], [T], tok, False)
        a, _ = _prefill(cfg, params, st, [1], [n], tok, False)
        b, _ = _prefill(cfg, params, st, [1], [T - n], {k: v[n:] for k, v in tok.items()}, False)
        _prefill(cfg, params, st, [2], [n], tok, False)
        slots = torch.tensor([2], dtype=torch.int32, device="cuda")
        dec = []
        for s in range(n, T):
            t = dev_tokens(tok, False, rows=slice(s, s + 1))
            o = torch.empty(1, H * d, device="cuda")
            K.kda_decode_token(cfg, params, st, slots, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], o)
            dec.append(to_np(o))
        S, tl = download_state(cfg, st, [0, 1, 2])
    finally:
        K.kda_state_free(st)
    assert rel_err(np.concatenate([a, b]), full) <= TOL_F32
    assert rel_err(np.concatenate(dec), full[n:]) <= TOL_F32
    assert rel_err(S[1], S[0]) <= TOL_F32 and rel_err(S[2], S[0]) <= TOL_F32
    assert np.array_equal(tl[1], tl[0]) and np.array_equal(tl[2], tl[0])


def test_snapshot_restore_bit_exact():
    """Restoring a snapshot and replaying the same decode steps reproduces every bit."""
    H, d = 4, 128
    p = KI.make_params(H, d, 4, 51)
    tok = KI.make_tokens(100, H, d, 51, bf16=True)
    cfg = K.kda_config(H, d, K.KDA_BF16)
    params = dev_params(p)
    st = K.kda_state_alloc(cfg, 4)
    try:
        _prefill(cfg, params, st, [1, 3], [40, 50], tok, True)
        for on_dev in (False, True):
            blob = torch.empty(K.kda_state_blob_bytes(st, 2), dtype=torch.uint8,
                               device="cuda" if on_dev else "cpu")
            K.kda_state_snapshot(st, [1, 3], blob)
            torch.cuda.synchronize()
            slots = torch.tensor([3, 1], dtype=torch.int32, device="cuda")

            def run():
                outs = []
                for s in range(3):
                    t = dev_tokens(tok, True, rows=slice(90 + 2 * s, 92 + 2 * s))
                    o = torch.empty(2, H * d, device="cuda", dtype=torch.bfloat16)
                    K.kda_decode_token(cfg, params, st, slots, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], o)
                    outs.append(o.clone())
                return torch.stack(outs)

            first = run()
            after_first = download_state(cfg, st, [1, 3])
            K.kda_state_reset(st, [1, 3])
            K.kda_state_restore(st, [1, 3], blob)
            second = run()
            after_second = download_state(cfg, st, [1, 3])
            assert torch.equal(first, second)
            assert np.array_equal(after_first[0], after_second[0]) and np.array_equal(after_first[1], after_second[1])
            K.kda_state_restore(st, [1, 3], blob)
    finally:
        K.kda_state_free(st)


def test_prefill_8192_bf16_full_size(oracle_mod):
    """1 sequence, T=8192, 96 heads x 128, BF16 inputs, chunk 64: outputs of the first
    1024 tokens and the final state against the sequential oracle (which runs all 8192)."""
    c = KI.CONFIGS["prefill_8192"]
    H, d, T, nchk = c["H"], c["d"], c["T"], c["check_tokens"]
    p = KI.make_params(H, d, 4, c["seed"])
    tok = KI.make_tokens(T, H, d, c["seed"], bf16=True)
    cfg = K.kda_config(H, d, K.KDA_BF16)
    st = K.kda_state_alloc(cfg, 1)
    try:
        got, _ = _prefill(cfg, dev_params(p), st, [0], [T], tok, True)
        Sg, tg = download_state(cfg, st, [0])
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    oc = oracle_mod.OracleCfg(H=H, d=d)
    S, tail = oracle_mod.new_state(oc)
    ref = oracle_mod.sequence(oc, p, S, tail, tok)
    print(f"prefill T=8192 bf16: first {nchk} tokens {rel_err(got[:nchk], ref[:nchk]):.2e} "
          f"all tokens {rel_err(got, ref):.2e} final state {rel_err(Sg[0], S):.2e}")
    assert rel_err(got[:nchk], ref[:nchk]) <= TOL_BF16
    assert rel_err(Sg[0], S) <= TOL_BF16
    assert np.array_equal(tg[0], tail.astype(np.float32))
    assert np.isfinite(got).all()


def test_prefill_is_bit_reproducible():
    """The same prefill, repeated into fresh slots, gives bit-identical outputs, states and
    conv histories (every reduction on the path runs in a fixed order)."""
    H, d = 8, 128
    p = KI.make_params(H, d, 4, 29)
    tok = KI.make_tokens(700, H, d, 29, bf16=True)
    cfg = K.kda_config(H, d, K.KDA_BF16)
    params = dev_params(p)
    st = K.kda_state_alloc(cfg, 4)
    try:
        runs = []
        for s in range(4):
            out, _ = _prefill(cfg, params, st, [s], [700], tok, True)
            S, t = download_state(cfg, st, [s])
            runs.append((out, S, t))
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    for out, S, t in runs[1:]:
        assert np.array_equal(out, runs[0][0]) and np.array_equal(S, runs[0][1]) and np.array_equal(t, runs[0][2])
