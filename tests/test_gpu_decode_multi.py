"""kda_decode_tokens (n decode tokens per row in one pass over the state) through the C ABI:
against the FP64 oracle run token by token, against n calls of kda_decode_token, and the
snapshot/restore rollback a speculative verifier uses."""
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


def _run_multi(cfg, params, st, slots_np, tok, bf16, n):
    B = len(slots_np)
    D = cfg.num_heads * cfg.head_dim
    t = dev_tokens(tok, bf16)
    out = torch.empty(B * n, D, device="cuda", dtype=t["q"].dtype)
    K.kda_decode_tokens(cfg, params, st, torch.tensor(slots_np, dtype=torch.int32, device="cuda"), n,
                        t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], out)
    return to_np(out).reshape(B, n, D)


def _run_single(cfg, params, st, slots_np, tok, bf16, n):
    B = len(slots_np)
    D = cfg.num_heads * cfg.head_dim
    slots = torch.tensor(slots_np, dtype=torch.int32, device="cuda")
    outs = []
    for s in range(n):
        t = dev_tokens(tok, bf16, rows=np.arange(B) * n + s)
        out = torch.empty(B, D, device="cuda", dtype=t["q"].dtype)
        K.kda_decode_token(cfg, params, st, slots, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], out)
        outs.append(to_np(out))
    return np.stack(outs, axis=1)  # [B][n][D]


# every n has its own kernel (the token count is a template parameter): each one runs, in both
# I/O types, at small sizes, and the workload's geometry at n = 4 and 8
@pytest.mark.parametrize("bf16,H,B,n", [(False, 2, 3, n) for n in range(1, 9)] + [(True, 4, 3, n) for n in range(1, 9)]
                         + [(False, 2, 2, 5), (True, 96, 3, 4), (True, 96, 2, 8)])
def test_decode_tokens_matches_oracle_and_single_calls(oracle_mod, bf16, H, B, n):
    d, seed = 128, 70 + n + H
    p = KI.make_params(H, d, 4, seed)
    tok = KI.make_tokens(B * n, H, d, seed, bf16=bf16)  # row r, token t at r * n + t
    S0 = KI.make_state(B, H, d, seed)
    T0 = KI.make_tail(B, H, d, 4, seed, bf16=bf16)
    cfg = K.kda_config(H, d, K.KDA_BF16 if bf16 else K.KDA_F32)
    params = dev_params(p)
    st = K.kda_state_alloc(cfg, 2 * B)
    try:
        multi_slots, single_slots = list(range(B)), list(range(B, 2 * B))
        upload_state(cfg, st, multi_slots, S0, T0)
        upload_state(cfg, st, single_slots, S0, T0)
        got = _run_multi(cfg, params, st, multi_slots, tok, bf16, n)
        one = _run_single(cfg, params, st, single_slots, tok, bf16, n)
        Sm, tm = download_state(cfg, st, multi_slots)
        Ss, ts = download_state(cfg, st, single_slots)
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    # one pass over n tokens is n single-token steps: the same arithmetic per token, bit for bit
    d_out, d_s = rel_err(got, one), rel_err(Sm, Ss)
    assert np.array_equal(got, one) and np.array_equal(Sm, Ss)
    assert np.array_equal(tm, ts)
    oc = oracle_mod.OracleCfg(H=H, d=d)
    worst_o = worst_s = 0.0
    for r in range(B):
        S = S0[r].astype(np.float64)
        tail = T0[r].astype(np.float64)
        ref = oracle_mod.sequence(oc, p, S, tail, {m: a[r * n:(r + 1) * n] for m, a in tok.items()})
        worst_o = max(worst_o, rel_err(got[r], ref))
        worst_s = max(worst_s, rel_err(Sm[r], S))
        assert np.array_equal(tm[r], tail.astype(np.float32))
    tol = TOL_BF16 if bf16 else TOL_F32
    print(f"decode_tokens {'bf16' if bf16 else 'fp32'} H={H} B={B} n={n}: out {worst_o:.2e} state {worst_s:.2e}; "
          f"vs single-token calls out {d_out:.1e} state {d_s:.1e} ({'bit-exact' if d_out == 0 and d_s == 0 else 'close'})")
    assert worst_o <= tol and worst_s <= tol


def test_speculative_rollback_and_argument_errors():
    """Verify a draft of 6 tokens from a snapshot, reject after 3: restore the snapshot and
    run the accepted 3 again. The slot then equals one that only ever saw those 3 tokens
    (bit for bit). Bad slot ids are skipped and recorded; n outside [1, 8] is refused."""
    H, d, B, n, j = 4, 128, 2, 6, 3
    p = KI.make_params(H, d, 4, 91)
    tok = KI.make_tokens(B * n, H, d, 91, bf16=True)
    acc = {m: a.reshape(B, n, -1)[:, :j].reshape(B * j, -1) for m, a in tok.items()}  # accepted prefix
    S0 = KI.make_state(B, H, d, 91)
    T0 = KI.make_tail(B, H, d, 4, 91, bf16=True)
    cfg = K.kda_config(H, d, K.KDA_BF16)
    params = dev_params(p)
    st = K.kda_state_alloc(cfg, 2 * B)
    try:
        spec, ref = list(range(B)), list(range(B, 2 * B))
        upload_state(cfg, st, spec, S0, T0)
        upload_state(cfg, st, ref, S0, T0)
        snap = torch.empty(K.kda_state_blob_bytes(st, B), dtype=torch.uint8, device="cuda")
        K.kda_state_snapshot(st, spec, snap)
        _run_multi(cfg, params, st, spec, tok, True, n)  # the draft
        K.kda_state_restore(st, spec, snap)              # rejected after j tokens
        out_spec = _run_multi(cfg, params, st, spec, acc, True, j)
        out_ref = _run_multi(cfg, params, st, ref, acc, True, j)
        Sa, ta = download_state(cfg, st, spec)
        Sb, tb = download_state(cfg, st, ref)
        assert K.kda_state_poll_error(st) == 0
        assert np.array_equal(out_spec, out_ref)
        assert np.array_equal(Sa, Sb) and np.array_equal(ta, tb)

        # a bad slot id: the row is skipped, the others run, the error word records it
        t = dev_tokens(acc, True)
        out = torch.empty(B * j, H * d, device="cuda", dtype=torch.bfloat16)
        bad = torch.tensor([0, 7 * B], dtype=torch.int32, device="cuda")
        K.kda_decode_tokens(cfg, params, st, bad, j, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], out)
        assert K.kda_state_poll_error(st) == K.KDA_ERR_DEVICE
        import ctypes
        sl = torch.tensor(spec, dtype=torch.int32, device="cuda")
        ptrs = [ctypes.c_void_p(x.data_ptr()) for x in (t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], out)]
        for bad_n in (0, K.KDA_DECODE_MAX_TOKENS + 1):
            rc = K.lib().kda_decode_tokens(ctypes.byref(cfg), ctypes.byref(params), st, ctypes.c_void_p(sl.data_ptr()),
                                           B, bad_n, *ptrs, None)
            assert rc == K.KDA_ERR_INVALID and "n must be" in K.kda_last_error()
        assert K.kda_state_poll_error(st) == 0  # nothing was enqueued
    finally:
        K.kda_state_free(st)


def test_bad_slot_then_good_units_in_one_cta():
    """384 units (B = 4 at H = 96) give some CTAs two units, so a skipped unit (row 0, bad
    slot) is followed by a good one in the same CTA: rows 1..3 must equal a run without
    the bad row, bit for bit, and the error word records the bad id."""
    H, d, B, n = 96, 128, 4, 2
    p = KI.make_params(H, d, 4, 17)
    tok = KI.make_tokens(B * n, H, d, 17, bf16=True)
    S0 = KI.make_state(B, H, d, 17)
    T0 = KI.make_tail(B, H, d, 4, 17, bf16=True)
    cfg = K.kda_config(H, d, K.KDA_BF16)
    params = dev_params(p)
    st = K.kda_state_alloc(cfg, 2 * B)
    try:
        upload_state(cfg, st, list(range(B)), S0, T0)
        upload_state(cfg, st, list(range(B, 2 * B)), S0, T0)
        t = dev_tokens(tok, True)
        out_bad = torch.zeros(B * n, H * d, device="cuda", dtype=torch.bfloat16)
        slots_bad = torch.tensor([9 * B, 1, 2, 3], dtype=torch.int32, device="cuda")
        K.kda_decode_tokens(cfg, params, st, slots_bad, n, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], out_bad)
        assert K.kda_state_poll_error(st) == K.KDA_ERR_DEVICE
        out_ok = torch.zeros(B * n, H * d, device="cuda", dtype=torch.bfloat16)
        slots_ok = torch.tensor([B, B + 1, B + 2, B + 3], dtype=torch.int32, device="cuda")
        K.kda_decode_tokens(cfg, params, st, slots_ok, n, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], out_ok)
        assert K.kda_state_poll_error(st) == 0
        assert torch.equal(out_bad[n:], out_ok[n:])
        Sa, ta = download_state(cfg, st, [1, 2, 3])
        Sb, tb = download_state(cfg, st, [B + 1, B + 2, B + 3])
        assert np.array_equal(Sa, Sb) and np.array_equal(ta, tb)
    finally:
        K.kda_state_free(st)


def test_decode_tokens_b256_n8_full_size(oracle_mod):
    """The bench's workload: 256 sequences x 8 tokens in one call, 96 heads x 128, BF16 I/O, FP32
    states (~1.6 GB) from the generator, slots a permutation inside a larger state. All units are
    checked bit for bit against 8 single-token calls on a copy of the state; sampled (sequence,
    head) units against the oracle, one by one."""
    c = KI.CONFIGS["decode_b256"]
    H, d, B, n = c["H"], c["d"], c["B"], 8
    n_slots = 2 * B
    rng = np.random.default_rng(c["seed"] + 8)
    perm = rng.permutation(n_slots).astype(np.int32)
    multi_slots, single_slots = perm[:B], perm[B:]
    p = KI.make_params(H, d, 4, c["seed"])
    tok = KI.make_tokens(B * n, H, d, c["seed"] + 8, bf16=True)  # row r, token t at r * n + t
    S0 = KI.make_state(B, H, d, c["seed"], std=0.05)
    T0 = KI.make_tail(B, H, d, 4, c["seed"], bf16=True)
    cfg = K.kda_config(H, d, K.KDA_BF16)
    params = dev_params(p)
    st = K.kda_state_alloc(cfg, n_slots)
    try:
        upload_state(cfg, st, multi_slots.tolist(), S0, T0)
        upload_state(cfg, st, single_slots.tolist(), S0, T0)
        got = _run_multi(cfg, params, st, multi_slots.tolist(), tok, True, n)     # [B][n][D]
        one = _run_single(cfg, params, st, single_slots.tolist(), tok, True, n)
        Sm, tm = download_state(cfg, st, multi_slots.tolist())
        Ss, ts = download_state(cfg, st, single_slots.tolist())
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    assert np.array_equal(got, one) and np.array_equal(Sm, Ss) and np.array_equal(tm, ts)
    oc = oracle_mod.OracleCfg(H=H, d=d)
    units = [(int(r), int(h)) for r, h in zip(rng.integers(0, B, 24), rng.integers(0, H, 24))]
    units += [(0, 0), (B - 1, H - 1)]
    errs, serrs = [], []
    for r, h in units:
        S_h = S0[r, h].astype(np.float64)
        tl = T0[r].astype(np.float64)
        ref = oracle_mod.unit(oc, h, p, S_h, tl, tok, rows=list(range(r * n, (r + 1) * n)))  # [n, d]
        g = got[r][:, h * d:(h + 1) * d]
        errs.append(np.abs(g - ref).max() / max(np.abs(ref).max(), 1e-30))
        serrs.append(rel_err(Sm[r, h], S_h))
        assert np.array_equal(tm[r][:, :, h * d:(h + 1) * d], tl[:, :, h * d:(h + 1) * d].astype(np.float32))
    print(f"decode_tokens B=256 n=8 bf16 ({len(units)} sampled units): out {max(errs):.2e} state {max(serrs):.2e}; "
          f"all units bit-exact against single-token calls")
    assert max(errs) <= TOL_BF16 and max(serrs) <= TOL_F32
