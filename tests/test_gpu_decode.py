"""Decode parity: kda_decode_token through the C ABI against the FP64 oracle."""
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


def _decode_steps(cfg, params, st, slots_np, tok, bf16, steps):
    slots = torch.tensor(slots_np, dtype=torch.int32, device="cuda")
    B = len(slots_np)
    D = cfg.num_heads * cfg.head_dim
    outs = []
    for s in range(steps):
        t = dev_tokens(tok, bf16, rows=slice(s * B, (s + 1) * B))
        out = torch.empty(B, D, device="cuda", dtype=t["q"].dtype)
        K.kda_decode_token(cfg, params, st, slots, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], out)
        outs.append(to_np(out))
    return np.stack(outs)


def test_tiny_fp32_decode_after_oracle_prefill(oracle_mod):
    """Tiny config: H=2, T=64 (32 prefill + 32 decode), FP32 throughout, zero start state.
    The first 32 tokens run in the oracle; its state (rounded to FP32) is uploaded and
    the GPU decodes the last 32; the oracle continues from the same rounded state."""
    c = KI.CONFIGS["tiny"]
    H, d, T, Tp = c["H"], c["d"], c["T"], c["T_prefill"]
    p = KI.make_params(H, d, 4, c["seed"])
    tok = KI.make_tokens(T, H, d, c["seed"], bf16=False)
    oc = oracle_mod.OracleCfg(H=H, d=d)
    S, tail = oracle_mod.new_state(oc)
    oracle_mod.sequence(oc, p, S, tail, {n: a[:Tp] for n, a in tok.items()})
    S32 = S.astype(np.float32)
    cfg = K.kda_config(H, d, K.KDA_F32)
    st = K.kda_state_alloc(cfg, 3)
    try:
        upload_state(cfg, st, [2], S32[None], tail[None])
        got = _decode_steps(cfg, dev_params(p), st, [2], {n: a[Tp:] for n, a in tok.items()}, False, T - Tp)
        Sg, tg = download_state(cfg, st, [2])
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    S_ref = S32.astype(np.float64)
    ref = oracle_mod.sequence(oc, p, S_ref, tail, {n: a[Tp:] for n, a in tok.items()})
    e_o, e_s = rel_err(got[:, 0], ref), rel_err(Sg[0], S_ref)
    print(f"tiny fp32 decode: out {e_o:.2e} state {e_s:.2e}")
    assert e_o <= TOL_F32
    assert e_s <= TOL_F32
    assert np.array_equal(tg[0], tail.astype(np.float32))  # history is raw inputs: exact


def test_decode_b1_bf16_prefilled_by_oracle(oracle_mod):
    """Batch 1, 96 heads x 128, state pre-filled by 256 oracle steps, BF16 inputs; 2 decode steps."""
    c = KI.CONFIGS["decode_b1"]
    H, d = c["H"], c["d"]
    npre = c["prefill_steps"]
    p = KI.make_params(H, d, 4, c["seed"])
    tok = KI.make_tokens(npre + 2, H, d, c["seed"], bf16=True)
    oc = oracle_mod.OracleCfg(H=H, d=d)
    S, tail = oracle_mod.new_state(oc)
    oracle_mod.sequence(oc, p, S, tail, {n: a[:npre] for n, a in tok.items()})
    S32 = S.astype(np.float32)
    cfg = K.kda_config(H, d, K.KDA_BF16)
    st = K.kda_state_alloc(cfg, 1)
    try:
        upload_state(cfg, st, [0], S32[None], tail[None])
        got = _decode_steps(cfg, dev_params(p), st, [0], {n: a[npre:] for n, a in tok.items()}, True, 2)
        Sg, tg = download_state(cfg, st, [0])
    finally:
        K.kda_state_free(st)
    S_ref = S32.astype(np.float64)
    ref = oracle_mod.sequence(oc, p, S_ref, tail, {n: a[npre:] for n, a in tok.items()})
    e_o, e_s = rel_err(got[:, 0], ref), rel_err(Sg[0], S_ref)
    print(f"decode B=1 bf16: out {e_o:.2e} state {e_s:.2e}")
    assert e_o <= TOL_BF16
    assert e_s <= TOL_F32  # the state itself stays FP32
    assert np.array_equal(tg[0], tail.astype(np.float32))


def test_decode_b256_full_size_sampled_units(oracle_mod):
    """Batch 256 independent sequences, 96 heads x 128, FP32 states (~1.6 GB) filled by the
    generator, BF16 inputs, 3 steps; slots are a permutation inside a larger state.
    Sampled (sequence, head) units are recomputed one by one by the oracle."""
    c = KI.CONFIGS["decode_b256"]
    H, d, B = c["H"], c["d"], c["B"]
    D = H * d
    n_slots = B + 16
    steps = 3
    rng = np.random.default_rng(c["seed"])
    slots = rng.permutation(n_slots)[:B].astype(np.int32)
    p = KI.make_params(H, d, 4, c["seed"])
    tok = KI.make_tokens(B * steps, H, d, c["seed"], bf16=True)
    S0 = KI.make_state(n_slots, H, d, c["seed"], std=0.05)
    T0 = KI.make_tail(n_slots, H, d, 4, c["seed"], bf16=True)
    cfg = K.kda_config(H, d, K.KDA_BF16)
    st = K.kda_state_alloc(cfg, n_slots)
    try:
        upload_state(cfg, st, list(range(n_slots)), S0, T0)
        got = _decode_steps(cfg, dev_params(p), st, slots, tok, True, steps)  # [steps, B, D]
        Sg, tg = download_state(cfg, st, list(range(n_slots)))
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    oc = oracle_mod.OracleCfg(H=H, d=d)
    units = [(int(r), int(h)) for r, h in zip(rng.integers(0, B, 40), rng.integers(0, H, 40))]
    units += [(0, h) for h in range(H)] + [(B - 1, h) for h in (0, H - 1)]
    errs, serrs = [], []
    for r, h in units:
        s = slots[r]
        S_h = S0[s, h].astype(np.float64)
        tl = T0[s].astype(np.float64)
        rows = [step * B + r for step in range(steps)]
        ref = oracle_mod.unit(oc, h, p, S_h, tl, tok, rows=rows)  # [steps, d]
        g = got[:, r, h * d:(h + 1) * d]
        errs.append(np.abs(g - ref).max() / max(np.abs(ref).max(), 1e-30))
        serrs.append(rel_err(Sg[s, h], S_h))
        assert np.array_equal(tg[s][:, :, h * d:(h + 1) * d], tl[:, :, h * d:(h + 1) * d].astype(np.float32))
    print(f"decode B=256 bf16 ({len(units)} sampled units): out {max(errs):.2e} state {max(serrs):.2e}")
    assert max(errs) <= TOL_BF16, max(errs)
    assert max(serrs) <= TOL_F32, max(serrs)
    # slots outside the batch are untouched
    untouched = sorted(set(range(n_slots)) - set(slots.tolist()))
    assert np.array_equal(Sg[untouched], S0[untouched])
    assert np.isfinite(got).all()


def test_decode_bad_slot_recorded_and_skipped():
    H, d = 2, 128
    cfg = K.kda_config(H, d, K.KDA_F32)
    p = KI.make_params(H, d, 4, 3)
    tok = KI.make_tokens(2, H, d, 3, bf16=False)
    st = K.kda_state_alloc(cfg, 2)
    try:
        slots = torch.tensor([1, 7], dtype=torch.int32, device="cuda")
        t = dev_tokens(tok, False)
        out = torch.zeros(2, H * d, device="cuda")
        K.kda_decode_token(cfg, dev_params(p), st, slots, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], out)
        assert K.kda_state_poll_error(st) == K.KDA_ERR_DEVICE
        assert K.kda_state_poll_error(st) == 0  # cleared by the read
        assert torch.all(out[1] == 0)          # the bad row was skipped
        assert torch.any(out[0] != 0)
    finally:
        K.kda_state_free(st)


def test_decode_argument_errors():
    import ctypes
    H, d = 2, 128
    cfg = K.kda_config(H, d, K.KDA_F32)
    p = dev_params(KI.make_params(H, d, 4, 3))
    st = K.kda_state_alloc(cfg, 2)
    try:
        t = dev_tokens(KI.make_tokens(1, H, d, 3, bf16=False), False)
        slots = torch.tensor([0], dtype=torch.int32, device="cuda")
        out = torch.empty(1, H * d, device="cuda")
        # a config that differs from the state's is rejected by the library itself
        other = K.kda_config(H, d, K.KDA_BF16)
        ptrs = [ctypes.c_void_p(x.data_ptr()) for x in (t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], out)]
        rc = K.lib().kda_decode_token(ctypes.byref(other), ctypes.byref(p), st, ctypes.c_void_p(slots.data_ptr()), 1,
                                      *ptrs, None)
        assert rc == K.KDA_ERR_INVALID and "config" in K.kda_last_error()
        # a tensor pointer that is not 16-byte aligned is rejected before anything is enqueued
        qbad = torch.empty(H * d + 4, device="cuda")[1:H * d + 1].view(1, H * d)
        bad = [ctypes.c_void_p(x.data_ptr()) for x in (qbad, t["k"], t["v"], t["z"], t["b"], t["g"], out)]
        rc = K.lib().kda_decode_token(ctypes.byref(cfg), ctypes.byref(p), st, ctypes.c_void_p(slots.data_ptr()), 1,
                                      *bad, None)
        assert rc == K.KDA_ERR_INVALID and "aligned" in K.kda_last_error()
        # the binding refuses tensors of the wrong dtype before calling in
        with pytest.raises(TypeError):
            K.kda_decode_token(other, p, st, slots, t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], out)
        # B == 0 is a no-op
        empty = torch.empty(0, dtype=torch.int32, device="cuda")
        e0 = torch.empty(0, H * d, device="cuda")
        K.kda_decode_token(cfg, p, st, empty, e0, e0, e0, e0, torch.empty(0, H, device="cuda"), e0, e0)
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
