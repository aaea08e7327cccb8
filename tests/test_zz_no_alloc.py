"""kda_prefill_noalloc: the prefill for callers that cannot allocate device memory
(runtimes that own every byte through their own arena, or loops that cannot take
the device synchronisation of cudaMalloc/cudaFree). It runs on caller-owned state
buffers with the library's static workspace.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test. It passes alone or after the others.
"""
import numpy as np
import pytest
import torch

import kda_inputs as KI
import linear_attention_mixer_gb300 as K
from tests.kda_testutil import TOL_BF16, TOL_F32, dev_params, dev_tokens, download_state, rel_err, to_np

pytestmark = pytest.mark.gpu


def _call_pair(lens_a, lens_b):
    cu_a = np.concatenate([[0], np.cumsum(lens_a)]).astype(np.int32)
    cu_b = np.concatenate([[0], np.cumsum(lens_b)]).astype(np.int32)
    return cu_a, cu_b


def test_noalloc_prefill_matches_kda_prefill_on_two_calls():
    from linear_attention_mixer_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    H, d, n_slots = 4, 128, 5
    slots_np = np.array([3, 0, 4], dtype=np.int32)
    lens_a, lens_b = [37, 70, 5], [64, 1, 130]
    cu_a, cu_b = _call_pair(lens_a, lens_b)
    p = KI.make_params(H, d, 4, 61)
    tok_a = KI.make_tokens(int(cu_a[-1]), H, d, 61, bf16=False, sub=0)
    tok_b = KI.make_tokens(int(cu_b[-1]), H, d, 61, bf16=False, sub=1)
    cfg = K.kda_config(H, d, K.KDA_F32)
    params = dev_params(p)
    slots = torch.tensor(slots_np, device="cuda")
    D = H * d

    # the existing entry point, on a library-owned state
    st = K.kda_state_alloc(cfg, n_slots)
    ref_out = []
    try:
        for tok, cu in ((tok_a, cu_a), (tok_b, cu_b)):
            t = dev_tokens(tok, False)
            o = torch.empty(int(cu[-1]), D, device="cuda")
            K.kda_prefill(cfg, params, st, slots, torch.tensor(cu, device="cuda"), cu,
                          t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], o)
            ref_out.append(to_np(o))
        S_ref, tail_ref = download_state(cfg, st, list(range(n_slots)))
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)

    # the no-allocation entry point, two calls in a row on caller-owned buffers
    S = torch.zeros(n_slots, H, d, d, device="cuda")
    tail = torch.zeros(n_slots, 3, 3, D, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = []
    for tok, cu in ((tok_a, cu_a), (tok_b, cu_b)):
        t = dev_tokens(tok, False)
        o = torch.empty(int(cu[-1]), D, device="cuda")
        K.kda_prefill_noalloc(cfg, params, S, tail, err, slots, torch.tensor(cu, device="cuda"), cu,
                              t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], o)
        got.append(to_np(o))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for g, r in zip(got, ref_out):
        assert rel_err(g, r) <= TOL_F32
    assert rel_err(S.cpu().numpy(), S_ref) <= TOL_F32
    assert np.array_equal(tail.cpu().numpy(), tail_ref)

    # a request beyond the static workspace is refused before anything is enqueued
    big = K.kda_config(96, 128, K.KDA_F32)
    Sb = torch.zeros(1, 96, d, d, device="cuda")
    tb = torch.zeros(1, 3, 3, 96 * d, device="cuda")
    T = 4096
    x = torch.zeros(T, 96 * d, device="cuda")
    with pytest.raises(K.KdaError) as ei:
        K.kda_prefill_noalloc(big, params, Sb, tb, None, torch.zeros(1, dtype=torch.int32, device="cuda"),
                              torch.tensor([0, T], dtype=torch.int32, device="cuda"), [0, T],
                              x, x, x, x, torch.zeros(T, 96, device="cuda"), x, x)
    assert ei.value.status == K.KDA_ERR_INVALID and "static workspace" in ei.value.message


@pytest.mark.parametrize("bf16", [False, True], ids=["fp32", "bf16"])
def test_noalloc_prefill_matches_oracle_on_two_calls(oracle_mod, bf16):
    """Against the FP64 oracle: two calls in a row on caller-owned buffers, ragged sequences
    that continue from the first call's state into the second. The first call passes an error
    word, the second passes none (the library's own word inside the static workspace, cleared
    at the start of the call), and both complete."""
    from linear_attention_mixer_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    H, d, n_slots = 4, 128, 4
    slots_np = np.array([2, 0, 3], dtype=np.int32)
    lens_a, lens_b = [130, 1, 64], [70, 129, 5]
    cu_a, cu_b = _call_pair(lens_a, lens_b)
    seed = 62 + int(bf16)
    p = KI.make_params(H, d, 4, seed)
    tok_a = KI.make_tokens(int(cu_a[-1]), H, d, seed, bf16=bf16, sub=0)
    tok_b = KI.make_tokens(int(cu_b[-1]), H, d, seed, bf16=bf16, sub=1)
    S0 = KI.make_state(n_slots, H, d, seed, std=0.05)
    T0 = KI.make_tail(n_slots, H, d, 4, seed, bf16=bf16)
    cfg = K.kda_config(H, d, K.KDA_BF16 if bf16 else K.KDA_F32)
    dt = torch.bfloat16 if bf16 else torch.float32
    params = dev_params(p)
    slots = torch.tensor(slots_np, device="cuda")
    D = H * d
    S = torch.from_numpy(S0).cuda()
    tail = torch.from_numpy(T0).cuda().to(dt).contiguous()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = []
    for (tok, cu), e in (((tok_a, cu_a), err), ((tok_b, cu_b), None)):
        t = dev_tokens(tok, bf16)
        o = torch.empty(int(cu[-1]), D, device="cuda", dtype=dt)
        K.kda_prefill_noalloc(cfg, params, S, tail, e, slots, torch.tensor(cu, device="cuda"), cu,
                              t["q"], t["k"], t["v"], t["z"], t["b"], t["g"], o)
        got.append(to_np(o))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    oc = oracle_mod.OracleCfg(H=H, d=d)
    tol = TOL_BF16 if bf16 else TOL_F32
    Sg, tg = S.cpu().numpy(), tail.float().cpu().numpy()
    for i, s in enumerate(slots_np):
        Sr = S0[s].astype(np.float64)
        tr = T0[s].astype(np.float64)
        for (tok, cu), g in zip(((tok_a, cu_a), (tok_b, cu_b)), got):
            rows = slice(cu[i], cu[i + 1])
            ref = oracle_mod.sequence(oc, p, Sr, tr, {n: a[rows] for n, a in tok.items()})
            assert rel_err(g[rows], ref) <= tol, (bf16, i)
        print(f"noalloc {'bf16' if bf16 else 'fp32'} slot {s}: state {rel_err(Sg[s], Sr):.2e}")
        assert rel_err(Sg[s], Sr) <= tol
        assert np.array_equal(tg[s], tr.astype(np.float32))
    untouched = sorted(set(range(n_slots)) - set(slots_np.tolist()))
    for s in untouched:
        assert np.array_equal(Sg[s], S0[s]) and np.array_equal(tg[s], T0[s])
