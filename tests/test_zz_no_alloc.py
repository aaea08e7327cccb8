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
from tests.kda_testutil import TOL_F32, dev_params, dev_tokens, download_state, rel_err, to_np

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
