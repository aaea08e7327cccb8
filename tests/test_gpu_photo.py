"""Recurrent-state photos (kda_photo_*): a prompt that diverges from an earlier one
resumes from the deepest photo whose token prefix it still starts with, then prefills
only the rest. The resumed run must equal, bit for bit, a run that prefilled the same
prefix and remainder itself, and both must match the FP64 oracle over the whole new
prompt. Also: least-recently-used eviction, same-prefix replacement, the store being
off, parked files, and the error paths."""
import os

import numpy as np
import pytest
import torch

import kda_inputs as KI
import linear_attention_mixer_gb300 as K
from tests.kda_testutil import TOL_BF16, dev_params, download_state, rel_err, to_np

pytestmark = pytest.mark.gpu

H, D_HEAD = 4, 128
SEED = 71


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_attention_mixer_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _prefill_rows(cfg, params, st, slot, x, a, b):
    """Prefill rows [a, b) of the input dict x into `slot`; returns the outputs as numpy."""
    n = b - a
    cu_h = np.array([0, n], dtype=np.int32)
    t = {k: torch.from_numpy(np.ascontiguousarray(v[a:b])).cuda().to(torch.bfloat16) for k, v in x.items()}
    out = torch.empty(n, cfg.num_heads * cfg.head_dim, device="cuda", dtype=torch.bfloat16)
    K.kda_prefill(cfg, params, st, torch.tensor([slot], dtype=torch.int32, device="cuda"),
                  torch.tensor(cu_h, device="cuda"), cu_h, *(t[k] for k in "qkvzbg"), out)
    return to_np(out)


def _prompts():
    """Prompt A (700 tokens, photographed after 300 and 560) and prompt B, which shares
    A's first 450 tokens and then diverges, with per-layer inputs that agree exactly on
    the shared prefix (as a causal model's layer inputs would)."""
    rng = np.random.default_rng(SEED)
    tok_a = rng.integers(0, 50_000, 700).astype(np.int32)
    tok_b = np.concatenate([tok_a[:450], rng.integers(0, 50_000, 250).astype(np.int32)])
    tok_b[450] = tok_a[450] + 1  # the prompts part at 450
    xa, xb = [], []
    for layer in range(2):
        a = KI.make_tokens(700, H, D_HEAD, SEED + 17 * layer, bf16=True, sub=0)
        nb = KI.make_tokens(700, H, D_HEAD, SEED + 17 * layer, bf16=True, sub=1)
        xa.append(a)
        xb.append({k: np.concatenate([a[k][:450], nb[k][450:]]) for k in a})
    return tok_a, tok_b, xa, xb


@pytest.mark.parametrize("mode", ["ram", "file"])
def test_photo_resume_equals_uninterrupted_and_oracle(oracle_mod, tmp_path, mode):
    tok_a, tok_b, xa, xb = _prompts()
    ps_ = [KI.make_params(H, D_HEAD, 4, SEED + 17 * layer) for layer in range(2)]
    params = [dev_params(p) for p in ps_]
    cfg = K.kda_config(H, D_HEAD, K.KDA_BF16)
    layers = [K.kda_state_alloc(cfg, 3) for _ in range(2)]  # slot 0: prompt A, 1: resumed B, 2: B in full
    store = K.kda_photo_store_create(2, str(tmp_path) if mode == "file" else None)
    try:
        # prompt A in two turns on slot 0, a photo after each
        ids = []
        for a, b in ((0, 300), (300, 560)):
            for layer in range(2):
                _prefill_rows(cfg, params[layer], layers[layer], 0, xa[layer], a, b)
            ids.append(K.kda_photo_take(store, layers, 0, tok_a[:b]))
        assert K.kda_photo_count(store) == 2
        if mode == "file":
            assert len([f for f in os.listdir(tmp_path) if f.startswith("kda_photo_")]) == 2

        # prompt B: the photo after 300 tokens is the deepest one that B still starts with
        pid, plen = K.kda_photo_find(store, tok_b)
        assert (pid, plen) == (ids[0], 300)
        K.kda_photo_restore(store, pid, layers, 1)
        resumed = [_prefill_rows(cfg, params[layer], layers[layer], 1, xb[layer], 300, 700) for layer in range(2)]

        # the same two calls without a photo: prefix, then the rest
        full = []
        for layer in range(2):
            _prefill_rows(cfg, params[layer], layers[layer], 2, xb[layer], 0, 300)
            full.append(_prefill_rows(cfg, params[layer], layers[layer], 2, xb[layer], 300, 700))
        for layer in range(2):
            assert np.array_equal(resumed[layer], full[layer]), layer
            S1, t1 = download_state(cfg, layers[layer], [1])
            S2, t2 = download_state(cfg, layers[layer], [2])
            assert np.array_equal(S1, S2) and np.array_equal(t1, t2), layer
            assert K.kda_state_poll_error(layers[layer]) == 0
        S_got = [download_state(cfg, layers[layer], [1])[0][0] for layer in range(2)]
    finally:
        for st in layers:
            K.kda_state_free(st)
        K.kda_photo_store_free(store)
    if mode == "file":  # parked photos never outlive their store
        assert not [f for f in os.listdir(tmp_path) if f.startswith("kda_photo_")]

    # the FP64 oracle over all of prompt B from a zero state
    oc = oracle_mod.OracleCfg(H=H, d=D_HEAD)
    for layer in range(2):
        S, tail = oracle_mod.new_state(oc)
        ref = oracle_mod.sequence(oc, ps_[layer], S, tail, xb[layer])
        e_out, e_s = rel_err(resumed[layer], ref[300:]), rel_err(S_got[layer], S)
        print(f"photo resume ({mode}) layer {layer}: out {e_out:.2e} state {e_s:.2e}")
        assert e_out <= TOL_BF16 and e_s <= TOL_BF16


def test_photo_eviction_replacement_and_errors(tmp_path):
    cfg = K.kda_config(2, D_HEAD, K.KDA_BF16)
    params = dev_params(KI.make_params(2, D_HEAD, 4, SEED))
    x = KI.make_tokens(96, 2, D_HEAD, SEED, bf16=True, sub=3)
    st = K.kda_state_alloc(cfg, 2)
    other = K.kda_state_alloc(K.kda_config(4, D_HEAD, K.KDA_BF16), 1)
    store = K.kda_photo_store_create(2)
    off = K.kda_photo_store_create(0, str(tmp_path))
    try:
        blob = torch.empty(K.kda_state_blob_bytes(st, 1), dtype=torch.uint8)
        snaps = []
        # three photos of slot 0 after 32, 64 and 96 tokens, each kept as a reference blob
        for i, b in enumerate((32, 64, 96)):
            _prefill_rows(cfg, params, st, 0, x, b - 32, b)
            K.kda_state_snapshot(st, [0], blob)
            torch.cuda.synchronize()
            snaps.append(blob.clone())
            if i < 2:
                K.kda_photo_take(store, [st], 0, list(range(b)))
            if i == 1:
                # using the first photo makes the second the least recently used
                p32, _ = K.kda_photo_find(store, list(range(40)))
                K.kda_photo_restore(store, p32, [st], 1)
        ids_before = K.kda_photo_find(store, list(range(100)))
        p96 = K.kda_photo_take(store, [st], 0, list(range(96)))
        assert K.kda_photo_count(store) == 2
        assert K.kda_photo_find(store, list(range(100))) == (p96, 96)
        assert K.kda_photo_find(store, list(range(70)))[1] == 32  # the 64-token photo was evicted
        with pytest.raises(K.KdaError) as e:
            K.kda_photo_restore(store, ids_before[0], [st], 1)
        assert e.value.status == K.KDA_ERR_INVALID
        # a restored photo is bit-identical to the state it was taken from
        p32, plen = K.kda_photo_find(store, list(range(32)) + [7, 7])
        assert plen == 32
        K.kda_photo_restore(store, p32, [st], 1)
        K.kda_state_snapshot(st, [1], blob)
        torch.cuda.synchronize()
        assert torch.equal(blob[64:], snaps[0][64:])
        # the same prefix again replaces its photo (new id, same count)
        p32b = K.kda_photo_take(store, [st], 1, list(range(32)))
        assert p32b != p32 and K.kda_photo_count(store) == 2
        assert K.kda_photo_find(store, list(range(33))) == (p32b, 32)
        # a store of capacity 0 is off
        assert K.kda_photo_take(off, [st], 0, [1, 2, 3]) == -1 and K.kda_photo_count(off) == 0
        assert not os.listdir(tmp_path)
        # errors: layer count, geometry, slot range
        with pytest.raises(K.KdaError) as e:
            K.kda_photo_restore(store, p96, [st, st], 1)
        assert e.value.status == K.KDA_ERR_INVALID
        with pytest.raises(K.KdaError) as e:
            K.kda_photo_restore(store, p96, [other], 0)
        assert e.value.status == K.KDA_ERR_BLOB
        with pytest.raises(K.KdaError) as e:
            K.kda_photo_take(store, [st, other], 0, [1])
        assert e.value.status == K.KDA_ERR_INVALID
        with pytest.raises(K.KdaError) as e:
            K.kda_photo_take(store, [st], 2, [1])
        assert e.value.status == K.KDA_ERR_INVALID
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
        K.kda_state_free(other)
        K.kda_photo_store_free(store)
        K.kda_photo_store_free(off)
