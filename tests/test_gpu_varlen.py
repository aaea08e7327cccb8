"""Varlen workload at full size: 16 sequences with lengths ~U[512, 16384] (seeded),
96 heads x 128, BF16 I/O, FP32 state. Prefill all, snapshot sequences 0-7, reset
and restore them, then 128 batched decode steps. Sampled heads of every sequence
are recomputed by the FP64 oracle from the same seeded inputs."""
import numpy as np
import pytest
import torch

import kda_inputs as KI
import linear_attention_mixer_gb300 as K
from tests.kda_testutil import TOL_BF16, dev_params, download_state, rel_err, to_np

pytestmark = pytest.mark.gpu

HEADS = (0, 37, 95)  # sampled heads checked against the oracle


def test_varlen_prefill_snapshot_restore_decode(oracle_mod):
    from linear_attention_mixer_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    c = KI.CONFIGS["varlen"]
    H, d, N, steps = c["H"], c["d"], c["n_seq"], c["decode_steps"]
    D = H * d
    lens = KI.varlen_lengths(N, c["len_lo"], c["len_hi"], c["seed"])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    p = KI.make_params(H, d, 4, c["seed"])
    params = dev_params(p)

    # device inputs drawn by the seeded device generator (BF16); the host keeps the sampled
    # heads' columns, which are exactly the values the library reads
    dev = KI.make_tokens_torch(T, H, d, c["seed"], sub=0)
    host = {h: {n: (dev[n][:, h:h + 1] if n == "b" else dev[n][:, h * d:(h + 1) * d]).float().cpu().numpy()
                for n in "qkvzbg"} for h in HEADS}
    dec = [{n: t.float().cpu().numpy() for n, t in KI.make_tokens_torch(N, H, d, c["seed"], sub=1000 + s).items()}
           for s in range(steps)]
    cfg = K.kda_config(H, d, K.KDA_BF16)
    st = K.kda_state_alloc(cfg, N)
    try:
        out = torch.empty(T, D, dtype=torch.bfloat16, device="cuda")
        slots = torch.arange(N, dtype=torch.int32, device="cuda")
        K.kda_prefill(cfg, params, st, slots, torch.tensor(cu, device="cuda"), cu,
                      *(dev[n] for n in "qkvzbg"), out)
        half = list(range(N // 2))
        before = download_state(cfg, st, half)
        blob = torch.empty(K.kda_state_blob_bytes(st, len(half)), dtype=torch.uint8)
        K.kda_state_snapshot(st, half, blob)
        torch.cuda.synchronize()
        K.kda_state_reset(st, half)
        zeroed = download_state(cfg, st, half)
        K.kda_state_restore(st, half, blob)
        after = download_state(cfg, st, half)
        assert np.all(zeroed[0] == 0) and np.all(zeroed[1] == 0)
        assert np.array_equal(before[0], after[0]) and np.array_equal(before[1], after[1])
        dec_out = []
        for s in range(steps):
            x = {n: torch.from_numpy(dec[s][n]).cuda().to(torch.bfloat16) for n in "qkvzbg"}
            o = torch.empty(N, D, dtype=torch.bfloat16, device="cuda")
            K.kda_decode_token(cfg, params, st, slots, *(x[n] for n in "qkvzbg"), o)
            dec_out.append(o)
        S_fin, _ = download_state(cfg, st, list(range(N)))
        assert K.kda_state_poll_error(st) == 0
        got_pre = {h: to_np(out[:, h * d:(h + 1) * d]) for h in HEADS}
        got_dec = {h: np.stack([to_np(o[:, h * d:(h + 1) * d]) for o in dec_out]) for h in HEADS}  # [steps, N, d]
    finally:
        K.kda_state_free(st)
    del dev, out

    def check(h, i):  # one (head, sequence) unit, as a one-head problem for the oracle
        rows = slice(int(cu[i]), int(cu[i + 1]))
        tok1 = {n: np.ascontiguousarray(host[h][n][rows]) for n in "qkvzbg"}
        dtok = {n: np.stack([dec[s][n][i, h:h + 1] if n == "b" else dec[s][n][i, h * d:(h + 1) * d]
                             for s in range(steps)]) for n in "qkvzbg"}
        p1 = KI.LayerParams(np.ascontiguousarray(p.conv_w[:, h * d:(h + 1) * d]),
                            np.ascontiguousarray(p.dt_bias[h * d:(h + 1) * d]),
                            np.ascontiguousarray(p.A_log[h:h + 1]), p.norm_w)
        oc1 = oracle_mod.OracleCfg(H=1, d=d)
        S, tail = oracle_mod.new_state(oc1)
        ref_pre = oracle_mod.sequence(oc1, p1, S, tail, tok1, nthreads=1)
        ref_dec = oracle_mod.sequence(oc1, p1, S, tail, dtok, nthreads=1)
        return (rel_err(got_pre[h][rows], ref_pre), rel_err(got_dec[h][:, i], ref_dec), rel_err(S_fin[i, h], S[0]))

    from concurrent.futures import ThreadPoolExecutor  # the oracle releases the GIL in its C calls
    with ThreadPoolExecutor(max_workers=max(1, oracle_mod.max_threads())) as ex:
        res = list(ex.map(lambda hi: check(*hi), [(h, i) for h in HEADS for i in range(N)]))
    worst_pre, worst_dec, worst_s = (max(r[j] for r in res) for j in range(3))
    print(f"varlen 16 seqs, {T} tokens, heads {HEADS}: prefill {worst_pre:.2e} decode {worst_dec:.2e} "
          f"final state {worst_s:.2e}")
    assert worst_pre <= TOL_BF16
    assert worst_dec <= TOL_BF16
    assert worst_s <= TOL_BF16
