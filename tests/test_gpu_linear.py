"""kda_linear (y = x W^T + r on the tensor cores, BF16 in and out) through the C ABI against
the FP64 layer oracle's product, over shapes that hit ragged row tiles, a single row, the
k-split path (partials added in split order), the column split into separate outputs and the
residual; and a whole KDA layer (projections, gate projections, mixer, W_o with the residual)
over several decode steps against the oracle's layer."""
import numpy as np
import pytest
import torch

import kda_inputs as KI
import linear_attention_mixer_gb300 as K
from oracle import layer as OL
from tests.kda_testutil import TOL_BF16, dev_params, download_state, rel_err, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_attention_mixer_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _bf(a):
    return KI.bf16_round(np.asarray(a, dtype=np.float32))


@pytest.mark.parametrize("M,N,K_,ysplit,res", [(1, 128, 64, 0, False), (37, 256, 192, 0, True),
                                               (256, 1024, 512, 256, False), (300, 384, 1024, 0, True),
                                               (256, 128, 4096, 0, True), (5, 512, 7168, 128, False),
                                               (513, 256, 128, 128, False)])
def test_linear_matches_oracle(M, N, K_, ysplit, res):
    rng = np.random.default_rng(M * 7 + N + K_)
    x = _bf(rng.standard_normal((M, K_)))
    w = _bf(rng.standard_normal((N, K_)) * K_ ** -0.5)
    r = _bf(rng.standard_normal((M, N))) if res else None
    dev = lambda a: torch.from_numpy(a).cuda().to(torch.bfloat16).contiguous()
    ws = torch.empty(K.kda_linear_workspace_bytes(M, N, K_), dtype=torch.uint8, device="cuda")
    y = torch.empty(N // (ysplit or N), M, ysplit or N, dtype=torch.bfloat16, device="cuda")
    K.kda_linear(dev(x), dev(w), y, ws, r=None if r is None else dev(r), ysplit=ysplit)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    got = to_np(y)
    got = np.concatenate(list(got), axis=1) if ysplit else got[0]
    ref = OL.linear(x, w, r)
    e = rel_err(got, ref)
    print(f"linear M={M} N={N} K={K_} ysplit={ysplit} res={res}: {e:.2e}")
    assert e <= TOL_BF16
    # repeatable bit for bit (the k split adds partials in split order)
    y2 = torch.empty_like(y)
    K.kda_linear(dev(x), dev(w), y2, ws, r=None if r is None else dev(r), ysplit=ysplit)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


def test_linear_argument_errors():
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(K.kda_linear_workspace_bytes(4, 128, 64), dtype=torch.uint8, device="cuda")
    for w, y, kw in ((torch.zeros(100, 64, dtype=torch.bfloat16, device="cuda"), torch.zeros(4, 100, dtype=torch.bfloat16, device="cuda"), {}),
                     (torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda"), torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda"), {"ysplit": 96})):
        with pytest.raises(K.KdaError) as ei:
            K.kda_linear(x, w, y, ws, **kw)
        assert ei.value.status == K.KDA_ERR_INVALID
    x48 = torch.zeros(4, 48, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(K.KdaError):
        K.kda_linear(x48, torch.zeros(128, 48, dtype=torch.bfloat16, device="cuda"),
                     torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda"), ws)


def test_layer_decode_matches_oracle(oracle_mod):
    """A whole layer (hidden 256, 2 heads): 3 sequences, 4 decode steps from filled states,
    each step x' = x + W_o mixer(W_q x, W_k x, W_v x, W_fb W_fa x, W_b x, W_g x)."""
    from linear_attention_mixer_gb300.layer import KdaLayerRunner, KdaLayerWeights
    H, d, hidden, B, steps = 2, 128, 256, 3, 4
    D = H * d
    rng = np.random.default_rng(81)
    p = KI.make_params(H, d, 4, 81)
    wn = {"w_qkvg": _bf(rng.standard_normal((4 * D, hidden)) * hidden ** -0.5),
          "w_fa": _bf(rng.standard_normal((d, hidden)) * hidden ** -0.5),
          "w_fb": _bf(rng.standard_normal((D, d)) * d ** -0.5),
          "w_b": _bf(rng.standard_normal((H, hidden)) * hidden ** -0.5),
          "w_o": _bf(rng.standard_normal((hidden, D)) * D ** -0.5)}
    dev = lambda a: torch.from_numpy(a).cuda().to(torch.bfloat16).contiguous()
    lw = KdaLayerWeights(dev(wn["w_qkvg"]), dev(wn["w_fa"]), dev(wn["w_fb"]), dev(wn["w_b"]), dev(wn["w_o"]),
                         dev_params(p))
    cfg = K.kda_config(H, d, K.KDA_BF16)
    S0 = KI.make_state(B, H, d, 81)
    T0 = KI.make_tail(B, H, d, 4, 81, bf16=True)
    st = K.kda_state_alloc(cfg, B)
    slots_np = np.array([2, 0, 1], dtype=np.int32)
    runner = KdaLayerRunner(cfg, hidden, B, "cuda")
    xs = [_bf(rng.standard_normal((B, hidden)))]
    outs = []
    try:
        from tests.kda_testutil import upload_state
        upload_state(cfg, st, list(range(B)), S0, T0)
        slots = torch.tensor(slots_np, device="cuda")
        x = dev(xs[0])
        for s in range(steps):
            y = torch.empty(B, hidden, dtype=torch.bfloat16, device="cuda")
            runner.decode(lw, st, slots, x, y)
            outs.append(to_np(y))
            x = y
        Sg, _ = download_state(cfg, st, list(range(B)))
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    oc = oracle_mod.OracleCfg(H=H, d=d)
    S_all, tail_all = S0.astype(np.float64), T0.astype(np.float64)
    x = xs[0].astype(np.float64)
    for s in range(steps):
        ref = OL.layer_decode(oc, p, wn, S_all, tail_all, slots_np, x)
        e = rel_err(outs[s], ref)
        print(f"layer decode step {s}: {e:.2e}")
        assert e <= TOL_BF16
        x = outs[s].astype(np.float64)  # the next step continues from the GPU's own output
    print(f"layer decode state: {rel_err(Sg, S_all):.2e}")
    assert rel_err(Sg, S_all) <= TOL_BF16


def test_layer_prefill_matches_oracle(oracle_mod):
    """A whole layer's packed prefill (hidden 256, 2 heads): sequences of 70 and 33 tokens
    (full chunks and ragged tails) from filled states, x' = x + W_o mixer(...), against the
    layer oracle's prefill, and the final states."""
    from linear_attention_mixer_gb300.layer import KdaLayerRunner, KdaLayerWeights
    H, d, hidden = 2, 128, 256
    D = H * d
    lens = [70, 33]
    cu_h = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu_h[-1])
    rng = np.random.default_rng(83)
    p = KI.make_params(H, d, 4, 83)
    wn = {"w_qkvg": _bf(rng.standard_normal((4 * D, hidden)) * hidden ** -0.5),
          "w_fa": _bf(rng.standard_normal((d, hidden)) * hidden ** -0.5),
          "w_fb": _bf(rng.standard_normal((D, d)) * d ** -0.5),
          "w_b": _bf(rng.standard_normal((H, hidden)) * hidden ** -0.5),
          "w_o": _bf(rng.standard_normal((hidden, D)) * D ** -0.5)}
    dev = lambda a: torch.from_numpy(a).cuda().to(torch.bfloat16).contiguous()
    lw = KdaLayerWeights(dev(wn["w_qkvg"]), dev(wn["w_fa"]), dev(wn["w_fb"]), dev(wn["w_b"]), dev(wn["w_o"]),
                         dev_params(p))
    cfg = K.kda_config(H, d, K.KDA_BF16)
    S0 = KI.make_state(2, H, d, 83)
    T0 = KI.make_tail(2, H, d, 4, 83, bf16=True)
    slots_np = np.array([1, 0], dtype=np.int32)
    x = _bf(rng.standard_normal((T, hidden)))
    st = K.kda_state_alloc(cfg, 2)
    runner = KdaLayerRunner(cfg, hidden, T, "cuda")
    try:
        from tests.kda_testutil import upload_state
        upload_state(cfg, st, [0, 1], S0, T0)
        y = torch.empty(T, hidden, dtype=torch.bfloat16, device="cuda")
        runner.prefill(lw, st, torch.tensor(slots_np, device="cuda"), torch.tensor(cu_h, device="cuda"), cu_h, dev(x),
                       y)
        got = to_np(y)
        Sg, tg = download_state(cfg, st, [0, 1])
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    oc = oracle_mod.OracleCfg(H=H, d=d)
    S_all, tail_all = S0.astype(np.float64), T0.astype(np.float64)
    ref = OL.layer_prefill(oc, p, wn, S_all, tail_all, slots_np, cu_h, x.astype(np.float64))
    e, es = rel_err(got, ref), rel_err(Sg, S_all)
    print(f"layer prefill, 2 sequences ({lens[0]} + {lens[1]} tokens): out {e:.2e} state {es:.2e}")
    assert e <= TOL_BF16 and es <= TOL_BF16



def test_linear_split_k_is_deterministic():
    """With few column tiles the K dimension is split over CTAs and the FP32 slices are added
    by a second kernel in slice order: repeated calls give identical bits."""
    rng = np.random.default_rng(91)
    M, N, K_ = 200, 256, 4096
    x = torch.from_numpy(_bf(rng.standard_normal((M, K_)))).cuda().to(torch.bfloat16)
    w = torch.from_numpy(_bf(rng.standard_normal((N, K_)) * K_ ** -0.5)).cuda().to(torch.bfloat16)
    ws_bytes = K.kda_linear_workspace_bytes(M, N, K_)
    assert ws_bytes > 256  # the split is in use at this shape
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ys = []
    for _ in range(3):
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        K.kda_linear(x, w, y, ws)
        ys.append(y)
    torch.cuda.synchronize()
    assert all(torch.equal(ys[0], y) for y in ys[1:])
