"""GPU parity of kda_gate_proj (the decay-gate and beta input projections,
z = W_fb (W_fa x) and b = W_b x) against the FP64 oracle in oracle/gate_proj.py, on
the same seeded inputs. With BF16 I/O the bound is max|diff| / max|ref| <= 2e-2 per
output tensor (the kernels round f to BF16 once and z, b on output, which puts the
error near 2^-9); with FP32 I/O it is 1e-3."""
import numpy as np
import pytest
import torch

import kda_inputs as KI
import linear_attention_mixer_gb300 as K
from kda_testutil import TOL_BF16, TOL_F32, rel_err
from oracle.gate_proj import gate_proj

pytestmark = pytest.mark.gpu


def _run(cfg, inp, dev="cuda", workspace=None, repeat=1):
    T, hidden = inp["x"].shape
    H, d = cfg.num_heads, cfg.head_dim
    dt = torch.bfloat16 if cfg.io_dtype == K.KDA_BF16 else torch.float32
    t = {n: torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(dt) for n, a in inp.items()}
    z = torch.full((T, H * d), float("nan"), device=dev, dtype=dt)
    b = torch.full((T, H), float("nan"), device=dev, dtype=dt)
    if workspace is None:
        workspace = torch.empty(K.kda_gate_proj_workspace_bytes(cfg, hidden, T), dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(repeat):
        K.kda_gate_proj(cfg, t["x"], t["w_fa"], t["w_fb"], t["w_b"], z, b, workspace)
        torch.cuda.synchronize()
        outs.append((z.float().cpu().numpy(), b.float().cpu().numpy()))
    err_word = int(workspace[:4].view(torch.int32).item())
    assert err_word == 0
    return outs


# (H, hidden, T): ragged token tiles, head counts that are not multiples of 16 (padded
# beta rows) or of 2 (a half-width last z tile), single-step and long hidden dimensions,
# split-K on and off, and the Kimi K3 geometry (96 heads, hidden 7168)
CASES = [(4, 192, 300), (1, 64, 5), (3, 128, 129), (2, 256, 1), (96, 512, 4096), (96, 7168, 1000),
         (17, 320, 777), (128, 1024, 2000)]


@pytest.mark.parametrize("H,hidden,T", CASES)
def test_gate_proj_matches_oracle(H, hidden, T):
    cfg = K.kda_config(H, 128, K.KDA_BF16)
    inp = KI.make_gate_proj(T, hidden, H, 128, seed=hidden + T + H)
    (z, b), = _run(cfg, inp)
    z_ref, b_ref = gate_proj(inp["x"], inp["w_fa"], inp["w_fb"], inp["w_b"])
    ez, eb = rel_err(z, z_ref), rel_err(b, b_ref)
    print(f"gate_proj H={H} hidden={hidden} T={T}: z {ez:.2e}, b {eb:.2e}")
    assert np.isfinite(z).all() and np.isfinite(b).all()
    assert ez <= TOL_BF16 and eb <= TOL_BF16


def test_gate_proj_full_size_sampled_rows():
    """T = 8192 tokens at hidden 7168 and 96 heads (the prefill workload's token count),
    in the launch configuration the benchmark times; 384 sampled rows against the oracle,
    including the first and last token tiles."""
    H, hidden, T = 96, 7168, 8192
    cfg = K.kda_config(H, 128, K.KDA_BF16)
    inp = KI.make_gate_proj(T, hidden, H, 128, seed=5)
    (z, b), = _run(cfg, inp)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(T - 64, T), rng.integers(0, T, 256)]))
    z_ref, b_ref = gate_proj(inp["x"][rows], inp["w_fa"], inp["w_fb"], inp["w_b"])
    ez, eb = rel_err(z[rows], z_ref), rel_err(b[rows], b_ref)
    print(f"gate_proj full size, {len(rows)} rows: z {ez:.2e}, b {eb:.2e}")
    assert np.isfinite(z).all() and np.isfinite(b).all()
    assert ez <= TOL_BF16 and eb <= TOL_BF16


def test_gate_proj_repeatable_and_workspace_checked():
    """Two calls on the same inputs give identical bits (the split-K partials are added in
    a fixed order); a workspace one byte short is refused before anything runs."""
    H, hidden, T = 96, 1024, 300
    cfg = K.kda_config(H, 128, K.KDA_BF16)
    inp = KI.make_gate_proj(T, hidden, H, 128, seed=9)
    (z1, b1), (z2, b2) = _run(cfg, inp, repeat=2)
    assert np.array_equal(z1, z2) and np.array_equal(b1, b2)
    need = K.kda_gate_proj_workspace_bytes(cfg, hidden, T)
    assert need > 0
    with pytest.raises(K.KdaError) as ei:
        _run(cfg, inp, workspace=torch.empty(need - 1, dtype=torch.uint8, device="cuda"))
    assert ei.value.status == K.KDA_ERR_INVALID



# T chosen so that the hidden dimension is split 3, 2 and 1 times on a 152-SM GB300 (tile pairs
# of 256 tokens: 50, 64 and 256 pairs); 1 means no cluster reduction at all. Rows are sampled,
# including the first and last token tiles.
@pytest.mark.parametrize("H,hidden,T", [(96, 1024, 12800), (96, 512, 16384), (8, 512, 65536)])
def test_gate_proj_large_T_sampled_rows(H, hidden, T):
    cfg = K.kda_config(H, 128, K.KDA_BF16)
    inp = KI.make_gate_proj(T, hidden, H, 128, seed=T + H)
    (z, b), = _run(cfg, inp)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([np.arange(0, 130), np.arange(T - 130, T), rng.integers(0, T, 256)]))
    z_ref, b_ref = gate_proj(inp["x"][rows], inp["w_fa"], inp["w_fb"], inp["w_b"])
    ez, eb = rel_err(z[rows], z_ref), rel_err(b[rows], b_ref)
    print(f"gate_proj H={H} hidden={hidden} T={T}, {len(rows)} rows: z {ez:.2e}, b {eb:.2e}")
    assert np.isfinite(z).all() and np.isfinite(b).all()
    assert ez <= TOL_BF16 and eb <= TOL_BF16


def test_gate_proj_zero_input_gives_exact_zeros():
    """x = 0 makes every product 0: z and b must be exactly zero (no stale workspace or
    staging data leaks into the outputs), also right after a call on nonzero inputs."""
    H, hidden, T = 96, 512, 700
    cfg = K.kda_config(H, 128, K.KDA_BF16)
    inp = KI.make_gate_proj(T, hidden, H, 128, seed=13)
    ws = torch.empty(K.kda_gate_proj_workspace_bytes(cfg, hidden, T), dtype=torch.uint8, device="cuda")
    _run(cfg, inp, workspace=ws)
    inp["x"] = np.zeros_like(inp["x"])
    (z, b), = _run(cfg, inp, workspace=ws)
    assert not z.any() and not b.any()


# FP32 I/O: the CUDA-core path, FP32 throughout, against the oracle on the same FP32 inputs
# (drawn as for BF16, so they happen to be BF16-representable; the arithmetic is FP32 anyway)
@pytest.mark.parametrize("H,hidden,T", [(2, 128, 64), (3, 192, 130), (96, 512, 300), (96, 7168, 70)])
def test_gate_proj_fp32_matches_oracle(H, hidden, T):
    cfg = K.kda_config(H, 128, K.KDA_F32)
    inp = KI.make_gate_proj(T, hidden, H, 128, seed=3 * T + H)
    (z, b), = _run(cfg, inp)
    z_ref, b_ref = gate_proj(inp["x"], inp["w_fa"], inp["w_fb"], inp["w_b"])
    ez, eb = rel_err(z, z_ref), rel_err(b, b_ref)
    print(f"gate_proj FP32 H={H} hidden={hidden} T={T}: z {ez:.2e}, b {eb:.2e}")
    assert ez <= TOL_F32 and eb <= TOL_F32


def test_gate_proj_feeds_the_mixer_fp32(oracle_mod):
    """The projection composed with the mixer, in FP32 (hidden state x -> kda_gate_proj -> z, b ->
    kda_prefill over two ragged sequences), against the oracle doing the same from x (its own
    projection, then its sequential recurrence): the mixer's FP32 bound of 1e-3."""
    from tests.kda_testutil import dev_params, to_np
    H, d, hidden, lens = 4, 128, 256, [70, 33]
    T = sum(lens)
    cfg = K.kda_config(H, d, K.KDA_F32)
    gp = KI.make_gate_proj(T, hidden, H, d, seed=21)
    p = KI.make_params(H, d, 4, seed=21)
    tok = KI.make_tokens(T, H, d, seed=21, bf16=False)
    (z, b), = _run(cfg, gp)
    dev = {n: torch.from_numpy(np.ascontiguousarray(tok[n])).cuda() for n in ("q", "k", "v", "g")}
    dev["z"], dev["b"] = torch.from_numpy(z).cuda(), torch.from_numpy(b).cuda()
    cu_h = np.array([0, lens[0], T], dtype=np.int32)
    st = K.kda_state_alloc(cfg, 2)
    try:
        out = torch.empty(T, H * d, device="cuda")
        K.kda_prefill(cfg, dev_params(p), st, torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                      torch.tensor(cu_h, device="cuda"), cu_h, dev["q"], dev["k"], dev["v"], dev["z"], dev["b"],
                      dev["g"], out)
        got = to_np(out)
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    z_o, b_o = gate_proj(gp["x"], gp["w_fa"], gp["w_fb"], gp["w_b"])
    oc = oracle_mod.OracleCfg(H=H, d=d)
    refs = []
    for s0, s1 in ((0, lens[0]), (lens[0], T)):
        seq = {n: tok[n][s0:s1] for n in ("q", "k", "v", "g")}
        seq["z"], seq["b"] = z_o[s0:s1], b_o[s0:s1]
        S, tail = oracle_mod.new_state(oc)
        refs.append(oracle_mod.sequence(oc, p, S, tail, seq))
    err = rel_err(got, np.concatenate(refs))
    print(f"gate_proj -> prefill, FP32, {T} tokens: rel err {err:.2e}")
    assert err <= TOL_F32


@pytest.mark.parametrize("H,hidden,lens", [(4, 256, [70, 33, 130]), (96, 1024, [300, 129])])
def test_gate_projection_fused_into_prefill_bf16(oracle_mod, H, hidden, lens):
    """x -> kda_gate_proj_in (f = W_fa x, b = W_b x) -> kda_prefill_gate_fused (z = W_fb f formed
    inside the prefill, never written) against the oracle's projection and recurrence, next to
    the separate path x -> kda_gate_proj -> kda_prefill; outputs and final states within the BF16
    bound, and b equal bit for bit between the two projection calls."""
    from tests.kda_testutil import TOL_BF16, dev_params, download_state, to_np
    d = 128
    T = sum(lens)
    N = len(lens)
    cfg = K.kda_config(H, d, K.KDA_BF16)
    gp = KI.make_gate_proj(T, hidden, H, d, seed=23)
    p = KI.make_params(H, d, 4, seed=23)
    tok = KI.make_tokens(T, H, d, seed=23, bf16=True)
    bf = torch.bfloat16
    dv = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(bf).contiguous()
    x, w_fa, w_fb, w_b = (dv(gp[n]) for n in ("x", "w_fa", "w_fb", "w_b"))
    ws = torch.empty(K.kda_gate_proj_workspace_bytes(cfg, hidden, T), dtype=torch.uint8, device="cuda")
    z = torch.empty(T, H * d, dtype=bf, device="cuda")
    b1 = torch.empty(T, H, dtype=bf, device="cuda")
    f = torch.empty(T, d, dtype=bf, device="cuda")
    b2 = torch.empty(T, H, dtype=bf, device="cuda")
    K.kda_gate_proj(cfg, x, w_fa, w_fb, w_b, z, b1, ws)
    K.kda_gate_proj_in(cfg, x, w_fa, w_b, f, b2, ws)
    torch.cuda.synchronize()
    assert torch.equal(b1, b2)
    q, k, v, g = (dv(tok[n]) for n in ("q", "k", "v", "g"))
    cu_h = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cu = torch.tensor(cu_h, device="cuda")
    slots = torch.arange(N, dtype=torch.int32, device="cuda")
    params = dev_params(p)
    res = {}
    for mode in ("separate", "fused"):
        st = K.kda_state_alloc(cfg, N)
        try:
            out = torch.empty(T, H * d, dtype=bf, device="cuda")
            if mode == "fused":
                K.kda_prefill_gate_fused(cfg, params, st, slots, cu, cu_h, q, k, v, f, w_fb, b2, g, out)
            else:
                K.kda_prefill(cfg, params, st, slots, cu, cu_h, q, k, v, z, b1, g, out)
            res[mode] = (to_np(out), download_state(cfg, st, list(range(N)))[0])
            assert K.kda_state_poll_error(st) == 0
        finally:
            K.kda_state_free(st)
    z_o, b_o = gate_proj(gp["x"], gp["w_fa"], gp["w_fb"], gp["w_b"])
    oc = oracle_mod.OracleCfg(H=H, d=d)
    refs, Ss = [], []
    for i in range(N):
        s0, s1 = cu_h[i], cu_h[i + 1]
        seq = {n: tok[n][s0:s1] for n in ("q", "k", "v", "g")}
        seq["z"], seq["b"] = z_o[s0:s1].astype(np.float32), b_o[s0:s1].astype(np.float32)
        S, tail = oracle_mod.new_state(oc)
        refs.append(oracle_mod.sequence(oc, p, S, tail, seq))
        Ss.append(S)
    ref = np.concatenate(refs)
    for mode, (got, Sg) in res.items():
        e, es = rel_err(got, ref), rel_err(Sg, np.stack(Ss))
        print(f"gate projection + prefill ({mode}), H={H}, {T} tokens: out {e:.2e} state {es:.2e}")
        assert e <= TOL_BF16 and es <= TOL_BF16
    # FP32 I/O has no fused path (the C entry point refuses it before enqueuing anything)
    import ctypes
    from linear_attention_mixer_gb300 import kda as KM
    cfg32 = K.kda_config(H, d, K.KDA_F32)
    st = K.kda_state_alloc(cfg32, N)
    try:
        P = lambda t: ctypes.c_void_p(t.data_ptr())
        rc = K.lib().kda_prefill_gate_fused(ctypes.byref(cfg32), ctypes.byref(params), st, P(slots), P(cu),
                                             KM._host_i32(cu_h)[1], N, P(q), P(k), P(v), P(f), P(w_fb), P(b2), P(g),
                                             P(q), ctypes.c_void_p(None))
        assert rc == K.KDA_ERR_INVALID and "BF16" in K.kda_last_error()
    finally:
        K.kda_state_free(st)


def test_gate_projection_fused_prefill_t8192_full_size(oracle_mod):
    """The hidden state of one 8192-token sequence (hidden 7168, 96 heads x 128, BF16) through
    kda_gate_proj_in and kda_prefill_gate_fused, against the FP64 projection oracle followed by
    the sequential oracle over all 8192 tokens; the final state too."""
    from tests.kda_testutil import dev_params, download_state
    c = KI.CONFIGS["prefill_8192"]
    H, d, T, hidden = c["H"], c["d"], c["T"], 7168
    cfg = K.kda_config(H, d, K.KDA_BF16)
    gp = KI.make_gate_proj(T, hidden, H, d, seed=31)
    p = KI.make_params(H, d, 4, 31)
    tok = KI.make_tokens(T, H, d, seed=31, bf16=True)
    bf = torch.bfloat16
    dv = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(bf).contiguous()
    f = torch.empty(T, d, dtype=bf, device="cuda")
    b = torch.empty(T, H, dtype=bf, device="cuda")
    ws = torch.empty(K.kda_gate_proj_workspace_bytes(cfg, hidden, T), dtype=torch.uint8, device="cuda")
    K.kda_gate_proj_in(cfg, dv(gp["x"]), dv(gp["w_fa"]), dv(gp["w_b"]), f, b, ws)
    st = K.kda_state_alloc(cfg, 1)
    try:
        cu_h = np.array([0, T], dtype=np.int32)
        out = torch.empty(T, H * d, dtype=bf, device="cuda")
        K.kda_prefill_gate_fused(cfg, dev_params(p), st, torch.zeros(1, dtype=torch.int32, device="cuda"),
                                 torch.tensor(cu_h, device="cuda"), cu_h, dv(tok["q"]), dv(tok["k"]), dv(tok["v"]), f,
                                 dv(gp["w_fb"]), b, dv(tok["g"]), out)
        got = out.float().cpu().numpy()
        Sg, _ = download_state(cfg, st, [0])
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    z_o, b_o = gate_proj(gp["x"], gp["w_fa"], gp["w_fb"], gp["w_b"])
    seq = {n: tok[n] for n in ("q", "k", "v", "g")}
    seq["z"], seq["b"] = z_o.astype(np.float32), b_o.astype(np.float32)
    oc = oracle_mod.OracleCfg(H=H, d=d)
    S, tail = oracle_mod.new_state(oc)
    ref = oracle_mod.sequence(oc, p, S, tail, seq)
    e, es = rel_err(got, ref), rel_err(Sg[0], S)
    print(f"gate projection fused into the prefill, T=8192, hidden 7168: out {e:.2e} final state {es:.2e}")
    assert e <= TOL_BF16 and es <= TOL_BF16 and np.isfinite(got).all()
