"""FP64 oracle of a whole KDA layer: the dense projections around the mixer.

TEST INFRASTRUCTURE ONLY. The tests use it to check the CUDA library's dense products
(kda_linear) and a layer built from them; the product path never imports it, and it
imports nothing from the product package.

What it computes, per token (kimi_k3.c header comment, block "KDA per-head recurrence":
q,k,v = SiLU(ShortConv4(W{q,k,v} x)), z = W_fb(W_fa x) + dt_bias, beta = sigmoid(W_b x),
out = W_o [sigmoid(W_g x) * RMSNorm_head(o)]; struct Kda: W q, k, v, o, g):
    q, k, v, g = W_q x, W_k x, W_v x, W_g x            numpy matmuls in float64
    z, b       = W_fb (W_fa x), W_b x                   oracle/gate_proj.py
    mixed      = the mixer on (q, k, v, z, b, g)        kda_oracle.c (sequential, FP64)
    x'         = x + W_o mixed                          a residual stream around the layer
The residual add is the plainest stand-in for the model's residual stream between layers
(the pages replace it by attention residuals, another component).
"""
from __future__ import annotations

import numpy as np

from oracle import oracle as O
from oracle.gate_proj import gate_proj


def linear(x, w, r=None) -> np.ndarray:
    """x [M][K] times w [N][K] transposed, plus r [M][N] if given, in float64."""
    y = np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T
    if r is not None:
        y = y + np.asarray(r, dtype=np.float64)
    return y


def layer_decode(cfg: O.OracleCfg, params, w: dict, S_all, tail_all, slots, x) -> np.ndarray:
    """One decode token for each row of x [B][hidden] (row r on slot slots[r] of S_all and
    tail_all, which advance in place). w holds float arrays w_qkvg [4 D][hidden] (rows of
    W_q, W_k, W_v, W_g), w_fa, w_fb, w_b and w_o [hidden][D]. Returns x' [B][hidden]."""
    D = cfg.H * cfg.d
    qkvg = linear(x, w["w_qkvg"])
    z, b = gate_proj(x, w["w_fa"], w["w_fb"], w["w_b"])
    tok = {"q": qkvg[:, 0:D], "k": qkvg[:, D:2 * D], "v": qkvg[:, 2 * D:3 * D], "g": qkvg[:, 3 * D:4 * D],
           "z": z, "b": b}
    tok = {n: np.ascontiguousarray(a, dtype=np.float32) for n, a in tok.items()}
    mixed = O.decode_batch(cfg, params, S_all, tail_all, slots, tok)
    return linear(mixed, w["w_o"], r=x)


def layer_prefill(cfg: O.OracleCfg, params, w: dict, S_all, tail_all, slots, cu_seqlens, x) -> np.ndarray:
    """Packed variable-length prefill of x [T][hidden]: sequence i is rows cu_seqlens[i] ..
    cu_seqlens[i + 1] - 1, on slot slots[i] of S_all and tail_all (which advance in place), its
    mixer run token by token by the sequential oracle. Returns x' [T][hidden]."""
    D = cfg.H * cfg.d
    qkvg = linear(x, w["w_qkvg"])
    z, b = gate_proj(x, w["w_fa"], w["w_fb"], w["w_b"])
    cols = {"q": qkvg[:, 0:D], "k": qkvg[:, D:2 * D], "v": qkvg[:, 2 * D:3 * D], "g": qkvg[:, 3 * D:4 * D],
            "z": z, "b": b}
    mixed = np.zeros((np.asarray(x).shape[0], D))
    for i, slot in enumerate(slots):
        a, e = int(cu_seqlens[i]), int(cu_seqlens[i + 1])
        tok = {n: np.ascontiguousarray(arr[a:e], dtype=np.float32) for n, arr in cols.items()}
        mixed[a:e] = O.sequence(cfg, params, S_all[slot], tail_all[slot], tok)
    return linear(mixed, w["w_o"], r=x)

