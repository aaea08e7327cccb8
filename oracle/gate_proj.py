"""FP64 oracle of the gate and beta input projections of a KDA layer.

TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's CPU-baseline leg
use it to check and time the CUDA library; the product path never imports it, and it
imports nothing from the product package.

What it computes (kimi_k3.c header comment, block "KDA per-head recurrence": the decay
gate's pre-activation is a low-rank projection of the hidden state, W_fb (W_fa x), and the
beta logit is a projection W_b x; struct Kda: fa is [hd][hidden], fb is [proj][hd], bp is
[heads][hidden], all FP32):
    f = W_fa x      (hd = 128 values per token)
    z = W_fb f      (proj = heads * hd values per token)
    b = W_b x       (heads values per token)
dt_bias and the sigmoids stay in the mixer (they act on z and b there). Matrix products
are numpy matmuls in float64, one step each, in the order the formula states.
"""
from __future__ import annotations

import numpy as np


def gate_proj(x: np.ndarray, fa: np.ndarray, fb: np.ndarray, bp: np.ndarray):
    """x [T][hidden] -> (z [T][proj], b [T][heads]) in float64."""
    x = np.asarray(x, dtype=np.float64)
    f = x @ np.asarray(fa, dtype=np.float64).T   # W_fa x, per token
    z = f @ np.asarray(fb, dtype=np.float64).T   # W_fb (W_fa x)
    b = x @ np.asarray(bp, dtype=np.float64).T   # W_b x
    return z, b
