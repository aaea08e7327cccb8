"""A whole KDA layer and a stack of them, on the library's kernels only.

Per token of each sequence (kimi_k3.c header comment, block "KDA per-head
recurrence"; struct Kda: W q, k, v, o, g, fa, fb, bp):

    q, k, v, g = W_q x, W_k x, W_v x, W_g x      one kda_linear over the stacked weights
    z, b       = W_fb (W_fa x), W_b x            kda_gate_proj
    o          = mixer(q, k, v, z, b, g)          kda_decode_token / kda_prefill (ShortConv4,
                                                  SiLU, L2, gates, delta rule, readout,
                                                  sigmoid(g) * RMSNorm_head)
    x'         = x + W_o o                        kda_linear with the residual

The residual add stands in for the model's residual stream (the pages' attention
residuals and the MoE/MLP blocks between KDA layers are other components). This module
only sequences library calls and owns their buffers; every product and every step of the
mixer runs in libkda's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import kda as K


@dataclass
class KdaLayerWeights:
    """Device weights of one KDA layer (BF16 products, FP32 mixer parameters)."""
    w_qkvg: torch.Tensor   # [4 H d, hidden]: rows of W_q, W_k, W_v, W_g in that order
    w_fa: torch.Tensor     # [d, hidden]
    w_fb: torch.Tensor     # [H d, d]
    w_b: torch.Tensor      # [H, hidden]
    w_o: torch.Tensor      # [hidden, H d]
    params: K.kda_layer_params  # conv_w, dt_bias, A_log, norm_w (FP32)


def random_layer_weights(H: int, d: int, hidden: int, gen: torch.Generator, device) -> KdaLayerWeights:
    """Synthetic weights: each projection ~ N(0, 1/fan_in) (so outputs come out ~ N(0, 1) for
    an input of unit variance), mixer parameters from the workload's distributions."""
    import math
    bf = torch.bfloat16
    D = H * d

    def mat(n, k):
        return (torch.randn(n, k, generator=gen, device=device) * k ** -0.5).to(bf).contiguous()

    conv_w = (torch.randn(3, D, 4, generator=gen, device=device) * 0.5).contiguous()
    dt_bias = torch.randn(D, generator=gen, device=device) * math.sqrt(0.5)
    A_log = torch.rand(H, generator=gen, device=device) * math.log(16.0)
    norm_w = 1.0 + torch.randn(d, generator=gen, device=device) * math.sqrt(0.1)
    return KdaLayerWeights(mat(4 * D, hidden), mat(d, hidden), mat(D, d), mat(H, hidden), mat(hidden, D),
                           K.kda_layer_params_from(conv_w, dt_bias, A_log, norm_w))


class KdaLayerRunner:
    """Buffers for running KDA layers on a batch of up to `rows` tokens at a time."""

    def __init__(self, cfg: K.kda_config_t, hidden: int, rows: int, device):
        self.cfg = cfg
        self.hidden = hidden
        H, d = cfg.num_heads, cfg.head_dim
        D = H * d
        bf = torch.bfloat16
        self.rows = rows
        self.qkvg = torch.empty(4, rows, D, dtype=bf, device=device)
        self.z = torch.empty(rows, D, dtype=bf, device=device)
        self.b = torch.empty(rows, H, dtype=bf, device=device)
        self.o = torch.empty(rows, D, dtype=bf, device=device)
        # the k split (and so the workspace) depends on the number of 256-row blocks: take the
        # largest need over every row count up to `rows`
        ws = 256
        for mb in range(1, (rows + 255) // 256 + 1):
            m = min(rows, 256 * mb)
            ws = max(ws, K.kda_linear_workspace_bytes(m, 4 * D, hidden), K.kda_linear_workspace_bytes(m, hidden, D))
        self.ws_lin = torch.empty(ws, dtype=torch.uint8, device=device)
        self.ws_gp = torch.empty(K.kda_gate_proj_workspace_bytes(cfg, hidden, rows), dtype=torch.uint8, device=device)

    def _inputs(self, lw: KdaLayerWeights, x: torch.Tensor, stream):
        n = x.shape[0]
        D = self.o.shape[1]
        qkvg = self.qkvg.view(-1)[:4 * n * D].view(4, n, D)  # four contiguous [n, D] matrices
        K.kda_linear(x, lw.w_qkvg, qkvg, self.ws_lin, ysplit=self.o.shape[1], stream=stream)
        z, b = self.z[:n], self.b[:n]
        K.kda_gate_proj(self.cfg, x, lw.w_fa, lw.w_fb, lw.w_b, z, b, self.ws_gp, stream)
        return qkvg, z, b

    def decode(self, lw: KdaLayerWeights, st, slots: torch.Tensor, x: torch.Tensor, x_out: torch.Tensor,
               stream=None) -> None:
        """One decode token for each of the x.shape[0] rows (row r on slot slots[r]): x_out = x + W_o o."""
        n = x.shape[0]
        qkvg, z, b = self._inputs(lw, x, stream)
        o = self.o[:n]
        K.kda_decode_token(self.cfg, lw.params, st, slots, qkvg[0], qkvg[1], qkvg[2], z, b, qkvg[3], o, stream)
        K.kda_linear(o, lw.w_o, x_out, self.ws_lin, r=x, stream=stream)

    def prefill(self, lw: KdaLayerWeights, st, slots: torch.Tensor, cu_seqlens: torch.Tensor, cu_seqlens_host,
                x: torch.Tensor, x_out: torch.Tensor, stream=None) -> None:
        """Packed variable-length prefill of x.shape[0] tokens: x_out = x + W_o o."""
        n = x.shape[0]
        qkvg, z, b = self._inputs(lw, x, stream)
        o = self.o[:n]
        K.kda_prefill(self.cfg, lw.params, st, slots, cu_seqlens, cu_seqlens_host, qkvg[0], qkvg[1], qkvg[2], z, b,
                      qkvg[3], o, stream)
        K.kda_linear(o, lw.w_o, x_out, self.ws_lin, r=x, stream=stream)
