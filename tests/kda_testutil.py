"""Helpers shared by the GPU tests: moving oracle-side numpy state into and out of
the library's slots through the public snapshot/restore blob, and the error metric."""
from __future__ import annotations

import numpy as np
import torch

import kda_inputs as KI
import linear_attention_mixer_gb300 as K

TOL_F32 = 1e-3   # max|diff| / max|ref| with FP32 I/O
TOL_BF16 = 2e-2  # max|diff| / max|ref| with BF16 I/O


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / den) if den > 0 else float(np.abs(got).max())


def dev_params(p: KI.LayerParams, dev="cuda"):
    return K.kda_layer_params_from(*(torch.from_numpy(np.ascontiguousarray(x)).to(dev)
                                     for x in (p.conv_w, p.dt_bias, p.A_log, p.norm_w)))


def dev_tokens(tok: dict, bf16: bool, dev="cuda", rows=None):
    dt = torch.bfloat16 if bf16 else torch.float32
    out = {}
    for n in ("q", "k", "v", "z", "b", "g"):
        a = tok[n] if rows is None else tok[n][rows]
        out[n] = torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(dt).contiguous()
    return out


def _hdr(cfg, n):
    H, d, Kc = cfg.num_heads, cfg.head_dim, cfg.conv_kernel
    h = K.kda_blob_header()
    h.magic, h.version = K.KDA_BLOB_MAGIC, K.KDA_BLOB_VERSION
    h.num_heads, h.head_dim, h.conv_kernel, h.io_dtype, h.n_slots = H, d, Kc, cfg.io_dtype, n
    h.state_bytes_per_slot = H * d * d * 4
    h.tail_bytes_per_slot = 3 * (Kc - 1) * H * d * (2 if cfg.io_dtype == K.KDA_BF16 else 4)
    return bytes(h)


def upload_state(cfg, st, slots, S: np.ndarray, tail: np.ndarray):
    """Write S [n,H,d,d] (rounded to float32) and the conv history [n,3,K-1,D] into the slots."""
    n = len(slots)
    parts = [_hdr(cfg, n)]
    for i in range(n):
        parts.append(np.ascontiguousarray(S[i], dtype=np.float32).tobytes())
        t = np.ascontiguousarray(tail[i], dtype=np.float32)
        parts.append(KI.to_bf16_bits(t).tobytes() if cfg.io_dtype == K.KDA_BF16 else t.tobytes())
    blob = torch.frombuffer(bytearray(b"".join(parts)), dtype=torch.uint8)
    K.kda_state_restore(st, slots, blob)
    torch.cuda.synchronize()


def download_state(cfg, st, slots):
    """Read (S [n,H,d,d] float32, tail [n,3,K-1,D] float32) of the slots."""
    n = len(slots)
    H, d, Kc = cfg.num_heads, cfg.head_dim, cfg.conv_kernel
    D = H * d
    blob = torch.empty(K.kda_state_blob_bytes(st, n), dtype=torch.uint8)
    K.kda_state_snapshot(st, slots, blob)
    torch.cuda.synchronize()
    raw = blob.numpy().tobytes()
    off = 64
    sb = H * d * d * 4
    tb = 3 * (Kc - 1) * D * (2 if cfg.io_dtype == K.KDA_BF16 else 4)
    S = np.empty((n, H, d, d), dtype=np.float32)
    tail = np.empty((n, 3, Kc - 1, D), dtype=np.float32)
    for i in range(n):
        S[i] = np.frombuffer(raw, dtype=np.float32, count=H * d * d, offset=off).reshape(H, d, d)
        off += sb
        if cfg.io_dtype == K.KDA_BF16:
            bits = np.frombuffer(raw, dtype=np.uint16, count=3 * (Kc - 1) * D, offset=off)
            tail[i] = KI.from_bf16_bits(bits).reshape(3, Kc - 1, D)
        else:
            tail[i] = np.frombuffer(raw, dtype=np.float32, count=3 * (Kc - 1) * D, offset=off).reshape(3, Kc - 1, D)
        off += tb
    return S, tail


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)
