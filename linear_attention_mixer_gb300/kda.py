"""Python binding of the KDA C ABI (include/kda.h), by ctypes.

Argument marshalling only: every function forwards to the entry point of the
same name in libkda.so; all arithmetic runs in the CUDA kernels behind it.
Device tensors are torch tensors (used for device memory and streams only).
There is no fallback: if libkda.so is missing or the call fails, an exception
is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

KDA_OK, KDA_ERR_INVALID, KDA_ERR_OOM, KDA_ERR_CUDA, KDA_ERR_BLOB, KDA_ERR_TIMEOUT, KDA_ERR_DEVICE, KDA_ERR_IO = range(8)
KDA_F32, KDA_BF16 = 0, 1
KDA_BLOB_MAGIC = 0x3141444B
KDA_BLOB_VERSION = 1
KDA_DECODE_MAX_TOKENS = 8  # most tokens per row in one kda_decode_tokens call
STATUS_NAMES = {0: "KDA_OK", 1: "KDA_ERR_INVALID", 2: "KDA_ERR_OOM", 3: "KDA_ERR_CUDA",
                4: "KDA_ERR_BLOB", 5: "KDA_ERR_TIMEOUT", 6: "KDA_ERR_DEVICE",
                7: "KDA_ERR_IO"}

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")


class KdaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


class kda_config_t(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("conv_kernel", ctypes.c_int32),
                ("io_dtype", ctypes.c_int32), ("chunk_size", ctypes.c_int32),
                ("gate_lower_bound", ctypes.c_float), ("l2_eps", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("q_scale", ctypes.c_float)]


class kda_layer_params(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("A_log", ctypes.c_void_p), ("norm_w", ctypes.c_void_p)]


class kda_blob_header(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_uint32), ("version", ctypes.c_uint32),
                ("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("conv_kernel", ctypes.c_int32), ("io_dtype", ctypes.c_int32),
                ("n_slots", ctypes.c_int32), ("reserved0", ctypes.c_int32),
                ("state_bytes_per_slot", ctypes.c_uint64), ("tail_bytes_per_slot", ctypes.c_uint64),
                ("reserved", ctypes.c_uint8 * 16)]


_VP = ctypes.c_void_p
_I32 = ctypes.c_int32
_PI32 = ctypes.POINTER(ctypes.c_int32)
_lib = None

# (name, restype, argtypes) for every entry point of include/kda.h
SIGNATURES = [
    ("kda_config", _I32, [ctypes.POINTER(kda_config_t), _I32, _I32, _I32]),
    ("kda_state_alloc", _I32, [ctypes.POINTER(kda_config_t), _I32, ctypes.POINTER(_VP)]),
    ("kda_state_free", _I32, [_VP]),
    ("kda_state_reset", _I32, [_VP, _PI32, _I32, _VP]),
    ("kda_state_max_slots", _I32, [_VP]),
    ("kda_state_blob_bytes", ctypes.c_size_t, [_VP, _I32]),
    ("kda_state_snapshot", _I32, [_VP, _PI32, _I32, _VP, _I32, _VP]),
    ("kda_state_restore", _I32, [_VP, _PI32, _I32, _VP, _I32, _VP]),
    ("kda_decode_token", _I32, [ctypes.POINTER(kda_config_t), ctypes.POINTER(kda_layer_params), _VP, _VP, _I32,
                                _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    ("kda_decode_tokens", _I32, [ctypes.POINTER(kda_config_t), ctypes.POINTER(kda_layer_params), _VP, _VP, _I32,
                                 _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    ("kda_prefill", _I32, [ctypes.POINTER(kda_config_t), ctypes.POINTER(kda_layer_params), _VP, _VP, _VP, _PI32,
                           _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    ("kda_prefill_noalloc", _I32, [ctypes.POINTER(kda_config_t), ctypes.POINTER(kda_layer_params), _VP, _VP, _I32,
                                   _VP, _VP, _VP, _PI32, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    ("kda_state_poll_error", _I32, [_VP, _PI32]),
    ("kda_gate_proj_workspace_bytes", ctypes.c_size_t, [ctypes.POINTER(kda_config_t), _I32, ctypes.c_int64]),
    ("kda_gate_proj", _I32, [ctypes.POINTER(kda_config_t), _I32, ctypes.c_int64, _VP, _VP, _VP, _VP, _VP, _VP,
                             _VP, ctypes.c_size_t, _VP]),
    ("kda_gate_proj_in", _I32, [ctypes.POINTER(kda_config_t), _I32, ctypes.c_int64, _VP, _VP, _VP, _VP, _VP, _VP,
                                ctypes.c_size_t, _VP]),
    ("kda_prefill_gate_fused", _I32, [ctypes.POINTER(kda_config_t), ctypes.POINTER(kda_layer_params), _VP, _VP, _VP,
                                      _PI32, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    ("kda_linear_workspace_bytes", ctypes.c_size_t, [_I32, _I32, _I32]),
    ("kda_linear", _I32, [_I32, _I32, _I32, _VP, _VP, _VP, _VP, _I32, _VP, ctypes.c_size_t, _VP]),
    ("kda_photo_store_create", _I32, [_I32, ctypes.c_char_p, ctypes.POINTER(_VP)]),
    ("kda_photo_store_free", _I32, [_VP]),
    ("kda_photo_count", _I32, [_VP]),
    ("kda_photo_capacity", _I32, [_VP]),
    ("kda_photo_take", _I32, [_VP, ctypes.POINTER(_VP), _I32, _I32, _PI32, ctypes.c_int64, _PI32, _VP]),
    ("kda_photo_find", _I32, [_VP, _PI32, ctypes.c_int64, _PI32, ctypes.POINTER(ctypes.c_int64)]),
    ("kda_photo_restore", _I32, [_VP, _I32, ctypes.POINTER(_VP), _I32, _I32, _VP]),
    ("kda_last_error", ctypes.c_char_p, []),
]


def lib() -> ctypes.CDLL:
    """Load libkda.so from the package directory (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"the KDA CUDA library is not built ({LIB_PATH} missing); "
                               "run linear_attention_mixer_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def kda_last_error() -> str:
    return lib().kda_last_error().decode()


def _check(status: int):
    if status != KDA_OK:
        raise KdaError(status, kda_last_error())


def _stream(stream):
    if stream is None:
        return _VP(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return _VP(stream.cuda_stream)
    return _VP(int(stream))


def _torch_io_dtype(cfg: kda_config_t):
    return torch.bfloat16 if cfg.io_dtype == KDA_BF16 else torch.float32


def _dev(t: torch.Tensor, dtype=None, name: str = "tensor"):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return _VP(t.data_ptr())


def _host_i32(x):
    import numpy as np
    a = np.ascontiguousarray(np.asarray(x, dtype=np.int32))
    return a, a.ctypes.data_as(_PI32)


# ---------------------------------------------------------------- entry points

def kda_config(num_heads: int, head_dim: int = 128, io_dtype: int = KDA_BF16) -> kda_config_t:
    cfg = kda_config_t()
    _check(lib().kda_config(ctypes.byref(cfg), num_heads, head_dim, io_dtype))
    return cfg


def kda_state_alloc(cfg: kda_config_t, max_slots: int) -> ctypes.c_void_p:
    h = _VP()
    _check(lib().kda_state_alloc(ctypes.byref(cfg), max_slots, ctypes.byref(h)))
    return h


def kda_state_free(st) -> None:
    _check(lib().kda_state_free(st))


def kda_state_max_slots(st) -> int:
    return int(lib().kda_state_max_slots(st))


def kda_state_blob_bytes(st, n_slots: int) -> int:
    return int(lib().kda_state_blob_bytes(st, n_slots))


def kda_state_reset(st, slots, stream=None) -> None:
    arr, p = _host_i32(slots)
    _check(lib().kda_state_reset(st, p, len(arr), _stream(stream)))


def _buf(t: torch.Tensor, need: int, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous torch tensor")
    if t.numel() * t.element_size() < need:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes, {need} needed")
    return _VP(t.data_ptr()), int(t.is_cuda)


def kda_state_snapshot(st, slots, dst: torch.Tensor, stream=None) -> None:
    arr, p = _host_i32(slots)
    ptr, on_dev = _buf(dst, kda_state_blob_bytes(st, len(arr)), "dst")
    _check(lib().kda_state_snapshot(st, p, len(arr), ptr, on_dev, _stream(stream)))


def kda_state_restore(st, slots, src: torch.Tensor, stream=None) -> None:
    arr, p = _host_i32(slots)
    ptr, on_dev = _buf(src, kda_state_blob_bytes(st, len(arr)), "src")
    _check(lib().kda_state_restore(st, p, len(arr), ptr, on_dev, _stream(stream)))


def kda_layer_params_from(conv_w: torch.Tensor, dt_bias: torch.Tensor, A_log: torch.Tensor,
                          norm_w: torch.Tensor) -> kda_layer_params:
    p = kda_layer_params(_dev(conv_w, torch.float32, "conv_w"), _dev(dt_bias, torch.float32, "dt_bias"),
                         _dev(A_log, torch.float32, "A_log"), _dev(norm_w, torch.float32, "norm_w"))
    p._keep = (conv_w, dt_bias, A_log, norm_w)
    return p


def kda_decode_token(cfg: kda_config_t, params: kda_layer_params, st, slots: torch.Tensor,
                     q, k, v, z, b, g, out, stream=None) -> None:
    dt = _torch_io_dtype(cfg)
    B = int(slots.numel())
    D = cfg.num_heads * cfg.head_dim
    for name, t, width in (("q", q, D), ("k", k, D), ("v", v, D), ("z", z, D), ("g", g, D),
                           ("b", b, cfg.num_heads), ("out", out, D)):
        if t.numel() != B * width:
            raise ValueError(f"{name} must hold {B} x {width} elements, got {tuple(t.shape)}")
    _check(lib().kda_decode_token(ctypes.byref(cfg), ctypes.byref(params), st, _dev(slots, torch.int32, "slots"), B,
                                  _dev(q, dt, "q"), _dev(k, dt, "k"), _dev(v, dt, "v"), _dev(z, dt, "z"),
                                  _dev(b, dt, "b"), _dev(g, dt, "g"), _dev(out, dt, "out"), _stream(stream)))


def kda_decode_tokens(cfg: kda_config_t, params: kda_layer_params, st, slots: torch.Tensor, n: int,
                      q, k, v, z, b, g, out, stream=None) -> None:
    """n consecutive decode tokens per row: q,k,v,z,g,out [B][n][H*d], b [B][n][H]."""
    dt = _torch_io_dtype(cfg)
    B = int(slots.numel())
    D = cfg.num_heads * cfg.head_dim
    for name, t, width in (("q", q, D), ("k", k, D), ("v", v, D), ("z", z, D), ("g", g, D),
                           ("b", b, cfg.num_heads), ("out", out, D)):
        if t.numel() != B * n * width:
            raise ValueError(f"{name} must hold {B} x {n} x {width} elements, got {tuple(t.shape)}")
    _check(lib().kda_decode_tokens(ctypes.byref(cfg), ctypes.byref(params), st, _dev(slots, torch.int32, "slots"),
                                   B, int(n), _dev(q, dt, "q"), _dev(k, dt, "k"), _dev(v, dt, "v"),
                                   _dev(z, dt, "z"), _dev(b, dt, "b"), _dev(g, dt, "g"), _dev(out, dt, "out"),
                                   _stream(stream)))


def kda_prefill(cfg: kda_config_t, params: kda_layer_params, st, slots: torch.Tensor, cu_seqlens: torch.Tensor,
                cu_seqlens_host, q, k, v, z, b, g, out, stream=None) -> None:
    dt = _torch_io_dtype(cfg)
    N = int(slots.numel())
    cu_h, cu_p = _host_i32(cu_seqlens_host)
    if len(cu_h) != N + 1 or cu_seqlens.numel() != N + 1:
        raise ValueError("cu_seqlens must hold N + 1 entries")
    T = int(cu_h[-1]) if N > 0 else 0
    D = cfg.num_heads * cfg.head_dim
    for name, t, width in (("q", q, D), ("k", k, D), ("v", v, D), ("z", z, D), ("g", g, D),
                           ("b", b, cfg.num_heads), ("out", out, D)):
        if t.numel() != T * width:
            raise ValueError(f"{name} must hold {T} x {width} elements, got {tuple(t.shape)}")
    _check(lib().kda_prefill(ctypes.byref(cfg), ctypes.byref(params), st, _dev(slots, torch.int32, "slots"),
                             _dev(cu_seqlens, torch.int32, "cu_seqlens"), cu_p, N,
                             _dev(q, dt, "q"), _dev(k, dt, "k"), _dev(v, dt, "v"), _dev(z, dt, "z"),
                             _dev(b, dt, "b"), _dev(g, dt, "g"), _dev(out, dt, "out"), _stream(stream)))


def kda_prefill_noalloc(cfg: kda_config_t, params: kda_layer_params, S: torch.Tensor, tail: torch.Tensor,
                        err, slots: torch.Tensor, cu_seqlens: torch.Tensor, cu_seqlens_host,
                        q, k, v, z, b, g, out, stream=None) -> None:
    """kda_prefill on caller-owned state buffers with the library's static workspace.

    S: FP32 [max_slots, H, d, d]; tail: io dtype [max_slots, 3, K-1, H*d]; err: int32
    device tensor of one element, or None.
    """
    dt = _torch_io_dtype(cfg)
    H, d, Kc = cfg.num_heads, cfg.head_dim, cfg.conv_kernel
    if S.dim() != 4 or tuple(S.shape[1:]) != (H, d, d):
        raise ValueError(f"S must be [max_slots, {H}, {d}, {d}]")
    max_slots = int(S.shape[0])
    if tuple(tail.shape) != (max_slots, 3, Kc - 1, H * d):
        raise ValueError(f"tail must be [{max_slots}, 3, {Kc - 1}, {H * d}]")
    N = int(slots.numel())
    cu_h, cu_p = _host_i32(cu_seqlens_host)
    if len(cu_h) != N + 1 or cu_seqlens.numel() != N + 1:
        raise ValueError("cu_seqlens must hold N + 1 entries")
    T = int(cu_h[-1]) if N > 0 else 0
    D = H * d
    for name, t, width in (("q", q, D), ("k", k, D), ("v", v, D), ("z", z, D), ("g", g, D),
                           ("b", b, H), ("out", out, D)):
        if t.numel() != T * width:
            raise ValueError(f"{name} must hold {T} x {width} elements, got {tuple(t.shape)}")
    errp = _VP(None) if err is None else _dev(err, torch.int32, "err")
    _check(lib().kda_prefill_noalloc(ctypes.byref(cfg), ctypes.byref(params), _dev(S, torch.float32, "S"),
                                     _dev(tail, dt, "tail"), max_slots, errp, _dev(slots, torch.int32, "slots"),
                                     _dev(cu_seqlens, torch.int32, "cu_seqlens"), cu_p, N,
                                     _dev(q, dt, "q"), _dev(k, dt, "k"), _dev(v, dt, "v"), _dev(z, dt, "z"),
                                     _dev(b, dt, "b"), _dev(g, dt, "g"), _dev(out, dt, "out"), _stream(stream)))


def kda_gate_proj_workspace_bytes(cfg: kda_config_t, hidden: int, T: int) -> int:
    return int(lib().kda_gate_proj_workspace_bytes(ctypes.byref(cfg), int(hidden), int(T)))


def kda_gate_proj(cfg: kda_config_t, x, w_fa, w_fb, w_b, z, b, workspace: torch.Tensor, stream=None) -> None:
    """z = W_fb (W_fa x), b = W_b x for x [T, hidden]; every tensor in the config's I/O dtype
    except the workspace (any dtype, at least kda_gate_proj_workspace_bytes bytes)."""
    H, d = cfg.num_heads, cfg.head_dim
    if x.dim() != 2:
        raise ValueError("x must be [T, hidden]")
    T, hidden = int(x.shape[0]), int(x.shape[1])
    for name, t, shape in (("w_fa", w_fa, (d, hidden)), ("w_fb", w_fb, (H * d, d)), ("w_b", w_b, (H, hidden)),
                           ("z", z, (T, H * d)), ("b", b, (T, H))):
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must be {list(shape)}, got {list(t.shape)}")
    bf = _torch_io_dtype(cfg)
    ws = _dev(workspace, None, "workspace")
    _check(lib().kda_gate_proj(ctypes.byref(cfg), hidden, T, _dev(x, bf, "x"), _dev(w_fa, bf, "w_fa"),
                               _dev(w_fb, bf, "w_fb"), _dev(w_b, bf, "w_b"), _dev(z, bf, "z"), _dev(b, bf, "b"),
                               ws, workspace.numel() * workspace.element_size(), _stream(stream)))


def kda_gate_proj_in(cfg: kda_config_t, x, w_fa, w_b, f, b, workspace: torch.Tensor, stream=None) -> None:
    """f = W_fa x [T, d] and b = W_b x [T, H] (BF16), the inputs of kda_prefill_gate_fused."""
    H, d = cfg.num_heads, cfg.head_dim
    if x.dim() != 2:
        raise ValueError("x must be [T, hidden]")
    T, hidden = int(x.shape[0]), int(x.shape[1])
    for name, t, shape in (("w_fa", w_fa, (d, hidden)), ("w_b", w_b, (H, hidden)), ("f", f, (T, d)), ("b", b, (T, H))):
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must be {list(shape)}, got {list(t.shape)}")
    bf = torch.bfloat16
    _check(lib().kda_gate_proj_in(ctypes.byref(cfg), hidden, T, _dev(x, bf, "x"), _dev(w_fa, bf, "w_fa"),
                                  _dev(w_b, bf, "w_b"), _dev(f, bf, "f"), _dev(b, bf, "b"),
                                  _dev(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
                                  _stream(stream)))


def kda_prefill_gate_fused(cfg: kda_config_t, params: kda_layer_params, st, slots: torch.Tensor,
                           cu_seqlens: torch.Tensor, cu_seqlens_host, q, k, v, f, w_fb, b, g, out, stream=None) -> None:
    """kda_prefill with z = W_fb f formed inside (f = W_fa x [T, d], w_fb [H d, d]; BF16)."""
    bf = torch.bfloat16
    N = int(slots.numel())
    cu_h, cu_p = _host_i32(cu_seqlens_host)
    if len(cu_h) != N + 1 or cu_seqlens.numel() != N + 1:
        raise ValueError("cu_seqlens must hold N + 1 entries")
    T = int(cu_h[-1]) if N > 0 else 0
    H, d = cfg.num_heads, cfg.head_dim
    D = H * d
    for name, t, width in (("q", q, D), ("k", k, D), ("v", v, D), ("f", f, d), ("g", g, D), ("b", b, H),
                           ("out", out, D)):
        if t.numel() != T * width:
            raise ValueError(f"{name} must hold {T} x {width} elements, got {tuple(t.shape)}")
    if tuple(w_fb.shape) != (D, d):
        raise ValueError(f"w_fb must be [{D}, {d}]")
    _check(lib().kda_prefill_gate_fused(ctypes.byref(cfg), ctypes.byref(params), st, _dev(slots, torch.int32, "slots"),
                                        _dev(cu_seqlens, torch.int32, "cu_seqlens"), cu_p, N, _dev(q, bf, "q"),
                                        _dev(k, bf, "k"), _dev(v, bf, "v"), _dev(f, bf, "f"), _dev(w_fb, bf, "w_fb"),
                                        _dev(b, bf, "b"), _dev(g, bf, "g"), _dev(out, bf, "out"), _stream(stream)))


def kda_linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().kda_linear_workspace_bytes(int(M), int(N), int(K)))


def kda_linear(x, w, y, workspace: torch.Tensor, r=None, ysplit: int = 0, stream=None) -> None:
    """y = x w^T (+ r), BF16: x [M, K], w [N, K], y [M, N] (or [N / ysplit, M, ysplit] with ysplit)."""
    bf = torch.bfloat16
    if x.dim() != 2 or w.dim() != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("x must be [M, K] and w [N, K]")
    M, K = int(x.shape[0]), int(x.shape[1])
    N = int(w.shape[0])
    if y.numel() != M * N:
        raise ValueError(f"y must hold {M} x {N} elements, got {tuple(y.shape)}")
    if r is not None and r.numel() != M * N:
        raise ValueError(f"r must hold {M} x {N} elements, got {tuple(r.shape)}")
    _check(lib().kda_linear(M, N, K, _dev(x, bf, "x"), _dev(w, bf, "w"),
                            _VP(None) if r is None else _dev(r, bf, "r"), _dev(y, bf, "y"), int(ysplit),
                            _dev(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
                            _stream(stream)))


def _layers(layers):
    hs = [layers] if isinstance(layers, _VP) else list(layers)
    arr = (_VP * len(hs))(*[h.value if isinstance(h, _VP) else h for h in hs])
    return arr, len(hs)


def kda_photo_store_create(capacity: int = -1, dir: str | None = None) -> ctypes.c_void_p:
    """A photo store: capacity < 0 means "not given" (2 with a directory, else 0 = off)."""
    h = _VP()
    _check(lib().kda_photo_store_create(capacity, None if dir is None else dir.encode(), ctypes.byref(h)))
    return h


def kda_photo_store_free(ps) -> None:
    _check(lib().kda_photo_store_free(ps))


def kda_photo_count(ps) -> int:
    return int(lib().kda_photo_count(ps))


def kda_photo_capacity(ps) -> int:
    return int(lib().kda_photo_capacity(ps))


def kda_photo_take(ps, layers, slot: int, tokens, stream=None) -> int:
    """Photo of `slot` of each state in `layers` after the host token prefix; returns its id (-1: store off)."""
    arr, n = _layers(layers)
    tok, tp = _host_i32(tokens)
    pid = ctypes.c_int32()
    _check(lib().kda_photo_take(ps, arr, n, slot, tp, len(tok), ctypes.byref(pid), _stream(stream)))
    return int(pid.value)


def kda_photo_find(ps, tokens) -> tuple[int, int]:
    """(photo id, prefix length) of the deepest photo whose prefix starts `tokens`, or (-1, 0)."""
    tok, tp = _host_i32(tokens)
    pid, plen = ctypes.c_int32(), ctypes.c_int64()
    _check(lib().kda_photo_find(ps, tp, len(tok), ctypes.byref(pid), ctypes.byref(plen)))
    return int(pid.value), int(plen.value)


def kda_photo_restore(ps, photo_id: int, layers, slot: int, stream=None) -> None:
    arr, n = _layers(layers)
    _check(lib().kda_photo_restore(ps, photo_id, arr, n, slot, _stream(stream)))


def kda_state_poll_error(st) -> int:
    code = ctypes.c_int32()
    _check(lib().kda_state_poll_error(st, ctypes.byref(code)))
    return int(code.value)
