"""Python access to the FP64 CPU oracle of the KDA mixer core (kda_oracle.c).

TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's
CPU-baseline leg use it to check and time the CUDA library; the product path
never imports it, and it imports nothing from the product package.

Every function here marshals numpy arrays into the C oracle; the arithmetic
lives in kda_oracle.c (sequential per token, double precision, following the
"KDA per-head recurrence" block of the kimi_k3.c header comment).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libkda_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile kda_oracle.c with gcc (portable C99, no FMA contraction, OpenMP)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC),
                                              os.path.getmtime(os.path.join(_HERE, "kda_oracle.h")))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=gnu99", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fopenmp",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("d", ctypes.c_int), ("K", ctypes.c_int),
                ("gate_lb", ctypes.c_double), ("l2_eps", ctypes.c_double),
                ("rms_eps", ctypes.c_double), ("q_scale", ctypes.c_double)]


@dataclass
class OracleCfg:
    H: int
    d: int
    K: int = 4
    gate_lb: float = -5.0
    l2_eps: float = 1e-6
    rms_eps: float = 1e-6
    q_scale: float | None = None  # default d^-1/2

    def c(self) -> _Cfg:
        qs = self.q_scale if self.q_scale is not None else self.d ** -0.5
        return _Cfg(self.H, self.d, self.K, self.gate_lb, self.l2_eps, self.rms_eps, qs)


_D = ctypes.POINTER(ctypes.c_double)
_F = ctypes.POINTER(ctypes.c_float)
_I = ctypes.POINTER(ctypes.c_int32)


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        # KDA_ORACLE_LIB lets the mutation test load a deliberately broken copy
        alt = os.environ.get("KDA_ORACLE_LIB")
        _lib = ctypes.CDLL(alt if alt else build())
        L = _lib
        L.kdao_sigmoid.restype = ctypes.c_double
        L.kdao_sigmoid.argtypes = [ctypes.c_double]
        L.kdao_silu.restype = ctypes.c_double
        L.kdao_silu.argtypes = [ctypes.c_double]
        L.kdao_conv_silu.restype = ctypes.c_double
        L.kdao_conv_silu.argtypes = [ctypes.c_int, _D, _D, ctypes.c_double]
        L.kdao_l2norm.restype = None
        L.kdao_l2norm.argtypes = [ctypes.c_int, _D, ctypes.c_double, ctypes.c_double, _D]
        L.kdao_gate_alpha.restype = ctypes.c_double
        L.kdao_gate_alpha.argtypes = [ctypes.c_double] * 4 + [_D]
        L.kdao_delta_step.restype = None
        L.kdao_delta_step.argtypes = [ctypes.c_int, _D, _D, ctypes.c_double, _D, _D, _D, _D]
        L.kdao_rmsnorm_gate.restype = None
        L.kdao_rmsnorm_gate.argtypes = [ctypes.c_int, _D, _D, _D, ctypes.c_double, _D]
        L.kdao_unit.restype = None
        L.kdao_unit.argtypes = [ctypes.POINTER(_Cfg), ctypes.c_int, _F, _F, _F, _F, _D, _D,
                                ctypes.c_long, ctypes.c_int, _F, _F, _F, _F, _F, ctypes.c_long,
                                _F, ctypes.c_long, _D, ctypes.c_long]
        L.kdao_sequence.restype = None
        L.kdao_sequence.argtypes = [ctypes.POINTER(_Cfg), _F, _F, _F, _F, _D, _D, ctypes.c_int,
                                    _F, _F, _F, _F, _F, _F, _D, ctypes.c_int]
        L.kdao_decode_batch.restype = None
        L.kdao_decode_batch.argtypes = [ctypes.POINTER(_Cfg), _F, _F, _F, _F, _D, _D, _I,
                                        ctypes.c_int, _F, _F, _F, _F, _F, _F, _D, ctypes.c_int]
        L.kdao_max_threads.restype = ctypes.c_int
        L.kdao_max_threads.argtypes = []
    return _lib


def _f(a: np.ndarray):
    assert a.dtype == np.float32 and a.flags.c_contiguous
    return a.ctypes.data_as(_F)


def _d(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_D)


def _dv(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


# ---------------- single-step helpers ----------------

def sigmoid(x: float) -> float:
    return lib().kdao_sigmoid(float(x))


def silu(x: float) -> float:
    return lib().kdao_silu(float(x))


def conv_silu(taps, hist, x: float) -> float:
    taps = _dv(taps)
    hist = _dv(hist) if len(hist) else np.zeros(1)
    return lib().kdao_conv_silu(len(taps), _d(taps), _d(hist), float(x))


def l2norm(x, eps: float = 1e-6, scale: float = 1.0) -> np.ndarray:
    x = _dv(x)
    y = np.empty_like(x)
    lib().kdao_l2norm(len(x), _d(x), eps, scale, _d(y))
    return y


def gate_alpha(A_log: float, z: float, dt: float, gmin: float = -5.0):
    gk = ctypes.c_double()
    a = lib().kdao_gate_alpha(float(A_log), float(z), float(dt), float(gmin), ctypes.byref(gk))
    return a, gk.value


def delta_step(S: np.ndarray, alpha, beta: float, k, v, q) -> np.ndarray:
    """Advance S ([d, d] float64, in place) by one token; returns o = S'^T q."""
    d = S.shape[0]
    assert S.dtype == np.float64 and S.flags.c_contiguous and S.shape == (d, d)
    alpha, k, v, q = _dv(alpha), _dv(k), _dv(v), _dv(q)
    o = np.empty(d)
    lib().kdao_delta_step(d, _d(S), _d(alpha), float(beta), _d(k), _d(v), _d(q), _d(o))
    return o


def rmsnorm_gate(o, w, g, eps: float = 1e-6) -> np.ndarray:
    o, w, g = _dv(o), _dv(w), _dv(g)
    out = np.empty_like(o)
    lib().kdao_rmsnorm_gate(len(o), _d(o), _d(w), _d(g), eps, _d(out))
    return out


# ---------------- whole-path drivers ----------------

def _params_ptrs(p):
    for a in (p.conv_w, p.dt_bias, p.A_log, p.norm_w):
        assert a.dtype == np.float32 and a.flags.c_contiguous
    return _f(p.conv_w), _f(p.dt_bias), _f(p.A_log), _f(p.norm_w)


def new_state(cfg: OracleCfg, n: int | None = None):
    """Zero state [H, d, d] and conv history [3, K-1, H*d] in float64 (n: leading slot dim)."""
    D = cfg.H * cfg.d
    if n is None:
        return np.zeros((cfg.H, cfg.d, cfg.d)), np.zeros((3, cfg.K - 1, D))
    return np.zeros((n, cfg.H, cfg.d, cfg.d)), np.zeros((n, 3, cfg.K - 1, D))


def sequence(cfg: OracleCfg, params, S: np.ndarray, tail: np.ndarray, tok: dict,
             nthreads: int = 0) -> np.ndarray:
    """Run T tokens of one sequence; S [H,d,d] and tail [3,K-1,D] (float64) advance in place.

    tok holds float32 arrays q,k,v,z,g [T, D] and b [T, H]. Returns out [T, D] float64.
    """
    H, d, K = cfg.H, cfg.d, cfg.K
    D = H * d
    T = tok["q"].shape[0]
    assert S.shape == (H, d, d) and tail.shape == (3, K - 1, D)
    arrs = [np.ascontiguousarray(tok[n], dtype=np.float32) for n in ("q", "k", "v", "z", "b", "g")]
    out = np.empty((T, D))
    nt = nthreads if nthreads > 0 else lib().kdao_max_threads()
    c = cfg.c()
    lib().kdao_sequence(ctypes.byref(c), *_params_ptrs(params), _d(S), _d(tail), T,
                        *[_f(a) for a in arrs], _d(out), nt)
    return out


def decode_batch(cfg: OracleCfg, params, S_all: np.ndarray, tail_all: np.ndarray, slots,
                 tok: dict, nthreads: int = 0) -> np.ndarray:
    """One token for each of B sequences; row r advances slot slots[r] of S_all / tail_all."""
    H, d, K = cfg.H, cfg.d, cfg.K
    D = H * d
    B = tok["q"].shape[0]
    slots = np.ascontiguousarray(slots, dtype=np.int32)
    assert slots.shape == (B,)
    assert S_all.shape[1:] == (H, d, d) and tail_all.shape[1:] == (3, K - 1, D)
    assert slots.min() >= 0 and slots.max() < S_all.shape[0]
    arrs = [np.ascontiguousarray(tok[n], dtype=np.float32) for n in ("q", "k", "v", "z", "b", "g")]
    out = np.empty((B, D))
    nt = nthreads if nthreads > 0 else lib().kdao_max_threads()
    c = cfg.c()
    lib().kdao_decode_batch(ctypes.byref(c), *_params_ptrs(params), _d(S_all), _d(tail_all),
                            slots.ctypes.data_as(_I), B, *[_f(a) for a in arrs], _d(out), nt)
    return out


def unit(cfg: OracleCfg, h: int, params, S_h: np.ndarray, tail_seq: np.ndarray, tok: dict,
         rows=None) -> np.ndarray:
    """Advance head h of one sequence over the given token rows (default: all).

    S_h is that head's [d, d] float64 state (in place); tail_seq the sequence's whole
    [3, K-1, D] float64 history (only head h's channels change). Returns [T, d].
    """
    H, d, K = cfg.H, cfg.d, cfg.K
    D = H * d
    arrs = {n: np.ascontiguousarray(tok[n] if rows is None else tok[n][rows], dtype=np.float32)
            for n in ("q", "k", "v", "z", "b", "g")}
    T = arrs["q"].shape[0]
    assert S_h.shape == (d, d) and S_h.dtype == np.float64 and S_h.flags.c_contiguous
    assert tail_seq.shape == (3, K - 1, D) and tail_seq.flags.c_contiguous
    out = np.empty((T, d))
    c = cfg.c()
    off_f = h * d * 4
    off_d = h * d * 8

    def fp(a, off):
        return ctypes.cast(a.ctypes.data + off, _F)

    lib().kdao_unit(ctypes.byref(c), h, *_params_ptrs(params), _d(S_h),
                    ctypes.cast(tail_seq.ctypes.data + off_d, _D), D, T,
                    fp(arrs["q"], off_f), fp(arrs["k"], off_f), fp(arrs["v"], off_f),
                    fp(arrs["z"], off_f), fp(arrs["g"], off_f), D,
                    fp(arrs["b"], h * 4), H, _d(out), d)
    return out


def max_threads() -> int:
    return lib().kdao_max_threads()
