"""ctypes front-end of the fp64 CPU oracle (``k3moe_oracle.c``).

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg may use it; the product path never does.  It imports nothing
from the CUDA package: callers hand it numpy arrays drawn by the seeded
generator.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k3moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(C.Structure):
    _fields_ = [("H", C.c_int), ("L", C.c_int), ("E", C.c_int), ("K", C.c_int),
                ("I", C.c_int), ("S", C.c_int), ("rms_eps", C.c_double),
                ("routed_scaling", C.c_double), ("router_bf16", C.c_int), ("has_bias", C.c_int),
                ("act", C.c_int), ("situ_beta", C.c_double), ("situ_linear_beta", C.c_double),
                ("a8", C.c_int)]


_PP = C.POINTER(C.c_void_p)


class _W(C.Structure):
    _fields_ = [("w_router", C.c_void_p), ("bias", C.c_void_p), ("w_down", C.c_void_p),
                ("w_up", C.c_void_p), ("gamma", C.c_void_p),
                ("w1p", _PP), ("w1s", _PP), ("w3p", _PP), ("w3s", _PP), ("w2p", _PP), ("w2s", _PP),
                ("ws1p", C.c_void_p), ("ws1s", C.c_void_p), ("ws3p", C.c_void_p),
                ("ws3s", C.c_void_p), ("ws2p", C.c_void_p), ("ws2s", C.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            d = C.c_double
            _lib.oracle_bf16.restype = d
            _lib.oracle_bf16.argtypes = [C.c_uint16]
            _lib.oracle_e2m1.restype = d
            _lib.oracle_e2m1.argtypes = [C.c_uint]
            _lib.oracle_e8m0.restype = d
            _lib.oracle_e8m0.argtypes = [C.c_uint]
            _lib.oracle_dequant_row.restype = None
            _lib.oracle_dequant_row.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_void_p]
            _lib.oracle_route.restype = None
            _lib.oracle_route.argtypes = [C.POINTER(_Cfg), C.POINTER(_W), C.c_void_p, C.c_void_p,
                                          C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                          C.c_int]
            _lib.oracle_forward.restype = C.c_int
            _lib.oracle_forward.argtypes = [C.POINTER(_Cfg), C.POINTER(_W), C.c_void_p, C.c_void_p,
                                            C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                            C.c_void_p, C.c_void_p, C.c_int]
            _lib.oracle_max_threads.restype = C.c_int
            _lib.oracle_act.restype = d
            _lib.oracle_act.argtypes = [C.c_int, d, d, d, d]
            _lib.oracle_round_bf16.restype = d
            _lib.oracle_round_bf16.argtypes = [d]
            _lib.oracle_e4m3.restype = d
            _lib.oracle_e4m3.argtypes = [d]
            _lib.oracle_mxfp8_row.restype = None
            _lib.oracle_mxfp8_row.argtypes = [C.c_void_p, C.c_int, C.c_void_p]
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def e2m1(code: int) -> float:
    return lib().oracle_e2m1(code)


def e8m0(e: int) -> float:
    return lib().oracle_e8m0(e)


def bf16(bits: int) -> float:
    return lib().oracle_bf16(bits)


def dequant(packed: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Dequantise an MXFP4 matrix [rows, cols] (fp64)."""
    packed = np.ascontiguousarray(packed, np.uint8)
    scale = np.ascontiguousarray(scale, np.uint8)
    rows, cols = packed.shape[0], packed.shape[1] * 2
    out = np.empty((rows, cols), np.float64)
    L = lib()
    for r in range(rows):
        L.oracle_dequant_row(packed[r].ctypes.data, scale[r].ctypes.data, cols,
                             out[r].ctypes.data)
    return out


def max_threads() -> int:
    return lib().oracle_max_threads()


class _Keep:
    """Holds numpy arrays alive while a C call uses pointers into them."""

    def __init__(self):
        self.items = []

    def __call__(self, a):
        if a is not None:
            self.items.append(a)
        return a


def _cfg(cfg) -> _Cfg:
    act = {"silu": 0, "situ": 1}[getattr(cfg, "act", "silu")]
    return _Cfg(cfg.H, cfg.L, cfg.E, cfg.K, cfg.I, cfg.S, cfg.rms_eps, cfg.routed_scaling,
                1 if cfg.router_dtype == "bf16" else 0, 1 if cfg.select_bias else 0, act,
                getattr(cfg, "situ_beta", 4.0), getattr(cfg, "situ_linear_beta", 25.0),
                1 if getattr(cfg, "a8", False) else 0)


def _weights(cfg, dense, experts, keep) -> _W:
    arr = lambda n: (C.c_void_p * n)()
    tabs = [arr(cfg.E) for _ in range(6)]
    for e, mats in (experts or {}).items():
        for m, (p, s) in enumerate(mats):
            p = keep(np.ascontiguousarray(p, np.uint8))
            s = keep(np.ascontiguousarray(s, np.uint8))
            tabs[2 * m][e] = p.ctypes.data
            tabs[2 * m + 1][e] = s.ctypes.data
    keep(tabs)
    c = lambda a: _ptr(keep(None if a is None else np.ascontiguousarray(a)))
    sh = [None] * 6
    if cfg.S and dense.shared is not None:
        sh = [c(a) for pair in dense.shared for a in pair]
    pp = lambda t: C.cast(t, _PP)
    return _W(c(dense.w_router), c(dense.select_bias), c(dense.w_down), c(dense.w_up),
              c(dense.gamma), pp(tabs[0]), pp(tabs[1]), pp(tabs[2]), pp(tabs[3]), pp(tabs[4]),
              pp(tabs[5]), *sh)


def act(kind: str, g, u, beta: float = 4.0, linear_beta: float = 25.0):
    """The oracle's GLU activation a(g, u) ("silu" or the "situ" reading), elementwise."""
    f = lib().oracle_act
    k = {"silu": 0, "situ": 1}[kind]
    g, u = np.broadcast_arrays(np.asarray(g, np.float64), np.asarray(u, np.float64))
    return np.array([f(k, beta, linear_beta, float(a), float(b)) for a, b in zip(g.ravel(), u.ravel())]
                    ).reshape(g.shape)


def mxfp8(x):
    """The oracle's MXFP8 rounding (step 6) of the last axis (length a multiple of 32)."""
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty_like(x)
    n = x.shape[-1]
    for xr, orow in zip(x.reshape(-1, n), out.reshape(-1, n)):
        lib().oracle_mxfp8_row(xr.ctypes.data, n, orow.ctypes.data)
    return out


def e4m3(v):
    f = lib().oracle_e4m3
    v = np.asarray(v, np.float64)
    return np.array([f(float(a)) for a in v.ravel()]).reshape(v.shape)


def round_bf16(v):
    f = lib().oracle_round_bf16
    v = np.asarray(v, np.float64)
    return np.array([f(float(a)) for a in v.ravel()]).reshape(v.shape)


def route(cfg, dense, x_rows: np.ndarray, nthreads: int = 0, want_logits: bool = False):
    """Route every row of ``x_rows`` [n, H] (BF16 bits).

    Returns (idx [n,K] int32, w [n,K] fp64, gap [n] fp64, logits [n,E] or None).
    """
    keep = _Keep()
    x_rows = keep(np.ascontiguousarray(x_rows, np.uint16))
    n = x_rows.shape[0]
    tok = keep(np.arange(n, dtype=np.int64))
    idx = np.empty((n, cfg.K), np.int32)
    w = np.empty((n, cfg.K), np.float64)
    gap = np.empty(n, np.float64)
    lg = np.empty((n, cfg.E), np.float64) if want_logits else None
    cc, ww = _cfg(cfg), _weights(cfg, dense, None, keep)
    lib().oracle_route(C.byref(cc), C.byref(ww), x_rows.ctypes.data, tok.ctypes.data, n,
                       idx.ctypes.data, w.ctypes.data, gap.ctypes.data, _ptr(lg), nthreads)
    return idx, w, gap, lg


def forward(cfg, dense, experts: dict, x_rows: np.ndarray, nthreads: int = 0,
            want_latent: bool = False):
    """Full fp64 forward of the rows of ``x_rows`` [n, H] (BF16 bits).

    ``experts`` maps expert index -> [(packed, scale)] for w1, w3, w2; it must
    hold every expert the rows select.  Returns a dict with out [n,H], idx,
    w, gap and, with ``want_latent``, h [n,L] and z [n,L].
    """
    keep = _Keep()
    x_rows = keep(np.ascontiguousarray(x_rows, np.uint16))
    n = x_rows.shape[0]
    tok = keep(np.arange(n, dtype=np.int64))
    out = np.zeros((n, cfg.H), np.float64)
    idx = np.empty((n, cfg.K), np.int32)
    w = np.empty((n, cfg.K), np.float64)
    gap = np.empty(n, np.float64)
    h = np.empty((n, cfg.L), np.float64) if want_latent else None
    z = np.empty((n, cfg.L), np.float64) if want_latent else None
    cc, ww = _cfg(cfg), _weights(cfg, dense, experts, keep)
    rc = lib().oracle_forward(C.byref(cc), C.byref(ww), x_rows.ctypes.data, tok.ctypes.data, n,
                              out.ctypes.data, idx.ctypes.data, w.ctypes.data, gap.ctypes.data,
                              _ptr(h), _ptr(z), nthreads)
    if rc == -1:
        raise KeyError("a selected expert's weights were not supplied")
    if rc == -2:
        raise ValueError("E8M0 scale 255 (NaN) in a selected expert")
    res = dict(out=out, idx=idx, w=w, gap=gap)
    if want_latent:
        res.update(h=h, z=z)
    return res


def touched_experts(idx: np.ndarray) -> np.ndarray:
    return np.unique(idx.reshape(-1))
