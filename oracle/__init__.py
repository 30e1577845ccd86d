"""Plain fp64 CPU oracle for Laplacian-kernel Nystrom attention.

TEST INFRASTRUCTURE ONLY.  This package is the independent reference the CUDA library is
checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the library under ``laplacian_nystr_attention_gb300/`` never does,
and this package imports nothing from there.

The arithmetic lives in ``lapl_oracle.c`` (plain loops in double precision, one function per
step of the method, each citing the explainer page it follows).  This module only builds that
file with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lapl_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liblapl_oracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: no fused multiply-add contraction, so x86 and Arm hosts round alike.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile ``lapl_oracle.c`` into ``liblapl_oracle.so`` next to it; return the path."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                          os.path.getmtime(os.path.join(_HERE, "lapl_oracle.h")))):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Config(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int), ("heads", ctypes.c_int),
        ("grid_h", ctypes.c_int), ("grid_w", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("num_landmarks", ctypes.c_int),
        ("lam", ctypes.c_double), ("eps", ctypes.c_double), ("delta", ctypes.c_double),
        ("ns_steps", ctypes.c_int), ("whiten", ctypes.c_int), ("kernel", ctypes.c_int),
        ("solver", ctypes.c_int),
    ]


_DP = ctypes.POINTER(ctypes.c_double)
_INTERMEDIATES = ["landmarks", "d_ql", "d_ll", "d_lk", "a", "b", "w", "x", "mu", "var",
                  "a_hat", "bv", "m_mat", "ns_resid"]


class _Intermediates(ctypes.Structure):
    _fields_ = [(name, _DP) for name in _INTERMEDIATES]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            for fn in (lib.orc_forward_slices, lib.orc_backward_slices):
                fn.restype = ctypes.c_int
            lib.orc_forward_slices.argtypes = [
                ctypes.POINTER(_Config), _DP, _DP, _DP, _DP, _DP,
                ctypes.POINTER(_Intermediates), ctypes.c_long, ctypes.c_long]
            lib.orc_backward_slices.argtypes = [
                ctypes.POINTER(_Config), _DP, _DP, _DP, _DP, _DP, _DP, _DP, _DP, _DP, _DP, _DP,
                ctypes.c_double, ctypes.c_long, ctypes.c_long]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_DP)


def _as_f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


class OracleError(RuntimeError):
    pass


def _config(cfg: dict) -> _Config:
    return _Config(int(cfg["batch"]), int(cfg["heads"]), int(cfg["grid_h"]), int(cfg["grid_w"]),
                   int(cfg["head_dim"]), int(cfg["num_landmarks"]), float(cfg["lam"]),
                   float(cfg["eps"]), float(cfg["delta"]), int(cfg["ns_steps"]),
                   int(cfg["whiten"]), int(cfg.get("kernel", 0)), int(cfg.get("solver", 0)))


def backward(cfg: dict, q, k, v, dout, bias=None, slices=None, tau: float = 2.0 ** -15):
    """Gradients of a loss with dLoss/dO = dout, through the whole forward (the chain rule
    step by step; see the C source).

    Returns (dq, dk, dv, dbias, amb_dq, amb_dk): float64 arrays [B,H,N,d] (zero outside the
    requested slices), dbias [H,m] (summed over the requested slices' batches), and for the
    Laplacian kernel the bounds on how far each dq / dk entry can move when a sign decision
    sgn(x - y) with |x - y| <= tau (|x| + |y|) is taken the other way (zeros otherwise)."""
    B, H = int(cfg["batch"]), int(cfg["heads"])
    N = int(cfg["grid_h"]) * int(cfg["grid_w"])
    d, m = int(cfg["head_dim"]), int(cfg["num_landmarks"])
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    for t in (q, k, v, dout):
        if t.shape != (B, H, N, d):
            raise ValueError(f"expected [B,H,N,d]={(B, H, N, d)}, got {t.shape}")
    bias = None if bias is None else _as_f64(bias)
    outs = [np.zeros((B, H, N, d)) for _ in range(5)]
    dbias = np.zeros((H, m))
    begin, count = (0, B * H) if slices is None else (int(slices[0]), int(slices[1]))
    c = _config(cfg)
    dq, dk, dv, aq, ak = outs
    rc = _load().orc_backward_slices(ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(bias),
                                     _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias),
                                     _ptr(aq), _ptr(ak), float(tau), begin, count)
    if rc != 0:
        raise OracleError(f"oracle backward returned status {rc}")
    return dq, dk, dv, dbias, aq, ak


def forward(cfg: dict, q, k, v, bias=None, intermediates: bool = False, slices=None):
    """Run the oracle.

    cfg: dict with batch, heads, grid_h, grid_w, head_dim, num_landmarks, lam, eps, delta,
    ns_steps, whiten, and optionally kernel (0 Laplacian, the default; 1 Gaussian) and solver
    (0 Newton-Schulz, the default; 1 conjugate gradient, ns_steps iterations).  q, k, v:
    [B,H,N,d] (converted exactly to float64).  bias: [H,m] or None.
    slices: None for all (b,h) slices, else (begin, count) over s = b*H + h; outputs of other
    slices are left at zero.  Returns (out, inter) where inter is a dict of float64 arrays
    (empty unless ``intermediates``).
    """
    B, H = int(cfg["batch"]), int(cfg["heads"])
    N = int(cfg["grid_h"]) * int(cfg["grid_w"])
    d, m, T = int(cfg["head_dim"]), int(cfg["num_landmarks"]), int(cfg["ns_steps"])
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    for t in (q, k, v):
        if t.shape != (B, H, N, d):
            raise ValueError(f"expected [B,H,N,d]={(B, H, N, d)}, got {t.shape}")
    bias = None if bias is None else _as_f64(bias)
    if bias is not None and bias.shape != (H, m):
        raise ValueError(f"bias must be [H,m]={(H, m)}, got {bias.shape}")
    out = np.zeros((B, H, N, d), dtype=np.float64)
    shapes = {
        "landmarks": (B, H, m, d), "d_ql": (B, H, N, m), "d_ll": (B, H, m, m),
        "d_lk": (B, H, m, N), "a": (B, H, N, m), "b": (B, H, m, N), "w": (B, H, m, m),
        "x": (B, H, m, m), "mu": (B, H, m), "var": (B, H, m), "a_hat": (B, H, N, m),
        "bv": (B, H, m, d), "m_mat": (B, H, m, d), "ns_resid": (B, H, T + 1),
    }
    inter = {}
    im = None
    if intermediates:
        inter = {name: np.zeros(shapes[name], dtype=np.float64) for name in _INTERMEDIATES}
        im = _Intermediates(**{name: _ptr(inter[name]) for name in _INTERMEDIATES})
    c = _config(cfg)
    begin, count = (0, B * H) if slices is None else (int(slices[0]), int(slices[1]))
    rc = _load().orc_forward_slices(ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(bias),
                                    _ptr(out), ctypes.byref(im) if im is not None else None,
                                    begin, count)
    if rc != 0:
        raise OracleError(f"oracle returned status {rc}")
    return out, inter
