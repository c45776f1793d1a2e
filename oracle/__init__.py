"""fmlp oracle: plain fp64 CPU implementation of the feed-forward block (C, via ctypes).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the package smoke check and by the
benchmark's CPU-baseline leg, never by the library. The arithmetic lives in
fmlp_oracle.c (plain loops, double precision, bf16 rounding only where the fused path
rounds); this wrapper only marshals numpy arrays of bf16 bit patterns.

Parity pins (tests/test_oracle.py): GELU against the normal CDF table and torch's fp64
GELU, ReLU against torch's relu, the MoE block against torch per expert and against the plain
block when every expert holds the same weights, the page's nn.Linear layout worked example, identity/zero weights, special cases with
distinguishable operands, rounding against an independent exact rounding, and brute force
against torch's fp64 nn.Linear / F.gelu on tiny shapes. No function here is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

GELU_TANH = 0
GELU_ERF = 1
RELU = 2        # the MLP's hidden activation may also be ReLU

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile fmlp_oracle.c with gcc (no fast-math, no FP contraction)."""
    src = os.path.join(_HERE, "fmlp_oracle.c")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src)):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                           "-ffp-contract=off", "-o", tmp, src, "-lm", "-lpthread"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_gelu.argtypes = [_P, _P, _I64, ctypes.c_int]
            lib.oracle_gelu.restype = None
            lib.oracle_linear.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _I64,
                                          ctypes.c_int]
            lib.oracle_linear.restype = ctypes.c_int
            lib.oracle_mlp_gelu.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64,
                                            _I64, ctypes.c_int, ctypes.c_int, _P, _I64,
                                            ctypes.c_int]
            lib.oracle_mlp_gelu.restype = ctypes.c_int
            lib.oracle_geglu.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64,
                                         ctypes.c_int, _P, _I64, ctypes.c_int]
            lib.oracle_geglu.restype = ctypes.c_int
            _lib = lib
    return _lib


def threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def _ptr(a):
    if a is None:
        return None
    assert a.flags.c_contiguous, "oracle inputs must be contiguous"
    return a.ctypes.data


def _u16(a, shape=None):
    a = np.ascontiguousarray(a, dtype=np.uint16)
    if shape is not None:
        assert a.shape == tuple(shape), (a.shape, shape)
    return a


def _rows(rows, T):
    if rows is None:
        return None, T
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    assert r.ndim == 1 and (r.size == 0 or (r.min() >= 0 and r.max() < T))
    return r, r.size


def round_bf16(v: float) -> int:
    """bf16 bit pattern nearest to the double v (ties to even)."""
    return int(_load().oracle_round_bf16(float(v)))


def gelu(x: np.ndarray, mode: int = GELU_TANH) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    _load().oracle_gelu(_ptr(x), _ptr(out), x.size, mode)
    return out



def moe_geglu(x, offsets, Wg, Wu, Wd, want_m=False, nthreads=None, rows=None):
    """Mixture-of-experts feed-forward (the ainews.cool article's MoE note: every expert is an
    MLP): tokens arrive grouped by expert, rows [offsets[e], offsets[e+1]) of x go through
    expert e's GeGLU block with Wg[e], Wu[e] [H, D] and Wd[e] [D, H]. Each expert's rows are
    exactly geglu() on those rows; nothing else is computed. rows: optional sorted token-row
    indices; then only those rows are computed and returned, in that order."""
    x = _u16(x)
    T, D = x.shape
    offsets = np.asarray(offsets, dtype=np.int64)
    E = offsets.size - 1
    if E < 1 or offsets[0] != 0 or offsets[-1] != T or np.any(np.diff(offsets) < 0):
        raise ValueError("offsets must rise from 0 to T")
    H = Wg.shape[1]
    sel = np.arange(T, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    if sel.size and (np.any(np.diff(sel) <= 0) or sel[0] < 0 or sel[-1] >= T):
        raise ValueError("rows must be sorted, unique and inside [0, T)")
    y = np.empty((sel.size, D), dtype=np.uint16)
    m = np.empty((sel.size, H), dtype=np.uint16)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        lo, hi = np.searchsorted(sel, a), np.searchsorted(sel, b)
        if b == a or hi == lo:
            continue
        ye, me = geglu(x[a:b], Wg[e], Wu[e], Wd[e], want_m=True, nthreads=nthreads,
                       rows=sel[lo:hi] - a)
        y[lo:hi], m[lo:hi] = ye, me
    return (y, m) if want_m else y

def linear(x, W, b, rows=None, nthreads=None, want_acc=False):
    """y = bf16(x W^T + b) for the selected rows; returns bf16 bits (and fp64 pre-round)."""
    T, K = x.shape
    N = W.shape[0]
    x, W = _u16(x), _u16(W, (N, K))
    b = None if b is None else _u16(b, (N,))
    r, n = _rows(rows, T)
    y = np.empty((n, N), dtype=np.uint16)
    acc = np.empty((n, N), dtype=np.float64) if want_acc else None
    rc = _load().oracle_linear(_ptr(x), _ptr(W), _ptr(b), _ptr(y), _ptr(acc), T, K, N,
                               _ptr(r), n, nthreads or threads())
    if rc != 0:
        raise RuntimeError(f"oracle_linear failed ({rc})")
    return (y, acc) if want_acc else y


def mlp_gelu(x, W1, b1, W2, b2, gelu_mode=GELU_ERF, eager=False, rows=None, nthreads=None,
             want_acc=False, want_h=False):
    """h = bf16(GELU(x W1^T + b1)); y = bf16(h W2^T + b2)."""
    T, D = x.shape
    H = W1.shape[0]
    Dout = W2.shape[0]
    x, W1, W2 = _u16(x), _u16(W1, (H, D)), _u16(W2, (Dout, H))
    b1 = None if b1 is None else _u16(b1, (H,))
    b2 = None if b2 is None else _u16(b2, (Dout,))
    r, n = _rows(rows, T)
    y = np.empty((n, Dout), dtype=np.uint16)
    acc = np.empty((n, Dout), dtype=np.float64) if want_acc else None
    h = np.empty((n, H), dtype=np.uint16) if want_h else None
    rc = _load().oracle_mlp_gelu(_ptr(x), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), _ptr(y),
                                 _ptr(acc), _ptr(h), T, D, H, Dout, int(gelu_mode),
                                 int(bool(eager)), _ptr(r), n, nthreads or threads())
    if rc != 0:
        raise RuntimeError(f"oracle_mlp_gelu failed ({rc})")
    out = [y]
    if want_acc:
        out.append(acc)
    if want_h:
        out.append(h)
    return out[0] if len(out) == 1 else tuple(out)


def geglu(x, Wg, Wu, Wd, eager=False, rows=None, nthreads=None, want_acc=False, want_m=False):
    """m = bf16(gelu_tanh(x Wg^T) * (x Wu^T)); y = bf16(m Wd^T)."""
    T, D = x.shape
    H = Wg.shape[0]
    x, Wg, Wu, Wd = _u16(x), _u16(Wg, (H, D)), _u16(Wu, (H, D)), _u16(Wd, (D, H))
    r, n = _rows(rows, T)
    y = np.empty((n, D), dtype=np.uint16)
    acc = np.empty((n, D), dtype=np.float64) if want_acc else None
    m = np.empty((n, H), dtype=np.uint16) if want_m else None
    rc = _load().oracle_geglu(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(y), _ptr(acc),
                              _ptr(m), T, D, H, int(bool(eager)), _ptr(r), n,
                              nthreads or threads())
    if rc != 0:
        raise RuntimeError(f"oracle_geglu failed ({rc})")
    out = [y]
    if want_acc:
        out.append(acc)
    if want_m:
        out.append(m)
    return out[0] if len(out) == 1 else tuple(out)
