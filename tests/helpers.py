"""Test helpers: an exact bf16 rounding written independently of the oracle, fp64 torch
references of the pages' modules, and the parity tolerance check.

The tolerance: per element |y - ref| <= 2e-2 * max(1, |ref|), and the relative Frobenius
error ||y - ref||_F / ||ref||_F <= 5e-3.
"""
from __future__ import annotations

import math
import struct

import numpy as np
import torch

ELEM_TOL = 2e-2
FROB_TOL = 5e-3


def rne_bf16_bits(v: float) -> int:
    """Nearest bf16 (ties to even) via frexp and Python's round-half-even on an exact
    scaled significand. Valid for finite values inside bf16's normal range and zero."""
    if v == 0.0:
        return 0x8000 if math.copysign(1.0, v) < 0 else 0
    m, e = math.frexp(abs(v))          # |v| = m 2^e, m in [0.5, 1)
    r = round(m * 256.0)               # exact product, banker's rounding
    q = math.ldexp(r, e - 8)
    bits = struct.unpack("<I", struct.pack("<f", q))[0] >> 16
    return bits | (0x8000 if v < 0 else 0)


def rne_bf16_array(a: np.ndarray) -> np.ndarray:
    flat = np.asarray(a, dtype=np.float64).ravel()
    return np.array([rne_bf16_bits(float(v)) for v in flat], dtype=np.uint16).reshape(np.shape(a))


def bits_to_f64(a: np.ndarray) -> np.ndarray:
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bits_via_torch(a: np.ndarray) -> np.ndarray:
    """bf16 bits of float64 values that are exactly representable in float32 (torch's own
    float -> bfloat16 conversion, ties to even)."""
    t = torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def t64(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(bits_to_f64(bits))


def torch_geglu_f64(x, Wg, Wu, Wd, round_m: bool = True):
    """The page's SimpleGeGLUMLP forward evaluated by torch in float64 on the CPU, with the
    intermediate m rounded to bf16 once (the fused path's single rounding).
    Returns (y_before_rounding, m_bits)."""
    xf, wg, wu, wd = t64(x), t64(Wg), t64(Wu), t64(Wd)
    g = torch.nn.functional.linear(xf, wg)
    u = torch.nn.functional.linear(xf, wu)
    h = torch.nn.functional.gelu(g, approximate="tanh")
    m = (h * u).numpy()
    m_bits = rne_bf16_array(m) if round_m else None
    mr = torch.from_numpy(bits_to_f64(m_bits)) if round_m else torch.from_numpy(m)
    y = torch.nn.functional.linear(mr, wd)
    return y.numpy(), m_bits


def torch_mlp_f64(x, W1, b1, W2, b2, approximate: str):
    xf, w1, w2 = t64(x), t64(W1), t64(W2)
    z = torch.nn.functional.linear(xf, w1, None if b1 is None else t64(b1))
    h = (torch.relu(z) if approximate == "relu"
         else torch.nn.functional.gelu(z, approximate=approximate)).numpy()
    h_bits = rne_bf16_array(h)
    y = torch.nn.functional.linear(torch.from_numpy(bits_to_f64(h_bits)), w2,
                                   None if b2 is None else t64(b2))
    return y.numpy(), h_bits


def _rne_t(t: torch.Tensor) -> torch.Tensor:
    """Round a float64 tensor to bf16 values with the independent rounding above."""
    return torch.from_numpy(bits_to_f64(rne_bf16_array(t.numpy())))


def torch_geglu_eager_f64(x, Wg, Wu, Wd):
    """The page's SimpleGeGLUMLP as eager PyTorch runs it in bf16: every tensor the module
    materialises (g, u, gelu(g), m) is rounded to bf16; products and sums in float64 by torch.
    Returns (y_before_rounding, m_bits)."""
    xf, wg, wu, wd = t64(x), t64(Wg), t64(Wu), t64(Wd)
    g = _rne_t(torch.nn.functional.linear(xf, wg))
    u = _rne_t(torch.nn.functional.linear(xf, wu))
    h = _rne_t(torch.nn.functional.gelu(g, approximate="tanh"))
    m = _rne_t(h * u)
    y = torch.nn.functional.linear(m, wd)
    return y.numpy(), rne_bf16_array(m.numpy())


def torch_mlp_eager_f64(x, W1, b1, W2, b2, approximate: str):
    """Linear -> activation -> Linear as eager PyTorch runs it in bf16: the first Linear's
    output (bias included) and the activation's output are each rounded to bf16.
    Returns (y_before_rounding, h_bits)."""
    xf, w1, w2 = t64(x), t64(W1), t64(W2)
    z = _rne_t(torch.nn.functional.linear(xf, w1, None if b1 is None else t64(b1)))
    h = _rne_t(torch.relu(z) if approximate == "relu"
               else torch.nn.functional.gelu(z, approximate=approximate))
    y = torch.nn.functional.linear(h, w2, None if b2 is None else t64(b2))
    return y.numpy(), rne_bf16_array(h.numpy())


def parity_stats(y_bits: np.ndarray, ref_bits: np.ndarray) -> dict:
    y = bits_to_f64(y_bits)
    r = bits_to_f64(ref_bits)
    assert y.shape == r.shape, (y.shape, r.shape)
    err = np.abs(y - r)
    bound = ELEM_TOL * np.maximum(1.0, np.abs(r))
    nref = float(np.linalg.norm(r))
    frob = float(np.linalg.norm(y - r)) / nref if nref > 0 else float(np.linalg.norm(y - r))
    ulp = np.abs(np.asarray(y_bits, np.int32) - np.asarray(ref_bits, np.int32))
    return {
        "max_abs": float(err.max()) if err.size else 0.0,
        "n_elem_fail": int((err > bound).sum()),
        "frob_rel": frob,
        "finite": bool(np.isfinite(y).all()),
        "mismatch_bits": int((np.asarray(y_bits) != np.asarray(ref_bits)).sum()),
        "max_ulp": int(ulp.max()) if ulp.size else 0,
        "n": int(y.size),
    }


def assert_parity(y_bits, ref_bits, what=""):
    s = parity_stats(y_bits, ref_bits)
    assert s["finite"], f"{what}: non-finite output {s}"
    assert s["n_elem_fail"] == 0, f"{what}: per-element tolerance exceeded {s}"
    assert s["frob_rel"] <= FROB_TOL, f"{what}: Frobenius tolerance exceeded {s}"
    return s
