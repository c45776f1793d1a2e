"""Pins for the oracle, each against something other than the oracle itself.

Sources: "Profiling in PyTorch (Part 2): From nn.Linear to a Fused MLP" (sections "From
matmul-add to Linear", "Where did the transpose go? Kernel layouts and pre-ops", "Stacking
three Linears: the MLP") and the ainews.cool fused-MLP article (technical deep-dive). The
GELU formulas are Hendrycks & Gimpel (2016); the page names only approximate="tanh".
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from helpers import (bits_to_f64, f64_to_bits_via_torch, parity_stats, rne_bf16_array, t64, torch_geglu_eager_f64, torch_mlp_eager_f64,
                     rne_bf16_bits, torch_geglu_f64, torch_mlp_f64)
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def rand_bits(shape, scale=1.0):
    return rne_bf16_array(rng.standard_normal(shape) * scale)


# ---------------------------------------------------------------------------- rounding

def test_round_bf16_matches_exact_rounding():
    vals = list(rng.standard_normal(2000) * 10.0 ** rng.integers(-6, 6, 2000))
    # exact ties: a bf16 value plus exactly half an ulp (even and odd neighbours)
    for base in (1.0, 1.0078125, 3.0, -5.5, 1e-3, 96.0):
        m, e = math.frexp(abs(base))
        half = math.ldexp(1.0, e - 9)
        vals += [base + half, base - half, base + half * 1.000001, base + half * 0.999999]
    for v in vals:
        assert oracle.round_bf16(v) == rne_bf16_bits(v), v
    assert oracle.round_bf16(0.0) == 0 and oracle.round_bf16(-0.0) == 0x8000
    assert oracle.round_bf16(1e39) == 0x7F80 and oracle.round_bf16(-1e39) == 0xFF80
    assert oracle.round_bf16(float("nan")) == 0x7FC0


def test_round_bf16_matches_torch_on_float_values():
    v = (rng.standard_normal(5000) * 3).astype(np.float32).astype(np.float64)
    ours = np.array([oracle.round_bf16(float(a)) for a in v], dtype=np.uint16)
    assert np.array_equal(ours, f64_to_bits_via_torch(v))


# ---------------------------------------------------------------------------- GELU

# Standard normal CDF table values: Phi(0.5), Phi(1), Phi(2), Phi(3).
PHI_TABLE = {0.5: 0.6914624612740131, 1.0: 0.8413447460685429, 2.0: 0.9772498680518208,
             3.0: 0.9986501019683699}


def test_gelu_erf_is_x_times_normal_cdf():
    xs = np.array(sorted(PHI_TABLE))
    got = oracle.gelu(xs, oracle.GELU_ERF)
    for x, g in zip(xs, got):
        assert abs(g - x * PHI_TABLE[x]) <= 1e-15 * max(1, x)
        # Phi(-x) = 1 - Phi(x)
        gm = oracle.gelu(np.array([-x]), oracle.GELU_ERF)[0]
        assert abs(gm - (-x) * (1 - PHI_TABLE[x])) <= 1e-15


@pytest.mark.parametrize("mode", [oracle.GELU_TANH, oracle.GELU_ERF])
def test_gelu_identities(mode):
    xs = np.linspace(-8, 8, 1601)
    g = oracle.gelu(xs, mode)
    gn = oracle.gelu(-xs, mode)
    # gelu(x) - gelu(-x) = x for both flavours (0.5 x (1 + odd(x)) structure)
    assert np.max(np.abs((g - gn) - xs)) <= 1e-14
    assert oracle.gelu(np.array([0.0]), mode)[0] == 0.0
    big = oracle.gelu(np.array([10.0, -10.0]), mode)
    assert abs(big[0] - 10.0) < 1e-12 and abs(big[1]) < 1e-12


@pytest.mark.parametrize("approx,mode", [("tanh", oracle.GELU_TANH), ("none", oracle.GELU_ERF)])
def test_gelu_matches_torch_fp64(approx, mode):
    xs = np.concatenate([np.linspace(-8, 8, 3201), [-0.5, 0.5, -1, 1, -2, 2, -3, 3, -6, 6]])
    ref = torch.nn.functional.gelu(torch.from_numpy(xs), approximate=approx).numpy()
    got = oracle.gelu(xs, mode)
    assert np.max(np.abs(got - ref) / np.maximum(1, np.abs(ref))) <= 1e-15


def test_gelu_tanh_differs_from_erf_but_is_close():
    xs = np.linspace(-8, 8, 16001)
    d = np.abs(oracle.gelu(xs, oracle.GELU_TANH) - oracle.gelu(xs, oracle.GELU_ERF))
    assert d.max() <= 2e-3     # the tanh form approximates the exact GELU ...
    assert d.max() >= 1e-4     # ... but is a different function (catches a swapped mode)


# ---------------------------------------------------------------------------- Linear

def test_linear_layout_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "linear_layout_example.json")))
    M = torch.tensor(g["M"])
    assert list(M.shape) == g["M_shape"] and list(M.stride()) == g["M_stride"]
    T_ = M.t()
    assert list(T_.shape) == g["MT_shape"] and list(T_.stride()) == g["MT_stride"]
    assert T_.tolist() == g["MT"] and T_.flatten().tolist() == g["MT_flatten"]
    # nn.Linear(in=2, out=3) with weight = M stored [out, in]; y = x @ w.T + b
    W = np.array(g["M"], dtype=np.float64)
    x = np.array([[1.0, 10.0]])
    b = np.array([1.0, 1.0, 1.0])
    expect = [sum(x[0][k] * W[n][k] for k in range(2)) + b[n] for n in range(3)]
    assert expect == [11.0, 33.0, 55.0]
    y = oracle.linear(rne_bf16_array(x), rne_bf16_array(W), rne_bf16_array(b))
    assert bits_to_f64(y).tolist() == [expect]
    # reading the weight transposed ([in, out]) is a different operation: wrong shape
    with pytest.raises(AssertionError):
        oracle.linear(rne_bf16_array(x), rne_bf16_array(W.T.copy()), rne_bf16_array(b))


def test_linear_identity_and_zero_are_bit_exact():
    T, K = 37, 24
    x = rand_bits((T, K))
    b = rand_bits((K,), 0.5)
    eye = rne_bf16_array(np.eye(K))
    y = oracle.linear(x, eye, b)
    expect = rne_bf16_array(bits_to_f64(x) + bits_to_f64(b)[None, :])
    assert np.array_equal(y, expect)
    z = oracle.linear(x, np.zeros((16, K), np.uint16), b[:16])
    assert np.array_equal(z, np.broadcast_to(b[:16], (T, 16)))
    z0 = oracle.linear(x, np.zeros((16, K), np.uint16), None)
    assert np.all(bits_to_f64(z0) == 0)


@pytest.mark.parametrize("T,K,N", [(1, 8, 8), (3, 16, 72), (17, 72, 32), (129, 32, 16)])
def test_linear_brute_force_vs_torch(T, K, N):
    x, W, b = rand_bits((T, K)), rand_bits((N, K), 0.2), rand_bits((N,), 0.2)
    y, acc = oracle.linear(x, W, b, want_acc=True)
    ref = torch.nn.functional.linear(torch.from_numpy(bits_to_f64(x)),
                                     torch.from_numpy(bits_to_f64(W)),
                                     torch.from_numpy(bits_to_f64(b))).numpy()
    assert np.max(np.abs(acc - ref) / np.maximum(1e-300, np.abs(ref) + 1e-12)) <= 1e-12
    assert np.array_equal(y, rne_bf16_array(acc))


def test_row_subset_equals_full_rows():
    x, W, b = rand_bits((50, 16)), rand_bits((24, 16)), rand_bits((24,))
    full = oracle.linear(x, W, b)
    rows = np.array([0, 7, 7, 49, 13])
    assert np.array_equal(oracle.linear(x, W, b, rows=rows), full[rows])


# ---------------------------------------------------------------------------- GeGLU

@pytest.mark.parametrize("T,D,H", [(1, 8, 8), (3, 16, 72), (17, 32, 16), (129, 72, 32)])
def test_geglu_brute_force_vs_torch_module(T, D, H):
    x = rand_bits((T, D))
    Wg, Wu = rand_bits((H, D), 1 / math.sqrt(D)), rand_bits((H, D), 1 / math.sqrt(D))
    Wd = rand_bits((D, H), 1 / math.sqrt(H))
    y, acc, m = oracle.geglu(x, Wg, Wu, Wd, want_acc=True, want_m=True)
    ref_y, ref_m = torch_geglu_f64(x, Wg, Wu, Wd)
    # m is rounded once from a double; a tie-breaking difference would need an exact tie
    assert np.array_equal(m, ref_m)
    assert np.max(np.abs(acc - ref_y)) <= 1e-12 * max(1.0, np.abs(ref_y).max())
    assert np.array_equal(y, rne_bf16_array(acc))


def test_geglu_zero_gate_or_up_gives_zero():
    x = rand_bits((20, 16))
    W = rand_bits((32, 16))
    Wd = rand_bits((16, 32))
    zero = np.zeros((32, 16), np.uint16)
    assert np.all(bits_to_f64(oracle.geglu(x, zero, W, Wd)) == 0)   # gelu(0) = 0
    assert np.all(bits_to_f64(oracle.geglu(x, W, zero, Wd)) == 0)   # u = 0


def test_geglu_identity_weights_distinguish_gate_from_up():
    # D = H, Wg = I, Wu = 2I, Wd = I  =>  y = bf16(gelu_tanh(x) * 2x) elementwise.
    # Swapping gate and up would give gelu(2x) * x instead.
    D = 32
    x = rand_bits((40, D))
    eye = rne_bf16_array(np.eye(D))
    two = rne_bf16_array(2 * np.eye(D))
    y = oracle.geglu(x, eye, two, eye)
    xf = torch.from_numpy(bits_to_f64(x))
    expect = rne_bf16_array((torch.nn.functional.gelu(xf, approximate="tanh") * 2 * xf).numpy())
    assert np.array_equal(y, expect)
    swapped = rne_bf16_array((torch.nn.functional.gelu(2 * xf, approximate="tanh") * xf).numpy())
    assert not np.array_equal(y, swapped)


def test_geglu_eager_and_fused_rounding_both_within_tolerance():
    w = synth.WORKLOADS["geglu_1024x32x64"]
    t = w.generate()
    fused = oracle.geglu(t["x"], t["Wg"], t["Wu"], t["Wd"])
    eager = oracle.geglu(t["x"], t["Wg"], t["Wu"], t["Wd"], eager=True)
    s = parity_stats(eager, fused)
    assert s["n_elem_fail"] == 0 and s["frob_rel"] <= 5e-3, s
    assert s["mismatch_bits"] > 0    # the two readings do differ


@pytest.mark.parametrize("T,D,H", [(3, 16, 72), (33, 64, 48)])
def test_geglu_eager_rounding_vs_torch_module(T, D, H):
    """The eager-rounding reading (g, u, gelu(g) and m each rounded to bf16, as the eager
    module materialises them) against torch's float64 evaluation of the page's module with
    those roundings written out: m bit-equal, y's sum to 1e-12. Dropping any one of the four
    roundings changes m somewhere, which the bit comparison catches."""
    x = rand_bits((T, D))
    Wg, Wu = rand_bits((H, D), 1 / math.sqrt(D)), rand_bits((H, D), 1 / math.sqrt(D))
    Wd = rand_bits((D, H), 1 / math.sqrt(H))
    y, acc, m = oracle.geglu(x, Wg, Wu, Wd, eager=True, want_acc=True, want_m=True)
    ref_y, ref_m = torch_geglu_eager_f64(x, Wg, Wu, Wd)
    assert np.array_equal(m, ref_m)
    assert np.max(np.abs(acc - ref_y)) <= 1e-12 * max(1.0, np.abs(ref_y).max())
    assert np.array_equal(y, rne_bf16_array(acc))
    _, m_fused = oracle.geglu(x, Wg, Wu, Wd, want_m=True)
    assert not np.array_equal(m, m_fused)       # the readings differ on these inputs


@pytest.mark.parametrize("approx,mode", [("tanh", oracle.GELU_TANH), ("none", oracle.GELU_ERF),
                                         ("relu", oracle.RELU)])
def test_mlp_eager_rounding_vs_torch(approx, mode):
    """Eager reading of Linear -> activation -> Linear: W1 x + b1 rounded to bf16 before the
    activation, and the activation's output rounded; h bit-equal to torch's float64
    evaluation with those roundings, y's sum to 1e-12."""
    T, D, H, Do = 9, 24, 40, 16
    x = rand_bits((T, D))
    W1, b1 = rand_bits((H, D), 1 / math.sqrt(D)), rand_bits((H,), 1 / math.sqrt(D))
    W2, b2 = rand_bits((Do, H), 1 / math.sqrt(H)), rand_bits((Do,), 1 / math.sqrt(H))
    y, acc, h = oracle.mlp_gelu(x, W1, b1, W2, b2, gelu_mode=mode, eager=True, want_acc=True,
                                want_h=True)
    ref_y, ref_h = torch_mlp_eager_f64(x, W1, b1, W2, b2, approx)
    assert np.array_equal(h, ref_h)
    assert np.max(np.abs(acc - ref_y)) <= 1e-12 * max(1.0, np.abs(ref_y).max())
    assert np.array_equal(y, rne_bf16_array(acc))


# ---------------------------------------------------------------------------- MLP

def test_relu_matches_torch():
    xs = np.array([-3.5, -1e-300, -0.0, 0.0, 1e-300, 0.25, 7.0, 1e300, -1e300, np.inf, -np.inf,
                   np.nan])
    got = oracle.gelu(xs, oracle.RELU)
    ref = torch.relu(torch.from_numpy(xs)).numpy()
    assert np.array_equal(got, ref, equal_nan=True)
    assert not np.signbit(got[2])                 # relu(-0) is +0
    rnd = np.random.default_rng(5).standard_normal(10000) * 4
    assert np.array_equal(oracle.gelu(rnd, oracle.RELU), np.maximum(rnd, 0.0))


@pytest.mark.parametrize("approx,mode", [("tanh", oracle.GELU_TANH), ("none", oracle.GELU_ERF),
                                         ("relu", oracle.RELU)])
@pytest.mark.parametrize("T,D,H,Do", [(1, 8, 16, 8), (17, 32, 72, 16), (129, 16, 32, 24)])
def test_mlp_brute_force_vs_torch(approx, mode, T, D, H, Do):
    x = rand_bits((T, D))
    W1, b1 = rand_bits((H, D), 0.3), rand_bits((H,), 0.3)
    W2, b2 = rand_bits((Do, H), 0.3), rand_bits((Do,), 0.3)
    y, acc, h = oracle.mlp_gelu(x, W1, b1, W2, b2, gelu_mode=mode, want_acc=True, want_h=True)
    ref_y, ref_h = torch_mlp_f64(x, W1, b1, W2, b2, approx)
    assert np.array_equal(h, ref_h)
    assert np.max(np.abs(acc - ref_y)) <= 1e-12 * max(1.0, np.abs(ref_y).max())
    assert np.array_equal(y, rne_bf16_array(acc))


def test_mlp_identity_weights():
    D = 24
    x = rand_bits((30, D))
    b1, b2 = rand_bits((D,), 0.5), rand_bits((D,), 0.5)
    eye = rne_bf16_array(np.eye(D))
    for approx, mode in (("tanh", oracle.GELU_TANH), ("none", oracle.GELU_ERF),
                         ("relu", oracle.RELU)):
        y = oracle.mlp_gelu(x, eye, b1, eye, b2, gelu_mode=mode)
        z = torch.from_numpy(bits_to_f64(x) + bits_to_f64(b1)[None, :])
        act = torch.relu(z) if approx == "relu" else torch.nn.functional.gelu(z, approximate=approx)
        h = bits_to_f64(rne_bf16_array(act.numpy()))
        assert np.array_equal(y, rne_bf16_array(h + bits_to_f64(b2)[None, :]))
    # bias-free and zero first layer: y = b2
    y0 = oracle.mlp_gelu(x, np.zeros((D, D), np.uint16), None, eye, b2)
    assert np.array_equal(y0, np.broadcast_to(b2, y0.shape))


# ---------------------------------------------------------------------------- MoE

def test_moe_geglu_brute_force_vs_torch_per_expert():
    T, D, H, E = 41, 16, 24, 4
    offsets = [0, 9, 9, 30, 41]                 # expert 1 gets no token
    x = rand_bits((T, D))
    Wg, Wu = rand_bits((E, H, D), 0.3), rand_bits((E, H, D), 0.3)
    Wd = rand_bits((E, D, H), 0.3)
    y, m = oracle.moe_geglu(x, offsets, Wg, Wu, Wd, want_m=True)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if a == b:
            continue
        xf = t64(x[a:b])
        g = torch.nn.functional.linear(xf, t64(Wg[e]))
        u = torch.nn.functional.linear(xf, t64(Wu[e]))
        me = rne_bf16_array((torch.nn.functional.gelu(g, approximate="tanh") * u).numpy())
        ye = torch.nn.functional.linear(torch.from_numpy(bits_to_f64(me)), t64(Wd[e])).numpy()
        assert np.array_equal(m[a:b], me)
        assert np.array_equal(y[a:b], rne_bf16_array(ye))


def test_moe_with_identical_experts_is_the_plain_block():
    T, D, H, E = 50, 32, 40, 3
    x = rand_bits((T, D))
    Wg, Wu, Wd = rand_bits((H, D), 0.2), rand_bits((H, D), 0.2), rand_bits((D, H), 0.2)
    stack = lambda w: np.stack([w] * E)
    y = oracle.moe_geglu(x, [0, 7, 33, 50], stack(Wg), stack(Wu), stack(Wd))
    assert np.array_equal(y, oracle.geglu(x, Wg, Wu, Wd))


def test_moe_rejects_bad_offsets():
    x = rand_bits((8, 16))
    W = rand_bits((2, 8, 16), 0.1)
    Wd = rand_bits((2, 16, 8), 0.1)
    for bad in ([0, 9, 8], [1, 4, 8], [0, 5, 3, 8][:3]):
        with pytest.raises(ValueError):
            oracle.moe_geglu(x, bad, W, W, Wd)


def test_moe_row_subset_equals_full_rows():
    """Selecting rows of the mixture-of-experts oracle returns exactly those rows of the full
    computation (groups with no selected row, and an empty group, included)."""
    E, D, H = 4, 16, 24
    counts = [5, 0, 9, 3]
    T = sum(counts)
    off = np.concatenate([[0], np.cumsum(counts)])
    x = rand_bits((T, D))
    Wg, Wu = rand_bits((E, H, D), 0.25), rand_bits((E, H, D), 0.25)
    Wd = rand_bits((E, D, H), 0.2)
    full = oracle.moe_geglu(x, off, Wg, Wu, Wd)
    rows = np.array([0, 3, 5, 6, 13])
    assert np.array_equal(oracle.moe_geglu(x, off, Wg, Wu, Wd, rows=rows), full[rows])
    with pytest.raises(ValueError):
        oracle.moe_geglu(x, off, Wg, Wu, Wd, rows=np.array([3, 1]))
