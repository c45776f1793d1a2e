"""CUDA path vs the oracle through the C ABI, on small and ragged shapes.

Tolerance: per element |y - ref| <= 2e-2 * max(1, |ref|) and relative Frobenius error
<= 5e-3. Special cases whose exact result the fused arithmetic reaches are compared bit for
bit.
"""
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
import oracle
import synth
from gpu_util import DEV, empty_bf16, guarded_bf16, to_dev, to_host, workspace
from helpers import assert_parity, bits_to_f64, rne_bf16_array

pytestmark = pytest.mark.gpu

rng = np.random.default_rng(20240611)


def rbits(shape, scale=1.0):
    return rne_bf16_array(rng.standard_normal(shape) * scale)


def ubits(shape, bound):
    return rne_bf16_array(rng.uniform(-bound, bound, shape))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fm.load()
    yield
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


# ------------------------------------------------------------------------ activation

@pytest.mark.parametrize("mode", [fm.FMLP_GELU_TANH, fm.FMLP_GELU_ERF])
def test_device_gelu_matches_oracle(mode):
    xs = np.concatenate([np.linspace(-12, 12, 20001), rng.standard_normal(20000) * 3])
    xs = xs.astype(np.float32)
    din = torch.from_numpy(xs).to(DEV)
    dout = torch.empty_like(din)
    fm.fmlp_gelu_eval(din, dout, xs.size, mode)
    got = dout.cpu().numpy().astype(np.float64)
    ref = oracle.gelu(xs.astype(np.float64), oracle.GELU_TANH if mode == 0 else oracle.GELU_ERF)
    err = np.abs(got - ref)
    assert np.all(err <= 1e-6 + 2e-5 * np.abs(ref)), float((err / (1e-6 + np.abs(ref))).max())
    # the two flavours differ by up to ~1e-3 near |x| ~ 2: the device uses the requested one
    other = oracle.gelu(xs.astype(np.float64), oracle.GELU_ERF if mode == 0 else oracle.GELU_TANH)
    assert np.abs(got - other).max() > 1e-4


def test_device_relu_is_exact():
    xs = np.concatenate([np.array([-0.0, 0.0, 1e-38, -1e-38, 3.5, -3.5, 1e38, -1e38,
                                   np.inf, -np.inf, np.nan]),
                         rng.standard_normal(20000) * 3]).astype(np.float32)
    din = torch.from_numpy(xs).to(DEV)
    dout = torch.empty_like(din)
    fm.fmlp_gelu_eval(din, dout, xs.size, fm.FMLP_RELU)
    got = dout.cpu().numpy()
    ref = oracle.gelu(xs.astype(np.float64), oracle.RELU).astype(np.float32)
    # NaN stays NaN (its payload is not part of ReLU's definition); everything else bit for bit
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    bad = np.flatnonzero(got[ok].view(np.uint32) != ref[ok].view(np.uint32))
    assert bad.size == 0, (xs[ok][bad[:5]], got[ok][bad[:5]], ref[ok][bad[:5]])


# ------------------------------------------------------------------------ Linear + bias

LINEAR_SHAPES = [
    (1, 32, 64), (3, 32, 64), (17, 72, 136), (127, 64, 64), (128, 128, 256), (129, 256, 200),
    (255, 96, 520), (1024, 32, 64), (300, 1024, 768), (640, 200, 1288),
]


@pytest.mark.parametrize("T,K,N", LINEAR_SHAPES)
@pytest.mark.parametrize("with_bias", [True, False])
def test_linear_bias_vs_oracle(T, K, N, with_bias):
    x, W = rbits((T, K)), ubits((N, K), 1 / math.sqrt(K))
    b = ubits((N,), 1 / math.sqrt(K)) if with_bias else None
    _, y, check = guarded_bf16(T, N)
    fm.fmlp_linear_bias(to_dev(x), to_dev(W), None if b is None else to_dev(b), y, T, K, N)
    torch.cuda.synchronize()
    check()
    assert_parity(to_host(y), oracle.linear(x, W, b), f"linear {T}x{K}->{N}")


def test_linear_identity_and_zero_bit_exact():
    T, K = 200, 136
    # |x| in [1/16, 4) and |b| < 1 keep x + b exact in fp32, so one rounding remains
    mag = rng.uniform(1 / 16, 4, (T, K)) * rng.choice([-1, 1], (T, K))
    x = rne_bf16_array(mag)
    b = ubits((K,), 1.0)
    eye = rne_bf16_array(np.eye(K))
    y = empty_bf16(T, K)
    fm.fmlp_linear_bias(to_dev(x), to_dev(eye), to_dev(b), y, T, K, K)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(y), oracle.linear(x, eye, b))
    z = empty_bf16(T, 64)
    fm.fmlp_linear_bias(to_dev(x), to_dev(np.zeros((64, K), np.uint16)), to_dev(b[:64]), z, T, K, 64)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(z), np.broadcast_to(b[:64], (T, 64)))


def test_linear_layout_worked_example_padded():
    # nn.Linear(2 -> 3) with weight [[0,1],[2,3],[4,5]], x = [1, 10], b = 1: y = [11, 33, 55]
    # (the transposed-view example of the nn.Linear page), zero-padded to the 8-multiple ABI.
    x = np.zeros((1, 8)); x[0, :2] = [1, 10]
    W = np.zeros((8, 8)); W[:3, :2] = [[0, 1], [2, 3], [4, 5]]
    b = np.zeros(8); b[:3] = 1
    y = empty_bf16(1, 8)
    fm.fmlp_linear_bias(to_dev(rne_bf16_array(x)), to_dev(rne_bf16_array(W)),
                        to_dev(rne_bf16_array(b)), y, 1, 8, 8)
    torch.cuda.synchronize()
    assert bits_to_f64(to_host(y))[0, :3].tolist() == [11.0, 33.0, 55.0]


@pytest.mark.parametrize("mode", [fm.FMLP_GELU_TANH, fm.FMLP_GELU_ERF, fm.FMLP_RELU])
@pytest.mark.parametrize("T,K,N", [(1, 64, 64), (129, 96, 520), (513, 512, 384)])
def test_linear_bias_gelu_vs_oracle(mode, T, K, N):
    x, W, b = rbits((T, K)), ubits((N, K), 1 / math.sqrt(K)), ubits((N,), 1 / math.sqrt(K))
    h = empty_bf16(T, N)
    fm.fmlp_linear_bias_gelu(to_dev(x), to_dev(W), to_dev(b), h, T, K, N, mode)
    torch.cuda.synchronize()
    # reference h: the oracle's MLP intermediate with an identity second layer
    _, ref_h = oracle.mlp_gelu(x, W, b, rne_bf16_array(np.eye(N)), None,
                               gelu_mode={0: oracle.GELU_TANH, 1: oracle.GELU_ERF, 2: oracle.RELU}[mode], want_h=True)
    assert_parity(to_host(h), ref_h, "linear+bias+activation")


# values whose activation is fixed exactly in bf16 (no tail of the approximations involved)
SPECIALS = [np.inf, -np.inf, np.nan, 3.0e38, -3.0e38, 1e30, -1e30, 0.0, -0.0, 100.0, -100.0,
            1e-30, -1e-30]


@pytest.mark.parametrize("mode", [fm.FMLP_GELU_TANH, fm.FMLP_GELU_ERF, fm.FMLP_RELU])
@pytest.mark.parametrize("T,policy", [(512, fm.FMLP_TILES_PAIR), (512, fm.FMLP_TILES_SINGLE),
                                      (40, fm.FMLP_TILES_AUTO)])
def test_activation_special_values_through_the_epilogues(mode, T, policy):
    """x = 0 and W = 0, so the pre-activation is the bias exactly: infinities, NaN, the bf16
    extremes, +-0 and values deep in either tail, through the CTA-pair, single-SM and
    few-token epilogues. Each output is the oracle's bf16 of act(0 + b), bit for bit (NaN as
    NaN; -inf gives NaN in both GELU forms, as the formula evaluated in IEEE arithmetic)."""
    K, N = 64, 1024
    vals = np.array(SPECIALS * (N // len(SPECIALS) + 1))[:N]
    b = np.array([oracle.round_bf16(float(v)) for v in vals], np.uint16)
    x = np.zeros((T, K), np.uint16)
    W = np.zeros((N, K), np.uint16)
    h = empty_bf16(T, N)
    fm.fmlp_set_tile_policy(policy)
    try:
        fm.fmlp_linear_bias_gelu(to_dev(x), to_dev(W), to_dev(b), h, T, K, N, mode)
        torch.cuda.synchronize()
    finally:
        fm.fmlp_set_tile_policy(fm.FMLP_TILES_AUTO)
    got = to_host(h)
    omode = {0: oracle.GELU_TANH, 1: oracle.GELU_ERF, 2: oracle.RELU}[mode]
    ref = np.array([oracle.round_bf16(float(v)) for v in
                    oracle.gelu(bits_to_f64(b).astype(np.float64) + 0.0, omode)], np.uint16)
    ref = np.broadcast_to(ref, got.shape)
    gnan, rnan = np.isnan(bits_to_f64(got)), np.isnan(bits_to_f64(ref))
    assert np.array_equal(gnan, rnan), (vals[np.flatnonzero(gnan[0] != rnan[0])[:5]])
    bad = np.flatnonzero((got[0] != ref[0]) & ~rnan[0])
    assert bad.size == 0, [(vals[i], hex(got[0, i]), hex(ref[0, i])) for i in bad[:6]]
    assert np.array_equal(got[:, ~rnan[0]], ref[:, ~rnan[0]])


# ------------------------------------------------------------------------ GeGLU

GEGLU_SHAPES = [(1, 32, 64), (3, 64, 128), (129, 32, 64), (200, 136, 264), (300, 192, 320),
                (1024, 32, 64), (257, 512, 1024)]


@pytest.mark.parametrize("T,D,H", GEGLU_SHAPES)
def test_geglu_gate_up_vs_oracle(T, D, H):
    x = rbits((T, D))
    Wg, Wu = ubits((H, D), 1 / math.sqrt(D)), ubits((H, D), 1 / math.sqrt(D))
    Wd = ubits((D, H), 1 / math.sqrt(H))
    _, m, check = guarded_bf16(T, H)
    fm.fmlp_geglu_gate_up(to_dev(x), to_dev(Wg), to_dev(Wu), m, T, D, H)
    torch.cuda.synchronize()
    check()
    _, ref_m = oracle.geglu(x, Wg, Wu, Wd, want_m=True)
    assert_parity(to_host(m), ref_m, f"gate/up {T}x{D}x{H}")


@pytest.mark.parametrize("T,D,H", GEGLU_SHAPES)
def test_geglu_vs_oracle(T, D, H):
    x = rbits((T, D))
    Wg, Wu = ubits((H, D), 1 / math.sqrt(D)), ubits((H, D), 1 / math.sqrt(D))
    Wd = ubits((D, H), 1 / math.sqrt(H))
    _, y, check = guarded_bf16(T, D)
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
    fm.fmlp_geglu(to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd), y, T, D, H, ws, ws.numel())
    torch.cuda.synchronize()
    check()
    assert_parity(to_host(y), oracle.geglu(x, Wg, Wu, Wd), f"geglu {T}x{D}x{H}")


def test_geglu_without_workspace_uses_stream_allocator():
    T, D, H = 130, 64, 128
    x, Wg, Wu, Wd = rbits((T, D)), ubits((H, D), .1), ubits((H, D), .1), ubits((D, H), .1)
    y = empty_bf16(T, D)
    fm.fmlp_geglu(to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd), y, T, D, H, None, 0)
    torch.cuda.synchronize()
    assert_parity(to_host(y), oracle.geglu(x, Wg, Wu, Wd), "geglu ws=NULL")


def test_geglu_special_cases_bit_exact():
    T, D = 150, 64
    x = rbits((T, D))
    W = ubits((D, D), 0.2)
    zero = np.zeros((D, D), np.uint16)
    eye = rne_bf16_array(np.eye(D))
    two = rne_bf16_array(2 * np.eye(D))
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, D))
    y = empty_bf16(T, D)
    for Wg, Wu, Wd in ((zero, W, W), (W, zero, W), (eye, two, eye)):
        fm.fmlp_geglu(to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd), y, T, D, D, ws, ws.numel())
        torch.cuda.synchronize()
        got, ref = to_host(y), oracle.geglu(x, Wg, Wu, Wd)
        if Wg is eye:
            # y = bf16(gelu_tanh(x) * 2x): the device's fp32 GELU may sit one bf16 ulp away
            assert np.abs(got.astype(np.int32) - ref.astype(np.int32)).max() <= 1
            assert (got != ref).mean() < 0.02
        else:
            assert np.array_equal(got, ref)


def test_geglu_deterministic_and_row_permutation_equivariant():
    T, D, H = 384, 256, 512
    x, Wg, Wu, Wd = rbits((T, D)), ubits((H, D), .06), ubits((H, D), .06), ubits((D, H), .04)
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
    dW = [to_dev(a) for a in (Wg, Wu, Wd)]
    outs = []
    for _ in range(2):
        y = empty_bf16(T, D)
        fm.fmlp_geglu(to_dev(x), *dW, y, T, D, H, ws, ws.numel())
        torch.cuda.synchronize()
        outs.append(to_host(y))
    assert np.array_equal(outs[0], outs[1])
    perm = rng.permutation(T)
    y = empty_bf16(T, D)
    fm.fmlp_geglu(to_dev(x[perm]), *dW, y, T, D, H, ws, ws.numel())
    torch.cuda.synchronize()
    assert np.array_equal(to_host(y), outs[0][perm])


# ------------------------------------------------------------------------ Linear -> GELU -> Linear

@pytest.mark.parametrize("mode", [fm.FMLP_GELU_ERF, fm.FMLP_GELU_TANH, fm.FMLP_RELU])
@pytest.mark.parametrize("T,D,H,Do", [(1, 64, 128, 64), (5, 256, 256, 256), (130, 64, 192, 72),
                                      (700, 512, 1024, 256)])
def test_mlp_gelu_vs_oracle(mode, T, D, H, Do):
    x = rbits((T, D))
    W1, b1 = ubits((H, D), 1 / math.sqrt(D)), ubits((H,), 1 / math.sqrt(D))
    W2, b2 = ubits((Do, H), 1 / math.sqrt(H)), ubits((Do,), 1 / math.sqrt(H))
    _, y, check = guarded_bf16(T, Do)
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(T, D, H, Do))
    fm.fmlp_mlp_gelu(to_dev(x), to_dev(W1), to_dev(b1), to_dev(W2), to_dev(b2), y, T, D, H, Do,
                     mode, ws, ws.numel())
    torch.cuda.synchronize()
    check()
    ref = oracle.mlp_gelu(x, W1, b1, W2, b2, gelu_mode={0: oracle.GELU_TANH, 1: oracle.GELU_ERF, 2: oracle.RELU}[mode])
    assert_parity(to_host(y), ref, f"mlp {T}x{D}x{H}x{Do} mode {mode}")


def test_mlp_without_biases():
    T, D, H = 64, 128, 256
    x, W1, W2 = rbits((T, D)), ubits((H, D), .09), ubits((D, H), .06)
    y = empty_bf16(T, D)
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(T, D, H, D))
    fm.fmlp_mlp_gelu(to_dev(x), to_dev(W1), None, to_dev(W2), None, y, T, D, H, D,
                     fm.FMLP_GELU_ERF, ws, ws.numel())
    torch.cuda.synchronize()
    assert_parity(to_host(y), oracle.mlp_gelu(x, W1, None, W2, None), "mlp no bias")


# ------------------------------------------------------------------------ small workloads

def test_small_workloads_vs_oracle():
    w = synth.WORKLOADS["geglu_1024x32x64"]
    t = w.generate()
    y = empty_bf16(w.T, w.D)
    fm.fmlp_geglu(to_dev(t["x"]), to_dev(t["Wg"]), to_dev(t["Wu"]), to_dev(t["Wd"]), y,
                  w.T, w.D, w.H, None, 0)
    w2 = synth.WORKLOADS["linear_1024x32x64"]
    t2 = w2.generate()
    y2 = empty_bf16(w2.T, w2.H)
    fm.fmlp_linear_bias(to_dev(t2["x"]), to_dev(t2["W"]), to_dev(t2["b"]), y2, w2.T, w2.D, w2.H)
    torch.cuda.synchronize()
    assert_parity(to_host(y), oracle.geglu(t["x"], t["Wg"], t["Wu"], t["Wd"]), "geglu C1")
    assert_parity(to_host(y2), oracle.linear(t2["x"], t2["W"], t2["b"]), "linear C2")


# ------------------------------------------------------------------------ device status

def test_bounded_wait_times_out_and_reports():
    assert fm.fmlp_device_status() == fm.FMLP_OK
    fm.fmlp_test_wait_timeout(20000)   # 20 ms
    st = fm.fmlp_device_status()
    assert st == fm.FMLP_ERR_DEVICE_TIMEOUT
    assert "test wait" in fm.fmlp_last_error()
    assert fm.fmlp_device_status() == fm.FMLP_OK       # read-and-clear
    # the context is still usable
    x = torch.ones(16, device=DEV)
    assert float(x.sum()) == 16.0
