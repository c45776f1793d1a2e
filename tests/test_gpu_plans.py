"""The fused single-kernel plan (small D) and the GEMV plan (a few tokens) against the oracle,
and the number of kernels each plan launches (counted in a captured CUDA graph)."""
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
import oracle
import synth
from gpu_util import DEV, count_graph_kernels, empty_bf16, guarded_bf16, to_dev, to_host, workspace
from helpers import assert_parity, rne_bf16_array

pytestmark = pytest.mark.gpu
rng = np.random.default_rng(777)


def ubits(shape, bound):
    return rne_bf16_array(rng.uniform(-bound, bound, shape))


def rbits(shape):
    return rne_bf16_array(rng.standard_normal(shape))


def geglu_inputs(T, D, H):
    return (rbits((T, D)), ubits((H, D), 1 / math.sqrt(D)), ubits((H, D), 1 / math.sqrt(D)),
            ubits((D, H), 1 / math.sqrt(H)))


def run_geglu(x, Wg, Wu, Wd):
    T, D = x.shape
    H = Wg.shape[0]
    _, y, check = guarded_bf16(T, D)
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
    fm.fmlp_geglu(to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd), y, T, D, H, ws, ws.numel())
    torch.cuda.synchronize()
    check()
    return to_host(y)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fm.load()
    yield
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


# ------------------------------------------------------------------------ fused small plan

@pytest.mark.parametrize("T,D,H", [(1, 32, 64), (100, 32, 64), (129, 16, 8), (1024, 32, 64),
                                   (300, 64, 200), (257, 96, 520), (128, 128, 1000),
                                   (513, 256, 2048), (64, 208, 72)])
def test_fused_small_geglu_vs_oracle(T, D, H):
    assert fm.fmlp_geglu_plan(T, D, H) == fm.FMLP_PLAN_FUSED_SMALL
    assert fm.fmlp_geglu_workspace_size(T, D, H) == 0
    x, Wg, Wu, Wd = geglu_inputs(T, D, H)
    assert_parity(run_geglu(x, Wg, Wu, Wd), oracle.geglu(x, Wg, Wu, Wd), f"fused {T}x{D}x{H}")


def test_fused_small_special_cases():
    T, D = 200, 64
    x = rbits((T, D))
    W = ubits((D, D), .2)
    zero = np.zeros((D, D), np.uint16)
    assert np.array_equal(run_geglu(x, zero, W, W), oracle.geglu(x, zero, W, W))
    assert np.array_equal(run_geglu(x, W, zero, W), oracle.geglu(x, W, zero, W))
    eye, two = rne_bf16_array(np.eye(D)), rne_bf16_array(2 * np.eye(D))
    got, ref = run_geglu(x, eye, two, eye), oracle.geglu(x, eye, two, eye)
    assert np.abs(got.astype(np.int32) - ref.astype(np.int32)).max() <= 1


def test_fused_small_workload_and_determinism():
    w = synth.WORKLOADS["geglu_1024x32x64"]
    t = w.generate()
    a = run_geglu(t["x"], t["Wg"], t["Wu"], t["Wd"])
    b = run_geglu(t["x"], t["Wg"], t["Wu"], t["Wd"])
    assert np.array_equal(a, b)
    assert_parity(a, oracle.geglu(t["x"], t["Wg"], t["Wu"], t["Wd"]), "geglu 1024x32x64")


# (T, D, H, Dout): the 1024 x 32 -> 64 -> 32 block; D a multiple of 8 only and H not a
# multiple of the 64-wide hidden chunk; the widest block the plan takes; a few tokens with tiny
# weights (which stay on this kernel rather than the decode one)
MLP_SMALL = [(1024, 32, 64, 32), (100, 40, 72, 48), (129, 256, 2048, 256), (300, 128, 1000, 64),
             (5, 64, 128, 16), (3, 32, 64, 32)]


@pytest.mark.parametrize("T,D,H,Dout", MLP_SMALL)
@pytest.mark.parametrize("mode", [fm.FMLP_GELU_TANH, fm.FMLP_GELU_ERF, fm.FMLP_RELU])
def test_fused_small_mlp_vs_oracle(T, D, H, Dout, mode):
    """Linear -> activation -> Linear with both biases in one kernel: h stays on chip."""
    assert fm.fmlp_mlp_gelu_plan(T, D, H, Dout) == fm.FMLP_PLAN_FUSED_SMALL
    assert fm.fmlp_mlp_gelu_workspace_size(T, D, H, Dout) == 0
    x = rbits((T, D))
    W1, b1 = ubits((H, D), 1 / math.sqrt(D)), ubits((H,), 1 / math.sqrt(D))
    W2, b2 = ubits((Dout, H), 1 / math.sqrt(H)), ubits((Dout,), 1 / math.sqrt(H))
    _, y, check = guarded_bf16(T, Dout)
    fm.fmlp_mlp_gelu(to_dev(x), to_dev(W1), to_dev(b1), to_dev(W2), to_dev(b2), y, T, D, H, Dout,
                     mode, None, 0)
    torch.cuda.synchronize()
    check()
    om = {0: oracle.GELU_TANH, 1: oracle.GELU_ERF, 2: oracle.RELU}[mode]
    assert_parity(to_host(y), oracle.mlp_gelu(x, W1, b1, W2, b2, gelu_mode=om),
                  f"fused mlp {T}x{D}x{H}x{Dout} mode {mode}")


def test_fused_small_mlp_nullable_biases_and_one_kernel():
    T, D, H, Dout = 1024, 32, 64, 32
    x = rbits((T, D))
    W1, b1 = ubits((H, D), 1 / math.sqrt(D)), ubits((H,), 1 / math.sqrt(D))
    W2, b2 = ubits((Dout, H), 1 / math.sqrt(H)), ubits((Dout,), 1 / math.sqrt(H))
    dx, dW1, db1, dW2, db2 = (to_dev(a) for a in (x, W1, b1, W2, b2))
    for bb1, bb2 in ((None, db2), (db1, None), (None, None)):
        y = empty_bf16(T, Dout)
        fm.fmlp_mlp_gelu(dx, dW1, bb1, dW2, bb2, y, T, D, H, Dout, fm.FMLP_GELU_ERF, None, 0)
        torch.cuda.synchronize()
        ref = oracle.mlp_gelu(x, W1, None if bb1 is None else b1, W2, None if bb2 is None else b2,
                              gelu_mode=oracle.GELU_ERF)
        assert_parity(to_host(y), ref, f"fused mlp biases {bb1 is not None} {bb2 is not None}")
    y = empty_bf16(T, Dout)
    nk, nall = count_graph_kernels(lambda s: fm.fmlp_mlp_gelu(
        dx, dW1, db1, dW2, db2, y, T, D, H, Dout, fm.FMLP_GELU_ERF, None, 0, stream=s))
    assert nk == 1 and nall == 1


# ------------------------------------------------------------------------ decode sizes

SMALL_WEIGHTS = 16 << 20   # the GEMV serves two tokens when a call's weights fit in this


def decode_plan(T, weight_bytes):
    """The plan a single Linear takes at a few tokens: the GEMV at one token, and at two when
    the weights are small; the few-token tcgen05 kernel (a TC plan) otherwise."""
    gemv = T == 1 or (T == 2 and weight_bytes <= SMALL_WEIGHTS)
    return fm.FMLP_PLAN_GEMV if gemv else fm.FMLP_PLAN_TC


def test_decode_crossover_table():
    """Blocks (GeGLU, MLP) of 1..4 tokens take the GEMV pair at one token (and at two for small
    weights) and the few-token kernels otherwise, tiny GeGLU blocks the single-CTA fused
    kernel; 5..128 tokens run the few-token kernels."""
    assert fm.fmlp_mlp_gelu_plan(1, 4096, 4096, 4096) == fm.FMLP_PLAN_GEMV
    assert fm.fmlp_mlp_gelu_plan(4, 4096, 4096, 4096) == fm.FMLP_PLAN_TC
    assert fm.fmlp_mlp_gelu_plan(5, 4096, 4096, 4096) == fm.FMLP_PLAN_TC
    assert fm.fmlp_geglu_plan(2, 768, 3072) == fm.FMLP_PLAN_GEMV
    assert fm.fmlp_geglu_plan(5, 768, 3072) == fm.FMLP_PLAN_TC
    assert fm.fmlp_geglu_plan(1, 32, 64) == fm.FMLP_PLAN_FUSED_SMALL
    assert "few-token" in fm.fmlp_describe_plan("mlp", 4, 4096, 4096, 4096)
    assert "few-token" in fm.fmlp_describe_plan("mlp", 5, 4096, 4096, 4096)
    assert "few-token" in fm.fmlp_describe_plan("mlp", 128, 4096, 4096, 4096)
    assert "few-token" not in fm.fmlp_describe_plan("mlp", 129, 4096, 4096, 4096)


def test_decode_crossover_table_with_the_decode_plan(prefer_decode):
    assert fm.fmlp_mlp_gelu_plan(1, 4096, 4096, 4096) == fm.FMLP_PLAN_DECODE
    assert fm.fmlp_mlp_gelu_plan(4, 4096, 4096, 4096) == fm.FMLP_PLAN_DECODE
    assert fm.fmlp_mlp_gelu_plan(5, 4096, 4096, 4096) == fm.FMLP_PLAN_TC
    assert fm.fmlp_geglu_plan(2, 768, 3072) == fm.FMLP_PLAN_DECODE
    assert fm.fmlp_geglu_plan(1, 32, 64) == fm.FMLP_PLAN_FUSED_SMALL
    assert "one weight-streaming kernel" in fm.fmlp_describe_plan("mlp", 4, 4096, 4096, 4096)


@pytest.mark.parametrize("T", [1, 2, 3, 4])
@pytest.mark.parametrize("K,N", [(256, 64), (512, 1000), (4096, 4096), (3072, 768)])
def test_gemv_linear_vs_oracle(T, K, N):
    assert fm.fmlp_linear_plan(T, K, N) == decode_plan(T, N * K * 2)
    x, W, b = rbits((T, K)), ubits((N, K), 1 / math.sqrt(K)), ubits((N,), 1 / math.sqrt(K))
    _, y, check = guarded_bf16(T, N)
    fm.fmlp_linear_bias(to_dev(x), to_dev(W), to_dev(b), y, T, K, N)
    torch.cuda.synchronize()
    check()
    assert_parity(to_host(y), oracle.linear(x, W, b), f"gemv {T}x{K}->{N}")


@pytest.mark.parametrize("decode", [False, True])
@pytest.mark.parametrize("T,D,H", [(1, 256, 512), (2, 768, 3072), (4, 512, 1280)])
def test_few_token_geglu_block_and_gemv_gate_up(T, D, H, decode):
    """The block at a few tokens (the default plans, or the decode kernel; the single-CTA fused
    kernel for tiny weights either way) and the gate/up stage on its own (the GEMV at one or
    two tokens) against the oracle."""
    fm.fmlp_test_prefer_decode(1 if decode else 0)
    try:
        plans = (fm.FMLP_PLAN_DECODE, fm.FMLP_PLAN_FUSED_SMALL) if decode else \
            (fm.FMLP_PLAN_GEMV, fm.FMLP_PLAN_TC, fm.FMLP_PLAN_FUSED_SMALL)
        assert fm.fmlp_geglu_plan(T, D, H) in plans
        x, Wg, Wu, Wd = geglu_inputs(T, D, H)
        assert_parity(run_geglu(x, Wg, Wu, Wd), oracle.geglu(x, Wg, Wu, Wd), f"geglu {T}x{D}x{H}")
    finally:
        fm.fmlp_test_prefer_decode(0)
    m = empty_bf16(T, H)
    fm.fmlp_geglu_gate_up(to_dev(x), to_dev(Wg), to_dev(Wu), m, T, D, H)
    torch.cuda.synchronize()
    _, ref_m = oracle.geglu(x, Wg, Wu, Wd, want_m=True)
    assert_parity(to_host(m), ref_m, "gate/up")


@pytest.mark.parametrize("decode", [False, True])
@pytest.mark.parametrize("mode", [fm.FMLP_GELU_ERF, fm.FMLP_GELU_TANH, fm.FMLP_RELU])
def test_decode_mlp_4096_vs_oracle(mode, decode, request):
    """The 4096-wide MLP at one token: the GEMV pair (default) and the one-kernel decode."""
    if decode:
        request.getfixturevalue("prefer_decode")
    w = synth.WORKLOADS["mlp_4096_t1"]
    assert fm.fmlp_mlp_gelu_plan(1, w.D, w.H, w.Dout) == \
        (fm.FMLP_PLAN_DECODE if decode else fm.FMLP_PLAN_GEMV)
    t = w.generate()
    d = {k: to_dev(v) for k, v in t.items()}
    _, y, check = guarded_bf16(1, w.Dout)
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(1, w.D, w.H, w.Dout))
    fm.fmlp_mlp_gelu(d["x"], d["W1"], d["b1"], d["W2"], d["b2"], y, 1, w.D, w.H, w.Dout, mode,
                     ws, ws.numel())
    torch.cuda.synchronize()
    check()
    ref = oracle.mlp_gelu(t["x"], t["W1"], t["b1"], t["W2"], t["b2"],
                          gelu_mode={0: oracle.GELU_TANH, 1: oracle.GELU_ERF, 2: oracle.RELU}[mode])
    assert_parity(to_host(y), ref, f"decode mlp 4096 mode {mode}")


def test_gemv_deterministic_across_calls():
    x, W, b = rbits((3, 4096)), ubits((4096, 4096), 1 / 64), ubits((4096,), 1 / 64)
    outs = []
    for _ in range(3):
        y = empty_bf16(3, 4096)
        fm.fmlp_linear_bias(to_dev(x), to_dev(W), to_dev(b), y, 3, 4096, 4096)
        torch.cuda.synchronize()
        outs.append(to_host(y))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


# ------------------------------------------------------------------------ kernel counts

@pytest.mark.parametrize("T,D,H,plan,kernels", [
    (1024, 32, 64, fm.FMLP_PLAN_FUSED_SMALL, 1),
    (1, 768, 3072, fm.FMLP_PLAN_DECODE, 1),
    (1, 768, 3072, fm.FMLP_PLAN_GEMV, 2),
    (512, 768, 3072, fm.FMLP_PLAN_TC, 2),
])
def test_geglu_kernel_count(T, D, H, plan, kernels, request):
    if plan == fm.FMLP_PLAN_DECODE:
        request.getfixturevalue("prefer_decode")
    assert fm.fmlp_geglu_plan(T, D, H) == plan
    x, Wg, Wu, Wd = (to_dev(a) for a in geglu_inputs(T, D, H))
    y = empty_bf16(T, D)
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
    nk, nall = count_graph_kernels(
        lambda s: fm.fmlp_geglu(x, Wg, Wu, Wd, y, T, D, H, ws, ws.numel(), stream=s))
    assert nk == kernels and nall == kernels


def test_linear_and_mlp_kernel_counts():
    T, K, N = 1024, 32, 64
    x, W, b = to_dev(rbits((T, K))), to_dev(ubits((N, K), .1)), to_dev(ubits((N,), .1))
    y = empty_bf16(T, N)
    nk, _ = count_graph_kernels(lambda s: fm.fmlp_linear_bias(x, W, b, y, T, K, N, stream=s))
    assert nk == 1     # the bias add is the GEMM's epilogue: one kernel
    x1 = to_dev(rbits((1, 4096)))
    W1, W2 = to_dev(ubits((4096, 4096), 1 / 64)), to_dev(ubits((4096, 4096), 1 / 64))
    b1, b2 = to_dev(ubits((4096,), 1 / 64)), to_dev(ubits((4096,), 1 / 64))
    y1 = empty_bf16(1, 4096)
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(1, 4096, 4096, 4096))
    nk, _ = count_graph_kernels(lambda s: fm.fmlp_mlp_gelu(
        x1, W1, b1, W2, b2, y1, 1, 4096, 4096, 4096, fm.FMLP_GELU_ERF, ws, ws.numel(), stream=s))
    assert nk == 2     # one GEMV per layer
    fm.fmlp_test_prefer_decode(1)
    try:
        nk, _ = count_graph_kernels(lambda s: fm.fmlp_mlp_gelu(
            x1, W1, b1, W2, b2, y1, 1, 4096, 4096, 4096, fm.FMLP_GELU_ERF, ws, ws.numel(),
            stream=s))
    finally:
        fm.fmlp_test_prefer_decode(0)
    assert nk == 1     # both layers in one decode kernel


@pytest.mark.parametrize("decode", [False, True])
def test_decode_repeated_and_on_two_streams(decode, request):
    """Decode calls in a row (the GEMV pair, or the one-kernel decode), alternating between two
    streams: every call gives the oracle's (and the first call's) result."""
    if decode:
        request.getfixturevalue("prefer_decode")
    T, D, H = 2, 1024, 2048
    x, W1, b1 = rbits((T, D)), ubits((H, D), 1 / 32), ubits((H,), 1 / 32)
    W2, b2 = ubits((D, H), 1 / 45), ubits((D,), 1 / 45)
    dx, dW1, db1, dW2, db2 = (to_dev(a) for a in (x, W1, b1, W2, b2))
    ref = oracle.mlp_gelu(x, W1, b1, W2, b2)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for i in range(12):
        s = streams[i % 2]
        y = empty_bf16(T, D)
        ws = workspace(fm.fmlp_mlp_gelu_workspace_size(T, D, H, D))
        with torch.cuda.stream(s):
            fm.fmlp_mlp_gelu(dx, dW1, db1, dW2, db2, y, T, D, H, D, fm.FMLP_GELU_ERF, ws,
                             ws.numel(), stream=s)
        s.synchronize()
        outs.append(to_host(y))
    for o in outs:
        assert np.array_equal(o, outs[0])
    assert_parity(outs[0], ref, "decode")
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


# ------------------------------------------------------------------------ decode ordering

@pytest.mark.parametrize("decode", [False, True])
def test_decode_weights_written_by_previous_kernels(decode, request):
    """Kernels of a decode block (the GEMV pair, or the one-kernel decode) start before the
    kernel queued ahead of them has finished (programmatic dependent launch); they must still
    see weights that kernels queued just before the block wrote. W2 of a block is written, on
    the same stream with no synchronisation, first by a tensor-core Linear and then by the
    last kernel of another block; both results must match the oracle run on the weights as
    written."""
    if decode:
        request.getfixturevalue("prefer_decode")
    s = torch.cuda.Stream()
    # (1) W2 [1024, 2048] is the output of a tensor-core Linear queued right before the block
    Tl, Kl, Nl = 1024, 256, 2048
    xl, Wl, bl = rbits((Tl, Kl)), ubits((Nl, Kl), 1 / 16), ubits((Nl,), 1 / 16)
    assert fm.fmlp_linear_plan(Tl, Kl, Nl) == fm.FMLP_PLAN_TC
    D, H, Dout = 1024, 2048, 1024
    x, W1, b1, b2 = rbits((1, D)), ubits((H, D), 1 / 32), ubits((H,), 1 / 32), ubits((Dout,), 1 / 45)
    dxl, dWl, dbl, dx, dW1, db1, db2 = (to_dev(a) for a in (xl, Wl, bl, x, W1, b1, b2))
    W2 = torch.zeros((Dout, H), dtype=torch.bfloat16, device="cuda")   # stale contents: zeros
    y = empty_bf16(1, Dout)
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(1, D, H, Dout))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        fm.fmlp_linear_bias(dxl, dWl, dbl, W2, Tl, Kl, Nl, stream=s)
        fm.fmlp_mlp_gelu(dx, dW1, db1, W2, db2, y, 1, D, H, Dout, fm.FMLP_GELU_ERF, ws,
                         ws.numel(), stream=s)
    s.synchronize()
    W2_bits = to_host(W2)
    assert np.any(W2_bits != 0)
    assert_parity(to_host(y), oracle.mlp_gelu(x, W1, b1, W2_bits, b2), "decode after linear")

    # (2) W2 of block B [8, 2048] is y [8, 2048] of few-token block A, queued right before B
    TA, DA, HA, DoA = 8, 1024, 2048, 2048
    xa, W1a, b1a = rbits((TA, DA)), ubits((HA, DA), 1 / 32), ubits((HA,), 1 / 32)
    W2a, b2a = ubits((DoA, HA), 1 / 45), ubits((DoA,), 1 / 45)
    DB, HB, DoB = 512, 2048, 8
    xb, W1b, b1b, b2b = rbits((1, DB)), ubits((HB, DB), 1 / 23), ubits((HB,), 1 / 23), ubits((DoB,), 1 / 45)
    dA = [to_dev(a) for a in (xa, W1a, b1a, W2a, b2a)]
    dB = [to_dev(a) for a in (xb, W1b, b1b, b2b)]
    yA = torch.zeros((TA, DoA), dtype=torch.bfloat16, device="cuda")
    yB = empty_bf16(1, DoB)
    wsA = workspace(fm.fmlp_mlp_gelu_workspace_size(TA, DA, HA, DoA))
    wsB = workspace(fm.fmlp_mlp_gelu_workspace_size(1, DB, HB, DoB))
    # block A runs the few-token tcgen05 kernels, block B the GEMV pair or the one-kernel decode
    assert fm.fmlp_mlp_gelu_plan(TA, DA, HA, DoA) == fm.FMLP_PLAN_TC
    assert fm.fmlp_mlp_gelu_plan(1, DB, HB, DoB) == \
        (fm.FMLP_PLAN_DECODE if decode else fm.FMLP_PLAN_GEMV)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(3):   # repeated, so that earlier blocks' kernels overlap later ones
            fm.fmlp_mlp_gelu(dA[0], dA[1], dA[2], dA[3], dA[4], yA, TA, DA, HA, DoA,
                             fm.FMLP_GELU_ERF, wsA, wsA.numel(), stream=s)
            fm.fmlp_mlp_gelu(dB[0], dB[1], dB[2], yA.view(DoB, HB), dB[3], yB, 1, DB, HB, DoB,
                             fm.FMLP_GELU_ERF, wsB, wsB.numel(), stream=s)
    s.synchronize()
    yA_bits = to_host(yA)
    assert_parity(yA_bits, oracle.mlp_gelu(xa, W1a, b1a, W2a, b2a), "decode block A")
    assert_parity(to_host(yB), oracle.mlp_gelu(xb, W1b, b1b, yA_bits.reshape(DoB, HB), b2b),
                  "decode block B on A's output")
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()

