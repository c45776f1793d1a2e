"""The one-kernel decode plan (both layers of the block in one launch for 1..4 tokens; taken
while fmlp_test_prefer_decode(1) is in effect, as in every test here) against the oracle: every activation, the GeGLU block, ragged and narrow shapes (rows split unevenly
over the CTAs, rows shorter than a warp's 32 chunks), rows longer than one 16-byte chunk per
thread, nullable biases, determinism, two streams, one kernel per call, and the bounded
grid-barrier wait running out and reporting."""
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
import oracle
import synth
from gpu_util import count_graph_kernels, empty_bf16, guarded_bf16, to_dev, to_host, workspace
from helpers import assert_parity, rne_bf16_array

pytestmark = pytest.mark.gpu
rng = np.random.default_rng(4242)


def ubits(shape, bound):
    return rne_bf16_array(rng.uniform(-bound, bound, shape))


def rbits(shape):
    return rne_bf16_array(rng.standard_normal(shape))


def fast_ubits(shape, bound, seed):
    """Large uniform tensors: torch's float -> bf16 conversion (round to nearest even) of
    float32 values, which is exact rounding for these."""
    g = torch.Generator().manual_seed(seed)
    v = (torch.rand(shape, generator=g, dtype=torch.float32) * 2 - 1) * bound
    return v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fm.load()
    fm.fmlp_test_prefer_decode(1)
    yield
    fm.fmlp_test_prefer_decode(0)
    fm.fmlp_test_decode_overload(0, 0)
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


def run_mlp(x, W1, b1, W2, b2, mode, stream=None):
    T, D = x.shape
    H, Dout = W1.shape[0], W2.shape[0]
    _, y, check = guarded_bf16(T, Dout)
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(T, D, H, Dout))
    dev = [None if a is None else to_dev(a) for a in (x, W1, b1, W2, b2)]
    fm.fmlp_mlp_gelu(dev[0], dev[1], dev[2], dev[3], dev[4], y, T, D, H, Dout, mode, ws,
                     ws.numel(), stream=stream)
    torch.cuda.synchronize()
    check()
    return to_host(y)


def run_geglu(x, Wg, Wu, Wd):
    T, D = x.shape
    H = Wg.shape[0]
    _, y, check = guarded_bf16(T, D)
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
    fm.fmlp_geglu(to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd), y, T, D, H, ws, ws.numel())
    torch.cuda.synchronize()
    check()
    return to_host(y)


MODES = [fm.FMLP_GELU_TANH, fm.FMLP_GELU_ERF, fm.FMLP_RELU]


@pytest.mark.parametrize("T", [1, 2, 3, 4])
@pytest.mark.parametrize("mode", MODES)
def test_decode_mlp_4096_all_token_counts(T, mode):
    D = H = Dout = 4096
    assert fm.fmlp_mlp_gelu_plan(T, D, H, Dout) == fm.FMLP_PLAN_DECODE
    x = rbits((T, D))
    W1, W2 = fast_ubits((H, D), 1 / 64, 11), fast_ubits((Dout, H), 1 / 64, 12)
    b1, b2 = ubits((H,), 1 / 64), ubits((Dout,), 1 / 64)
    got = run_mlp(x, W1, b1, W2, b2, mode)
    assert_parity(got, oracle.mlp_gelu(x, W1, b1, W2, b2, gelu_mode=mode), f"decode T={T} {mode}")


# (T, D, H, Dout): ragged row splits over the CTAs; rows shorter than one warp's 32 chunks
# (several thread groups per CTA); D > H and H > D; inner dims that are multiples of 8 only
MLP_SHAPES = [(1, 264, 1032, 520), (3, 1032, 264, 8), (2, 8, 16, 24), (4, 2048, 6144, 1024),
              (1, 4104, 2056, 4096), (1, 12288, 1536, 3000)]


@pytest.mark.parametrize("T,D,H,Dout", MLP_SHAPES)
def test_decode_mlp_shapes(T, D, H, Dout):
    assert fm.fmlp_mlp_gelu_plan(T, D, H, Dout) == fm.FMLP_PLAN_DECODE
    x = rbits((T, D))
    W1, W2 = fast_ubits((H, D), 1 / math.sqrt(D), 21), fast_ubits((Dout, H), 1 / math.sqrt(H), 22)
    b1, b2 = ubits((H,), 0.1), ubits((Dout,), 0.1)
    got = run_mlp(x, W1, b1, W2, b2, fm.FMLP_GELU_ERF)
    assert_parity(got, oracle.mlp_gelu(x, W1, b1, W2, b2, gelu_mode=fm.FMLP_GELU_ERF),
                  f"decode {T}x{D}x{H}x{Dout}")


def test_decode_mlp_without_biases():
    T, D, H, Dout = 2, 1024, 3072, 1024
    x = rbits((T, D))
    W1, W2 = fast_ubits((H, D), 1 / 32, 31), fast_ubits((Dout, H), 1 / 55, 32)
    got = run_mlp(x, W1, None, W2, None, fm.FMLP_GELU_TANH)
    assert_parity(got, oracle.mlp_gelu(x, W1, None, W2, None, gelu_mode=fm.FMLP_GELU_TANH),
                  "decode no bias")


def test_decode_long_rows():
    """H = 16384: a layer-2 row of 32 KB fills a ring stage by itself and every consumer thread
    covers four 16-byte chunks of it (the layer-1 rows are short enough for four thread
    groups)."""
    T, D, H, Dout = 1, 1024, 16384, 4096
    assert fm.fmlp_mlp_gelu_plan(T, D, H, Dout) == fm.FMLP_PLAN_DECODE
    x = rbits((T, D))
    W1, W2 = fast_ubits((H, D), 1 / 32, 41), fast_ubits((Dout, H), 1 / 128, 42)
    b1, b2 = ubits((H,), 0.05), ubits((Dout,), 0.05)
    got = run_mlp(x, W1, b1, W2, b2, fm.FMLP_GELU_ERF)
    assert_parity(got, oracle.mlp_gelu(x, W1, b1, W2, b2, gelu_mode=fm.FMLP_GELU_ERF),
                  "decode long rows")


def test_rows_too_long_for_two_stages_take_the_gemv():
    """With H = 40960 the token vector (80 KB) and two ring stages of one 80 KB layer-2 row do
    not fit in shared memory: the block runs as two GEMVs."""
    assert fm.fmlp_mlp_gelu_plan(1, 1024, 40960, 1024) == fm.FMLP_PLAN_GEMV


@pytest.mark.parametrize("T,D,H", [(1, 768, 3072), (2, 768, 3072), (3, 768, 3072),
                                   (4, 768, 3072), (1, 4096, 11008), (2, 520, 1288)])
def test_decode_geglu_vs_oracle(T, D, H):
    assert fm.fmlp_geglu_plan(T, D, H) == fm.FMLP_PLAN_DECODE
    x = rbits((T, D))
    Wg, Wu = fast_ubits((H, D), 1 / math.sqrt(D), 51), fast_ubits((H, D), 1 / math.sqrt(D), 52)
    Wd = fast_ubits((D, H), 1 / math.sqrt(H), 53)
    assert_parity(run_geglu(x, Wg, Wu, Wd), oracle.geglu(x, Wg, Wu, Wd), f"decode geglu {T}x{D}x{H}")


def test_geglu_70b_class_one_token():
    """The 70B-class block (D 8192, H 28672) at one token: 1.41 GB of weights (two GEMVs)."""
    w = synth.WORKLOADS["geglu_8192x8192x28672"]
    t = w.generate(names=["Wg", "Wu", "Wd"])
    x = rbits((1, w.D))
    assert_parity(run_geglu(x, t["Wg"], t["Wu"], t["Wd"]), oracle.geglu(x, t["Wg"], t["Wu"], t["Wd"]),
                  "decode geglu 70B-class")


def test_decode_special_cases_bit_exact():
    """Zero gate weights make m = gelu(0) * u = 0 and y = 0 exactly; identity weights of the
    MLP with ReLU give y = bf16(relu(x + b1) + b2) with one rounding of h in between."""
    T, D, H = 3, 512, 512
    assert fm.fmlp_geglu_plan(T, D, H) == fm.FMLP_PLAN_DECODE
    assert fm.fmlp_mlp_gelu_plan(T, D, H, D) == fm.FMLP_PLAN_DECODE
    x = rbits((T, D))
    zero = np.zeros((H, D), np.uint16)
    W = ubits((H, D), 0.1)
    got = run_geglu(x, zero, W, W)
    assert np.array_equal(got, oracle.geglu(x, zero, W, W))
    eye = rne_bf16_array(np.eye(D))
    b1, b2 = ubits((D,), 0.5), ubits((D,), 0.5)
    got = run_mlp(x, eye, b1, eye, b2, fm.FMLP_RELU)
    assert np.array_equal(got, oracle.mlp_gelu(x, eye, b1, eye, b2, gelu_mode=fm.FMLP_RELU))


def test_decode_deterministic_one_kernel_and_two_streams():
    T, D, H, Dout = 2, 4096, 4096, 4096
    x, b1, b2 = rbits((T, D)), ubits((H,), 1 / 64), ubits((Dout,), 1 / 64)
    W1, W2 = fast_ubits((H, D), 1 / 64, 61), fast_ubits((Dout, H), 1 / 64, 62)
    dx, dW1, db1, dW2, db2 = (to_dev(a) for a in (x, W1, b1, W2, b2))
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(T, D, H, Dout))
    y = empty_bf16(T, Dout)
    nk, _ = count_graph_kernels(lambda s: fm.fmlp_mlp_gelu(
        dx, dW1, db1, dW2, db2, y, T, D, H, Dout, fm.FMLP_GELU_ERF, ws, ws.numel(), stream=s))
    assert nk == 1     # both layers in one kernel
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for i in range(10):
        s = streams[i % 2]
        yi = empty_bf16(T, Dout)
        wsi = workspace(ws.numel())
        with torch.cuda.stream(s):
            fm.fmlp_mlp_gelu(dx, dW1, db1, dW2, db2, yi, T, D, H, Dout, fm.FMLP_GELU_ERF, wsi,
                             wsi.numel(), stream=s)
        outs.append((s, yi))
    torch.cuda.synchronize()
    first = to_host(outs[0][1])
    for _, yi in outs:
        assert np.array_equal(to_host(yi), first)
    assert_parity(first, oracle.mlp_gelu(x, W1, b1, W2, b2, gelu_mode=fm.FMLP_GELU_ERF), "decode")
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


def test_decode_weights_written_just_before():
    """W2 of this block is y of another decode block queued right before it on the same
    stream (the previous kernel lets this one launch early); W1 is written by a tensor-core
    Linear before that. The results must match the oracle on the weights as written."""
    s = torch.cuda.Stream()
    DA, HA, DoA = 1024, 2048, 4096          # block A: y [4, 4096] becomes W2 of block B
    xa, W1a, b1a = rbits((4, DA)), ubits((HA, DA), 1 / 32), ubits((HA,), 1 / 32)
    W2a, b2a = fast_ubits((DoA, HA), 1 / 45, 71), ubits((DoA,), 1 / 45)
    DB, HB, DoB = 512, 2048, 8
    xb, b1b, b2b = rbits((1, DB)), ubits((HB,), 1 / 23), ubits((DoB,), 1 / 45)
    xl, Wl = rbits((HB, 256)), ubits((DB, 256), 1 / 16)   # Linear writing W1 of block B
    dA = [to_dev(a) for a in (xa, W1a, b1a, W2a, b2a)]
    dxb, db1b, db2b, dxl, dWl = (to_dev(a) for a in (xb, b1b, b2b, xl, Wl))
    W1b = torch.zeros((HB, DB), dtype=torch.bfloat16, device="cuda")
    yA = torch.zeros((4, DoA), dtype=torch.bfloat16, device="cuda")
    yB = empty_bf16(1, DoB)
    wsA = workspace(fm.fmlp_mlp_gelu_workspace_size(4, DA, HA, DoA))
    wsB = workspace(fm.fmlp_mlp_gelu_workspace_size(1, DB, HB, DoB))
    assert fm.fmlp_mlp_gelu_plan(4, DA, HA, DoA) == fm.FMLP_PLAN_DECODE
    assert fm.fmlp_mlp_gelu_plan(1, DB, HB, DoB) == fm.FMLP_PLAN_DECODE
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(3):
            fm.fmlp_linear_bias(dxl, dWl, None, W1b, HB, 256, DB, stream=s)
            fm.fmlp_mlp_gelu(dA[0], dA[1], dA[2], dA[3], dA[4], yA, 4, DA, HA, DoA,
                             fm.FMLP_GELU_ERF, wsA, wsA.numel(), stream=s)
            fm.fmlp_mlp_gelu(dxb, W1b, db1b, yA.view(DoB, HB), db2b, yB, 1, DB, HB, DoB,
                             fm.FMLP_GELU_ERF, wsB, wsB.numel(), stream=s)
    s.synchronize()
    yA_bits, W1b_bits = to_host(yA), to_host(W1b)
    assert np.any(W1b_bits != 0)
    assert_parity(yA_bits, oracle.mlp_gelu(xa, W1a, b1a, W2a, b2a), "decode block A")
    assert_parity(to_host(yB), oracle.mlp_gelu(xb, W1b_bits, b1b, yA_bits.reshape(DoB, HB), b2b),
                  "decode block B on A's output")
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


def test_decode_grid_barrier_wait_runs_out_and_reports():
    """With more CTAs than can be resident, the resident ones wait at the grid barrier for CTAs
    that cannot start until they leave: the bounded wait runs out (2 ms here), the kernel
    records the timeout and returns; the status word reports it. The barrier counter heals
    (every CTA still arrives once), so the next normal call is correct."""
    T, D, H, Dout = 1, 2048, 2048, 2048
    x, b1, b2 = rbits((T, D)), ubits((H,), 0.02), ubits((Dout,), 0.02)
    W1, W2 = fast_ubits((H, D), 1 / 45, 81), fast_ubits((Dout, H), 1 / 45, 82)
    assert fm.fmlp_device_status() == fm.FMLP_OK
    # three times the SM count more CTAs than one per SM: whatever the residency, some wait
    fm.fmlp_test_decode_overload(3 * torch.cuda.get_device_properties(0).multi_processor_count,
                                 2000)
    try:
        run_mlp(x, W1, b1, W2, b2, fm.FMLP_GELU_ERF)
    finally:
        fm.fmlp_test_decode_overload(0, 0)
    assert fm.fmlp_device_status() == fm.FMLP_ERR_DEVICE_TIMEOUT
    assert "grid barrier" in fm.fmlp_last_error()
    assert fm.fmlp_device_status() == fm.FMLP_OK          # read and cleared
    for _ in range(2):
        got = run_mlp(x, W1, b1, W2, b2, fm.FMLP_GELU_ERF)
        assert_parity(got, oracle.mlp_gelu(x, W1, b1, W2, b2), "decode after a timeout")
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()
