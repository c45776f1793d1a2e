"""The two-stage block launch (both layers of a GeGLU or MLP block in one persistent CTA-pair
kernel, the down tiles of a 256-row band waiting on a counter for that band's first-layer
tiles): against the oracle, bit for bit against the two-launch path on the same tiles, in a
CUDA graph replayed several times (the band counters are put back to zero by each launch),
back to back on one stream, on row-strided views, and with a band count that is never reached
(every down tile's bounded wait runs out, the status says where, later calls are correct)."""
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
import oracle
from gpu_util import count_graph_kernels, empty_bf16, guarded_bf16, to_dev, to_host, workspace
from helpers import assert_parity, rne_bf16_array

pytestmark = pytest.mark.gpu
rng = np.random.default_rng(4242)
ONE_LAUNCH = "one tcgen05 CTA-pair launch for both layers"


def ubits(shape, bound):
    return rne_bf16_array(rng.uniform(-bound, bound, shape))


def rbits(shape):
    return rne_bf16_array(rng.standard_normal(shape))


def geglu_inputs(T, D, H):
    return (rbits((T, D)), ubits((H, D), 1 / math.sqrt(D)), ubits((H, D), 1 / math.sqrt(D)),
            ubits((D, H), 1 / math.sqrt(H)))


def mlp_inputs(T, D, H, Dout):
    return (rbits((T, D)), ubits((H, D), 1 / math.sqrt(D)), ubits((H,), 1 / math.sqrt(D)),
            ubits((Dout, H), 1 / math.sqrt(H)), ubits((Dout,), 1 / math.sqrt(H)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fm.load()
    yield
    fm.fmlp_test_two_stage(0)
    fm.fmlp_test_inject(fm.FMLP_INJECT_NONE)
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


@pytest.fixture
def two_stage():
    fm.fmlp_test_two_stage(1)
    yield
    fm.fmlp_test_two_stage(0)


def run_geglu(ins, T, D, H, stream=None):
    x, Wg, Wu, Wd = (to_dev(a) for a in ins)
    _, y, check = guarded_bf16(T, D)
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
    fm.fmlp_geglu(x, Wg, Wu, Wd, y, T, D, H, ws, ws.numel(), stream=stream)
    torch.cuda.synchronize()
    check()
    return to_host(y)


def run_mlp(ins, T, D, H, Dout, mode):
    x, W1, b1, W2, b2 = (to_dev(a) for a in ins)
    _, y, check = guarded_bf16(T, Dout)
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(T, D, H, Dout))
    fm.fmlp_mlp_gelu(x, W1, b1, W2, b2, y, T, D, H, Dout, mode, ws, ws.numel())
    torch.cuda.synchronize()
    check()
    return to_host(y)


# T ragged against the 256-row bands, H against the 128/256-wide first-stage tiles, D against
# the 256-wide down tiles; the GPT-2-small block at 8192 tokens (sampled rows)
GEGLU_CASES = [(300, 320, 512), (1000, 512, 1032), (777, 776, 2056), (2048, 768, 3072)]


@pytest.mark.parametrize("T,D,H", GEGLU_CASES)
def test_geglu_two_stage_vs_oracle(T, D, H, two_stage):
    assert ONE_LAUNCH in fm.fmlp_describe_plan("geglu", T, D, H)
    ins = geglu_inputs(T, D, H)
    assert_parity(run_geglu(ins, T, D, H), oracle.geglu(*ins), f"two-stage geglu {T}x{D}x{H}")


def test_geglu_gpt2_small_8192_tokens_sampled_rows():
    """The automatic plan takes the two-stage launch at T=8192, D=768, H=3072."""
    T, D, H = 8192, 768, 3072
    assert ONE_LAUNCH in fm.fmlp_describe_plan("geglu", T, D, H)
    ins = geglu_inputs(T, D, H)
    y = run_geglu(ins, T, D, H)
    rows = np.sort(rng.choice(T, 96, replace=False))
    rows[:2] = [0, T - 1]
    rows = np.unique(np.concatenate([rows, [255, 256, 4095, 4096, 8191 - 256]]))
    assert_parity(np.ascontiguousarray(y[rows]), oracle.geglu(*ins, rows=rows),
                  "two-stage GPT-2-small block, sampled rows")


@pytest.mark.parametrize("T,D,H,Dout,mode", [(520, 512, 1024, 776, fm.FMLP_GELU_TANH),
                                             (1000, 1024, 2048, 1024, fm.FMLP_GELU_ERF),
                                             (257, 264, 784, 256, fm.FMLP_RELU)])
def test_mlp_two_stage_vs_oracle(T, D, H, Dout, mode, two_stage):
    assert ONE_LAUNCH in fm.fmlp_describe_plan("mlp", T, D, H, Dout)
    ins = mlp_inputs(T, D, H, Dout)
    assert_parity(run_mlp(ins, T, D, H, Dout, mode), oracle.mlp_gelu(*ins, gelu_mode=mode),
                  f"two-stage mlp {T}x{D}x{H}x{Dout}")


@pytest.mark.parametrize("T,D,H", [(1000, 512, 1032), (2048, 768, 3072), (777, 776, 2056)])
def test_geglu_two_stage_bit_identical_to_two_launches(T, D, H):
    """Same 256-row tiles, same K order, same roundings: the one-launch and two-launch paths
    agree bit for bit under the CTA-pair tile policy."""
    ins = geglu_inputs(T, D, H)
    fm.fmlp_set_tile_policy(fm.FMLP_TILES_PAIR)
    try:
        fm.fmlp_test_two_stage(-1)
        assert ONE_LAUNCH not in fm.fmlp_describe_plan("geglu", T, D, H)
        y2 = run_geglu(ins, T, D, H)
        fm.fmlp_test_two_stage(1)
        assert ONE_LAUNCH in fm.fmlp_describe_plan("geglu", T, D, H)
        y1 = run_geglu(ins, T, D, H)
    finally:
        fm.fmlp_test_two_stage(0)
        fm.fmlp_set_tile_policy(fm.FMLP_TILES_AUTO)
    assert np.array_equal(y1, y2)


def test_mlp_two_stage_bit_identical_to_two_launches():
    T, D, H, Dout = 1000, 1024, 2048, 776
    ins = mlp_inputs(T, D, H, Dout)
    fm.fmlp_set_tile_policy(fm.FMLP_TILES_PAIR)
    try:
        fm.fmlp_test_two_stage(-1)
        y2 = run_mlp(ins, T, D, H, Dout, fm.FMLP_GELU_TANH)
        fm.fmlp_test_two_stage(1)
        y1 = run_mlp(ins, T, D, H, Dout, fm.FMLP_GELU_TANH)
    finally:
        fm.fmlp_test_two_stage(0)
        fm.fmlp_set_tile_policy(fm.FMLP_TILES_AUTO)
    assert np.array_equal(y1, y2)


def test_two_stage_is_one_kernel(two_stage):
    T, D, H = 1000, 512, 1032
    x, Wg, Wu, Wd = (to_dev(a) for a in geglu_inputs(T, D, H))
    y = empty_bf16(T, D)
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
    nk, nall = count_graph_kernels(
        lambda s: fm.fmlp_geglu(x, Wg, Wu, Wd, y, T, D, H, ws, ws.numel(), stream=s))
    assert nk == 1 and nall == 1


def test_two_stage_graph_replays_and_back_to_back_calls(two_stage):
    """Each launch leaves its band counters at zero for the next one on the stream: replays of
    one captured graph, and calls queued without a synchronize in between, all match."""
    T, D, H = 777, 776, 2056
    ins = geglu_inputs(T, D, H)
    ref = run_geglu(ins, T, D, H)
    assert_parity(ref, oracle.geglu(*ins), "reference run")
    x, Wg, Wu, Wd = (to_dev(a) for a in ins)
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
    ys = [empty_bf16(T, D) for _ in range(4)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for y in ys:
            fm.fmlp_geglu(x, Wg, Wu, Wd, y, T, D, H, ws, ws.numel(), stream=s)
    torch.cuda.synchronize()
    for y in ys:
        assert np.array_equal(to_host(y), ref)
    g = torch.cuda.CUDAGraph()
    y = empty_bf16(T, D)
    with torch.cuda.stream(s):
        fm.fmlp_geglu(x, Wg, Wu, Wd, y, T, D, H, ws, ws.numel(), stream=s)   # warm-up
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        fm.fmlp_geglu(x, Wg, Wu, Wd, y, T, D, H, ws, ws.numel(), stream=s)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(to_host(y), ref)
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


def test_two_stage_on_row_strided_views(two_stage):
    T, D, H, xpad, ypad = 700, 512, 1024, 32, 64
    x, Wg, Wu, Wd = geglu_inputs(T, D, H)
    xbuf = rbits((T, xpad + D + 24))
    xbuf[:, xpad:xpad + D] = x
    ybuf = np.full((T, ypad + D + 8), 0x7FBF, np.uint16)
    dx, dy = to_dev(xbuf), to_dev(ybuf)
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
    assert ONE_LAUNCH in fm.fmlp_describe_plan("geglu", T, D, H)
    fm.fmlp_geglu_strided(dx[:, xpad:xpad + D], to_dev(Wg), to_dev(Wu), to_dev(Wd),
                          dy[:, ypad:ypad + D], T, D, H, ws, ws.numel())
    torch.cuda.synchronize()
    out = to_host(dy)
    assert_parity(np.ascontiguousarray(out[:, ypad:ypad + D]), oracle.geglu(x, Wg, Wu, Wd),
                  "two-stage strided")
    assert np.all(out[:, :ypad] == 0x7FBF) and np.all(out[:, ypad + D:] == 0x7FBF)


def test_two_stage_band_wait_runs_out(two_stage):
    """A band count one above what the first-layer tiles add: every down tile's wait runs out
    after 2 ms, the launch records FMLP_ERR_DEVICE_TIMEOUT and ends; the counters are back at
    zero, so the next calls are correct."""
    T, D, H = 1000, 512, 1032
    ins = geglu_inputs(T, D, H)
    x, Wg, Wu, Wd = (to_dev(a) for a in ins)
    y = empty_bf16(T, D)
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
    fm.fmlp_test_inject(fm.FMLP_INJECT_SKIP_LOAD, 1, 2000)
    fm.fmlp_geglu(x, Wg, Wu, Wd, y, T, D, H, ws, ws.numel())
    torch.cuda.synchronize()
    assert fm.fmlp_device_status() == fm.FMLP_ERR_DEVICE_TIMEOUT
    # the first wait to run out records its site: the band wait, or (started a little later,
    # but polled more often) the MMA's wait for the loads the band wait holds back
    msg = fm.fmlp_last_error()
    assert "band of the intermediate" in msg or "MMA (full slot)" in msg, msg
    assert fm.fmlp_device_status() == fm.FMLP_OK
    ref = oracle.geglu(*ins)
    for _ in range(2):
        assert_parity(run_geglu(ins, T, D, H), ref, "after the band wait ran out")
    assert fm.fmlp_device_status() == fm.FMLP_OK
