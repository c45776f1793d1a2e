"""Both layers of a few-token block in one launch (fmlp_test_fewtoken_block(1)): against the
oracle over the token counts of the band, bit for bit against the two few-token launches where
both layers take the same tiling, one kernel in a captured graph, graph replays and calls back
to back (the grid-barrier counter is never reset), interleaved with one-kernel decode calls on
the same stream (they share the counter), and on row-strided views."""
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
import oracle
from gpu_util import count_graph_kernels, empty_bf16, guarded_bf16, to_dev, to_host, workspace
from helpers import assert_parity, rne_bf16_array

pytestmark = pytest.mark.gpu
rng = np.random.default_rng(9090)
ONE_LAUNCH = "one few-token tcgen05 launch for both layers"


def ubits(shape, bound):
    return rne_bf16_array(rng.uniform(-bound, bound, shape))


def rbits(shape):
    return rne_bf16_array(rng.standard_normal(shape))


def mlp_inputs(T, D, H, Dout):
    return (rbits((T, D)), ubits((H, D), 1 / math.sqrt(D)), ubits((H,), 1 / math.sqrt(D)),
            ubits((Dout, H), 1 / math.sqrt(H)), ubits((Dout,), 1 / math.sqrt(H)))


def geglu_inputs(T, D, H):
    return (rbits((T, D)), ubits((H, D), 1 / math.sqrt(D)), ubits((H, D), 1 / math.sqrt(D)),
            ubits((D, H), 1 / math.sqrt(H)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fm.load()
    yield
    fm.fmlp_test_fewtoken_block(0)
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


@pytest.fixture
def fused():
    fm.fmlp_test_fewtoken_block(1)
    yield
    fm.fmlp_test_fewtoken_block(0)


def run_mlp(ins, T, D, H, Dout, mode, stream=None):
    x, W1, b1, W2, b2 = (to_dev(a) for a in ins)
    _, y, check = guarded_bf16(T, Dout)
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(T, D, H, Dout))
    fm.fmlp_mlp_gelu(x, W1, b1, W2, b2, y, T, D, H, Dout, mode, ws, ws.numel(), stream=stream)
    torch.cuda.synchronize()
    check()
    return to_host(y)


def run_geglu(ins, T, D, H):
    x, Wg, Wu, Wd = (to_dev(a) for a in ins)
    _, y, check = guarded_bf16(T, D)
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
    fm.fmlp_geglu(x, Wg, Wu, Wd, y, T, D, H, ws, ws.numel())
    torch.cuda.synchronize()
    check()
    return to_host(y)


@pytest.mark.parametrize("T", [3, 5, 16, 33, 64, 100, 128])
def test_mlp_one_launch_vs_oracle(T, fused):
    D, H, Dout = 1024, 2048, 1032
    assert ONE_LAUNCH in fm.fmlp_describe_plan("mlp", T, D, H, Dout)
    ins = mlp_inputs(T, D, H, Dout)
    mode = [fm.FMLP_GELU_ERF, fm.FMLP_GELU_TANH, fm.FMLP_RELU][T % 3]
    omode = {0: oracle.GELU_TANH, 1: oracle.GELU_ERF, 2: oracle.RELU}[mode]
    assert_parity(run_mlp(ins, T, D, H, Dout, mode), oracle.mlp_gelu(*ins, gelu_mode=omode),
                  f"one-launch mlp T={T}")


@pytest.mark.parametrize("T", [2, 16, 64, 128])
def test_mlp_4096_one_launch_vs_oracle_and_two_launches(T):
    """The 4096-wide MLP: both layers take 36 tiles of 116 rows split 4 ways, as the two
    few-token launches do, so the results agree bit for bit."""
    D = H = Dout = 4096
    ins = mlp_inputs(T, D, H, Dout)
    fm.fmlp_test_fewtoken_block(-1)
    try:
        assert ONE_LAUNCH not in fm.fmlp_describe_plan("mlp", T, D, H, Dout)
        y2 = run_mlp(ins, T, D, H, Dout, fm.FMLP_GELU_ERF)
        fm.fmlp_test_fewtoken_block(1)
        assert ONE_LAUNCH in fm.fmlp_describe_plan("mlp", T, D, H, Dout)
        y1 = run_mlp(ins, T, D, H, Dout, fm.FMLP_GELU_ERF)
    finally:
        fm.fmlp_test_fewtoken_block(0)
    assert np.array_equal(y1, y2)
    assert_parity(y1, oracle.mlp_gelu(*ins, gelu_mode=oracle.GELU_ERF), f"4096 mlp T={T}")


@pytest.mark.parametrize("T,D,H", [(3, 768, 3072), (16, 768, 3072), (40, 520, 1032),
                                   (64, 768, 3072)])
def test_geglu_one_launch_vs_oracle(T, D, H, fused):
    assert ONE_LAUNCH in fm.fmlp_describe_plan("geglu", T, D, H)
    ins = geglu_inputs(T, D, H)
    assert_parity(run_geglu(ins, T, D, H), oracle.geglu(*ins), f"one-launch geglu T={T}")


def test_one_launch_is_one_kernel(fused):
    T, D, H = 16, 1024, 2048
    x, W1, b1, W2, b2 = (to_dev(a) for a in mlp_inputs(T, D, H, D))
    y = empty_bf16(T, D)
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(T, D, H, D))
    nk, nall = count_graph_kernels(lambda s: fm.fmlp_mlp_gelu(
        x, W1, b1, W2, b2, y, T, D, H, D, fm.FMLP_GELU_TANH, ws, ws.numel(), stream=s))
    assert nk == 1 and nall == 1


def test_graph_replays_back_to_back_and_beside_the_decode_plan(fused, prefer_decode):
    """The grid-barrier counter is shared with the one-kernel decode on a stream and never
    reset: calls queued without a synchronize, replays of a captured graph and decode-plan
    calls in between all give the same result."""
    T, D, H = 24, 1024, 2048
    ins = mlp_inputs(T, D, H, D)
    ref = run_mlp(ins, T, D, H, D, fm.FMLP_GELU_TANH)
    assert_parity(ref, oracle.mlp_gelu(*ins, gelu_mode=oracle.GELU_TANH), "reference run")
    x, W1, b1, W2, b2 = (to_dev(a) for a in ins)
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(T, D, H, D))
    x1 = to_dev(rbits((1, D)))
    y1 = empty_bf16(1, D)
    ws1 = workspace(fm.fmlp_mlp_gelu_workspace_size(1, D, H, D))
    assert fm.fmlp_mlp_gelu_plan(1, D, H, D) == fm.FMLP_PLAN_DECODE
    ys = [empty_bf16(T, D) for _ in range(4)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for y in ys:
            fm.fmlp_mlp_gelu(x, W1, b1, W2, b2, y, T, D, H, D, fm.FMLP_GELU_TANH, ws, ws.numel(),
                             stream=s)
            fm.fmlp_mlp_gelu(x1, W1, b1, W2, b2, y1, 1, D, H, D, fm.FMLP_GELU_TANH, ws1,
                             ws1.numel(), stream=s)
    torch.cuda.synchronize()
    for y in ys:
        assert np.array_equal(to_host(y), ref)
    g = torch.cuda.CUDAGraph()
    y = empty_bf16(T, D)
    with torch.cuda.graph(g, stream=s):
        fm.fmlp_mlp_gelu(x, W1, b1, W2, b2, y, T, D, H, D, fm.FMLP_GELU_TANH, ws, ws.numel(),
                         stream=s)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(to_host(y), ref)
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


def test_one_launch_on_row_strided_views(fused):
    T, D, H, xpad, ypad = 20, 1024, 2048, 16, 40
    x, W1, b1, W2, b2 = mlp_inputs(T, D, H, D)
    xbuf = rbits((T, xpad + D + 8))
    xbuf[:, xpad:xpad + D] = x
    ybuf = np.full((T, ypad + D + 24), 0x7FBF, np.uint16)
    dx, dy = to_dev(xbuf), to_dev(ybuf)
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(T, D, H, D))
    fm.fmlp_mlp_gelu_strided(dx[:, xpad:xpad + D], to_dev(W1), to_dev(b1), to_dev(W2), to_dev(b2),
                             dy[:, ypad:ypad + D], T, D, H, D, fm.FMLP_GELU_ERF, ws, ws.numel())
    torch.cuda.synchronize()
    out = to_host(dy)
    assert_parity(np.ascontiguousarray(out[:, ypad:ypad + D]),
                  oracle.mlp_gelu(x, W1, b1, W2, b2, gelu_mode=oracle.GELU_ERF), "strided")
    assert np.all(out[:, :ypad] == 0x7FBF) and np.all(out[:, ypad + D:] == 0x7FBF)


def test_one_launch_grid_barrier_wait_runs_out_and_reports(fused):
    """More CTAs than can be resident (whole clusters whose tiles lie past the last weight
    row): the resident ones wait at the grid barrier for CTAs that cannot start until they
    leave; the bounded wait runs out (2 ms), the status says where, and the counter heals
    (every CTA still arrives once), so the next calls are correct."""
    T, D, H = 16, 1024, 2048
    ins = mlp_inputs(T, D, H, D)
    assert fm.fmlp_device_status() == fm.FMLP_OK
    fm.fmlp_test_decode_overload(3 * torch.cuda.get_device_properties(0).multi_processor_count,
                                 2000)
    try:
        run_mlp(ins, T, D, H, D, fm.FMLP_GELU_TANH)
    finally:
        fm.fmlp_test_decode_overload(0, 0)
    assert fm.fmlp_device_status() == fm.FMLP_ERR_DEVICE_TIMEOUT
    assert "few-token block (grid barrier)" in fm.fmlp_last_error(), fm.fmlp_last_error()
    assert fm.fmlp_device_status() == fm.FMLP_OK
    ref = oracle.mlp_gelu(*ins, gelu_mode=oracle.GELU_TANH)
    for _ in range(2):
        assert_parity(run_mlp(ins, T, D, H, D, fm.FMLP_GELU_TANH), ref, "after a timeout")
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()
