"""The few-token tcgen05 kernel (T <= 128 tokens: the weights are the MMA's M side and each
weight tile of up to 128 rows is split along K over a cluster of 1, 2, 4 or 8 CTAs, which
add their slices through distributed shared memory) against the oracle: ragged T, N and K,
partial tiles, every epilogue, the tiling rules, and the same bits from call to call."""
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
import oracle
from gpu_util import empty_bf16, guarded_bf16, to_dev, to_host, workspace
from helpers import assert_parity, rne_bf16_array

pytestmark = pytest.mark.gpu

rng = np.random.default_rng(2026)


def rbits(shape, scale=1.0):
    return rne_bf16_array(rng.standard_normal(shape) * scale)


def ubits(shape, bound):
    return rne_bf16_array(rng.uniform(-bound, bound, shape))


def tiling_of(text):
    """(weight rows per tile, K split, grid) from a few-token plan description."""
    rows = int(text.split(" weight rows")[0].split(", ")[-1])
    split = int(text.split("K split ")[1].split(" ")[0])
    grid = int(text.split("grid=")[1].split()[0].rstrip(","))
    return rows, split, grid


# T, K, N and the K split where the sizes force it: 128-row tiles already outnumber the SMs
# (no split), a single partial K step (none), two K steps (at most 2); the others (2 tiles of
# N over 17 K steps, the 4096-wide layer, one token with K not a multiple of 256, 7 tiles of
# 10 K steps) take whatever split fills the most SMs in one wave
LINEAR_CASES = [(33, 1032, 136, None), (5, 4096, 4096, None), (100, 72, 1000, 2),
                (128, 256, 28672, 1), (64, 8, 64, 1), (1, 4104, 520, None), (97, 640, 776, None)]


@pytest.mark.parametrize("T,K,N,split", LINEAR_CASES)
@pytest.mark.parametrize("with_bias", [True, False])
def test_fewtoken_linear_vs_oracle(T, K, N, split, with_bias):
    text = fm.fmlp_describe_plan("linear", T, K, N)
    assert "few-token" in text, text
    rows, S, grid = tiling_of(text)
    assert rows % 4 == 0 and 4 <= rows <= 128 and S in (1, 2, 4, 8), text
    assert grid == -(-N // rows) * S and S <= -(-K // 64), text
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert grid <= sms or (rows == 128 and S == 1), text     # one wave
    if split is not None:
        assert S == split, text
    x, W = rbits((T, K)), ubits((N, K), 1 / math.sqrt(K))
    b = ubits((N,), 1 / math.sqrt(K)) if with_bias else None
    _, y, check = guarded_bf16(T, N)
    fm.fmlp_linear_bias(to_dev(x), to_dev(W), None if b is None else to_dev(b), y, T, K, N)
    torch.cuda.synchronize()
    check()
    assert_parity(to_host(y), oracle.linear(x, W, b), f"few-token linear {T}x{K}->{N}")


def test_fewtoken_4096_layer_fills_more_sms_than_128_row_tiles():
    """The 4096-row layer: partial tiles (fewer than 128 weight rows) let more CTAs stream
    than the 32 x 4 = 128 of full 128-row tiles."""
    rows, S, grid = tiling_of(fm.fmlp_describe_plan("linear", 16, 4096, 4096))
    assert grid > 128 or rows == 128, (rows, S, grid)


@pytest.mark.parametrize("mode", [fm.FMLP_GELU_TANH, fm.FMLP_GELU_ERF, fm.FMLP_RELU])
def test_fewtoken_mlp_vs_oracle(mode):
    T, D, H, Do = 50, 1024, 2048, 520
    x = rbits((T, D))
    W1, b1 = ubits((H, D), 1 / math.sqrt(D)), ubits((H,), 1 / math.sqrt(D))
    W2, b2 = ubits((Do, H), 1 / math.sqrt(H)), ubits((Do,), 1 / math.sqrt(H))
    assert fm.fmlp_describe_plan("mlp", T, D, H, Do).count("few-token") == 2
    _, y, check = guarded_bf16(T, Do)
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(T, D, H, Do))
    fm.fmlp_mlp_gelu(to_dev(x), to_dev(W1), to_dev(b1), to_dev(W2), to_dev(b2), y, T, D, H, Do,
                     mode, ws, ws.numel())
    torch.cuda.synchronize()
    check()
    om = {0: oracle.GELU_TANH, 1: oracle.GELU_ERF, 2: oracle.RELU}[mode]
    assert_parity(to_host(y), oracle.mlp_gelu(x, W1, b1, W2, b2, gelu_mode=om),
                  f"few-token mlp mode {mode}")


@pytest.mark.parametrize("T,D,H", [(17, 768, 3072), (96, 512, 1288), (5, 8192, 1024)])
def test_fewtoken_geglu_vs_oracle(T, D, H):
    """Gate and up share the token tile: two accumulators per CTA, gelu_tanh(g)*u after the
    cluster adds the slices."""
    assert fm.fmlp_geglu_plan(T, D, H) == fm.FMLP_PLAN_TC
    assert fm.fmlp_describe_plan("geglu", T, D, H).count("few-token") == 2
    x, Wg, Wu = rbits((T, D)), ubits((H, D), 1 / math.sqrt(D)), ubits((H, D), 1 / math.sqrt(D))
    Wd = ubits((D, H), 1 / math.sqrt(H))
    dx, dg, du, dd = to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd)
    _, y, check = guarded_bf16(T, D)
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
    fm.fmlp_geglu(dx, dg, du, dd, y, T, D, H, ws, ws.numel())
    m = empty_bf16(T, H)
    fm.fmlp_geglu_gate_up(dx, dg, du, m, T, D, H)
    torch.cuda.synchronize()
    check()
    ref_y, ref_m = oracle.geglu(x, Wg, Wu, Wd, want_m=True)
    assert_parity(to_host(y), ref_y, f"few-token geglu {T}x{D}x{H}")
    assert_parity(to_host(m), ref_m, f"few-token gate/up {T}x{D}x{H}")


def test_fewtoken_same_bits_every_call():
    T, K, N = 33, 1032, 136
    x, W, b = to_dev(rbits((T, K))), to_dev(ubits((N, K), 0.03)), to_dev(ubits((N,), 0.03))
    outs = []
    for _ in range(4):
        y = empty_bf16(T, N)
        fm.fmlp_linear_bias(x, W, b, y, T, K, N)
        torch.cuda.synchronize()
        outs.append(to_host(y))
    assert all(np.array_equal(o, outs[0]) for o in outs[1:])
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


def test_single_sm_tiles_policy_keeps_the_batched_kernel():
    """With the tile policy forced to single-SM tiles the same call runs the batched kernel;
    both give the oracle's result."""
    T, K, N = 40, 512, 384
    x, W, b = rbits((T, K)), ubits((N, K), 1 / math.sqrt(K)), ubits((N,), 1 / math.sqrt(K))
    ref = oracle.linear(x, W, b)
    try:
        fm.fmlp_set_tile_policy(fm.FMLP_TILES_SINGLE)
        assert "single-SM" in fm.fmlp_describe_plan("linear", T, K, N)
        y = empty_bf16(T, N)
        fm.fmlp_linear_bias(to_dev(x), to_dev(W), to_dev(b), y, T, K, N)
        torch.cuda.synchronize()
        assert_parity(to_host(y), ref, "single-SM tiles at 40 tokens")
    finally:
        fm.fmlp_set_tile_policy(fm.FMLP_TILES_AUTO)
