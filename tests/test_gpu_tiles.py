"""The single-SM (128-row) and CTA-pair (256-row, cta_group::2) tile kernels give the oracle's
result on the same shapes, including ragged M, N and K tails."""
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
import oracle
from gpu_util import guarded_bf16, to_dev, to_host, workspace
from helpers import assert_parity, rne_bf16_array

pytestmark = pytest.mark.gpu
rng = np.random.default_rng(4242)


def ubits(shape, bound):
    return rne_bf16_array(rng.uniform(-bound, bound, shape))


def rbits(shape):
    return rne_bf16_array(rng.standard_normal(shape))


@pytest.fixture(params=[fm.FMLP_TILES_SINGLE, fm.FMLP_TILES_PAIR], ids=["single", "pair"])
def policy(request):
    fm.load()
    fm.fmlp_set_tile_policy(request.param)
    yield request.param
    fm.fmlp_set_tile_policy(fm.FMLP_TILES_AUTO)
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


@pytest.mark.parametrize("T,K,N", [(129, 64, 64), (256, 256, 256), (300, 520, 776),
                                   (1000, 1024, 1032), (2048, 768, 3072)])
def test_linear_bias_both_tilings(policy, T, K, N):
    x, W, b = rbits((T, K)), ubits((N, K), 1 / math.sqrt(K)), ubits((N,), 1 / math.sqrt(K))
    _, y, check = guarded_bf16(T, N)
    fm.fmlp_linear_bias(to_dev(x), to_dev(W), to_dev(b), y, T, K, N)
    torch.cuda.synchronize()
    check()
    assert_parity(to_host(y), oracle.linear(x, W, b), f"linear {T}x{K}x{N} policy {policy}")


@pytest.mark.parametrize("T,D,H", [(257, 264, 200), (512, 512, 1024), (700, 320, 1544)])
def test_geglu_both_tilings(policy, T, D, H):
    x = rbits((T, D))
    Wg, Wu = ubits((H, D), 1 / math.sqrt(D)), ubits((H, D), 1 / math.sqrt(D))
    Wd = ubits((D, H), 1 / math.sqrt(H))
    assert fm.fmlp_geglu_plan(T, D, H) == fm.FMLP_PLAN_TC
    _, y, check = guarded_bf16(T, D)
    ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
    fm.fmlp_geglu(to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd), y, T, D, H, ws, ws.numel())
    torch.cuda.synchronize()
    check()
    assert_parity(to_host(y), oracle.geglu(x, Wg, Wu, Wd), f"geglu {T}x{D}x{H} policy {policy}")


@pytest.mark.parametrize("mode", [fm.FMLP_GELU_ERF, fm.FMLP_GELU_TANH])
def test_mlp_both_tilings(policy, mode):
    T, D, H, Do = 520, 384, 1040, 264
    x = rbits((T, D))
    W1, b1 = ubits((H, D), 1 / math.sqrt(D)), ubits((H,), 1 / math.sqrt(D))
    W2, b2 = ubits((Do, H), 1 / math.sqrt(H)), ubits((Do,), 1 / math.sqrt(H))
    _, y, check = guarded_bf16(T, Do)
    ws = workspace(fm.fmlp_mlp_gelu_workspace_size(T, D, H, Do))
    fm.fmlp_mlp_gelu(to_dev(x), to_dev(W1), to_dev(b1), to_dev(W2), to_dev(b2), y, T, D, H, Do,
                     mode, ws, ws.numel())
    torch.cuda.synchronize()
    check()
    om = oracle.GELU_ERF if mode == fm.FMLP_GELU_ERF else oracle.GELU_TANH
    assert_parity(to_host(y), oracle.mlp_gelu(x, W1, b1, W2, b2, gelu_mode=om), "mlp tilings")


def test_pair_and_single_agree_closely():
    T, K, N = 1024, 2048, 2048
    x, W = to_dev(rbits((T, K))), to_dev(ubits((N, K), 1 / math.sqrt(K)))
    outs = []
    for p in (fm.FMLP_TILES_SINGLE, fm.FMLP_TILES_PAIR):
        fm.fmlp_set_tile_policy(p)
        y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        fm.fmlp_linear_bias(x, W, None, y, T, K, N)
        torch.cuda.synchronize()
        outs.append(to_host(y))
    fm.fmlp_set_tile_policy(fm.FMLP_TILES_AUTO)
    # same products, fp32 sums in the same K order per tile: expect (near) bit equality
    diff = np.abs(outs[0].astype(np.int32) - outs[1].astype(np.int32))
    assert diff.max() <= 1
