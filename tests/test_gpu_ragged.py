"""Inner dimensions that are not multiples of 8 (packed rows): the Linear, the gate/up stage
and both blocks run on zero-padded copies and must give the oracle's result on the original
sizes, writing nothing past the output. Sizes cover the GEMV, the few-token and the batched
tiles, the single-kernel fused block, one-element tails and a dimension below 8."""
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
import oracle
from gpu_util import guarded_bf16, to_dev, to_host
from helpers import assert_parity, rne_bf16_array

pytestmark = pytest.mark.gpu
rng = np.random.default_rng(8080)


def rbits(shape):
    return rne_bf16_array(rng.standard_normal(shape))


def ubits(shape, bound):
    return rne_bf16_array(rng.uniform(-bound, bound, shape))


@pytest.mark.parametrize("T,K,N", [(1, 100, 37), (5, 12, 300), (130, 1000, 6), (300, 72, 130),
                                   (3, 4097, 33)])
@pytest.mark.parametrize("with_bias", [True, False])
def test_ragged_linear_vs_oracle(T, K, N, with_bias):
    assert "zero-padded" in fm.fmlp_describe_plan("linear", T, K, N)
    x, W = rbits((T, K)), ubits((N, K), 1 / math.sqrt(K))
    b = ubits((N,), 1 / math.sqrt(K)) if with_bias else None
    _, y, check = guarded_bf16(T, N)
    fm.fmlp_linear_bias(to_dev(x), to_dev(W), None if b is None else to_dev(b), y, T, K, N)
    torch.cuda.synchronize()
    check()
    assert_parity(to_host(y), oracle.linear(x, W, b), f"ragged linear {T}x{K}->{N}")
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


@pytest.mark.parametrize("mode", [fm.FMLP_GELU_TANH, fm.FMLP_GELU_ERF, fm.FMLP_RELU])
def test_ragged_linear_gelu_vs_oracle(mode):
    T, K, N = 40, 90, 110
    x, W, b = rbits((T, K)), ubits((N, K), 1 / math.sqrt(K)), ubits((N,), 0.1)
    _, h, check = guarded_bf16(T, N)
    fm.fmlp_linear_bias_gelu(to_dev(x), to_dev(W), to_dev(b), h, T, K, N, mode)
    torch.cuda.synchronize()
    check()
    om = {0: oracle.GELU_TANH, 1: oracle.GELU_ERF, 2: oracle.RELU}[mode]
    # the MLP oracle's h is bf16(act(x W^T + b)), the Linear + activation itself
    _, ref_h = oracle.mlp_gelu(x, W, b, rne_bf16_array(np.eye(N)), None, gelu_mode=om, want_h=True)
    assert_parity(to_host(h), ref_h, f"ragged linear+act mode {mode}")


@pytest.mark.parametrize("T,D,H", [(3, 20, 50), (200, 100, 36)])
def test_ragged_gate_up_vs_oracle(T, D, H):
    x, Wg, Wu = rbits((T, D)), ubits((H, D), 1 / math.sqrt(D)), ubits((H, D), 1 / math.sqrt(D))
    Wd = ubits((D, H), 1 / math.sqrt(H))
    _, m, check = guarded_bf16(T, H)
    fm.fmlp_geglu_gate_up(to_dev(x), to_dev(Wg), to_dev(Wu), m, T, D, H)
    torch.cuda.synchronize()
    check()
    _, ref_m = oracle.geglu(x, Wg, Wu, Wd, want_m=True)
    assert_parity(to_host(m), ref_m, f"ragged gate/up {T}x{D}x{H}")


@pytest.mark.parametrize("T,D,H", [(1, 100, 300), (7, 60, 44), (300, 100, 250), (2000, 36, 100),
                                   (64, 5, 9)])
def test_ragged_geglu_vs_oracle(T, D, H):
    assert fm.fmlp_geglu_workspace_size(T, D, H) == 0
    x, Wg, Wu = rbits((T, D)), ubits((H, D), 1 / math.sqrt(D)), ubits((H, D), 1 / math.sqrt(D))
    Wd = ubits((D, H), 1 / math.sqrt(H))
    _, y, check = guarded_bf16(T, D)
    fm.fmlp_geglu(to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd), y, T, D, H, None, 0)
    torch.cuda.synchronize()
    check()
    assert_parity(to_host(y), oracle.geglu(x, Wg, Wu, Wd), f"ragged geglu {T}x{D}x{H}")
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


@pytest.mark.parametrize("T,D,H,Do", [(1, 100, 250, 36), (64, 24, 40, 20), (513, 300, 100, 70),
                                      (4, 4093, 4096, 4090)])
@pytest.mark.parametrize("mode", [fm.FMLP_GELU_ERF, fm.FMLP_RELU])
def test_ragged_mlp_vs_oracle(T, D, H, Do, mode):
    x = rbits((T, D))
    W1, b1 = ubits((H, D), 1 / math.sqrt(D)), ubits((H,), 1 / math.sqrt(D))
    W2, b2 = ubits((Do, H), 1 / math.sqrt(H)), ubits((Do,), 1 / math.sqrt(H))
    _, y, check = guarded_bf16(T, Do)
    fm.fmlp_mlp_gelu(to_dev(x), to_dev(W1), to_dev(b1), to_dev(W2), to_dev(b2), y, T, D, H, Do,
                     mode, None, 0)
    torch.cuda.synchronize()
    check()
    om = {1: oracle.GELU_ERF, 2: oracle.RELU}[mode]
    assert_parity(to_host(y), oracle.mlp_gelu(x, W1, b1, W2, b2, gelu_mode=om),
                  f"ragged mlp {T}x{D}x{H}x{Do}")
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()
