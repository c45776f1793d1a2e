"""fmlp_linear_bias_wt: the Linear with its weight given transposed ([in, out], out
contiguous), read by the tcgen05 GEMM as an MN-major operand, against the oracle run on the
same weight in nn.Linear's [out, in] layout: ragged T, N tiles of 128 and 256, K of one
and many 64-deep steps, with and without bias, and the same result as fmlp_linear_bias."""
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
import oracle
from gpu_util import empty_bf16, guarded_bf16, to_dev, to_host
from helpers import assert_parity, rne_bf16_array

pytestmark = pytest.mark.gpu
rng = np.random.default_rng(5151)


def rbits(shape):
    return rne_bf16_array(rng.standard_normal(shape))


def ubits(shape, bound):
    return rne_bf16_array(rng.uniform(-bound, bound, shape))


@pytest.mark.parametrize("T,K,N", [(8, 64, 64), (300, 256, 384), (1000, 512, 1000),
                                   (130, 4096, 4096), (1, 72, 136)])
@pytest.mark.parametrize("with_bias", [True, False])
def test_transposed_weight_linear_vs_oracle(T, K, N, with_bias):
    x, W = rbits((T, K)), ubits((N, K), 1 / math.sqrt(K))
    b = ubits((N,), 1 / math.sqrt(K)) if with_bias else None
    Wt = np.ascontiguousarray(W.T)                       # [K, N], N contiguous
    _, y, check = guarded_bf16(T, N)
    fm.fmlp_linear_bias_wt(to_dev(x), to_dev(Wt), None if b is None else to_dev(b), y, T, K, N)
    torch.cuda.synchronize()
    check()
    got = to_host(y)
    assert_parity(got, oracle.linear(x, W, b), f"transposed-weight linear {T}x{K}->{N}")
    y2 = empty_bf16(T, N)
    fm.fmlp_linear_bias(to_dev(x), to_dev(W), None if b is None else to_dev(b), y2, T, K, N)
    torch.cuda.synchronize()
    assert_parity(got, to_host(y2), "transposed vs stored layout")
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


def test_transposed_weight_special_cases_bit_exact():
    """Identity weights give y = bf16(x + b) exactly; a weight that is one column of ones picks
    the sum of x's row (small integers: exact in fp32)."""
    T, K = 64, 256
    x = rne_bf16_array(rng.integers(-4, 5, (T, K)).astype(np.float64))
    b = rne_bf16_array(rng.integers(-3, 4, (K,)).astype(np.float64))
    eye = rne_bf16_array(np.eye(K))
    y = empty_bf16(T, K)
    fm.fmlp_linear_bias_wt(to_dev(x), to_dev(eye), to_dev(b), y, T, K, K)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(y), oracle.linear(x, eye, b))
    # W[n, k] = 1 for n == 3 only: Wt[k, 3] = 1
    W = np.zeros((128, K)); W[3, :] = 1.0
    W = rne_bf16_array(W)
    y = empty_bf16(T, 128)
    fm.fmlp_linear_bias_wt(to_dev(x), to_dev(np.ascontiguousarray(W.T)), None, y, T, K, 128)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(y), oracle.linear(x, W, None))
