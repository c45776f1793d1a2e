"""Failure detection on the real pipeline, made without faulting or hanging the GPU: a launch
refused on the host (injected), and the CTA-pair tcgen05 GEMM whose producers skip the loads
of one K step, so its MMA, producer and epilogue waits run out (bounded at 2 ms here), the
kernel returns and the status word reports the timeout. After each, a normal call gives the
oracle's result."""
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
import oracle
from gpu_util import empty_bf16, to_dev, to_host
from helpers import assert_parity, rne_bf16_array

pytestmark = pytest.mark.gpu
rng = np.random.default_rng(5150)


def bits(shape, bound):
    return rne_bf16_array(rng.uniform(-bound, bound, shape))


@pytest.fixture(autouse=True)
def _clean():
    fm.load()
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()
    yield
    fm.fmlp_test_inject(fm.FMLP_INJECT_NONE)


def linear_case(T, K, N):
    x, W, b = bits((T, K), 2.0), bits((N, K), 1 / math.sqrt(K)), bits((N,), 1 / math.sqrt(K))
    return x, W, b, to_dev(x), to_dev(W), to_dev(b)


def test_injected_launch_failure_is_reported_and_the_next_call_works():
    T, K, N = 512, 256, 512
    x, W, b, dx, dW, db = linear_case(T, K, N)
    y = empty_bf16(T, N)
    fm.fmlp_test_inject(fm.FMLP_INJECT_LAUNCH, 1)
    st = fm.fmlp_linear_bias(dx, dW, db, y, T, K, N, raise_on_error=False)
    assert st == fm.FMLP_ERR_CUDA
    assert "injected" in fm.fmlp_last_error()
    fm.fmlp_linear_bias(dx, dW, db, y, T, K, N)     # the injection was used up
    torch.cuda.synchronize()
    assert_parity(to_host(y), oracle.linear(x, W, b), "after an injected launch failure")
    assert fm.fmlp_device_status() == fm.FMLP_OK


def test_injected_failure_of_a_block_call():
    """A two-kernel block whose first launch is refused returns the error and launches
    nothing; the workspace it allocated itself is released (a later call still works)."""
    T, D, H = 300, 512, 1024
    x, Wg, Wu, Wd = (bits((T, D), 2.0), bits((H, D), 1 / math.sqrt(D)),
                     bits((H, D), 1 / math.sqrt(D)), bits((D, H), 1 / math.sqrt(H)))
    d = [to_dev(a) for a in (x, Wg, Wu, Wd)]
    y = empty_bf16(T, D)
    fm.fmlp_test_inject(fm.FMLP_INJECT_LAUNCH, 1)
    st = fm.fmlp_geglu(d[0], d[1], d[2], d[3], y, T, D, H, None, 0, raise_on_error=False)
    assert st == fm.FMLP_ERR_CUDA and "injected" in fm.fmlp_last_error()
    fm.fmlp_geglu(d[0], d[1], d[2], d[3], y, T, D, H, None, 0)
    torch.cuda.synchronize()
    assert_parity(to_host(y), oracle.geglu(x, Wg, Wu, Wd), "block after an injected failure")


@pytest.fixture
def pair_tiles():
    fm.fmlp_set_tile_policy(fm.FMLP_TILES_PAIR)
    yield
    fm.fmlp_set_tile_policy(fm.FMLP_TILES_AUTO)


def test_pair_gemm_skipped_load_runs_its_waits_out(pair_tiles):
    T, K, N = 1024, 1024, 2048
    assert "CTA-pair" in fm.fmlp_describe_plan("linear", T, K, N)
    x, W, b, dx, dW, db = linear_case(T, K, N)
    y = empty_bf16(T, N)
    fm.fmlp_test_inject(fm.FMLP_INJECT_SKIP_LOAD, 1, 2000)
    fm.fmlp_linear_bias(dx, dW, db, y, T, K, N)
    torch.cuda.synchronize()
    assert fm.fmlp_device_status() == fm.FMLP_ERR_DEVICE_TIMEOUT
    msg = fm.fmlp_last_error()
    assert any(site in msg for site in ("MMA (full slot)", "producer (empty slot)",
                                        "epilogue (accumulator)", "drain")), msg
    assert fm.fmlp_device_status() == fm.FMLP_OK          # read and cleared
    for _ in range(2):
        fm.fmlp_linear_bias(dx, dW, db, y, T, K, N)
        torch.cuda.synchronize()
        assert_parity(to_host(y), oracle.linear(x, W, b), "after the skipped load")
    assert fm.fmlp_device_status() == fm.FMLP_OK
