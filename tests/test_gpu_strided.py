"""fmlp_linear_bias_strided on row-strided views (slices of wider tensors, as in "What's the
transpose doing?") through every plan: the GEMV (one token), the few-token kernel, and the
single-SM and CTA-pair tcgen05 GEMMs; the columns outside the output view stay untouched."""
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
import oracle
from gpu_util import to_dev, to_host
from helpers import assert_parity, rne_bf16_array

pytestmark = pytest.mark.gpu

rng = np.random.default_rng(77)
FILL = 0x7FBF   # a NaN pattern: any stray write into the untouched columns shows


def bits(shape, scale):
    return rne_bf16_array(rng.uniform(-scale, scale, shape))


# T, in, out, extra columns left of x / of y, and the plan each size takes
CASES = [(1, 4096, 1024, 64, 128, fm.FMLP_PLAN_GEMV),      # GEMV
         (40, 520, 776, 8, 24, fm.FMLP_PLAN_TC),            # few-token kernel
         (300, 256, 200, 16, 8, fm.FMLP_PLAN_TC),           # single-SM tiles (narrow)
         (1000, 1024, 2048, 32, 64, fm.FMLP_PLAN_TC)]       # CTA-pair tiles


@pytest.mark.parametrize("T,K,N,xpad,ypad,plan", CASES)
def test_linear_on_column_slices(T, K, N, xpad, ypad, plan):
    assert fm.fmlp_linear_plan(T, K, N) == plan
    x, W, b = bits((T, K), 2.0), bits((N, K), 1 / math.sqrt(K)), bits((N,), 1 / math.sqrt(K))
    xbuf = rne_bf16_array(rng.standard_normal((T, xpad + K + 40)))
    xbuf[:, xpad:xpad + K] = x
    ybuf = np.full((T, ypad + N + 16), FILL, np.uint16)
    dx, dy = to_dev(xbuf), to_dev(ybuf)
    xv, yv = dx[:, xpad:xpad + K], dy[:, ypad:ypad + N]
    fm.fmlp_linear_bias_strided(xv, to_dev(W), to_dev(b), yv, T, K, N)
    torch.cuda.synchronize()
    out = to_host(dy)
    assert_parity(np.ascontiguousarray(out[:, ypad:ypad + N]), oracle.linear(x, W, b),
                  f"strided linear {T}x{K}->{N}")
    assert np.all(out[:, :ypad] == FILL) and np.all(out[:, ypad + N:] == FILL)
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


@pytest.mark.parametrize("T", [1, 64, 512])
def test_input_and_output_are_column_blocks_of_one_buffer(T):
    """x = buf[:, :K] and y = buf[:, K:K+N]: same stride, rows interleaved, no element shared."""
    K, N = 512, 256
    x, W, b = bits((T, K), 2.0), bits((N, K), 1 / math.sqrt(K)), bits((N,), 1 / math.sqrt(K))
    buf = np.full((T, K + N), FILL, np.uint16)
    buf[:, :K] = x
    d = to_dev(buf)
    fm.fmlp_linear_bias_strided(d[:, :K], to_dev(W), to_dev(b), d[:, K:], T, K, N)
    torch.cuda.synchronize()
    out = to_host(d)
    assert np.array_equal(out[:, :K], x)                   # the input block is unchanged
    assert_parity(np.ascontiguousarray(out[:, K:]), oracle.linear(x, W, b), f"one buffer T={T}")
