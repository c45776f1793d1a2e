"""The *_strided calls on row-strided views (slices of wider tensors, as in "What's the
transpose doing?") through every plan: fmlp_linear_bias_strided on the GEMV (one token), the
few-token kernel and the single-SM and CTA-pair tcgen05 GEMMs; fmlp_geglu_strided and
fmlp_mlp_gelu_strided on the single-kernel fused block, the one-kernel decode, the few-token
and the batched kernels. The columns outside the output view stay untouched."""
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


def _views(x, T, K, N, xpad, ypad):
    xbuf = rne_bf16_array(rng.standard_normal((T, xpad + K + 24)))
    xbuf[:, xpad:xpad + K] = x
    ybuf = np.full((T, ypad + N + 8), FILL, np.uint16)
    dx, dy = to_dev(xbuf), to_dev(ybuf)
    return dx, dy, dx[:, xpad:xpad + K], dy[:, ypad:ypad + N]


# T, D, H, extra columns left of x / of y, and the plan each size takes
GEGLU_CASES = [(300, 64, 200, 8, 16, fm.FMLP_PLAN_FUSED_SMALL),
               (3, 768, 3072, 16, 8, fm.FMLP_PLAN_DECODE),
               (1, 768, 3072, 16, 8, fm.FMLP_PLAN_GEMV),
               (40, 520, 1032, 8, 24, fm.FMLP_PLAN_TC),             # few-token kernels
               (700, 512, 1024, 32, 64, fm.FMLP_PLAN_TC)]           # batched tiles


@pytest.mark.parametrize("T,D,H,xpad,ypad,plan", GEGLU_CASES)
def test_geglu_on_column_slices(T, D, H, xpad, ypad, plan, request):
    if plan == fm.FMLP_PLAN_DECODE:
        request.getfixturevalue("prefer_decode")
    assert fm.fmlp_geglu_plan(T, D, H) == plan
    x = bits((T, D), 2.0)
    Wg, Wu = bits((H, D), 1 / math.sqrt(D)), bits((H, D), 1 / math.sqrt(D))
    Wd = bits((D, H), 1 / math.sqrt(H))
    dx, dy, xv, yv = _views(x, T, D, D, xpad, ypad)
    ws = torch.empty(max(1, fm.fmlp_geglu_workspace_size(T, D, H)), dtype=torch.uint8,
                     device="cuda")
    fm.fmlp_geglu_strided(xv, to_dev(Wg), to_dev(Wu), to_dev(Wd), yv, T, D, H, ws, ws.numel())
    torch.cuda.synchronize()
    out = to_host(dy)
    assert_parity(np.ascontiguousarray(out[:, ypad:ypad + D]), oracle.geglu(x, Wg, Wu, Wd),
                  f"strided geglu {T}x{D}x{H}")
    assert np.all(out[:, :ypad] == FILL) and np.all(out[:, ypad + D:] == FILL)
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


MLP_CASES = [(100, 40, 72, 48, 8, 16, fm.FMLP_PLAN_FUSED_SMALL),
             (1, 4096, 4096, 4096, 64, 128, fm.FMLP_PLAN_DECODE),
             (1, 4096, 4096, 4096, 64, 128, fm.FMLP_PLAN_GEMV),
             (20, 1024, 2048, 520, 8, 8, fm.FMLP_PLAN_TC),
             (600, 384, 1040, 264, 16, 32, fm.FMLP_PLAN_TC)]


@pytest.mark.parametrize("T,D,H,Do,xpad,ypad,plan", MLP_CASES)
def test_mlp_on_column_slices(T, D, H, Do, xpad, ypad, plan, request):
    if plan == fm.FMLP_PLAN_DECODE:
        request.getfixturevalue("prefer_decode")
    assert fm.fmlp_mlp_gelu_plan(T, D, H, Do) == plan
    x = bits((T, D), 2.0)
    W1, b1 = bits((H, D), 1 / math.sqrt(D)), bits((H,), 1 / math.sqrt(D))
    W2, b2 = bits((Do, H), 1 / math.sqrt(H)), bits((Do,), 1 / math.sqrt(H))
    dx, dy, xv, yv = _views(x, T, D, Do, xpad, ypad)
    ws = torch.empty(max(1, fm.fmlp_mlp_gelu_workspace_size(T, D, H, Do)), dtype=torch.uint8,
                     device="cuda")
    fm.fmlp_mlp_gelu_strided(xv, to_dev(W1), to_dev(b1), to_dev(W2), to_dev(b2), yv, T, D, H, Do,
                             fm.FMLP_GELU_ERF, ws, ws.numel())
    torch.cuda.synchronize()
    out = to_host(dy)
    assert_parity(np.ascontiguousarray(out[:, ypad:ypad + Do]),
                  oracle.mlp_gelu(x, W1, b1, W2, b2, gelu_mode=oracle.GELU_ERF),
                  f"strided mlp {T}x{D}x{H}x{Do}")
    assert np.all(out[:, :ypad] == FILL) and np.all(out[:, ypad + Do:] == FILL)
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


def test_strided_block_rejects_bad_strides():
    T, D, H = 8, 64, 128
    a = 0x10000
    with pytest.raises(fm.FmlpError) as e:
        fm.fmlp_geglu_strided(a, a, a, a, a + (1 << 24), T, D, H, ldx=60, ldy=64)
    assert e.value.status == fm.FMLP_ERR_SHAPE          # ldx < D
    with pytest.raises(fm.FmlpError) as e:
        fm.fmlp_mlp_gelu_strided(a, a, None, a, None, a + (1 << 24), T, D, H, D, ldx=68, ldy=64)
    assert e.value.status == fm.FMLP_ERR_ALIGN          # ldx not a multiple of 8
