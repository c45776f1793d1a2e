"""fmlp_geglu_noalloc, the entry point for callers that cannot allocate device memory, gives
the same result as fmlp_geglu with a caller-provided workspace and as the oracle, on two calls
in a row (the second call reuses the shared scratch the first one left behind), and it
allocates nothing: the high-water mark of the device's default memory pool (the pool that
cudaMallocAsync draws from) stays at zero across its calls, while a plain fmlp_geglu call
without a workspace moves it."""
import ctypes
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
import oracle
from gpu_util import _cudart, empty_bf16, to_dev, to_host, workspace
from helpers import assert_parity, rne_bf16_array

pytestmark = pytest.mark.gpu

POOL_USED_MEM_HIGH = 8   # cudaMemPoolAttrUsedMemHigh


def inputs(T, D, H, seed):
    rng = np.random.default_rng(seed)

    def u(shape, bound):
        return rne_bf16_array(rng.uniform(-bound, bound, shape))
    x = rne_bf16_array(rng.standard_normal((T, D)))
    return x, u((H, D), 1 / math.sqrt(D)), u((H, D), 1 / math.sqrt(D)), u((D, H), 1 / math.sqrt(H))


class DefaultPool:
    """The current device's default memory pool, read through the CUDA runtime."""

    def __init__(self):
        self.rt = _cudart()
        self.pool = ctypes.c_void_p()
        dev = torch.cuda.current_device()
        assert self.rt.cudaDeviceGetDefaultMemPool(ctypes.byref(self.pool), ctypes.c_int(dev)) == 0

    def reset_high(self):
        zero = ctypes.c_uint64(0)
        assert self.rt.cudaMemPoolSetAttribute(self.pool, ctypes.c_int(POOL_USED_MEM_HIGH),
                                               ctypes.byref(zero)) == 0

    def used_high(self) -> int:
        v = ctypes.c_uint64(0)
        assert self.rt.cudaMemPoolGetAttribute(self.pool, ctypes.c_int(POOL_USED_MEM_HIGH),
                                               ctypes.byref(v)) == 0
        return v.value


# a batched block (two tcgen05 kernels), the GEMV pair at two tokens, ragged sizes
@pytest.mark.parametrize("T,D,H", [(512, 768, 3072), (2, 768, 3072), (1000, 264, 1032)])
def test_noalloc_matches_workspace_call_and_oracle_twice(T, D, H):
    fm.load()
    assert fm.fmlp_geglu_workspace_size(T, D, H) > 0        # these sizes use the scratch
    pool = DefaultPool()
    for call in range(2):
        x, Wg, Wu, Wd = inputs(T, D, H, seed=100 * call + T)
        dx, dg, du, dd = to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd)
        y_ref = empty_bf16(T, D)
        ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
        fm.fmlp_geglu(dx, dg, du, dd, y_ref, T, D, H, ws, ws.numel())
        y = empty_bf16(T, D)
        torch.cuda.synchronize()
        pool.reset_high()
        fm.fmlp_geglu_noalloc(dx, dg, du, dd, y, T, D, H)
        torch.cuda.synchronize()
        assert pool.used_high() == 0, "fmlp_geglu_noalloc drew memory from the default pool"
        got = to_host(y)
        assert_parity(got, to_host(y_ref), f"noalloc call {call} {T}x{D}x{H} vs fmlp_geglu")
        assert_parity(got, oracle.geglu(x, Wg, Wu, Wd), f"noalloc call {call} {T}x{D}x{H} vs oracle")
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


def test_the_pool_probe_sees_an_allocating_call():
    """Positive control: fmlp_geglu without a workspace takes its T*H*2 bytes from the default
    pool (cudaMallocAsync), and the high-water mark shows it."""
    fm.load()
    T, D, H = 512, 768, 3072
    x, Wg, Wu, Wd = (to_dev(a) for a in inputs(T, D, H, seed=7))
    y = empty_bf16(T, D)
    pool = DefaultPool()
    torch.cuda.synchronize()
    pool.reset_high()
    fm.fmlp_geglu(x, Wg, Wu, Wd, y, T, D, H, None, 0)
    torch.cuda.synchronize()
    assert pool.used_high() >= T * H * 2


def test_noalloc_rejects_sizes_beyond_the_scratch_and_bad_shapes():
    fm.load()
    st = fm.fmlp_geglu_noalloc(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 65536, 768, 3072,
                               raise_on_error=False)
    assert st == fm.FMLP_ERR_WORKSPACE
    assert "scratch" in fm.fmlp_last_error()
    # a negative H (a multiple of 256, so T*H*2 would wrap to a huge size) is a shape error
    st = fm.fmlp_geglu_noalloc(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 4, 768, -256,
                               raise_on_error=False)
    assert st == fm.FMLP_ERR_SHAPE
    st = fm.fmlp_geglu_noalloc(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, -1, 768, 3072,
                               raise_on_error=False)
    assert st == fm.FMLP_ERR_SHAPE
