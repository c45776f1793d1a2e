"""fmlp_geglu_noalloc, the entry point for callers that cannot allocate device memory, gives
the same result as fmlp_geglu with a caller-provided workspace, on two calls in a row (the
second call reuses the shared scratch the first one left behind)."""
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
from gpu_util import empty_bf16, to_dev, to_host, workspace
from helpers import assert_parity, rne_bf16_array

pytestmark = pytest.mark.gpu


def inputs(T, D, H, seed):
    rng = np.random.default_rng(seed)

    def u(shape, bound):
        return to_dev(rne_bf16_array(rng.uniform(-bound, bound, shape)))
    x = to_dev(rne_bf16_array(rng.standard_normal((T, D))))
    return x, u((H, D), 1 / math.sqrt(D)), u((H, D), 1 / math.sqrt(D)), u((D, H), 1 / math.sqrt(H))


@pytest.mark.parametrize("T,D,H", [(512, 768, 3072), (2, 768, 3072), (1000, 264, 1032)])
def test_noalloc_matches_workspace_call_twice(T, D, H):
    fm.load()
    assert fm.fmlp_geglu_workspace_size(T, D, H) > 0        # these sizes use the scratch
    for call in range(2):
        x, Wg, Wu, Wd = inputs(T, D, H, seed=100 * call + T)
        y_ref = empty_bf16(T, D)
        ws = workspace(fm.fmlp_geglu_workspace_size(T, D, H))
        fm.fmlp_geglu(x, Wg, Wu, Wd, y_ref, T, D, H, ws, ws.numel())
        y = empty_bf16(T, D)
        fm.fmlp_geglu_noalloc(x, Wg, Wu, Wd, y, T, D, H)
        torch.cuda.synchronize()
        assert_parity(to_host(y), to_host(y_ref), f"noalloc call {call} {T}x{D}x{H}")
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()


def test_noalloc_rejects_sizes_beyond_the_scratch():
    fm.load()
    st = fm.fmlp_geglu_noalloc(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 65536, 768, 3072,
                               raise_on_error=False)
    assert st == fm.FMLP_ERR_WORKSPACE
    assert "scratch" in fm.fmlp_last_error()
