"""fmlp_moe_geglu (per-expert GeGLU over tokens grouped by expert, one launch per GEMM stage
over all experts) against the oracle: uneven groups with empty experts and groups that end
inside a 128-row tile, one expert, identical experts, offsets written on the stream just
before the call, and the same bits from call to call."""
import math

import numpy as np
import pytest
import torch

import feed_forward_gemm_gb300 as fm
import oracle
from gpu_util import DEV, guarded_bf16, to_dev, to_host, workspace
from helpers import assert_parity, rne_bf16_array

pytestmark = pytest.mark.gpu

rng = np.random.default_rng(8)


def bits(shape, bound):
    return rne_bf16_array(rng.uniform(-bound, bound, shape))


def experts(E, D, H):
    return (bits((E, H, D), 1 / math.sqrt(D)), bits((E, H, D), 1 / math.sqrt(D)),
            bits((E, D, H), 1 / math.sqrt(H)))


def run(x, offsets, Wg, Wu, Wd, T, D, H, E):
    dev = [to_dev(a) for a in (x, Wg, Wu, Wd)]
    off = torch.tensor(offsets, dtype=torch.int32, device=DEV)
    _, y, check = guarded_bf16(T, D)
    ws = workspace(fm.fmlp_moe_geglu_workspace_size(T, D, H))
    fm.fmlp_moe_geglu(dev[0], off, dev[1], dev[2], dev[3], y, T, D, H, E, ws, ws.numel())
    torch.cuda.synchronize()
    check()
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()
    return to_host(y)


@pytest.mark.parametrize("counts", [[130, 0, 257, 1, 300, 12, 200, 100],   # T = 1000
                                    [0, 0, 640, 0],                         # one busy expert
                                    [5, 3, 0, 7, 1, 9, 2, 4, 6, 8, 0, 11]])  # tiny groups
def test_moe_vs_oracle(counts):
    E, D, H = len(counts), 512, 1024
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    T = int(offsets[-1])
    x = bits((T, D), 2.0)
    Wg, Wu, Wd = experts(E, D, H)
    y = run(x, offsets, Wg, Wu, Wd, T, D, H, E)
    assert_parity(y, oracle.moe_geglu(x, offsets, Wg, Wu, Wd), f"moe {counts}")


def test_moe_single_sm_tiles_vs_oracle():
    """The grouped single-SM kernel (tile policy forced to single-SM tiles) on uneven groups."""
    counts = [130, 0, 257, 1, 300, 12]
    E, D, H = len(counts), 512, 768
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    T = int(offsets[-1])
    x = bits((T, D), 2.0)
    Wg, Wu, Wd = experts(E, D, H)
    try:
        fm.fmlp_set_tile_policy(fm.FMLP_TILES_SINGLE)
        y = run(x, offsets, Wg, Wu, Wd, T, D, H, E)
    finally:
        fm.fmlp_set_tile_policy(fm.FMLP_TILES_AUTO)
    assert_parity(y, oracle.moe_geglu(x, offsets, Wg, Wu, Wd), "moe single-SM tiles")


def test_moe_one_expert_and_identical_experts_are_the_plain_block():
    T, D, H = 300, 256, 768
    x = bits((T, D), 2.0)
    Wg, Wu, Wd = experts(1, D, H)
    ref = oracle.geglu(x, Wg[0], Wu[0], Wd[0])
    assert_parity(run(x, [0, T], Wg, Wu, Wd, T, D, H, 1), ref, "one expert")
    stack = lambda w: np.ascontiguousarray(np.repeat(w, 5, axis=0))
    y5 = run(x, [0, 10, 150, 151, 290, T], stack(Wg), stack(Wu), stack(Wd), T, D, H, 5)
    assert_parity(y5, ref, "identical experts")


def test_moe_offsets_written_just_before_and_same_bits():
    """A routing step writes the offsets on the stream right before the call; the kernels read
    them only after waiting for it. Repeated calls give the same bits."""
    E, D, H = 6, 512, 512
    counts = [100, 0, 333, 64, 1, 2]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(offsets[-1])
    x = bits((T, D), 2.0)
    Wg, Wu, Wd = experts(E, D, H)
    dx, dg, du, dd = (to_dev(a) for a in (x, Wg, Wu, Wd))
    ws = workspace(fm.fmlp_moe_geglu_workspace_size(T, D, H))
    host = torch.from_numpy(offsets).pin_memory()
    s = torch.cuda.Stream()
    outs = []
    for _ in range(3):
        off = torch.full((E + 1,), 12345, dtype=torch.int32, device=DEV)   # stale contents
        y = torch.empty((T, D), dtype=torch.bfloat16, device=DEV)
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            off.copy_(host, non_blocking=True)
            fm.fmlp_moe_geglu(dx, off, dg, du, dd, y, T, D, H, E, ws, ws.numel(), stream=s)
        s.synchronize()
        outs.append(to_host(y))
    assert all(np.array_equal(o, outs[0]) for o in outs[1:])
    assert_parity(outs[0], oracle.moe_geglu(x, offsets, Wg, Wu, Wd), "moe after routing")


def test_moe_mixtral_shaped_layer_at_the_benchmarked_size():
    """The benchmarked layer: 8 experts, D 4096, H 14336, 16,384 routed rows in groups of
    768..4096 (seeded synth inputs, the benchmark's own). Long K (64 K steps per tile) and
    groups spanning many 256-row tiles; 256 seeded rows of every expert group against the
    oracle."""
    import synth
    w = synth.MOE_WORKLOADS["moe_geglu_8x4096x14336"]
    t = w.generate()
    off = w.offsets()
    dx, dg, du, dd = (to_dev(t[k]) for k in ("x", "Wg", "Wu", "Wd"))
    y = torch.empty((w.T, w.D), dtype=torch.bfloat16, device=DEV)
    ws = workspace(fm.fmlp_moe_geglu_workspace_size(w.T, w.D, w.H))
    fm.fmlp_moe_geglu(dx, torch.tensor(off, dtype=torch.int32, device=DEV), dg, du, dd, y, w.T,
                      w.D, w.H, w.E, ws, ws.numel())
    torch.cuda.synchronize()
    assert fm.fmlp_device_status() == fm.FMLP_OK, fm.fmlp_last_error()
    pick = np.random.default_rng(2024)
    rows = np.sort(np.concatenate([
        off[e] + pick.choice(off[e + 1] - off[e], 256, replace=False) for e in range(w.E)]))
    ref = oracle.moe_geglu(t["x"], off, t["Wg"], t["Wu"], t["Wd"], rows=rows)
    got = to_host(y)[rows]
    for e in range(w.E):
        sel = (rows >= off[e]) & (rows < off[e + 1])
        assert_parity(got[sel], ref[sel], f"mixtral-shaped layer, expert {e}")
