"""The seeded input generator against its published definition (SplitMix64 + Box-Muller)."""
import math

import numpy as np

import synth

MASK = (1 << 64) - 1


def splitmix_mix(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def test_words_match_splitmix64_definition():
    for seed in (0, 1, 5003, 2**63 + 7):
        key = splitmix_mix(seed & MASK)
        for i in (0, 1, 2, 12345, 2**40 + 3):
            expect = splitmix_mix((key + (i + 1) * 0x9E3779B97F4A7C15) & MASK)
            assert synth.word(seed, i) == expect


def test_splitmix64_reference_sequence():
    # SplitMix64 seeded with 0 (state += golden gamma, then mix): published first outputs.
    state = 0
    outs = []
    for _ in range(3):
        state = (state + 0x9E3779B97F4A7C15) & MASK
        outs.append(splitmix_mix(state))
    assert outs[0] == 0xE220A8397B1DCDAF
    assert outs[1] == 0x6E789E6AA1B965F4
    assert outs[2] == 0x06C45D188009454F


def test_uniform_values_follow_definition():
    seed, bound, n = 2001, 0.125, 4096
    a = np.empty(n, dtype=np.uint16)
    synth.fill_bf16(a, n, seed, "uniform", bound, threads=1)
    v = synth.bf16_bits_to_f32(a).astype(np.float64)
    key = splitmix_mix(seed)
    for i in (0, 1, 77, 4095):
        w = splitmix_mix((key + (i + 1) * 0x9E3779B97F4A7C15) & MASK)
        u = (w >> 11) * 2.0 ** -53
        exact = bound * (2 * u - 1)
        # nearest bf16: |v - exact| <= half an ulp of bf16 at that magnitude
        half_ulp = 2.0 ** (math.frexp(abs(exact))[1] - 9) if exact != 0 else 0
        assert abs(v[i] - exact) <= half_ulp + 1e-300
    assert np.all(np.abs(v) <= bound)


def test_normal_moments_and_threads_independence():
    n = 1 << 20
    a1 = np.empty(n, dtype=np.uint16)
    a8 = np.empty(n, dtype=np.uint16)
    synth.fill_bf16(a1, n, 77, "normal", threads=1)
    synth.fill_bf16(a8, n, 77, "normal", threads=8)
    assert np.array_equal(a1, a8)
    v = synth.bf16_bits_to_f32(a1).astype(np.float64)
    assert abs(v.mean()) < 5e-3
    assert abs(v.std() - 1.0) < 5e-3
    assert abs((v > 1.0).mean() - 0.158655) < 3e-3     # 1 - Phi(1)


def test_workloads_shapes_and_seeds():
    w = synth.WORKLOADS["geglu_8192x768x3072"]
    assert w.spec("Wg").shape == (3072, 768) and w.spec("Wd").shape == (768, 3072)
    assert w.seed(w.spec("x")) == 4000 and w.seed(w.spec("Wd")) == 4003
    # GEMM flop count of one GeGLU GEMM at [8192, 768, 3072]: 2*8192*768*3072 ~ 38.7 GFLOP
    assert w.flops() // 3 == 38_654_705_664
    t1 = synth.WORKLOADS["mlp_4096_t1"].generate(["x"])["x"]
    t4 = synth.WORKLOADS["mlp_4096_t4096"].generate(["x"])["x"]
    assert np.array_equal(t1[0], t4[0])   # same seed: decode row == first row of the batch
