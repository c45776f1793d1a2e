"""Seeded synthetic inputs for the feed-forward block's workloads.

This module only draws input tensors (activations, weights, biases) as bfloat16 bit
patterns. It holds none of the block's arithmetic. Both the CUDA path's harness and the
oracle take their inputs from here, so the two see identical bits.

Workload shapes follow "Profiling in PyTorch (Part 2): From nn.Linear to a Fused MLP"
(sections "From matmul-add to Linear" for the single Linear, "Stacking three Linears:
the MLP" and "Why are there two kinds of GEMM kernels?" for the [64*128, 768, 3072]
GeGLU block) and the ainews.cool fused-MLP article's benchmark section (4096-wide
Linear->GELU->Linear). Values: activations ~ N(0, 1); weights and biases
~ U(-1/sqrt(in), 1/sqrt(in)), the nn.Linear default init bound; the 4096-wide MLP uses
U(-1/64, 1/64). The seed of tensor j of workload c is 1000*c + j (+100*r for the r-th
extra copy used to rotate weights through L2 in timing runs).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the generator (plain C, gcc, no fast-math) into synth/_build/libsynth.so."""
    src = os.path.join(_HERE, "synth.c")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src)):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                           "-ffp-contract=off", "-o", tmp, src, "-lm", "-lpthread"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.synth_fill_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64,
                                                   ctypes.c_uint64, ctypes.c_int]
            lib.synth_fill_normal_bf16.restype = ctypes.c_int
            lib.synth_fill_uniform_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64,
                                                    ctypes.c_uint64, ctypes.c_double,
                                                    ctypes.c_int]
            lib.synth_fill_uniform_bf16.restype = ctypes.c_int
            lib.synth_word.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.synth_word.restype = ctypes.c_uint64
            _lib = lib
    return _lib


def host_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def word(seed: int, i: int) -> int:
    """The raw 64-bit generator word for element i of seed `seed`."""
    return int(_load().synth_word(seed, i))


def fill_bf16(out: np.ndarray | int, n: int, seed: int, dist: str, bound: float = 0.0,
              threads: int | None = None) -> None:
    """Fill n bf16 values (as uint16 bits) into a numpy array or a raw host pointer."""
    lib = _load()
    ptr = out.ctypes.data if isinstance(out, np.ndarray) else int(out)
    if isinstance(out, np.ndarray):
        assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size >= n
    th = threads or host_threads()
    if dist == "normal":
        rc = lib.synth_fill_normal_bf16(ptr, n, seed, th)
    elif dist == "uniform":
        rc = lib.synth_fill_uniform_bf16(ptr, n, seed, float(bound), th)
    else:
        raise ValueError(dist)
    if rc != 0:
        raise RuntimeError("synth fill failed")


@dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple
    dist: str          # "normal" or "uniform"
    bound: float       # uniform half-width
    tid: int           # tensor id within the workload (seed = 1000*cid + tid)

    @property
    def numel(self) -> int:
        return int(np.prod(self.shape)) if self.shape else 1


@dataclass(frozen=True)
class Workload:
    name: str
    cid: int
    op: str            # "linear_bias" | "mlp_gelu" | "geglu"
    T: int
    D: int
    H: int             # hidden (GeGLU / MLP) or out_dim (linear)
    Dout: int
    tensors: tuple = field(default_factory=tuple)
    gelu: str = "tanh"

    def seed(self, spec: TensorSpec, replica: int = 0) -> int:
        return 1000 * self.cid + spec.tid + 100 * replica

    def spec(self, name: str) -> TensorSpec:
        for s in self.tensors:
            if s.name == name:
                return s
        raise KeyError(name)

    def flops(self) -> int:
        """GEMM flops (2 per multiply-add) of one forward; activations excluded."""
        if self.op == "linear_bias":
            return 2 * self.T * self.D * self.H
        if self.op == "mlp_gelu":
            return 2 * self.T * self.D * self.H + 2 * self.T * self.H * self.Dout
        return 3 * 2 * self.T * self.D * self.H   # gate, up, down

    def generate(self, names=None, replica: int = 0, threads: int | None = None) -> dict:
        """Draw the workload's tensors as numpy uint16 (bf16 bit) arrays."""
        out = {}
        for s in self.tensors:
            if names is not None and s.name not in names:
                continue
            arr = np.empty(s.shape, dtype=np.uint16)
            fill_bf16(arr, s.numel, self.seed(s, replica), s.dist, s.bound, threads)
            out[s.name] = arr
        return out


def _lin_bound(fan_in: int) -> float:
    return 1.0 / math.sqrt(fan_in)


def geglu_workload(name: str, cid: int, T: int, D: int, H: int) -> Workload:
    return Workload(name, cid, "geglu", T, D, H, D, (
        TensorSpec("x", (T, D), "normal", 0.0, 0),
        TensorSpec("Wg", (H, D), "uniform", _lin_bound(D), 1),
        TensorSpec("Wu", (H, D), "uniform", _lin_bound(D), 2),
        TensorSpec("Wd", (D, H), "uniform", _lin_bound(H), 3),
    ))


def linear_workload(name: str, cid: int, T: int, din: int, dout: int) -> Workload:
    return Workload(name, cid, "linear_bias", T, din, dout, dout, (
        TensorSpec("x", (T, din), "normal", 0.0, 0),
        TensorSpec("W", (dout, din), "uniform", _lin_bound(din), 1),
        TensorSpec("b", (dout,), "uniform", _lin_bound(din), 2),
    ))


def mlp_workload(name: str, cid: int, T: int, D: int, H: int, Dout: int, bound: float,
                 gelu: str = "erf") -> Workload:
    return Workload(name, cid, "mlp_gelu", T, D, H, Dout, (
        TensorSpec("x", (T, D), "normal", 0.0, 0),
        TensorSpec("W1", (H, D), "uniform", bound, 1),
        TensorSpec("b1", (H,), "uniform", bound, 2),
        TensorSpec("W2", (Dout, H), "uniform", bound, 3),
        TensorSpec("b2", (Dout,), "uniform", bound, 4),
    ), gelu)


# The five workloads: a small fully fused GeGLU block, a single Linear with bias, the
# 4096-wide Linear->GELU->Linear at one token (decode) and at 4096 tokens, the GPT-2-small
# GeGLU FFN (64*128 tokens, 768 -> 3072) and a 70B-class GeGLU FFN (8192 -> 28672).
WORKLOADS = {
    "geglu_1024x32x64": geglu_workload("geglu_1024x32x64", 1, 1024, 32, 64),
    "linear_1024x32x64": linear_workload("linear_1024x32x64", 2, 1024, 32, 64),
    "mlp_4096_t1": mlp_workload("mlp_4096_t1", 3, 1, 4096, 4096, 4096, 1.0 / 64),
    "mlp_4096_t4096": mlp_workload("mlp_4096_t4096", 3, 4096, 4096, 4096, 4096, 1.0 / 64),
    "geglu_8192x768x3072": geglu_workload("geglu_8192x768x3072", 4, 8192, 768, 3072),
    "geglu_8192x8192x28672": geglu_workload("geglu_8192x8192x28672", 5, 8192, 8192, 28672),
}


@dataclass(frozen=True)
class MoeWorkload(Workload):
    """E experts, each a GeGLU block; the T token rows arrive grouped by expert, `counts[e]`
    rows for expert e (a fixed routing layout: no trained router exists here)."""
    E: int = 1
    counts: tuple = ()

    def offsets(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.counts)]).astype(np.int32)

    def flops(self) -> int:
        return 3 * 2 * self.T * self.D * self.H


def moe_workload(name: str, cid: int, D: int, H: int, counts) -> MoeWorkload:
    E, T = len(counts), int(sum(counts))
    return MoeWorkload(name, cid, "moe_geglu", T, D, H, D, (
        TensorSpec("x", (T, D), "normal", 0.0, 0),
        TensorSpec("Wg", (E, H, D), "uniform", _lin_bound(D), 1),
        TensorSpec("Wu", (E, H, D), "uniform", _lin_bound(D), 2),
        TensorSpec("Wd", (E, D, H), "uniform", _lin_bound(H), 3),
    ), "tanh", E, tuple(int(c) for c in counts))


# A Mixtral-shaped mixture-of-experts layer (the ainews.cool article's MoE note names Mixtral
# 8x7B): 8 GeGLU experts, D 4096, H 14336, 16,384 routed token rows in uneven groups.
MOE_WORKLOADS = {
    "moe_geglu_8x4096x14336": moe_workload("moe_geglu_8x4096x14336", 6, 4096, 14336,
                                           (4096, 3072, 2560, 2048, 1536, 1280, 1024, 768)),
}


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 values (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32)
