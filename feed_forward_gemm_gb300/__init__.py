"""Python binding of the fmlp C ABI (include/fmlp.h): argument marshalling only.

Every entry point here has the C name and forwards plain device pointers and sizes to the
shared library built from csrc/. No computation happens in Python: if the library is
missing the import of a function fails loudly (there is no fallback of any kind).

Tensors may be passed as torch tensors (their data_ptr() is used; they must be contiguous
CUDA tensors of the documented shape) or as raw integer device addresses. `stream` may be a
torch.cuda.Stream, a raw cudaStream_t integer, or None for torch's current stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = [
    "FmlpError", "load", "build", "library_path",
    "fmlp_linear_bias", "fmlp_linear_bias_strided", "fmlp_linear_bias_gelu", "fmlp_linear_bias_wt",
    "fmlp_geglu_strided", "fmlp_mlp_gelu_strided",
    "fmlp_geglu_gate_up", "fmlp_geglu", "fmlp_moe_geglu", "fmlp_moe_geglu_workspace_size",
    "fmlp_mlp_gelu", "fmlp_geglu_workspace_size", "fmlp_mlp_gelu_workspace_size",
    "fmlp_geglu_plan", "fmlp_mlp_gelu_plan", "fmlp_linear_plan", "fmlp_gelu_eval",
    "fmlp_device_status", "fmlp_test_wait_timeout", "fmlp_status_string", "fmlp_last_error",
    "fmlp_version", "fmlp_set_tile_policy", "fmlp_describe_plan", "fmlp_geglu_noalloc", "FMLP_TILES_AUTO", "FMLP_TILES_SINGLE",
    "FMLP_TILES_PAIR",
    "FMLP_OK", "FMLP_ERR_NULL", "FMLP_ERR_SHAPE", "FMLP_ERR_ALIGN", "FMLP_ERR_ALIAS",
    "FMLP_ERR_WORKSPACE", "FMLP_ERR_CUDA", "FMLP_ERR_DEVICE_TIMEOUT", "FMLP_ERR_DEVICE",
    "FMLP_GELU_TANH", "FMLP_GELU_ERF", "FMLP_PLAN_NONE", "FMLP_PLAN_TC",
    "FMLP_PLAN_FUSED_SMALL", "FMLP_PLAN_GEMV", "FMLP_PLAN_DECODE", "fmlp_test_decode_overload",
    "fmlp_test_prefer_decode",
    "fmlp_test_two_stage",
    "fmlp_test_fewtoken_block",
    "fmlp_test_two_stage_schedule",
    "fmlp_test_inject", "FMLP_INJECT_NONE", "FMLP_INJECT_LAUNCH", "FMLP_INJECT_SKIP_LOAD",
]

FMLP_OK, FMLP_ERR_NULL, FMLP_ERR_SHAPE, FMLP_ERR_ALIGN, FMLP_ERR_ALIAS = 0, 1, 2, 3, 4
FMLP_ERR_WORKSPACE, FMLP_ERR_CUDA, FMLP_ERR_DEVICE_TIMEOUT, FMLP_ERR_DEVICE = 5, 6, 7, 8
FMLP_GELU_TANH, FMLP_GELU_ERF, FMLP_RELU = 0, 1, 2
FMLP_PLAN_NONE, FMLP_PLAN_TC, FMLP_PLAN_FUSED_SMALL, FMLP_PLAN_GEMV, FMLP_PLAN_DECODE = 0, 1, 2, 3, 4
FMLP_TILES_AUTO, FMLP_TILES_SINGLE, FMLP_TILES_PAIR = 0, 1, 2
FMLP_INJECT_NONE, FMLP_INJECT_LAUNCH, FMLP_INJECT_SKIP_LOAD = 0, 1, 2

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_INT = ctypes.c_int

# name -> (restype, argtypes); the order matches include/fmlp.h
_SIGNATURES = {
    "fmlp_linear_bias": (_INT, [_P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "fmlp_linear_bias_wt": (_INT, [_P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "fmlp_linear_bias_strided": (_INT, [_P, _I64, _P, _P, _P, _I64, _I64, _I64, _I64, _P]),
    "fmlp_moe_geglu": (_INT, [_P, _P, _I64, _P, _P, _P, _P, _I64, _I64, _I64, _P, ctypes.c_size_t,
                              _P]),
    "fmlp_moe_geglu_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64]),
    "fmlp_linear_bias_gelu": (_INT, [_P, _P, _P, _P, _I64, _I64, _I64, _INT, _P]),
    "fmlp_geglu_gate_up": (_INT, [_P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "fmlp_geglu": (_INT, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    "fmlp_mlp_gelu": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _INT, _P, _SZ, _P]),
    "fmlp_geglu_strided": (_INT, [_P, _I64, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _SZ, _P]),
    "fmlp_mlp_gelu_strided": (_INT, [_P, _I64, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64,
                                     _INT, _P, _SZ, _P]),
    "fmlp_geglu_workspace_size": (_SZ, [_I64, _I64, _I64]),
    "fmlp_mlp_gelu_workspace_size": (_SZ, [_I64, _I64, _I64, _I64]),
    "fmlp_geglu_plan": (_INT, [_I64, _I64, _I64]),
    "fmlp_mlp_gelu_plan": (_INT, [_I64, _I64, _I64, _I64]),
    "fmlp_linear_plan": (_INT, [_I64, _I64, _I64]),
    "fmlp_gelu_eval": (_INT, [_P, _P, _I64, _INT, _P]),
    "fmlp_device_status": (_INT, [_P]),
    "fmlp_test_wait_timeout": (_INT, [_I64, _P]),
    "fmlp_test_decode_overload": (_INT, [_I64, _I64]),
    "fmlp_test_prefer_decode": (_INT, [_INT]),
    "fmlp_test_two_stage": (_INT, [_INT]),
    "fmlp_test_fewtoken_block": (_INT, [_INT]),
    "fmlp_test_two_stage_schedule": (_INT, [_INT, _INT, _INT, _INT, _INT, _INT, _P, _P, _P]),
    "fmlp_test_inject": (_INT, [_INT, _I64, _I64]),
    "fmlp_status_string": (ctypes.c_char_p, [_INT]),
    "fmlp_last_error": (ctypes.c_char_p, []),
    "fmlp_version": (_INT, []),
    "fmlp_set_tile_policy": (_INT, [_INT]),
    "fmlp_describe_plan": (_INT, [_INT, _I64, _I64, _I64, _I64, ctypes.c_char_p, _SZ]),
    "fmlp_geglu_noalloc": (_INT, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
}


class FmlpError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where} -> status {status} ({_status_text(status)}): {detail}")


def library_path() -> str:
    return _build.LIB


def build(force: bool = False) -> str:
    return _build.build(force=force)


def load(build_if_missing: bool = False):
    """Load the shared library (raising if it is absent and build_if_missing is False)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise ImportError(
                    f"fmlp CUDA library not built ({path} missing); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            _build.build()
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _status_text(st: int) -> str:
    try:
        return load().fmlp_status_string(st).decode()
    except Exception:  # pragma: no cover
        return "?"


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        if hasattr(t, "is_contiguous") and not t.is_contiguous():
            raise ValueError("fmlp tensors must be contiguous")
        return t.data_ptr() or None
    raise TypeError(f"cannot take a device pointer from {type(t)!r}")


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(s, int):
        return s or None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream or None
    raise TypeError(f"cannot take a CUDA stream from {type(s)!r}")


def _check(st: int, where: str, raise_on_error: bool):
    if st != FMLP_OK and raise_on_error:
        raise FmlpError(st, where, fmlp_last_error())
    return st


def fmlp_status_string(st: int) -> str:
    return load().fmlp_status_string(int(st)).decode()


def fmlp_last_error() -> str:
    return load().fmlp_last_error().decode()


def fmlp_version() -> int:
    return int(load().fmlp_version())


def fmlp_linear_bias(x, W, b, y, T, in_dim, out_dim, stream=None, raise_on_error=True):
    st = load().fmlp_linear_bias(_ptr(x), _ptr(W), _ptr(b), _ptr(y), T, in_dim, out_dim,
                                 _stream(stream))
    return _check(st, "fmlp_linear_bias", raise_on_error)


def fmlp_linear_bias_wt(x, Wt, b, y, T, in_dim, out_dim, stream=None, raise_on_error=True):
    """y = x @ Wt + b with the weight given as [in, out] (the transposed layout)."""
    st = load().fmlp_linear_bias_wt(_ptr(x), _ptr(Wt), _ptr(b), _ptr(y), T, in_dim, out_dim,
                                    _stream(stream))
    return _check(st, "fmlp_linear_bias_wt", raise_on_error)


def _view(t, ld):
    """(device pointer, row stride in elements) of a row-major view whose rows may be apart."""
    if t is None or isinstance(t, int):
        return t, (0 if ld is None else int(ld))
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("fmlp strided views must be 2-D with unit column stride")
    return (t.data_ptr() or None), (t.stride(0) if ld is None else int(ld))


def fmlp_linear_bias_strided(x, W, b, y, T, in_dim, out_dim, ldx=None, ldy=None, stream=None,
                             raise_on_error=True):
    """fmlp_linear_bias on row-strided views; ldx/ldy default to the views' row strides."""
    px, lx = _view(x, ldx)
    py, ly = _view(y, ldy)
    st = load().fmlp_linear_bias_strided(px, lx, _ptr(W), _ptr(b), py, ly, T, in_dim, out_dim,
                                         _stream(stream))
    return _check(st, "fmlp_linear_bias_strided", raise_on_error)


def fmlp_moe_geglu(x, offsets, Wg, Wu, Wd, y, T, D, H, E, ws=None, ws_bytes=0, stream=None,
                   raise_on_error=True):
    """Per-expert GeGLU over tokens grouped by expert (offsets: E + 1 int32 on the device)."""
    st = load().fmlp_moe_geglu(_ptr(x), _ptr(offsets), E, _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(y),
                               T, D, H, _ptr(ws), int(ws_bytes), _stream(stream))
    return _check(st, "fmlp_moe_geglu", raise_on_error)


def fmlp_moe_geglu_workspace_size(T, D, H) -> int:
    return int(load().fmlp_moe_geglu_workspace_size(T, D, H))


def fmlp_linear_bias_gelu(x, W, b, h, T, in_dim, out_dim, mode=FMLP_GELU_TANH, stream=None,
                          raise_on_error=True):
    st = load().fmlp_linear_bias_gelu(_ptr(x), _ptr(W), _ptr(b), _ptr(h), T, in_dim, out_dim,
                                      int(mode), _stream(stream))
    return _check(st, "fmlp_linear_bias_gelu", raise_on_error)


def fmlp_geglu_gate_up(x, Wg, Wu, m, T, D, H, stream=None, raise_on_error=True):
    st = load().fmlp_geglu_gate_up(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(m), T, D, H,
                                   _stream(stream))
    return _check(st, "fmlp_geglu_gate_up", raise_on_error)


def fmlp_geglu(x, Wg, Wu, Wd, y, T, D, H, ws=None, ws_bytes=0, stream=None,
               raise_on_error=True):
    st = load().fmlp_geglu(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(y), T, D, H, _ptr(ws),
                           int(ws_bytes), _stream(stream))
    return _check(st, "fmlp_geglu", raise_on_error)


def fmlp_geglu_noalloc(x, Wg, Wu, Wd, y, T, D, H, stream=None, raise_on_error=True):
    """fmlp_geglu with the intermediate in the library's fixed device array (allocates
    nothing; T*H*2 bytes must fit in 64 MiB; overlapping calls race on the array)."""
    st = load().fmlp_geglu_noalloc(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(y), T, D, H,
                                   _stream(stream))
    return _check(st, "fmlp_geglu_noalloc", raise_on_error)


def fmlp_mlp_gelu(x, W1, b1, W2, b2, y, T, D, H, Dout, mode=FMLP_GELU_ERF, ws=None, ws_bytes=0,
                  stream=None, raise_on_error=True):
    st = load().fmlp_mlp_gelu(_ptr(x), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), _ptr(y), T, D, H,
                              Dout, int(mode), _ptr(ws), int(ws_bytes), _stream(stream))
    return _check(st, "fmlp_mlp_gelu", raise_on_error)


def fmlp_geglu_strided(x, Wg, Wu, Wd, y, T, D, H, ws=None, ws_bytes=0, ldx=None, ldy=None,
                       stream=None, raise_on_error=True):
    """fmlp_geglu on row-strided views of x and y; ldx/ldy default to the views' row strides."""
    px, lx = _view(x, ldx)
    py, ly = _view(y, ldy)
    st = load().fmlp_geglu_strided(px, lx, _ptr(Wg), _ptr(Wu), _ptr(Wd), py, ly, T, D, H,
                                   _ptr(ws), int(ws_bytes), _stream(stream))
    return _check(st, "fmlp_geglu_strided", raise_on_error)


def fmlp_mlp_gelu_strided(x, W1, b1, W2, b2, y, T, D, H, Dout, mode=FMLP_GELU_ERF, ws=None,
                          ws_bytes=0, ldx=None, ldy=None, stream=None, raise_on_error=True):
    """fmlp_mlp_gelu on row-strided views of x and y; ldx/ldy default to the views' strides."""
    px, lx = _view(x, ldx)
    py, ly = _view(y, ldy)
    st = load().fmlp_mlp_gelu_strided(px, lx, _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), py, ly, T,
                                      D, H, Dout, int(mode), _ptr(ws), int(ws_bytes),
                                      _stream(stream))
    return _check(st, "fmlp_mlp_gelu_strided", raise_on_error)


def fmlp_geglu_workspace_size(T, D, H) -> int:
    return int(load().fmlp_geglu_workspace_size(T, D, H))


def fmlp_mlp_gelu_workspace_size(T, D, H, Dout) -> int:
    return int(load().fmlp_mlp_gelu_workspace_size(T, D, H, Dout))


def fmlp_geglu_plan(T, D, H) -> int:
    return int(load().fmlp_geglu_plan(T, D, H))


def fmlp_mlp_gelu_plan(T, D, H, Dout) -> int:
    return int(load().fmlp_mlp_gelu_plan(T, D, H, Dout))


def fmlp_linear_plan(T, in_dim, out_dim) -> int:
    return int(load().fmlp_linear_plan(T, in_dim, out_dim))


def fmlp_gelu_eval(x, out, n, mode=FMLP_GELU_TANH, stream=None, raise_on_error=True):
    st = load().fmlp_gelu_eval(_ptr(x), _ptr(out), n, int(mode), _stream(stream))
    return _check(st, "fmlp_gelu_eval", raise_on_error)


PLAN_OPS = {"linear": 0, "linear_gelu": 1, "gate_up": 2, "geglu": 3, "mlp": 4}


def fmlp_describe_plan(op, T, D, H, Dout=0) -> str:
    """The kernels a call with these sizes launches on the current device, as text."""
    buf = ctypes.create_string_buffer(512)
    code = PLAN_OPS[op] if isinstance(op, str) else int(op)
    st = load().fmlp_describe_plan(code, T, D, H, Dout, buf, len(buf))
    _check(st, "fmlp_describe_plan", True)
    return buf.value.decode()


def fmlp_set_tile_policy(policy: int, raise_on_error=True):
    st = load().fmlp_set_tile_policy(int(policy))
    return _check(st, "fmlp_set_tile_policy", raise_on_error)


def fmlp_device_status(stream=None) -> int:
    return int(load().fmlp_device_status(_stream(stream)))


def fmlp_test_inject(kind, count=0, timeout_us=0, raise_on_error=True):
    """Failure-injection test hook (FMLP_INJECT_*); FMLP_INJECT_NONE clears everything."""
    st = load().fmlp_test_inject(int(kind), int(count), int(timeout_us))
    return _check(st, "fmlp_test_inject", raise_on_error)


def fmlp_test_decode_overload(extra_ctas, timeout_us, raise_on_error=True):
    """Test hook: later one-kernel decode launches get extra_ctas CTAs that cannot be resident
    and a wait limit of timeout_us (0: default); (0, 0) restores normal launches."""
    st = load().fmlp_test_decode_overload(int(extra_ctas), int(timeout_us))
    return _check(st, "fmlp_test_decode_overload", raise_on_error)


def fmlp_test_prefer_decode(on, raise_on_error=True):
    """Route 1..4-token GeGLU/MLP blocks to the one-kernel decode (process-wide switch)."""
    st = load().fmlp_test_prefer_decode(int(on))
    return _check(st, "fmlp_test_prefer_decode", raise_on_error)


def fmlp_test_two_stage(mode, raise_on_error=True):
    """Two-stage block launch: 0 automatic, 1 whenever accepted, -1 never (process-wide)."""
    st = load().fmlp_test_two_stage(int(mode))
    return _check(st, "fmlp_test_two_stage", raise_on_error)


def fmlp_test_two_stage_schedule(num_m, num_n1, num_n2, kb1, kb2, pairs):
    """The two-stage launch's item lists for a shape (host only): (start, items) as lists."""
    start = (ctypes.c_uint16 * (int(pairs) + 1))()
    item = (ctypes.c_uint16 * 2048)()
    n = ctypes.c_int64(0)
    st = load().fmlp_test_two_stage_schedule(int(num_m), int(num_n1), int(num_n2), int(kb1),
                                             int(kb2), int(pairs), start, item, ctypes.byref(n))
    _check(st, "fmlp_test_two_stage_schedule", True)
    return list(start), list(item[:n.value])


def fmlp_test_fewtoken_block(mode, raise_on_error=True):
    """Few-token block in one launch: 0 automatic, 1 whenever accepted, -1 never."""
    st = load().fmlp_test_fewtoken_block(int(mode))
    return _check(st, "fmlp_test_fewtoken_block", raise_on_error)


def fmlp_test_wait_timeout(timeout_us, stream=None, raise_on_error=True):
    st = load().fmlp_test_wait_timeout(int(timeout_us), _stream(stream))
    return _check(st, "fmlp_test_wait_timeout", raise_on_error)
