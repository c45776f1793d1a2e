"""Moving bf16 bit patterns between numpy and CUDA tensors for the GPU tests."""
import numpy as np
import torch

DEV = torch.device("cuda:0")


def to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def to_host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def empty_bf16(*shape) -> torch.Tensor:
    return torch.empty(shape, dtype=torch.bfloat16, device=DEV)


def guarded_bf16(rows: int, cols: int, guard: int = 4096, pattern: int = 0x7FBF):
    """An output buffer with `guard` bf16 canaries before and after it. Returns (buffer,
    view, check) where check() asserts the canaries are intact."""
    n = rows * cols
    buf = torch.full((guard + n + guard,), pattern, dtype=torch.int16, device=DEV)
    view = buf[guard:guard + n].view(torch.bfloat16).view(rows, cols)

    def check():
        h = buf.cpu().numpy()
        assert np.all(h[:guard] == pattern), "write before the output buffer"
        assert np.all(h[guard + n:] == pattern), "write past the output buffer"
    return buf, view, check


def workspace(nbytes: int) -> torch.Tensor:
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=DEV)


def _cudart():
    """The CUDA runtime torch has already loaded (matched by soname)."""
    import ctypes
    for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    raise RuntimeError("no CUDA runtime library found")


def count_graph_kernels(fn):
    """Capture fn(stream) on a fresh stream into a CUDA graph; return (#kernel nodes, #nodes)."""
    import ctypes
    rt = _cudart()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn(s)                                   # warm-up outside the capture
    torch.cuda.synchronize()
    h = ctypes.c_void_p(s.cuda_stream)
    assert rt.cudaStreamBeginCapture(h, ctypes.c_int(1)) == 0   # thread-local mode
    try:
        fn(s)
    finally:
        graph = ctypes.c_void_p()
        rc = rt.cudaStreamEndCapture(h, ctypes.byref(graph))
    assert rc == 0, rc
    n = ctypes.c_size_t(0)
    assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * max(1, n.value))()
    assert rt.cudaGraphGetNodes(graph, nodes, ctypes.byref(n)) == 0
    kinds = []
    for i in range(n.value):
        ty = ctypes.c_int(-1)
        assert rt.cudaGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(ty)) == 0
        kinds.append(ty.value)
    rt.cudaGraphDestroy(graph)
    return sum(1 for k in kinds if k == 0), len(kinds)   # cudaGraphNodeTypeKernel == 0
