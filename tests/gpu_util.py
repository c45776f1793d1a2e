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
