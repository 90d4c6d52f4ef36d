"""Helpers for the GPU parity tests: numpy <-> torch transfers of raw bit
patterns (bf16 as uint16, e4m3 / scale bytes as uint8) and sentinel buffers."""
import numpy as np
import torch

DEV = "cuda:0"


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(DEV)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(DEV)
    return torch.from_numpy(a).to(DEV)


def to_host(t: torch.Tensor, like: np.ndarray) -> np.ndarray:
    h = t.detach().cpu().contiguous().numpy()
    return h.view(like.dtype).reshape(like.shape)


def bf16_dev(a_u16: np.ndarray) -> torch.Tensor:
    return to_dev(a_u16).view(torch.bfloat16)


def bits_equal(a: np.ndarray, b: np.ndarray) -> bool:
    return a.shape == b.shape and np.array_equal(np.ascontiguousarray(a).view(np.uint8),
                                                 np.ascontiguousarray(b).view(np.uint8))


def first_mismatch(a: np.ndarray, b: np.ndarray):
    ia = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
    ib = np.ascontiguousarray(b).view(np.uint8).reshape(-1)
    d = np.flatnonzero(ia != ib)
    return None if d.size == 0 else (int(d[0]), int(d.size))


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (2^(floor(log2|x|) - 7)); 2^-133 at 0."""
    ax = np.abs(x)
    e = np.frexp(np.where(ax > 0, ax, 2.0 ** -126))[1] - 1
    return np.ldexp(1.0, e - 7)
