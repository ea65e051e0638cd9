"""Moving numpy arrays to and from CUDA tensors for the parity tests (uint32 via int32 views)."""

import numpy as np
import torch


def dev(a: np.ndarray, offset: int = 0) -> torch.Tensor:
    """Copy to a CUDA tensor of the same dtype.  offset > 0 places the data
    `offset` elements into a larger allocation, so the pointer is 4-byte but
    not 16-byte aligned (exercises the scalar kernels)."""
    a = np.ascontiguousarray(a)
    base = a.view(np.int32) if a.dtype == np.uint32 else a
    t = torch.from_numpy(base.copy())
    if offset:
        big = torch.zeros(t.numel() + offset, dtype=t.dtype)
        big[offset:] = t
        g = big.cuda()[offset:]
    else:
        g = t.cuda()
    return g.view(torch.uint32) if a.dtype == np.uint32 else g


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.uint32:
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    return t.cpu().numpy()


def empty_like_offset(t: torch.Tensor, offset: int = 0, fill: int = 0) -> torch.Tensor:
    """An output buffer of t's size and dtype, prefilled with a sentinel, optionally misaligned."""
    base_dtype = torch.int32 if t.dtype == torch.uint32 else t.dtype
    big = torch.full((t.numel() + offset,), fill, dtype=base_dtype, device=t.device)
    g = big[offset:]
    return g.view(torch.uint32) if t.dtype == torch.uint32 else g


def f32_within(got: np.ndarray, want64: np.ndarray, rel: float = 1e-5):
    """Every element within rel of the float64 value; exact where that value is 0."""
    got64 = got.astype(np.float64)
    err = np.abs(got64 - want64)
    bound = rel * np.abs(want64)
    bad = np.flatnonzero(err > bound)
    return bad, (float((err / np.maximum(np.abs(want64), 1e-300)).max()) if got.size else 0.0)
