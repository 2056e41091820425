"""Helpers for the GPU parity tests: move the seeded numpy inputs to CUDA
tensors and bring results back as float64.  No arithmetic of the method."""

import numpy as np

import synth_inputs as S

try:
    import torch
except ImportError:  # pragma: no cover
    torch = None


TORCH_DT = {}
if torch is not None:
    TORCH_DT = {S.F16: torch.float16, S.BF16: torch.bfloat16, S.F32: torch.float32}


def to_cuda(arr: np.ndarray, dtype: str, pitch: int | None = None):
    """Upload a stored array; optionally pad the last dimension to `pitch`
    elements and return a view of the original width (row pitch = pitch)."""
    if dtype == S.BF16:
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr))
    if pitch is not None and pitch != arr.shape[-1]:
        padded = torch.zeros(*arr.shape[:-1], pitch, dtype=t.dtype)
        padded[..., :arr.shape[-1]] = t
        return padded.cuda()[..., :arr.shape[-1]]
    return t.cuda()


def to_f64(t) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def empty_out(shape, dtype: str, pitch: int | None = None, fill: float = float("nan")):
    if pitch is None:
        return torch.full(shape, fill, dtype=TORCH_DT[dtype], device="cuda")
    full = torch.full((*shape[:-1], pitch), fill, dtype=TORCH_DT[dtype], device="cuda")
    return full[..., :shape[-1]]
