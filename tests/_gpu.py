"""Shared set-up for the GPU tests: the built library on cuda:0 and the
conversions between numpy arrays (oracle side) and CUDA tensors."""
from __future__ import annotations

import numpy as np
import pytest


def require_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_fine_grained_fp8bs_gb300 as fp8bs
    fp8bs.build()
    fp8bs.load_library()
    return torch, fp8bs


def to_dev_bf16(bits: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to("cuda:0")


def to_dev(arr: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr)).to("cuda:0")


def to_host(t) -> np.ndarray:
    import torch
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy()
