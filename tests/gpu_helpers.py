"""Device transfer helpers of the GPU tests (not collected as tests)."""
from __future__ import annotations

import numpy as np
import torch


def dev():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA GPU"
    return torch.device("cuda:0")


def bf(bits: np.ndarray) -> torch.Tensor:
    """bf16 bits (uint16) -> a bf16 CUDA tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev()).view(torch.bfloat16)


def f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


def i32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev())


def f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def npi(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def lib():
    import token_dispatch_grouped_softmax_gb300 as moe

    moe.build()
    moe.load()
    return moe
