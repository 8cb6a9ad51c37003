"""Helpers for the GPU parity tests: move seeded numpy inputs to the device
and bring results back as raw bits."""
import numpy as np
import pytest
import torch

requires_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def dev():
    return torch.device("cuda:0")


def bf16(a):
    """uint16 bf16 bit patterns (numpy) -> bf16 CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev())


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def bits(t):
    """bf16 CUDA tensor -> uint16 bit patterns (numpy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
