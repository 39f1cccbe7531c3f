"""Helpers for the GPU tests: move generator output to the device and back."""
import numpy as np
import torch


def bf16_dev(bits, device="cuda"):
    """uint16 BF16 patterns -> torch.bfloat16 tensor on the device (exact)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def bf16_host_bits(t):
    """torch.bfloat16 tensor -> uint16 numpy patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_values(t):
    """torch.bfloat16 tensor -> float64 numpy values (exact)."""
    return t.detach().cpu().float().numpy().astype(np.float64)


def dev(arr, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)
