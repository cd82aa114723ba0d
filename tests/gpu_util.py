"""Helpers for the GPU parity tests: numpy bf16 bit arrays <-> torch tensors."""

import numpy as np
import torch


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def padded_bf16(bits: np.ndarray, ld: int, device="cuda") -> torch.Tensor:
    """[rows, V] bits placed in a [rows, ld] bf16 buffer (padding = NaN, so a
    kernel that reads past V would be caught by a wrong answer), returned as a
    [rows, V] strided view."""
    rows, V = bits.shape
    full = np.full((rows, ld), 0x7FC0, np.uint16)
    full[:, :V] = bits
    return dev_bf16(full, device)[:, :V]
