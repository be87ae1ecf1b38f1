"""Torch tensor -> numpy raw-code conversions used by the tests (no arithmetic)."""

import numpy as np
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy array of its bit patterns."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint8)


def i32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().astype(np.int32)


def oracle_args(inp):
    """Positional oracle inputs of a workloads.Inputs (all numpy, CPU)."""
    return dict(q_bits=bf16_bits(inp.q), kv_codes=u8(inp.kv), pages=i32(inp.pages),
                indptr=i32(inp.indptr), scale=inp.scale, kv_scale=inp.kv_scale,
                heads=inp.heads, qlen=inp.qlen)
