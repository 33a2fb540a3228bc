"""Test helpers: host <-> device transfer of the workload's bf16 bits and
the comparison metrics the parity tests use (no method arithmetic)."""

import numpy as np
import torch


def dev_bf16(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).cuda()


def host_bf16_bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def rownorm_rel(x, y):
    """Per-row ||x - y||_2 / ||y||_2 over the last axis (flattened leading axes)."""
    x = np.asarray(x, np.float64).reshape(-1, np.shape(x)[-1])
    y = np.asarray(y, np.float64).reshape(-1, np.shape(y)[-1])
    return np.linalg.norm(x - y, axis=1) / np.maximum(np.linalg.norm(y, axis=1), 1e-300)
