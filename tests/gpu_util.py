"""Helpers for the GPU parity tests (device buffers via torch; oracle on the CPU)."""
import numpy as np
import torch

import quantized_transformer_decode_ql_gb300 as ql
from quantized_transformer_decode_ql_gb300 import build as _build

_built = False


def lib():
    global _built
    if not _built:
        _build.build()
        _built = True
    return ql


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def q4_dev(scales: np.ndarray, quants: np.ndarray):
    """Upload q4_0 bytes (u16 scale bits, u8 codes) as device tensors."""
    s = torch.from_numpy(np.ascontiguousarray(scales).view(np.int16)).cuda()
    q = torch.from_numpy(np.ascontiguousarray(quants)).cuda()
    return s, q


def rel_err(got, want):
    """max |got - want| / rms(want) (a scale-free error for one output vector set)."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    scale = np.sqrt(np.mean(want * want)) + 1e-300
    return float(np.max(np.abs(got - want)) / scale)
