"""Activation quantisation to int8 by absmax, stated plainly (test infrastructure; see the
package docstring).

inferencelayer ``cuda_llm.rs``: before every GEMV of an activation vector the engine computes
``xs = [max|x|, 1/max|x|]`` (``CudaQwen3::absmax``, the ``xs`` buffer "for the GEMV currently
in flight"), and the q4_0 GEMV reads the vector with that scale. The kernel body is not printed,
so the reading taken here is the plainest one for an int8 (dp4a) product:

* the scale is one per activation vector: ``m = max|x|`` over the vector;
* each element's code is ``q = round_half_even(x * (127 / m))`` in [-127, 127], a zero vector
  gives all-zero codes;
* the GEMV then multiplies the weights by ``x^ = q * (m / 127)``.

Where floating point decides the integer code, the decision is taken in f32 as on the page (its
``x`` and ``xs`` are f32): ``127 / m`` is one f32 division, ``x * (127 / m)`` one f32
multiplication, then the rounding to an integer. ``x^`` is returned in f64.
"""
from __future__ import annotations

import numpy as np

QMAX = 127


def absmax_codes(x) -> tuple[np.ndarray, np.ndarray]:
    """``x [..., n]`` -> (int8 codes ``[..., n]``, per-vector ``m = max|x|`` as f32 ``[..., 1]``)."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    m = np.max(np.abs(x32), axis=-1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        s = np.where(m > 0, np.float32(QMAX) / m, np.float32(0)).astype(np.float32)
        prod = (x32 * s).astype(np.float32)                 # one f32 multiplication
    q = np.clip(np.rint(prod), -QMAX, QMAX).astype(np.int8)  # np.rint: half to even
    return q, m


def absmax_dequant(x) -> np.ndarray:
    """The activation the int8 GEMV multiplies: ``q * (m / 127)`` in f64."""
    q, m = absmax_codes(x)
    return q.astype(np.float64) * (m.astype(np.float64) / QMAX)
