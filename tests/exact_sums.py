"""Exact projection sums and their accumulation-error bounds, for the MATCH
acceptance check.

The GPU accumulates the gate and up projections in f32 (tensor-core MMAs and
f32 adds) in an order of its own; the oracle's f64 sums are exact for these
sizes (every product of two bf16 or f16 values is exact in f64, and the sums
carry far more bits than the projections are rounded to).  A stored projection
that differs from the correctly rounded value is a valid result only if it is
the rounding of some value the f32 accumulation can reach, i.e. within the
accumulation's error bound of the exact sum.

Bound (stated model, not a proof about the hardware): every accumulation step
-- one MMA instruction folding 16 products into the f32 accumulator, or one
f32 add of partial sums -- rounds or truncates once, with an error of at most
two f32 ulps of the magnitudes it combines, i.e. at most 2^-22 times
|accumulator| + the step's sum of |products| <= 2^-22 * sum_k |x_k * w_k|.
With `steps` such steps on the longest path of any term, the stored f32 sum is
within steps * 2^-22 * sum_k |x_k * w_k| of the exact sum.  The step counts of
the two kernels:

  tensor-core kernel: a chain of at most 22 K steps of 4 MMAs (K = 16 each),
    then one X += Y merge per later chain (ceil(nk / 22) chains, nk = K / 64
    steps), and at most one f32 add per stream-K contributor of a split tile
    (each contributor holds at least 8 K steps: ceil(nk / 8));
  small-M kernels: 8 chained MMAs per 128-code block into a fresh fragment,
    then f32 adds of the blocks' fragments and of partial sums.  Both kernels
    cut a unit's nkb = K / 128 blocks into P contiguous or interleaved pieces,
    one running sum each (at most nkb - P + 1 blocks, as many adds), and add
    the P partials: at most nkb + 1 adds on any path, whatever the split.
"""
from __future__ import annotations

import math

import numpy as np

import oracle
from tests.tolerances import TO_F64

F32_STEP = 2.0 ** -22


def accumulation_steps(kernel: str, K: int) -> int:
    if kernel == "tensor_core":
        nk = math.ceil(K / 64)
        return 4 * 22 + math.ceil(nk / 22) + math.ceil(nk / 8)
    if kernel == "small_m":
        nkb = math.ceil(K / 128)
        return 8 + nkb + 1
    raise ValueError(kernel)


def _operand_rows(q, rows, K, dtype):
    """Dequantised rows `rows` of a quantised operand, as exact doubles."""
    rows = np.asarray(rows)
    return oracle.dequant(q.packed[rows], q.scales[rows], q.biases[rows], K, q.gs, q.bits, dtype=dtype)


def projection_context(case, kernel: str, rows=None, pairs=None):
    """(g64, u64, bound_g, bound_u) for the selected outputs: all rows, the
    listed rows (all I columns), or the listed (m, i) pairs."""
    dt = case.dtype
    K = case.H
    x = TO_F64[dt](case.x)
    steps = accumulation_steps(kernel, K)
    out = []
    for q in (case.gate, case.up):
        if pairs is not None:
            m_idx, i_idx = pairs[:, 0], pairs[:, 1]
            uniq, pos = np.unique(i_idx, return_inverse=True)
            w = _operand_rows(q, uniq, K, dt)[pos]
            xs = x[m_idx]
            exact = np.einsum("nk,nk->n", xs, w)
            sabs = np.einsum("nk,nk->n", np.abs(xs), np.abs(w))
        else:
            xs = x if rows is None else x[np.asarray(rows)]
            w = _operand_rows(q, np.arange(case.I), K, dt)
            exact = xs @ w.T
            sabs = np.abs(xs) @ np.abs(w).T
        out.append((exact, steps * F32_STEP * sabs))
    (g64, bg), (u64, bu) = out
    return g64, u64, bg, bu
