"""The pages' online-softmax algebra, restated in fp64 (test infrastructure).

Each function follows the steps in the order the pages give them, on one
query row.  They exist to pin the oracle and to check, on the CPU, that the
blocked / conditionally rescaled formulation the kernel uses reaches the plain
definition.

* ``block_state`` / ``merge``: "Infra: Flash Attention", section "How softmax
  is computed in pieces" -- a processed block A keeps (m_A, l_A, u_A) with
  l_A = sum e^{x_j - m_A}, u_A = sum e^{x_j - m_A} V_j; two blocks merge with
  m = max(m_A, m_B), alpha = e^{m_A - m}, beta = e^{m_B - m},
  l = alpha l_A + beta l_B, u = alpha u_A + beta u_B, O = u / l.
* ``flash_scan``: the same page, Algorithm 1 (FlashAttention forward): the
  running (m, l, U) updated per key/value tile with the exponent taken against
  the new maximum, fully masked tiles skipped, O = U / l and L = m + log l at
  the end.
* ``conditional_scan``: "Flash Attention 4 on Blackwell", section "Online
  softmax and conditional rescaling": scores in base 2 with the scale folded
  in (scale_log2 = log2(e) * scale); per block the candidate maximum is
  compared with the kept reference through
  delta = (row_max - candidate_max) * scale_log2; the first block takes its
  own maximum; delta >= -tau keeps the reference (acc_scale = 1); otherwise the
  reference moves to the candidate and the state is scaled by 2^delta.  The
  "Infra: Flash Attention" section "Why the exponent base need not be updated
  yet" gives the invariant that makes the result independent of the
  reference: u(r) / l(r) does not depend on r.
"""
from __future__ import annotations

import math

import numpy as np

LOG2E = 1.0 / math.log(2.0)


def block_state(x, values):
    """(m, l, u) of one block of scores x (natural units) and values [n, dv]."""
    x = np.asarray(x, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64).reshape(len(x), -1)
    m = float(np.max(x))
    w = np.exp(x - m)
    return m, float(np.sum(w)), w @ values


def merge(a, b):
    """Merge two block states into one against the common maximum."""
    m_a, l_a, u_a = a
    m_b, l_b, u_b = b
    m = max(m_a, m_b)
    alpha = math.exp(m_a - m)
    beta = math.exp(m_b - m)
    return m, alpha * l_a + beta * l_b, alpha * np.asarray(u_a) + beta * np.asarray(u_b)


def finish(state):
    """O = u / l and L = m + log l of a merged state."""
    m, l, u = state
    return np.asarray(u) / l, m + math.log(l)


def flash_scan(x, values, block: int, valid=None):
    """Algorithm 1 on one row: x [n] scores (scale applied), values [n, dv].

    ``valid`` (bool [n]) marks visible keys; tiles with no visible key are
    skipped.  Returns (O, L); a row with no visible key gives (0, -inf).
    """
    x = np.asarray(x, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64).reshape(len(x), -1)
    if valid is None:
        valid = np.ones(len(x), dtype=bool)
    m, l, U = -math.inf, 0.0, np.zeros(values.shape[1])
    for j0 in range(0, len(x), block):
        s = np.where(valid[j0:j0 + block], x[j0:j0 + block], -np.inf)
        if not np.any(np.isfinite(s)):
            continue  # whole tile masked for this row: skip the update
        m_new = max(m, float(np.max(s)))
        alpha = math.exp(m - m_new)  # 0 on the first visible tile
        w = np.exp(s - m_new)
        l = alpha * l + float(np.sum(w))
        U = alpha * U + w @ values[j0:j0 + block]
        m = m_new
    if l == 0.0:
        return np.zeros(values.shape[1]), -math.inf
    return U / l, m + math.log(l)


def conditional_scan(raw, values, block: int, scale: float, tau: float = 8.0, valid=None):
    """Conditional-rescaling scan on one row, in base 2 with the scale folded in.

    raw [n]: unscaled scores q.k; values [n, dv].  Returns (O, L, n_rescales)
    with L in natural-log units.  tau = inf never moves the reference after the
    first block; tau = 0 moves it whenever the maximum grows.
    """
    raw = np.asarray(raw, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64).reshape(len(raw), -1)
    if valid is None:
        valid = np.ones(len(raw), dtype=bool)
    scale_log2 = scale * LOG2E
    row_max = -math.inf  # kept reference, raw units
    row_sum = 0.0
    acc_o = np.zeros(values.shape[1])
    rescales = 0
    for j0 in range(0, len(raw), block):
        s = np.where(valid[j0:j0 + block], raw[j0:j0 + block], -np.inf)
        block_max = float(np.max(s))
        if block_max == -math.inf:
            continue  # no visible key in this block for this row
        if row_max == -math.inf:
            row_max = block_max  # first block: take its own maximum
            acc_scale = 1.0
        else:
            cand = max(row_max, block_max)
            delta = (row_max - cand) * scale_log2
            if delta >= -tau:
                acc_scale = 1.0  # keep the old reference
            else:
                acc_scale = 2.0 ** delta
                row_max = cand
                rescales += 1
        p = np.exp2(s * scale_log2 - row_max * scale_log2)
        row_sum = row_sum * acc_scale + float(np.sum(p))
        acc_o = acc_o * acc_scale + p @ values[j0:j0 + block]
    if row_sum == 0.0:
        return np.zeros(values.shape[1]), -math.inf, rescales
    lse = (row_max * scale_log2 + math.log2(row_sum)) * math.log(2.0)
    return acc_o / row_sum, lse, rescales
