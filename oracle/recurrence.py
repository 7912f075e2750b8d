"""Tiled online-softmax recurrences from the pages, in fp64 numpy (test infrastructure).

These follow the pages' steps in their order and notation.  They exist to pin the oracle's
three-pass definition in ``attn_oracle.c``: Theorem 1 of the FlashAttention paper says that
after every outer step the running statistics equal the softmax statistics of the prefix seen
so far, so the recurrence and the definition must agree at every block boundary.

Readings taken (the pages disagree with themselves here):
  * The FlashAttention-2 reading notes write the rescale of the running output in eq. (10) and
    Algorithm 1 (forward) line "O_i = diag(exp(m_old - m_new))^{-1} O_i + P V_j" with an
    inverse.  Their own two-block proof, eq. (13), and the worked example on the wmrh.cn page
    multiply by exp(m_old - m_new).  We multiply: that is the only form under which eq. (14)
    holds.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np


def online_softmax_tiles(tiles: Sequence[Sequence[float]]) -> List[Tuple[float, float]]:
    """Running (m, l) after each tile of one score row.

    wmrh.cn page, "Online Softmax" walk-through: for each tile, m_new = max(m, max(tile)),
    l_new = l * exp(m - m_new) + sum(exp(tile - m_new)); start from m = -inf, l = 0.
    """
    m, l = -np.inf, 0.0
    out = []
    for t in tiles:
        x = np.asarray(t, dtype=np.float64)
        m_new = max(m, float(np.max(x)))
        corr = 0.0 if m == -np.inf else float(np.exp(m - m_new))
        l = l * corr + float(np.sum(np.exp(x - m_new)))
        m = m_new
        out.append((m, l))
    return out


def online_softmax_scalar(x: Sequence[float]) -> Tuple[float, float]:
    """One element at a time: d_j = d_{j-1} e^{m_{j-1}-m_j} + e^{x_j - m_j}.

    "Flash Attention v1" (languisher.top), section "Online Softmax", incremental softmax.
    """
    m, dsum = -np.inf, 0.0
    for xj in x:
        m_new = max(m, float(xj))
        corr = 0.0 if m == -np.inf else float(np.exp(m - m_new))
        dsum = dsum * corr + float(np.exp(float(xj) - m_new))
        m = m_new
    return m, dsum


def merge_stats(m1: float, l1: float, m2: float, l2: float) -> Tuple[float, float]:
    """Statistics of a concatenated vector from those of its two halves.

    FlashAttention paper-detail page, "Technique 1 (Tiling)": m = max(m1, m2),
    l = e^{m1 - m} l1 + e^{m2 - m} l2.
    """
    m = max(m1, m2)
    return m, float(np.exp(m1 - m) * l1 + np.exp(m2 - m) * l2)


def fa2_forward_steps(S: np.ndarray, V: np.ndarray, block_c: int):
    """FlashAttention-2 Algorithm 1 (forward) for one row block, keeping every step.

    S: [Br, N] scores (already scaled, -inf where masked); V: [N, d].
    Per column block j: m_new = max(m, rowmax(S_j)); P~ = exp(S_j - m_new);
    l = exp(m - m_new) l + rowsum(P~); O~ = diag(exp(m - m_new)) O~ + P~ V_j
    (multiplying, per the reading in the module docstring).  After the loop
    O = diag(l)^{-1} O~ and L = m + log(l).
    Returns a list with (m, l, O~) after every step, and the final (O, L).
    """
    Br, N = S.shape
    d = V.shape[1]
    m = np.full(Br, -np.inf)
    l = np.zeros(Br)
    Ot = np.zeros((Br, d))
    steps = []
    for c0 in range(0, N, block_c):
        Sj = S[:, c0:c0 + block_c]
        m_new = np.maximum(m, Sj.max(axis=1))
        safe = np.where(np.isfinite(m_new), m_new, 0.0)
        Pt = np.exp(Sj - safe[:, None])
        corr = np.where(np.isfinite(m), np.exp(m - safe), 0.0)
        l = corr * l + Pt.sum(axis=1)
        Ot = corr[:, None] * Ot + Pt @ V[c0:c0 + block_c]
        m = m_new
        steps.append((m.copy(), l.copy(), Ot.copy()))
    with np.errstate(divide="ignore", invalid="ignore"):
        O = np.where(l[:, None] > 0, Ot / np.where(l > 0, l, 1.0)[:, None], 0.0)
        L = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return steps, (O, L)


def fa1_forward(S: np.ndarray, V: np.ndarray, block_c: int) -> np.ndarray:
    """FlashAttention-1 per-step normalised update, FlashAttention-2 reading notes eq. (7)/(9).

    O^(j) = diag(l^(j))^{-1} [ e^{m^(j-1) - m^(j)} l^(j-1) O^(j-1) + e^{S^(j) - m^(j)} V^(j) ]
    """
    Br, N = S.shape
    d = V.shape[1]
    m = np.full(Br, -np.inf)
    l = np.zeros(Br)
    O = np.zeros((Br, d))
    for c0 in range(0, N, block_c):
        Sj = S[:, c0:c0 + block_c]
        m_new = np.maximum(m, Sj.max(axis=1))
        safe = np.where(np.isfinite(m_new), m_new, 0.0)
        Pt = np.exp(Sj - safe[:, None])
        corr = np.where(np.isfinite(m), np.exp(m - safe), 0.0)
        l_new = corr * l + Pt.sum(axis=1)
        with np.errstate(divide="ignore", invalid="ignore"):
            inv = np.where(l_new > 0, 1.0 / np.where(l_new > 0, l_new, 1.0), 0.0)
        O = inv[:, None] * ((corr * l)[:, None] * O + Pt @ V[c0:c0 + block_c])
        m, l = m_new, l_new
    return O
