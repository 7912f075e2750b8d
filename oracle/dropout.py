"""Attention with dropout on the probabilities, and the counter-based generator that draws the
dropout decisions, in plain fp64 numpy (test infrastructure, like the rest of ``oracle``).

The FlashAttention paper detail page lists dropout among the operations fused into the
attention kernel (O = dropout(softmax(S)) V), and the FlashAttention-2 reading notes keep it in
the backward; neither page fixes a random-number generator.  The reading taken here:

* Generator: Philox4x64-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as
  1, 2, 3", SC 2011): a 256-bit counter and a 128-bit key, ten rounds of two 64 x 64 -> 128-bit
  multiplications, with the key bumped by two Weyl constants between rounds.  It is pinned
  against numpy's ``np.random.Philox`` (the same generator) in the tests.
* Decisions: score (q, k) of head bh (b * H + h) takes byte (k mod 32) of the 32 output bytes
  (4 little-endian 64-bit words) of Philox4x64-10 with counter (k div 32, q, bh, 0) and key
  (seed, offset); it is dropped when that byte is below t = nearest integer to 256 p (ties to
  even), so the drop probability is t / 256, and kept probabilities are scaled by 256 / (256 - t).
* Forward: P = softmax(S) (masked as usual), P_d = P o Z * 256 / (256 - t), O = P_d V; LSE is the
  logsumexp of the scores (dropout does not change it).
* Backward: dV = P_d^T dO, dP = (dO V^T) o Z * 256 / (256 - t), D = rowsum(P o dP)
  (= rowsum(dO o O)), dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.
"""
from __future__ import annotations

import numpy as np

from . import _f64, probabilities

_M0, _M1 = np.uint64(0xD2E7470EE14C6C93), np.uint64(0xCA5A826395121157)
_W0, _W1 = np.uint64(0x9E3779B97F4A7C15), np.uint64(0xBB67AE8584CAA73B)
_LO = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)


def _mulhilo(a: np.uint64, b: np.ndarray):
    """(high, low) 64-bit halves of the 128-bit products a * b, from 32-bit partial products."""
    a_lo, a_hi = a & _LO, a >> _S32
    b_lo, b_hi = b & _LO, b >> _S32
    ll, lh, hl, hh = a_lo * b_lo, a_lo * b_hi, a_hi * b_lo, a_hi * b_hi
    mid = (ll >> _S32) + (lh & _LO) + (hl & _LO)
    lo = (ll & _LO) | ((mid & _LO) << _S32)
    hi = hh + (lh >> _S32) + (hl >> _S32) + (mid >> _S32)
    return hi, lo


def philox4x64_10(counter, key) -> np.ndarray:
    """Philox4x64-10 of counters [..., 4] (uint64) under key (k0, k1): [..., 4] uint64."""
    c = np.asarray(counter, dtype=np.uint64)
    c0, c1, c2, c3 = (c[..., i].copy() for i in range(4))
    k0, k1 = np.uint64(key[0]), np.uint64(key[1])
    with np.errstate(over="ignore"):
        for _ in range(10):
            hi0, lo0 = _mulhilo(_M0, c0)
            hi1, lo1 = _mulhilo(_M1, c2)
            c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
            k0, k1 = k0 + _W0, k1 + _W1
    return np.stack([c0, c1, c2, c3], axis=-1)


def threshold(p: float) -> int:
    """Byte threshold t of drop probability p: the nearest integer to 256 p (ties to even)."""
    t = int(np.rint(256.0 * p))
    if not 0 <= t <= 255:
        raise ValueError("dropout probability must be in [0, 255/256]")
    return t


def keep_mask(bh: int, Nq: int, Nk: int, seed: int, offset: int, t: int) -> np.ndarray:
    """keep[q, k] (bool) for every score of head bh."""
    nkb = (Nk + 31) // 32
    q, kb = np.meshgrid(np.arange(Nq, dtype=np.uint64), np.arange(nkb, dtype=np.uint64),
                        indexing="ij")
    ctr = np.stack([kb, q, np.full_like(q, bh), np.zeros_like(q)], axis=-1)
    words = philox4x64_10(ctr, (seed, offset))                   # [Nq, nkb, 4]
    b = words.astype("<u8").view(np.uint8).reshape(Nq, nkb * 32)  # byte k mod 32 of block k div 32
    return b[:, :Nk] >= t


def attention_dropout(q, k, v, scale: float, p: float, seed: int, offset: int = 0,
                      causal: bool = False, block_mask=None, block: int = 128, dout=None) -> dict:
    """Forward (and backward with ``dout``) of attention with dropout: q, k, v [B, H, N, d]."""
    qa, ka, va = _f64(q), _f64(k), _f64(v)
    B, H, N, d = qa.shape
    t = threshold(p)
    keep_scale = 256.0 / (256.0 - t)
    da = None if dout is None else _f64(dout)
    res = {x: np.zeros_like(qa) for x in ("o", "dq", "dk", "dv")}
    res["lse"] = np.zeros((B, H, N))
    res["delta"] = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            bh = b * H + h
            Q, K, V = qa[b, h], ka[b, h], va[b, h]
            P = probabilities(Q, K, scale, causal, block_mask, block)
            S = scale * (Q @ K.T)
            if causal:
                S = np.where(np.tril(np.ones((N, N), dtype=bool)), S, -np.inf)
            if block_mask is not None:
                bm = np.asarray(block_mask, dtype=bool)
                idx = np.arange(N) // block
                S = np.where(bm[idx][:, idx], S, -np.inf)
            m = S.max(axis=1)
            fin = np.isfinite(m)
            lse = np.full(N, -np.inf)
            lse[fin] = m[fin] + np.log(np.exp(S[fin] - m[fin, None]).sum(axis=1))
            Z = keep_mask(bh, N, N, seed, offset, t)
            Pd = np.where(Z, P * keep_scale, 0.0)
            O = Pd @ V
            res["o"][b, h], res["lse"][b, h] = O, lse
            if da is not None:
                dO = da[b, h]
                dP = np.where(Z, (dO @ V.T) * keep_scale, 0.0)
                D = np.sum(P * dP, axis=1)
                dS = P * (dP - D[:, None])
                res["dv"][b, h] = Pd.T @ dO
                res["dq"][b, h] = scale * (dS @ K)
                res["dk"][b, h] = scale * (dS.T @ Q)
                res["delta"][b, h] = D
    return res
