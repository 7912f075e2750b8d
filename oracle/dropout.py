"""Attention with dropout on the probabilities, and the counter-based generator that draws the
dropout decisions, in plain fp64 numpy (test infrastructure, like the rest of ``oracle``).

The FlashAttention paper detail page lists dropout among the operations fused into the
attention kernel (O = dropout(softmax(S)) V), and the FlashAttention-2 reading notes keep it in
the backward; neither page fixes a random-number generator.  The reading taken here:

* Generator: Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as
  1, 2, 3", SC 2011): a 128-bit counter of four 32-bit words and a 64-bit key, ten rounds of two
  32 x 32 -> 64-bit multiplications whose halves are swapped and xored into the other words,
  with the key bumped by two Weyl constants between rounds.  It is pinned in the tests against
  cuRAND's host Philox4_32_10 generator (an independent implementation of the same generator).
* Decisions: score (q, k) of head bh (b * H + h) takes byte (k mod 16) of the 16 output bytes
  (4 little-endian 32-bit words) of Philox4x32-10 with counter (k div 16, q, bh, offset) and key
  (seed mod 2^32, seed div 2^32); it is dropped when that byte is below t = nearest integer to
  256 p (ties to even), so the drop probability is t / 256, and kept probabilities are scaled by
  256 / (256 - t).  The offset is below 2^32.
* Forward: P = softmax(S) (masked as usual), P_d = P o Z * 256 / (256 - t), O = P_d V; LSE is the
  logsumexp of the scores (dropout does not change it).
* Backward: dV = P_d^T dO, dP = (dO V^T) o Z * 256 / (256 - t), D = rowsum(P o dP)
  (= rowsum(dO o O)), dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.
"""
from __future__ import annotations

import numpy as np

from . import _f64, probabilities

_M0, _M1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)  # round multipliers
_W0, _W1 = np.uint64(0x9E3779B9), np.uint64(0xBB67AE85)  # key increments (Weyl constants)
_LO = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)


def philox4x32_10(counter, key) -> np.ndarray:
    """Philox4x32-10 of counters [..., 4] (32-bit words) under key (k0, k1): [..., 4] uint32.

    Each round multiplies counter words 0 and 2 by the two multipliers (a 32 x 32 -> 64-bit
    product, exact in uint64); the new words are (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2),
    hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); then the key words advance by the Weyl constants (mod 2^32).
    """
    c = np.asarray(counter, dtype=np.uint64) & _LO
    c0, c1, c2, c3 = (c[..., i].copy() for i in range(4))
    k0, k1 = np.uint64(int(key[0]) & 0xFFFFFFFF), np.uint64(int(key[1]) & 0xFFFFFFFF)
    for _ in range(10):
        p0, p1 = _M0 * c0, _M1 * c2
        c0, c1, c2, c3 = (p1 >> _S32) ^ c1 ^ k0, p1 & _LO, (p0 >> _S32) ^ c3 ^ k1, p0 & _LO
        k0, k1 = (k0 + _W0) & _LO, (k1 + _W1) & _LO
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def threshold(p: float) -> int:
    """Byte threshold t of drop probability p: the nearest integer to 256 p (ties to even)."""
    t = int(np.rint(256.0 * p))
    if not 0 <= t <= 255:
        raise ValueError("dropout probability must be in [0, 255/256]")
    return t


def keep_mask(bh: int, Nq: int, Nk: int, seed: int, offset: int, t: int) -> np.ndarray:
    """keep[q, k] (bool) for every score of head bh."""
    if not 0 <= offset < 2 ** 32:
        raise ValueError("the dropout offset is a 32-bit counter word")
    nkb = (Nk + 15) // 16
    q, kb = np.meshgrid(np.arange(Nq, dtype=np.uint64), np.arange(nkb, dtype=np.uint64),
                        indexing="ij")
    ctr = np.stack([kb, q, np.full_like(q, bh), np.full_like(q, offset)], axis=-1)
    words = philox4x32_10(ctr, (seed & 0xFFFFFFFF, seed >> 32))   # [Nq, nkb, 4]
    b = words.astype("<u4").view(np.uint8).reshape(Nq, nkb * 16)  # byte k mod 16 of block k div 16
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
