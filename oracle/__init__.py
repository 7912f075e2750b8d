"""fp64 CPU oracle for exact attention.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares nothing with the CUDA library; the two meet
only through the seeded inputs of ``exact_attention_staged_gb300.workloads``.

``attn_oracle.c`` holds the definition (see its header for the citations); ``recurrence.py``
holds the tiled online-softmax recurrences the pages derive, used to pin the definition.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py`` (worked example,
closed forms, invariants, finite differences, library special cases).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_lp = ctypes.POINTER(ctypes.c_long)


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (plain -O2, IEEE arithmetic, OpenMP)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC,
                               "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            lib.oracle_attention.argtypes = [ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                             ctypes.c_long, _dp, _dp, _dp, _dp, ctypes.c_double,
                                             ctypes.c_int, _u8p, ctypes.c_int, _dp, _dp, _dp, _dp,
                                             _dp, _dp]
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_forward_rows.argtypes = [ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                                _dp, _dp, _dp,
                                                ctypes.c_double, ctypes.c_int, _u8p, ctypes.c_int,
                                                ctypes.c_long, _lp, _dp, _dp]
            lib.oracle_forward_rows.restype = ctypes.c_int
            for name in ("oracle_scores", "oracle_probabilities"):
                fn = getattr(lib, name)
                fn.argtypes = [ctypes.c_long, ctypes.c_long, ctypes.c_long, _dp, _dp,
                               ctypes.c_double,
                               ctypes.c_int, _u8p, ctypes.c_int, _dp]
                fn.restype = ctypes.c_int
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact upcast of fp16/bf16/fp32 values (numpy arrays or CPU torch tensors) to fp64."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _mask_arg(block_mask, N: int, block: int):
    """N is max(Nq, Nk): the mask is square with ceil(N / block) tiles per side."""
    if block_mask is None:
        return None, None
    m = block_mask
    if hasattr(m, "detach"):
        m = m.detach().cpu().numpy()
    m = np.ascontiguousarray(np.asarray(m, dtype=np.uint8))
    tiles = (N + block - 1) // block
    if m.shape != (tiles, tiles):
        raise ValueError(f"block mask must be [{tiles},{tiles}], got {m.shape}")
    return m, m.ctypes.data_as(_u8p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def attention(q, k, v, scale: float, causal: bool = False, block_mask=None, block: int = 128,
              dout=None) -> dict:
    """Forward (and backward when ``dout`` is given): q [..., Nq, d], k and v [..., Nk, d].

    Returns fp64 arrays: o, lse and, with ``dout``, dq, dk, dv and delta (D_i = <P_i, dP_i>).
    """
    qa, ka, va = _f64(q), _f64(k), _f64(v)
    if qa.ndim < 2 or ka.shape != va.shape or qa.shape[:-2] != ka.shape[:-2] \
            or qa.shape[-1] != ka.shape[-1]:
        raise ValueError("q must be [..., Nq, d] and k, v [..., Nk, d]")
    *lead, Nq, d = qa.shape
    Nk = ka.shape[-2]
    BH = int(np.prod(lead)) if lead else 1
    mk, mptr = _mask_arg(block_mask, max(Nq, Nk), block)
    o = np.empty_like(qa)
    lse = np.empty(tuple(lead) + (Nq,), dtype=np.float64)
    res = {"o": o, "lse": lse}
    null = ctypes.cast(None, _dp)
    if dout is not None:
        da = _f64(dout)
        if da.shape != qa.shape:
            raise ValueError("dout must match q")
        dq, dk, dv = np.empty_like(qa), np.empty_like(ka), np.empty_like(ka)
        delta = np.empty_like(lse)
        rc = _load().oracle_attention(BH, Nq, Nk, d, _ptr(qa), _ptr(ka), _ptr(va), _ptr(da),
                                      float(scale), int(bool(causal)), mptr, block, _ptr(o),
                                      _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(delta))
        res.update(dq=dq, dk=dk, dv=dv, delta=delta)
    else:
        rc = _load().oracle_attention(BH, Nq, Nk, d, _ptr(qa), _ptr(ka), _ptr(va), null,
                                      float(scale),
                                      int(bool(causal)), mptr, block, _ptr(o), _ptr(lse), null,
                                      null, null, null)
    if rc != 0:
        raise RuntimeError(f"oracle_attention failed ({rc})")
    del mk
    return res


def forward_rows(q, k, v, scale: float, rows, causal: bool = False, block_mask=None,
                 block: int = 128):
    """O and LSE for the given query rows of ONE head (q: [Nq, d]; k, v: [Nk, d])."""
    qa, ka, va = _f64(q), _f64(k), _f64(v)
    Nq, d = qa.shape
    Nk = ka.shape[0]
    mk, mptr = _mask_arg(block_mask, max(Nq, Nk), block)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    o = np.empty((len(r), d), dtype=np.float64)
    lse = np.empty((len(r),), dtype=np.float64)
    rc = _load().oracle_forward_rows(Nq, Nk, d, _ptr(qa), _ptr(ka), _ptr(va), float(scale),
                                     int(bool(causal)), mptr, block, len(r),
                                     r.ctypes.data_as(_lp), _ptr(o), _ptr(lse))
    if rc != 0:
        raise RuntimeError(f"oracle_forward_rows failed ({rc})")
    del mk
    return o, lse


def _square(name, q, k, scale, causal, block_mask, block):
    qa, ka = _f64(q), _f64(k)
    Nq, d = qa.shape
    Nk = ka.shape[0]
    mk, mptr = _mask_arg(block_mask, max(Nq, Nk), block)
    out = np.empty((Nq, Nk), dtype=np.float64)
    rc = getattr(_load(), name)(Nq, Nk, d, _ptr(qa), _ptr(ka), float(scale), int(bool(causal)), mptr,
                                block, _ptr(out))
    if rc != 0:
        raise RuntimeError(f"{name} failed ({rc})")
    del mk
    return out


def scores(q, k, scale: float, causal: bool = False, block_mask=None, block: int = 128):
    """S = scale * Q K^T of ONE head with -inf at masked entries."""
    return _square("oracle_scores", q, k, scale, causal, block_mask, block)


def probabilities(q, k, scale: float, causal: bool = False, block_mask=None, block: int = 128):
    """P = softmax(S) of ONE head (three-pass safe softmax)."""
    return _square("oracle_probabilities", q, k, scale, causal, block_mask, block)


def attention_gqa(q, k, v, scale: float, causal: bool = False, block_mask=None, block: int = 128,
                  dout=None) -> dict:
    """Grouped-query attention: q [B, H, N, d]; k, v [B, H_kv, N, d] with H_kv dividing H.

    FlashAttention-2 reading notes, section on MQA/GQA support: query head h reads the K/V head
    of its group, and because a K/V head is shared by the query heads of its group, its
    gradients dK, dV are the sums of theirs.  Group g holds the H / H_kv consecutive query heads
    h with h // (H / H_kv) == g (H_kv = 1 is MQA, H_kv = H is MHA).  Written as the plain
    definition: K and V are indexed per query head and the MHA oracle runs on that, then the
    per-query-head dK and dV are summed over each group.
    """
    qa, ka, va = _f64(q), _f64(k), _f64(v)
    if qa.ndim != 4 or ka.ndim != 4 or ka.shape != va.shape or qa.shape[0] != ka.shape[0] \
            or qa.shape[3] != ka.shape[3]:
        raise ValueError("q must be [B, H, N, d] and k, v [B, H_kv, N, d]")
    B, H, Nq, d = qa.shape
    Hkv, Nk = ka.shape[1], ka.shape[2]
    if Hkv < 1 or H % Hkv != 0:
        raise ValueError("H_kv must divide H")
    rep = H // Hkv
    kv_head = np.arange(H) // rep
    res = attention(qa, np.ascontiguousarray(ka[:, kv_head]), np.ascontiguousarray(va[:, kv_head]),
                    scale, causal, block_mask, block, dout)
    if dout is not None:
        res["dk"] = res["dk"].reshape(B, Hkv, rep, Nk, d).sum(axis=2)
        res["dv"] = res["dv"].reshape(B, Hkv, rep, Nk, d).sum(axis=2)
    return res


def decode(q, k, v, scale: float, causal: bool = False, kv_len=None) -> dict:
    """Attention of a few new query rows against a KV cache, in plain fp64 numpy.

    FlashAttention-2 reading notes, section on the KV cache: in the decode phase each step's
    query is 1 x d (or a few rows) and attends to the N cached keys.  q [B, H, Nq, d];
    k, v [B, H_kv, Nk, d] with H_kv dividing H (query head h reads K/V head h // (H / H_kv), as
    in ``attention_gqa``); batch b uses its first ``kv_len[b]`` cached keys (all Nk when None).
    With ``causal`` the Nq new rows are the last positions of the sequence: row r is position
    kv_len - Nq + r and sees keys j <= that position (rows and keys aligned at the end).
    Per row this is the definition itself: s = scale * K q, P = exp(s - max s) / sum,
    O = P V, LSE = max s + ln sum exp(s - max s); a row that sees no key gets O = 0 and
    LSE = -inf.
    """
    qa, ka, va = _f64(q), _f64(k), _f64(v)
    B, H, Nq, d = qa.shape
    Hkv, Nk = ka.shape[1], ka.shape[2]
    if ka.shape != va.shape or ka.shape[0] != B or ka.shape[3] != d or H % Hkv != 0:
        raise ValueError("q [B, H, Nq, d], k and v [B, H_kv, Nk, d] with H_kv dividing H")
    lens = np.full(B, Nk, dtype=np.int64) if kv_len is None else \
        np.asarray(kv_len.detach().cpu().numpy() if hasattr(kv_len, "detach") else kv_len,
                   dtype=np.int64)
    rep = H // Hkv
    o = np.zeros_like(qa)
    lse = np.full((B, H, Nq), -np.inf)
    for b in range(B):
        L = int(min(max(lens[b], 0), Nk))
        for h in range(H):
            K, V = ka[b, h // rep, :L], va[b, h // rep, :L]
            for r in range(Nq):
                last = L - Nq + r if causal else L - 1  # last key this row sees
                if last < 0:
                    continue
                s = scale * (K[:last + 1] @ qa[b, h, r])
                m = s.max()
                p = np.exp(s - m)
                o[b, h, r] = (p @ V[:last + 1]) / p.sum()
                lse[b, h, r] = m + np.log(p.sum())
    return {"o": o, "lse": lse}


def e4m3_to_f64(codes) -> np.ndarray:
    """Values of e4m3 bytes (OCP 8-bit floating point, E4M3: 1 sign bit, 4 exponent bits with
    bias 7, 3 mantissa bits; exponent 0 is subnormal, 2^-6 * m / 8; exponent 15 with mantissa 7
    is NaN; no infinities; largest finite 448)."""
    c = np.asarray(codes.detach().cpu().numpy() if hasattr(codes, "detach") else codes,
                   dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def attention_fp8(q, k, v, scale: float, descale_q: float, descale_k: float,
                  descale_v: float, causal: bool = False, block_mask=None,
                  block: int = 128) -> dict:
    """Forward of attention on e4m3 inputs: q [B, H, N, d], k, v [B, H_kv, N, d] as e4m3
    codes, each tensor standing for code value * its descale.  The attention itself is the
    plain definition (``attention_gqa``) on those values in fp64; the e4m3 format only decides
    which values the inputs are."""
    qa = e4m3_to_f64(q) * descale_q
    ka = e4m3_to_f64(k) * descale_k
    va = e4m3_to_f64(v) * descale_v
    return attention_gqa(qa, ka, va, scale, causal, block_mask, block)
