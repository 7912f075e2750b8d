"""GPU parity of attention with dropout (fa_fwd_dropout, fa_bwd_dropout) against the fp64
oracle (``oracle.dropout``), which draws the same Philox4x32-10 decisions independently.

Tolerances as in test_parity_gpu: dropout only zeroes probabilities and scales the rest by
256 / (256 - t), so the rounding behaviour of O and the gradients is that of the plain path,
on values that factor larger: the relative bars are unchanged and O's max-abs bar is scaled by
256 / (256 - t) (at p = 0.9 O is about ten times the plain output, and so is its rounding).
"""
import math

import numpy as np
import pytest
import torch

from oracle import dropout as odrop
from exact_attention_staged_gb300.workloads import (BLOCK, WORKLOADS, make_block_mask,
                                                    make_inputs, workload_inputs)
from test_parity_gpu import DEV, check_bwd, check_fwd, np64

pytestmark = pytest.mark.gpu


def run_drop(api, t, scale, causal, p, seed, offset, mask=None):
    q, k, v, do = (t[x].to(DEV) for x in ("q", "k", "v", "do"))
    m = None if mask is None else mask.to(DEV)
    o, lse = api.fwd_dropout(q, k, v, p, seed, offset, scale, causal, m)
    grads = api.bwd_dropout(q, k, v, o, lse, do, p, seed, offset, scale, causal, m)
    assert api.sync_status() == 0
    return o, lse, grads


CASES = [  # B, H, N, d, causal, p
    (1, 2, 128, 64, False, 0.1),
    (1, 2, 200, 128, True, 0.25),
    (2, 2, 513, 64, True, 0.5),
    (1, 3, 384, 128, False, 0.1),
    (1, 1, 17, 64, True, 0.3),
    # thresholds above 128 (256 - t below 128: the other branch of the kernels' byte compare),
    # the largest one, and the smallest nonzero one
    (1, 2, 256, 64, False, 0.75),
    (1, 1, 200, 128, True, 0.9),
    (1, 2, 130, 128, False, 0.99),
    (1, 2, 130, 64, True, 1 / 256),
]


def keep_scale(p):
    return 256.0 / (256.0 - odrop.threshold(p))


@pytest.mark.parametrize("B,H,N,d,causal,p", CASES)
def test_dropout_small(cuda_lib, B, H, N, d, causal, p):
    t = make_inputs(B, H, N, d, torch.bfloat16, seed=700 + N + d)
    scale = 1 / math.sqrt(d)
    o, lse, grads = run_drop(cuda_lib, t, scale, causal, p, seed=1234 + N, offset=7)
    ref = odrop.attention_dropout(t["q"], t["k"], t["v"], scale, p, 1234 + N, 7, causal,
                                  dout=t["do"])
    what = f"B={B} H={H} N={N} d={d} causal={causal} p={p}"
    check_fwd(o, lse, ref, what, o_scale=keep_scale(p))
    check_bwd(grads, ref, what)


def test_dropout_block_sparse_and_seed_dependence(cuda_lib):
    N, d = 700, 128
    T = (N + BLOCK - 1) // BLOCK
    mask = make_block_mask(T, 31, 0.5)
    t = make_inputs(1, 2, N, d, torch.bfloat16, seed=760)
    o, lse, grads = run_drop(cuda_lib, t, 0.1, True, 0.2, 99, 3, mask)
    ref = odrop.attention_dropout(t["q"], t["k"], t["v"], 0.1, 0.2, 99, 3, True, mask,
                                  dout=t["do"])
    check_fwd(o, lse, ref, "dropout sparse")
    check_bwd(grads, ref, "dropout sparse")
    # same arguments: same result; another offset: other decisions, same LSE
    o2, lse2, g2 = run_drop(cuda_lib, t, 0.1, True, 0.2, 99, 3, mask)
    assert torch.equal(o, o2) and all(torch.equal(a, b) for a, b in zip(grads, g2))
    o3, lse3, _ = run_drop(cuda_lib, t, 0.1, True, 0.2, 99, 4, mask)
    assert not torch.equal(o, o3) and torch.equal(lse, lse3)
    # a seed above 2^32 fills both key words of the generator; the largest 32-bit offset
    seed, off = 0xDEADBEEF12345678, 2 ** 32 - 1
    o4, lse4, g4 = run_drop(cuda_lib, t, 0.1, True, 0.2, seed, off, mask)
    ref4 = odrop.attention_dropout(t["q"], t["k"], t["v"], 0.1, 0.2, seed, off, True, mask,
                                   dout=t["do"])
    check_fwd(o4, lse4, ref4, "dropout 64-bit seed")
    check_bwd(g4, ref4, "dropout 64-bit seed")


def test_dropout_zero_probability_is_the_plain_path(cuda_lib):
    t = make_inputs(1, 2, 300, 64, torch.bfloat16, seed=770)
    q, k, v, do = (t[x].to(DEV) for x in ("q", "k", "v", "do"))
    a = cuda_lib.fwd_dropout(q, k, v, 0.0, 5, 0, 0.125, True)
    b = cuda_lib.fwd(q, k, v, 0.125, causal=True)
    ga = cuda_lib.bwd_dropout(q, k, v, a[0], a[1], do, 0.0, 5, 0, 0.125, True)
    gb = cuda_lib.bwd(q, k, v, b[0], b[1], do, 0.125, causal=True)
    assert cuda_lib.sync_status() == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for x, y in zip(ga, gb):
        assert torch.equal(x, y)


def test_dropout_with_grouped_kv_heads(cuda_lib):
    # the grouped-query path with dropout: decisions are per query head
    t = make_inputs(1, 4, 260, 64, torch.bfloat16, seed=780, h_kv=2)
    o, lse, grads = run_drop(cuda_lib, t, 0.125, True, 0.15, 5, 1)
    ref = odrop.attention_dropout(t["q"], t["k"].repeat_interleave(2, 1),
                                  t["v"].repeat_interleave(2, 1), 0.125, 0.15, 5, 1, True,
                                  dout=t["do"])
    ref["dk"] = ref["dk"].reshape(1, 2, 2, 260, 64).sum(axis=2)
    ref["dv"] = ref["dv"].reshape(1, 2, 2, 260, 64).sum(axis=2)
    check_fwd(o, lse, ref, "dropout gqa")
    check_bwd(grads, ref, "dropout gqa")


def test_dropout_workload_sampled_rows(cuda_lib):
    # the 8k workload: whole-head oracle checks are too large for numpy's generator, so the
    # first and last 256 query rows of two heads are checked; those rows only need keys below
    # them (first rows) or the full key range (last rows)
    w = WORKLOADS["dropout_causal_d128_n8k"]
    t = workload_inputs(w)
    o, lse, grads = run_drop(cuda_lib, t, w.scale, w.causal, w.dropout, w.seed, 0)
    assert torch.isfinite(o).all() and all(torch.isfinite(g).all() for g in grads)
    n0 = 256
    sub = {x: t[x][:, :1, :n0] for x in ("q", "k", "v", "do")}
    ref = odrop.attention_dropout(sub["q"], sub["k"], sub["v"], w.scale, w.dropout, w.seed, 0,
                                  True, dout=sub["do"])
    check_fwd(o[:, :1, :n0], lse[:, :1, :n0], ref, "first rows of head 0")
