"""GPU parity of the e4m3 forward (fa_fwd_fp8) with the fp64 oracle on the decoded inputs.

Tolerance, derived from the arithmetic: the kernel rounds each probability P~ to e4m3 before
the PV product, a relative error of at most 2^-4 (3 mantissa bits, round to nearest) per
probability, independent from one probability to the next.  O is a P-weighted mean of V rows,
so its error is bounded elementwise by 2^-4 * max |V| and, over a tensor, its relative
Frobenius error by 2^-4 (the RMS estimate is 2^-4 / sqrt(3) = 0.036).  LSE is computed from the
fp32 probabilities and keeps the forward's 1e-3.  Scores accumulate exactly-representable e4m3
products in fp32, as in the bf16 path.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_staged_gb300.workloads import (BLOCK, FP8_WORKLOADS, fp8_workload_inputs,
                                                    make_block_mask, make_fp8_inputs)
from test_parity_gpu import DEV, expected_visits, np64, relf

pytestmark = pytest.mark.gpu

U = 2.0 ** -4  # e4m3 unit roundoff (relative spacing / 2 is 2^-4 for round to nearest)


def check_fp8(o, lse, ref, vmax, what):
    o, lse = np64(o), np64(lse)
    fin = np.isfinite(ref["lse"])
    assert np.array_equal(np.isneginf(lse), ~fin), f"{what}: -inf LSE rows differ"
    err = float(np.max(np.abs(o - ref["o"])))
    rel = relf(o, ref["o"])
    lerr = float(np.max(np.abs(lse[fin] - ref["lse"][fin]))) if fin.any() else 0.0
    assert rel <= U and err <= U * vmax, f"{what}: O relF {rel:.3e} maxabs {err:.3e}"
    assert lerr <= 1e-3, f"{what}: LSE maxabs {lerr:.3e}"
    return rel, err


def run_fp8(api, t, scale, causal, mask=None):
    q, k, v = (t[x].to(DEV) for x in ("q", "k", "v"))
    m = None if mask is None else mask.to(DEV)
    o, lse = api.fwd_fp8(q, k, v, t["descale_q"], t["descale_k"], t["descale_v"], scale,
                         causal=causal, block_mask=m)
    assert api.sync_status() == 0
    return o, lse


CASES = [  # B, H, H_kv, N, d, causal
    (1, 2, 2, 128, 128, False),
    (1, 2, 2, 200, 64, True),
    (2, 4, 2, 513, 128, True),
    (1, 3, 1, 1000, 64, False),
    (1, 2, 2, 1, 128, False),
    (1, 2, 2, 17, 64, True),
]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal", CASES)
def test_fp8_small_shapes(cuda_lib, B, H, Hkv, N, d, causal):
    t = make_fp8_inputs(B, H, N, d, seed=600 + N + d, h_kv=Hkv)
    scale = 1 / math.sqrt(d)
    o, lse = run_fp8(cuda_lib, t, scale, causal)
    ref = oracle.attention_fp8(t["q"], t["k"], t["v"], scale, t["descale_q"], t["descale_k"],
                               t["descale_v"], causal)
    vmax = float(np.max(np.abs(oracle.e4m3_to_f64(t["v"])))) * t["descale_v"]
    check_fp8(o, lse, ref, vmax, f"B={B} H={H} Hkv={Hkv} N={N} d={d} causal={causal}")


def test_fp8_block_sparse_visits_and_dead_rows(cuda_lib):
    N, d = 900, 128
    T = (N + BLOCK - 1) // BLOCK
    mask = make_block_mask(T, 23, 0.4)
    mask[3, :] = 0
    t = make_fp8_inputs(1, 2, N, d, seed=640, qk_mult=2.0)
    log = torch.zeros(2 * T * T, dtype=torch.uint8, device=DEV)
    cuda_lib.debug_set_visit_log(log)
    try:
        o, lse = run_fp8(cuda_lib, t, 0.1, True, mask)
    finally:
        cuda_lib.debug_set_visit_log(None)
    ref = oracle.attention_fp8(t["q"], t["k"], t["v"], 0.1, t["descale_q"], t["descale_k"],
                               t["descale_v"], True, mask)
    vmax = float(np.max(np.abs(oracle.e4m3_to_f64(t["v"])))) * t["descale_v"]
    check_fp8(o, lse, ref, vmax, "fp8 sparse")
    assert torch.all(o[:, :, 384:512].cpu() == 0)
    got = log.cpu().numpy().reshape(2, T, T)
    assert np.array_equal(got, expected_visits(2, T, True, mask) & 1)


def test_fp8_is_deterministic(cuda_lib):
    t = make_fp8_inputs(1, 4, 700, 128, seed=650, h_kv=2)
    a = run_fp8(cuda_lib, t, 0.09, True)
    b = run_fp8(cuda_lib, t, 0.09, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fp8_workload_parity(cuda_lib):
    w = FP8_WORKLOADS["fp8_causal_d128_n8k"]
    t = fp8_workload_inputs(w)
    o, lse = run_fp8(cuda_lib, t, w.scale, w.causal)
    vmax = float(np.max(np.abs(oracle.e4m3_to_f64(t["v"])))) * t["descale_v"]
    for h in sorted({0, w.H - 1}):
        ref = oracle.attention_fp8(t["q"][:, h:h + 1], t["k"][:, h:h + 1], t["v"][:, h:h + 1],
                                   w.scale, t["descale_q"], t["descale_k"], t["descale_v"],
                                   w.causal)
        check_fp8(o[:, h:h + 1], lse[:, h:h + 1], ref, vmax, f"{w.name} head {h}")
    assert torch.isfinite(o).all()
