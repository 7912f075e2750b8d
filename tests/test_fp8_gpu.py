"""GPU parity of the e4m3 forward (fa_fwd_fp8) with the fp64 oracle on the decoded inputs.

Tolerance, derived from the arithmetic.  The kernel rounds each probability P~ to e4m3 (3
mantissa bits, round to nearest, unit roundoff u = 2^-4) before the PV product; everything
else matches the bf16 path (scores are sums of exactly representable e4m3 products in fp32,
the softmax statistics are fp32, O is rounded once to bf16).  With P^_j = P~_j (1 + e_j):

  elementwise   |dO| = |sum_j P_j e_j V_j| <= u max|V| (the weights P_j sum to 1), plus the
                bf16 rounding of O, 2^-9 |O| <= 2^-9 max|V|:  bound (2^-4 + 2^-9) max|V|;
  Frobenius     with the rounding position uniform within each spacing interval (the
                standard model of round to nearest), E[e_j^2] <= u^2 / 3 whatever P~ is, and
                for V with independent zero-mean entries E|dO|^2 = sum_j P_j^2 E[e_j^2] E[V^2]
                while E|O|^2 = sum_j P_j^2 E[V^2]: the relative Frobenius error of O is at most
                u / sqrt(3) = 0.0361 (the bf16 rounding of O adds 2^-9 / sqrt(3) in
                quadrature, below 1 % of it).  With mantissas spread evenly in log scale the
                same model predicts 0.0265.
LSE is computed from the fp32 probabilities and keeps the forward's 1e-3.  Each test records
the measured errors (junit properties fp8_relF, fp8_maxabs_over_vmax).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_staged_gb300.workloads import (BLOCK, FP8_WORKLOADS, fp8_workload_inputs,
                                                    make_block_mask, make_fp8_inputs)
from test_parity_gpu import DEV, expected_visits, np64, relf, visit_log_buffer

pytestmark = pytest.mark.gpu

U = 2.0 ** -4                      # e4m3 unit roundoff (round to nearest, 3 mantissa bits)
REL_BOUND = U / math.sqrt(3.0)     # relative Frobenius error of O (module docstring)
ABS_FACTOR = U + 2.0 ** -9         # elementwise error of O, in units of max |V|


def check_fp8(o, lse, ref, vmax, what, record=None):
    o, lse = np64(o), np64(lse)
    fin = np.isfinite(ref["lse"])
    assert np.array_equal(np.isneginf(lse), ~fin), f"{what}: -inf LSE rows differ"
    err = float(np.max(np.abs(o - ref["o"])))
    rel = relf(o, ref["o"])
    lerr = float(np.max(np.abs(lse[fin] - ref["lse"][fin]))) if fin.any() else 0.0
    if record is not None:
        record("fp8_relF", rel)
        record("fp8_maxabs_over_vmax", err / vmax if vmax > 0 else 0.0)
        record("fp8_lse_maxabs", lerr)
    assert rel <= REL_BOUND and err <= ABS_FACTOR * vmax, \
        f"{what}: O relF {rel:.3e} maxabs {err:.3e} (max|V| {vmax:.3e})"
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
def test_fp8_small_shapes(cuda_lib, record_property, B, H, Hkv, N, d, causal):
    t = make_fp8_inputs(B, H, N, d, seed=600 + N + d, h_kv=Hkv)
    scale = 1 / math.sqrt(d)
    o, lse = run_fp8(cuda_lib, t, scale, causal)
    ref = oracle.attention_fp8(t["q"], t["k"], t["v"], scale, t["descale_q"], t["descale_k"],
                               t["descale_v"], causal)
    vmax = float(np.max(np.abs(oracle.e4m3_to_f64(t["v"])))) * t["descale_v"]
    check_fp8(o, lse, ref, vmax, f"B={B} H={H} Hkv={Hkv} N={N} d={d} causal={causal}",
              record_property)


def test_fp8_block_sparse_visits_and_dead_rows(cuda_lib, record_property):
    N, d = 900, 128
    T = (N + BLOCK - 1) // BLOCK
    mask = make_block_mask(T, 23, 0.4)
    mask[3, :] = 0
    t = make_fp8_inputs(1, 2, N, d, seed=640, qk_mult=2.0)
    log = visit_log_buffer(2 * T * T)
    cuda_lib.debug_set_visit_log(log)
    try:
        o, lse = run_fp8(cuda_lib, t, 0.1, True, mask)
    finally:
        cuda_lib.debug_set_visit_log(None)
    ref = oracle.attention_fp8(t["q"], t["k"], t["v"], 0.1, t["descale_q"], t["descale_k"],
                               t["descale_v"], True, mask)
    vmax = float(np.max(np.abs(oracle.e4m3_to_f64(t["v"])))) * t["descale_v"]
    check_fp8(o, lse, ref, vmax, "fp8 sparse", record_property)
    assert torch.all(o[:, :, 384:512].cpu() == 0)
    got = log.cpu().numpy()[:2 * T * T].reshape(2, T, T)
    assert np.array_equal(got, expected_visits(2, T, True, mask) & 1)


def test_fp8_is_deterministic(cuda_lib):
    t = make_fp8_inputs(1, 4, 700, 128, seed=650, h_kv=2)
    a = run_fp8(cuda_lib, t, 0.09, True)
    b = run_fp8(cuda_lib, t, 0.09, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fp8_workload_parity(cuda_lib, record_property):
    w = FP8_WORKLOADS["fp8_causal_d128_n8k"]
    t = fp8_workload_inputs(w)
    o, lse = run_fp8(cuda_lib, t, w.scale, w.causal)
    vmax = float(np.max(np.abs(oracle.e4m3_to_f64(t["v"])))) * t["descale_v"]
    for h in sorted({0, w.H - 1}):
        ref = oracle.attention_fp8(t["q"][:, h:h + 1], t["k"][:, h:h + 1], t["v"][:, h:h + 1],
                                   w.scale, t["descale_q"], t["descale_k"], t["descale_v"],
                                   w.causal)
        check_fp8(o[:, h:h + 1], lse[:, h:h + 1], ref, vmax, f"{w.name} head {h}",
                  record_property)
    assert torch.isfinite(o).all()
