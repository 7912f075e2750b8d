"""GPU parity of grouped-query attention (fa_fwd_gqa, fa_bwd_gqa) against the fp64 oracle.

FlashAttention-2 reading notes, MQA/GQA section: query head h reads K/V head h // (H / H_kv);
dK and dV of a shared head are sums over its query heads.  Tolerances as in test_parity_gpu.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_staged_gb300.workloads import (BLOCK, WORKLOADS, make_block_mask,
                                                    make_inputs, workload_inputs)
from test_parity_gpu import DEV, check_bwd, check_fwd, expected_visits, np64, visit_log_buffer

pytestmark = pytest.mark.gpu


def run_gqa(api, t, scale, causal, mask=None):
    q, k, v, do = (t[x].to(DEV) for x in ("q", "k", "v", "do"))
    m = None if mask is None else mask.to(DEV)
    o, lse = api.fwd_gqa(q, k, v, scale, causal=causal, block_mask=m)
    grads = api.bwd_gqa(q, k, v, o, lse, do, scale, causal=causal, block_mask=m)
    assert api.sync_status() == 0
    return o, lse, grads


CASES = [  # B, H, H_kv, N, d, causal
    (2, 4, 2, 200, 64, False),
    (1, 6, 3, 513, 128, True),
    (1, 8, 1, 384, 64, True),     # MQA
    (2, 4, 1, 130, 128, False),   # MQA, ragged tail
    (1, 4, 2, 1000, 128, True),
]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal", CASES)
@pytest.mark.parametrize("splits", [0, 1, 2])
def test_gqa_small_shapes(cuda_lib, B, H, Hkv, N, d, causal, splits):
    t = make_inputs(B, H, N, d, torch.bfloat16, seed=400 + N + H, h_kv=Hkv)
    scale = 1 / math.sqrt(d)
    cuda_lib.debug_set_dkdv_splits(splits)
    try:
        o, lse, grads = run_gqa(cuda_lib, t, scale, causal)
    finally:
        cuda_lib.debug_set_dkdv_splits(0)
    ref = oracle.attention_gqa(t["q"], t["k"], t["v"], scale, causal, dout=t["do"])
    what = f"B={B} H={H} Hkv={Hkv} N={N} d={d} causal={causal} splits={splits}"
    check_fwd(o, lse, ref, what)
    check_bwd(grads, ref, what)


def test_gqa_block_sparse_with_dead_rows(cuda_lib):
    N, d = 900, 64
    T = (N + BLOCK - 1) // BLOCK
    mask = make_block_mask(T, 17, 0.4)
    mask[2, :] = 0  # query block 2 sees no key
    t = make_inputs(1, 6, N, d, torch.bfloat16, seed=417, h_kv=2)
    o, lse, grads = run_gqa(cuda_lib, t, 0.125, True, mask)
    ref = oracle.attention_gqa(t["q"], t["k"], t["v"], 0.125, True, mask, dout=t["do"])
    check_fwd(o, lse, ref, "gqa sparse")
    check_bwd(grads, ref, "gqa sparse")
    assert torch.all(o[:, :, 256:384].cpu() == 0)


def test_gqa_with_equal_heads_is_mha_bitwise(cuda_lib):
    # H_kv = H goes through the same kernels as fa_fwd / fa_bwd with identical arguments
    t = make_inputs(2, 3, 333, 128, torch.bfloat16, seed=420)
    q, k, v, do = (t[x].to(DEV) for x in ("q", "k", "v", "do"))
    a = cuda_lib.fwd_gqa(q, k, v, 0.1, causal=True)
    b = cuda_lib.fwd(q, k, v, 0.1, causal=True)
    ga = cuda_lib.bwd_gqa(q, k, v, a[0], a[1], do, 0.1, causal=True)
    gb = cuda_lib.bwd(q, k, v, b[0], b[1], do, 0.1, causal=True)
    assert cuda_lib.sync_status() == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for x, y in zip(ga, gb):
        assert torch.equal(x, y)


@pytest.mark.parametrize("splits", [1, 3])
def test_gqa_tile_visits_and_determinism(cuda_lib, splits):
    B, H, Hkv, N, d = 1, 6, 2, 700, 64
    T = (N + BLOCK - 1) // BLOCK
    t = make_inputs(B, H, N, d, torch.bfloat16, seed=430, h_kv=Hkv)
    log = visit_log_buffer(B * H * T * T)
    cuda_lib.debug_set_dkdv_splits(splits)
    cuda_lib.debug_set_visit_log(log)
    try:
        first = run_gqa(cuda_lib, t, 0.125, True)
    finally:
        cuda_lib.debug_set_visit_log(None)
    try:
        second = run_gqa(cuda_lib, t, 0.125, True)
    finally:
        cuda_lib.debug_set_dkdv_splits(0)
    got = log.cpu().numpy()[:B * H * T * T].reshape(B * H, T, T)
    assert np.array_equal(got, expected_visits(B * H, T, True, None))
    for x, y in zip(first[2], second[2]):
        assert torch.equal(x, y)


def test_gqa_workload_parity(cuda_lib):
    w = WORKLOADS["gqa_causal_d128_n8k"]
    t = workload_inputs(w)
    o, lse, grads = run_gqa(cuda_lib, t, w.scale, w.causal)
    rep = w.H // w.kv_heads
    for g in sorted({0, w.kv_heads - 1}):  # first and last K/V group, all their query heads
        hs = slice(g * rep, (g + 1) * rep)
        ref = oracle.attention_gqa(t["q"][:, hs], t["k"][:, g:g + 1], t["v"][:, g:g + 1],
                                   w.scale, w.causal, dout=t["do"][:, hs])
        check_fwd(o[:, hs], lse[:, hs], ref, f"group {g}")
        check_bwd([grads[0][:, hs], grads[1][:, g:g + 1], grads[2][:, g:g + 1]], ref,
                  f"group {g}")
    assert torch.isfinite(o).all()
    for x in grads:
        assert torch.isfinite(x).all()


def test_gqa_split_groups_with_partial_last_head_group(cuda_lib):
    # dK/dV with each K/V head's query group split over 2 CTAs per key tile: its CTA order then
    # has B * H_kv * 2 = 24 work-unit heads, taken in groups of 16 at N = 4096, d = 128 (the
    # streamed Q and dO tiles of a group stay near 32 MiB of L2), so the last group is partial
    from test_parity_gpu import heads_per_group
    B, H, Hkv, N, d = 2, 12, 6, 4096, 128
    units = B * Hkv * 2
    grp = heads_per_group(units, N, d, 2.0)
    assert units > grp and units % grp != 0
    t = make_inputs(B, H, N, d, torch.bfloat16, seed=440, h_kv=Hkv)
    scale = 1 / math.sqrt(d)
    cuda_lib.debug_set_dkdv_splits(2)
    try:
        o, lse, grads = run_gqa(cuda_lib, t, scale, True)
    finally:
        cuda_lib.debug_set_dkdv_splits(0)
    ref = oracle.attention_gqa(t["q"], t["k"], t["v"], scale, True, dout=t["do"])
    check_fwd(o, lse, ref, "gqa split, partial group")
    check_bwd(grads, ref, "gqa split, partial group")
