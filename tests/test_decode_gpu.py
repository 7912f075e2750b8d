"""GPU parity of decode against a KV cache (fa_decode) with the fp64 oracle's ``decode``.

FlashAttention-2 reading notes, KV-cache section: a few new query rows per sequence against the
cache.  O and LSE tolerances as for the forward (test_parity_gpu).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_staged_gb300.workloads import (DECODE_WORKLOADS, decode_inputs,
                                                    make_decode_inputs)
from test_parity_gpu import DEV, check_fwd

pytestmark = pytest.mark.gpu


def run_decode(api, t, scale, causal, kv_len=None):
    q, k, v = (t[x].to(DEV) for x in ("q", "k", "v"))
    lens = None if kv_len is None else kv_len.to(DEV)
    o, lse = api.decode(q, k, v, scale, causal=causal, kv_len=lens)
    assert api.sync_status() == 0
    return o, lse


CASES = [  # B, H, H_kv, Nq, Nk, d, causal, ragged
    (2, 4, 4, 1, 300, 64, False, False),    # MHA, two key ranges
    (2, 4, 4, 1, 200, 128, False, False),   # one key range: written directly
    (3, 8, 2, 1, 1000, 128, False, True),   # GQA, ragged cache lengths
    (2, 4, 1, 4, 777, 128, True, True),     # MQA, 4 new rows, end-aligned causal: 16 rows
    (1, 32, 1, 1, 5000, 64, False, False),  # 32 rows per K/V head: two row groups
    (2, 6, 3, 3, 4096, 64, True, False),
    (2, 4, 2, 1, 513, 128, False, False),   # 2 rows per K/V head
    (1, 8, 1, 1, 1500, 128, True, True),    # 8 rows per K/V head at d = 128
]


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,d,causal,ragged", CASES)
def test_decode_small(cuda_lib, B, H, Hkv, Nq, Nk, d, causal, ragged):
    t = make_decode_inputs(B, H, Hkv, Nq, Nk, d, torch.bfloat16, seed=500 + Nk, ragged=ragged)
    scale = 1 / math.sqrt(d)
    o, lse = run_decode(cuda_lib, t, scale, causal, t.get("kv_len"))
    ref = oracle.decode(t["q"], t["k"], t["v"], scale, causal, t.get("kv_len"))
    check_fwd(o, lse, ref, f"B={B} H={H} Hkv={Hkv} Nq={Nq} Nk={Nk} d={d} causal={causal}")


def test_decode_fp16_and_short_or_empty_caches(cuda_lib):
    B, H, Hkv, Nq, Nk, d = 4, 4, 2, 3, 600, 64
    t = make_decode_inputs(B, H, Hkv, Nq, Nk, d, torch.float16, seed=520)
    lens = torch.tensor([0, 2, 600, 1], dtype=torch.int32)  # empty, shorter than Nq, full
    o, lse = run_decode(cuda_lib, t, 0.2, True, lens)
    ref = oracle.decode(t["q"], t["k"], t["v"], 0.2, True, lens)
    check_fwd(o, lse, ref, "fp16 short caches")
    assert torch.all(o[0].cpu() == 0) and torch.all(torch.isneginf(lse[0].cpu()))
    # lengths above the capacity are clamped to it
    o2, lse2 = run_decode(cuda_lib, t, 0.2, True, torch.tensor([0, 2, 9999, 1], dtype=torch.int32))
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_decode_is_deterministic(cuda_lib):
    t = make_decode_inputs(2, 8, 2, 2, 3000, 128, torch.bfloat16, seed=530, ragged=True)
    a = run_decode(cuda_lib, t, 0.09, True, t["kv_len"])
    b = run_decode(cuda_lib, t, 0.09, True, t["kv_len"])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_decode_workload_parity(cuda_lib):
    w = DECODE_WORKLOADS["decode_gqa_d128_kv8k"]
    t = decode_inputs(w)
    o, lse = run_decode(cuda_lib, t, w.scale, w.causal, t.get("kv_len"))
    ref = oracle.decode(t["q"], t["k"], t["v"], w.scale, w.causal, t.get("kv_len"))
    check_fwd(o, lse, ref, w.name)
