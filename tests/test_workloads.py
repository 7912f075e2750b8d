"""Seeded workload generator: shapes, determinism and the block-mask recipe (CPU only)."""
import torch

from exact_attention_staged_gb300.workloads import (EXTENSIONS, ORDER, WORKLOADS,
                                                    make_block_mask, make_inputs, workload_inputs)


def test_five_workloads_in_order():
    assert ORDER + EXTENSIONS == list(WORKLOADS)
    shapes = [(WORKLOADS[n].B, WORKLOADS[n].H, WORKLOADS[n].N, WORKLOADS[n].d) for n in ORDER]
    assert shapes == [(1, 1, 128, 64), (4, 16, 1024, 64), (2, 16, 4096, 128),
                      (1, 32, 8192, 128), (1, 8, 16384, 64)]
    assert [WORKLOADS[n].seed for n in ORDER] == [1, 2, 3, 4, 5]
    assert WORKLOADS["tiny_fwd_fp16"].dtype == "fp16"
    assert WORKLOADS["causal_d128_n4k"].causal and WORKLOADS["gpt_causal_d128_n8k"].causal


def test_inputs_are_seeded_and_ordered():
    a = make_inputs(1, 2, 33, 8, torch.bfloat16, seed=7)
    b = make_inputs(1, 2, 33, 8, torch.bfloat16, seed=7)
    for key in ("q", "k", "v", "do"):
        assert torch.equal(a[key], b[key])
        assert a[key].dtype == torch.bfloat16 and a[key].shape == (1, 2, 33, 8)
    g = torch.Generator().manual_seed(7)
    q = torch.randn((1, 2, 33, 8), generator=g)
    assert torch.equal(a["q"], q.to(torch.bfloat16))
    k = torch.randn((1, 2, 33, 8), generator=g)
    assert torch.equal(a["k"], k.to(torch.bfloat16))


def test_qk_doubling_is_exact():
    a = make_inputs(1, 1, 64, 16, torch.bfloat16, seed=4, qk_mult=2.0)
    b = make_inputs(1, 1, 64, 16, torch.bfloat16, seed=4)
    assert torch.equal(a["q"].float(), 2 * b["q"].float())
    assert torch.equal(a["k"].float(), 2 * b["k"].float())
    assert torch.equal(a["v"], b["v"])


def test_block_mask_recipe():
    m = make_block_mask(128, 1005, 0.25)
    assert m.dtype == torch.uint8 and m.shape == (128, 128)
    assert torch.all(m.diagonal() == 1)
    density = m.float().mean().item()
    assert abs(density - (128 + 0.25 * 128 * 127) / 128 ** 2) < 0.02
    w = WORKLOADS["blocksparse_d64_n16k"]
    assert w.tiles == 128


def test_small_workload_inputs():
    t = workload_inputs(WORKLOADS["tiny_fwd_fp16"])
    assert t["q"].dtype == torch.float16 and t["q"].shape == (1, 1, 128, 64)


def test_grouped_kv_heads_shapes():
    w = WORKLOADS["gqa_causal_d128_n8k"]
    assert (w.H, w.kv_heads, w.N, w.d) == (32, 8, 8192, 128) and w.causal
    a = make_inputs(2, 6, 40, 8, torch.bfloat16, seed=9, h_kv=2)
    assert a["q"].shape == (2, 6, 40, 8) and a["do"].shape == (2, 6, 40, 8)
    assert a["k"].shape == (2, 2, 40, 8) and a["v"].shape == (2, 2, 40, 8)


def test_decode_inputs():
    from exact_attention_staged_gb300.workloads import DECODE_WORKLOADS, make_decode_inputs
    w = DECODE_WORKLOADS["decode_gqa_d128_kv8k"]
    assert (w.B, w.H, w.h_kv, w.Nq, w.Nk, w.d) == (16, 32, 8, 1, 8192, 128)
    a = make_decode_inputs(3, 4, 2, 2, 64, 8, torch.bfloat16, seed=5, ragged=True)
    b = make_decode_inputs(3, 4, 2, 2, 64, 8, torch.bfloat16, seed=5, ragged=True)
    assert a["q"].shape == (3, 4, 2, 8) and a["k"].shape == (3, 2, 64, 8)
    assert a["kv_len"].dtype == torch.int32 and a["kv_len"].shape == (3,)
    assert torch.all((a["kv_len"] >= 32) & (a["kv_len"] <= 64))
    for key in a:
        assert torch.equal(a[key], b[key])
