"""Seeded synthetic inputs shared by the CUDA path's tests, the benchmark and the oracle's tests.

This module only draws random numbers and names shapes.  It holds none of the attention
arithmetic, so importing it from both sides keeps the oracle and the CUDA path independent.

Recipe (one per workload):
  * ``torch.Generator('cpu').manual_seed(seed)``; Q, K, V, dO drawn in that order with
    ``randn`` in fp32 of shape [B, H, N, d], then cast to the workload dtype.
  * The long-context workload multiplies Q and K by 2 before the cast (a power of two, so the
    cast of the doubled value equals the double of the cast value).
  * The block-sparse workload's 128x128 block mask: generator seeded with ``seed + 1000``;
    off-diagonal blocks kept iid with probability 0.25, every diagonal block kept.
  * Grouped-query workloads draw K and V with H_kv heads ([B, H_kv, N, d]); Q and dO keep H.
  * FP8 workloads draw Q, K, V as above in fp32, then quantise each tensor to e4m3 with one
    scale: descale = amax / 448, code = e4m3(clamp(x / descale, -448, 448)) (round to nearest);
    the value a code stands for is e4m3(code) * descale.
  * Decode workloads draw Q [B, H, Nq, d], then the cache K, V [B, H_kv, Nk, d], then (ragged
    ones) the per-batch cache lengths uniform in [Nk / 2, Nk], from one seeded generator.

The five workloads follow the shapes of the FlashAttention-2 reading notes' kernel benchmark
(seq 512-16k, hidden 2048, heads of 64/128) and the GPT-style 8k training shape the notes quote.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

BLOCK = 128  # block-mask granularity (rows and columns of the score matrix per mask entry)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str            # "fp16" or "bf16"
    causal: bool
    seed: int
    qk_mult: float = 1.0  # multiplier applied to Q and K before the cast
    sparse_p: Optional[float] = None  # Bernoulli keep-probability of off-diagonal mask blocks
    backward: bool = True
    h_kv: Optional[int] = None  # K/V heads (grouped-query attention); None means H
    dropout: float = 0.0        # probability of dropping a probability (generator seed = seed)

    @property
    def kv_heads(self) -> int:
        return self.H if self.h_kv is None else self.h_kv

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float16 if self.dtype == "fp16" else torch.bfloat16

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def tiles(self) -> int:
        return (self.N + BLOCK - 1) // BLOCK

    def describe(self) -> str:
        kind = "block-sparse" if self.sparse_p is not None else ("causal" if self.causal else "dense")
        passes = "fwd+bwd" if self.backward else "fwd"
        heads = f"H={self.H}" if self.h_kv is None else f"H={self.H} H_kv={self.h_kv}"
        drop = f", dropout {self.dropout}" if self.dropout else ""
        return (f"{self.name}: {passes} {kind} B={self.B} {heads} N={self.N} d={self.d} "
                f"{self.dtype}{drop}")


WORKLOADS: Dict[str, Workload] = {
    # single-tile forward case, small enough for the fp64 oracle in well under a second
    "tiny_fwd_fp16": Workload("tiny_fwd_fp16", 1, 1, 128, 64, "fp16", False, 1, backward=False),
    # non-causal head-64 forward+backward
    "dense_d64_n1k": Workload("dense_d64_n1k", 4, 16, 1024, 64, "bf16", False, 2),
    # causal head-128 forward+backward
    "causal_d128_n4k": Workload("causal_d128_n4k", 2, 16, 4096, 128, "bf16", True, 3),
    # GPT-style long-context training shape, scores widened by doubling Q and K
    "gpt_causal_d128_n8k": Workload("gpt_causal_d128_n8k", 1, 32, 8192, 128, "bf16", True, 4,
                                    qk_mult=2.0),
    # block-sparse head-64 forward+backward at 16k tokens, density about 0.256
    "blocksparse_d64_n16k": Workload("blocksparse_d64_n16k", 1, 8, 16384, 64, "bf16", False, 5,
                                     sparse_p=0.25),
    # the GPT-style 8k shape with grouped K/V heads: 32 query heads over 8 K/V heads
    "gqa_causal_d128_n8k": Workload("gqa_causal_d128_n8k", 1, 32, 8192, 128, "bf16", True, 6,
                                    qk_mult=2.0, h_kv=8),
    # the GPT-style 8k training shape with dropout 0.1 on the attention probabilities
    "dropout_causal_d128_n8k": Workload("dropout_causal_d128_n8k", 1, 32, 8192, 128, "bf16",
                                        True, 9, qk_mult=2.0, dropout=0.1),
}

# the five workloads of the method's scope, in order; the rest extend it (grouped K/V heads)
ORDER = ["tiny_fwd_fp16", "dense_d64_n1k", "causal_d128_n4k", "gpt_causal_d128_n8k",
         "blocksparse_d64_n16k"]
EXTENSIONS = ["gqa_causal_d128_n8k", "dropout_causal_d128_n8k"]

# e4m3 forward workloads: the GPT-style 8k shape with Q, K, V quantised per tensor
FP8_WORKLOADS: Dict[str, Workload] = {
    "fp8_causal_d128_n8k": Workload("fp8_causal_d128_n8k", 1, 32, 8192, 128, "e4m3", True, 8,
                                    qk_mult=2.0, backward=False),
}


def make_inputs(B: int, H: int, N: int, d: int, dtype: torch.dtype, seed: int,
                qk_mult: float = 1.0, with_dout: bool = True,
                h_kv: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Draw Q, K, V (and dO) on the CPU from one seeded generator, in that order."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (B, H, N, d)
    kv_shape = (B, H if h_kv is None else h_kv, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(kv_shape, generator=g, dtype=torch.float32)
    v = torch.randn(kv_shape, generator=g, dtype=torch.float32)
    out = {}
    if qk_mult != 1.0:
        q = q * qk_mult
        k = k * qk_mult
    out["q"] = q.to(dtype)
    out["k"] = k.to(dtype)
    out["v"] = v.to(dtype)
    if with_dout:
        out["do"] = torch.randn(shape, generator=g, dtype=torch.float32).to(dtype)
    return out


def make_block_mask(tiles: int, seed: int, p: float, keep_diagonal: bool = True) -> torch.Tensor:
    """uint8 [tiles, tiles] row-major: 1 keeps a 128x128 score block, 0 skips it."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    m = (torch.rand((tiles, tiles), generator=g) < p).to(torch.uint8)
    if keep_diagonal:
        idx = torch.arange(tiles)
        m[idx, idx] = 1
    return m.contiguous()


def workload_inputs(w: Workload) -> Dict[str, torch.Tensor]:
    out = make_inputs(w.B, w.H, w.N, w.d, w.torch_dtype, w.seed, w.qk_mult, with_dout=True,
                      h_kv=w.h_kv)
    if w.sparse_p is not None:
        out["block_mask"] = make_block_mask(w.tiles, w.seed + 1000, w.sparse_p)
    return out


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """A few new query rows per sequence against a KV cache of Nk positions."""
    name: str
    B: int
    H: int
    h_kv: int
    Nq: int
    Nk: int
    d: int
    dtype: str
    causal: bool
    seed: int
    ragged: bool = False  # per-batch cache lengths in [Nk / 2, Nk] instead of all Nk

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float16 if self.dtype == "fp16" else torch.bfloat16

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def describe(self) -> str:
        lens = "ragged cache lengths" if self.ragged else "full cache"
        return (f"{self.name}: decode B={self.B} H={self.H} H_kv={self.h_kv} Nq={self.Nq} "
                f"Nk={self.Nk} d={self.d} {self.dtype}, {lens}")


DECODE_WORKLOADS: Dict[str, DecodeWorkload] = {
    # one new token per sequence, 16 sequences of 8k cached tokens, 32 query / 8 K/V heads
    "decode_gqa_d128_kv8k": DecodeWorkload("decode_gqa_d128_kv8k", 16, 32, 8, 1, 8192, 128,
                                           "bf16", False, 7),
}


def make_decode_inputs(B: int, H: int, h_kv: int, Nq: int, Nk: int, d: int, dtype: torch.dtype,
                       seed: int, ragged: bool = False) -> Dict[str, torch.Tensor]:
    """Q, the K/V cache and (ragged) int32 cache lengths, in that order from one generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = {"q": torch.randn((B, H, Nq, d), generator=g, dtype=torch.float32).to(dtype),
           "k": torch.randn((B, h_kv, Nk, d), generator=g, dtype=torch.float32).to(dtype),
           "v": torch.randn((B, h_kv, Nk, d), generator=g, dtype=torch.float32).to(dtype)}
    if ragged:
        out["kv_len"] = torch.randint(Nk // 2, Nk + 1, (B,), generator=g, dtype=torch.int32)
    return out


def decode_inputs(w: DecodeWorkload) -> Dict[str, torch.Tensor]:
    return make_decode_inputs(w.B, w.H, w.h_kv, w.Nq, w.Nk, w.d, w.torch_dtype, w.seed, w.ragged)


def quantize_e4m3(x: torch.Tensor):
    """One-scale e4m3 quantisation of an fp32 tensor: (uint8 codes, descale as a float)."""
    amax = float(x.abs().max())
    descale = amax / 448.0 if amax > 0 else 1.0
    codes = (x / descale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), descale


def make_fp8_inputs(B: int, H: int, N: int, d: int, seed: int, qk_mult: float = 1.0,
                    h_kv: Optional[int] = None) -> Dict[str, object]:
    """Q, K, V drawn as in make_inputs (fp32, same order), each quantised to e4m3 codes."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    kv_shape = (B, H if h_kv is None else h_kv, N, d)
    q = torch.randn((B, H, N, d), generator=g, dtype=torch.float32) * qk_mult
    k = torch.randn(kv_shape, generator=g, dtype=torch.float32) * qk_mult
    v = torch.randn(kv_shape, generator=g, dtype=torch.float32)
    out: Dict[str, object] = {}
    for name, x in (("q", q), ("k", k), ("v", v)):
        out[name], out["descale_" + name] = quantize_e4m3(x)
    return out


def fp8_workload_inputs(w: Workload) -> Dict[str, object]:
    return make_fp8_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult, w.h_kv)
