"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such a caller (a plug-in handed only its input and output buffers by an application that owns
every device allocation, or code that may not take cudaMalloc's device-wide synchronisation)
gets the same gradients as fa_bwd without passing a workspace: the D scratch is a fixed array
inside libfa.so.  This file is collected last so that a failure here stops a `-x` run only
after every other test has run.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_staged_gb300.workloads import make_block_mask, make_inputs

pytestmark = pytest.mark.gpu

G_REL = 1e-2  # the gradient tolerance of the parity tests


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _relf(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    return float((a - b).norm() / b.norm())


def _noalloc(lib, q, k, v, o, lse, do, dq, dk, dv, scale, causal, mask):
    B, H, N, d = q.shape
    dt = 1 if q.dtype == torch.bfloat16 else 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                              _ptr(dk), _ptr(dv), B, H, N, d, dt, float(scale), int(causal),
                              _ptr(mask), stream)


def test_noalloc_backward_matches_workspace_backward_twice(cuda_lib):
    lib = cuda_lib.load()
    dev = "cuda:0"
    # two calls in a row with different shapes: the second must not see the first's scratch
    cases = [(2, 4, 1000, 128, True, None, 61), (1, 3, 640, 64, False, 0.5, 62)]
    for B, H, N, d, causal, sparse, seed in cases:
        t = make_inputs(B, H, N, d, torch.bfloat16, seed=seed)
        q, k, v, do = (t[x].to(dev) for x in ("q", "k", "v", "do"))
        mask = None
        if sparse is not None:
            T = (N + 127) // 128
            mask = make_block_mask(T, seed, sparse).to(dev)
        scale = 1.0 / math.sqrt(d)
        o, lse = cuda_lib.fwd(q, k, v, scale, causal=causal, block_mask=mask)
        ref = cuda_lib.bwd(q, k, v, o, lse, do, scale, causal=causal, block_mask=mask)
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        rc = _noalloc(lib, q, k, v, o, lse, do, dq, dk, dv, scale, causal, mask)
        assert rc == cuda_lib.FA_OK, cuda_lib.status_string(rc)
        assert cuda_lib.sync_status() == 0
        # no device memory was taken by the call (cudaMalloc works in pages of at least 2 MiB)
        assert torch.cuda.mem_get_info()[0] == free_before
        for got, want in zip((dq, dk, dv), ref):
            assert torch.isfinite(got).all()
            assert _relf(got, want) <= G_REL
        # and against the fp64 oracle itself, not only the workspace backward
        want = oracle.attention(t["q"], t["k"], t["v"], scale, causal,
                                None if mask is None else mask.cpu(), dout=t["do"])
        for name, got in zip(("dq", "dk", "dv"), (dq, dk, dv)):
            r = _relf(got, torch.from_numpy(want[name]))
            assert r <= G_REL, f"{name} relF {r:.3e} against the oracle"


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_lib):
    lib = cuda_lib.load()
    # B*H*N one past the limit: refused on the host before any launch, nothing touched
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda:0")
    lse = torch.zeros(4, dtype=torch.float32, device="cuda:0")
    N = cuda_lib.FA_NOALLOC_MAX_ROWS + 1
    p = _ptr(x)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.fa_bwd_noalloc(p, p, p, p, p, _ptr(lse), p, p, p, 1, 1, N, 64, 1, 0.125, 0, None,
                            stream)
    assert rc == cuda_lib.FA_ERR_INVALID
    assert cuda_lib.sync_status() == 0
