"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element by element.

Tolerances (fixed for this method):
  O      max |O - O_ref| <= 2e-2 and ||O - O_ref||_F / ||O_ref||_F <= 5e-3
  LSE    max |LSE - LSE_ref| <= 1e-3
  dQ, dK, dV   ||x - x_ref||_F / ||x_ref||_F <= 1e-2
  tile skipping (which score tiles each kernel computes): bit-exact
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_staged_gb300.workloads import (BLOCK, WORKLOADS, make_block_mask,
                                                    make_inputs, workload_inputs)

pytestmark = pytest.mark.gpu

O_MAX, O_REL, LSE_MAX, G_REL = 2e-2, 5e-3, 1e-3, 1e-2
DEV = "cuda:0"


def relf(a, b):
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def np64(t):
    return t.detach().double().cpu().numpy()


def check_fwd(o, lse, ref, what="", o_scale=1.0):
    """O within O_MAX * o_scale (max abs) and O_REL (relative Frobenius), LSE within LSE_MAX.
    o_scale > 1 where the outputs are that much larger than plain attention's (dropout)."""
    o, lse = np64(o), np64(lse)
    err = float(np.max(np.abs(o - ref["o"])))
    rel = relf(o, ref["o"])
    fin = np.isfinite(ref["lse"])
    assert np.array_equal(np.isneginf(lse), ~fin), f"{what}: -inf LSE rows differ"
    lerr = float(np.max(np.abs(lse[fin] - ref["lse"][fin]))) if fin.any() else 0.0
    assert err <= O_MAX * o_scale and rel <= O_REL, f"{what}: O maxabs {err:.3e} relF {rel:.3e}"
    assert lerr <= LSE_MAX, f"{what}: LSE maxabs {lerr:.3e}"


def check_bwd(grads, ref, what=""):
    for name, g in zip(("dq", "dk", "dv"), grads):
        r = relf(np64(g), ref[name])
        assert r <= G_REL, f"{what}: {name} relF {r:.3e}"


def run_pair(api, t, scale, causal, mask=None, backward=True):
    q, k, v, do = (t[x].to(DEV) for x in ("q", "k", "v", "do"))
    m = None if mask is None else mask.to(DEV)
    o, lse = api.fwd(q, k, v, scale, causal=causal, block_mask=m)
    grads = api.bwd(q, k, v, o, lse, do, scale, causal=causal, block_mask=m) if backward else None
    assert api.sync_status() == 0
    return o, lse, grads


SMALL = [(n, d) for d in (64, 128) for n in (1, 17, 128, 200, 256, 384, 513)]


@pytest.mark.parametrize("N,d", SMALL)
@pytest.mark.parametrize("causal", [False, True])
def test_small_shapes_bf16(cuda_lib, N, d, causal):
    t = make_inputs(1, 2, N, d, torch.bfloat16, seed=100 + N + d)
    scale = 1 / math.sqrt(d)
    o, lse, grads = run_pair(cuda_lib, t, scale, causal)
    ref = oracle.attention(t["q"], t["k"], t["v"], scale, causal, dout=t["do"])
    check_fwd(o, lse, ref, f"N={N} d={d} causal={causal}")
    check_bwd(grads, ref, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("N,d", [(128, 64), (300, 128), (640, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_small_shapes_fp16(cuda_lib, N, d, causal):
    t = make_inputs(2, 1, N, d, torch.float16, seed=200 + N)
    scale = 1 / math.sqrt(d)
    o, lse, grads = run_pair(cuda_lib, t, scale, causal)
    ref = oracle.attention(t["q"], t["k"], t["v"], scale, causal, dout=t["do"])
    check_fwd(o, lse, ref, f"fp16 N={N} d={d} causal={causal}")
    check_bwd(grads, ref, f"fp16 N={N} d={d} causal={causal}")


def test_wide_scores_and_odd_scale(cuda_lib):
    # scores of std ~8 make the running max move often (many rescales of O and l)
    t = make_inputs(1, 2, 700, 128, torch.bfloat16, seed=7, qk_mult=2.0)
    o, lse, grads = run_pair(cuda_lib, t, 0.17, True)
    ref = oracle.attention(t["q"], t["k"], t["v"], 0.17, True, dout=t["do"])
    check_fwd(o, lse, ref, "wide")
    check_bwd(grads, ref, "wide")


@pytest.mark.parametrize("N,d,causal,seed", [(640, 64, False, 1), (640, 128, True, 2),
                                             (1000, 64, True, 3), (1000, 128, False, 4)])
def test_block_sparse_small(cuda_lib, N, d, causal, seed):
    T = (N + BLOCK - 1) // BLOCK
    mask = make_block_mask(T, seed, 0.4, keep_diagonal=(seed % 2 == 0))
    mask[1, :] = 0  # one query block with no key at all: O = 0, LSE = -inf, zero gradients
    t = make_inputs(1, 2, N, d, torch.bfloat16, seed=300 + seed)
    scale = 1 / math.sqrt(d)
    o, lse, grads = run_pair(cuda_lib, t, scale, causal, mask)
    ref = oracle.attention(t["q"], t["k"], t["v"], scale, causal, mask, dout=t["do"])
    check_fwd(o, lse, ref, "sparse")
    check_bwd(grads, ref, "sparse")
    assert torch.all(o[:, :, 128:256].cpu() == 0)
    assert torch.all(grads[0][:, :, 128:256].cpu() == 0)


@pytest.mark.parametrize("T", [2048, 2049, 4096, 4097])
def test_block_mask_wider_than_shared_copy(cuda_lib, T):
    # The forward copies the mask rows of its query tiles into shared memory as bits when the
    # mask is at most 2048 tiles wide, the backward kernels a row or column of up to 4096 tiles;
    # wider masks are read from global memory.  A mask of 2 x 2 diagonal super-blocks (and a lone
    # last block when T is odd) splits the attention into independent problems of 256 rows
    # (keys and queries alike), which the oracle solves one at a time.
    N, d = T * BLOCK, 64
    sb = torch.arange(T) // 2
    mask = (sb[:, None] == sb[None, :]).to(torch.uint8).contiguous()
    t = make_inputs(1, 1, N, d, torch.bfloat16, seed=41)
    o, lse, grads = run_pair(cuda_lib, t, 0.125, False, mask)
    for a in (0, 1400, 2 * ((T - 1) // 2)):
        rows = slice(a * BLOCK, min(a + 2, T) * BLOCK)
        sub = {x: t[x][0, 0, rows] for x in ("q", "k", "v", "do")}
        ref = oracle.attention(sub["q"], sub["k"], sub["v"], 0.125, False, None, dout=sub["do"])
        check_fwd(o[0, 0, rows], lse[0, 0, rows], ref, f"T={T} block {a}")
        check_bwd([g[0, 0, rows] for g in grads], ref, f"T={T} block {a}")


def visit_log_buffer(n):
    """A zeroed device log for n tile entries, rounded up to whole 32-bit words (the kernels mark
    it with 32-bit atomic ORs)."""
    return torch.zeros((n + 3) // 4 * 4, dtype=torch.uint8, device=DEV)


def expected_visits(BH, T, causal, mask):
    i = np.arange(T)
    live = np.ones((T, T), dtype=bool)
    if causal:
        live &= i[None, :] <= i[:, None]
    if mask is not None:
        live &= mask.numpy().astype(bool)
    return np.broadcast_to(live.astype(np.uint8) * 7, (BH, T, T)).copy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("sparse", [False, True])
def test_tile_skipping_is_bit_exact(cuda_lib, causal, sparse):
    B, H, N, d = 1, 3, 1100, 64
    T = (N + BLOCK - 1) // BLOCK
    mask = make_block_mask(T, 9, 0.3) if sparse else None
    t = make_inputs(B, H, N, d, torch.bfloat16, seed=9)
    log = visit_log_buffer(B * H * T * T)
    cuda_lib.debug_set_visit_log(log)
    try:
        run_pair(cuda_lib, t, 0.125, causal, mask)
    finally:
        cuda_lib.debug_set_visit_log(None)
    got = log.cpu().numpy()[:B * H * T * T].reshape(B * H, T, T)
    assert np.array_equal(got, expected_visits(B * H, T, causal, mask))


def test_dead_key_blocks_are_never_read(cuda_lib):
    # key block 2 is masked for every query block: NaNs there must not reach any output
    N, d = 768, 128
    T = N // BLOCK
    mask = torch.ones(T, T, dtype=torch.uint8)
    mask[:, 2] = 0
    t = make_inputs(1, 2, N, d, torch.bfloat16, seed=21)
    clean = run_pair(cuda_lib, t, 0.1, False, mask)
    p = dict(t)
    p["k"] = t["k"].clone()
    p["v"] = t["v"].clone()
    p["k"][:, :, 256:384] = float("nan")
    p["v"][:, :, 256:384] = float("nan")
    dirty = run_pair(cuda_lib, p, 0.1, False, mask)
    assert torch.equal(clean[0], dirty[0]) and torch.equal(clean[1], dirty[1])
    for a, b in zip(clean[2], dirty[2]):
        assert torch.equal(a, b)


def test_deterministic(cuda_lib):
    t = make_inputs(2, 2, 900, 128, torch.bfloat16, seed=31)
    a = run_pair(cuda_lib, t, 0.09, True)
    b = run_pair(cuda_lib, t, 0.09, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for x, y in zip(a[2], b[2]):
        assert torch.equal(x, y)


@pytest.mark.parametrize("d, causal", [(64, False), (64, True), (128, False)])
def test_dkdv_repeatable_over_long_key_walks(cuda_lib, d, causal):
    # dK/dV at head dimension 64 issues the next S^T before dV of the current query tile, so its
    # compute warps can drift a tile apart; each S^T buffer has its own probability-ready
    # barrier for that reason.  Long key walks (128 query tiles a key tile) and many CTAs per
    # SM give the drift room: dK and dV must come out bit for bit the same every call.
    t = make_inputs(1, 8, 16384, d, torch.bfloat16, seed=37)
    q, k, v, do = (t[x].to(DEV) for x in ("q", "k", "v", "do"))
    o, lse = cuda_lib.fwd(q, k, v, d ** -0.5, causal=causal)
    delta = torch.empty_like(lse)
    cuda_lib.bwd_preprocess(o, do, delta)
    first = None
    for _ in range(4):
        dk, dv = cuda_lib.bwd_dkdv(q, k, v, do, lse, delta, torch.empty_like(q),
                                   torch.empty_like(q), d ** -0.5, causal)
        assert cuda_lib.sync_status() == 0
        assert bool(torch.isfinite(dv).all()) and bool(torch.isfinite(dk).all())
        if first is None:
            first = (dk.clone(), dv.clone())
        else:
            assert torch.equal(first[0], dk) and torch.equal(first[1], dv)


def test_backward_stages_match_fused_call(cuda_lib):
    t = make_inputs(1, 2, 500, 64, torch.bfloat16, seed=41)
    q, k, v, do = (t[x].to(DEV) for x in ("q", "k", "v", "do"))
    o, lse = cuda_lib.fwd(q, k, v, 0.125, causal=True)
    dq, dk, dv = cuda_lib.bwd(q, k, v, o, lse, do, 0.125, causal=True)
    delta = torch.empty_like(lse)
    cuda_lib.bwd_preprocess(o, do, delta)
    dk2, dv2 = cuda_lib.bwd_dkdv(q, k, v, do, lse, delta, torch.empty_like(q),
                                 torch.empty_like(q), 0.125, True)
    dq2 = cuda_lib.bwd_dq(q, k, v, do, lse, delta, torch.empty_like(q), 0.125, True)
    assert cuda_lib.sync_status() == 0
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)
    ref = oracle.attention(t["q"], t["k"], t["v"], 0.125, True, dout=t["do"])
    # D = rowsum(dO o O) from the kernel's own O agrees with the oracle's <P, dP>
    assert float(np.max(np.abs(np64(delta) - ref["delta"]))) <= 2e-2


def test_timeout_is_reported_not_hung(cuda_lib):
    # the forward's load warp skips its first key tile: every wait on it runs out after 50 ms,
    # the kernel returns early, and the status word says so; the context stays usable
    t = make_inputs(1, 1, 256, 64, torch.bfloat16, seed=51)
    q, k, v = (t[x].to(DEV) for x in ("q", "k", "v"))
    cuda_lib.debug_set_wait_limit_ns(50_000_000)
    cuda_lib.debug_set_fault(1)
    try:
        cuda_lib.fwd(q, k, v, 0.125)
        assert cuda_lib.sync_status() == cuda_lib.FA_ERR_TIMEOUT
    finally:
        cuda_lib.debug_set_fault(0)
        cuda_lib.debug_set_wait_limit_ns(0)
    o, lse = cuda_lib.fwd(q, k, v, 0.125)
    assert cuda_lib.sync_status() == 0
    ref = oracle.attention(t["q"], t["k"], t["v"], 0.125)
    check_fwd(o, lse, ref, "after timeout")


@pytest.mark.parametrize("mode,stage", [(2, "dkdv"), (3, "dq")])
def test_backward_timeout_is_reported_not_hung(cuda_lib, mode, stage):
    # the dK/dV (mode 2) or dQ (mode 3) load warp skips its first tile: the bounded waits run
    # out after 50 ms, the kernel returns early, and the context stays usable
    t = make_inputs(1, 1, 256, 64, torch.bfloat16, seed=52)
    q, k, v, do = (t[x].to(DEV) for x in ("q", "k", "v", "do"))
    o, lse = cuda_lib.fwd(q, k, v, 0.125)
    delta = torch.empty_like(lse)
    cuda_lib.bwd_preprocess(o, do, delta)
    assert cuda_lib.sync_status() == 0
    cuda_lib.debug_set_wait_limit_ns(50_000_000)
    cuda_lib.debug_set_fault(mode)
    try:
        if stage == "dkdv":
            cuda_lib.bwd_dkdv(q, k, v, do, lse, delta, torch.empty_like(q), torch.empty_like(q),
                              0.125, False)
        else:
            cuda_lib.bwd_dq(q, k, v, do, lse, delta, torch.empty_like(q), 0.125, False)
        assert cuda_lib.sync_status() == cuda_lib.FA_ERR_TIMEOUT
    finally:
        cuda_lib.debug_set_fault(0)
        cuda_lib.debug_set_wait_limit_ns(0)
    grads = cuda_lib.bwd(q, k, v, o, lse, do, 0.125)
    assert cuda_lib.sync_status() == 0
    ref = oracle.attention(t["q"], t["k"], t["v"], 0.125, dout=t["do"])
    check_bwd(grads, ref, f"after {stage} timeout")


def test_invalid_arguments_on_device(cuda_lib):
    q = torch.zeros(1, 1, 128, 96, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(cuda_lib.FAError) as e:
        cuda_lib.fwd(q, q, q)
    assert e.value.code == cuda_lib.FA_ERR_UNSUPPORTED
    x = torch.zeros(1 * 1 * 128 * 64 + 1, dtype=torch.bfloat16, device=DEV)[1:].view(1, 1, 128, 64)
    with pytest.raises(cuda_lib.FAError) as e:
        cuda_lib.fwd(x, x, x)
    assert e.value.code == cuda_lib.FA_ERR_INVALID


# ---------------------------------------------------------------- the five workloads

def _spread(total, pick):
    """`pick` indices spread evenly over range(total), first and last included."""
    if total <= pick:
        return list(range(total))
    return sorted({round(i * (total - 1) / (pick - 1)) for i in range(pick)})


def sample_rows(N, seed, edge=16, mid=32):
    """The first and last `edge` rows of a head and `mid` seeded random rows in between."""
    rng = np.random.default_rng(seed)
    rows = set(range(min(edge, N))) | set(range(max(0, N - edge), N))
    rows |= set(rng.choice(N, size=min(mid, N), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def check_fwd_rows(o, lse, rows, ref_o, ref_lse, what):
    """Sampled rows of one head against oracle.forward_rows, with the forward's tolerances."""
    got_o, got_l = np64(o)[rows], np64(lse)[rows]
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isneginf(got_l), ~fin), f"{what}: -inf LSE rows differ"
    err = float(np.max(np.abs(got_o - ref_o)))
    rel = relf(got_o, ref_o)
    lerr = float(np.max(np.abs(got_l[fin] - ref_lse[fin]))) if fin.any() else 0.0
    assert err <= O_MAX and rel <= O_REL, f"{what}: O maxabs {err:.3e} relF {rel:.3e}"
    assert lerr <= LSE_MAX, f"{what}: LSE maxabs {lerr:.3e}"


# heads compared in full (forward and backward) per workload: every head where the oracle is
# quick, otherwise heads spread over the whole B*H range, so that every group of heads in the
# kernels' CTA order (heads are scheduled in groups that share L2) has a head checked in full
FULL_HEADS = {"tiny_fwd_fp16": 1, "dense_d64_n1k": 64, "causal_d128_n4k": 32,
              "gpt_causal_d128_n8k": 8, "blocksparse_d64_n16k": 3}


@pytest.mark.parametrize("name", ["tiny_fwd_fp16", "dense_d64_n1k", "causal_d128_n4k",
                                  "gpt_causal_d128_n8k", "blocksparse_d64_n16k"])
def test_workload_parity(cuda_lib, name):
    w = WORKLOADS[name]
    t = workload_inputs(w)
    mask = t.get("block_mask")
    o, lse, grads = run_pair(cuda_lib, t, w.scale, w.causal, mask, backward=w.backward)
    BH = w.B * w.H
    flat = {x: t[x].reshape(BH, w.N, w.d) for x in ("q", "k", "v", "do")}
    of, lf = o.reshape(BH, w.N, w.d), lse.reshape(BH, w.N)
    # every head: 64 sampled rows of O and LSE, each row computed alone by the oracle
    for h in range(BH):
        rows = sample_rows(w.N, 1000 * w.seed + h)
        ro, rl = oracle.forward_rows(flat["q"][h], flat["k"][h], flat["v"][h], w.scale, rows,
                                     w.causal, mask)
        check_fwd_rows(of[h], lf[h], rows, ro, rl, f"{name} head {h} sampled rows")
    # heads spread over the CTA order: the whole head, forward and backward
    for h in _spread(BH, FULL_HEADS[name]):
        ref = oracle.attention(flat["q"][h], flat["k"][h], flat["v"][h], w.scale, w.causal,
                               mask, dout=flat["do"][h] if w.backward else None)
        check_fwd(of[h], lf[h], ref, f"{name} head {h}")
        if w.backward:
            check_bwd([g.reshape(BH, w.N, w.d)[h] for g in grads], ref, f"{name} head {h}")
    assert torch.isfinite(o).all()
    if w.backward:
        for g in grads:
            assert torch.isfinite(g).all()


def heads_per_group(units, N, d, tensors_per_unit):
    """The host's CTA-order group size: as many work-unit heads as keep about 32 MiB of
    streamed 16-bit [N, d] tensors in flight (at least 1, at most `units`)."""
    g = int((32.0 * 1024 * 1024) // (2.0 * N * d * tensors_per_unit))
    return max(1, min(g, units))


@pytest.mark.parametrize("B,H,N,d,causal", [(3, 4, 8192, 128, True), (5, 8, 4096, 64, False)])
def test_partial_last_head_group(cuda_lib, B, H, N, d, causal):
    # B*H is larger than the CTA-order group and not a multiple of it (8192 x 128: groups of 8
    # heads for 12 heads; 4096 x 64: groups of 32 for 40), so the last group is partial in the
    # forward, dK/dV and dQ grids; every head is compared in full with the oracle
    BH = B * H
    grp = heads_per_group(BH, N, d, 2.0)
    assert BH > grp and BH % grp != 0
    t = make_inputs(B, H, N, d, torch.bfloat16, seed=70 + d)
    scale = 1 / math.sqrt(d)
    o, lse, grads = run_pair(cuda_lib, t, scale, causal)
    flat = {x: t[x].reshape(BH, N, d) for x in ("q", "k", "v", "do")}
    for h in range(BH):
        ref = oracle.attention(flat["q"][h], flat["k"][h], flat["v"][h], scale, causal,
                               dout=flat["do"][h])
        check_fwd(o.reshape(BH, N, d)[h], lse.reshape(BH, N)[h], ref, f"head {h}")
        check_bwd([g.reshape(BH, N, d)[h] for g in grads], ref, f"head {h}")
