"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Every check compares the oracle with something other than itself: the worked example printed
on the wmrh.cn page, closed forms, library routines (scipy, torch autograd), the pages' own
tiled recurrences, brute force and finite differences.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import recurrence
from exact_attention_staged_gb300.workloads import make_block_mask, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- worked example (wmrh.cn page)

def _golden():
    with open(os.path.join(GOLDEN, "online_softmax_worked_example.json")) as f:
        return json.load(f)


def test_worked_example_recurrence_matches_printed_m_and_terms():
    g = _golden()
    steps = recurrence.online_softmax_tiles(g["tiles"])
    ms = [s[0] for s in steps]
    ls = [s[1] for s in steps]
    assert ms == g["printed_row_m"]                       # 2.0, 3.0, 3.0 exactly
    assert round(ls[0], 2) == g["printed_row_l"][0]       # 1.37 as printed
    prev = None
    for i, term in enumerate(g["printed_terms"]):
        # evaluate the page's own written term on the exact previous l
        want = sum(math.exp(e) for e in term["exponents"])
        if term["prev_factor_exponent"] is not None:
            want += prev * math.exp(term["prev_factor_exponent"])
        assert ls[i] == pytest.approx(want, rel=1e-14), term["text"]
        prev = ls[i]
    # the page's printed 1.88 and 3.03 are arithmetic slips (reading recorded in the fixture)
    assert abs(ls[1] - g["printed_row_l"][1]) > 0.2
    assert abs(ls[2] - g["printed_row_l"][2]) > 0.5


def test_worked_example_final_stats_equal_three_pass_oracle():
    g = _golden()
    x = np.concatenate([np.asarray(t) for t in g["tiles"]])
    n = len(x)
    # one query row with q = 1 against keys k_j = x_j (d = 1, scale 1) makes S_0j = x_j
    q = np.zeros((n, 1)); q[0, 0] = 1.0
    k = x.reshape(n, 1).copy()
    v = rand((n, 1), 0)
    res = oracle.attention(q, k, v, scale=1.0)
    steps = recurrence.online_softmax_tiles(g["tiles"])
    m, l = steps[-1]
    assert res["lse"][0] == pytest.approx(m + math.log(l), abs=1e-13)
    assert res["lse"][0] == pytest.approx(scipy.special.logsumexp(x), abs=1e-13)
    # scalar (element-by-element) recurrence of the "Flash Attention v1" page agrees too
    ms, ds = recurrence.online_softmax_scalar(x)
    assert ms == 3.0 and ds == pytest.approx(l, rel=1e-14)
    # merging two halves' statistics gives the same (FlashAttention paper-detail page)
    m1, l1 = recurrence.online_softmax_scalar(x[:3])
    m2, l2 = recurrence.online_softmax_scalar(x[3:])
    mm, lm = recurrence.merge_stats(m1, l1, m2, l2)
    assert mm == 3.0 and lm == pytest.approx(l, rel=1e-14)


# ---------------------------------------------------------------- forward: library and closed forms

@pytest.mark.parametrize("N,d", [(1, 4), (7, 3), (33, 16), (64, 8)])
def test_forward_matches_scipy_softmax(N, d):
    q, k, v = rand((N, d), 1), rand((N, d), 2), rand((N, d), 3)
    scale = 0.37
    res = oracle.attention(q, k, v, scale)
    S = scale * (q @ k.T)
    np.testing.assert_allclose(res["lse"], scipy.special.logsumexp(S, axis=1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(res["o"], scipy.special.softmax(S, axis=1) @ v, rtol=0, atol=1e-12)


def test_two_keys_reduce_to_a_sigmoid():
    # softmax over two scores is the logistic function of their difference
    rng = np.random.default_rng(5)
    d = 6
    q, k, v = rng.standard_normal((2, d)), rng.standard_normal((2, d)), rng.standard_normal((2, d))
    scale = 0.8
    res = oracle.attention(q, k, v, scale)
    for i in range(2):
        z = scale * float(q[i] @ (k[0] - k[1]))
        sig = 1.0 / (1.0 + math.exp(-z))
        np.testing.assert_allclose(res["o"][i], v[1] + (v[0] - v[1]) * sig, atol=1e-14)
        s0, s1 = scale * float(q[i] @ k[0]), scale * float(q[i] @ k[1])
        assert res["lse"][i] == pytest.approx(max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))),
                                              abs=1e-14)


def test_equal_value_rows_give_that_row():
    N, d = 40, 8
    q, k = rand((N, d), 7, 3.0), rand((N, d), 8, 3.0)
    row = rand((d,), 9)
    v = np.tile(row, (N, 1))
    for causal in (False, True):
        res = oracle.attention(q, k, v, 0.5, causal=causal)
        np.testing.assert_allclose(res["o"], np.tile(row, (N, 1)), atol=1e-12)


def test_uniform_scores_average_the_values():
    N, d = 21, 5
    q = np.zeros((N, d))
    k, v = rand((N, d), 10), rand((N, d), 11)
    res = oracle.attention(q, k, v, 1.0)
    np.testing.assert_allclose(res["o"], np.tile(v.mean(axis=0), (N, 1)), atol=1e-13)
    np.testing.assert_allclose(res["lse"], np.full(N, math.log(N)), atol=1e-13)
    res = oracle.attention(q, k, v, 1.0, causal=True)
    want = np.cumsum(v, axis=0) / np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(res["o"], want, atol=1e-13)
    np.testing.assert_allclose(res["lse"], np.log(np.arange(1, N + 1)), atol=1e-13)


def test_rows_of_p_sum_to_one_and_scores_never_exceed_lse():
    N, d = 300, 16
    q, k, v = rand((N, d), 12, 2.0), rand((N, d), 13, 2.0), rand((N, d), 14)
    mask = make_block_mask(3, 99, 0.5).numpy()
    for causal, m in ((False, None), (True, None), (False, mask), (True, mask)):
        P = oracle.probabilities(q, k, 0.25, causal=causal, block_mask=m)
        S = oracle.scores(q, k, 0.25, causal=causal, block_mask=m)
        lse = oracle.attention(q, k, v, 0.25, causal=causal, block_mask=m)["lse"]
        assert np.all(np.abs(P.sum(axis=1) - 1.0) <= 1e-12)
        assert np.all(P >= 0) and np.all(P <= 1)
        assert np.all(S - lse[:, None] <= 0)


def test_causal_matches_brute_force_row_loop():
    N, d = 19, 4
    q, k, v = rand((N, d), 15), rand((N, d), 16), rand((N, d), 17)
    res = oracle.attention(q, k, v, 0.9, causal=True)
    for i in range(N):
        s = [0.9 * float(q[i] @ k[j]) for j in range(i + 1)]
        mx = max(s)
        w = [math.exp(x - mx) for x in s]
        tot = sum(w)
        o = sum(w[j] / tot * v[j] for j in range(i + 1))
        np.testing.assert_allclose(res["o"][i], o, atol=1e-13)
        assert res["lse"][i] == pytest.approx(mx + math.log(tot), abs=1e-13)


def test_block_mask_all_ones_equals_dense_and_masking_drops_blocks():
    N, d, blk = 70, 4, 16
    q, k, v = rand((N, d), 18), rand((N, d), 19), rand((N, d), 20)
    tiles = (N + blk - 1) // blk
    ones = np.ones((tiles, tiles), dtype=np.uint8)
    a = oracle.attention(q, k, v, 0.5, block_mask=ones, block=blk)
    b = oracle.attention(q, k, v, 0.5)
    assert np.array_equal(a["o"], b["o"]) and np.array_equal(a["lse"], b["lse"])
    m = make_block_mask(tiles, 3, 0.4).numpy()
    c = oracle.attention(q, k, v, 0.5, block_mask=m, block=blk)
    for i in range(N):
        keep = [j for j in range(N) if m[i // blk, j // blk]]
        S = 0.5 * (q[i] @ k[keep].T)
        np.testing.assert_allclose(c["o"][i], scipy.special.softmax(S) @ v[keep], atol=1e-13)


def test_fully_masked_rows_are_zero():
    N, d, blk = 48, 4, 16
    q, k, v, do = (rand((N, d), s) for s in (21, 22, 23, 24))
    m = np.ones((3, 3), dtype=np.uint8)
    m[1, :] = 0
    res = oracle.attention(q, k, v, 0.5, block_mask=m, block=blk, dout=do)
    rows = slice(16, 32)
    assert np.all(res["o"][rows] == 0) and np.all(np.isneginf(res["lse"][rows]))
    assert np.all(res["dq"][rows] == 0)
    assert np.all(np.isfinite(res["dk"])) and np.all(np.isfinite(res["dv"]))


def test_forward_rows_match_full_forward():
    N, d = 200, 16
    q, k, v = rand((N, d), 25), rand((N, d), 26), rand((N, d), 27)
    mask = make_block_mask(2, 4, 0.5).numpy()
    full = oracle.attention(q, k, v, 0.3, causal=True, block_mask=mask)
    rows = [0, 5, 127, 128, 199]
    o, lse = oracle.forward_rows(q, k, v, 0.3, rows, causal=True, block_mask=mask)
    np.testing.assert_allclose(o, full["o"][rows], atol=1e-14)
    np.testing.assert_allclose(lse, full["lse"][rows], atol=1e-14)


# ---------------------------------------------------------------- Theorem 1 and the recurrences

@pytest.mark.parametrize("bc", [1, 2, 3, 5, 16])
@pytest.mark.parametrize("causal", [False, True])
def test_theorem1_invariant_at_every_block_boundary(bc, causal):
    N, d, scale = 48, 8, 0.6
    q, k, v = rand((N, d), 30, 2.0), rand((N, d), 31, 2.0), rand((N, d), 32)
    S = oracle.scores(q, k, scale, causal=causal)
    steps, (O, L) = recurrence.fa2_forward_steps(S, v, bc)
    for j, (m, l, Ot) in enumerate(steps):
        n = min((j + 1) * bc, N)
        pref = oracle.attention(q, k[:n], v[:n], scale) if not causal else None
        if causal:
            # prefix of a causal row: keys 0..min(i, n-1); rows with none are still empty
            for i in range(N):
                kk = min(i + 1, n)
                r = oracle.attention(q[i:i + 1], k[:kk], v[:kk], scale)
                assert m[i] + math.log(l[i]) == pytest.approx(r["lse"][0], abs=1e-12)
                np.testing.assert_allclose(Ot[i] / l[i], r["o"][0], atol=1e-12)
        else:
            np.testing.assert_allclose(m + np.log(l), pref["lse"], atol=1e-12)
            np.testing.assert_allclose(Ot / l[:, None], pref["o"], atol=1e-12)
            # m is the running row max of the prefix
            np.testing.assert_array_equal(m, S[:, :n].max(axis=1))
    full = oracle.attention(q, k, v, scale, causal=causal)
    np.testing.assert_allclose(O, full["o"], atol=1e-12)
    np.testing.assert_allclose(L, full["lse"], atol=1e-12)


def test_fa1_normalised_update_gives_same_output():
    N, d = 37, 6
    q, k, v = rand((N, d), 33), rand((N, d), 34), rand((N, d), 35)
    S = oracle.scores(q, k, 1.1)
    for bc in (1, 4, 10):
        np.testing.assert_allclose(recurrence.fa1_forward(S, v, bc),
                                   oracle.attention(q, k, v, 1.1)["o"], atol=1e-12)


# ---------------------------------------------------------------- backward

def _loss(q, k, v, do, scale, causal, mask, blk):
    return float(np.sum(oracle.attention(q, k, v, scale, causal, mask, blk)["o"] * do))


@pytest.mark.parametrize("N,d,causal,masked", [(5, 4, False, False), (16, 8, True, False),
                                               (12, 4, False, True), (16, 4, True, True)])
def test_gradients_match_central_differences(N, d, causal, masked):
    blk = 4
    q, k, v, do = rand((N, d), 40), rand((N, d), 41), rand((N, d), 42), rand((N, d), 43)
    mask = make_block_mask((N + blk - 1) // blk, 7, 0.5).numpy() if masked else None
    scale = 0.7
    res = oracle.attention(q, k, v, scale, causal, mask, blk, dout=do)
    h = 1e-6
    for name, x, g in (("q", q, res["dq"]), ("k", k, res["dk"]), ("v", v, res["dv"])):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], do, scale, causal, mask, blk)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], do, scale, causal, mask, blk)
            fd[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(fd - g) / max(np.linalg.norm(g), 1e-300)
        assert err <= 1e-6, (name, err)


def test_gradients_match_torch_autograd_fp64():
    N, d, blk = 96, 16, 32
    q, k, v, do = (rand((2, N, d), s) for s in (50, 51, 52, 53))
    mask = make_block_mask(3, 11, 0.5).numpy()
    scale = 0.25
    res = oracle.attention(q, k, v, scale, True, mask, blk, dout=do)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    S = scale * tq @ tk.transpose(-1, -2)
    i = torch.arange(N)
    keep = (i[None, :] <= i[:, None]) & torch.tensor(mask, dtype=torch.bool)[i // blk][:, i // blk]
    S = S.masked_fill(~keep, float("-inf"))
    O = torch.softmax(S, dim=-1) @ tv
    O.backward(torch.tensor(do))
    np.testing.assert_allclose(res["o"], O.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(res["lse"], torch.logsumexp(S, -1).detach().numpy(), atol=1e-12)
    for name, t in (("dq", tq), ("dk", tk), ("dv", tv)):
        np.testing.assert_allclose(res[name], t.grad.numpy(), atol=1e-11)


def test_delta_equals_rowsum_of_do_times_o():
    N, d = 50, 8
    q, k, v, do = (rand((N, d), s) for s in (60, 61, 62, 63))
    for causal in (False, True):
        res = oracle.attention(q, k, v, 0.4, causal, dout=do)
        np.testing.assert_allclose(res["delta"], np.sum(do * res["o"], axis=1), atol=1e-12)


def test_single_key_special_cases():
    d = 6
    q, k, v, do = (rand((1, d), s) for s in (70, 71, 72, 73))
    res = oracle.attention(q, k, v, 0.5, dout=do)
    np.testing.assert_allclose(res["o"], v, atol=0)
    assert res["lse"][0] == pytest.approx(0.5 * float(q[0] @ k[0]), abs=1e-15)
    assert np.all(res["dq"] == 0) and np.all(res["dk"] == 0)
    np.testing.assert_allclose(res["dv"], do, atol=0)
    # causal row 0 sees only key 0: same closed forms for that row
    N = 9
    q, k, v, do = (rand((N, d), s) for s in (74, 75, 76, 77))
    res = oracle.attention(q, k, v, 0.5, causal=True, dout=do)
    np.testing.assert_allclose(res["o"][0], v[0], atol=0)
    assert np.all(res["dq"][0] == 0)


def test_accepts_seeded_low_precision_inputs_exactly():
    t = make_inputs(1, 2, 33, 8, torch.bfloat16, seed=3)
    res = oracle.attention(t["q"], t["k"], t["v"], 0.35, dout=t["do"])
    q = t["q"].double().numpy()
    assert res["o"].shape == q.shape and res["lse"].shape == q.shape[:-1]
    # the bf16 values are carried into fp64 without change
    S = 0.35 * q[0, 1] @ t["k"].double().numpy()[0, 1].T
    np.testing.assert_allclose(res["lse"][0, 1], scipy.special.logsumexp(S, axis=1), atol=1e-12)


# ---------------------------------------------------------------- grouped-query attention
# FlashAttention-2 reading notes, MQA/GQA section: query head h uses K/V head h // (H / H_kv),
# and the gradient of a shared K/V head is the sum over its query heads.

def _gqa_torch(q, k, v, do, scale, causal):
    """Independent fp64 autograd: every query head indexes its K/V head directly (no expansion,
    no explicit group sum: autograd accumulates the shared leaves' gradients itself)."""
    B, H, N, d = q.shape
    rep = H // k.shape[1]
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    outs, lses = [], []
    i = torch.arange(N)
    for h in range(H):
        S = scale * tq[:, h] @ tk[:, h // rep].transpose(-1, -2)
        if causal:
            S = S.masked_fill(i[None, :] > i[:, None], float("-inf"))
        outs.append(torch.softmax(S, dim=-1) @ tv[:, h // rep])
        lses.append(torch.logsumexp(S, dim=-1))
    O = torch.stack(outs, dim=1)
    O.backward(torch.tensor(do))
    return (O.detach().numpy(), torch.stack(lses, 1).detach().numpy(), tq.grad.numpy(),
            tk.grad.numpy(), tv.grad.numpy())


@pytest.mark.parametrize("H,Hkv,causal", [(4, 2, False), (6, 3, True), (4, 1, True),
                                           (3, 3, False)])
def test_gqa_matches_per_head_torch_autograd(H, Hkv, causal):
    B, N, d = 2, 20, 8
    q, do = rand((B, H, N, d), 80), rand((B, H, N, d), 81)
    k, v = rand((B, Hkv, N, d), 82), rand((B, Hkv, N, d), 83)
    res = oracle.attention_gqa(q, k, v, 0.45, causal, dout=do)
    o, lse, dq, dk, dv = _gqa_torch(q, k, v, do, 0.45, causal)
    np.testing.assert_allclose(res["o"], o, atol=1e-12)
    np.testing.assert_allclose(res["lse"], lse, atol=1e-12)
    for name, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(res[name], ref, atol=1e-11)


def test_gqa_with_one_head_per_group_is_mha():
    q, k, v, do = (rand((2, 3, 17, 4), s) for s in (84, 85, 86, 87))
    a = oracle.attention_gqa(q, k, v, 0.6, True, dout=do)
    b = oracle.attention(q, k, v, 0.6, True, dout=do)
    for name in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_array_equal(a[name], b[name])


def test_mqa_with_identical_query_heads_scales_kv_gradients():
    # all H query heads equal (and their dO equal): every head produces the same dK, dV, so the
    # shared head's gradients are exactly H times one head's, while O and dQ repeat per head
    H, N, d = 5, 12, 4
    q1, do1 = rand((1, 1, N, d), 88), rand((1, 1, N, d), 89)
    k, v = rand((1, 1, N, d), 90), rand((1, 1, N, d), 91)
    q, do = np.repeat(q1, H, axis=1), np.repeat(do1, H, axis=1)
    many = oracle.attention_gqa(q, k, v, 0.8, False, dout=do)
    one = oracle.attention(q1, k, v, 0.8, False, dout=do1)
    np.testing.assert_allclose(many["dk"], H * one["dk"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(many["dv"], H * one["dv"], rtol=1e-13, atol=1e-14)
    for h in range(H):
        np.testing.assert_array_equal(many["o"][:, h], one["o"][:, 0])
        np.testing.assert_array_equal(many["dq"][:, h], one["dq"][:, 0])


def test_gqa_gradients_match_central_differences():
    B, H, Hkv, N, d = 1, 4, 2, 6, 3
    q, do = rand((B, H, N, d), 92), rand((B, H, N, d), 93)
    k, v = rand((B, Hkv, N, d), 94), rand((B, Hkv, N, d), 95)
    res = oracle.attention_gqa(q, k, v, 0.9, True, dout=do)

    def loss(kk, vv):
        return float(np.sum(oracle.attention_gqa(q, kk, vv, 0.9, True)["o"] * do))

    h = 1e-6
    for name, x, g in (("k", k, res["dk"]), ("v", v, res["dv"])):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            if name == "k":
                fd[idx] = (loss(xp, v) - loss(xm, v)) / (2 * h)
            else:
                fd[idx] = (loss(k, xp) - loss(k, xm)) / (2 * h)
        err = np.linalg.norm(fd - g) / np.linalg.norm(g)
        assert err <= 1e-6, (name, err)


def test_gqa_rejects_heads_that_do_not_divide():
    with pytest.raises(ValueError):
        oracle.attention_gqa(rand((1, 4, 8, 4), 1), rand((1, 3, 8, 4), 2), rand((1, 3, 8, 4), 3),
                             0.5)


# ---------------------------------------------------------------- decode against a KV cache
# FlashAttention-2 reading notes, KV-cache section: a few new query rows against the cache.

def test_decode_with_every_row_new_is_causal_attention():
    # Nq = Nk = kv_len: the new rows are the whole sequence, so end alignment is the usual
    # causal mask of the (pinned) three-pass oracle
    q, k, v = (rand((2, 3, 19, 8), s) for s in (100, 101, 102))
    a = oracle.decode(q, k, v, 0.3, causal=True)
    b = oracle.attention(q, k, v, 0.3, True)
    np.testing.assert_allclose(a["o"], b["o"], atol=1e-13)
    np.testing.assert_allclose(a["lse"], b["lse"], atol=1e-13)


def test_decode_noncausal_ragged_lengths_match_truncated_attention():
    B, H, Hkv, Nq, Nk, d = 3, 4, 2, 3, 40, 8
    q = rand((B, H, Nq, d), 103)
    k, v = rand((B, Hkv, Nk, d), 104), rand((B, Hkv, Nk, d), 105)
    lens = [40, 17, 1]
    a = oracle.decode(q, k, v, 0.5, kv_len=lens)
    for b, L in enumerate(lens):
        ref = oracle.attention_gqa(q[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L], 0.5)
        np.testing.assert_allclose(a["o"][b:b + 1], ref["o"], atol=1e-13)
        np.testing.assert_allclose(a["lse"][b:b + 1], ref["lse"], atol=1e-13)


def test_decode_causal_rows_are_the_last_rows_of_a_square_problem():
    # Nq new rows at the end of a length-L sequence: rows L-Nq .. L-1 of the square causal
    # problem whose earlier query rows are anything (here zeros)
    L, Nq, d = 37, 5, 8
    q, k, v = rand((1, 1, Nq, d), 106), rand((1, 1, L, d), 107), rand((1, 1, L, d), 108)
    a = oracle.decode(q, k, v, 0.4, causal=True)
    qfull = np.zeros((L, d))
    qfull[L - Nq:] = q[0, 0]
    o, lse = oracle.forward_rows(qfull, k[0, 0], v[0, 0], 0.4, list(range(L - Nq, L)), True)
    np.testing.assert_allclose(a["o"][0, 0], o, atol=1e-13)
    np.testing.assert_allclose(a["lse"][0, 0], lse, atol=1e-13)


def test_decode_rows_that_see_nothing():
    q, k, v = rand((2, 1, 4, 4), 109), rand((2, 1, 10, 4), 110), rand((2, 1, 10, 4), 111)
    a = oracle.decode(q, k, v, 1.0, causal=True, kv_len=[0, 2])
    assert np.all(a["o"][0] == 0) and np.all(np.isneginf(a["lse"][0]))
    # batch 1: length 2 with 4 new rows: rows 0, 1 are positions -2, -1 (nothing), rows 2, 3
    # are positions 0 and 1
    assert np.all(a["o"][1, 0, :2] == 0) and np.all(np.isneginf(a["lse"][1, 0, :2]))
    np.testing.assert_allclose(a["o"][1, 0, 2], v[1, 0, 0], atol=1e-15)
    assert a["lse"][1, 0, 2] == pytest.approx(float(q[1, 0, 2] @ k[1, 0, 0]), abs=1e-14)


def test_split_key_ranges_merge_to_the_whole_row():
    # FlashAttention paper detail, Technique 1: the statistics (and, scaled the same way, the
    # outputs) of two key ranges combine into those of their concatenation
    q, k, v = rand((1, 1, 1, 16), 112), rand((1, 1, 300, 16), 113), rand((1, 1, 300, 16), 114)
    whole = oracle.decode(q, k, v, 0.25)
    a = oracle.decode(q, k[:, :, :123], v[:, :, :123], 0.25)
    b = oracle.decode(q, k[:, :, 123:], v[:, :, 123:], 0.25)
    la, lb = a["lse"][0, 0, 0], b["lse"][0, 0, 0]
    m, l = recurrence.merge_stats(la, 1.0, lb, 1.0)  # each part's l is e^{LSE - LSE} = 1
    wa, wb = np.exp(la - m) / l, np.exp(lb - m) / l
    np.testing.assert_allclose(m + np.log(l), whole["lse"][0, 0, 0], atol=1e-13)
    np.testing.assert_allclose(wa * a["o"][0, 0, 0] + wb * b["o"][0, 0, 0], whole["o"][0, 0, 0],
                               atol=1e-13)



# ---------------------------------------------------------------- e4m3 inputs

def test_e4m3_decoder_matches_the_format_and_torch():
    # values fixed by the format: bias 7, 3 mantissa bits, subnormals below 2^-6, max 448
    fixed = {0x00: 0.0, 0x80: -0.0, 0x38: 1.0, 0x7E: 448.0, 0xFE: -448.0, 0x08: 2.0 ** -6,
             0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x40: 2.0, 0x3C: 1.5, 0x30: 0.5}
    got = oracle.e4m3_to_f64(np.array(list(fixed), dtype=np.uint8))
    np.testing.assert_array_equal(got, np.array(list(fixed.values())))
    assert np.isnan(oracle.e4m3_to_f64(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    # every code against torch's float8_e4m3fn conversion (a library routine)
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = oracle.e4m3_to_f64(codes)
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(mine[ok], ref[ok])


def test_fp8_attention_is_attention_of_the_decoded_values():
    from exact_attention_staged_gb300.workloads import make_fp8_inputs
    t = make_fp8_inputs(1, 4, 40, 8, seed=12, h_kv=2)
    a = oracle.attention_fp8(t["q"], t["k"], t["v"], 0.3, t["descale_q"], t["descale_k"],
                             t["descale_v"], causal=True)
    # decode through torch instead, then the (pinned) grouped-query oracle
    dec = {x: t[x].view(torch.float8_e4m3fn).to(torch.float64) * t["descale_" + x]
           for x in ("q", "k", "v")}
    b = oracle.attention_gqa(dec["q"], dec["k"], dec["v"], 0.3, True)
    np.testing.assert_array_equal(a["o"], b["o"])
    np.testing.assert_array_equal(a["lse"], b["lse"])
    for x in ("q", "k", "v"):  # the quantisation leaves every code finite
        assert not np.isnan(oracle.e4m3_to_f64(t[x])).any()


def test_fp8_descales_in_a_two_key_closed_form():
    # one query against two keys is a logistic choice between the two value rows; written out
    # by hand from the codes: q = 1.0 (0x38), k0 = 2.0 (0x40), k1 = 0.5 (0x30), v0 = 1.5 (0x3C),
    # v1 = -1.0 (0xB8), so s_i = scale * dq * dk * q k_i and O = dv (1.5 s(s0 - s1) - s(s1 - s0))
    # with s the logistic function; the descales of Q and K enter only through the scores, the
    # descale of V only as a factor of O
    q = np.array([[[[0x38]]]], dtype=np.uint8)
    k = np.array([[[[0x40], [0x30]]]], dtype=np.uint8)
    v = np.array([[[[0x3C], [0xB8]]]], dtype=np.uint8)
    for scale, dq, dk, dv in ((0.5, 1.0, 1.0, 1.0), (0.7, 0.25, 3.0, 2.5), (1.3, 2.0, 0.125, 0.1)):
        s0, s1 = scale * dq * dk * 2.0, scale * dq * dk * 0.5
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        want_o = dv * (1.5 * w0 - 1.0 * (1.0 - w0))
        want_lse = math.log(math.exp(s0) + math.exp(s1))
        # two query rows: row 0 sees only key 0 under the causal mask, row 1 sees both
        qq = np.concatenate([q, q], axis=2)
        got = oracle.attention_fp8(qq, k, v, scale, dq, dk, dv, causal=True)
        np.testing.assert_allclose(got["o"][0, 0, 1, 0], want_o, rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(got["lse"][0, 0, 1], want_lse, rtol=1e-14)
        np.testing.assert_allclose(got["o"][0, 0, 0, 0], dv * 1.5, rtol=1e-15)
        np.testing.assert_allclose(got["lse"][0, 0, 0], s0, rtol=1e-14)


# ---------------------------------------------------------------- dropout
from oracle import dropout as odrop  # noqa: E402


def _curand():
    """cuRAND (an NVIDIA library with its own Philox4x32-10) through ctypes, or None."""
    import ctypes
    import ctypes.util
    names = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64", "libcurand.so"),
             ctypes.util.find_library("curand"), "libcurand.so", "libcurand.so.10"]
    for n in names:
        if not n:
            continue
        try:
            return ctypes.CDLL(n)
        except OSError:
            continue
    return None


def _curand_philox_words(lib, seed, offset, n):
    import ctypes
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0  # PSEUDO_PHILOX4_32_10
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out


def test_philox_matches_curand_host_generator():
    # cuRAND's host Philox4_32_10 generator is another implementation of the same generator:
    # for seed s its value 4 i + j is word j of Philox4x32-10 with counter (0, 0, i, 0) and key
    # (s mod 2^32, s div 2^32), so whole blocks, every round and the key schedule are compared
    lib = _curand()
    if lib is None:
        pytest.skip("cuRAND is not installed")
    for seed in (0, 1, 0x123456789ABCDEF0, 2 ** 64 - 1):
        ref = _curand_philox_words(lib, seed, 0, 256).reshape(64, 4)
        ctr = np.zeros((64, 4), dtype=np.uint64)
        ctr[:, 2] = np.arange(64)
        mine = odrop.philox4x32_10(ctr, (seed & 0xFFFFFFFF, seed >> 32))
        np.testing.assert_array_equal(mine, ref)
    # a start offset lands on block offset / 4 of the same stream
    ref = _curand_philox_words(lib, 77, 4 * 1000, 8).reshape(2, 4)
    ctr = np.zeros((2, 4), dtype=np.uint64)
    ctr[:, 2] = [1000, 1001]
    np.testing.assert_array_equal(odrop.philox4x32_10(ctr, (77, 0)), ref)


def test_dropout_rate_and_threshold():
    assert odrop.threshold(0.1) == 26 and odrop.threshold(0.0) == 0
    with pytest.raises(ValueError):
        odrop.threshold(1.0)
    z = odrop.keep_mask(3, 512, 2048, seed=7, offset=1, t=64)  # p = 0.25
    frac = 1.0 - z.mean()
    sigma = math.sqrt(0.25 * 0.75 / z.size)
    assert abs(frac - 0.25) < 5 * sigma
    # different heads, rows, offsets give different decisions
    assert not np.array_equal(z, odrop.keep_mask(4, 512, 2048, seed=7, offset=1, t=64))
    assert not np.array_equal(z, odrop.keep_mask(3, 512, 2048, seed=7, offset=2, t=64))


def test_dropout_zero_is_attention():
    q, k, v, do = (rand((1, 2, 70, 8), s) for s in (120, 121, 122, 123))
    a = odrop.attention_dropout(q, k, v, 0.4, 0.0, seed=1, causal=True, dout=do)
    b = oracle.attention(q, k, v, 0.4, True, dout=do)
    for name in ("o", "lse", "dq", "dk", "dv", "delta"):
        np.testing.assert_allclose(a[name], b[name], atol=1e-12)


def test_dropout_gradients_match_torch_autograd_and_delta_identity():
    B, H, N, d, blk = 1, 2, 48, 8, 16
    q, k, v, do = (rand((B, H, N, d), s) for s in (124, 125, 126, 127))
    mask = make_block_mask(3, 13, 0.6).numpy()
    p, seed, off = 0.3, 99, 5
    res = odrop.attention_dropout(q, k, v, 0.35, p, seed, off, True, mask, blk, dout=do)
    t = odrop.threshold(p)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    i = torch.arange(N)
    keep = (i[None, :] <= i[:, None]) & torch.tensor(mask, dtype=torch.bool)[i // blk][:, i // blk]
    outs = []
    for h in range(H):
        S = (0.35 * tq[0, h] @ tk[0, h].T).masked_fill(~keep, float("-inf"))
        Z = torch.tensor(odrop.keep_mask(h, N, N, seed, off, t))
        Pd = torch.softmax(S, -1) * Z * (256.0 / (256 - t))
        outs.append(Pd @ tv[0, h])
    O = torch.stack(outs)[None]
    O.backward(torch.tensor(do))
    np.testing.assert_allclose(res["o"], O.detach().numpy(), atol=1e-12)
    for name, x in (("dq", tq), ("dk", tk), ("dv", tv)):
        np.testing.assert_allclose(res[name], x.grad.numpy(), atol=1e-11)
    # D = rowsum(P o dP) equals rowsum(dO o O) with dropout too
    np.testing.assert_allclose(res["delta"], np.sum(do * res["o"], axis=-1), atol=1e-12)
