"""Pins for the oracle's forward over packed sequences of different lengths.

Each packed sequence is an attention problem of its own.  Checked against: a pure-Python
brute force per sequence on tiny inputs (with grouped heads, empty sequences and
sequences with more keys than queries), isolation (changing one sequence's data leaves
every other sequence's rows bit for bit unchanged, so a wrong offset anywhere fails), and
a single sequence, which must equal the unpacked forward.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import make_inputs, make_varlen_inputs


def brute_seq(q, k, v, causal, scale):
    """One head of one sequence: q [nq,d], k/v [nk,d]; query i stands at key i + nk - nq."""
    q, k, v = q.double().tolist(), k.double().tolist(), v.double().tolist()
    nq, nk, d = len(q), len(k), len(k[0])
    O, L = [], []
    for i in range(nq):
        js = range(i + nk - nq + 1) if causal else range(nk)
        s = {j: scale * sum(q[i][t] * k[j][t] for t in range(d)) for j in js}
        mx = max(s.values())
        e = {j: math.exp(s[j] - mx) for j in js}
        z = sum(e.values())
        O.append([sum(e[j] / z * v[j][c] for j in js) for c in range(d)])
        L.append(mx + math.log(z))
    return np.array(O).reshape(nq, d), np.array(L)


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_per_sequence(causal):
    lens_q = [3, 0, 1, 6, 2]
    lens_k = [5, 2, 1, 6, 9] if causal else [4, 3, 7, 2, 1]
    Hq, Hkv, d = 4, 2, 4
    x = make_varlen_inputs(410 + causal, lens_q, lens_k, Hq, Hkv, d)
    O, L = oracle.attn_fwd_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], causal, 0.45)
    cq, ck = x["cu_q"].tolist(), x["cu_k"].tolist()
    for b in range(len(lens_q)):
        for h in range(Hq):
            hk = h // (Hq // Hkv)
            if lens_q[b] == 0:
                continue
            Ob, Lb = brute_seq(x["q"][h, cq[b]:cq[b + 1]], x["k"][hk, ck[b]:ck[b + 1]],
                               x["v"][hk, ck[b]:ck[b + 1]], causal, 0.45)
            np.testing.assert_allclose(O[h, cq[b]:cq[b + 1]], Ob, rtol=0, atol=1e-12)
            np.testing.assert_allclose(L[h, cq[b]:cq[b + 1]], Lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_sequences_are_isolated(causal):
    lens = [37, 5, 80, 19]
    x = make_varlen_inputs(420, lens, lens, 2, 1, 8)
    O0, L0 = oracle.attn_fwd_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], causal, 0.3)
    cq = x["cu_q"].tolist()
    # Replace every value of sequence 2 (its queries, keys and values).
    y = {n: x[n].clone() for n in ("q", "k", "v")}
    g = torch.Generator().manual_seed(421)
    for n in ("q", "k", "v"):
        part = y[n][:, cq[2]:cq[3]]
        y[n][:, cq[2]:cq[3]] = torch.randn(part.shape, generator=g).to(torch.bfloat16)
    O1, L1 = oracle.attn_fwd_varlen(y["q"], y["k"], y["v"], x["cu_q"], x["cu_k"], causal, 0.3)
    other = np.r_[0:cq[2], cq[3]:cq[-1]]
    np.testing.assert_array_equal(O1[:, other], O0[:, other])
    np.testing.assert_array_equal(L1[:, other], L0[:, other])
    assert np.abs(O1[:, cq[2]:cq[3]] - O0[:, cq[2]:cq[3]]).max() > 1e-3


def test_single_sequence_is_the_unpacked_forward():
    x = make_inputs(430, 1, 4, 2, 45, 8)
    cu = torch.tensor([0, 45], dtype=torch.int32)
    for causal in (False, True):
        O, L = oracle.attn_fwd_varlen(x["q"][0], x["k"][0], x["v"][0], cu, cu, causal, 0.25)
        O0, L0 = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, 0.25)
        np.testing.assert_allclose(O, O0[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(L, L0[0], rtol=0, atol=1e-13)


def test_invalid_offsets_are_rejected():
    x = make_varlen_inputs(440, [3, 4], [3, 4], 1, 1, 4)
    q, k, v = x["q"], x["k"], x["v"]
    bad = [([0, 9, 7], [0, 3, 7]),    # decreasing (the end is right)
           ([1, 3, 7], [0, 3, 7]),    # does not start at 0
           ([0, 3, 6], [0, 3, 7])]    # does not end at the packed length
    for cq, ck in bad:
        with pytest.raises(ValueError):
            oracle.attn_fwd_varlen(q, k, v, cq, ck, False, 0.5)
    with pytest.raises(ValueError):   # a sequence with queries and no keys
        oracle.attn_fwd_varlen(q, k[:, :3], v[:, :3], [0, 3, 7], [0, 3, 3], False, 0.5)
    with pytest.raises(ValueError):   # causal with fewer keys than queries
        oracle.attn_fwd_varlen(q, k[:, :5], v[:, :5], [0, 3, 7], [0, 3, 5], True, 0.5)


# ---------------------------------------------------------------------------- backward
def _fd_loss_kv(q, k, v, do, causal, scale):
    """L = sum(dO o O) for one head of one sequence, fp64, query i at key i + nk - nq."""
    nq, nk = q.shape[0], k.shape[0]
    s = scale * q @ k.T
    if causal:
        s = np.where(np.arange(nk)[None, :] <= np.arange(nq)[:, None] + nk - nq, s, -np.inf)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return float((do * (p @ v)).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_finite_differences_more_keys_than_queries(causal):
    # One sequence of 3 queries after 5 keys, one head: central differences of sum(dO o O).
    x = make_varlen_inputs(450 + causal, [3], [5], 1, 1, 4)
    do = make_varlen_inputs(451, [3], [5], 1, 1, 4)["q"]
    scale = 0.4
    dQ, dK, dV = oracle.attn_bwd_varlen(x["q"], x["k"], x["v"], do, x["cu_q"], x["cu_k"], causal, scale)
    q, k, v, dd = (t[0].double().numpy() for t in (x["q"], x["k"], x["v"], do))
    O, _ = oracle.attn_fwd_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], causal, scale)
    assert abs(_fd_loss_kv(q, k, v, dd, causal, scale) - float((dd * O[0]).sum())) < 1e-12
    h = 1e-6
    for name, arr, grad in (("q", q, dQ[0]), ("k", k, dK[0]), ("v", v, dV[0])):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args = {"q": q, "k": k, "v": v}
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args[name] = plus
            lp = _fd_loss_kv(args["q"], args["k"], args["v"], dd, causal, scale)
            args[name] = minus
            lm = _fd_loss_kv(args["q"], args["k"], args["v"], dd, causal, scale)
            fd[idx] = (lp - lm) / (2 * h)
        assert np.abs(fd - grad).max() / max(1.0, np.abs(grad).max()) < 1e-6, name


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_square_sequences_match_the_unpacked_oracle(causal):
    # Each square sequence against the (separately pinned) C oracle's backward on it alone,
    # with grouped heads (dK, dV summed over the group).
    lens = [9, 1, 30]
    x = make_varlen_inputs(460 + causal, lens, lens, 4, 2, 8)
    do = make_varlen_inputs(461, lens, lens, 4, 2, 8)["q"]
    dQ, dK, dV = oracle.attn_bwd_varlen(x["q"], x["k"], x["v"], do, x["cu_q"], x["cu_k"], causal, 0.3)
    cq = x["cu_q"].tolist()
    for b in range(len(lens)):
        sl = slice(cq[b], cq[b + 1])
        sq = lambda t: t[:, sl].unsqueeze(0).contiguous()
        rq, rk, rv = oracle.attn_bwd(sq(x["q"]), sq(x["k"]), sq(x["v"]), sq(do), causal, 0.3)
        np.testing.assert_allclose(dQ[:, sl], rq[0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dK[:, sl], rk[0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dV[:, sl], rv[0], rtol=0, atol=1e-12)


def test_bwd_keys_without_queries_get_zero_gradients():
    x = make_varlen_inputs(470, [4, 0, 3], [4, 6, 5], 2, 1, 4)
    do = make_varlen_inputs(471, [4, 0, 3], [4, 6, 5], 2, 1, 4)["q"]
    dQ, dK, dV = oracle.attn_bwd_varlen(x["q"], x["k"], x["v"], do, x["cu_q"], x["cu_k"], True, 0.5)
    assert not dK[:, 4:10].any() and not dV[:, 4:10].any()
    assert np.abs(dV[:, :4]).max() > 0 and np.abs(dV[:, 10:]).max() > 0
    # rows of P sum to one: sum over keys of dV equals sum over queries of dO, per sequence
    dof = do.double().numpy()
    np.testing.assert_allclose(dV[0, 10:].sum(axis=0), dof[:, 4:].sum(axis=(0, 1)), atol=1e-12)
