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
