"""Pins for the oracle's forward with Nq queries after a cache of Nk >= Nq keys.

Query i stands at key position i + Nk - Nq; with causal it sees keys j <= i + Nk - Nq.
Checked against: a pure-Python brute force on tiny inputs, the last Nq rows of the
(separately pinned) square oracle run on the full sequence, the single-query case (a
query at the end sees every key, so causal = non-causal), and Nq = Nk.
"""
import math

import numpy as np
import pytest

import oracle
from attn_inputs import make_inputs


def brute_kv(q, k, v, causal, scale):
    """Pure-Python loops on one head: q [Nq,d], k/v [Nk,d]."""
    q = q.double().tolist()
    k = k.double().tolist()
    v = v.double().tolist()
    Nq, Nk, d = len(q), len(k), len(q[0])
    O, L = [], []
    for i in range(Nq):
        js = range(i + Nk - Nq + 1) if causal else range(Nk)
        s = {j: scale * sum(q[i][t] * k[j][t] for t in range(d)) for j in js}
        mx = max(s.values())
        e = {j: math.exp(s[j] - mx) for j in js}
        z = sum(e.values())
        O.append([sum(e[j] / z * v[j][c] for j in js) for c in range(d)])
        L.append(mx + math.log(z))
    return np.array(O), np.array(L)


@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 6), (3, 7), (5, 5), (4, 13)])
@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(Nq, Nk, causal):
    d = 4
    x = make_inputs(300 + Nq * 16 + Nk, 1, 2, 1, Nk, d)
    q = x["q"][:, :, Nk - Nq:]
    O, L = oracle.attn_fwd_kv(q, x["k"], x["v"], causal, 0.41)
    for h in range(2):
        Ob, Lb = brute_kv(q[0, h], x["k"][0, 0], x["v"][0, 0], causal, 0.41)
        np.testing.assert_allclose(O[0, h], Ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(L[0, h], Lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq", [1, 9, 40])
def test_suffix_of_square_problem(causal, Nq):
    # The last Nq queries of a square problem over the whole sequence are exactly the
    # problem of those Nq queries against the whole key sequence.
    B, Hq, Hkv, N, d = 2, 4, 2, 40, 8
    x = make_inputs(320 + Nq, B, Hq, Hkv, N, d)
    O_full, L_full = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, 0.3)
    O, L = oracle.attn_fwd_kv(x["q"][:, :, N - Nq:], x["k"], x["v"], causal, 0.3)
    np.testing.assert_allclose(O, O_full[:, :, N - Nq:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, L_full[:, :, N - Nq:], rtol=0, atol=1e-12)


def test_single_query_sees_every_key():
    x = make_inputs(340, 1, 3, 1, 57, 8)
    q = x["q"][:, :, -1:]
    O1, L1 = oracle.attn_fwd_kv(q, x["k"], x["v"], True, 0.2)
    O0, L0 = oracle.attn_fwd_kv(q, x["k"], x["v"], False, 0.2)
    np.testing.assert_array_equal(O1, O0)
    np.testing.assert_array_equal(L1, L0)


def test_square_case_matches_attn_fwd():
    x = make_inputs(350, 1, 2, 2, 33, 8)
    for causal in (False, True):
        O1, L1 = oracle.attn_fwd_kv(x["q"], x["k"], x["v"], causal, 0.25)
        O0, L0 = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, 0.25)
        np.testing.assert_allclose(O1, O0, rtol=0, atol=1e-13)
        np.testing.assert_allclose(L1, L0, rtol=0, atol=1e-13)


def test_causal_needs_enough_keys():
    x = make_inputs(360, 1, 1, 1, 8, 4)
    with pytest.raises(ValueError):
        oracle.attn_fwd_kv(x["q"], x["k"][:, :, :5], x["v"][:, :, :5], True, 0.5)
