"""Pins for the fp64 CPU oracle's forward pass.

Each test checks the oracle against something other than itself: a brute-force
pure-Python evaluation on tiny inputs, closed forms (equal scores, one-hot dominant
scores, causal row 0, N = 1), and invariants (probability rows sum to one, key
permutation, grouped-head mapping).  A dropped term, a wrong sign or index or a
transposed operand in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import make_inputs


def bf(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def brute_fwd(q, k, v, causal, scale):
    """Pure-Python loops, math.exp, no numpy reductions: [N,d] x [N,d] x [N,d]."""
    q = q.to(torch.float64).tolist()
    k = k.to(torch.float64).tolist()
    v = v.to(torch.float64).tolist()
    N, d = len(q), len(q[0])
    O, L = [], []
    for i in range(N):
        js = range(i + 1) if causal else range(N)
        s = {j: scale * sum(q[i][t] * k[j][t] for t in range(d)) for j in js}
        mx = max(s.values())
        e = {j: math.exp(s[j] - mx) for j in js}
        z = sum(e.values())
        O.append([sum(e[j] / z * v[j][c] for j in js) for c in range(d)])
        L.append(mx + math.log(z))
    return np.array(O), np.array(L)


@pytest.mark.parametrize("N,d", [(1, 1), (2, 4), (3, 8), (7, 4), (16, 8)])
@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(N, d, causal):
    x = make_inputs(11 + N + d, 1, 2, 2, N, d)
    scale = 0.37
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, scale)
    for h in range(2):
        Ob, Lb = brute_fwd(x["q"][0, h], x["k"][0, h], x["v"][0, h], causal, scale)
        np.testing.assert_allclose(O[0, h], Ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(L[0, h], Lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one(causal):
    # V = identity rows (d = N) makes O_i equal to the probability row P_i.
    N = 24
    x = make_inputs(5, 1, 1, 1, N, N)
    v = bf(np.eye(N))[None, None]
    O, _ = oracle.attn_fwd(x["q"], x["k"], v, causal, 0.3)
    P = O[0, 0]
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert (P >= 0).all()
    if causal:
        assert np.all(np.triu(P, 1) == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_scores_mean_of_v(causal):
    # Q = 0: every score is 0, so P is uniform over the visible keys.
    N, d = 37, 8
    x = make_inputs(6, 1, 1, 1, N, d)
    q = torch.zeros_like(x["q"])
    O, L = oracle.attn_fwd(q, x["k"], x["v"], causal, 0.125)
    V = x["v"][0, 0].double().numpy()
    if causal:
        want = np.cumsum(V, axis=0) / np.arange(1, N + 1)[:, None]
        want_l = np.log(np.arange(1, N + 1))
    else:
        want = np.broadcast_to(V.mean(axis=0), (N, d))
        want_l = np.full(N, math.log(N))
    np.testing.assert_allclose(O[0, 0], want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L[0, 0], want_l, rtol=0, atol=1e-12)


def test_one_hot_dominant():
    # K_j = e_j (unit rows), Q_i = alpha * e_{pi(i)} with alpha*scale = 60: row i's score
    # for key pi(i) beats every other by 60 nats, so O_i = V_{pi(i)} to ~N e^-60.
    N = d = 16
    rng = np.random.default_rng(0)
    perm = rng.permutation(N)
    scale = 0.25
    alpha = 60.0 / scale
    Q = np.zeros((N, d)); Q[np.arange(N), perm] = alpha
    K = np.eye(N)
    x = make_inputs(7, 1, 1, 1, N, d)
    O, L = oracle.attn_fwd(bf(Q)[None, None], bf(K)[None, None], x["v"], False, scale)
    V = x["v"][0, 0].double().numpy()
    np.testing.assert_allclose(O[0, 0], V[perm], rtol=0, atol=8 * N * math.exp(-60))
    np.testing.assert_allclose(L[0, 0], 60.0, rtol=0, atol=1e-12)


def test_causal_row0_and_single_key():
    N, d = 9, 4
    x = make_inputs(8, 1, 1, 1, N, d)
    scale = 0.5
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], True, scale)
    q0 = x["q"][0, 0, 0].double().numpy(); k0 = x["k"][0, 0, 0].double().numpy()
    np.testing.assert_array_equal(O[0, 0, 0], x["v"][0, 0, 0].double().numpy())
    assert abs(L[0, 0, 0] - scale * float(q0 @ k0)) < 1e-12
    # N = 1 reduces to O = V for either mask.
    y = make_inputs(9, 1, 1, 1, 1, d)
    for causal in (False, True):
        O1, L1 = oracle.attn_fwd(y["q"], y["k"], y["v"], causal, scale)
        np.testing.assert_array_equal(O1[0, 0], y["v"][0, 0].double().numpy())


def test_key_permutation_invariance():
    N, d = 20, 8
    x = make_inputs(10, 1, 1, 1, N, d)
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(3))
    O1, L1 = oracle.attn_fwd(x["q"], x["k"], x["v"], False, 0.2)
    O2, L2 = oracle.attn_fwd(x["q"], x["k"][:, :, perm], x["v"][:, :, perm], False, 0.2)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L1, L2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("Hkv", [1, 2])
def test_grouped_heads_match_repeated_kv(Hkv):
    # Query head h reads key/value head h // (Hq/Hkv): same as repeating each K/V head
    # Hq/Hkv times along the head axis.
    B, Hq, N, d = 2, 4, 12, 8
    x = make_inputs(12, B, Hq, Hkv, N, d)
    g = Hq // Hkv
    kr = x["k"].repeat_interleave(g, dim=1)
    vr = x["v"].repeat_interleave(g, dim=1)
    for causal in (False, True):
        O1, L1 = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, 0.3)
        O2, L2 = oracle.attn_fwd(x["q"], kr, vr, causal, 0.3)
        np.testing.assert_array_equal(O1, O2)
        np.testing.assert_array_equal(L1, L2)


def test_head_subset_matches_full():
    B, Hq, Hkv, N, d = 2, 4, 2, 10, 8
    x = make_inputs(13, B, Hq, Hkv, N, d)
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], True, 0.3)
    heads = [(1, 3), (0, 1)]
    Os, Ls = oracle.attn_fwd(x["q"], x["k"], x["v"], True, 0.3, heads=heads)
    for s, (b, h) in enumerate(heads):
        np.testing.assert_array_equal(Os[s], O[b, h])
        np.testing.assert_array_equal(Ls[s], L[b, h])


def test_golden_two_by_two():
    # Hand-worked case stored under tests/golden (see the file for the derivation).
    import json, os
    with open(os.path.join(os.path.dirname(__file__), "golden", "fwd_2x2.json")) as f:
        g = json.load(f)
    q = bf(g["q"])[None, None]; k = bf(g["k"])[None, None]; v = bf(g["v"])[None, None]
    for case in g["cases"]:
        O, L = oracle.attn_fwd(q, k, v, case["causal"], g["scale"])
        np.testing.assert_allclose(O[0, 0], np.array(case["O"]), rtol=0, atol=2e-15)
        np.testing.assert_allclose(L[0, 0], np.array(case["LSE"]), rtol=0, atol=2e-15)
