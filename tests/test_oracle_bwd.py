"""Pins for the fp64 CPU oracle's backward pass.

The gradients are checked against central finite differences of the scalar
L = sum(dO o O), computed from the oracle's own forward (which the forward pins fix),
and against invariants that hold for any inputs: softmax shift invariance
(sum_j dK_j = 0), rows of P summing to one (sum_j dV_j = sum_i dO_i), causal row 0
(dQ_0 = 0), a closed form for equal scores, and grouped-head summation.
"""
import numpy as np
import pytest
import torch

import oracle
from attn_inputs import make_inputs


def _fd_loss(qd, kd, vd, dod, causal, scale):
    """L = sum(dO * O) with O from a plain fp64 numpy evaluation of the definition on
    already-double inputs (perturbed entries are not bf16, so the bf16 oracle cannot
    take them)."""
    N = qd.shape[0]
    S = scale * qd @ kd.T
    if causal:
        S = np.where(np.triu(np.ones((N, N), bool), 1), -np.inf, S)
    S = S - S.max(axis=1, keepdims=True)
    P = np.exp(S)
    P /= P.sum(axis=1, keepdims=True)
    return float((dod * (P @ vd)).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(3, 2), (6, 4)])
def test_finite_differences(causal, N, d):
    x = make_inputs(21 + N, 1, 1, 1, N, d, with_grad=True)
    scale = 0.45
    dQ, dK, dV = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, scale)
    q, k, v, do = (x[n][0, 0].double().numpy() for n in ("q", "k", "v", "do"))
    # The forward of the finite-difference loss must agree with the oracle's forward.
    O, _ = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, scale)
    assert abs(_fd_loss(q, k, v, do, causal, scale) - float((do * O[0, 0]).sum())) < 1e-12
    h = 1e-6
    for name, arr, grad in (("q", q, dQ[0, 0]), ("k", k, dK[0, 0]), ("v", v, dV[0, 0])):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = plus
            lp = _fd_loss(args["q"], args["k"], args["v"], do, causal, scale)
            args[name] = minus
            lm = _fd_loss(args["q"], args["k"], args["v"], do, causal, scale)
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(fd - grad).max() / max(1.0, np.abs(grad).max())
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_invariants(causal):
    B, H, N, d = 1, 2, 33, 8
    x = make_inputs(31, B, H, H, N, d, with_grad=True)
    dQ, dK, dV = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, 0.35)
    do = x["do"].double().numpy()
    # Adding a constant to a row of scores leaves P unchanged: sum over keys of dS is 0,
    # hence sum_j dK_j = scale * sum_i (sum_j dS_ij) Q_i = 0.
    np.testing.assert_allclose(dK.sum(axis=2), 0.0, atol=1e-12)
    # Rows of P sum to one: sum_j dV_j = sum_j sum_i P_ij dO_i = sum_i dO_i.
    np.testing.assert_allclose(dV.sum(axis=2), do.sum(axis=2), atol=1e-12)
    if causal:
        # Query 0 sees only key 0, its probability is exactly 1: dQ_0 = 0.
        np.testing.assert_array_equal(dQ[:, :, 0], 0.0)


def test_equal_scores_closed_form():
    # Q = 0 (non-causal): P_ij = 1/N.  Then dP_ij = dO_i . V_j, D_i = mean_j dP_ij,
    # dQ_i = scale/N * sum_j (dP_ij - D_i) K_j, dV_j = (1/N) sum_i dO_i.
    N, d = 10, 4
    x = make_inputs(41, 1, 1, 1, N, d, with_grad=True)
    q = torch.zeros_like(x["q"])
    scale = 0.7
    dQ, dK, dV = oracle.attn_bwd(q, x["k"], x["v"], x["do"], False, scale)
    k, v, do = (x[n][0, 0].double().numpy() for n in ("k", "v", "do"))
    dP = do @ v.T
    D = dP.mean(axis=1, keepdims=True)
    np.testing.assert_allclose(dQ[0, 0], scale / N * (dP - D) @ k, atol=1e-12)
    np.testing.assert_allclose(dV[0, 0], np.broadcast_to(do.sum(axis=0) / N, (N, d)), atol=1e-12)
    np.testing.assert_allclose(dK[0, 0], 0.0, atol=1e-12)  # Q = 0 => dK = scale dS^T Q = 0


@pytest.mark.parametrize("Hkv", [1, 2])
def test_grouped_heads_sum(Hkv):
    # dK, dV of a shared key/value head are the sums of the per-query-head gradients
    # computed with K/V repeated per head.
    B, Hq, N, d = 1, 4, 9, 4
    x = make_inputs(51, B, Hq, Hkv, N, d, with_grad=True)
    g = Hq // Hkv
    kr = x["k"].repeat_interleave(g, dim=1)
    vr = x["v"].repeat_interleave(g, dim=1)
    for causal in (False, True):
        dQ, dK, dV = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, 0.3)
        dQr, dKr, dVr = oracle.attn_bwd(x["q"], kr, vr, x["do"], causal, 0.3)
        np.testing.assert_allclose(dQ, dQr, atol=1e-13)
        np.testing.assert_allclose(dK, dKr.reshape(B, Hkv, g, N, d).sum(axis=2), atol=1e-13)
        np.testing.assert_allclose(dV, dVr.reshape(B, Hkv, g, N, d).sum(axis=2), atol=1e-13)


def test_kv_subset_matches_full():
    B, Hq, Hkv, N, d = 2, 4, 2, 7, 4
    x = make_inputs(61, B, Hq, Hkv, N, d, with_grad=True)
    dQ, dK, dV = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], True, 0.3)
    sel = [(1, 1), (0, 0)]
    dQs, dKs, dVs = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], True, 0.3, kv_heads=sel)
    g = Hq // Hkv
    for s, (b, h) in enumerate(sel):
        np.testing.assert_array_equal(dQs[s], dQ[b, h * g:(h + 1) * g])
        np.testing.assert_array_equal(dKs[s], dK[b, h])
        np.testing.assert_array_equal(dVs[s], dV[b, h])
