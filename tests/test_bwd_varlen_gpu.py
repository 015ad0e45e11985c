"""Backward over packed sequences (attn_bwd_varlen): dQ, dK, dV from the CUDA path (with
O and LSE from attn_fwd_varlen) against the fp64 oracle, against the single-sequence
backward bit for bit where the order of additions is the same, reproducible when
deterministic, and with offsets that fail the device check."""
import numpy as np
import pytest
import torch

import oracle
from attn_inputs import default_scale, make_varlen_inputs, varlen_workload
from parity import GRAD_REL_FRO, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import attention_attn_fwd_09_gb300 as A
    A.attn_set_debug_knobs()
    A.attn_set_varlen_order(True)
    A.attn_device_status(True)
    yield A
    A.attn_set_varlen_order(True)


CASES = {  # name: (lens_q, lens_k or None for equal, Hq, Hkv, d)
    "ragged_mha_d128": ([1, 127, 128, 129, 300, 257], None, 4, 4, 128),
    "gqa_d64": ([700, 64, 3, 513], None, 8, 2, 64),
    "odd_group_d128": ([333, 129, 640], None, 6, 2, 128),
    "longer_keys_d128": ([100, 0, 300, 40, 1], [229, 50, 301, 40, 130], 4, 2, 128),
}


def _inputs(name):
    lens_q, lens_k, Hq, Hkv, d = CASES[name]
    lens_k = list(lens_q) if lens_k is None else lens_k
    x = make_varlen_inputs(700 + sum(lens_q) % 89 + d, lens_q, lens_k, Hq, Hkv, d)
    x["do"] = make_varlen_inputs(701 + d, lens_q, lens_k, Hq, Hkv, d)["q"]
    return x, default_scale(d)


def _run(A, x, causal, scale, deterministic=False, order=True):
    dev = torch.device("cuda")
    q, k, v, do, cq, ck = (x[n].to(dev) for n in ("q", "k", "v", "do", "cu_q", "cu_k"))
    o, lse = A.attn_fwd_varlen(q, k, v, cq, ck, causal=causal, scale=scale)
    A.attn_set_varlen_order(order)
    dq, dk, dv = A.attn_bwd_varlen(q, k, v, o, lse, do, cq, ck, causal=causal, scale=scale,
                                   deterministic=deterministic)
    torch.cuda.synchronize()
    A.attn_set_varlen_order(True)
    assert A.attn_device_status(True) == 0
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("deterministic", [False, True])
def test_varlen_bwd_matches_oracle(A, name, causal, deterministic):
    x, scale = _inputs(name)
    _, _, dq, dk, dv = _run(A, x, causal, scale, deterministic)
    ref = oracle.attn_bwd_varlen(x["q"], x["k"], x["v"], x["do"], x["cu_q"], x["cu_k"], causal, scale)
    for nm, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        g = g.float().cpu().numpy()
        assert np.isfinite(g).all(), f"{name} {nm}: non-finite"
        e = rel_fro(g, r)
        assert e <= GRAD_REL_FRO, f"{name} causal={causal} det={deterministic} {nm}: rel Frobenius {e:.3e}"


def test_keys_without_queries_get_zero_gradients(A):
    x, scale = _inputs("longer_keys_d128")
    _, _, _, dk, dv = _run(A, x, True, scale)
    ck = x["cu_k"].tolist()
    assert not bool(dk[:, ck[1]:ck[2]].any()) and not bool(dv[:, ck[1]:ck[2]].any())


@pytest.mark.parametrize("name", ["ragged_mha_d128", "gqa_d64", "odd_group_d128"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("deterministic", [False, True])
def test_varlen_bwd_equals_each_sequence_alone(A, name, causal, deterministic):
    # dK and dV: every key block visits the same query tiles in the same order as in a
    # call on its sequence alone, so they agree bit for bit (except deterministic and
    # non-causal, where a short single sequence takes the rotating order and packed ones
    # the shared descending order).  dQ too when the additions are ordered the same way
    # (deterministic and causal: ascending key blocks in both).
    x, scale = _inputs(name)
    o, lse, dq, dk, dv = _run(A, x, causal, scale, deterministic)
    exact_kv = causal or not deterministic
    dev = torch.device("cuda")
    cq = x["cu_q"].tolist()
    for b in range(len(cq) - 1):
        sl = slice(cq[b], cq[b + 1])
        one = lambda t: t[:, sl].unsqueeze(0).contiguous().to(dev)
        rq, rk, rv = A.attn_bwd(one(x["q"]), one(x["k"]), one(x["v"]), one(o), one(lse), one(x["do"]),
                                causal=causal, scale=scale, deterministic=deterministic)
        if exact_kv:
            assert torch.equal(dk[:, sl], rk[0]), f"sequence {b}: dK differs"
            assert torch.equal(dv[:, sl], rv[0]), f"sequence {b}: dV differs"
        else:
            for nm, g, r in (("dK", dk, rk), ("dV", dv, rv)):
                e = rel_fro(g[:, sl].float().cpu().numpy(), r[0].float().cpu().numpy())
                assert e <= 1e-2, f"sequence {b}: {nm} rel Frobenius {e:.3e} against the single-sequence call"
        if deterministic and causal:
            assert torch.equal(dq[:, sl], rq[0]), f"sequence {b}: dQ differs"
        else:
            e = rel_fro(dq[:, sl].float().cpu().numpy(), rq[0].float().cpu().numpy())
            assert e <= 1e-2, f"sequence {b}: dQ rel Frobenius {e:.3e} against the single-sequence call"
    assert A.attn_device_status(True) == 0


@pytest.mark.parametrize("causal", [False, True])
def test_deterministic_runs_are_identical(A, causal):
    x, scale = _inputs("gqa_d64")
    first = _run(A, x, causal, scale, deterministic=True)[2:]
    for _ in range(4):
        again = _run(A, x, causal, scale, deterministic=True)[2:]
        for a, b in zip(first, again):
            assert torch.equal(a, b)


def test_order_does_not_change_dk_dv(A):
    x, scale = _inputs("ragged_mha_d128")
    a = _run(A, x, True, scale, deterministic=True, order=True)[2:]
    b = _run(A, x, True, scale, deterministic=True, order=False)[2:]
    for u, w in zip(a, b):
        assert torch.equal(u, w)


def test_bad_offsets_fail_the_device_check(A):
    x = make_varlen_inputs(750, [200, 100], [200, 100], 2, 2, 64)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = q.clone()
    lse = torch.zeros((2, 300), dtype=torch.float32, device=dev)
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(v, 7.0)
    for cu in ([0, 250, 200, 300], [0, 100, 290], [5, 100, 300]):
        c = torch.tensor(cu, dtype=torch.int32, device=dev)
        A.attn_bwd_varlen(q, k, v, o, lse, q, c, c, causal=False, scale=0.125, dk=dk, dv=dv)
        assert A.attn_device_status(True) == -1, cu
        assert bool((dk == 7.0).all()) and bool((dv == 7.0).all()), "dK/dV written despite bad offsets"


@pytest.mark.parametrize("causal", [False, True])
def test_mixed_length_batch_full_size(A, causal):
    # The packed mixed-length batch (65536 tokens, 16 heads, d = 128): dK and dV of every
    # sequence bit for bit against the single-sequence backward, dQ close to it, and the
    # shortest sequence against the oracle.
    w = varlen_workload()
    x = make_varlen_inputs(w["seed"], w["lens"], w["lens"], w["Hq"], w["Hkv"], w["d"])
    x["do"] = make_varlen_inputs(w["seed"] + 1, w["lens"], w["lens"], w["Hq"], w["Hkv"], w["d"])["q"]
    scale = default_scale(w["d"])
    o, lse, dq, dk, dv = _run(A, x, causal, scale)
    dev = torch.device("cuda")
    cq = x["cu_q"].tolist()
    for b in range(len(cq) - 1):
        sl = slice(cq[b], cq[b + 1])
        one = lambda t: t[:, sl].unsqueeze(0).contiguous().to(dev)
        rq, rk, rv = A.attn_bwd(one(x["q"]), one(x["k"]), one(x["v"]), one(o), one(lse), one(x["do"]),
                                causal=causal, scale=scale)
        assert torch.equal(dk[:, sl], rk[0]) and torch.equal(dv[:, sl], rv[0]), f"sequence {b}"
        assert rel_fro(dq[:, sl].float().cpu().numpy(), rq[0].float().cpu().numpy()) <= 1e-2, f"sequence {b}"
    b = int(np.argmin(w["lens"]))
    sl = slice(cq[b], cq[b + 1])
    cu = torch.tensor([0, w["lens"][b]], dtype=torch.int32)
    part = lambda t: t[:, sl].contiguous()
    ref = oracle.attn_bwd_varlen(part(x["q"]), part(x["k"]), part(x["v"]), part(x["do"]), cu, cu, causal, scale)
    for nm, g, r in zip(("dq", "dk", "dv"), (dq[:, sl], dk[:, sl], dv[:, sl]), ref):
        e = rel_fro(g.float().cpu().numpy(), r)
        assert e <= GRAD_REL_FRO, f"sequence {b} {nm}: rel Frobenius {e:.3e}"
