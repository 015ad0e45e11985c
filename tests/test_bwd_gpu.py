"""Backward parity: dQ, dK, dV from the CUDA path (through the C ABI, with O and LSE
from the CUDA forward) against the fp64 chain-rule oracle on the same seeded inputs."""
import hashlib

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import WORKLOADS, default_scale, long_bwd_workload, make_inputs
from parity import GRAD_REL_FRO, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import attention_attn_fwd_09_gb300 as A
    A.attn_set_debug_knobs()
    A.attn_device_status(True)
    return A


def run_bwd(A, x, causal, scale, deterministic=False):
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = A.attn_fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = A.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale, deterministic=deterministic)
    torch.cuda.synchronize()
    assert A.attn_device_status(True) == 0
    return dq.float().cpu().numpy(), dk.float().cpu().numpy(), dv.float().cpu().numpy()


def check(got, ref, what):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.isfinite(g).all(), f"{what} {name}: non-finite"
        e = rel_fro(g, r)
        assert e <= GRAD_REL_FRO, f"{what} {name}: rel Frobenius {e:.3e}"


SHAPES = [(1, 2, 2, 128, 64), (1, 2, 2, 200, 128), (1, 4, 2, 256, 128), (1, 4, 1, 300, 64), (2, 2, 2, 1, 128),
          (1, 3, 1, 130, 128), (2, 2, 1, 512, 64),
          # one row short of, one past, and one past two whole 128-row tiles
          (1, 2, 2, 127, 128), (1, 2, 1, 129, 64), (1, 2, 2, 257, 128)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dHq%dHkv%dN%dd%d" % s)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("deterministic", [False, True])
def test_shapes(A, shape, causal, deterministic):
    B, Hq, Hkv, N, d = shape
    x = make_inputs(700 + N + d + Hq, B, Hq, Hkv, N, d, with_grad=True)
    scale = default_scale(d)
    got = run_bwd(A, x, causal, scale, deterministic)
    ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, scale)
    check(got, ref, f"{shape} causal={causal} det={deterministic}")


@pytest.mark.parametrize("causal", [False, True])
def test_train_workload(A, causal):
    w = WORKLOADS["train2k"]
    x = make_inputs(w["seed"], w["B"], w["Hq"], w["Hkv"], w["N"], w["d"], with_grad=True)
    scale = default_scale(w["d"])
    dq, dk, dv = run_bwd(A, x, causal, scale)
    sel = [(0, 0), (3, 15)]
    dQ, dK, dV = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, scale, kv_heads=sel)
    for s, (b, h) in enumerate(sel):
        check((dq[b, h:h + 1], dk[b, h], dv[b, h]), (dQ[s], dK[s], dV[s]), f"train2k b{b} h{h}")


@pytest.mark.parametrize("N", [8192, 16384])
@pytest.mark.parametrize("causal", [False, True])
def test_long_atomic_and_deterministic(A, N, causal):
    w = long_bwd_workload(N)
    x = make_inputs(w["seed"], w["B"], w["Hq"], w["Hkv"], w["N"], w["d"], with_grad=True)
    scale = default_scale(w["d"])
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = A.attn_fwd(q, k, v, causal=causal, scale=scale)
    outs = {}
    for det in (False, True):
        dq, dk, dv = A.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale, deterministic=det)
        torch.cuda.synchronize()
        assert A.attn_device_status(True) == 0
        outs[det] = tuple(t.float().cpu().numpy() for t in (dq, dk, dv))
    # The first and the last K/V head: the grid's first CTAs and its tail.
    sel = [(0, 0), (w["B"] - 1, w["Hkv"] - 1)]
    dQ, dK, dV = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, scale, kv_heads=sel)
    for s, (b, h) in enumerate(sel):
        for det in (False, True):
            dq, dk, dv = outs[det]
            check((dq[b, h:h + 1], dk[b, h], dv[b, h]), (dQ[s], dK[s], dV[s]),
                  f"N{N} causal={causal} det={det} b{b} h{h}")
    for i in range(3):   # atomic and ordered accumulation agree everywhere
        assert rel_fro(outs[True][i], outs[False][i]) <= GRAD_REL_FRO


def _digest(ts):
    h = hashlib.sha256()
    for t in ts:
        h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())
    return h.hexdigest()


@pytest.mark.parametrize("causal", [False, True])
def test_deterministic_bit_identical(A, causal):
    w = long_bwd_workload(8192)
    x = make_inputs(w["seed"], w["B"], w["Hq"], w["Hkv"], w["N"], w["d"], with_grad=True)
    scale = default_scale(w["d"])
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = A.attn_fwd(q, k, v, causal=causal, scale=scale)
    ws = torch.empty(A.attn_bwd_workspace_size(w["B"], w["Hq"], w["Hkv"], w["N"], w["d"], True),
                     dtype=torch.uint8, device=dev)
    digests = set()
    for _ in range(10):
        ws.fill_(0xA5)            # workspace contents on entry must not matter
        grads = A.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale, deterministic=True, workspace=ws)
        torch.cuda.synchronize()
        digests.add(_digest(grads))
    assert A.attn_device_status(True) == 0
    assert len(digests) == 1


@pytest.mark.parametrize("shape", [(1, 4, 4, 16384), (1, 8, 2, 4096)], ids=["shared_order_N16384", "gqa_N4096"])
def test_deterministic_other_orders(A, shape):
    # Non-causal at N = 16384 (128 key blocks per head, more than half the SMs): one shared
    # tile order per head, contributions split into two classes.  Grouped heads at N = 4096:
    # the rotating order walks each of a K/V head's query heads in turn.  Both repeat bit for
    # bit and agree with the atomic order.
    B, Hq, Hkv, N = shape
    d = 128
    x = make_inputs(77 + N, B, Hq, Hkv, N, d, with_grad=True)
    scale = default_scale(d)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = A.attn_fwd(q, k, v, causal=False, scale=scale)
    ws = torch.empty(A.attn_bwd_workspace_size(B, Hq, Hkv, N, d, True), dtype=torch.uint8, device=dev)
    digests = set()
    for _ in range(3):
        ws.fill_(0x5A)
        grads = A.attn_bwd(q, k, v, o, lse, do, causal=False, scale=scale, deterministic=True, workspace=ws)
        torch.cuda.synchronize()
        digests.add(_digest(grads))
    atomic = A.attn_bwd(q, k, v, o, lse, do, causal=False, scale=scale, deterministic=False)
    torch.cuda.synchronize()
    assert A.attn_device_status(True) == 0
    assert len(digests) == 1
    for g, a in zip(grads, atomic):
        assert rel_fro(g.float().cpu().numpy(), a.float().cpu().numpy()) <= GRAD_REL_FRO


@pytest.mark.parametrize("deterministic", [False, True])
def test_inputs_written_just_before(A, deterministic):
    # The backward's kernels are launched as programmatic dependents, and the main kernel
    # starts loading Q, K, V and dO before it waits on the kernel before it: inputs written by
    # the stream's previous kernels, with no synchronisation in between, must still be seen.
    B, H, N, d = 2, 4, 1024, 128
    x = make_inputs(88, B, H, H, N, d, with_grad=True)
    scale = default_scale(d)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = A.attn_fwd(q, k, v, causal=False, scale=scale)
    ref = [t.clone() for t in A.attn_bwd(q, k, v, o, lse, do, causal=False, scale=scale, deterministic=True)]
    saved = [t.clone() for t in (q, k, v, do)]
    torch.cuda.synchronize()
    for _ in range(3):
        for t in (q, k, v, do):
            t.zero_()
        torch.cuda.synchronize()
        for t, src in zip((q, k, v, do), saved):
            t.copy_(src)                       # kernels immediately ahead of the backward
        got = A.attn_bwd(q, k, v, o, lse, do, causal=False, scale=scale, deterministic=deterministic)
        torch.cuda.synchronize()
        if deterministic:
            assert all(torch.equal(g, r) for g, r in zip(got, ref))
        else:
            for g, r in zip(got, ref):
                assert rel_fro(g.float().cpu().numpy(), r.float().cpu().numpy()) <= 1e-3
    assert A.attn_device_status(True) == 0


def test_grouped_long(A):
    # GQA group of 4 sharing each K/V head; dK/dV sum over the group inside one CTA.
    w = WORKLOADS["gqa8k"]
    B, Hq, Hkv, N, d = 1, 8, 2, 2048, 128
    x = make_inputs(w["seed"], B, Hq, Hkv, N, d, recipe=w["recipe"], with_grad=True)
    scale = default_scale(d)
    dq, dk, dv = run_bwd(A, x, True, scale)
    sel = [(0, 1)]
    dQ, dK, dV = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], True, scale, kv_heads=sel)
    check((dq[0, 4:8], dk[0, 1], dv[0, 1]), (dQ[0], dK[0], dV[0]), "gqa group")
