"""Backward parity at d = 64 and 128 with the 64-row query-tile kernel
(attn_set_bwd_query_tile(64)): dQ, dK, dV against the fp64 chain-rule oracle, rel.
Frobenius <= 2e-2 each; deterministic mode bit-identical over 10 runs."""
import hashlib

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import default_scale, long_bwd_workload, make_inputs
from parity import GRAD_REL_FRO, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import attention_attn_fwd_09_gb300 as A
    A.attn_set_debug_knobs()
    A.attn_device_status(True)
    A.attn_set_bwd_query_tile(64)
    yield A
    A.attn_set_bwd_query_tile(128)


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


SHAPES = [(1, 2, 2, 1), (1, 2, 2, 63), (1, 2, 1, 65), (1, 2, 2, 127), (2, 2, 2, 128), (1, 4, 2, 129),
          (1, 3, 1, 200), (2, 2, 1, 300), (1, 2, 2, 513)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dHq%dHkv%dN%d" % s)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("deterministic", [False, True])
def test_shapes(A, d, shape, causal, deterministic):
    B, Hq, Hkv, N = shape
    x = make_inputs(700 + N + d + Hq, B, Hq, Hkv, N, d, with_grad=True)
    scale = default_scale(d)
    got = run_bwd(A, x, causal, scale, deterministic)
    ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, scale)
    check(got, ref, f"d{d} {shape} causal={causal} det={deterministic}")


@pytest.mark.parametrize("causal", [False, True])
def test_train_and_long(A, causal):
    for B, H, N in ((4, 16, 2048), (2, 16, 8192)):
        w = long_bwd_workload(N) if N == 8192 else dict(seed=2, B=B, Hq=H, Hkv=H, N=N, d=128)
        x = make_inputs(w["seed"], B, H, H, N, 128, with_grad=True)
        scale = default_scale(128)
        for det in (False, True):
            dq, dk, dv = run_bwd(A, x, causal, scale, det)
            sel = [(0, 0), (B - 1, H - 1)]
            dQ, dK, dV = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, scale, kv_heads=sel)
            for s, (b, h) in enumerate(sel):
                check((dq[b, h:h + 1], dk[b, h], dv[b, h]), (dQ[s], dK[s], dV[s]),
                      f"N{N} causal={causal} det={det} b{b} h{h}")


def test_deterministic_bit_identical(A):
    w = long_bwd_workload(8192)
    x = make_inputs(w["seed"], w["B"], w["Hq"], w["Hkv"], w["N"], w["d"], with_grad=True)
    scale = default_scale(w["d"])
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = A.attn_fwd(q, k, v, causal=False, scale=scale)
    ws = torch.empty(A.attn_bwd_workspace_size(w["B"], w["Hq"], w["Hkv"], w["N"], w["d"], True), dtype=torch.uint8,
                     device=dev)
    digests = set()
    for _ in range(10):
        ws.fill_(0xA5)
        grads = A.attn_bwd(q, k, v, o, lse, do, causal=False, scale=scale, deterministic=True, workspace=ws)
        torch.cuda.synchronize()
        h = hashlib.sha256()
        for t in grads:
            h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())
        digests.add(h.hexdigest())
    assert A.attn_device_status(True) == 0
    assert len(digests) == 1
