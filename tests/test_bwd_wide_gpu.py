"""Backward parity for wide heads (d = 192, 256): dQ, dK, dV from the CUDA path (through
the C ABI, with O and LSE from the CUDA forward) against the fp64 chain-rule oracle on the
same seeded inputs; rel. Frobenius <= 2e-2 each."""
import hashlib

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import default_scale, make_inputs
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


SHAPES = [  # B, Hq, Hkv, N
    (1, 2, 2, 1), (1, 2, 2, 63), (1, 2, 2, 64), (1, 2, 1, 65), (1, 2, 2, 127), (2, 2, 2, 128), (1, 4, 2, 129),
    (1, 3, 1, 200), (2, 2, 1, 300), (1, 2, 2, 513),
]


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dHq%dHkv%dN%d" % s)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("deterministic", [False, True])
def test_shapes(A, d, shape, causal, deterministic):
    B, Hq, Hkv, N = shape
    x = make_inputs(900 + N + d + Hq, B, Hq, Hkv, N, d, with_grad=True)
    scale = default_scale(d)
    got = run_bwd(A, x, causal, scale, deterministic)
    ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, scale)
    check(got, ref, f"d{d} {shape} causal={causal} det={deterministic}")


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [4096, 8192])
def test_long_sampled_heads(A, d, causal, N):
    B, H = 8192 // N, 8
    x = make_inputs(5, B, H, H, N, d, with_grad=True)
    scale = default_scale(d)
    dq, dk, dv = run_bwd(A, x, causal, scale)
    sel = [(0, 0), (B - 1, H - 1)]
    dQ, dK, dV = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, scale, kv_heads=sel)
    for s, (b, h) in enumerate(sel):
        check((dq[b, h:h + 1], dk[b, h], dv[b, h]), (dQ[s], dK[s], dV[s]), f"d{d} N{N} causal={causal} b{b} h{h}")


def test_grouped_outliers(A):
    # Four query heads per K/V head with the outlier inputs; dK, dV sum over the group.
    B, Hq, Hkv, N, d = 1, 8, 2, 1024, 256
    x = make_inputs(4, B, Hq, Hkv, N, d, recipe="outliers", with_grad=True)
    scale = default_scale(d)
    dq, dk, dv = run_bwd(A, x, True, scale)
    sel = [(0, 1)]
    dQ, dK, dV = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], True, scale, kv_heads=sel)
    check((dq[0, 4:8], dk[0, 1], dv[0, 1]), (dQ[0], dK[0], dV[0]), "d256 gqa outliers")


def _digest(ts):
    h = hashlib.sha256()
    for t in ts:
        h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())
    return h.hexdigest()


@pytest.mark.parametrize("d", [192, 256])
def test_deterministic_bit_identical(A, d):
    B, H, N = 2, 4, 2048
    x = make_inputs(6, B, H, H, N, d, with_grad=True)
    scale = default_scale(d)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = A.attn_fwd(q, k, v, causal=True, scale=scale)
    ws = torch.empty(A.attn_bwd_workspace_size(B, H, H, N, d, True), dtype=torch.uint8, device=dev)
    digests = set()
    for _ in range(10):
        ws.fill_(0xA5)            # workspace contents on entry must not matter
        grads = A.attn_bwd(q, k, v, o, lse, do, causal=True, scale=scale, deterministic=True, workspace=ws)
        torch.cuda.synchronize()
        digests.add(_digest(grads))
    assert A.attn_device_status(True) == 0
    assert len(digests) == 1


def test_outputs_stay_in_bounds(A):
    B, Hq, Hkv, N, d = 1, 2, 1, 200, 192
    x = make_inputs(910, B, Hq, Hkv, N, d, with_grad=True)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = A.attn_fwd(q, k, v, causal=True, scale=0.1)
    bufs = []
    views = []
    for shp in ((B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d)):
        n = int(np.prod(shp))
        buf = torch.full((n + 4096,), -7.0, dtype=torch.bfloat16, device=dev)
        bufs.append((buf, n))
        views.append(buf[:n].view(shp))
    A.attn_bwd(q, k, v, o, lse, do, causal=True, scale=0.1, dq=views[0], dk=views[1], dv=views[2])
    torch.cuda.synchronize()
    for buf, n in bufs:
        assert bool((buf[n:] == -7.0).all())
