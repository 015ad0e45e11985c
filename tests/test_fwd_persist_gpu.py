"""The persistent forward (one CTA per SM walking the work list, fwd_persist.cu) against
the per-unit forward bit for bit (same arithmetic per tile), against the fp64 oracle, and
through the bounded-wait abort path."""
import numpy as np
import pytest
import torch

import oracle
from attn_inputs import default_scale, make_inputs
from parity import check_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import attention_attn_fwd_09_gb300 as A
    A.attn_set_debug_knobs()
    A.attn_set_fwd_persistent(False)
    A.attn_device_status(True)
    yield A
    A.attn_set_fwd_persistent(False)


def _fwd(A, q, k, v, causal, scale, persistent):
    A.attn_set_fwd_persistent(persistent)
    try:
        o, lse = A.attn_fwd(q, k, v, causal=causal, scale=scale)
        torch.cuda.synchronize()
    finally:
        A.attn_set_fwd_persistent(False)
    assert A.attn_device_status(True) == 0
    return o, lse


SHAPES = [  # B, Hq, Hkv, N, d: units per CTA from one to many, ragged ends, split last waves
    (1, 2, 2, 100, 128),
    (1, 6, 2, 257, 128),      # grouped heads, pairs
    (2, 3, 3, 1000, 64),      # odd row-tile count (an empty split half)
    (4, 16, 16, 2048, 128),   # the training shape: 512 units, split last wave
    (2, 16, 16, 4096, 128),
    (1, 32, 8, 3000, 128),    # grouped heads, ragged
    (3, 81, 81, 256, 128),    # many short units per CTA
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dHq%dHkv%dN%dd%d" % s)
@pytest.mark.parametrize("causal", [False, True])
def test_persistent_equals_per_unit(A, shape, causal):
    B, Hq, Hkv, N, d = shape
    x = make_inputs(1100 + N + Hq + d, B, Hq, Hkv, N, d)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    scale = default_scale(d)
    o1, l1 = _fwd(A, q, k, v, causal, scale, True)
    o0, l0 = _fwd(A, q, k, v, causal, scale, False)
    assert torch.equal(o1, o0) and torch.equal(l1, l0)


@pytest.mark.parametrize("shape", [(1, 4, 2, 700, 128), (2, 2, 2, 300, 64)], ids=lambda s: "B%dHq%dHkv%dN%dd%d" % s)
@pytest.mark.parametrize("causal", [False, True])
def test_persistent_matches_oracle(A, shape, causal):
    B, Hq, Hkv, N, d = shape
    x = make_inputs(1150 + N + d, B, Hq, Hkv, N, d, recipe="outliers")
    dev = torch.device("cuda")
    scale = default_scale(d)
    o, lse = _fwd(A, x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), causal, scale, True)
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, scale)
    check_fwd(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, f"{shape} causal={causal}")


def test_persistent_queries_after_cache(A):
    x = make_inputs(1170, 1, 8, 2, 900, 128)
    q = x["q"][:, :, 300:].contiguous()
    dev = torch.device("cuda")
    none = torch.empty((0,), dtype=torch.uint8, device=dev)
    args = (q.to(dev), x["k"].to(dev), x["v"].to(dev))
    A.attn_set_fwd_persistent(True)
    try:
        o1, l1 = A.attn_fwd_kv(*args, causal=True, scale=0.1, workspace=none)
    finally:
        A.attn_set_fwd_persistent(False)
    o0, l0 = A.attn_fwd_kv(*args, causal=True, scale=0.1, workspace=none)
    torch.cuda.synchronize()
    assert A.attn_device_status(True) == 0
    assert torch.equal(o1, o0) and torch.equal(l1, l0)


def test_persistent_bounded_wait_gives_up_cleanly(A):
    # The K/V loader never issues the first K tile: the MMA warp's wait runs out, every
    # role of every CTA stops, TMEM is freed, and the status word says so.
    x = make_inputs(1180, 2, 4, 4, 1024, 128)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    A.attn_device_status(True)
    A.attn_set_debug_knobs(wait_limit_ns=20_000_000)
    A.attn_set_test_hooks(True)
    A.attn_set_fwd_persistent(True)
    try:
        A.attn_fwd(q, k, v, causal=False, scale=0.1)
        torch.cuda.synchronize()
        assert A.attn_device_status(True) == -6
    finally:
        A.attn_set_fwd_persistent(False)
        A.attn_set_test_hooks(False)
        A.attn_set_debug_knobs()
    o, lse = _fwd(A, q, k, v, False, 0.1, True)
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], False, 0.1)
    check_fwd(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, "after timeout")
