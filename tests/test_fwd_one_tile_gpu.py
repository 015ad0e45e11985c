"""Forward parity for d = 128 through the one-tile kernel (one query tile per CTA, the
softmax of each key block split over two warpgroups that exchange their row maxima):
the CUDA path against the fp64 oracle, and against the two-tile kernel."""
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
    A.attn_set_fwd_one_tile(True)
    A.attn_device_status(True)
    yield A
    A.attn_set_fwd_one_tile(False)


def run(A, x, causal, scale):
    dev = torch.device("cuda")
    o, lse = A.attn_fwd(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert A.attn_device_status(True) == 0
    return o, lse


SHAPES = [  # B, Hq, Hkv, N
    (1, 2, 2, 1), (1, 2, 2, 5), (1, 2, 2, 100), (1, 4, 1, 300), (1, 2, 2, 384), (1, 6, 2, 257),
    (2, 4, 2, 1000), (1, 2, 2, 2048),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dHq%dHkv%dN%d" % s)
@pytest.mark.parametrize("causal", [False, True])
def test_one_tile_shapes(A, shape, causal):
    B, Hq, Hkv, N = shape
    x = make_inputs(900 + N + Hq, B, Hq, Hkv, N, 128)
    scale = default_scale(128)
    o, lse = run(A, x, causal, scale)
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, scale)
    check_fwd(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, f"{shape} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_one_tile_outliers(A, causal):
    # Outliers make the maximum sit in either half of a block and jump by more than tau.
    x = make_inputs(950 + causal, 1, 2, 2, 1024, 128, recipe="outliers")
    scale = default_scale(128)
    A.attn_rescale_counter(True)
    o, lse = run(A, x, causal, scale)
    assert A.attn_rescale_counter(False) > 0
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, scale)
    check_fwd(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, f"outliers causal={causal}")


def test_one_tile_agrees_with_two_tile(A):
    # Same probabilities and the same PV products; only the row sums are added in another
    # order, so the outputs agree to a few bf16 ulps.
    x = make_inputs(960, 2, 8, 4, 1500, 128)
    scale = default_scale(128)
    o1, l1 = run(A, x, True, scale)
    A.attn_set_fwd_one_tile(False)
    try:
        o2, l2 = run(A, x, True, scale)
    finally:
        A.attn_set_fwd_one_tile(True)
    d = (o1.float() - o2.float()).abs()
    assert float(d.max()) <= 2 ** -6 * max(1.0, float(o2.float().abs().max()))
    assert float((l1 - l2).abs().max()) <= 1e-5


def test_one_tile_queries_after_cache(A):
    x = make_inputs(970, 1, 4, 2, 700, 128)
    q = x["q"][:, :, 600:].contiguous()
    scale = default_scale(128)
    dev = torch.device("cuda")
    none = torch.empty((0,), dtype=torch.uint8, device=dev)
    o, lse = A.attn_fwd_kv(q.to(dev), x["k"].to(dev), x["v"].to(dev), causal=True, scale=scale, workspace=none)
    torch.cuda.synchronize()
    assert A.attn_device_status(True) == 0
    O, L = oracle.attn_fwd_kv(q, x["k"], x["v"], True, scale)
    check_fwd(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, "kv causal")
