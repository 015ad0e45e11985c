"""Forward parity with Nq queries after a cache of Nk >= Nq keys (attn_fwd_kv): the CUDA
path against the fp64 oracle's bottom-right-aligned definition, element by element."""
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
    A.attn_device_status(True)
    yield A


SHAPES = [  # B, Hq, Hkv, Nq, Nk, d
    (1, 2, 2, 1, 300, 128),      # one new token against a cache
    (2, 4, 1, 16, 1000, 64),     # a few tokens, multi-query
    (1, 8, 2, 128, 640, 128),    # one query tile, grouped heads (pairs share K/V)
    (1, 4, 4, 200, 333, 128),    # ragged on both sides
    (2, 2, 2, 257, 257, 64),     # the square case through the same entry point
    (1, 2, 1, 130, 4096, 128),   # long cache
    # grouped decode: the g query heads x Nq queries of a group packed into one tile,
    # keys split over CTAs
    (2, 8, 2, 1, 5000, 128),     # one token, g = 4
    (1, 32, 8, 4, 2048, 128),    # 16 rows per tile
    (1, 16, 1, 8, 1000, 64),     # multi-query: exactly 128 rows
    (1, 8, 1, 15, 777, 128),     # 120 rows, ragged cache
    (3, 6, 3, 3, 130, 128),      # g = 2, two key blocks
    (1, 9, 3, 5, 500, 128),      # g = 3, 15 rows
    (2, 5, 1, 7, 333, 64),       # odd g = 5, 35 rows
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dHq%dHkv%dNq%dNk%dd%d" % s)
@pytest.mark.parametrize("causal", [False, True])
def test_kv_shapes(A, shape, causal):
    B, Hq, Hkv, Nq, Nk, d = shape
    x = make_inputs(500 + Nq + Nk + d, B, Hq, Hkv, Nk, d)
    q = x["q"][:, :, Nk - Nq:].contiguous()
    scale = default_scale(d)
    dev = torch.device("cuda")
    o, lse = A.attn_fwd_kv(q.to(dev), x["k"].to(dev), x["v"].to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert A.attn_device_status(True) == 0
    O, L = oracle.attn_fwd_kv(q, x["k"], x["v"], causal, scale)
    check_fwd(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, f"{shape} causal={causal}")


def test_kv_square_equals_attn_fwd(A):
    B, H, N, d = 1, 4, 300, 128
    x = make_inputs(561, B, H, H, N, d)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    for causal in (False, True):
        o1, l1 = A.attn_fwd(q, k, v, causal=causal)
        o2, l2 = A.attn_fwd_kv(q, k, v, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_decode_matches_ordinary_tiling(A, causal):
    # The packed, key-split path and the ordinary tiling (no workspace) agree.
    B, Hq, Hkv, Nq, Nk, d = 2, 16, 4, 4, 3000, 128
    x = make_inputs(570, B, Hq, Hkv, Nk, d)
    dev = torch.device("cuda")
    q = x["q"][:, :, Nk - Nq:].contiguous().to(dev)
    k, v = x["k"].to(dev), x["v"].to(dev)
    assert A.attn_fwd_kv_workspace_size(B, Hq, Hkv, Nq, Nk, d) > 0
    o1, l1 = A.attn_fwd_kv(q, k, v, causal=causal)
    o2, l2 = A.attn_fwd_kv(q, k, v, causal=causal, workspace=torch.empty(0, dtype=torch.uint8, device=dev))
    torch.cuda.synchronize()
    assert A.attn_device_status(True) == 0
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


GROUPED = [s for s in SHAPES if s[2] < s[1] and s[1] // s[2] * s[3] <= 128]


@pytest.mark.parametrize("shape", GROUPED, ids=lambda s: "B%dHq%dHkv%dNq%dNk%dd%d" % s)
@pytest.mark.parametrize("causal", [False, True])
def test_grouped_decode_two_tile_kernel(A, shape, causal):
    # The grouped decode through the two-tile kernel (the one-tile kernel serves d = 128 by
    # default; d = 64 always takes this path) against the oracle.
    B, Hq, Hkv, Nq, Nk, d = shape
    x = make_inputs(500 + Nq + Nk + d, B, Hq, Hkv, Nk, d)
    q = x["q"][:, :, Nk - Nq:].contiguous()
    scale = default_scale(d)
    dev = torch.device("cuda")
    A.attn_set_decode_one_tile(False)
    try:
        o, lse = A.attn_fwd_kv(q.to(dev), x["k"].to(dev), x["v"].to(dev), causal=causal, scale=scale)
        torch.cuda.synchronize()
    finally:
        A.attn_set_decode_one_tile(True)
    assert A.attn_device_status(True) == 0
    O, L = oracle.attn_fwd_kv(q, x["k"], x["v"], causal, scale)
    check_fwd(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, f"two-tile {shape} causal={causal}")


# Larger grouped-decode shapes, compared in full: 40 groups of 10 key blocks, 4 groups of 71
# blocks with 16 queries each, and the decode benchmark's B8 Hq32 Hkv8 Nk8192.
LARGER = [  # B, Hq, Hkv, Nq, Nk, d
    (5, 32, 8, 1, 1280, 128),
    (2, 8, 2, 16, 9000, 128),
    (8, 32, 8, 1, 8192, 128),
]


@pytest.mark.parametrize("shape", LARGER, ids=lambda s: "B%dHq%dHkv%dNq%dNk%dd%d" % s)
@pytest.mark.parametrize("causal", [False, True])
def test_grouped_decode_larger(A, shape, causal):
    B, Hq, Hkv, Nq, Nk, d = shape
    x = make_inputs(640 + Nq + Nk, B, Hq, Hkv, Nk, d)
    q = x["q"][:, :, Nk - Nq:].contiguous()
    scale = default_scale(d)
    dev = torch.device("cuda")
    assert A.attn_fwd_kv_workspace_size(B, Hq, Hkv, Nq, Nk, d) > 0
    o, lse = A.attn_fwd_kv(q.to(dev), x["k"].to(dev), x["v"].to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert A.attn_device_status(True) == 0
    O, L = oracle.attn_fwd_kv(q, x["k"], x["v"], causal, scale)
    check_fwd(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, f"larger {shape} causal={causal}")
