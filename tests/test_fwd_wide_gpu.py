"""Forward parity for wide heads (d = 192 and 256, the one-tile kernel): the CUDA path
against the fp64 oracle element by element, including ragged lengths, grouped heads,
causal masks, queries after a longer key cache, and the outlier inputs that make the
running maximum jump (conditional rescale)."""
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


SHAPES = [  # B, Hq, Hkv, N, d
    (1, 2, 2, 256, 256),
    (1, 2, 1, 300, 192),
    (2, 4, 2, 129, 256),     # grouped heads, one row past a tile
    (1, 3, 3, 1000, 192),    # ragged, 8 key blocks
    (1, 2, 2, 1, 256),       # a single query
    (1, 4, 1, 513, 256),     # multi-query
    (1, 2, 2, 2048, 256),    # 16 key blocks: both S buffers and the whole ring cycle many times
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dHq%dHkv%dN%dd%d" % s)
@pytest.mark.parametrize("causal", [False, True])
def test_wide_shapes(A, shape, causal):
    B, Hq, Hkv, N, d = shape
    x = make_inputs(800 + N + d, B, Hq, Hkv, N, d)
    scale = default_scale(d)
    dev = torch.device("cuda")
    o, lse = A.attn_fwd(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert A.attn_device_status(True) == 0
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, scale)
    check_fwd(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, f"{shape} causal={causal}")


@pytest.mark.parametrize("d", [192, 256])
def test_wide_outliers_rescale(A, d):
    # Outlier scores move the running maximum by far more than tau between key blocks.
    B, H, N = 1, 2, 1024
    x = make_inputs(850 + d, B, H, H, N, d, recipe="outliers")
    scale = default_scale(d)
    dev = torch.device("cuda")
    A.attn_rescale_counter(True)
    o, lse = A.attn_fwd(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), causal=True, scale=scale)
    torch.cuda.synchronize()
    rescales = A.attn_rescale_counter(False)
    assert A.attn_device_status(True) == 0
    assert rescales > 0
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], True, scale)
    check_fwd(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, f"outliers d={d}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [192, 256])
def test_wide_queries_after_cache(A, causal, d):
    B, Hq, Hkv, Nq, Nk = 1, 4, 2, 100, 700
    x = make_inputs(870 + d, B, Hq, Hkv, Nk, d)
    q = x["q"][:, :, Nk - Nq:].contiguous()
    scale = default_scale(d)
    dev = torch.device("cuda")
    o, lse = A.attn_fwd_kv(q.to(dev), x["k"].to(dev), x["v"].to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert A.attn_device_status(True) == 0
    O, L = oracle.attn_fwd_kv(q, x["k"], x["v"], causal, scale)
    check_fwd(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, f"kv d={d} causal={causal}")


def test_wide_full_size_sampled(A):
    # The benchmark's wide shape (B=2, H=16, N=8192, d=256, causal): sampled heads against
    # the oracle, every LSE finite.
    B, H, N, d = 2, 16, 8192, 256
    x = make_inputs(880, B, H, H, N, d)
    q, k, v = x["q"], x["k"], x["v"]
    dev = torch.device("cuda")
    o, lse = A.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True, scale=default_scale(d))
    torch.cuda.synchronize()
    assert A.attn_device_status(True) == 0
    assert bool(torch.isfinite(lse).all())
    heads = [(0, 0), (1, 9)]
    O, L = oracle.attn_fwd(q, k, v, True, default_scale(d), heads=heads)
    got_o = np.stack([o[b, h].float().cpu().numpy() for b, h in heads])
    got_l = np.stack([lse[b, h].cpu().numpy() for b, h in heads])
    check_fwd(got_o, got_l, O, L, "B2 H16 N8192 d256 causal (sampled heads)")
