"""Software exp2 (FMA-pipe cubic) on the GPU against fp64 exp2.

Bound: max relative error <= 2e-4 over [-127, 0] (the pages only require that a
cubic beat the bf16 quantisation error of 3.9e-3, "Hotelren FA4 summary" section 3.2).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def grid_points():
    # Every 97th fp32 value in [-127, 0], plus all integers and half-integers.
    lo = np.float32(-127.0).view(np.uint32)       # negative floats: larger bit pattern = more negative
    bits = np.arange(0x80000000, int(lo) + 1, 97, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    extra = np.concatenate([np.arange(-127, 1, dtype=np.float32), np.arange(-126.5, 0, 1, dtype=np.float32)])
    return np.concatenate([x, extra, np.float32([0.0, -0.0, -127.0])])


def test_poly_full_range_bound():
    import attention_attn_fwd_09_gb300 as A
    x = grid_points()
    y = A.attn_exp2_sw(torch.from_numpy(x).cuda(), variant=1).cpu().numpy().astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y - ref) / ref
    assert rel.max() <= 2e-4, (rel.max(), x[np.argmax(rel)])
    print(f"full-range poly: max rel err {rel.max():.3e} over {len(x)} points")


def test_poly_production_form():
    import attention_attn_fwd_09_gb300 as A
    x = grid_points()
    x = x[x >= -126.0]
    y = A.attn_exp2_sw(torch.from_numpy(x).cuda(), variant=0).cpu().numpy().astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y - ref) / ref
    assert rel.max() <= 2e-4, rel.max()
    # Masked scores: -inf and anything at or below -127 give exactly +0.
    z = A.attn_exp2_sw(torch.tensor([-np.inf, -127.0, -1000.0], dtype=torch.float32).cuda(), variant=0).cpu()
    assert z.tolist() == [0.0, 0.0, 0.0]
    # The values the stale maximum allows (up to 2^8) stay accurate too.
    xp = np.linspace(0.0, 8.0, 10001, dtype=np.float32)
    yp = A.attn_exp2_sw(torch.from_numpy(xp).cuda(), variant=0).cpu().numpy().astype(np.float64)
    assert (np.abs(yp - np.exp2(xp.astype(np.float64))) / np.exp2(xp.astype(np.float64))).max() <= 2e-4


def test_mufu_reference_point():
    import attention_attn_fwd_09_gb300 as A
    x = np.linspace(-20, 0, 4097, dtype=np.float32)
    y = A.attn_exp2_sw(torch.from_numpy(x).cuda(), variant=2).cpu().numpy().astype(np.float64)
    rel = np.abs(y - np.exp2(x.astype(np.float64))) / np.exp2(x.astype(np.float64))
    assert rel.max() <= 1e-5
