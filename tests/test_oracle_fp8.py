"""Pins for the FP8 oracle (oracle/fp8.py), on the CPU.

The e4m3 decoder and encoder are checked against PyTorch's own float8_e4m3fn type (a
library implementation of the same format); the block quantiser against scales and codes
computed with torch operations; the fp64 forward on dequantised values against the C
oracle (oracle/attn_oracle.c, pinned separately) on inputs whose dequantised values are
exactly representable in bf16 (power-of-two block scales), so that both see the same
numbers.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def _torch_decode(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def _torch_encode(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours, ref = fp8.e4m3_decode(codes), _torch_decode(codes)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert fp8.e4m3_decode(np.uint8(0x7E)) == 448.0 and fp8.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9


def test_encode_matches_torch():
    rng = np.random.default_rng(0)
    finite = fp8.e4m3_decode(np.arange(0x7F, dtype=np.uint8))          # 0 .. 448
    mids = (finite[:-1] + finite[1:]) / 2                                 # every tie
    mags = np.exp(rng.uniform(np.log(1e-4), np.log(460.0), 20000))
    vals = np.concatenate([finite, mids, mags, rng.uniform(0, 448, 20000), [1e-12, 2.0 ** -10, 3 * 2.0 ** -11]])
    vals = np.concatenate([vals, -vals]).astype(np.float32)
    vals = vals[np.abs(vals) < 464]                                      # torch does not saturate above
    assert np.array_equal(fp8.e4m3_encode(vals), _torch_encode(vals))
    # saturation and round trips
    assert np.array_equal(fp8.e4m3_encode(np.float32([500.0, -1e6, 448.5])), np.uint8([0x7E, 0xFE, 0x7E]))
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes).astype(np.float32)), codes)


@pytest.mark.parametrize("N", [1, 100, 128, 300])
def test_quantize_against_torch_ops(N):
    g = torch.Generator().manual_seed(N)
    x = (torch.randn((2, 3, N, 128), generator=g) * 3).to(torch.bfloat16)
    x[1, 2] = 0                                                          # an all-zero head: scale 1
    codes, scales = fp8.quantize(x)
    xf = x.float()
    nb = (N + 127) // 128
    for blk in range(nb):
        part = xf[:, :, blk * 128:(blk + 1) * 128]
        amax = part.abs().amax(dim=(2, 3))
        s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        assert np.array_equal(scales[:, :, blk], s.numpy())
        want = (part / s[:, :, None, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(codes[:, :, blk * 128:(blk + 1) * 128], want)
    # dequantised values are within half a step of x (relative 2^-4, or 2^-10 * s near 0)
    deq = fp8.dequantize(codes, scales)
    s_rows = np.repeat(scales, 128, axis=2)[:, :, :N, None].astype(np.float64)
    err = np.abs(deq - xf.double().numpy())
    # (the factor 1 + 2^-20 covers x / s being rounded to fp32 before the tie-breaking)
    bound = np.maximum(np.abs(xf.double().numpy()) * 2.0 ** -4, s_rows * 2.0 ** -10) * (1 + 2.0 ** -20)
    assert np.all(err <= bound)


def _pow2_inputs(seed, B, H, N, d):
    """Random finite codes (|value| <= 4) and power-of-two block scales: every dequantised
    value is exactly a bf16 number."""
    rng = np.random.default_rng(seed)
    small = np.array([c for c in range(256) if (c & 0x7F) <= 0x48], dtype=np.uint8)   # |v| <= 4
    codes = rng.choice(small, size=(B, H, N, d)).astype(np.uint8)
    scales = (2.0 ** rng.integers(-3, 3, size=(B, H, (N + 127) // 128))).astype(np.float32)
    return codes, scales


def _as_bf16(codes, scales):
    """The same values through torch: decode by torch's float8 type, scale each 128-row
    block, round to bf16 (exact for these inputs)."""
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).double()
    s = torch.from_numpy(scales).double().repeat_interleave(128, dim=2)[:, :, :codes.shape[2]]
    vals = dec * s[..., None]
    out = vals.to(torch.bfloat16)
    assert torch.equal(out.double(), vals)
    return out


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 2, 130), (2, 4, 2, 257), (1, 3, 1, 64)])
def test_fp8_forward_equals_c_oracle_on_exact_values(shape, causal):
    B, Hq, Hkv, N = shape
    d = 128
    q8, sq = _pow2_inputs(1, B, Hq, N, d)
    k8, sk = _pow2_inputs(2, B, Hkv, N, d)
    v8, sv = _pow2_inputs(3, B, Hkv, N, d)
    scale = d ** -0.5
    O, L = fp8.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal, scale)
    Oc, Lc = oracle.attn_fwd(_as_bf16(q8, sq), _as_bf16(k8, sk), _as_bf16(v8, sv), causal, scale)
    np.testing.assert_allclose(O, Oc, rtol=0, atol=1e-11)
    np.testing.assert_allclose(L, Lc, rtol=0, atol=1e-11)


def test_fp8_forward_head_selection_and_chunking():
    q8, sq = _pow2_inputs(4, 1, 4, 300, 128)
    k8, sk = _pow2_inputs(5, 1, 2, 300, 128)
    v8, sv = _pow2_inputs(6, 1, 2, 300, 128)
    O, L = fp8.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, True, 0.1)
    q, k, v = fp8.dequantize(q8, sq), fp8.dequantize(k8, sk), fp8.dequantize(v8, sv)
    Os, Ls = fp8.attn_fwd_values(q, k, v, True, 0.1, heads=[(0, 3), (0, 0)], row_chunk=7)
    np.testing.assert_allclose(Os[0], O[0, 3], rtol=0, atol=1e-12)
    np.testing.assert_allclose(Ls[1], L[0, 0], rtol=0, atol=1e-12)
