"""CPU oracle for the FP8 forward (e4m3 Q/K/V with per-block scales).  TEST INFRASTRUCTURE
ONLY: imported by the tests, the smoke check and the benchmark's CPU leg, never by the
product path, and it imports nothing from the product path.

The pages name an FP8 forward as the next step ("Hotelren FA4 summary", section 6.3,
future directions: FP8 inputs; the reverse-engineering page's FP8 path) without fixing a
format or a scaling rule.  The reading implemented here (one fp32 scale per block of 128
consecutive rows of one head, the tile the kernels load):

  encoding   e4m3 (OCP FP8 "E4M3FN"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
             bits; exponent field 0 holds the subnormals m * 2^-9; exponent 15 with
             mantissa 7 is NaN; no infinities; largest finite value 448.
  quantise   per block b of 128 rows x d columns of one head:
               amax_b = max |x| over the block,
               s_b    = amax_b / 448 in fp32 (round to nearest), or 1 when amax_b = 0,
               code   = e4m3 nearest to fp32(x / s_b) (ties to the even code; values
                        beyond 448 saturate to +-448).
  dequantise x~ = decode(code) * s_b, exact in fp64.
  forward    the attention definition (oracle/attn_oracle.c) applied to the dequantised
             Q~, K~, V~ in fp64: O = softmax(scale Q~ K~^T [causal]) V~, LSE by rows.

So the FP8 path is compared against the exact attention of the values it was actually given;
the quantisation error itself is a property of the inputs, not of the kernel.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BLOCK_ROWS = 128


def _e4m3_table() -> np.ndarray:
    """Value of each of the 256 codes (fp64; NaN for the two NaN codes), from the format's
    definition: sign, exponent field e (bias 7) and mantissa field m."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = sign * m * 2.0 ** -9
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_TABLE = _e4m3_table()
# The 127 finite non-negative values in increasing order, with their codes 0x00..0x7E.
_POS_VALUES = _TABLE[:0x7F]
_POS_CODES = np.arange(0x7F, dtype=np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    """uint8 codes -> fp64 values."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x) -> np.ndarray:
    """fp32 values -> e4m3 codes, round to nearest with ties to the even code, saturating
    at +-448 (finite inputs only).  A brute-force search over the 127 non-negative finite
    values: the candidates just below and just above |x|, the nearer one wins."""
    a = np.abs(np.asarray(x, dtype=np.float32)).astype(np.float64)
    if not np.all(np.isfinite(a)):
        raise ValueError("e4m3_encode: finite inputs only")
    neg = np.signbit(np.asarray(x, dtype=np.float32))
    a = np.minimum(a, E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a, side="left")          # first value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((_POS_CODES[hi] & 1) == 0))
    code = np.where(take_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    # The sign bit follows the input's sign, also when the magnitude rounds to zero (-0).
    return np.where(neg, code | 0x80, code).astype(np.uint8)


def _bf16_to_f32(t) -> np.ndarray:
    """bf16 torch tensor (or uint16 numpy bit patterns) -> fp32 numpy values."""
    if isinstance(t, np.ndarray):
        bits = t.astype(np.uint32)
    else:
        import torch
        assert t.dtype == torch.bfloat16
        bits = t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).astype(np.uint32)
    return (bits << 16).view(np.float32)


def quantize(x):
    """x: bf16 [B, H, N, d] (torch tensor or uint16 bit patterns).  Returns (codes uint8
    [B, H, N, d], scales fp32 [B, H, ceil(N / 128)]) by the block rule in the module
    docstring."""
    xf = _bf16_to_f32(x)
    B, H, N, d = xf.shape
    nb = (N + BLOCK_ROWS - 1) // BLOCK_ROWS
    codes = np.zeros(xf.shape, dtype=np.uint8)
    scales = np.ones((B, H, nb), dtype=np.float32)
    for blk in range(nb):
        r0, r1 = blk * BLOCK_ROWS, min(N, (blk + 1) * BLOCK_ROWS)
        part = xf[:, :, r0:r1, :]
        amax = np.abs(part).max(axis=(2, 3)).astype(np.float32)               # [B, H]
        s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        scales[:, :, blk] = s
        y = (part / s[:, :, None, None]).astype(np.float32)                    # fp32 division
        codes[:, :, r0:r1, :] = e4m3_encode(y)
    return codes, scales


def dequantize(codes, scales) -> np.ndarray:
    """codes uint8 [B, H, N, d], scales fp32 [B, H, ceil(N / 128)] -> fp64 values."""
    codes = np.asarray(codes, dtype=np.uint8)
    B, H, N, d = codes.shape
    s = np.repeat(np.asarray(scales, dtype=np.float64), BLOCK_ROWS, axis=2)[:, :, :N]
    return e4m3_decode(codes) * s[..., None]


def attn_fwd_values(q, k, v, causal: bool, scale: float, heads=None, row_chunk: int = 2048):
    """The attention definition in fp64 on given fp64 values: q [B, Hq, N, d], k/v
    [B, Hkv, N, d]; query head h reads key/value head h / (Hq / Hkv).  Returns (O, LSE)
    for ``heads`` (list of (b, hq); default all) shaped [S, N, d] and [S, N], or
    [B, Hq, N, d] and [B, Hq, N] when ``heads`` is None.  Rows are processed in chunks;
    every row's scores, maximum, exponentials and sums are those of the definition."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    sel = [(b, h) for b in range(B) for h in range(Hq)] if heads is None else list(heads)
    O = np.zeros((len(sel), N, d))
    L = np.zeros((len(sel), N))
    for s_i, (b, h) in enumerate(sel):
        kk, vv = k[b, h // g], v[b, h // g]
        for r0 in range(0, N, row_chunk):
            r1 = min(N, r0 + row_chunk)
            s = scale * (q[b, h, r0:r1] @ kk.T)                         # [rows, N]
            if causal:
                i = np.arange(r0, r1)[:, None]
                j = np.arange(N)[None, :]
                s = np.where(j <= i, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            l = p.sum(axis=1, keepdims=True)
            O[s_i, r0:r1] = (p / l) @ vv
            L[s_i, r0:r1] = (m + np.log(l))[:, 0]
    if heads is None:
        return O.reshape(B, Hq, N, d), L.reshape(B, Hq, N)
    return O, L


def attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal: bool, scale: float, heads=None):
    """fp64 forward of the FP8 inputs: dequantise each operand by its block scales, then
    the attention definition (``attn_fwd_values``)."""
    return attn_fwd_values(dequantize(q8, q_scale), dequantize(k8, k_scale), dequantize(v8, v_scale), causal, scale,
                           heads)
