"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds no attention arithmetic: it only draws random tensors and rounds
them to bf16, so that the CUDA path and the CPU oracle see the same bytes.

Workload shapes follow the sizes the FlashAttention-4 pages discuss (head dim 64/128,
tiles of 128, sequence lengths 512..16384, GQA/MQA groups).  The value recipe:

* ``normal``   : every entry i.i.d. N(0, 1), drawn in fp32 by ``torch.randn`` from a
                 CPU ``torch.Generator`` seeded with ``seed``, then rounded to bf16
                 (round-to-nearest-even).  Tensors are drawn in the order Q, K, V, dO.
* ``outliers`` : Q and K are N(0, 3^2) (``randn * 3``); then exactly
                 ``round(0.001 * numel)`` positions of each, chosen without
                 replacement, are set to +20 or -20 with equal probability.  This makes
                 the running row maximum jump by far more than 8 (log2 units) between
                 key tiles, which exercises the conditional rescale.  V and dO stay N(0, 1).
"""
from __future__ import annotations

import math

import torch


def _outlier_fill(t: torch.Tensor, g: torch.Generator) -> torch.Tensor:
    flat = t.reshape(-1)
    n_out = int(round(0.001 * flat.numel()))
    if n_out:
        idx = torch.randperm(flat.numel(), generator=g)[:n_out]
        sign = torch.randint(0, 2, (n_out,), generator=g).to(torch.float32) * 2.0 - 1.0
        flat[idx] = 20.0 * sign
    return t


def make_inputs(seed: int, B: int, Hq: int, Hkv: int, N: int, d: int, *,
                recipe: str = "normal", with_grad: bool = False) -> dict:
    """Return CPU bf16 tensors ``q [B,Hq,N,d]``, ``k``/``v [B,Hkv,N,d]`` and, when
    ``with_grad``, ``do [B,Hq,N,d]``.  Same seed and shape give the same bytes."""
    if recipe not in ("normal", "outliers"):
        raise ValueError(f"unknown recipe {recipe!r}")
    g = torch.Generator().manual_seed(int(seed))
    qs, ks = (B, Hq, N, d), (B, Hkv, N, d)
    sigma = 3.0 if recipe == "outliers" else 1.0
    q = torch.randn(qs, generator=g, dtype=torch.float32) * sigma
    k = torch.randn(ks, generator=g, dtype=torch.float32) * sigma
    if recipe == "outliers":
        q = _outlier_fill(q, g)
        k = _outlier_fill(k, g)
    v = torch.randn(ks, generator=g, dtype=torch.float32)
    out = {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}
    if with_grad:
        out["do"] = torch.randn(qs, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out


def default_scale(d: int) -> float:
    """1/sqrt(d), the softmax scale used by every workload."""
    return 1.0 / math.sqrt(d)


# The workloads (shapes, recipe, seed).  Seeds: 0 for the small case, 2..5 for the rest.
WORKLOADS = {
    "small": dict(seed=0, B=1, Hq=2, Hkv=2, N=256, d=64, recipe="normal", causal=(False,)),
    "train2k": dict(seed=2, B=4, Hq=16, Hkv=16, N=2048, d=128, recipe="normal", causal=(False, True)),
    "gqa8k": dict(seed=4, B=2, Hq=32, Hkv=8, N=8192, d=128, recipe="outliers", causal=(True,)),
    "mqa8k": dict(seed=4, B=2, Hq=32, Hkv=1, N=8192, d=128, recipe="outliers", causal=(True,)),
}


def sweep_workload(N: int, d: int) -> dict:
    """Sequence sweep with 16384 total tokens: B = 16384 / N, 16 heads."""
    return dict(seed=3, B=16384 // N, Hq=16, Hkv=16, N=N, d=d, recipe="normal")


def long_bwd_workload(N: int) -> dict:
    """Backward at length: B=2, 16 heads, d=128."""
    return dict(seed=5, B=2, Hq=16, Hkv=16, N=N, d=128, recipe="normal")


# ------------------------------------------------------------------ packed variable-length inputs
def varlen_lengths(seed: int, total: int, lo: int, hi: int) -> list:
    """Sequence lengths drawn i.i.d. uniform on the integers [lo, hi] (CPU generator seeded
    with ``seed``) until they reach ``total`` tokens; the last length is cut so that the
    lengths sum to exactly ``total``."""
    g = torch.Generator().manual_seed(int(seed))
    lens, acc = [], 0
    while acc < total:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        n = min(n, total - acc)
        lens.append(n)
        acc += n
    return lens


def offsets(lens) -> torch.Tensor:
    """Row offsets [0, l0, l0 + l1, ...] (int32) of sequences packed one after another."""
    out = [0]
    for n in lens:
        out.append(out[-1] + int(n))
    return torch.tensor(out, dtype=torch.int32)


def make_varlen_inputs(seed: int, lens_q, lens_k, Hq: int, Hkv: int, d: int, *, recipe: str = "normal") -> dict:
    """Packed sequences: ``q [Hq, sum(lens_q), d]``, ``k``/``v [Hkv, sum(lens_k), d]`` (CPU
    bf16, drawn as ``make_inputs`` draws them, Q then K then V) and the int32 offsets
    ``cu_q``/``cu_k`` (B + 1 entries each)."""
    if len(lens_q) != len(lens_k):
        raise ValueError("lens_q and lens_k need one entry per sequence")
    tq, tk = sum(int(n) for n in lens_q), sum(int(n) for n in lens_k)
    x = make_inputs(seed, 1, Hq, Hkv, max(tq, tk), d, recipe=recipe)
    return {"q": x["q"][0, :, :tq].contiguous(), "k": x["k"][0, :, :tk].contiguous(),
            "v": x["v"][0, :, :tk].contiguous(), "cu_q": offsets(lens_q), "cu_k": offsets(lens_k)}


def varlen_workload() -> dict:
    """Packed training batch of mixed lengths: 65536 tokens in sequences of 256..8192
    tokens (uniform), 16 heads, d = 128."""
    lens = varlen_lengths(7, 65536, 256, 8192)
    return dict(seed=7, lens=lens, Hq=16, Hkv=16, d=128)
