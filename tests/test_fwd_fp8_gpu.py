"""FP8 forward parity: the quantiser bit for bit against the oracle's, and the FP8 forward
(through the C ABI) against the fp64 attention of the dequantised inputs, element by
element, with the forward's tolerances (O max-abs 2e-2, rel. Frobenius 1e-2, LSE 1e-3).

Inputs: seeded bf16 tensors from attn_inputs, quantised on the CPU by the oracle's
quantiser; the GPU forward and the oracle read the same codes and scales."""
import numpy as np
import pytest
import torch

from attn_inputs import default_scale, make_inputs
from oracle import fp8 as ofp8
from parity import check_fwd, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import attention_attn_fwd_09_gb300 as A
    A.attn_set_debug_knobs()
    A.attn_device_status(True)
    yield A
    A.attn_set_debug_knobs()


def _quantised(x):
    """CPU-quantised codes and scales of each of q, k, v (the oracle's quantiser)."""
    return {n: ofp8.quantize(x[n]) for n in ("q", "k", "v")}


def _run(A, qz, causal, scale):
    dev = torch.device("cuda")
    t = {n: (torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev)) for n, (c, s) in qz.items()}
    o, lse = A.attn_fwd_fp8(t["q"][0], t["k"][0], t["v"][0], t["q"][1], t["k"][1], t["v"][1], causal=causal,
                            scale=scale)
    torch.cuda.synchronize()
    assert A.attn_device_status(True) == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _oracle(qz, causal, scale, heads=None):
    """fp64 attention of the dequantised inputs; with ``heads`` only those (b, hq) (their
    K/V heads are sliced out first so that only what is needed is dequantised)."""
    (q8, sq), (k8, sk), (v8, sv) = qz["q"], qz["k"], qz["v"]
    if heads is None:
        return ofp8.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal, scale)
    g = q8.shape[1] // k8.shape[1]
    O, L = [], []
    for b, h in heads:
        o, l = ofp8.attn_fwd_fp8(q8[b:b + 1, h:h + 1], k8[b:b + 1, h // g:h // g + 1], v8[b:b + 1, h // g:h // g + 1],
                                 sq[b:b + 1, h:h + 1], sk[b:b + 1, h // g:h // g + 1], sv[b:b + 1, h // g:h // g + 1],
                                 causal, scale)
        O.append(o[0, 0])
        L.append(l[0, 0])
    return np.stack(O), np.stack(L)


QSHAPES = [(1, 2, 1), (2, 3, 100), (1, 2, 128), (2, 2, 300), (1, 1, 1000)]


@pytest.mark.parametrize("shape", QSHAPES, ids=lambda s: "B%dH%dN%d" % s)
@pytest.mark.parametrize("recipe", ["normal", "outliers"])
def test_quantiser_bit_exact(A, shape, recipe):
    B, H, N = shape
    x = make_inputs(40 + N, B, H, H, N, 128, recipe=recipe)["q"]
    if B > 1:
        x[1, 0] = 0                                   # an all-zero head: scale 1, codes 0
    codes, scales = ofp8.quantize(x)
    x8, s = A.attn_quantize_fp8(x.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy(), scales)
    assert np.array_equal(x8.cpu().numpy(), codes)


SHAPES = [  # B, Hq, Hkv, N
    (1, 2, 2, 1), (1, 2, 2, 100), (2, 4, 2, 129), (1, 4, 1, 300), (1, 3, 1, 200), (1, 6, 2, 257), (2, 2, 1, 640),
    (1, 2, 2, 384),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dHq%dHkv%dN%d" % s)
@pytest.mark.parametrize("causal", [False, True])
def test_shapes_ragged_grouped(A, shape, causal):
    B, Hq, Hkv, N = shape
    x = make_inputs(800 + N + Hq, B, Hq, Hkv, N, 128)
    qz = _quantised(x)
    scale = default_scale(128)
    o, lse = _run(A, qz, causal, scale)
    O, L = _oracle(qz, causal, scale)
    check_fwd(o, lse, O, L, f"fp8 {shape} causal={causal}")


def test_last_wave_one_tile_ctas(A):
    # 2 x 81 heads of N = 256: 162 two-tile units, the last wave's split into one-tile CTAs.
    B, H, N = 2, 81, 256
    x = make_inputs(855, B, H, H, N, 128)
    qz = _quantised(x)
    scale = default_scale(128)
    o, lse = _run(A, qz, False, scale)
    heads = [(0, 0), (1, 78), (1, 80)]
    O, L = _oracle(qz, False, scale, heads)
    for s, (b, h) in enumerate(heads):
        check_fwd(o[b, h], lse[b, h], O[s], L[s], f"fp8 b{b} h{h}")


@pytest.mark.parametrize("N", [2048, 8192, 16384])
@pytest.mark.parametrize("causal", [False, True])
def test_long_sampled_heads(A, N, causal):
    B, H = max(1, 16384 // N), 16
    x = make_inputs(3, B, H, H, N, 128)
    qz = _quantised(x)
    scale = default_scale(128)
    o, lse = _run(A, qz, causal, scale)
    heads = [(0, 0), (B - 1, H - 1)]
    O, L = _oracle(qz, causal, scale, heads)
    for s, (b, h) in enumerate(heads):
        check_fwd(o[b, h], lse[b, h], O[s], L[s], f"fp8 N{N} b{b} h{h}")


def test_grouped_outliers_rescale(A):
    # Q, K with large outliers (running maxima jump by far more than 8): tau = 0 and 8 both
    # meet the bounds and agree with each other.
    B, Hq, Hkv, N = 1, 8, 2, 2048
    x = make_inputs(4, B, Hq, Hkv, N, 128, recipe="outliers")
    qz = _quantised(x)
    scale = default_scale(128)
    heads = [(0, 0), (0, 1), (0, Hq - 1)]
    O, L = _oracle(qz, True, scale, heads)
    outs = {}
    for tau in (0.0, 8.0):
        A.attn_set_debug_knobs(tau=tau)
        o, lse = _run(A, qz, True, scale)
        outs[tau] = o
        for s, (b, h) in enumerate(heads):
            check_fwd(o[b, h], lse[b, h], O[s], L[s], f"fp8 outliers tau={tau} h{h}")
    A.attn_set_debug_knobs()
    assert rel_fro(outs[0.0], outs[8.0]) <= 1e-2


def test_repeatable_and_bounded_wait(A):
    x = make_inputs(860, 1, 4, 4, 700, 128)
    qz = _quantised(x)
    a = _run(A, qz, True, 0.1)
    b = _run(A, qz, True, 0.1)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # The load warp never issues the first K tile: the waits run out, the CTAs give up
    # cleanly, the status word says so, and the next call works.
    dev = torch.device("cuda")
    t = {n: (torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev)) for n, (c, s) in qz.items()}
    A.attn_set_debug_knobs(wait_limit_ns=20_000_000)
    A.attn_set_test_hooks(True)
    try:
        A.attn_fwd_fp8(t["q"][0], t["k"][0], t["v"][0], t["q"][1], t["k"][1], t["v"][1], causal=False, scale=0.1)
        torch.cuda.synchronize()
        assert A.attn_device_status(True) == -6
    finally:
        A.attn_set_test_hooks(False)
        A.attn_set_debug_knobs()
    c = _run(A, qz, True, 0.1)
    assert np.array_equal(a[0], c[0])


def test_outputs_stay_in_bounds(A):
    B, Hq, Hkv, N = 1, 2, 1, 200
    x = make_inputs(870, B, Hq, Hkv, N, 128)
    qz = _quantised(x)
    dev = torch.device("cuda")
    t = {n: (torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev)) for n, (c, s) in qz.items()}
    n_o = B * Hq * N * 128
    o_buf = torch.full((n_o + 4096,), -7.0, dtype=torch.bfloat16, device=dev)
    l_buf = torch.full((B * Hq * N + 1024,), -7.0, dtype=torch.float32, device=dev)
    o = o_buf[:n_o].view(B, Hq, N, 128)
    lse = l_buf[:B * Hq * N].view(B, Hq, N)
    A.attn_fwd_fp8(t["q"][0], t["k"][0], t["v"][0], t["q"][1], t["k"][1], t["v"][1], causal=True, scale=0.1,
                   o=o, lse=lse)
    torch.cuda.synchronize()
    assert bool((o_buf[n_o:] == -7.0).all())
    assert bool((l_buf[B * Hq * N:] == -7.0).all())
