"""Forward parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on the
same seeded bf16 inputs, element by element."""
import numpy as np
import pytest
import torch

import oracle
from attn_inputs import WORKLOADS, default_scale, make_inputs, sweep_workload
from parity import check_fwd, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import attention_attn_fwd_09_gb300 as A
    A.attn_set_debug_knobs()
    A.attn_device_status(True)
    yield A
    A.attn_set_debug_knobs()


def run(A, x, causal, scale):
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o, lse = A.attn_fwd(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert A.attn_device_status(True) == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def test_small_workload(A):
    w = WORKLOADS["small"]
    x = make_inputs(w["seed"], w["B"], w["Hq"], w["Hkv"], w["N"], w["d"])
    scale = default_scale(w["d"])
    o, lse = run(A, x, False, scale)
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], False, scale)
    check_fwd(o, lse, O, L, "small")


SHAPES = [  # B, Hq, Hkv, N, d
    (1, 2, 2, 1, 64), (1, 2, 2, 5, 128), (1, 2, 2, 100, 128), (2, 4, 2, 129, 64), (1, 4, 1, 300, 128),
    (1, 3, 1, 200, 64), (1, 2, 2, 384, 128), (1, 6, 2, 257, 128), (2, 2, 1, 640, 64),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dHq%dHkv%dN%dd%d" % s)
@pytest.mark.parametrize("causal", [False, True])
def test_shapes_ragged_grouped(A, shape, causal):
    B, Hq, Hkv, N, d = shape
    x = make_inputs(100 + N + d + Hq, B, Hq, Hkv, N, d)
    scale = default_scale(d)
    o, lse = run(A, x, causal, scale)
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, scale)
    check_fwd(o, lse, O, L, f"{shape} causal={causal}")


def test_last_wave_one_tile_ctas(A):
    # 2 x 81 heads of N = 256 (two query tiles) are 162 two-tile units.  On GPUs with 132
    # to 152 SMs the last wave holds 10 to 30 of them, which run as one-tile CTAs; the last
    # heads are in that wave and the first ones are not.
    B, H, N, d = 2, 81, 256, 128
    x = make_inputs(55, B, H, H, N, d)
    scale = default_scale(d)
    o, lse = run(A, x, False, scale)
    heads = [(0, 0), (1, 78), (1, 80)]
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], False, scale, heads=heads)
    for s, (b, h) in enumerate(heads):
        check_fwd(o[b, h], lse[b, h], O[s], L[s], f"b{b} h{h}")


@pytest.mark.parametrize("causal", [False, True])
def test_train_workload_heads(A, causal):
    w = WORKLOADS["train2k"]
    x = make_inputs(w["seed"], w["B"], w["Hq"], w["Hkv"], w["N"], w["d"])
    scale = default_scale(w["d"])
    o, lse = run(A, x, causal, scale)
    heads = [(0, 0), (1, 7), (3, 15)]
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, scale, heads=heads)
    for s, (b, h) in enumerate(heads):
        check_fwd(o[b, h], lse[b, h], O[s], L[s], f"train2k b{b} h{h}")


@pytest.mark.parametrize("N", [512, 1024, 2048, 4096, 8192, 16384])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_sequence_sweep(A, N, d, causal):
    w = sweep_workload(N, d)
    x = make_inputs(w["seed"], w["B"], w["Hq"], w["Hkv"], w["N"], w["d"])
    scale = default_scale(d)
    o, lse = run(A, x, causal, scale)
    B, H = w["B"], w["Hq"]
    # The first head (first CTAs of the grid) and the last one at every length, so that
    # the first wave and the tail are both compared.
    heads = [(0, 0), (B - 1, H - 1)]
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, scale, heads=heads)
    for s, (b, h) in enumerate(heads):
        check_fwd(o[b, h], lse[b, h], O[s], L[s], f"sweep N{N} d{d} b{b} h{h}")


@pytest.mark.parametrize("name", ["gqa8k", "mqa8k"])
def test_grouped_outliers_rescale(A, name):
    w = WORKLOADS[name]
    x = make_inputs(w["seed"], w["B"], w["Hq"], w["Hkv"], w["N"], w["d"], recipe=w["recipe"])
    scale = default_scale(w["d"])
    g = w["Hq"] // w["Hkv"]
    heads = [(0, 0), (0, 1), (1, w["Hq"] - 1)]        # two heads of one K/V group, and the last head
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], True, scale, heads=heads)
    counts = {}
    outs = {}
    for tau in (0.0, 8.0):
        A.attn_set_debug_knobs(tau=tau)
        A.attn_rescale_counter(True)
        o, lse = run(A, x, True, scale)
        counts[tau] = A.attn_rescale_counter(False)
        outs[tau] = o
        for s, (b, h) in enumerate(heads):
            check_fwd(o[b, h], lse[b, h], O[s], L[s], f"{name} tau={tau} b{b} h{h}")
    A.attn_set_debug_knobs()
    # Both runs meet the forward bounds against the oracle (above).  Against each other,
    # over every head: rel. Frobenius <= 1e-2, and elementwise at most one bf16 ulp of the
    # value (an absolute 2e-2 is below one bf16 ulp once |O| >= 4).
    a, b8 = outs[0.0].astype(np.float64), outs[8.0].astype(np.float64)
    assert rel_fro(a, b8) <= 1e-2
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(a), np.abs(b8)) + 1e-30)) - 7)
    assert (np.abs(a - b8) <= np.maximum(2e-2, ulp)).all(), np.abs(a - b8).max()
    assert counts[8.0] < counts[0.0], counts
    print(f"{name}: rescales tau=0 {counts[0.0]}, tau=8 {counts[8.0]} "
          f"({100.0 * (1 - counts[8.0] / max(counts[0.0], 1)):.1f}% skipped), g={g}")


@pytest.mark.parametrize("poly", [0, 4, 16])
@pytest.mark.parametrize("d", [64, 128])
def test_poly_fraction(A, poly, d):
    x = make_inputs(200 + poly + d, 2, 4, 2, 1000, d)
    scale = default_scale(d)
    A.attn_set_debug_knobs(poly_per_16=poly)
    try:
        for causal in (False, True):
            o, lse = run(A, x, causal, scale)
            O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, scale)
            check_fwd(o, lse, O, L, f"poly={poly} d={d} causal={causal}")
    finally:
        A.attn_set_debug_knobs()


def test_outputs_stay_in_bounds(A):
    # Canary: a ragged problem written into the front of larger buffers leaves the tail alone.
    B, Hq, Hkv, N, d = 1, 2, 1, 200, 128
    x = make_inputs(300, B, Hq, Hkv, N, d)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    n_o = B * Hq * N * d
    o_buf = torch.full((n_o + 4096,), -7.0, dtype=torch.bfloat16, device=dev)
    l_buf = torch.full((B * Hq * N + 1024,), -7.0, dtype=torch.float32, device=dev)
    o = o_buf[:n_o].view(B, Hq, N, d)
    lse = l_buf[:B * Hq * N].view(B, Hq, N)
    A.attn_fwd(q, k, v, causal=True, scale=0.1, o=o, lse=lse)
    torch.cuda.synchronize()
    assert bool((o_buf[n_o:] == -7.0).all())
    assert bool((l_buf[B * Hq * N:] == -7.0).all())


def test_repeatable(A):
    x = make_inputs(400, 1, 4, 4, 700, 128)
    a = run(A, x, True, 0.1)
    b = run(A, x, True, 0.1)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bounded_wait_gives_up_cleanly(A):
    # The load warp never issues the first K tile: the MMA warp's wait runs out after the
    # (short) limit, every role of the CTA stops, TMEM is freed, and the status word says
    # so.  The next normal call must then work on the same context.
    x = make_inputs(500, 1, 2, 2, 512, 128)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    A.attn_device_status(True)
    A.attn_set_debug_knobs(wait_limit_ns=20_000_000)
    A.attn_set_test_hooks(True)
    try:
        A.attn_fwd(q, k, v, causal=False, scale=0.1)
        torch.cuda.synchronize()
        assert A.attn_device_status(True) == -6
    finally:
        A.attn_set_test_hooks(False)
        A.attn_set_debug_knobs()
    o, lse = run(A, x, False, 0.1)
    O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], False, 0.1)
    check_fwd(o, lse, O, L, "after timeout")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_single_key_is_exact(A, d, causal):
    # With one key every probability is exactly 1, so O must be V bit for bit (any error
    # in the row maximum or the normaliser shows up as a one-ulp change) and LSE the score.
    B, Hq, Hkv = 2, 4, 2
    x = make_inputs(600 + d, B, Hq, Hkv, 1, d)
    scale = default_scale(d)
    o, lse = run(A, x, causal, scale)
    v = x["v"].float().numpy().repeat(Hq // Hkv, axis=1)
    assert np.array_equal(o, v)
    s = (x["q"].double() * x["k"].double().repeat_interleave(Hq // Hkv, dim=1)).sum(-1).numpy() * scale
    np.testing.assert_allclose(lse, s, rtol=0, atol=1e-5)
