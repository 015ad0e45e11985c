"""The library's calls are stream-ordered and never synchronise with the host, so a whole
training step (forward and backward, at d = 128 with either query tile and at d = 192 and
256), the packed-sequence pair, the wide-head forward, the FP8 quantiser plus forward and a
grouped decode step can each be captured once in a CUDA graph and replayed: each replay on
new inputs must give, bit for bit, what the eager calls give (deterministic dQ order, so
that the backward is reproducible)."""
import pytest
import torch

from attn_inputs import default_scale, make_inputs, make_varlen_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import attention_attn_fwd_09_gb300 as A
    A.attn_set_debug_knobs()
    A.attn_device_status(True)
    yield A


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                                   # warm-up outside the graph (one-time setup)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_training_step_graph(A):
    B, H, N, d = 2, 4, 640, 128
    dev = torch.device("cuda")
    scale = default_scale(d)
    x0 = make_inputs(1000, B, H, H, N, d, with_grad=True)
    q, k, v, do = (x0[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty((A.attn_bwd_workspace_size(B, H, H, N, d, True),), dtype=torch.uint8, device=dev)

    def step():
        A.attn_fwd(q, k, v, causal=True, scale=scale, o=o, lse=lse)
        A.attn_bwd(q, k, v, o, lse, do, causal=True, scale=scale, deterministic=True, dq=dq, dk=dk, dv=dv,
                   workspace=ws)

    g = _capture(step)
    for seed in (1001, 1002):
        x = make_inputs(seed, B, H, H, N, d, with_grad=True)
        for t, nm in ((q, "q"), (k, "k"), (v, "v"), (do, "do")):
            t.copy_(x[nm].to(dev))
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (o, lse, dq, dk, dv)]
        step()
        torch.cuda.synchronize()
        for a, b in zip(got, (o, lse, dq, dk, dv)):
            assert torch.equal(a, b)
    assert A.attn_device_status(True) == 0


def test_packed_sequences_graph(A):
    lens = [300, 17, 129, 512]
    Hq, Hkv, d = 4, 2, 128
    dev = torch.device("cuda")
    scale = default_scale(d)
    x0 = make_varlen_inputs(1010, lens, lens, Hq, Hkv, d)
    q, k, v, cq, ck = (x0[n].to(dev) for n in ("q", "k", "v", "cu_q", "cu_k"))
    do = torch.zeros_like(q)
    o, lse = torch.empty_like(q), torch.empty((Hq, q.shape[1]), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    T = q.shape[1]
    wf = torch.empty((A.attn_fwd_varlen_workspace_size(len(lens), Hq, Hkv, T, d),), dtype=torch.uint8, device=dev)
    wb = torch.empty((A.attn_bwd_varlen_workspace_size(len(lens), Hq, Hkv, T, T, d, True),), dtype=torch.uint8,
                     device=dev)

    def step():
        A.attn_fwd_varlen(q, k, v, cq, ck, causal=True, scale=scale, o=o, lse=lse, workspace=wf)
        A.attn_bwd_varlen(q, k, v, o, lse, do, cq, ck, causal=True, scale=scale, deterministic=True, dq=dq, dk=dk,
                          dv=dv, workspace=wb)

    g = _capture(step)
    for seed in (1011, 1012):
        x = make_varlen_inputs(seed, lens, lens, Hq, Hkv, d)
        for t, nm in ((q, "q"), (k, "k"), (v, "v")):
            t.copy_(x[nm].to(dev))
        do.copy_(make_varlen_inputs(seed + 50, lens, lens, Hq, Hkv, d)["q"].to(dev))
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (o, lse, dq, dk, dv)]
        step()
        torch.cuda.synchronize()
        for a, b in zip(got, (o, lse, dq, dk, dv)):
            assert torch.equal(a, b)
    assert A.attn_device_status(True) == 0


def test_wide_forward_graph(A):
    B, H, N, d = 1, 4, 1000, 256
    dev = torch.device("cuda")
    x0 = make_inputs(1020, B, H, H, N, d)
    q, k, v = (x0[n].to(dev) for n in ("q", "k", "v"))
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev)
    g = _capture(lambda: A.attn_fwd(q, k, v, causal=False, scale=default_scale(d), o=o, lse=lse))
    x = make_inputs(1021, B, H, H, N, d)
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        t.copy_(x[nm].to(dev))
    g.replay()
    torch.cuda.synchronize()
    got = (o.clone(), lse.clone())
    A.attn_fwd(q, k, v, causal=False, scale=default_scale(d), o=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(got[0], o) and torch.equal(got[1], lse)
    assert A.attn_device_status(True) == 0


def _replay_matches_eager(g, step, refill, outs, seeds):
    """Refill the inputs for each seed, replay the graph, then run the same calls eagerly:
    every output must agree bit for bit."""
    for seed in seeds:
        refill(seed)
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in outs]
        step()
        torch.cuda.synchronize()
        for a, b in zip(got, outs):
            assert torch.equal(a, b)


def test_fp8_quantise_and_forward_graph(A):
    # The quantiser and the FP8 forward in one graph: bf16 inputs in, O and LSE out.
    B, Hq, Hkv, N, d = 1, 4, 2, 700, 128
    dev = torch.device("cuda")
    x0 = make_inputs(1030, B, Hq, Hkv, N, d)
    q, k, v = (x0[n].to(dev) for n in ("q", "k", "v"))
    nb = (N + 127) // 128
    q8, k8, v8 = (torch.empty(t.shape, dtype=torch.uint8, device=dev) for t in (q, k, v))
    sq = torch.empty((B, Hq, nb), dtype=torch.float32, device=dev)
    sk, sv = (torch.empty((B, Hkv, nb), dtype=torch.float32, device=dev) for _ in range(2))
    o, lse = torch.empty_like(q), torch.empty((B, Hq, N), dtype=torch.float32, device=dev)

    def step():
        A.attn_quantize_fp8(q, q8, sq)
        A.attn_quantize_fp8(k, k8, sk)
        A.attn_quantize_fp8(v, v8, sv)
        A.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal=True, scale=default_scale(d), o=o, lse=lse)

    def refill(seed):
        x = make_inputs(seed, B, Hq, Hkv, N, d)
        for t, nm in ((q, "q"), (k, "k"), (v, "v")):
            t.copy_(x[nm].to(dev))

    g = _capture(step)
    _replay_matches_eager(g, step, refill, (q8, sq, k8, sk, v8, sv, o, lse), (1031, 1032))
    assert A.attn_device_status(True) == 0


@pytest.mark.parametrize("d", [192, 256])
def test_wide_training_step_graph(A, d):
    # Forward and deterministic backward at a wide head dimension (the 64-row backward).
    B, Hq, Hkv, N = 1, 4, 2, 520
    dev = torch.device("cuda")
    scale = default_scale(d)
    x0 = make_inputs(1040 + d, B, Hq, Hkv, N, d, with_grad=True)
    q, k, v, do = (x0[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = torch.empty_like(q), torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty((A.attn_bwd_workspace_size(B, Hq, Hkv, N, d, True),), dtype=torch.uint8, device=dev)

    def step():
        A.attn_fwd(q, k, v, causal=True, scale=scale, o=o, lse=lse)
        A.attn_bwd(q, k, v, o, lse, do, causal=True, scale=scale, deterministic=True, dq=dq, dk=dk, dv=dv,
                   workspace=ws)

    def refill(seed):
        x = make_inputs(seed, B, Hq, Hkv, N, d, with_grad=True)
        for t, nm in ((q, "q"), (k, "k"), (v, "v"), (do, "do")):
            t.copy_(x[nm].to(dev))

    g = _capture(step)
    _replay_matches_eager(g, step, refill, (o, lse, dq, dk, dv), (1050 + d, 1051 + d))
    assert A.attn_device_status(True) == 0


@pytest.mark.parametrize("one_tile", [True, False])
def test_grouped_decode_graph(A, one_tile):
    # A decode step (8 queries per KV head group packed into one tile, keys split across
    # CTAs, then the merge) captured with its workspace; the cache grows by refilling.
    B, Hq, Hkv, Nq, Nk, d = 2, 16, 4, 2, 3000, 128
    dev = torch.device("cuda")
    x0 = make_inputs(1060, B, Hq, Hkv, Nk, d)
    q = x0["q"][:, :, Nk - Nq:].contiguous().to(dev)
    k, v = x0["k"].to(dev), x0["v"].to(dev)
    o, lse = torch.empty_like(q), torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    n = A.attn_fwd_kv_workspace_size(B, Hq, Hkv, Nq, Nk, d)
    assert n > 0
    ws = torch.empty((n,), dtype=torch.uint8, device=dev)

    def step():
        A.attn_fwd_kv(q, k, v, causal=True, scale=default_scale(d), o=o, lse=lse, workspace=ws)

    def refill(seed):
        x = make_inputs(seed, B, Hq, Hkv, Nk, d)
        q.copy_(x["q"][:, :, Nk - Nq:].to(dev))
        k.copy_(x["k"].to(dev))
        v.copy_(x["v"].to(dev))

    A.attn_set_decode_one_tile(one_tile)
    try:
        g = _capture(step)
        _replay_matches_eager(g, step, refill, (o, lse), (1061, 1062))
    finally:
        A.attn_set_decode_one_tile(True)
    assert A.attn_device_status(True) == 0


def test_tile64_training_step_graph(A):
    # The 64-row backward at d = 128 (chosen by attn_set_bwd_query_tile) inside a graph.
    B, H, N, d = 1, 4, 700, 128
    dev = torch.device("cuda")
    scale = default_scale(d)
    x0 = make_inputs(1070, B, H, H, N, d, with_grad=True)
    q, k, v, do = (x0[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    A.attn_set_bwd_query_tile(64)
    try:
        ws = torch.empty((A.attn_bwd_workspace_size(B, H, H, N, d, True),), dtype=torch.uint8, device=dev)

        def step():
            A.attn_fwd(q, k, v, causal=False, scale=scale, o=o, lse=lse)
            A.attn_bwd(q, k, v, o, lse, do, causal=False, scale=scale, deterministic=True, dq=dq, dk=dk, dv=dv,
                       workspace=ws)

        def refill(seed):
            x = make_inputs(seed, B, H, H, N, d, with_grad=True)
            for t, nm in ((q, "q"), (k, "k"), (v, "v"), (do, "do")):
                t.copy_(x[nm].to(dev))

        g = _capture(step)
        _replay_matches_eager(g, step, refill, (o, lse, dq, dk, dv), (1071, 1072))
    finally:
        A.attn_set_bwd_query_tile(128)
    assert A.attn_device_status(True) == 0
