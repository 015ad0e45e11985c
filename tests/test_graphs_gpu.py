"""The library's calls are stream-ordered and never synchronise with the host, so a whole
training step (forward and backward), the packed-sequence pair and the wide-head forward
can be captured once in a CUDA graph and replayed: each replay on new inputs must give,
bit for bit, what the eager calls give (deterministic dQ order, so that the backward is
reproducible)."""
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
