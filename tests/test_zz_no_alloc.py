"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory on the
call path (plugins inside another runtime's memory pool, latency-critical loops where a
cudaMalloc would synchronise the device).  It must give what attn_bwd gives with a
caller workspace.

Collected last on purpose (file name), so a run that stops at the first failure has
already run every other test.  Calls go through the C ABI with ctypes.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import default_scale, make_inputs
from parity import GRAD_REL_FRO, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import attention_attn_fwd_09_gb300 as A
    L = ctypes.CDLL(A.LIB_PATH)
    p, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.attn_bwd_noalloc.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, i, f, i, p]
    L.attn_bwd_noalloc.restype = i
    L.attn_bwd.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, i, f, i, p, sz, p]
    L.attn_bwd.restype = i
    L.attn_bwd_workspace_size.argtypes = [i, i, i, i, i, i]
    L.attn_bwd_workspace_size.restype = sz
    L.attn_last_error.restype = ctypes.c_char_p
    return L, A


def P(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("causal,deterministic", [(False, False), (True, True)])
def test_noalloc_matches_workspace_entry_point(lib, causal, deterministic):
    L, A = lib
    B, Hq, Hkv, N, d = 2, 4, 2, 300, 128
    dev = torch.device("cuda")
    scale = default_scale(d)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):           # two calls in a row: the shared array's old contents must not leak in
        x = make_inputs(900 + call, B, Hq, Hkv, N, d, with_grad=True)
        q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
        o, lse = A.attn_fwd(q, k, v, causal=causal, scale=scale)
        ref = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
        got = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
        ws_bytes = L.attn_bwd_workspace_size(B, Hq, Hkv, N, d, int(deterministic))
        ws = torch.empty((ws_bytes,), dtype=torch.uint8, device=dev)
        rc = L.attn_bwd(P(q), P(k), P(v), P(o), P(lse), P(do), P(ref[0]), P(ref[1]), P(ref[2]), B, Hq, Hkv, N, d,
                        int(causal), scale, int(deterministic), P(ws), ws_bytes, stream)
        assert rc == 0, L.attn_last_error()
        rc = L.attn_bwd_noalloc(P(q), P(k), P(v), P(o), P(lse), P(do), P(got[0]), P(got[1]), P(got[2]), B, Hq,
                                Hkv, N, d, int(causal), scale, int(deterministic), stream)
        assert rc == 0, L.attn_last_error()
        torch.cuda.synchronize()
        assert A.attn_device_status(True) == 0
        # Against the fp64 oracle on the same inputs, and against attn_bwd (bit for bit when
        # deterministic: the same kernels add in the same order).
        truth = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, scale)
        for name, g, r, t in zip(("dq", "dk", "dv"), got, ref, truth):
            g, r = g.float().cpu().numpy(), r.float().cpu().numpy()
            assert np.isfinite(g).all()
            assert rel_fro(g, t) <= GRAD_REL_FRO, (call, name, "oracle", rel_fro(g, t))
            assert rel_fro(g, r) <= GRAD_REL_FRO, (call, name, rel_fro(g, r))
            if deterministic:
                assert np.array_equal(g, r), (call, name)


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    L, _ = lib
    B, Hq, Hkv, N, d = 8, 16, 16, 4096, 128        # needs far more than 64 MiB
    assert L.attn_bwd_workspace_size(B, Hq, Hkv, N, d, 0) > (64 << 20)
    fake = ctypes.c_void_p(0x10000)
    rc = L.attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, B, Hq, Hkv, N, d, 0, 0.1, 0, None)
    assert rc == -4
    assert b"64 MiB" in L.attn_last_error()
