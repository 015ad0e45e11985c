"""Forward over packed sequences of different lengths (attn_fwd_varlen): the CUDA path
against the fp64 oracle element by element, against the single-sequence entry point bit
for bit, independent of the tile order, and with offsets that fail the device check."""
import numpy as np
import pytest
import torch

import oracle
from attn_inputs import default_scale, make_varlen_inputs, varlen_workload
from parity import check_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import attention_attn_fwd_09_gb300 as A
    A.attn_set_debug_knobs()
    A.attn_set_varlen_order(True)
    A.attn_device_status(True)
    yield A
    A.attn_set_varlen_order(True)


CASES = {  # name: (lens_q, extra keys per sequence or None for nk = nq, Hq, Hkv, d)
    "ragged_mha_d128": ([1, 127, 128, 129, 300, 1000, 256, 257], None, 4, 4, 128),
    "empty_seqs_d64": ([0, 5, 0, 0, 130, 0, 383], None, 2, 2, 64),
    "gqa_pairs_d128": ([700, 64, 512, 3, 1200], None, 8, 2, 128),
    "odd_group_d128": ([333, 129, 1, 640], None, 6, 2, 128),
    "mqa_d64": ([900, 17, 256, 511], None, 4, 1, 64),
    "longer_keys_d128": ([100, 1, 300, 128, 40], [29, 700, 1, 128, 0], 4, 2, 128),
    "single_seq_d128": ([1500], None, 2, 2, 128),
    # wide heads: the one-tile kernel, one table record per tile
    "wide_d256": ([300, 1, 640, 129], None, 4, 2, 256),
    "wide_d192_longer_keys": ([100, 7, 300, 0], [229, 7, 900, 3], 2, 1, 192),
}


def _run(A, x, causal, scale, order=True):
    dev = torch.device("cuda")
    A.attn_set_varlen_order(order)
    o, lse = A.attn_fwd_varlen(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), x["cu_q"].to(dev),
                               x["cu_k"].to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    A.attn_set_varlen_order(True)
    assert A.attn_device_status(True) == 0
    return o, lse


def _inputs(name, causal):
    lens_q, extra, Hq, Hkv, d = CASES[name]
    lens_k = list(lens_q) if extra is None else [n + e for n, e in zip(lens_q, extra)]
    seed = 600 + sum(lens_q) % 97 + d
    return make_varlen_inputs(seed, lens_q, lens_k, Hq, Hkv, d), default_scale(d)


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_oracle(A, name, causal):
    x, scale = _inputs(name, causal)
    o, lse = _run(A, x, causal, scale)
    O, L = oracle.attn_fwd_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], causal, scale)
    check_fwd(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, f"{name} causal={causal}")


@pytest.mark.parametrize("name", ["ragged_mha_d128", "gqa_pairs_d128", "longer_keys_d128", "odd_group_d128",
                                  "wide_d256", "wide_d192_longer_keys"])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_each_sequence_alone(A, name, causal):
    # Every tile does the same arithmetic as in a call on its sequence alone: keys past the
    # sequence's end are masked whether they are zero fill or the next sequence's keys.
    x, scale = _inputs(name, causal)
    o, lse = _run(A, x, causal, scale)
    dev = torch.device("cuda")
    cq, ck = x["cu_q"].tolist(), x["cu_k"].tolist()
    none = torch.empty((0,), dtype=torch.uint8, device=dev)   # ordinary tiling in attn_fwd_kv
    for b in range(len(cq) - 1):
        if cq[b + 1] == cq[b]:
            continue
        qb = x["q"][:, cq[b]:cq[b + 1]].unsqueeze(0).contiguous().to(dev)
        kb = x["k"][:, ck[b]:ck[b + 1]].unsqueeze(0).contiguous().to(dev)
        vb = x["v"][:, ck[b]:ck[b + 1]].unsqueeze(0).contiguous().to(dev)
        ob, lb = A.attn_fwd_kv(qb, kb, vb, causal=causal, scale=scale, workspace=none)
        assert torch.equal(o[:, cq[b]:cq[b + 1]], ob[0]), f"sequence {b}: O differs"
        assert torch.equal(lse[:, cq[b]:cq[b + 1]], lb[0]), f"sequence {b}: LSE differs"
    assert A.attn_device_status(True) == 0


@pytest.mark.parametrize("causal", [False, True])
def test_tile_order_does_not_change_results(A, causal):
    x, scale = _inputs("ragged_mha_d128", causal)
    o1, l1 = _run(A, x, causal, scale, order=True)
    o0, l0 = _run(A, x, causal, scale, order=False)
    assert torch.equal(o1, o0) and torch.equal(l1, l0)


def test_bad_offsets_fail_the_device_check(A):
    x = make_varlen_inputs(650, [200, 100], [200, 100], 2, 2, 64)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.full_like(q, 7.0)
    lse = torch.full((2, 300), 7.0, dtype=torch.float32, device=dev)
    bad = [[0, 250, 200, 300],   # decreasing
           [0, 100, 290],        # does not end at the packed length
           [5, 100, 300]]        # does not start at 0
    for cu in bad:
        c = torch.tensor(cu, dtype=torch.int32, device=dev)
        A.attn_fwd_varlen(q, k, v, c, c, causal=False, scale=0.125, o=o, lse=lse)
        assert A.attn_device_status(True) == -1, cu
        assert bool((o == 7.0).all()) and bool((lse == 7.0).all()), "outputs written despite bad offsets"
    # causal needs at least as many keys as queries in every sequence
    cq = torch.tensor([0, 200, 300], dtype=torch.int32, device=dev)
    ck = torch.tensor([0, 150, 300], dtype=torch.int32, device=dev)
    A.attn_fwd_varlen(q, k, v, cq, ck, causal=True, scale=0.125, o=o, lse=lse)
    assert A.attn_device_status(True) == -1
    assert bool((o == 7.0).all())
    # the same offsets are valid without causal
    A.attn_fwd_varlen(q, k, v, cq, ck, causal=False, scale=0.125, o=o, lse=lse)
    assert A.attn_device_status(True) == 0


@pytest.mark.parametrize("causal", [False, True])
def test_mixed_length_batch_full_size(A, causal):
    # The packed mixed-length batch the benchmark times (65536 tokens, 16 heads, d = 128):
    # every sequence bit for bit against the single-sequence entry point, and the shortest
    # and the longest sequence against the oracle on two heads.
    w = varlen_workload()
    x = make_varlen_inputs(w["seed"], w["lens"], w["lens"], w["Hq"], w["Hkv"], w["d"])
    scale = default_scale(w["d"])
    o, lse = _run(A, x, causal, scale)
    assert bool(torch.isfinite(lse).all())
    dev = torch.device("cuda")
    cq = x["cu_q"].tolist()
    none = torch.empty((0,), dtype=torch.uint8, device=dev)
    for b in range(len(cq) - 1):
        sl = slice(cq[b], cq[b + 1])
        qb, kb, vb = (x[n][:, sl].unsqueeze(0).contiguous().to(dev) for n in ("q", "k", "v"))
        ob, lb = A.attn_fwd_kv(qb, kb, vb, causal=causal, scale=scale, workspace=none)
        assert torch.equal(o[:, sl], ob[0]) and torch.equal(lse[:, sl], lb[0]), f"sequence {b}"
    lens = w["lens"]
    for b in (int(np.argmin(lens)), int(np.argmax(lens))):
        sl = slice(cq[b], cq[b + 1])
        heads = [(0, 0), (0, 11)]
        O, L = oracle.attn_fwd_kv(x["q"][:, sl].unsqueeze(0).contiguous(), x["k"][:, sl].unsqueeze(0).contiguous(),
                                  x["v"][:, sl].unsqueeze(0).contiguous(), causal, scale, heads=heads)
        got_o = o[[0, 11], sl].float().cpu().numpy()
        got_l = lse[[0, 11], sl].cpu().numpy()
        check_fwd(got_o, got_l, O, L, f"sequence {b} (length {lens[b]}) causal={causal}")
