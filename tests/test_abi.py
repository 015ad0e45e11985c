"""The C ABI library loads, exports every declared entry point, and rejects bad
arguments with the documented status codes before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    L = ctypes.CDLL(path)
    p, i, f, ll, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong, ctypes.c_size_t
    L.attn_fwd.argtypes = [p, p, p, p, p, i, i, i, i, i, i, f, p]
    L.attn_fwd.restype = i
    L.attn_fwd_kv.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, f, p, sz, p]
    L.attn_fwd_kv.restype = i
    L.attn_fwd_varlen.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, i, f, p, sz, p]
    L.attn_fwd_varlen.restype = i
    L.attn_fwd_varlen_workspace_size.argtypes = [i, i, i, i, i]
    L.attn_fwd_varlen_workspace_size.restype = sz
    L.attn_bwd_varlen.argtypes = [p, p, p, p, p, p, p, p, p, p, p, i, i, i, i, i, i, i, f, i, p, sz, p]
    L.attn_bwd_varlen.restype = i
    L.attn_bwd_varlen_workspace_size.argtypes = [i, i, i, i, i, i, i]
    L.attn_bwd_varlen_workspace_size.restype = sz
    L.attn_bwd.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, i, f, i, p, sz, p]
    L.attn_bwd.restype = i
    L.attn_bwd_workspace_size.argtypes = [i, i, i, i, i, i]
    L.attn_bwd_workspace_size.restype = sz
    L.attn_last_error.restype = ctypes.c_char_p
    L.attn_set_debug_knobs.argtypes = [f, i, ll, i]
    L.attn_set_debug_knobs.restype = i
    L.attn_exp2_sw.argtypes = [p, p, ll, i, p]
    L.attn_exp2_sw.restype = i
    return L


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "attn_fwd" in names and "attn_bwd" in names
    for n in names:
        assert hasattr(lib, n), n


FAKE = ctypes.c_void_p(0x10000)       # aligned, never dereferenced on the error paths
MIS = ctypes.c_void_p(0x10008)


def fwd(lib, B=1, Hq=2, Hkv=2, N=128, d=64, causal=0, scale=0.125, ptrs=None):
    q = k = v = o = lse = FAKE
    if ptrs:
        q, k, v, o, lse = ptrs
    return lib.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, None)


def test_fwd_argument_errors(lib):
    assert fwd(lib, d=96) == -2
    assert b"d=96" in lib.attn_last_error()
    assert fwd(lib, Hq=3, Hkv=2) == -1
    assert fwd(lib, Hkv=0) == -1
    assert fwd(lib, N=-1) == -1
    assert fwd(lib, scale=0.0) == -1
    assert fwd(lib, scale=float("nan")) == -1
    assert fwd(lib, ptrs=(FAKE, FAKE, MIS, FAKE, FAKE)) == -3
    assert fwd(lib, ptrs=(FAKE, None, FAKE, FAKE, FAKE)) == -1
    # Nothing to do: OK without any device work.
    assert fwd(lib, B=0) == 0
    assert fwd(lib, N=0) == 0


def test_bwd_workspace_and_errors(lib):
    assert lib.attn_bwd_workspace_size(0, 2, 2, 128, 64, 0) == 0
    n = lib.attn_bwd_workspace_size(2, 4, 2, 300, 128, 1)
    assert n >= 2 * 4 * 300 * 128 * 4      # at least the fp32 dQ accumulator
    assert n % 16 == 0
    assert lib.attn_bwd_workspace_size(1, 3, 2, 128, 64, 0) == ctypes.c_size_t(-1).value
    rc = lib.attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 2, 128, 96, 0, 0.1, 0,
                      FAKE, 1 << 30, None)
    assert rc == -2
    rc = lib.attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 2, 128, 64, 0, 0.1, 0,
                      FAKE, 16, None)
    assert rc == -4                          # workspace too small
    # d <= 128: dQ accumulator (rows padded to 128-row tiles), D and LSE2; deterministic adds
    # four counter sets per (head, 128-row tile) and a second accumulator.  The size covers
    # the 64-row-tile layout too, which is never larger at these sizes.
    al = lambda x: (x + 255) // 256 * 256
    B, Hq, N, d = 2, 4, 300, 128
    acc = al(B * Hq * 384 * d * 4)
    base = acc + 2 * al(B * Hq * N * 4)
    assert lib.attn_bwd_workspace_size(B, Hq, 2, N, d, 0) == base
    assert lib.attn_bwd_workspace_size(B, Hq, 2, N, d, 1) == base + al(4 * B * Hq * 3 * 4) + acc
    # from 64 query tiles per head (N > 8064) on, three more accumulators
    B, Hq, N, d = 1, 2, 8065, 64
    acc = al(B * Hq * 64 * 128 * d * 4)
    base = acc + 2 * al(B * Hq * N * 4)
    assert lib.attn_bwd_workspace_size(B, Hq, 2, N, d, 1) == base + al(4 * B * Hq * 64 * 4) + 3 * acc
    assert lib.attn_bwd_workspace_size(B, Hq, 2, 8064, d, 1) == (
        al(B * Hq * 8064 * d * 4) + 2 * al(B * Hq * 8064 * 4) + al(4 * B * Hq * 63 * 4) + al(B * Hq * 8064 * d * 4))
    # wide heads (192, 256): dQ accumulator rows padded to whole 64-row tiles, counters per
    # (head, 64-row tile, column half) when deterministic
    for d in (192, 256):
        B, Hq, N = 2, 4, 300
        base = al(B * Hq * 320 * d * 4) + 2 * al(B * Hq * N * 4)
        assert lib.attn_bwd_workspace_size(B, Hq, 2, N, d, 0) == base
        assert lib.attn_bwd_workspace_size(B, Hq, 2, N, d, 1) == base + al(B * Hq * 5 * 2 * 4)
        rc = lib.attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 2, 128, d, 0, 0.1, 0,
                          FAKE, 16, None)
        assert rc == -4


def test_knobs_validate(lib):
    assert lib.attn_set_debug_knobs(-1.0, 0, 1000, 0) == -1
    assert lib.attn_set_debug_knobs(8.0, 3, 1000, 0) == -2
    assert lib.attn_set_debug_knobs(8.0, 0, 0, 0) == -1
    assert lib.attn_set_debug_knobs(8.0, 0, 2_000_000_000, 0) == 0


def test_exp2_entry_validates(lib):
    assert lib.attn_exp2_sw(None, None, -1, 0, None) == -1
    assert lib.attn_exp2_sw(FAKE, FAKE, 16, 7, None) == -1
    assert lib.attn_exp2_sw(None, None, 0, 0, None) == 0


def test_fwd_kv_argument_errors(lib):
    # Checked before any device work.
    args = lambda Nq, Nk, causal: (FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 2, Nq, Nk, 64, causal, 0.1, None, 0, None)
    assert lib.attn_fwd_kv(*args(4, 0, 0)) == -1          # queries but no keys
    assert b"no keys" in lib.attn_last_error()
    assert lib.attn_fwd_kv(*args(9, 8, 1)) == -1          # causal with more queries than keys
    assert b"N <= Nk" in lib.attn_last_error()
    assert lib.attn_fwd_kv(*args(4, -1, 0)) == -1
    assert lib.attn_fwd_kv(*args(0, 8, 1)) == 0           # nothing to do


def test_fwd_varlen_argument_errors(lib):
    # Host-side checks, before any device work (the offsets themselves are checked on the
    # device).  The workspace bound: B=2 sequences, 4 heads (no head pairs), 300 rows:
    # floor(300/128) + 2 = 4 tiles per head at most, ceil((4 + 2) / 2) = 3 records per head.
    assert lib.attn_fwd_varlen_workspace_size(2, 4, 4, 300, 64) == 256 + 3 * 4 * 16
    assert lib.attn_fwd_varlen_workspace_size(2, 4, 2, 300, 64) == 256 + 4 * 2 * 16   # head pairs
    assert lib.attn_fwd_varlen_workspace_size(0, 4, 4, 300, 64) == 0
    assert lib.attn_fwd_varlen_workspace_size(2, 4, 3, 300, 64) == ctypes.c_size_t(-1).value

    def call(B=2, Hq=4, Hkv=4, tq=300, tk=300, d=64, causal=0, cu=FAKE, ws=FAKE, ws_bytes=1 << 20):
        return lib.attn_fwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, cu, cu, B, Hq, Hkv, tq, tk, d, causal, 0.1,
                                   ws, ws_bytes, None)
    assert call(d=96) == -2
    # wide heads: one tile per record, floor(300/128) + 2 = 4 tiles per head at most
    assert lib.attn_fwd_varlen_workspace_size(2, 4, 4, 300, 256) == 256 + 4 * 4 * 16
    assert call(tk=0) == -1 and b"no keys" in lib.attn_last_error()
    assert call(Hq=70000, Hkv=70000) == -2
    assert call(cu=ctypes.c_void_p(0x10002)) == -3
    assert call(ws_bytes=100) == -4
    assert call(ws=MIS) == -3
    assert call(B=0) == 0 and call(tq=0) == 0


def test_bwd_varlen_workspace_and_errors(lib):
    # Layout: dQ accumulator Hq x (total_q + 128 B) x d fp32, D and LSE2 Hq x total_q fp32
    # (each rounded up to 256 bytes), counters Hq x ((total_q + 128 B) / 128 + 1) when
    # deterministic, then a 256-byte header and Hkv x (total_k / 128 + B) 16-byte records.
    al = lambda x: (x + 255) // 256 * 256
    B, Hq, Hkv, tq, tk, d = 3, 4, 2, 500, 700, 64
    rows_pad = tq + 128 * B
    base = al(Hq * rows_pad * d * 4) + 2 * al(Hq * tq * 4) + 256 + Hkv * (tk // 128 + B) * 16
    assert lib.attn_bwd_varlen_workspace_size(B, Hq, Hkv, tq, tk, d, 0) == base
    assert lib.attn_bwd_varlen_workspace_size(B, Hq, Hkv, tq, tk, d, 1) == base + al(Hq * (rows_pad // 128 + 1) * 4)
    assert lib.attn_bwd_varlen_workspace_size(0, Hq, Hkv, tq, tk, d, 0) == 0
    assert lib.attn_bwd_varlen_workspace_size(B, Hq, 3, tq, tk, d, 0) == ctypes.c_size_t(-1).value

    def call(tq=500, tk=700, d=64, ws=FAKE, ws_bytes=1 << 30, cu=FAKE):
        return lib.attn_bwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, cu, cu, 3, 4, 2, tq, tk, d,
                                   0, 0.1, 0, ws, ws_bytes, None)
    assert call(d=96) == -2
    assert call(tk=0) == -1 and b"no keys" in lib.attn_last_error()
    assert call(ws_bytes=1000) == -4
    assert call(ws=MIS) == -3
    assert call(cu=ctypes.c_void_p(0x10001)) == -3
    assert call(tq=0, tk=0) == 0


def test_fp8_argument_errors(lib):
    # Host-side checks of the FP8 entry points, before any device work.
    lib.attn_quantize_fp8.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    lib.attn_quantize_fp8.restype = ctypes.c_int
    p, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_fwd_fp8.argtypes = [p] * 8 + [i] * 6 + [f, p]
    lib.attn_fwd_fp8.restype = i
    assert lib.attn_quantize_fp8(FAKE, FAKE, FAKE, 1, 2, 128, 64, None) == -2
    assert b"128" in lib.attn_last_error()
    assert lib.attn_quantize_fp8(FAKE, FAKE, None, 1, 2, 128, 128, None) == -1
    assert lib.attn_quantize_fp8(FAKE, MIS, FAKE, 1, 2, 128, 128, None) == -3
    assert lib.attn_quantize_fp8(FAKE, FAKE, FAKE, 1, 2, 0, 128, None) == 0

    def call(d=128, Hq=2, Hkv=2, N=128, scale=0.1, q8=FAKE, ks=FAKE):
        return lib.attn_fwd_fp8(q8, FAKE, FAKE, FAKE, ks, FAKE, FAKE, FAKE, 1, Hq, Hkv, N, d, 0, scale, None)
    assert call(d=64) == -2 and b"FP8" in lib.attn_last_error()
    assert call(Hq=3) == -1
    assert call(scale=-1.0) == -1
    assert call(q8=None) == -1
    assert call(q8=MIS) == -3
    assert call(ks=ctypes.c_void_p(0x10002)) == -3
    assert call(N=0) == 0
