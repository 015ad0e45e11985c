"""Python binding for libattn.so: fused exact attention on GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  If the compiled
library is missing this module raises at import time; there is no fallback.

Names match the C ABI in include/attn.h: ``attn_fwd``, ``attn_fwd_kv``,
``attn_fwd_varlen`` and ``attn_bwd_varlen`` (packed sequences of different lengths), ``attn_bwd``,
``attn_bwd_noalloc``, ``attn_quantize_fp8`` and ``attn_fwd_fp8`` (e4m3 inputs with
per-block scales), the ``*_workspace_size`` queries, ``attn_last_error`` and the
test/tuning knobs.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() (or python -m "
                      "attention_attn_fwd_09_gb300._build) first")

_lib = ctypes.CDLL(LIB_PATH)
_p, _i, _f, _ll, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong, ctypes.c_size_t
_lib.attn_fwd.argtypes = [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _p]
_lib.attn_fwd.restype = _i
_lib.attn_fwd_kv.argtypes = [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _p, _sz, _p]
_lib.attn_fwd_kv.restype = _i
_lib.attn_fwd_kv_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i]
_lib.attn_fwd_kv_workspace_size.restype = _sz
_lib.attn_fwd_varlen.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _p, _sz, _p]
_lib.attn_fwd_varlen.restype = _i
_lib.attn_fwd_varlen_workspace_size.argtypes = [_i, _i, _i, _i, _i]
_lib.attn_fwd_varlen_workspace_size.restype = _sz
_lib.attn_bwd_varlen.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _i, _p,
                                 _sz, _p]
_lib.attn_bwd_varlen.restype = _i
_lib.attn_bwd_varlen_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i, _i]
_lib.attn_bwd_varlen_workspace_size.restype = _sz
_lib.attn_set_fwd_persistent.argtypes = [_i]
_lib.attn_set_fwd_persistent.restype = _i
_lib.attn_set_fwd_one_tile.argtypes = [_i]
_lib.attn_set_fwd_one_tile.restype = _i
_lib.attn_set_decode_one_tile.argtypes = [_i]
_lib.attn_set_decode_one_tile.restype = _i
_lib.attn_set_bwd_query_tile.argtypes = [_i]
_lib.attn_set_bwd_query_tile.restype = _i
_lib.attn_set_varlen_order.argtypes = [_i]
_lib.attn_set_varlen_order.restype = _i
_lib.attn_bwd.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _i, _p, _sz, _p]
_lib.attn_bwd.restype = _i
_lib.attn_bwd_noalloc.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _i, _p]
_lib.attn_bwd_noalloc.restype = _i
_lib.attn_bwd_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i]
_lib.attn_bwd_workspace_size.restype = _sz
_lib.attn_last_error.argtypes = []
_lib.attn_last_error.restype = ctypes.c_char_p
_lib.attn_version.argtypes = []
_lib.attn_version.restype = ctypes.c_char_p
_lib.attn_set_debug_knobs.argtypes = [_f, _i, _ll, _i]
_lib.attn_set_debug_knobs.restype = _i
_lib.attn_get_debug_knobs.argtypes = [ctypes.POINTER(_f), ctypes.POINTER(_i), ctypes.POINTER(_ll), ctypes.POINTER(_i)]
_lib.attn_get_debug_knobs.restype = _i
_lib.attn_device_status.argtypes = [_i]
_lib.attn_device_status.restype = _i
_lib.attn_rescale_counter.argtypes = [_i, ctypes.POINTER(ctypes.c_ulonglong)]
_lib.attn_rescale_counter.restype = _i
_lib.attn_set_test_hooks.argtypes = [_i]
_lib.attn_set_test_hooks.restype = _i
_lib.attn_quantize_fp8.argtypes = [_p, _p, _p, _i, _i, _i, _i, _p]
_lib.attn_quantize_fp8.restype = _i
_lib.attn_fwd_fp8.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _p]
_lib.attn_fwd_fp8.restype = _i
_lib.attn_exp2_sw.argtypes = [_p, _p, _ll, _i, _p]
_lib.attn_exp2_sw.restype = _i

STATUS = {0: "ATTN_OK", -1: "ATTN_ERR_INVALID_ARG", -2: "ATTN_ERR_UNSUPPORTED", -3: "ATTN_ERR_MISALIGNED",
          -4: "ATTN_ERR_WORKSPACE", -5: "ATTN_ERR_CUDA", -6: "ATTN_ERR_TIMEOUT"}


class AttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


def attn_last_error() -> str:
    return (_lib.attn_last_error() or b"").decode()


def attn_version() -> str:
    return _lib.attn_version().decode()


def _check(rc: int):
    if rc != 0:
        raise AttnError(rc, attn_last_error())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _dev_bf16(name, t, shape):
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected a contiguous CUDA bf16 tensor of shape {tuple(shape)}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device} (contiguous={t.is_contiguous()})")


def _dev_f32(name, t, shape):
    if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected a contiguous CUDA fp32 tensor of shape {tuple(shape)}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device} (contiguous={t.is_contiguous()})")


def _bwd_tensors(q, k, v, o, lse, do, dq, dk, dv):
    """Checks the backward's inputs and outputs ([B,Hq,N,d] / [B,Hkv,N,d] bf16, lse [B,Hq,N]
    fp32, all on one device) and allocates the outputs not given."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    for name, t, shp in (("q", q, (B, Hq, N, d)), ("k", k, (B, Hkv, N, d)), ("v", v, (B, Hkv, N, d)),
                         ("o", o, (B, Hq, N, d)), ("do", do, (B, Hq, N, d))):
        _dev_bf16(name, t, shp)
    _dev_f32("lse", lse, (B, Hq, N))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _dev_bf16("dq", dq, (B, Hq, N, d))
    _dev_bf16("dk", dk, (B, Hkv, N, d))
    _dev_bf16("dv", dv, (B, Hkv, N, d))
    for name, t in (("k", k), ("v", v), ("o", o), ("lse", lse), ("do", do), ("dq", dq), ("dk", dk), ("dv", dv)):
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
    return B, Hq, Hkv, N, d, dq, dk, dv


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None, stream=None):
    """O, LSE = attention(q, k, v).  q [B,Hq,N,d], k/v [B,Hkv,N,d] CUDA bf16.

    ``o`` ([B,Hq,N,d] bf16) and ``lse`` ([B,Hq,N] fp32) may be given to reuse buffers."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    _dev_bf16("q", q, (B, Hq, N, d))
    _dev_bf16("k", k, (B, Hkv, N, d))
    _dev_bf16("v", v, (B, Hkv, N, d))
    if scale is None:
        scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    _dev_bf16("o", o, (B, Hq, N, d))
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, Hq, N):
        raise ValueError("lse: expected a contiguous fp32 tensor [B,Hq,N]")
    _check(_lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, int(bool(causal)),
                         float(scale), _stream(stream)))
    return o, lse


def attn_fwd_kv_workspace_size(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int) -> int:
    n = _lib.attn_fwd_kv_workspace_size(B, Hq, Hkv, Nq, Nk, d)
    if n == ctypes.c_size_t(-1).value:
        raise AttnError(-1, attn_last_error())
    return int(n)


def attn_fwd_kv(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None, workspace=None,
                stream=None):
    """O, LSE for Nq queries after a cache of Nk >= Nq keys.  q [B,Hq,Nq,d], k/v [B,Hkv,Nk,d]
    CUDA bf16; query i stands at key position i + Nk - Nq (causal: sees keys up to there).
    ``workspace``: a uint8 CUDA tensor of at least attn_fwd_kv_workspace_size(...) bytes
    (allocated here when None and needed; pass an empty tensor to use the ordinary tiling)."""
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    _dev_bf16("q", q, (B, Hq, Nq, d))
    _dev_bf16("k", k, (B, Hkv, Nk, d))
    _dev_bf16("v", v, (B, Hkv, Nk, d))
    if scale is None:
        scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    _dev_bf16("o", o, (B, Hq, Nq, d))
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("lse: expected a contiguous fp32 tensor [B,Hq,Nq]")
    if workspace is None:
        n = attn_fwd_kv_workspace_size(B, Hq, Hkv, Nq, Nk, d)
        workspace = torch.empty((n,), dtype=torch.uint8, device=q.device)
    ws_ptr = _ptr(workspace) if workspace.numel() > 0 else ctypes.c_void_p(0)
    _check(_lib.attn_fwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                            int(bool(causal)), float(scale), ws_ptr, workspace.numel() * workspace.element_size(),
                            _stream(stream)))
    return o, lse


def attn_fwd_varlen_workspace_size(B: int, Hq: int, Hkv: int, total_q: int, d: int) -> int:
    n = _lib.attn_fwd_varlen_workspace_size(B, Hq, Hkv, total_q, d)
    if n == ctypes.c_size_t(-1).value:
        raise AttnError(-1, attn_last_error())
    return int(n)


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool = False, scale: float | None = None,
                    o=None, lse=None, workspace=None, stream=None):
    """O, LSE for packed sequences of different lengths.  q [Hq, total_q, d], k/v [Hkv,
    total_k, d] CUDA bf16; ``cu_seqlens_q``/``cu_seqlens_k``: CUDA int32 offsets (B + 1
    each) of the sequences along the row axis.  Within a sequence, query i stands at key
    position i + nk - nq (causal: sees keys up to there).  ``workspace``: a uint8 CUDA
    tensor of at least attn_fwd_varlen_workspace_size(...) bytes (allocated when None).
    The offsets are checked on the device; a failed check shows in attn_device_status()."""
    Hq, Tq, d = q.shape
    Hkv, Tk = k.shape[0], k.shape[1]
    _dev_bf16("q", q, (Hq, Tq, d))
    _dev_bf16("k", k, (Hkv, Tk, d))
    _dev_bf16("v", v, (Hkv, Tk, d))
    for name, c in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if c.dtype != torch.int32 or not c.is_cuda or not c.is_contiguous() or c.dim() != 1:
            raise ValueError(f"{name}: expected a contiguous 1-D CUDA int32 tensor")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k need B + 1 entries each")
    B = cu_seqlens_q.numel() - 1
    if scale is None:
        scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    _dev_bf16("o", o, (Hq, Tq, d))
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (Hq, Tq):
        raise ValueError("lse: expected a contiguous fp32 tensor [Hq, total_q]")
    if workspace is None:
        n = attn_fwd_varlen_workspace_size(B, Hq, Hkv, Tq, d)
        workspace = torch.empty((max(n, 16),), dtype=torch.uint8, device=q.device)
    _check(_lib.attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens_q),
                                _ptr(cu_seqlens_k), B, Hq, Hkv, Tq, Tk, d, int(bool(causal)), float(scale),
                                _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return o, lse


def attn_bwd_varlen_workspace_size(B: int, Hq: int, Hkv: int, total_q: int, total_k: int, d: int,
                                   deterministic: bool = False) -> int:
    n = _lib.attn_bwd_varlen_workspace_size(B, Hq, Hkv, total_q, total_k, d, int(bool(deterministic)))
    if n == ctypes.c_size_t(-1).value:
        raise AttnError(-1, attn_last_error())
    return int(n)


def attn_bwd_varlen(q, k, v, o, lse, do, cu_seqlens_q, cu_seqlens_k, causal: bool = False,
                    scale: float | None = None, deterministic: bool = False, dq=None, dk=None, dv=None,
                    workspace=None, stream=None):
    """dQ, dK, dV over packed sequences (layouts and offsets as ``attn_fwd_varlen``; ``o``
    and ``lse`` as it returned them, ``do`` like ``q``)."""
    Hq, Tq, d = q.shape
    Hkv, Tk = k.shape[0], k.shape[1]
    for name, t, shp in (("q", q, (Hq, Tq, d)), ("o", o, (Hq, Tq, d)), ("do", do, (Hq, Tq, d)),
                         ("k", k, (Hkv, Tk, d)), ("v", v, (Hkv, Tk, d))):
        _dev_bf16(name, t, shp)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (Hq, Tq):
        raise ValueError("lse: expected a contiguous fp32 tensor [Hq, total_q]")
    for name, c in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if c.dtype != torch.int32 or not c.is_cuda or not c.is_contiguous() or c.dim() != 1:
            raise ValueError(f"{name}: expected a contiguous 1-D CUDA int32 tensor")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k need B + 1 entries each")
    B = cu_seqlens_q.numel() - 1
    if scale is None:
        scale = d ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _dev_bf16("dq", dq, (Hq, Tq, d))
    _dev_bf16("dk", dk, (Hkv, Tk, d))
    _dev_bf16("dv", dv, (Hkv, Tk, d))
    if workspace is None:
        n = attn_bwd_varlen_workspace_size(B, Hq, Hkv, Tq, Tk, d, deterministic)
        workspace = torch.empty((max(n, 16),), dtype=torch.uint8, device=q.device)
    _check(_lib.attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                                _ptr(dv), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, Hq, Hkv, Tq, Tk, d,
                                int(bool(causal)), float(scale), int(bool(deterministic)), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)))
    return dq, dk, dv


def attn_set_fwd_persistent(enable: bool):
    """d = 64/128 forward: one CTA per SM walking the work list (True) or one per unit."""
    _check(_lib.attn_set_fwd_persistent(int(bool(enable))))


def attn_set_fwd_one_tile(enable: bool):
    """d = 128 forward kernel: one query tile per CTA (True) or two (False)."""
    _check(_lib.attn_set_fwd_one_tile(int(bool(enable))))


def attn_set_decode_one_tile(enable: bool):
    """attn_fwd_kv grouped decode at d = 128: the one-tile kernel (True, default) or the
    two-tile kernel (False)."""
    _check(_lib.attn_set_decode_one_tile(int(bool(enable))))


def attn_set_bwd_query_tile(rows: int):
    """d = 64/128 backward: 128-row query tiles (dQ^T in dP^T's columns) or 64-row tiles
    (dQ^T in columns of its own, next tile's products issued ahead)."""
    _check(_lib.attn_set_bwd_query_tile(int(rows)))


def attn_set_varlen_order(longest_first: bool = True):
    _check(_lib.attn_set_varlen_order(int(bool(longest_first))))


def attn_bwd_workspace_size(B: int, Hq: int, Hkv: int, N: int, d: int, deterministic: bool = False) -> int:
    n = _lib.attn_bwd_workspace_size(B, Hq, Hkv, N, d, int(bool(deterministic)))
    if n == ctypes.c_size_t(-1).value:
        raise AttnError(-1, attn_last_error())
    return int(n)


def attn_bwd(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None, deterministic: bool = False,
             dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV of attention given the forward's o, lse and the upstream gradient do."""
    B, Hq, Hkv, N, d, dq, dk, dv = _bwd_tensors(q, k, v, o, lse, do, dq, dk, dv)
    if scale is None:
        scale = d ** -0.5
    ws_bytes = attn_bwd_workspace_size(B, Hq, Hkv, N, d, deterministic)
    if workspace is None:
        workspace = torch.empty((max(ws_bytes, 16),), dtype=torch.uint8, device=q.device)
    _check(_lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                         B, Hq, Hkv, N, d, int(bool(causal)), float(scale), int(bool(deterministic)),
                         _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return dq, dk, dv


def attn_bwd_noalloc(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None,
                     deterministic: bool = False, dq=None, dk=None, dv=None, stream=None):
    """attn_bwd without a workspace, for callers that cannot allocate device memory on
    the call path; the library's own fixed 64 MiB array serves as the workspace (sizes
    needing more are rejected).  Overlapping calls on different streams race on it."""
    B, Hq, Hkv, N, d, dq, dk, dv = _bwd_tensors(q, k, v, o, lse, do, dq, dk, dv)
    if scale is None:
        scale = d ** -0.5
    _check(_lib.attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                                 _ptr(dv), B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                                 int(bool(deterministic)), _stream(stream)))
    return dq, dk, dv


def attn_quantize_fp8(x, x8=None, scales=None, stream=None):
    """e4m3 codes and per-128-row-block fp32 scales of x [B,H,N,128] bf16 (CUDA).  Returns
    (x8 uint8 [B,H,N,128], scales fp32 [B,H,ceil(N/128)])."""
    B, H, N, d = x.shape
    _dev_bf16("x", x, (B, H, N, d))
    nb = (N + 127) // 128
    x8 = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device) if x8 is None else x8
    scales = torch.empty((B, H, nb), dtype=torch.float32, device=x.device) if scales is None else scales
    if x8.dtype != torch.uint8 or not x8.is_contiguous() or tuple(x8.shape) != (B, H, N, d) or x8.device != x.device:
        raise ValueError("x8: expected a contiguous uint8 tensor shaped like x on its device")
    _dev_f32("scales", scales, (B, H, nb))
    _check(_lib.attn_quantize_fp8(_ptr(x), _ptr(x8), _ptr(scales), B, H, N, d, _stream(stream)))
    return x8, scales


def attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal: bool = False, scale: float | None = None, o=None,
                 lse=None, stream=None):
    """O, LSE of the FP8 inputs (e4m3 codes as uint8 tensors q8 [B,Hq,N,128], k8/v8
    [B,Hkv,N,128], fp32 block scales [.., ceil(N/128)] as attn_quantize_fp8 returns them).
    O is bf16, LSE fp32."""
    B, Hq, N, d = q8.shape
    Hkv = k8.shape[1]
    nb = (N + 127) // 128
    for name, t, shp in (("q8", q8, (B, Hq, N, d)), ("k8", k8, (B, Hkv, N, d)), ("v8", v8, (B, Hkv, N, d))):
        if t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != shp:
            raise ValueError(f"{name}: expected a contiguous CUDA uint8 tensor of shape {shp}")
    _dev_f32("q_scale", q_scale, (B, Hq, nb))
    _dev_f32("k_scale", k_scale, (B, Hkv, nb))
    _dev_f32("v_scale", v_scale, (B, Hkv, nb))
    if scale is None:
        scale = d ** -0.5
    o = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device=q8.device) if o is None else o
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    _dev_bf16("o", o, (B, Hq, N, d))
    _dev_f32("lse", lse, (B, Hq, N))
    _check(_lib.attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), _ptr(o),
                             _ptr(lse), B, Hq, Hkv, N, d, int(bool(causal)), float(scale), _stream(stream)))
    return o, lse


def attn_set_debug_knobs(tau: float = 8.0, poly_per_16: int = 0, wait_limit_ns: int = 2_000_000_000,
                         sync_check: bool = False):
    _check(_lib.attn_set_debug_knobs(float(tau), int(poly_per_16), int(wait_limit_ns), int(bool(sync_check))))


def attn_get_debug_knobs():
    tau, poly, wl, sc = _f(), _i(), _ll(), _i()
    _check(_lib.attn_get_debug_knobs(ctypes.byref(tau), ctypes.byref(poly), ctypes.byref(wl), ctypes.byref(sc)))
    return {"tau": tau.value, "poly_per_16": poly.value, "wait_limit_ns": wl.value, "sync_check": bool(sc.value)}


def attn_set_test_hooks(skip_first_kv_load: bool = False):
    _check(_lib.attn_set_test_hooks(int(bool(skip_first_kv_load))))


def attn_device_status(clear: bool = True) -> int:
    """Synchronise and return the raw status (0 = fine, ATTN_ERR_TIMEOUT = a kernel gave up)."""
    return int(_lib.attn_device_status(int(bool(clear))))


def attn_rescale_counter(enable: bool) -> int:
    v = ctypes.c_ulonglong(0)
    _check(_lib.attn_rescale_counter(int(bool(enable)), ctypes.byref(v)))
    return int(v.value)


def attn_exp2_sw(x, variant: int = 0, stream=None):
    """y = 2^x on the GPU: variant 0 = polynomial as used in the forward, 1 = polynomial
    with correct subnormals, 2 = MUFU ex2.approx."""
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x: contiguous CUDA fp32 tensor expected")
    y = torch.empty_like(x)
    _check(_lib.attn_exp2_sw(_ptr(x), _ptr(y), x.numel(), int(variant), _stream(stream)))
    return y


__all__ = ["attn_fwd", "attn_fwd_fp8", "attn_quantize_fp8", "attn_bwd", "attn_bwd_noalloc", "attn_bwd_workspace_size", "attn_last_error", "attn_version",
           "attn_set_debug_knobs", "attn_get_debug_knobs", "attn_device_status", "attn_rescale_counter",
           "attn_exp2_sw", "attn_set_test_hooks", "AttnError", "LIB_PATH"]
