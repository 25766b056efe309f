"""Python binding of ``libmpfa.so`` (the MpFA QK4PV8 attention forward).

Argument marshalling only: this module allocates outputs and workspaces with
torch on the caller's device, passes raw pointers and the current CUDA stream
through the C ABI (``include/mpfa.h``) and raises on a non-zero status.  Every
step of the computation runs in the library's CUDA kernels; there is no
fallback.  If the library is missing this import fails.

Method: "MpFA: Hardware-Efficient Train-Free QK4V8 FlashAttention Kernels on
Blackwell GPUs" (abstract) -- NVFP4 Q/K, FP8 P/V, rank-one smoothing
compensation, split work for decode.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmpfa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first "
        "(python -c 'import __graft_entry__ as g; g.build()' or "
        "python flashattention_mpfa_quantize_gb300/build.py)")

_lib = ctypes.CDLL(LIB_PATH)

D = 128
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4


class MpfaError(RuntimeError):
    def __init__(self, status: int, where: str):
        name = _lib.mpfa_status_string(status).decode()
        extra = ""
        if status == ERR_CUDA:
            extra = f" [{_lib.mpfa_last_cuda_error().decode()}]"
        super().__init__(f"{where}: {name} ({status}){extra}")
        self.status = status


class NVFP4(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p)]


class FP8(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p)]


class Rank1(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


class KSmooth(ctypes.Structure):
    _fields_ = [("kbar", ctypes.c_void_p), ("lse_shift", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_lib.mpfa_status_string.restype = ctypes.c_char_p
_lib.mpfa_status_string.argtypes = [_I]
_lib.mpfa_last_cuda_error.restype = ctypes.c_char_p
_lib.mpfa_last_cuda_error.argtypes = []
_lib.mpfa_quantize_workspace_size.restype = _SZ
_lib.mpfa_quantize_workspace_size.argtypes = [_I, _I, _I, _I, _I, _I, _I]
_lib.mpfa_quantize_qkv.restype = _I
_lib.mpfa_quantize_qkv.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                   ctypes.POINTER(NVFP4), ctypes.POINTER(Rank1),
                                   ctypes.POINTER(NVFP4), ctypes.POINTER(FP8),
                                   ctypes.POINTER(KSmooth), _P, _SZ, _P]
_lib.mpfa_prefill.restype = _I
_lib.mpfa_prefill.argtypes = [ctypes.POINTER(NVFP4), ctypes.POINTER(Rank1),
                              ctypes.POINTER(NVFP4), ctypes.POINTER(FP8), _I, _I, _I, _I, _I,
                              _I, _I, _I, _P, _P, _P, _P]
_lib.mpfa_quantize_v_fp4.restype = _I
_lib.mpfa_quantize_v_fp4.argtypes = [_P, _I, _I, _I, _I, ctypes.POINTER(NVFP4), _P, _SZ, _P]
_lib.mpfa_prefill_fp4pv.restype = _I
_lib.mpfa_prefill_fp4pv.argtypes = [ctypes.POINTER(NVFP4), ctypes.POINTER(Rank1),
                                    ctypes.POINTER(NVFP4), ctypes.POINTER(NVFP4), _I, _I, _I, _I,
                                    _I, _I, _I, _I, _P, _P, _P]
_lib.mpfa_decode_workspace_size.restype = _SZ
_lib.mpfa_decode_workspace_size.argtypes = [_I, _I, _I, _I, _I, _I]
_lib.mpfa_decode.restype = _I
_lib.mpfa_decode.argtypes = [_P, ctypes.POINTER(NVFP4), ctypes.POINTER(FP8), _P, _P, _I, _I, _I,
                             _I, _I, _I, _I, _I, _P, _P, ctypes.POINTER(NVFP4),
                             ctypes.POINTER(Rank1), ctypes.POINTER(_I), _P, _SZ, _P]
_lib.mpfa_append_kv.restype = _I
_lib.mpfa_append_kv.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, ctypes.POINTER(NVFP4),
                                ctypes.POINTER(FP8), _P, _P]
_lib.mpfa_decode_paged.restype = _I
_lib.mpfa_decode_paged.argtypes = [_P, ctypes.POINTER(NVFP4), ctypes.POINTER(FP8), _P, _I, _I, _P,
                                   _I, _I, _I, _I, _I, _I, _I, _P, _P, ctypes.POINTER(NVFP4),
                                   ctypes.POINTER(Rank1), ctypes.POINTER(_I), _P, _SZ, _P]
_lib.mpfa_append_kv_paged.restype = _I
_lib.mpfa_append_kv_paged.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                      ctypes.POINTER(NVFP4), ctypes.POINTER(FP8), _P]
_lib.mpfa_get_error.restype = _I
_lib.mpfa_get_error.argtypes = [_P]

lib = _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(status, where):
    if status != OK:
        raise MpfaError(status, where)


def get_error(device=None) -> int:
    """Synchronize the current stream and return (and clear) the device status."""
    return _lib.mpfa_get_error(_stream(device))


# --------------------------------------------------------------------------
# quantization
# --------------------------------------------------------------------------

def alloc_nvfp4(rows_shape, device):
    """codes [..., 64] u8, tiled scales (rows*8 bytes) u8, tensor scale f32[1]."""
    rows = 1
    for s in rows_shape:
        rows *= s
    return dict(codes=torch.empty(*rows_shape, 64, dtype=torch.uint8, device=device),
                scales=torch.empty(rows * 8, dtype=torch.uint8, device=device),
                scale=torch.empty(1, dtype=torch.float32, device=device))


def quantize_qkv(q=None, k=None, v=None, *, compensate=True, T=2, k_smooth=False,
                 workspace=None):
    """Quantize bf16 q [B,Nq,Hq,128], k / v [B,Nk,Hkv,128] (any may be None).

    Returns a dict with ``q`` (codes [B,Hq,Nq,64], scales, scale), ``qbar``
    (codes [B,Hq,Nq/128,T,64], scales [B,Hq,Nq/128,T,8]) when compensating,
    ``k`` (codes [B,Hkv,Nk,64], scales, scale), ``v`` (codes [B,Hkv,Nk,128],
    scale), plus the shape fields.  k_smooth (needs k): key-side smoothing,
    adding ``kbar`` (f32 [B,Hkv,128]) and, with q, ``lse_shift`` (f32
    [B,Hq,Nq]); prefill and decode pick them up from the dict."""
    ref = next(t for t in (q, k, v) if t is not None)
    dev = ref.device
    B = ref.shape[0]
    Nq, Hq = (q.shape[1], q.shape[2]) if q is not None else (0, 0)
    src_kv = k if k is not None else v
    Nk, Hkv = (src_kv.shape[1], src_kv.shape[2]) if src_kv is not None else (0, 0)
    comp = bool(compensate) and q is not None
    for t in (q, k, v):
        if t is not None:
            assert t.dtype == torch.bfloat16 and t.is_contiguous() and t.shape[-1] == D
    out = dict(B=B, Nq=Nq, Nk=Nk, Hq=Hq, Hkv=Hkv, compensate=comp, T=T if comp else 0)
    qs = ks = vs = None
    rb = None
    if q is not None:
        out["q"] = alloc_nvfp4((B, Hq, Nq), dev)
        qs = NVFP4(out["q"]["codes"].data_ptr(), out["q"]["scales"].data_ptr(),
                   out["q"]["scale"].data_ptr())
        if comp:
            out["qbar"] = dict(
                codes=torch.empty(B, Hq, Nq // 128, T, 64, dtype=torch.uint8, device=dev),
                scales=torch.empty(B, Hq, Nq // 128, T, 8, dtype=torch.uint8, device=dev))
            rb = Rank1(out["qbar"]["codes"].data_ptr(), out["qbar"]["scales"].data_ptr())
    if k is not None:
        out["k"] = alloc_nvfp4((B, Hkv, Nk), dev)
        ks = NVFP4(out["k"]["codes"].data_ptr(), out["k"]["scales"].data_ptr(),
                   out["k"]["scale"].data_ptr())
    if v is not None:
        out["v"] = dict(codes=torch.empty(B, Hkv, Nk, 128, dtype=torch.uint8, device=dev),
                        scale=torch.empty(1, dtype=torch.float32, device=dev))
        vs = FP8(out["v"]["codes"].data_ptr(), out["v"]["scale"].data_ptr())
    ksm = None
    if k_smooth:
        assert k is not None, "key-side smoothing needs k"
        out["kbar"] = torch.empty(B, Hkv, D, dtype=torch.float32, device=dev)
        if q is not None:
            out["lse_shift"] = torch.empty(B, Hq, Nq, dtype=torch.float32, device=dev)
        ksm = KSmooth(out["kbar"].data_ptr(),
                      out["lse_shift"].data_ptr() if q is not None else None)
    ws_bytes = _lib.mpfa_quantize_workspace_size(B, Nq, Nk if k is not None else 0, Hq, Hkv,
                                                 int(comp), int(bool(k_smooth)))
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    st = _lib.mpfa_quantize_qkv(
        _ptr(q), _ptr(k), _ptr(v), B, Nq, Nk, Hq, Hkv, D, int(comp), int(T),
        ctypes.byref(qs) if qs is not None else None, ctypes.byref(rb) if rb is not None else None,
        ctypes.byref(ks) if ks is not None else None, ctypes.byref(vs) if vs is not None else None,
        ctypes.byref(ksm) if ksm is not None else None,
        _ptr(workspace), workspace.numel(), _stream(dev))
    _check(st, "mpfa_quantize_qkv")
    out["_workspace"] = workspace
    return out


# --------------------------------------------------------------------------
# prefill / decode
# --------------------------------------------------------------------------

def _nvfp4(d):
    return NVFP4(d["codes"].data_ptr(), d["scales"].data_ptr(), d["scale"].data_ptr())


def prefill(qz, *, causal, out=None, lse=None, want_lse=True):
    """Attention forward on the output of quantize_qkv (q, k and v given).
    Returns (o bf16 [B,N,Hq,128], lse f32 [B,Hq,N] or None)."""
    B, N, Hq, Hkv = qz["B"], qz["Nq"], qz["Hq"], qz["Hkv"]
    assert qz["Nk"] == N, "prefill takes N_q == N_k"
    dev = qz["q"]["codes"].device
    if out is None:
        out = torch.empty(B, N, Hq, D, dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
    qs, ks = _nvfp4(qz["q"]), _nvfp4(qz["k"])
    vs = FP8(qz["v"]["codes"].data_ptr(), qz["v"]["scale"].data_ptr())
    comp = qz["compensate"]
    rb = Rank1(qz["qbar"]["codes"].data_ptr(), qz["qbar"]["scales"].data_ptr()) if comp else None
    st = _lib.mpfa_prefill(ctypes.byref(qs), ctypes.byref(rb) if rb is not None else None,
                           ctypes.byref(ks), ctypes.byref(vs), B, N, Hq, Hkv, D, int(bool(causal)),
                           int(comp), int(qz["T"]), _ptr(out), _ptr(lse),
                           _ptr(qz.get("lse_shift")), _stream(dev))
    _check(st, "mpfa_prefill")
    return out, lse


def quantize_v_fp4(v, *, workspace=None):
    """Full-FP4 PV ablation: V^T of bf16 v [B,Nk,Hkv,128] in NVFP4 along the
    keys.  Returns dict(codes u8 [B,Hkv,128,Nk/2], scales u8 (one 1 KB tile
    per 128-key tile), scale f32[1])."""
    assert v.dtype == torch.bfloat16 and v.is_contiguous() and v.shape[-1] == D
    B, Nk, Hkv = v.shape[0], v.shape[1], v.shape[2]
    dev = v.device
    out = dict(codes=torch.empty(B, Hkv, D, Nk // 2, dtype=torch.uint8, device=dev),
               scales=torch.empty(B * Hkv * (Nk // 128) * 1024, dtype=torch.uint8, device=dev),
               scale=torch.empty(1, dtype=torch.float32, device=dev))
    if workspace is None or workspace.numel() < 256:
        workspace = torch.empty(256, dtype=torch.uint8, device=dev)
    vt = _nvfp4(out)
    st = _lib.mpfa_quantize_v_fp4(_ptr(v), B, Nk, Hkv, D, ctypes.byref(vt), _ptr(workspace),
                                  workspace.numel(), _stream(dev))
    _check(st, "mpfa_quantize_v_fp4")
    out["_workspace"] = workspace
    return out


def prefill_fp4pv(qz, vt, *, causal, out=None, lse=None, want_lse=True):
    """The prefill with the full-FP4 PV of the ablation: q, k (and qbar) from
    quantize_qkv, vt from quantize_v_fp4.  Returns (o, lse) as prefill."""
    B, N, Hq, Hkv = qz["B"], qz["Nq"], qz["Hq"], qz["Hkv"]
    assert qz["Nk"] == N, "prefill takes N_q == N_k"
    assert qz.get("lse_shift") is None, "the full-FP4 PV kernel takes no key-side smoothing"
    dev = qz["q"]["codes"].device
    if out is None:
        out = torch.empty(B, N, Hq, D, dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
    qs, ks, vs = _nvfp4(qz["q"]), _nvfp4(qz["k"]), _nvfp4(vt)
    comp = qz["compensate"]
    rb = Rank1(qz["qbar"]["codes"].data_ptr(), qz["qbar"]["scales"].data_ptr()) if comp else None
    st = _lib.mpfa_prefill_fp4pv(ctypes.byref(qs), ctypes.byref(rb) if rb is not None else None,
                                 ctypes.byref(ks), ctypes.byref(vs), B, N, Hq, Hkv, D,
                                 int(bool(causal)), int(comp), int(qz["T"]), _ptr(out), _ptr(lse),
                                 _stream(dev))
    _check(st, "mpfa_prefill_fp4pv")
    return out, lse


def decode_workspace_bytes(B, Hq, Hkv, Lmax, kv_chunk=0) -> int:
    return int(_lib.mpfa_decode_workspace_size(B, Hq, Hkv, D, Lmax, kv_chunk))


def decode(q, cache, seqlens, *, compensate=True, T=2, kv_chunk=0, out=None, lse=None,
           want_lse=True, return_query_codes=False, workspace=None):
    """One decode step: q bf16 [B,Hq,128] against a cache from quantize_qkv
    (k and v given, q None), seqlens int32 [B] on the device.  A cache built
    with k_smooth carries its ``kbar``, which adds the smoothing's LSE term.
    Returns dict(o, lse, chunk[, q, qbar])."""
    B, Hq, _ = q.shape
    Hkv, Lmax = cache["Hkv"], cache["Nk"]
    dev = q.device
    assert q.dtype == torch.bfloat16 and q.is_contiguous()
    assert seqlens.dtype == torch.int32 and seqlens.device == dev
    if out is None:
        out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    ws_bytes = decode_workspace_bytes(B, Hq, Hkv, Lmax, kv_chunk)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ks = _nvfp4(cache["k"])
    vs = FP8(cache["v"]["codes"].data_ptr(), cache["v"]["scale"].data_ptr())
    res = dict(o=out, lse=lse)
    qq = rb = None
    if return_query_codes:
        res["q"] = dict(codes=torch.empty(B, Hq, 64, dtype=torch.uint8, device=dev),
                        scales=torch.empty(B, Hq, 8, dtype=torch.uint8, device=dev),
                        scale=torch.empty(1, dtype=torch.float32, device=dev))
        qq = _nvfp4(res["q"])
        if compensate:
            res["qbar"] = dict(codes=torch.empty(B, Hkv, T, 64, dtype=torch.uint8, device=dev),
                               scales=torch.empty(B, Hkv, T, 8, dtype=torch.uint8, device=dev))
            rb = Rank1(res["qbar"]["codes"].data_ptr(), res["qbar"]["scales"].data_ptr())
    used = ctypes.c_int(0)
    st = _lib.mpfa_decode(_ptr(q), ctypes.byref(ks), ctypes.byref(vs), _ptr(cache.get("kbar")),
                          _ptr(seqlens), B, Hq, Hkv,
                          D, Lmax, int(bool(compensate)), int(T), int(kv_chunk), _ptr(out),
                          _ptr(lse), ctypes.byref(qq) if qq is not None else None,
                          ctypes.byref(rb) if rb is not None else None, ctypes.byref(used),
                          _ptr(workspace), workspace.numel(), _stream(dev))
    _check(st, "mpfa_decode")
    res["chunk"] = used.value
    res["_workspace"] = workspace
    return res


def append_kv(k_new, v_new, cache, seqlens):
    """Quantize-on-append: k_new / v_new bf16 [B, n_new, Hkv, 128] on the
    device, quantized with the cache's own tensor scales and written into
    the cache (from quantize_qkv(None, k, v)) at rows seqlens[b] ..
    seqlens[b] + n_new - 1 (int32 [B] on the device, not advanced: pass
    seqlens + n_new to the next decode); a cache built with k_smooth has
    its ``kbar`` subtracted from the new keys first.  A sequence that would run past the
    cache is left as it is and get_error() then reports
    MPFA_ERR_INVALID_ARG."""
    B, n_new, Hkv, d = k_new.shape
    dev = k_new.device
    for t in (k_new, v_new):
        assert t.dtype == torch.bfloat16 and t.is_contiguous() and t.shape == (B, n_new, Hkv, D)
        assert t.device == dev
    assert seqlens.dtype == torch.int32 and seqlens.device == dev and seqlens.numel() == B
    assert cache["Hkv"] == Hkv and cache["B"] == B
    ks = _nvfp4(cache["k"])
    vs = FP8(cache["v"]["codes"].data_ptr(), cache["v"]["scale"].data_ptr())
    st = _lib.mpfa_append_kv(_ptr(k_new), _ptr(v_new), _ptr(seqlens), B, n_new, Hkv, d,
                             cache["Nk"], ctypes.byref(ks), ctypes.byref(vs),
                             _ptr(cache.get("kbar")), _stream(dev))
    _check(st, "mpfa_append_kv")
    return cache


# --------------------------------------------------------------------------
# layout utility (inspection only; not on the compute path)
# --------------------------------------------------------------------------

def untile_scales(tiled: torch.Tensor, rows: int) -> torch.Tensor:
    """Tiled block scales (rows*8 bytes) -> row-major [rows, 8]."""
    r = torch.arange(rows, device=tiled.device).view(-1, 1)
    j = torch.arange(8, device=tiled.device).view(1, -1)
    off = (r // 128) * 1024 + (j // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (j % 4)
    return tiled.view(-1)[off.view(-1)].view(rows, 8)


# --------------------------------------------------------------------------
# paged KV pool
# --------------------------------------------------------------------------

def quantize_pool(k_pages, v_pages, workspace=None):
    """A paged pool from bf16 K / V pages [num_pages, 128, Hkv, 128]: page p
    holds, for every KV head, 128 token rows (see include/mpfa.h)."""
    assert k_pages.shape[1] == 128 and v_pages.shape == k_pages.shape
    pool = quantize_qkv(None, k_pages, v_pages, workspace=workspace)
    pool["num_pages"] = k_pages.shape[0]
    return pool


def decode_paged(q, pool, block_table, seqlens, *, compensate=True, T=2, kv_chunk=0, out=None,
                 lse=None, want_lse=True, workspace=None):
    """Split-KV decode over a paged pool: block_table int32 [B, max_pages] on
    the device (page of each sequence's 128-token block), seqlens int32 [B].
    Returns dict(o, lse, chunk)."""
    B, Hq, _ = q.shape
    Hkv, num_pages = pool["Hkv"], pool["num_pages"]
    max_pages = block_table.shape[1]
    dev = q.device
    assert q.dtype == torch.bfloat16 and q.is_contiguous()
    assert block_table.dtype == torch.int32 and block_table.is_contiguous()
    assert block_table.shape[0] == B and block_table.device == dev
    assert seqlens.dtype == torch.int32 and seqlens.device == dev
    if out is None:
        out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    ws_bytes = decode_workspace_bytes(B, Hq, Hkv, 128 * max_pages, kv_chunk)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ks = _nvfp4(pool["k"])
    vs = FP8(pool["v"]["codes"].data_ptr(), pool["v"]["scale"].data_ptr())
    used = ctypes.c_int(0)
    st = _lib.mpfa_decode_paged(_ptr(q), ctypes.byref(ks), ctypes.byref(vs), _ptr(block_table),
                                num_pages, max_pages, _ptr(seqlens), B, Hq, Hkv, D,
                                int(bool(compensate)), int(T), int(kv_chunk), _ptr(out),
                                _ptr(lse), None, None, ctypes.byref(used), _ptr(workspace),
                                workspace.numel(), _stream(dev))
    _check(st, "mpfa_decode_paged")
    return dict(o=out, lse=lse, chunk=used.value, _workspace=workspace)


def append_kv_paged(k_new, v_new, pool, block_table, seqlens):
    """Quantize-on-append into a paged pool: token seqlens[b] + t of sequence
    b goes to row (seqlens[b] + t) % 128 of page block_table[b][(...) / 128],
    coded with the pool's own tensor scales."""
    B, n_new, Hkv, d = k_new.shape
    dev = k_new.device
    for t in (k_new, v_new):
        assert t.dtype == torch.bfloat16 and t.is_contiguous() and t.shape == (B, n_new, Hkv, D)
    assert block_table.dtype == torch.int32 and block_table.shape[0] == B
    assert seqlens.dtype == torch.int32 and seqlens.numel() == B
    ks = _nvfp4(pool["k"])
    vs = FP8(pool["v"]["codes"].data_ptr(), pool["v"]["scale"].data_ptr())
    st = _lib.mpfa_append_kv_paged(_ptr(k_new), _ptr(v_new), _ptr(seqlens), _ptr(block_table),
                                   pool["num_pages"], block_table.shape[1], B, n_new, Hkv, d,
                                   ctypes.byref(ks), ctypes.byref(vs), _stream(dev))
    _check(st, "mpfa_append_kv_paged")
    return pool
