"""The C-ABI library builds, loads and exports every symbol include/mpfa.h
declares (no compute calls: these run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mpfa.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mpfa_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._builder().build()
    return ctypes.CDLL(path)


def test_header_declares_entry_points():
    names = _declared()
    for n in ("mpfa_quantize_qkv", "mpfa_prefill", "mpfa_decode", "mpfa_get_error",
              "mpfa_status_string", "mpfa_quantize_workspace_size",
              "mpfa_decode_workspace_size", "mpfa_append_kv"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    lib.mpfa_status_string.restype = ctypes.c_char_p
    assert lib.mpfa_status_string(0) == b"MPFA_OK"
    assert lib.mpfa_status_string(4) == b"MPFA_ERR_TIMEOUT"


def test_last_cuda_error_starts_clear(lib):
    """The CUDA error behind an MPFA_ERR_CUDA is reported by name; before any
    CUDA failure on this thread it is cudaSuccess."""
    lib.mpfa_last_cuda_error.restype = ctypes.c_char_p
    assert lib.mpfa_last_cuda_error() == b"cudaSuccess"


def test_host_side_validation_without_gpu(lib):
    """Bad arguments are rejected on the host before anything is enqueued."""
    f = lib.mpfa_prefill
    f.restype = ctypes.c_int
    # d != 128 -> unsupported; null tensors -> invalid
    assert f(None, None, None, None, 1, 128, 1, 1, 64, 0, 0, 0, None, None, None, None) == 2
    assert f(None, None, None, None, 1, 128, 1, 1, 128, 0, 0, 0, None, None, None, None) == 1
    f4 = lib.mpfa_prefill_fp4pv
    f4.restype = ctypes.c_int
    assert f4(None, None, None, None, 1, 128, 1, 1, 64, 0, 0, 0, None, None, None) == 2
    assert f4(None, None, None, None, 1, 128, 1, 1, 128, 0, 0, 0, None, None, None) == 1
    v4 = lib.mpfa_quantize_v_fp4
    v4.restype = ctypes.c_int
    assert v4(None, 1, 128, 1, 64, None, None, ctypes.c_size_t(0), None) == 2
    assert v4(None, 1, 128, 1, 128, None, None, ctypes.c_size_t(0), None) == 1
    q = lib.mpfa_quantize_qkv
    q.restype = ctypes.c_int
    assert q(None, None, None, 1, 128, 128, 1, 1, 128, 0, 2, None, None, None, None, None, None,
             0, None) == 1
    assert q(None, None, None, 1, 128, 128, 1, 1, 96, 0, 2, None, None, None, None, None, None,
             0, None) == 2


def test_workspace_size_queries(lib):
    lib.mpfa_quantize_workspace_size.restype = ctypes.c_size_t
    n0 = lib.mpfa_quantize_workspace_size(1, 256, 384, 2, 1, 0, 0)
    n1 = lib.mpfa_quantize_workspace_size(1, 256, 384, 2, 1, 1, 0)
    n2 = lib.mpfa_quantize_workspace_size(1, 256, 384, 2, 1, 1, 1)
    assert n1 - n0 == 2 * 2 * 128 * 4                  # Q block means
    assert n2 - n1 == 1 * 3 * 3 * 128 * 4              # key block mean, max, min


def _fake(addr):
    return ctypes.c_void_p(addr)


def test_host_validation_rejects_bad_shapes_and_pointers(lib):
    """Every host-checkable fault returns before any CUDA call (these run
    with no GPU: a call that passed validation would fail with MPFA_ERR_CUDA)."""
    class NV(ctypes.Structure):
        _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                    ("tensor_scale", ctypes.c_void_p)]

    class F8(ctypes.Structure):
        _fields_ = [("codes", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p)]

    ok = 0x10000
    q = NV(ok, ok, ok)
    k = NV(ok, ok, ok)
    v = F8(ok, ok)
    f = lib.mpfa_prefill
    f.restype = ctypes.c_int
    R = ctypes.byref
    # N not a multiple of 128
    assert f(R(q), None, R(k), R(v), 1, 100, 4, 2, 128, 1, 0, 0, _fake(ok), None, None, None) == 1
    # Hq % Hkv != 0
    assert f(R(q), None, R(k), R(v), 1, 128, 5, 2, 128, 1, 0, 0, _fake(ok), None, None,
             None) == 1
    # misaligned output
    assert f(R(q), None, R(k), R(v), 1, 128, 4, 2, 128, 1, 0, 0, _fake(ok + 2), None, None,
             None) == 1
    # compensation without its terms, and T out of range
    assert f(R(q), None, R(k), R(v), 1, 128, 4, 2, 128, 1, 1, 2, _fake(ok), None, None,
             None) == 1
    assert f(R(q), None, R(k), R(v), 1, 128, 4, 2, 128, 1, 1, 3, _fake(ok), None, None,
             None) == 2
    d = lib.mpfa_decode
    d.restype = ctypes.c_int
    used = ctypes.c_int(0)
    # kv_chunk not a multiple of 128; Lmax not a multiple of 128
    assert d(_fake(ok), R(k), R(v), None, _fake(ok), 2, 8, 2, 128, 256, 1, 2, 100, _fake(ok), None,
             None, None, R(used), _fake(ok), 1 << 20, None) == 1
    assert d(_fake(ok), R(k), R(v), None, _fake(ok), 2, 8, 2, 128, 200, 1, 2, 0, _fake(ok), None,
             None, None, R(used), _fake(ok), 1 << 20, None) == 1
    # more than 16 query heads per KV head
    assert d(_fake(ok), R(k), R(v), None, _fake(ok), 2, 64, 2, 128, 256, 1, 2, 0, _fake(ok), None,
             None, None, R(used), _fake(ok), 1 << 20, None) == 2
    # 2^31 cache rows or more (B * Hkv * Lmax)
    assert d(_fake(ok), R(k), R(v), None, _fake(ok), 4096, 8, 8, 128, 1 << 16, 1, 2, 0, _fake(ok),
             None, None, None, R(used), _fake(ok), ctypes.c_size_t(1 << 50), None) == 1
    # 2^31 rows or more in prefill
    assert f(R(q), None, R(k), R(v), 1024, 1 << 21, 4, 2, 128, 1, 0, 0, _fake(ok), None,
             None, None) == 1
    # and in quantize (q rows; k/v rows)
    qq = lib.mpfa_quantize_qkv
    qq.restype = ctypes.c_int
    assert qq(_fake(ok), None, None, 1024, 1 << 21, 0, 4, 2, 128, 0, 2, R(q), None, None, None,
              None, _fake(ok), ctypes.c_size_t(1 << 50), None) == 1
    assert qq(None, _fake(ok), _fake(ok), 1024, 0, 1 << 21, 4, 2, 128, 0, 2, None, None, R(k),
              R(v), None, _fake(ok), ctypes.c_size_t(1 << 50), None) == 1

    # key-side smoothing: needs the keys and a kbar buffer; its LSE term needs the queries
    class KS(ctypes.Structure):
        _fields_ = [("kbar", ctypes.c_void_p), ("lse_shift", ctypes.c_void_p)]

    big = ctypes.c_size_t(1 << 40)
    assert qq(_fake(ok), None, None, 1, 256, 256, 4, 2, 128, 0, 2, R(q), None, None, None,
              R(KS(ok, ok)), _fake(ok), big, None) == 1
    assert qq(None, _fake(ok), None, 1, 0, 256, 4, 2, 128, 0, 2, None, None, R(k), None,
              R(KS(ok, ok)), _fake(ok), big, None) == 1
    assert qq(None, _fake(ok), None, 1, 0, 256, 4, 2, 128, 0, 2, None, None, R(k), None,
              R(KS(None, None)), _fake(ok), big, None) == 1
    # a workspace without room for the key statistics
    lib.mpfa_quantize_workspace_size.restype = ctypes.c_size_t
    need = lib.mpfa_quantize_workspace_size(1, 0, 256, 4, 2, 0, 1)
    assert qq(None, _fake(ok), None, 1, 0, 256, 4, 2, 128, 0, 2, None, None, R(k), None,
              R(KS(ok, None)), _fake(ok), ctypes.c_size_t(need - 1), None) == 1


def test_append_kv_host_validation(lib):
    """mpfa_append_kv rejects bad shapes and pointers before any CUDA call."""
    class NV(ctypes.Structure):
        _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                    ("tensor_scale", ctypes.c_void_p)]

    class F8(ctypes.Structure):
        _fields_ = [("codes", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p)]

    ok = 0x10000
    k, v, R = NV(ok, ok, ok), F8(ok, ok), ctypes.byref
    a = lib.mpfa_append_kv
    a.restype = ctypes.c_int
    args = dict(kn=_fake(ok), vn=_fake(ok), sl=_fake(ok), B=2, n=1, H=2, d=128, L=256)

    def call(**kw):
        x = {**args, **kw}
        return a(x["kn"], x["vn"], x["sl"], x["B"], x["n"], x["H"], x["d"], x["L"],
                 kw.get("k", R(k)), kw.get("v", R(v)), None, None)

    assert call(d=64) == 2                      # head dim other than 128
    assert call(kn=None) == 1                   # null new K
    assert call(vn=_fake(ok + 8)) == 1          # misaligned new V
    assert call(sl=None) == 1                   # no lengths
    assert call(L=200) == 1                     # Lmax not a multiple of 128
    assert call(n=0) == 1                       # nothing to append
    assert call(n=257) == 1                     # more new tokens than the cache holds
    assert call(k=None) == 1                    # no cache
    assert call(k=R(NV(ok, None, ok))) == 1     # cache without scales
    assert call(v=R(F8(ok, None))) == 1         # cache without its tensor scale
    assert call(B=4096, H=8, L=1 << 16) == 1    # 2^31 cache rows or more



def test_paged_entry_points_host_validation(lib):
    """mpfa_decode_paged / mpfa_append_kv_paged reject a missing block table,
    non-positive pool sizes and pools of 2^31 rows or more before any CUDA
    call."""
    class NV(ctypes.Structure):
        _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                    ("tensor_scale", ctypes.c_void_p)]

    class F8(ctypes.Structure):
        _fields_ = [("codes", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p)]

    ok = 0x10000
    k, v, R = NV(ok, ok, ok), F8(ok, ok), ctypes.byref
    d = lib.mpfa_decode_paged
    d.restype = ctypes.c_int
    used = ctypes.c_int(0)

    def dec(table=_fake(ok), pages=8, maxp=4, dh=128):
        return d(_fake(ok), R(k), R(v), table, pages, maxp, _fake(ok), 2, 8, 2, dh, 1, 2, 0,
                 _fake(ok), None, None, None, R(used), _fake(ok), ctypes.c_size_t(1 << 40), None)

    assert dec(dh=64) == 2
    assert dec(table=None) == 1
    assert dec(pages=0) == 1
    assert dec(maxp=0) == 1
    assert dec(pages=1 << 24) == 1        # 2^24 pages x 2 heads x 128 rows = 2^32
    a = lib.mpfa_append_kv_paged
    a.restype = ctypes.c_int

    def app(table=_fake(ok), pages=8, maxp=4, n=1):
        return a(_fake(ok), _fake(ok), _fake(ok), table, pages, maxp, 2, n, 2, 128, R(k), R(v), None)

    assert app(table=None) == 1
    assert app(pages=-1) == 1
    assert app(n=513) == 1                # more new tokens than 4 pages hold
    assert app(pages=1 << 24) == 1
