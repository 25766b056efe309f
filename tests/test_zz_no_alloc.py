"""mpfa_quantize_qkv_noalloc (the quantization entry point for callers that
cannot allocate device memory, e.g. a serving process whose HBM is owned by
its own pool) against mpfa_quantize_qkv with a caller workspace, called
through the C ABI twice in a row: codes, block scales and tensor scales must
be identical.  The second call uses inputs with a smaller amax than the first,
so state left in the shared scratch array by the first call would show.

This file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

import mpfa_inputs as mi

pytestmark = pytest.mark.gpu


def _call_noalloc(mp, Q, K, V, compensate, T):
    lib = mp.lib
    f = lib.mpfa_quantize_qkv_noalloc
    f.restype = ctypes.c_int
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, P, I, I, I, I, I, I, I, I, ctypes.POINTER(mp.NVFP4),
                  ctypes.POINTER(mp.Rank1), ctypes.POINTER(mp.NVFP4), ctypes.POINTER(mp.FP8), P]
    B, N, Hq, _ = Q.shape
    Hkv = K.shape[2]
    dev = Q.device
    q = mp.alloc_nvfp4((B, Hq, N), dev)
    k = mp.alloc_nvfp4((B, Hkv, N), dev)
    v = dict(codes=torch.empty(B, Hkv, N, 128, dtype=torch.uint8, device=dev),
             scale=torch.empty(1, dtype=torch.float32, device=dev))
    qb = dict(codes=torch.empty(B, Hq, N // 128, T, 64, dtype=torch.uint8, device=dev),
              scales=torch.empty(B, Hq, N // 128, T, 8, dtype=torch.uint8, device=dev))
    qs = mp.NVFP4(q["codes"].data_ptr(), q["scales"].data_ptr(), q["scale"].data_ptr())
    ks = mp.NVFP4(k["codes"].data_ptr(), k["scales"].data_ptr(), k["scale"].data_ptr())
    vs = mp.FP8(v["codes"].data_ptr(), v["scale"].data_ptr())
    rb = mp.Rank1(qb["codes"].data_ptr(), qb["scales"].data_ptr())
    st = f(Q.data_ptr(), K.data_ptr(), V.data_ptr(), B, N, N, Hq, Hkv, 128, int(compensate), T,
           ctypes.byref(qs), ctypes.byref(rb) if compensate else None, ctypes.byref(ks),
           ctypes.byref(vs), torch.cuda.current_stream(dev).cuda_stream)
    assert st == 0, mp.lib.mpfa_status_string(st)
    return dict(q=q, k=k, v=v, qbar=qb if compensate else None)


def _same(a, b, compensate):
    for name in ("q", "k"):
        assert torch.equal(a[name]["codes"], b[name]["codes"])
        assert torch.equal(a[name]["scales"], b[name]["scales"])
        assert torch.equal(a[name]["scale"], b[name]["scale"])
    assert torch.equal(a["v"]["codes"], b["v"]["codes"])
    assert torch.equal(a["v"]["scale"], b["v"]["scale"])
    if compensate:
        assert torch.equal(a["qbar"]["codes"], b["qbar"]["codes"])
        assert torch.equal(a["qbar"]["scales"], b["qbar"]["scales"])


@pytest.mark.parametrize("compensate", [True, False])
def test_noalloc_matches_workspace_entry_point_twice(compensate):
    import flashattention_mpfa_quantize_gb300 as mp
    dev = torch.device("cuda:0")
    cfg = mi.custom_prefill(2, 4, 2, 384, True, k_outliers=2, v_outlier_p=0.01, q_offset=True)
    for seed, scale in ((0, 4.0), (1, 0.5)):   # second call: smaller amax
        Q, K, V = (t.to(dev) for t in mi.prefill_inputs(cfg, "cpu", seed))
        Q, K, V = ((t.float() * scale).to(torch.bfloat16).contiguous() for t in (Q, K, V))
        want = mp.quantize_qkv(Q, K, V, compensate=compensate, T=2)
        got = _call_noalloc(mp, Q, K, V, compensate, 2)
        torch.cuda.synchronize()
        assert mp.get_error() == 0
        _same(got, want, compensate)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import flashattention_mpfa_quantize_gb300 as mp
    dev = torch.device("cuda:0")
    # 40 heads x 131072 rows = 40960 query blocks > 32768: rejected, nothing enqueued
    f = mp.lib.mpfa_quantize_qkv_noalloc
    f.restype = ctypes.c_int
    q = torch.empty(16, dtype=torch.bfloat16, device=dev)
    dummy = mp.NVFP4(q.data_ptr(), q.data_ptr(), q.data_ptr())
    rb = mp.Rank1(q.data_ptr(), q.data_ptr())
    st = f(ctypes.c_void_p(q.data_ptr()), None, None, 1, 131072, 0, 40, 8, 128, 1, 2,
           ctypes.byref(dummy), ctypes.byref(rb), None, None,
           ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    assert st == mp.ERR_INVALID_ARG
