"""Failure detection without a GPU fault: a kernel's bounded barrier wait that
runs out records MPFA_ERR_TIMEOUT in the device status word, mpfa_get_error
reports and clears it, and the context stays usable for real work."""
import ctypes

import numpy as np
import pytest
import torch

import mpfa_inputs as mi

pytestmark = pytest.mark.gpu


def test_bounded_wait_expiry_is_reported_and_context_survives():
    import flashattention_mpfa_quantize_gb300 as mp
    dev = torch.device("cuda:0")
    lib = mp.lib
    lib.mpfa_selftest_wait_timeout.restype = ctypes.c_int
    lib.mpfa_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p]
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    assert mp.get_error() == mp.OK
    assert lib.mpfa_selftest_wait_timeout(50_000_000, stream) == mp.OK   # 50 ms
    assert mp.get_error() == mp.ERR_TIMEOUT
    assert mp.get_error() == mp.OK                                         # cleared
    # the context still runs the real path correctly
    cfg = mi.PREFILL["tiny_n256"]
    Q, K, V = (t.to(dev) for t in mi.prefill_inputs(cfg, "cpu", 0))
    qz = mp.quantize_qkv(Q, K, V, compensate=True, T=2)
    o, lse = mp.prefill(qz, causal=False)
    torch.cuda.synchronize()
    assert mp.get_error() == mp.OK
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_selftest_rejects_bad_limits():
    import flashattention_mpfa_quantize_gb300 as mp
    lib = mp.lib
    lib.mpfa_selftest_wait_timeout.restype = ctypes.c_int
    lib.mpfa_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p]
    assert lib.mpfa_selftest_wait_timeout(0, None) == mp.ERR_INVALID_ARG
    assert lib.mpfa_selftest_wait_timeout(3_000_000_000, None) == mp.ERR_INVALID_ARG
