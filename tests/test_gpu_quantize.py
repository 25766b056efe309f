"""GPU parity: the quantization kernels against the oracle, bit for bit
(codes, block scales, tensor scales, rank-one terms)."""
import numpy as np
import pytest
import torch

import mpfa_inputs as mi
from helpers import oracle_quantize, tiled_to_rows

pytestmark = pytest.mark.gpu


def _run(cfg, compensate, T, seed=0):
    import flashattention_mpfa_quantize_gb300 as mp
    Q, K, V = mi.prefill_inputs(cfg, "cpu", seed)
    dev = torch.device("cuda:0")
    qz = mp.quantize_qkv(Q.to(dev), K.to(dev), V.to(dev), compensate=compensate, T=T)
    torch.cuda.synchronize()
    ref = oracle_quantize(Q, K, V, compensate, T)
    return qz, ref


def _check(qz, ref, compensate):
    B, Hq, N, Hkv = qz["B"], qz["Hq"], qz["Nq"], qz["Hkv"]
    q = ref["q"]
    assert qz["q"]["scale"].item() == q["s_q"]
    np.testing.assert_array_equal(qz["q"]["codes"].cpu().numpy(), q["qc"])
    np.testing.assert_array_equal(
        tiled_to_rows(qz["q"]["scales"].cpu().numpy(), B * Hq * N), q["qs"].reshape(-1, 8))
    if compensate:
        np.testing.assert_array_equal(qz["qbar"]["codes"].cpu().numpy(), q["qbc"])
        np.testing.assert_array_equal(qz["qbar"]["scales"].cpu().numpy(), q["qbs"])
    k = ref["k"]
    assert qz["k"]["scale"].item() == k["s_k"]
    np.testing.assert_array_equal(qz["k"]["codes"].cpu().numpy(), k["kc"])
    np.testing.assert_array_equal(
        tiled_to_rows(qz["k"]["scales"].cpu().numpy(), B * Hkv * N), k["ks"].reshape(-1, 8))
    v = ref["v"]
    assert qz["v"]["scale"].item() == v["s_v"]
    np.testing.assert_array_equal(qz["v"]["codes"].cpu().numpy(), v["vc"])


@pytest.mark.parametrize("name", ["tiny_n256", "tiny_n256_qoffset"])
@pytest.mark.parametrize("compensate,T", [(False, 2), (True, 1), (True, 2)])
def test_quantize_tiny_bit_exact(name, compensate, T):
    qz, ref = _run(mi.PREFILL[name], compensate, T)
    _check(qz, ref, compensate)


@pytest.mark.parametrize("compensate", [False, True])
def test_quantize_gqa_multi_batch_bit_exact(compensate):
    cfg = mi.custom_prefill(2, 6, 2, 640, True, k_outliers=2, v_outlier_p=0.01, q_offset=True)
    qz, ref = _run(cfg, compensate, 2, seed=3)
    _check(qz, ref, compensate)


def test_quantize_zero_tensor():
    import flashattention_mpfa_quantize_gb300 as mp
    dev = torch.device("cuda:0")
    z = torch.zeros(1, 128, 1, 128, dtype=torch.bfloat16, device=dev)
    qz = mp.quantize_qkv(z, z, z, compensate=True, T=2)
    torch.cuda.synchronize()
    assert qz["q"]["scale"].item() == 1.0 and qz["k"]["scale"].item() == 1.0
    assert qz["v"]["scale"].item() == 1.0
    assert int(qz["q"]["codes"].sum()) == 0 and int(qz["k"]["scales"].sum()) == 0
    assert int(qz["v"]["codes"].sum()) == 0


def test_quantize_kv_only_cache():
    """q = None quantizes a KV cache alone (the decode producer)."""
    import flashattention_mpfa_quantize_gb300 as mp
    cfg = mi.custom_decode(3, 8, 2, 256, 100, 256)
    _, K, V, _ = mi.decode_inputs(cfg, "cpu", 1)
    dev = torch.device("cuda:0")
    qz = mp.quantize_qkv(None, K.to(dev), V.to(dev))
    torch.cuda.synchronize()
    ref = oracle_quantize(None, K, V, False, 2)
    np.testing.assert_array_equal(qz["k"]["codes"].cpu().numpy(), ref["k"]["kc"])
    np.testing.assert_array_equal(
        tiled_to_rows(qz["k"]["scales"].cpu().numpy(), 3 * 2 * 256), ref["k"]["ks"].reshape(-1, 8))
    np.testing.assert_array_equal(qz["v"]["codes"].cpu().numpy(), ref["v"]["vc"])
