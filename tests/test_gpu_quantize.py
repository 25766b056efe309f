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


def _edge_column_q(rng, n_blocks=2, Hq=2, big=False):
    """Q [1, 128 n_blocks, Hq, 128] bf16 whose columns exercise every path of
    the exact block mean: ordinary values, cancellation, a spread of more
    than 26 binades, tiny and subnormal values (subnormal means), an all-zero
    column, one nonzero value, an exact tie, and (big=True) values near the
    bf16 maximum."""
    x = rng.standard_normal((n_blocks * 128, Hq, 128)).astype(np.float32)
    r = np.arange(n_blocks * 128)
    x[:, :, 8] = np.where(r % 4 == 0, 100.0, np.where(r % 4 == 2, -100.0, 1e-3))[:, None] * (
        1.0 + np.where(r % 2 == 1, 1.0, 0.0)[:, None] * x[:, :, 8])
    x[:, :, 9] = x[:, :, 9] * np.exp2(rng.integers(-22, 22, (n_blocks * 128, Hq)))
    x[:, :, 10] = 1e-37 * x[:, :, 10]
    x[:, :, 11] = 3e-39 * x[:, :, 11]            # bf16 subnormals
    x[:, :, 12] = 0.0
    x[:, :, 13] = 0.0
    x[::128, :, 13] = -2.5
    x[:, :, 14] = 1.0
    x[::128, :, 14] = 1.0 + 2.0 ** -7               # the exact mean lies on a tie
    x[:, :, 15] = np.exp2(-10.0) * (1.0 + (r % 128)[:, None] / 128.0)
    x[5::128, :, 15] = 192.0                        # 17 binades above the rest
    x[:, :, 17] = np.where(r % 3 == 0, 1.0, -np.exp2(-26.0))[:, None]   # spread 26
    x[:, :, 18] = np.where(r % 3 == 0, 1.0, np.exp2(-27.0))[:, None]    # spread 27
    if big:
        x[:, :, 16] = 2.5e38 * (0.5 + 0.5 * np.abs(x[:, :, 16]) / (1 + np.abs(x[:, :, 16])))
    return torch.from_numpy(x[None]).to(torch.bfloat16)


@pytest.mark.parametrize("big", [False, True])
def test_quantize_block_means_edge_columns(big):
    """The fp32 block means the kernels leave in the workspace equal the
    oracle's correctly rounded means bit for bit, and the codes and tensor
    scales that follow from them match too."""
    import flashattention_mpfa_quantize_gb300 as mp
    import oracle as orc
    rng = np.random.default_rng(11)
    Q = _edge_column_q(rng, big=big)
    K = torch.from_numpy(rng.standard_normal((1, 256, 1, 128)).astype(np.float32)).to(torch.bfloat16)
    dev = torch.device("cuda:0")
    qz = mp.quantize_qkv(Q.to(dev), K.to(dev), K.to(dev), compensate=True, T=2)
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    B, N, Hq = 1, Q.shape[1], Q.shape[2]
    ws = qz["_workspace"][256:256 + B * Hq * (N // 128) * 128 * 4].cpu().numpy().view(np.float32)
    got = ws.reshape(Hq, N // 128, 128)
    xs = Q.float().numpy()[0]
    for h in range(Hq):
        want, _ = orc.block_means(xs[:, h, :], 128)
        np.testing.assert_array_equal(got[h].view(np.uint32), want.view(np.uint32))
    _check(qz, oracle_quantize(Q, K, K, True, 2), True)


@pytest.mark.parametrize("scale", [1e-36, 1e-26, 1e31])
def test_quantize_extreme_magnitudes(scale):
    """Tensors scaled so that the block divisors fall outside [2^-90, 2^100]
    (tiny and huge scales take the IEEE-division path, the others the
    reciprocal-and-correction path, some blocks of each in one tensor):
    codes, block scales and tensor scales stay bit-exact with the oracle."""
    import flashattention_mpfa_quantize_gb300 as mp
    cfg = mi.custom_prefill(1, 2, 1, 256, False, k_outliers=2, v_outlier_p=0.01, q_offset=True)
    Q, K, V = mi.prefill_inputs(cfg, "cpu", 5)
    # per-row magnitudes spread over 2^±10 around `scale` (bf16 subnormals
    # for the smallest, far from overflow for the largest)
    rng = np.random.default_rng(2)
    def spread(t):
        f = np.exp2(rng.integers(-10, 11, size=(1, t.shape[1], t.shape[2], 1))).astype(np.float32)
        x = t.float().numpy() * f * np.float32(scale)
        assert np.isfinite(x).all()
        return torch.from_numpy(x).to(torch.bfloat16)
    Q, K, V = spread(Q), spread(K), spread(V)
    dev = torch.device("cuda:0")
    for comp in (False, True):
        qz = mp.quantize_qkv(Q.to(dev), K.to(dev), V.to(dev), compensate=comp, T=2)
        torch.cuda.synchronize()
        assert mp.get_error() == 0
        _check(qz, oracle_quantize(Q, K, V, comp, 2), comp)
