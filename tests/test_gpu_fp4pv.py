"""GPU parity of the full-FP4 PV ablation (the MpFA abstract weighs QK4PV8
against full FP4): the V^T quantize kernel bit for bit against the oracle's
NVFP4 of V^T along the keys, and the FP4-PV prefill kernel against the
oracle's emulation of the same pipeline (P in NVFP4 per 16 keys with the
fixed tensor scale, V^T in NVFP4), at the prefill tests' tolerances."""
import numpy as np
import pytest
import torch

import mpfa_inputs as mi
import oracle as orc
from helpers import fp4p_flip_allowance, np_f32, oracle_quantize, rel_l2, tiled_to_rows

pytestmark = pytest.mark.gpu

O_MAX_ABS = 2e-2
O_REL_L2 = 5e-3
LSE_ABS = 2e-3


def _vt_check(V, vt):
    """GPU V^T codes, tiled block scales and tensor scale against the oracle."""
    ref = orc.quantize_v_fp4(np_f32(V))
    B, N, Hkv, d = V.shape
    assert vt["scale"].item() == ref["s_v"]
    np.testing.assert_array_equal(vt["codes"].cpu().numpy(), ref["vc4"])
    nt = N // 128
    rows = tiled_to_rows(vt["scales"].cpu().numpy(), B * Hkv * nt * 128)
    got = rows.reshape(B * Hkv, nt, 128, 8)
    want = ref["vs4"].reshape(B * Hkv, d, nt, 8).transpose(0, 2, 1, 3)
    np.testing.assert_array_equal(got, want)
    return ref


@pytest.mark.parametrize("cfg", [mi.PREFILL["tiny_n256"],
                                 mi.custom_prefill(2, 6, 3, 640, True, k_outliers=2,
                                                   v_outlier_p=0.01, q_offset=True)],
                         ids=["tiny_n256", "b2_hkv3_n640_outliers"])
def test_quantize_v_fp4_bit_exact(cfg):
    import flashattention_mpfa_quantize_gb300 as mp
    _, _, V = mi.prefill_inputs(cfg, "cpu", 4)
    vt = mp.quantize_v_fp4(V.to("cuda:0"))
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    _vt_check(V, vt)


def test_quantize_v_fp4_zero_tensor():
    import flashattention_mpfa_quantize_gb300 as mp
    V = torch.zeros(1, 256, 2, 128, dtype=torch.bfloat16)
    vt = mp.quantize_v_fp4(V.to("cuda:0"))
    torch.cuda.synchronize()
    _vt_check(V, vt)
    assert not vt["codes"].any()


def _fp4pv_case(cfg, compensate, T=2, seed=0, heads=None):
    import flashattention_mpfa_quantize_gb300 as mp
    Q, K, V = mi.prefill_inputs(cfg, "cpu", seed)
    dev = torch.device("cuda:0")
    Vd = V.to(dev)
    qz = mp.quantize_qkv(Q.to(dev), K.to(dev), Vd, compensate=compensate, T=T)
    vt = mp.quantize_v_fp4(Vd)
    o, lse = mp.prefill_fp4pv(qz, vt, causal=cfg.causal)
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    ref = oracle_quantize(Q, K, None, compensate, T)
    vz = _vt_check(V, vt)
    em = orc.prefill_emulate(ref["q"], ref["k"], vz, causal=cfg.causal, heads=heads)
    o_gpu, lse_gpu = np_f32(o), lse.cpu().numpy()
    got, want, lg, lw = [], [], [], []
    for (b, h), (oe, le) in em.items():
        got.append(o_gpu[b, :, h, :])
        want.append(orc.bf16_bits_to_float(orc.bf16_round(oe)))
        lg.append(lse_gpu[b, h])
        lw.append(le)
    return np.concatenate(got), np.concatenate(want), np.concatenate(lg), np.concatenate(lw)


def _assert_close(got, want, lg, lw):
    err = np.abs(got - want)
    assert np.isfinite(got).all()
    assert err.max() <= O_MAX_ABS, (err.max(), np.unravel_index(err.argmax(), err.shape))
    assert rel_l2(got, want) <= O_REL_L2, rel_l2(got, want)
    assert np.abs(lg - lw).max() <= LSE_ABS, np.abs(lg - lw).max()


@pytest.mark.parametrize("compensate", [False, True])
def test_prefill_fp4pv_tiny(compensate):
    _assert_close(*_fp4pv_case(mi.PREFILL["tiny_n256"], compensate))


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_fp4pv_gqa_multitile(causal):
    cfg = mi.custom_prefill(2, 4, 2, 640, causal, k_outliers=1, v_outlier_p=0.001,
                            q_offset=True)
    _assert_close(*_fp4pv_case(cfg, True, 2, seed=5))


def test_prefill_fp4pv_many_items_per_cta():
    """More items than SMs, so the carries across a CTA's items (P banks,
    the P and V^T scale slots, the ones operand copied once) take part."""
    cfg = mi.custom_prefill(2, 32, 4, 1024, True, k_outliers=1, v_outlier_p=0.001,
                            q_offset=True)
    heads = [(0, 0), (0, 13), (1, 7), (1, 31)]
    _assert_close(*_fp4pv_case(cfg, True, 2, seed=11, heads=heads))


def test_prefill_fp4pv_single_tile_items():
    """One-tile items back to back (every tile starts an item).  Causal rows
    with few keys: one FP4 decision near a rounding boundary moves O by up to
    a few 1e-2 here (and the LSE by up to ~2e-2), so O and the LSE are
    checked against the oracle within O_MAX_ABS and LSE_ABS plus the row's
    flip allowance."""
    import flashattention_mpfa_quantize_gb300 as mp
    cfg = mi.custom_prefill(2, 128, 8, 128, True, k_outliers=1, v_outlier_p=0.001,
                            q_offset=True)
    heads = [(0, 0), (0, 77), (1, 3), (1, 127)]
    Q, K, V = mi.prefill_inputs(cfg, "cpu", 12)
    dev = torch.device("cuda:0")
    Vd = V.to(dev)
    qz = mp.quantize_qkv(Q.to(dev), K.to(dev), Vd, compensate=True, T=2)
    vt = mp.quantize_v_fp4(Vd)
    o, lse = mp.prefill_fp4pv(qz, vt, causal=True)
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    ref = oracle_quantize(Q, K, None, True, 2)
    vz = _vt_check(V, vt)
    em = orc.prefill_emulate(ref["q"], ref["k"], vz, causal=True, heads=heads)
    o_gpu, lse_gpu = np_f32(o), lse.cpu().numpy()
    g = cfg.Hq // cfg.Hkv
    got, want = [], []
    for (b, h), (oe, le) in em.items():
        w = orc.bf16_bits_to_float(orc.bf16_round(oe))
        allow, allow_lse = fp4p_flip_allowance(ref["q"], ref["k"], vz, b, h, g)
        err = np.abs(o_gpu[b, :, h, :] - w)
        assert (err <= O_MAX_ABS + allow).all(), (err.max(), (err - allow).max())
        lerr = np.abs(lse_gpu[b, h] - le)
        assert (lerr <= LSE_ABS + allow_lse).all(), (lerr.max(), (lerr - allow_lse).max())
        got.append(o_gpu[b, :, h, :])
        want.append(w)
    got, want = np.concatenate(got), np.concatenate(want)
    assert np.isfinite(got).all()
    assert rel_l2(got, want) <= O_REL_L2, rel_l2(got, want)
