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
from helpers import (fp4p_first_tile_allowance, fp4p_flip_allowance, np_f32,
                     oracle_quantize, rel_l2, tiled_to_rows)

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


def _amax_bf16_chunks(t):
    m = 0
    for b in range(t.shape[0]):
        bits = t[b].contiguous().view(torch.int16).cpu().numpy().view(np.uint16) & 0x7FFF
        m = max(m, int(bits.max()))
    return np.uint32(m << 16).view(np.float32)


def _fp4pv_fullsize(cfg, heads, seed=0):
    """The benchmark workload at full size, as bench.py's PV ablation runs
    it: Vᵀ codes and scales of the sampled KV heads bit for bit, and sampled
    query rows (first rows, tile boundaries, the last rows, random ones)
    emulated one by one.  Rows below 128 see only the first key tile, where
    one FP4 decision can move a short row's O; they get the flip allowance."""
    import flashattention_mpfa_quantize_gb300 as mp
    dev = torch.device("cuda:0")
    Q, K, V = mi.prefill_inputs(cfg, dev, seed)
    qz = mp.quantize_qkv(Q, K, None, compensate=True, T=2)
    vt = mp.quantize_v_fp4(V)
    o, lse = mp.prefill_fp4pv(qz, vt, causal=cfg.causal)
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    B, N, Hq, Hkv, g = cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.Hq // cfg.Hkv
    s_q, s_k = qz["q"]["scale"].item(), qz["k"]["scale"].item()
    s_v = orc.tensor_scale(_amax_bf16_chunks(V), 2688.0)
    assert vt["scale"].item() == s_v
    rng = np.random.default_rng(7)
    rows = np.array(sorted({0, 1, 2, 63, 100, 127, 128, 129, 255, 256, N // 2, N - 129,
                            N - 128, N - 1} | set(rng.integers(0, N, 6).tolist())), np.int64)
    cs = orc.score_scale_log2(np.float32(s_q), np.float32(s_k))
    nt = N // 128
    for (b, h) in heads:
        hk = h // g
        vc, vs = orc.nvfp4_quantize(np.ascontiguousarray(np_f32(V[b, :, hk, :]).T), np.float32(s_v))
        np.testing.assert_array_equal(vt["codes"][b, hk].cpu().numpy(), vc)
        t0 = (b * Hkv + hk) * nt * 1024
        got_s = tiled_to_rows(vt["scales"][t0:t0 + nt * 1024].cpu().numpy(), nt * 128)
        np.testing.assert_array_equal(got_s.reshape(nt, 128, 8).transpose(1, 0, 2).reshape(128, -1),
                                      vs)
        mb, xp = orc.block_means(np_f32(Q[b, :, h, :]), 128)
        qc, qs = orc.nvfp4_quantize(xp, np.float32(s_q))
        tc, ts = orc.rank_one_terms(mb, np.float32(s_q), 2)
        np.testing.assert_array_equal(qz["q"]["codes"][b, h].cpu().numpy(), qc)
        kc, ks = orc.nvfp4_quantize(np_f32(K[b, :, hk, :]), np.float32(s_k))
        q = orc.nvfp4_dequant(qc, qs)
        qadd = np.repeat(sum(orc.nvfp4_dequant(np.ascontiguousarray(tc[:, t]),
                                               np.ascontiguousarray(ts[:, t])) for t in range(2)),
                         128, axis=0)
        k = orc.nvfp4_dequant(kc, ks)
        v = orc.nvfp4_dequant(vc, vs).T
        oe, le = orc.attn_online(q, qadd, k, v, score_scale=cs, out_scale=float(s_v),
                                 causal=cfg.causal, round_p=2, rows=rows)
        want = orc.bf16_bits_to_float(orc.bf16_round(oe))
        got = np_f32(o[b, rows, h, :])
        lg = lse[b, h, rows].cpu().numpy()
        allow = np.zeros_like(want)
        allow_lse = np.zeros(len(rows))
        first = rows < 128
        a_o, a_l = fp4p_first_tile_allowance((q + qadd)[rows[first]], k, v * np.float64(s_v),
                                             cs, rows[first])
        allow[first], allow_lse[first] = a_o, a_l
        assert np.isfinite(got).all()
        err = np.abs(got - want)
        assert (err <= O_MAX_ABS + allow).all(), (err.max(), (err - allow).max())
        assert (np.abs(lg - le) <= LSE_ABS + allow_lse).all(), np.abs(lg - le).max()
        assert rel_l2(got, want) <= O_REL_L2, rel_l2(got, want)


def test_fp4pv_fullsize_llama8b_n16k_causal():
    _fp4pv_fullsize(mi.PREFILL["llama8b_n16k_causal"], [(0, 0), (0, 31)])


def test_fp4pv_fullsize_qwen14b_n128k_causal():
    _fp4pv_fullsize(mi.PREFILL["qwen14b_n128k_causal"], [(0, 0), (0, 39)])
