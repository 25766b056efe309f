"""GPU parity of key-side smoothing (K' = K - kbar, an addition to the pages'
method resting on the softmax's invariance to one shift of a row's logits)
against the oracle: kbar, the K' codes, block scales and s_k bit for bit;
the per-row LSE term within 1e-4; prefill and split-KV decode O within the
usual tolerances (max-abs 2e-2, rel-L2 5e-3) and LSE within 2e-3 of the
oracle's emulation on its own smoothed codes; quantize-on-append into a
smoothed cache bit for bit."""
import numpy as np
import pytest
import torch

import mpfa_inputs as mi
import oracle as orc
from helpers import np_f32, rel_l2, tiled_to_rows

pytestmark = pytest.mark.gpu

O_MAX_ABS = 2e-2
O_REL_L2 = 5e-3
LSE_ABS = 2e-3
SHIFT_ABS = 1e-4


def _quantize(cfg, compensate, T, seed=0):
    import flashattention_mpfa_quantize_gb300 as mp
    Q, K, V = mi.prefill_inputs(cfg, "cpu", seed)
    dev = torch.device("cuda:0")
    z = mp.quantize_qkv(Q.to(dev), K.to(dev), V.to(dev), compensate=compensate, T=T,
                        k_smooth=True)
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    qz = orc.quantize_q_prefill(np_f32(Q), compensate, T)
    kz = orc.quantize_k(np_f32(K), smooth=True)
    vz = orc.quantize_v(np_f32(V))
    return z, qz, kz, vz


def _check_codes(z, qz, kz):
    B, Hq, N, Hkv = z["B"], z["Hq"], z["Nq"], z["Hkv"]
    np.testing.assert_array_equal(z["kbar"].cpu().numpy(), kz["kbar"])
    assert z["k"]["scale"].item() == kz["s_k"]
    np.testing.assert_array_equal(z["k"]["codes"].cpu().numpy(), kz["kc"])
    np.testing.assert_array_equal(
        tiled_to_rows(z["k"]["scales"].cpu().numpy(), B * Hkv * N), kz["ks"].reshape(-1, 8))
    g = Hq // Hkv
    sh = z["lse_shift"].cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            want = orc.lse_shift(qz, kz, b, h, g)
            assert np.abs(sh[b, h] - want).max() <= SHIFT_ABS * max(1.0, np.abs(want).max())


@pytest.mark.parametrize("compensate,T", [(False, 2), (True, 1), (True, 2)])
def test_ksmooth_codes_tiny(compensate, T):
    z, qz, kz, _ = _quantize(mi.PREFILL["tiny_n256"], compensate, T)
    _check_codes(z, qz, kz)


def test_ksmooth_codes_gqa_multi_batch():
    cfg = mi.custom_prefill(2, 6, 2, 640, True, k_outliers=2, v_outlier_p=0.01, q_offset=True)
    z, qz, kz, _ = _quantize(cfg, True, 2, seed=5)
    _check_codes(z, qz, kz)


@pytest.mark.parametrize("causal,compensate,T", [(False, True, 2), (True, True, 2),
                                                 (True, False, 2), (False, True, 1)])
def test_ksmooth_prefill_parity(causal, compensate, T):
    import flashattention_mpfa_quantize_gb300 as mp
    cfg = mi.custom_prefill(2, 4, 2, 640, causal, k_outliers=1, v_outlier_p=0.001, q_offset=True)
    z, qz, kz, vz = _quantize(cfg, compensate, T, seed=7)
    o, lse = mp.prefill(z, causal=causal)
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    em = orc.prefill_emulate(qz, kz, vz, causal=causal)
    o_gpu, lse_gpu = np_f32(o), lse.cpu().numpy()
    got = np.concatenate([o_gpu[b, :, h, :] for (b, h) in em])
    want = np.concatenate([orc.bf16_bits_to_float(orc.bf16_round(v[0])) for v in em.values()])
    lg = np.concatenate([lse_gpu[b, h] for (b, h) in em])
    lw = np.concatenate([v[1] for v in em.values()])
    assert np.isfinite(got).all()
    assert np.abs(got - want).max() <= O_MAX_ABS
    assert rel_l2(got, want) <= O_REL_L2
    assert np.abs(lg - lw).max() <= LSE_ABS


def test_ksmooth_lowers_error_against_exact():
    """On the tiny configuration (K channel offsets, four x20 outlier
    channels) the smoothed forward is closer to exact fp64 attention."""
    import flashattention_mpfa_quantize_gb300 as mp
    cfg = mi.PREFILL["tiny_n256"]
    Q, K, V = mi.prefill_inputs(cfg, "cpu", 0)
    dev = torch.device("cuda:0")
    a = mp.quantize_qkv(Q.to(dev), K.to(dev), V.to(dev), k_smooth=True)
    b = mp.quantize_qkv(Q.to(dev), K.to(dev), V.to(dev))
    oa, la = mp.prefill(a, causal=False)
    ob, lb = mp.prefill(b, causal=False)
    torch.cuda.synchronize()
    ex = orc.prefill_exact(np_f32(Q), np_f32(K), np_f32(V), causal=False)[(0, 0)]
    ea = rel_l2(np_f32(oa)[0, :, 0, :], ex[0])
    eb = rel_l2(np_f32(ob)[0, :, 0, :], ex[0])
    print(f"\ntiny_n256 rel-L2 vs exact: K smoothing off {eb:.4f}, on {ea:.4f}")
    assert ea < eb
    assert np.isfinite(la.cpu().numpy()).all() and np.isfinite(lb.cpu().numpy()).all()


@pytest.mark.parametrize("compensate", [False, True])
def test_ksmooth_decode_parity(compensate):
    import flashattention_mpfa_quantize_gb300 as mp
    B, Hq, Hkv, Lmax = 3, 8, 2, 640
    cfg = mi.custom_decode(B, Hq, Hkv, Lmax, 1, Lmax)
    q, K, V, _ = mi.decode_inputs(cfg, "cpu", 11)
    lens = [640, 300, 0]
    dev = torch.device("cuda:0")
    cache = mp.quantize_qkv(None, K.to(dev), V.to(dev), k_smooth=True)
    res = mp.decode(q.to(dev), cache, torch.tensor(lens, dtype=torch.int32, device=dev),
                    compensate=compensate, T=2, kv_chunk=256)
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    kz = orc.quantize_k(np_f32(K), smooth=True)
    np.testing.assert_array_equal(cache["kbar"].cpu().numpy(), kz["kbar"])
    qz = orc.quantize_q_decode(np_f32(q), Hkv, compensate, 2)
    vz = orc.quantize_v(np_f32(V))
    em = orc.decode_emulate(qz, kz, vz, lens, chunk=res["chunk"])
    o_gpu, lse_gpu = np_f32(res["o"]), res["lse"].cpu().numpy()
    got = np.stack([o_gpu[b, h] for (b, h) in em])
    want = np.stack([orc.bf16_bits_to_float(orc.bf16_round(v[0])) for v in em.values()])
    lg = np.array([lse_gpu[b, h] for (b, h) in em])
    lw = np.array([v[1] for v in em.values()])
    assert np.abs(got - want).max() <= O_MAX_ABS
    fin = np.isfinite(lw)
    assert np.array_equal(fin, np.isfinite(lg)) and (~fin).sum() == Hq   # the empty sequence
    assert np.abs(lg[fin] - lw[fin]).max() <= LSE_ABS


def test_ksmooth_append_bit_exact():
    """New keys appended to a smoothed cache are coded as fp32(K - kbar) with
    the cache's own s_k, exactly like its rows."""
    import flashattention_mpfa_quantize_gb300 as mp
    B, Hkv, Lmax, n_new = 2, 2, 384, 5
    cfg = mi.custom_decode(B, 4, Hkv, Lmax, 1, Lmax)
    _, K, V, _ = mi.decode_inputs(cfg, "cpu", 13)
    kn, vn = mi.append_inputs(B, n_new, Hkv, "cpu", 14)
    dev = torch.device("cuda:0")
    cache = mp.quantize_qkv(None, K.to(dev), V.to(dev), k_smooth=True)
    start = [100, 379]
    mp.append_kv(kn.to(dev), vn.to(dev), cache, torch.tensor(start, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    kz = orc.quantize_k(np_f32(K), smooth=True)
    kbar = kz["kbar"]
    kc = cache["k"]["codes"].cpu().numpy()
    ks = tiled_to_rows(cache["k"]["scales"].cpu().numpy(), B * Hkv * Lmax).reshape(B, Hkv, Lmax, 8)
    knf = np_f32(kn)
    for b in range(B):
        for h in range(Hkv):
            x = (knf[b, :, h, :] - kbar[b, h][None, :]).astype(np.float32)
            c, s = orc.nvfp4_quantize(x, kz["s_k"])
            rows = slice(start[b], start[b] + n_new)
            np.testing.assert_array_equal(kc[b, h, rows], c)
            np.testing.assert_array_equal(ks[b, h, rows], s)
