"""CPU check of the full-FP4 PV parity test's flip allowance (the oracle's
single-tile emulation; no GPU): perturbing the scores by up to T_SLACK moves
O by no more than the allowance, and on the test's draw some row does move,
so the allowance is not vacuous."""
import numpy as np

import mpfa_inputs as mi
import oracle as orc
from helpers import S_P, T_SLACK, fp4p_flip_allowance, np_f32, oracle_quantize


def test_flip_allowance_finds_the_sensitive_rows():
    """CPU check of the allowance itself: perturbing the scores by up to
    T_SLACK moves the single-tile emulation's O by no more than the
    allowance, and on this draw some row does move (so it is not vacuous)."""
    cfg = mi.custom_prefill(2, 128, 8, 128, True, k_outliers=1, v_outlier_p=0.001,
                            q_offset=True)
    Q, K, V = mi.prefill_inputs(cfg, "cpu", 12)
    ref = oracle_quantize(Q, K, None, True, 2)
    vz = orc.quantize_v_fp4(np_f32(V))
    qz, kz = ref["q"], ref["k"]
    g = cfg.Hq // cfg.Hkv
    rng = np.random.default_rng(3)
    moved = 0.0
    for (b, h) in [(0, 0), (0, 77), (1, 3), (1, 127)]:
        allow, allow_lse = fp4p_flip_allowance(qz, kz, vz, b, h, g)
        q, qadd, k, _ = orc._head_operands(qz, kz, None, b, h, g)
        t = (q + qadd) @ k.T * orc.score_scale_log2(qz["s_q"], kz["s_k"])
        n = t.shape[0]
        t = np.where(np.arange(n)[None, :] > np.arange(n)[:, None], -np.inf, t)
        m = t.max(axis=1, keepdims=True)
        v = orc.nvfp4_dequant(vz["vc4"][b, h // g], vz["vs4"][b, h // g]).T * np.float64(vz["s_v"])

        def out(tt):
            c, sc = orc.nvfp4_quantize(np.exp2(tt - m + 4).astype(np.float32), S_P)
            P = orc.nvfp4_dequant(c, sc) * np.float64(S_P)
            l = P.sum(axis=1, keepdims=True)
            return P @ v / l, np.log(l[:, 0])

        o0, ll0 = out(t)
        for _ in range(4):
            o1, ll1 = out(t + rng.uniform(-T_SLACK, T_SLACK, t.shape))
            d = np.abs(o1 - o0)
            assert (d <= 1.05 * allow + 1e-12).all()
            assert (np.abs(ll1 - ll0) <= 1.05 * allow_lse + 1e-12).all()
            moved = max(moved, d.max())
    assert moved > 1e-3
