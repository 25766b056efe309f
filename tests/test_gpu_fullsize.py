"""GPU parity at the benchmark workloads' full sizes, in the launch
configuration bench.py times (inputs drawn on the GPU with the same seeds,
compensation on with T=2, the library's default decode chunk).

The oracle cannot emulate a whole 16K-128K forward in seconds, so each case
checks sampled outputs it can compute one by one: the tensor scales come from
the whole tensors (as the method defines them), the codes of a few sampled
heads are compared bit for bit, and sampled query rows (first and last rows,
tile boundaries, random rows) are emulated and compared within the parity
tolerance (O max-abs 2e-2, rel-L2 5e-3; LSE 2e-3)."""
import numpy as np
import pytest
import torch

import mpfa_inputs as mi
import oracle as orc
from helpers import np_f32, rel_l2, tiled_to_rows

pytestmark = pytest.mark.gpu

O_MAX_ABS, O_REL_L2, LSE_ABS = 2e-2, 5e-3, 2e-3


def _amax_bf16_chunks(t: torch.Tensor) -> np.float32:
    """max |x| of a bf16 GPU tensor, reduced on the host one batch row at a time."""
    m = 0
    for b in range(t.shape[0]):
        bits = t[b].contiguous().view(torch.int16).cpu().numpy().view(np.uint16) & 0x7FFF
        m = max(m, int(bits.max()))
    return np.uint32(m << 16).view(np.float32)


def _sample_rows(n, rng, extra=6):
    base = {0, 1, 63, 127, 128, 129, 255, 256, n // 2 - 1, n // 2, n - 129, n - 128, n - 2, n - 1}
    base |= set(rng.integers(0, n, extra).tolist())
    return np.array(sorted(r for r in base if 0 <= r < n), dtype=np.int64)


def _prefill_fullsize(cfg, heads, seed=0):
    import flashattention_mpfa_quantize_gb300 as mp
    dev = torch.device("cuda:0")
    Q, K, V = mi.prefill_inputs(cfg, dev, seed)
    qz = mp.quantize_qkv(Q, K, V, compensate=True, T=2)
    o, lse = mp.prefill(qz, causal=cfg.causal)
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    B, N, Hq, Hkv, g = cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.Hq // cfg.Hkv
    # tensor scales of the whole tensors (rank-one smoothing on)
    amax_q = np.float32(0)
    for b in range(B):
        for h in range(Hq):
            mb, xp = orc.block_means(np_f32(Q[b, :, h, :]), 128)
            amax_q = max(amax_q, np.float32(np.abs(xp).max()), np.float32(np.abs(mb).max()))
    s_q = orc.tensor_scale(amax_q, 2688.0)
    s_k = orc.tensor_scale(_amax_bf16_chunks(K), 2688.0)
    s_v = orc.tensor_scale(_amax_bf16_chunks(V), 448.0)
    assert qz["q"]["scale"].item() == s_q
    assert qz["k"]["scale"].item() == s_k and qz["v"]["scale"].item() == s_v
    rng = np.random.default_rng(7)
    rows = _sample_rows(N, rng)
    cs = orc.score_scale_log2(s_q, s_k)
    got, want, lg, lw = [], [], [], []
    for (b, h) in heads:
        hk = h // g
        mb, xp = orc.block_means(np_f32(Q[b, :, h, :]), 128)
        qc, qs = orc.nvfp4_quantize(xp, s_q)
        tc, ts = orc.rank_one_terms(mb, s_q, 2)
        kc, ks = orc.nvfp4_quantize(np_f32(K[b, :, hk, :]), s_k)
        vc = orc.fp8_quantize(np_f32(V[b, :, hk, :]), s_v)
        # codes and scales of this head, bit for bit
        r0 = (b * Hq + h) * N
        np.testing.assert_array_equal(qz["q"]["codes"][b, h].cpu().numpy(), qc)
        np.testing.assert_array_equal(
            tiled_to_rows(qz["q"]["scales"][r0 * 8:(r0 + N) * 8].cpu().numpy(), N), qs)
        np.testing.assert_array_equal(qz["qbar"]["codes"][b, h].cpu().numpy(), tc)
        np.testing.assert_array_equal(qz["qbar"]["scales"][b, h].cpu().numpy(), ts)
        k0 = (b * Hkv + hk) * N
        np.testing.assert_array_equal(qz["k"]["codes"][b, hk].cpu().numpy(), kc)
        np.testing.assert_array_equal(
            tiled_to_rows(qz["k"]["scales"][k0 * 8:(k0 + N) * 8].cpu().numpy(), N), ks)
        np.testing.assert_array_equal(qz["v"]["codes"][b, hk].cpu().numpy(), vc)
        # emulated rows
        q = orc.nvfp4_dequant(qc, qs)
        qadd = np.repeat(sum(orc.nvfp4_dequant(np.ascontiguousarray(tc[:, t]),
                                               np.ascontiguousarray(ts[:, t])) for t in range(2)),
                         128, axis=0)
        oe, le = orc.attn_online(q, qadd, orc.nvfp4_dequant(kc, ks), orc.fp8_dequant(vc),
                                 score_scale=cs, out_scale=float(s_v), causal=cfg.causal,
                                 rows=rows)
        got.append(np_f32(o[b, rows, h, :]))
        want.append(orc.bf16_bits_to_float(orc.bf16_round(oe)))
        lg.append(lse[b, h, rows].cpu().numpy())
        lw.append(le)
    got, want = np.concatenate(got), np.concatenate(want)
    lg, lw = np.concatenate(lg), np.concatenate(lw)
    assert np.isfinite(got).all()
    assert np.abs(got - want).max() <= O_MAX_ABS, np.abs(got - want).max()
    assert rel_l2(got, want) <= O_REL_L2, rel_l2(got, want)
    assert np.abs(lg - lw).max() <= LSE_ABS, np.abs(lg - lw).max()


def test_fullsize_llama8b_n16k_causal():
    _prefill_fullsize(mi.PREFILL["llama8b_n16k_causal"], [(0, 0), (0, 17), (0, 31)])


def test_fullsize_qwen14b_n128k_causal():
    _prefill_fullsize(mi.PREFILL["qwen14b_n128k_causal"], [(0, 0), (0, 39)])


def test_fullsize_b1_s4096_h24():
    _prefill_fullsize(mi.PREFILL["b1_s4096_h24"], [(0, 0), (0, 23)])


def test_fullsize_b1_s8192_h64():
    _prefill_fullsize(mi.PREFILL["b1_s8192_h64"], [(0, 5), (0, 63)])


def _decode_fullsize(cfg, pick, seed=1):
    import flashattention_mpfa_quantize_gb300 as mp
    dev = torch.device("cuda:0")
    q, K, V, seqlens = mi.decode_inputs(cfg, dev, seed)
    cache = mp.quantize_qkv(None, K, V)
    res = mp.decode(q, cache, seqlens, return_query_codes=True)
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    s_k = orc.tensor_scale(_amax_bf16_chunks(K), 2688.0)
    s_v = orc.tensor_scale(_amax_bf16_chunks(V), 448.0)
    assert cache["k"]["scale"].item() == s_k and cache["v"]["scale"].item() == s_v
    qz = orc.quantize_q_decode(np_f32(q), cfg.Hkv, True, 2)
    np.testing.assert_array_equal(res["q"]["codes"].cpu().numpy(), qz["qc"])
    np.testing.assert_array_equal(res["q"]["scales"].cpu().numpy(), qz["qs"])
    np.testing.assert_array_equal(res["qbar"]["codes"].cpu().numpy(), qz["qbc"])
    np.testing.assert_array_equal(res["qbar"]["scales"].cpu().numpy(), qz["qbs"])
    assert res["q"]["scale"].item() == qz["s_q"]
    lens = seqlens.cpu().numpy()
    pairs = pick(lens)
    g = cfg.Hq // cfg.Hkv
    cs = orc.score_scale_log2(qz["s_q"], s_k)
    got, want, lg, lw = [], [], [], []
    L = cfg.Lmax
    for (b, h) in pairs:
        hk = h // g
        kc, ks = orc.nvfp4_quantize(np_f32(K[b, :, hk, :]), s_k)
        vc = orc.fp8_quantize(np_f32(V[b, :, hk, :]), s_v)
        r0 = (b * cfg.Hkv + hk) * L
        np.testing.assert_array_equal(cache["k"]["codes"][b, hk].cpu().numpy(), kc)
        np.testing.assert_array_equal(
            tiled_to_rows(cache["k"]["scales"][r0 * 8:(r0 + L) * 8].cpu().numpy(), L), ks)
        np.testing.assert_array_equal(cache["v"]["codes"][b, hk].cpu().numpy(), vc)
        qd = orc.nvfp4_dequant(qz["qc"][b, h][None], qz["qs"][b, h][None])
        qadd = sum(orc.nvfp4_dequant(qz["qbc"][b, hk, t][None], qz["qbs"][b, hk, t][None])
                   for t in range(2))
        oe, le = orc.attn_online(qd, qadd, orc.nvfp4_dequant(kc, ks), orc.fp8_dequant(vc),
                                 score_scale=cs, out_scale=float(s_v), causal=False,
                                 kv_len=int(lens[b]), chunk=res["chunk"])
        got.append(np_f32(res["o"][b, h]))
        want.append(orc.bf16_bits_to_float(orc.bf16_round(oe[0])))
        lg.append(res["lse"][b, h].item())
        lw.append(le[0])
    got, want = np.stack(got), np.stack(want)
    assert np.abs(got - want).max() <= O_MAX_ABS, np.abs(got - want).max()
    assert rel_l2(got, want) <= O_REL_L2, rel_l2(got, want)
    assert np.abs(np.array(lg) - np.array(lw)).max() <= LSE_ABS


def test_fullsize_decode_b64_l32k():
    _decode_fullsize(mi.DECODE["decode_b64_l32k"],
                     lambda lens: [(0, 0), (17, 9), (40, 22), (63, 31)])


def test_fullsize_decode_b64_l4k_64k():
    # the shortest and the longest sequence of the ragged batch, plus one more
    _decode_fullsize(mi.DECODE["decode_b64_l4k_64k"],
                     lambda lens: [(int(np.argmin(lens)), 0), (int(np.argmax(lens)), 31), (5, 12)])
