"""GPU parity of quantize-on-append into a decode cache: the new tokens'
codes and tiled block scales are bit-identical to the oracle's NVFP4 / FP8
quantizers at the cache's own tensor scales (values beyond the cache's range
saturate on both sides), every other cache row is untouched, a decode step
over the extended cache matches the oracle's split emulation of the same
codes, and a sequence that would run past the cache is refused on the
device and left as it was."""
import numpy as np
import pytest
import torch

import mpfa_inputs as mi
import oracle as orc
from helpers import np_f32, rel_l2, tiled_to_rows

pytestmark = pytest.mark.gpu


def _cache_arrays(cache, B, Hkv, Lmax):
    kc = cache["k"]["codes"].cpu().numpy().reshape(B, Hkv, Lmax, 64)
    ks = tiled_to_rows(cache["k"]["scales"].cpu().numpy(), B * Hkv * Lmax).reshape(B, Hkv,
                                                                                   Lmax, 8)
    vc = cache["v"]["codes"].cpu().numpy().reshape(B, Hkv, Lmax, 128)
    return kc, ks, vc


def _append_case(B, Hq, Hkv, Lmax, lens, n_new, seed, spike=0.0):
    import flashattention_mpfa_quantize_gb300 as mp
    dev = torch.device("cuda:0")
    cfg = mi.custom_decode(B, Hq, Hkv, Lmax, 1, Lmax)
    q, K, V, _ = mi.decode_inputs(cfg, "cpu", seed)
    Kn, Vn = mi.append_inputs(B, n_new, Hkv, "cpu", seed + 1, spike=spike)
    cache = mp.quantize_qkv(None, K.to(dev), V.to(dev))
    before = _cache_arrays(cache, B, Hkv, Lmax)
    seq = torch.tensor(lens, dtype=torch.int32, device=dev)
    mp.append_kv(Kn.to(dev), Vn.to(dev), cache, seq)
    status = mp.get_error()
    after = _cache_arrays(cache, B, Hkv, Lmax)
    return mp, dev, q, K, V, Kn, Vn, cache, before, after, status


def test_append_bit_exact_and_other_rows_untouched():
    B, Hq, Hkv, Lmax, n_new = 3, 8, 2, 384, 5
    lens = [0, 130, Lmax - n_new]   # empty, mid-tile, filling the cache exactly
    mp, dev, q, K, V, Kn, Vn, cache, before, after, status = _append_case(
        B, Hq, Hkv, Lmax, lens, n_new, seed=3, spike=1000.0)
    assert status == 0
    kz, vz = orc.quantize_k(np_f32(K)), orc.quantize_v(np_f32(V))
    # the cache keeps its tensor scales
    assert cache["k"]["scale"].item() == kz["s_k"] and cache["v"]["scale"].item() == vz["s_v"]
    kc, ks, vc = after
    touched = np.zeros((B, Hkv, Lmax), bool)
    for b in range(B):
        for h in range(Hkv):
            rows = slice(lens[b], lens[b] + n_new)
            c, s = orc.nvfp4_quantize(np_f32(Kn[b, :, h, :]), kz["s_k"])
            np.testing.assert_array_equal(kc[b, h, rows], c)
            np.testing.assert_array_equal(ks[b, h, rows], s)
            np.testing.assert_array_equal(vc[b, h, rows],
                                          orc.fp8_quantize(np_f32(Vn[b, :, h, :]), vz["s_v"]))
            touched[b, h, rows] = True
    # the spikes (far beyond the cache's range) saturate: the largest E4M3
    # block scale of K and the largest E4M3 codes of V appear in the new rows
    assert (ks[touched] == 0x7E).any()
    assert ((vc[touched] & 0x7F) == 0x7E).any()
    for x, y in zip(before, after):
        np.testing.assert_array_equal(x[~touched], y[~touched])


@pytest.mark.parametrize("compensate", [False, True])
def test_decode_over_appended_cache(compensate):
    B, Hq, Hkv, Lmax, n_new = 2, 8, 2, 512, 3
    lens = [127, 300]
    mp, dev, q, K, V, Kn, Vn, cache, _, _, status = _append_case(B, Hq, Hkv, Lmax, lens, n_new,
                                                                 seed=5)
    assert status == 0
    new_lens = [n + n_new for n in lens]
    res = mp.decode(q.to(dev), cache, torch.tensor(new_lens, dtype=torch.int32, device=dev),
                    compensate=compensate, T=2, return_query_codes=True)
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    # the oracle's cache with the oracle's codes of the new tokens in place
    kz, vz = orc.quantize_k(np_f32(K)), orc.quantize_v(np_f32(V))
    for b in range(B):
        for h in range(Hkv):
            rows = slice(lens[b], lens[b] + n_new)
            kz["kc"][b, h, rows], kz["ks"][b, h, rows] = orc.nvfp4_quantize(
                np_f32(Kn[b, :, h, :]), kz["s_k"])
            vz["vc"][b, h, rows] = orc.fp8_quantize(np_f32(Vn[b, :, h, :]), vz["s_v"])
    qz = orc.quantize_q_decode(np_f32(q), Hkv, compensate, 2)
    em = orc.decode_emulate(qz, kz, vz, new_lens, chunk=res["chunk"])
    o_gpu = np_f32(res["o"])
    got = np.stack([o_gpu[b, h] for (b, h) in em])
    want = np.stack([orc.bf16_bits_to_float(orc.bf16_round(v[0])) for v in em.values()])
    assert np.abs(got - want).max() <= 2e-2
    assert rel_l2(got, want) <= 5e-3
    lg = res["lse"].cpu().numpy()
    assert max(abs(lg[b, h] - v[1]) for (b, h), v in em.items()) <= 2e-3


def test_append_overrun_refused_on_device():
    B, Hq, Hkv, Lmax, n_new = 2, 4, 1, 256, 4
    lens = [10, Lmax - 2]   # the second sequence would run past the cache
    mp, dev, q, K, V, Kn, Vn, cache, before, after, status = _append_case(
        B, Hq, Hkv, Lmax, lens, n_new, seed=7)
    assert status == 1   # MPFA_ERR_INVALID_ARG from the device status word
    assert mp.get_error() == 0   # read and cleared
    kz = orc.quantize_k(np_f32(K))
    c, s = orc.nvfp4_quantize(np_f32(Kn[0, :, 0, :]), kz["s_k"])
    np.testing.assert_array_equal(after[0][0, 0, 10:10 + n_new], c)
    for x, y in zip(before, after):
        np.testing.assert_array_equal(x[1], y[1])   # the refused sequence is as it was
