"""GPU parity: split-KV decode against the oracle's split emulation on the
oracle's own codes of the same seeded cache (query codes bit-exact; O within
max-abs 2e-2 and rel-L2 5e-3; LSE within 2e-3), with the chunk the library
reports, ragged and empty lengths, forced chunk sizes and several GQA ratios."""
import numpy as np
import pytest
import torch

import mpfa_inputs as mi
import oracle as orc
from helpers import np_f32, rel_l2

pytestmark = pytest.mark.gpu

O_MAX_ABS = 2e-2
O_REL_L2 = 5e-3
LSE_ABS = 2e-3


def _decode_case(B, Hq, Hkv, Lmax, lens, compensate=True, T=2, kv_chunk=0, seed=0):
    import flashattention_mpfa_quantize_gb300 as mp
    cfg = mi.custom_decode(B, Hq, Hkv, Lmax, 1, Lmax)
    q, K, V, _ = mi.decode_inputs(cfg, "cpu", seed)
    seqlens = torch.tensor(lens, dtype=torch.int32)
    dev = torch.device("cuda:0")
    cache = mp.quantize_qkv(None, K.to(dev), V.to(dev))
    res = mp.decode(q.to(dev), cache, seqlens.to(dev), compensate=compensate, T=T,
                    kv_chunk=kv_chunk, return_query_codes=True)
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    qz = orc.quantize_q_decode(np_f32(q), Hkv, compensate, T)
    kz, vz = orc.quantize_k(np_f32(K)), orc.quantize_v(np_f32(V))
    # query codes: bit-exact
    np.testing.assert_array_equal(res["q"]["codes"].cpu().numpy(), qz["qc"])
    np.testing.assert_array_equal(res["q"]["scales"].cpu().numpy(), qz["qs"])
    assert res["q"]["scale"].item() == qz["s_q"]
    if compensate:
        np.testing.assert_array_equal(res["qbar"]["codes"].cpu().numpy(), qz["qbc"])
        np.testing.assert_array_equal(res["qbar"]["scales"].cpu().numpy(), qz["qbs"])
    em = orc.decode_emulate(qz, kz, vz, lens, chunk=res["chunk"])
    o_gpu = np_f32(res["o"])
    lse_gpu = res["lse"].cpu().numpy()
    got = np.stack([o_gpu[b, h] for (b, h) in em])
    want = np.stack([orc.bf16_bits_to_float(orc.bf16_round(v[0])) for v in em.values()])
    lg = np.array([lse_gpu[b, h] for (b, h) in em])
    lw = np.array([v[1] for v in em.values()])
    return got, want, lg, lw, res["chunk"]


def _assert_close(got, want, lg, lw):
    assert np.isfinite(got).all()
    err = np.abs(got - want)
    assert err.max() <= O_MAX_ABS, err.max()
    if np.linalg.norm(want) > 0:
        assert rel_l2(got, want) <= O_REL_L2, rel_l2(got, want)
    fin = np.isfinite(lw)
    assert np.array_equal(fin, np.isfinite(lg))
    assert np.abs(lg[fin] - lw[fin]).max() <= LSE_ABS


@pytest.mark.parametrize("compensate,T", [(False, 2), (True, 1), (True, 2)])
def test_decode_ragged_lengths(compensate, T):
    got, want, lg, lw, _ = _decode_case(4, 8, 2, 768, [1, 129, 700, 768], compensate, T)
    _assert_close(got, want, lg, lw)


@pytest.mark.parametrize("kv_chunk", [128, 256, 768])
def test_decode_forced_chunks(kv_chunk):
    got, want, lg, lw, chunk = _decode_case(2, 8, 2, 768, [500, 768], kv_chunk=kv_chunk, seed=1)
    assert chunk == kv_chunk
    _assert_close(got, want, lg, lw)


def test_decode_empty_sequence():
    got, want, lg, lw, _ = _decode_case(3, 4, 1, 256, [0, 256, 37], seed=2)
    _assert_close(got, want, lg, lw)
    assert (got[:4] == 0).all() and np.isneginf(lg[:4]).all()


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (16, 2), (32, 8)])
def test_decode_gqa_ratios(Hq, Hkv):
    got, want, lg, lw, _ = _decode_case(2, Hq, Hkv, 512, [512, 300], seed=3)
    _assert_close(got, want, lg, lw)
