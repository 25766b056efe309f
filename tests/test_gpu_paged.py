"""GPU checks of the paged KV pool (block table over 128-token pages): a
pool holding the same tokens as a contiguous cache gives bit-identical
codes, and split-KV decode over it gives bit-identical O and LSE (same
tiles in the same order); quantize-on-append into the pool writes the same
codes as into the contiguous cache; a block-table entry outside the pool is
reported, not followed."""
import numpy as np
import pytest
import torch

import mpfa_inputs as mi
import oracle as orc
from helpers import np_f32, tiled_to_rows

pytestmark = pytest.mark.gpu


def _pool_case(B, Hq, Hkv, max_pages, seed):
    cfg = mi.custom_decode(B, Hq, Hkv, 128 * max_pages, 1, 128 * max_pages)
    q, K, V, _ = mi.decode_inputs(cfg, "cpu", seed)
    num_pages = B * max_pages
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed + 100))
    table = perm.view(B, max_pages).to(torch.int32)
    kp = torch.empty(num_pages, 128, Hkv, 128, dtype=torch.bfloat16)
    vp = torch.empty_like(kp)
    for b in range(B):
        for lp in range(max_pages):
            kp[table[b, lp]] = K[b, lp * 128:(lp + 1) * 128]
            vp[table[b, lp]] = V[b, lp * 128:(lp + 1) * 128]
    return q, K, V, kp, vp, table


def test_paged_pool_codes_and_decode_match_contiguous():
    import flashattention_mpfa_quantize_gb300 as mp
    B, Hq, Hkv, max_pages = 3, 8, 2, 5
    q, K, V, kp, vp, table = _pool_case(B, Hq, Hkv, max_pages, 21)
    dev = torch.device("cuda:0")
    cache = mp.quantize_qkv(None, K.to(dev), V.to(dev))
    pool = mp.quantize_pool(kp.to(dev), vp.to(dev))
    torch.cuda.synchronize()
    assert pool["k"]["scale"].item() == cache["k"]["scale"].item()
    assert pool["v"]["scale"].item() == cache["v"]["scale"].item()
    ck, pk = cache["k"]["codes"].cpu(), pool["k"]["codes"].cpu()
    cks = tiled_to_rows(cache["k"]["scales"].cpu().numpy(), B * Hkv * 128 * max_pages)
    pks = tiled_to_rows(pool["k"]["scales"].cpu().numpy(), B * max_pages * Hkv * 128)
    cv, pv = cache["v"]["codes"].cpu(), pool["v"]["codes"].cpu()
    for b in range(B):
        for h in range(Hkv):
            for lp in range(max_pages):
                p = int(table[b, lp])
                rows = slice(lp * 128, (lp + 1) * 128)
                assert torch.equal(ck[b, h, rows], pk[p, h])
                assert torch.equal(cv[b, h, rows], pv[p, h])
                c0 = ((b * Hkv + h) * max_pages + lp) * 128
                p0 = (p * Hkv + h) * 128
                np.testing.assert_array_equal(cks[c0:c0 + 128], pks[p0:p0 + 128])
    lens = torch.tensor([640, 300, 1], dtype=torch.int32, device=dev)
    for chunk in (0, 256):
        a = mp.decode(q.to(dev), cache, lens, kv_chunk=chunk)
        p_ = mp.decode_paged(q.to(dev), pool, table.to(dev), lens, kv_chunk=chunk)
        torch.cuda.synchronize()
        assert mp.get_error() == 0
        assert a["chunk"] == p_["chunk"]
        assert torch.equal(a["o"], p_["o"])
        assert torch.equal(a["lse"], p_["lse"])


def test_paged_append_matches_contiguous_append():
    import flashattention_mpfa_quantize_gb300 as mp
    B, Hq, Hkv, max_pages, n_new = 3, 8, 2, 4, 6
    q, K, V, kp, vp, table = _pool_case(B, Hq, Hkv, max_pages, 23)
    kn, vn = mi.append_inputs(B, n_new, Hkv, "cpu", 24)
    dev = torch.device("cuda:0")
    cache = mp.quantize_qkv(None, K.to(dev), V.to(dev))
    pool = mp.quantize_pool(kp.to(dev), vp.to(dev))
    start = torch.tensor([125, 300, 0], dtype=torch.int32, device=dev)   # 125: crosses a page
    mp.append_kv(kn.to(dev), vn.to(dev), cache, start)
    mp.append_kv_paged(kn.to(dev), vn.to(dev), pool, table.to(dev), start)
    torch.cuda.synchronize()
    assert mp.get_error() == 0
    ck, pk = cache["k"]["codes"].cpu(), pool["k"]["codes"].cpu()
    cv, pv = cache["v"]["codes"].cpu(), pool["v"]["codes"].cpu()
    s_k = pool["k"]["scale"].item()
    knf = np_f32(kn)
    for b in range(B):
        for h in range(Hkv):
            c, _ = orc.nvfp4_quantize(np.ascontiguousarray(knf[b, :, h, :]), np.float32(s_k))
            for t in range(n_new):
                pos = int(start[b]) + t
                p = int(table[b, pos // 128])
                assert torch.equal(pk[p, h, pos % 128], ck[b, h, pos])
                assert torch.equal(pv[p, h, pos % 128], cv[b, h, pos])
                np.testing.assert_array_equal(pk[p, h, pos % 128].numpy(), c[t])
    lens = start + n_new
    a = mp.decode(q.to(dev), cache, lens, kv_chunk=128)
    p_ = mp.decode_paged(q.to(dev), pool, table.to(dev), lens, kv_chunk=128)
    torch.cuda.synchronize()
    assert torch.equal(a["o"], p_["o"]) and torch.equal(a["lse"], p_["lse"])


def test_paged_bad_table_entry_is_reported():
    import flashattention_mpfa_quantize_gb300 as mp
    B, Hq, Hkv, max_pages = 2, 4, 1, 2
    q, K, V, kp, vp, table = _pool_case(B, Hq, Hkv, max_pages, 25)
    dev = torch.device("cuda:0")
    pool = mp.quantize_pool(kp.to(dev), vp.to(dev))
    bad = table.clone()
    bad[1, 1] = 1000                      # outside the 4-page pool
    lens = torch.tensor([256, 256], dtype=torch.int32, device=dev)
    mp.decode_paged(q.to(dev), pool, bad.to(dev), lens)
    assert mp.get_error() == mp.ERR_INVALID_ARG
    assert mp.get_error() == 0            # read and cleared
