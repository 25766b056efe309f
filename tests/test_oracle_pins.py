"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the
codebook the FP4 explainer prints, torch's float8 cast (a library routine),
an independent arithmetic formulation of round-to-nearest-even, closed forms
(softmax on a single tile, V = 1), the exactness of the online softmax, and
invariants of the rank-one smoothing.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LOG2E_RSQRT_D = math.log2(math.e) / math.sqrt(128)


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    return rows


# --------------------------------------------------------------------------
# formats
# --------------------------------------------------------------------------

def test_e2m1_codebook_matches_page():
    mags = sorted(r[0] for r in _read_golden("e2m1_codebook.txt"))
    pos = sorted(orc.e2m1_value(c) for c in range(8))
    assert pos == mags
    for c in range(8):
        v = orc.e2m1_value(c + 8)
        assert v == -orc.e2m1_value(c) and math.copysign(1.0, v) == -1.0
    # about 15 distinct values (+0 and -0 coincide), range +-6
    vals = {orc.e2m1_value(c) for c in range(16)}
    assert len(vals) == 15 and max(vals) == 6 and min(vals) == -6


def test_e2m1_rounding_examples():
    for x, want in _read_golden("e2m1_rounding_examples.txt"):
        for sgn in (1.0, -1.0):
            code = int(orc.e2m1_encode([sgn * x])[0])
            assert abs(orc.e2m1_value(code)) == want, (x, code)
            assert (code >> 3) == (1 if sgn < 0 else 0)


def _rne_grid_e2m1(a):
    """Independent formulation: round |a| on the local grid spacing with
    numpy's half-to-even rint; spacing 0.5 below 2, 1 below 4, 2 above."""
    a = np.abs(a)
    h = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    v = h * np.rint(a / h)
    return np.minimum(v, 6.0)


def test_e2m1_encode_matches_rint_formulation():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.uniform(-8, 8, 200000),
        np.arange(-700, 701) / 100.0,                    # dense sweep incl. every tie point
        np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 6.5, -0.0, 0.0]),
    ])
    codes = orc.e2m1_encode(x)
    got = np.array([abs(orc.e2m1_value(int(c))) for c in codes])
    np.testing.assert_array_equal(got, _rne_grid_e2m1(x))
    np.testing.assert_array_equal(codes >> 3, np.signbit(x).astype(np.uint8))


def test_e4m3_table_matches_torch():
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    ours = np.array([orc.e4m3_value(c) for c in range(256)])
    nan = np.isnan(t)
    assert nan.sum() == 2 and np.array_equal(nan, np.isnan(ours))
    np.testing.assert_array_equal(ours[~nan], t[~nan])
    assert orc.e4m3_value(0x7E) == 448.0 and orc.e4m3_value(1) == 2.0 ** -9


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(2)
    mags = np.exp2(rng.uniform(-14, math.log2(463.0), 300000))
    x = (mags * rng.choice([-1.0, 1.0], mags.size)).astype(np.float32).astype(np.float64)
    vals = np.array([orc.e4m3_value(c) for c in range(0x7F)])
    mids = (vals[:-1] + vals[1:]) / 2                    # every tie point
    x = np.concatenate([x, mids, -mids, [0.0, -0.0, 2.0 ** -10, 3 * 2.0 ** -11, 460.0]])
    x32 = x.astype(np.float32)                           # the encoder is fed fp32 values
    assert np.array_equal(x32.astype(np.float64), x)     # all of these are fp32-exact
    ref = torch.from_numpy(x32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(orc.e4m3_encode(x), ref)


def test_e4m3_encode_saturates():
    x = np.array([448.0, 464.0, 470.0, 1e4, 1e30])
    assert (orc.e4m3_encode(x) == 0x7E).all()
    assert (orc.e4m3_encode(-x) == 0xFE).all()


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(100000) * np.exp2(rng.uniform(-20, 20, 100000))).astype(np.float32)
    x = np.concatenate([x, np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(orc.bf16_round(x.astype(np.float64)), ref)


# --------------------------------------------------------------------------
# quantizers
# --------------------------------------------------------------------------

def test_nvfp4_representable_roundtrip():
    """A tensor built from codes x block scales x s round-trips exactly when
    each block contains a magnitude-6 element and one block has scale 448."""
    rng = np.random.default_rng(4)
    rows, d = 64, 128
    s = np.float32(2.0 ** -5)                             # amax = 6*448*s = 84
    e4m3_vals = np.array([orc.e4m3_value(c) for c in range(1, 0x7F)])
    sb = rng.choice(e4m3_vals[e4m3_vals >= 2 ** -3], (rows, d // 16))
    sb[0, 0] = 448.0
    codes = rng.integers(0, 16, (rows, d))
    codes[:, ::16] = 7                                     # magnitude 6 in every block
    vals = np.array([orc.e2m1_value(int(c)) for c in range(16)])[codes]
    x = (vals * np.repeat(sb, 16, axis=1) * float(s)).astype(np.float32)
    assert np.array_equal(x.astype(np.float64), vals * np.repeat(sb, 16, axis=1) * float(s))
    amax = np.float32(np.abs(x).max())
    assert orc.tensor_scale(amax, 2688.0) == s
    qc, qs = orc.nvfp4_quantize(x, s)
    np.testing.assert_array_equal(np.array([orc.e4m3_value(int(c)) for c in qs.ravel()]),
                                  sb.ravel())
    deq = orc.nvfp4_dequant(qc, qs) * float(s)
    # codes compare by value (+0 and -0 both decode to 0)
    np.testing.assert_array_equal(deq, x.astype(np.float64))
    lo = (qc & 15).astype(np.int64)
    hi = (qc >> 4).astype(np.int64)
    interleaved = np.stack([lo, hi], axis=-1).reshape(rows, d)
    nz = vals != 0
    np.testing.assert_array_equal(interleaved[nz], codes[nz])   # low nibble = lower index


def _nvfp4_error_bound(x, s, qs):
    sbs = np.repeat(np.array([orc.e4m3_value(int(c)) for c in qs.ravel()]).reshape(qs.shape),
                    16, axis=1) * float(s)
    y = np.abs(x.astype(np.float64)) / np.where(sbs > 0, sbs, 1)
    half = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0))
    bound = np.maximum(half, y - 6.0) * sbs
    return np.where(sbs > 0, bound * (1 + 1e-6), np.abs(x))


@pytest.mark.parametrize("dist", ["normal", "outliers", "tiny"])
def test_nvfp4_invariants(dist):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((512, 128)).astype(np.float32)
    if dist == "outliers":
        x[:, 7] *= 20
        x += rng.standard_normal(128).astype(np.float32) * 1.4
    if dist == "tiny":
        x *= 1e-30
    x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    amax = np.float32(np.abs(x).max())
    s = orc.tensor_scale(amax, 2688.0)
    assert s == np.float32(amax / np.float32(2688.0))
    qc, qs = orc.nvfp4_quantize(x, s)
    assert qs.max() <= 0x7E                                # block scales never exceed 448
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert qs[r, c // 16] == 0x7E                          # the amax block gets scale 448
    deq = orc.nvfp4_dequant(qc, qs) * float(s)
    err = np.abs(deq - x.astype(np.float64))
    assert (err <= _nvfp4_error_bound(x, s, qs)).all()


def test_nvfp4_zero_tensor():
    x = np.zeros((4, 128), np.float32)
    s = orc.tensor_scale(0.0, 2688.0)
    assert s == 1.0
    qc, qs = orc.nvfp4_quantize(x, s)
    assert (qc == 0).all() and (qs == 0).all()


def test_fp8_v_quantizer():
    rng = np.random.default_rng(6)
    v = torch.from_numpy(rng.standard_normal((300, 128)).astype(np.float32) * 3)
    v = v.to(torch.bfloat16).float().numpy()
    s = orc.tensor_scale(np.abs(v).max(), 448.0)
    codes = orc.fp8_quantize(v, s)
    ref = torch.from_numpy((v / s).astype(np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()
    np.testing.assert_array_equal(codes, ref)
    assert np.abs(orc.fp8_dequant(codes)).max() == 448.0


def test_block_means_match_numpy():
    rng = np.random.default_rng(7)
    x = torch.from_numpy(rng.standard_normal((4 * 128, 128)).astype(np.float32) * 2 + 0.7)
    x = x.to(torch.bfloat16).float().numpy()
    qbar, xp = orc.block_means(x, 128)
    ref = x.astype(np.float64).reshape(4, 128, 128).mean(axis=1).astype(np.float32)
    np.testing.assert_array_equal(qbar, ref)
    np.testing.assert_array_equal(xp, (x.reshape(4, 128, 128) - qbar[:, None, :]).reshape(-1, 128))


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def _rand_qkv(n, nk=None, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    nk = n if nk is None else nk
    q = rng.standard_normal((n, 128)) * scale
    k = rng.standard_normal((nk, 128)) * scale
    v = rng.standard_normal((nk, 128))
    return q, k, v


@pytest.mark.parametrize("n,causal", [(16, False), (32, True), (64, False), (300, True),
                                      (300, False), (257, True)])
def test_online_softmax_equals_full_softmax(n, causal):
    """Quantizers off (identity, unrounded P): the tiled online softmax equals
    the exact softmax (the FlashAttention-2 identity)."""
    q, k, v = _rand_qkv(n, seed=n, scale=1.5)
    o1, l1 = orc.attn_online(q, None, k, v, score_scale=LOG2E_RSQRT_D, out_scale=1.0,
                             causal=causal, round_p=False)
    o2, l2 = orc.attn_exact(q, k, v, causal=causal)
    np.testing.assert_allclose(o1, o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-11)


@pytest.mark.parametrize("chunk,kv_len", [(128, 300), (256, 513), (128, 129), (384, 1000)])
def test_split_kv_combine_equals_full_softmax(chunk, kv_len):
    q, k, v = _rand_qkv(4, nk=1024, seed=chunk + kv_len)
    o1, l1 = orc.attn_online(q, None, k, v, score_scale=LOG2E_RSQRT_D, out_scale=1.0,
                             causal=False, kv_len=kv_len, chunk=chunk, round_p=False)
    o2, l2 = orc.attn_exact(q, k, v, causal=False, kv_len=kv_len)
    np.testing.assert_allclose(o1, o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-11)


def test_qadd_is_added_to_every_score():
    """S = (q + qadd).k: one row of qadd shared by all rows equals adding it to q."""
    q, k, v = _rand_qkv(200, seed=11)
    u = np.random.default_rng(12).standard_normal(128)
    qadd = np.tile(u, (200, 1))
    o1, l1 = orc.attn_online(q, qadd, k, v, score_scale=LOG2E_RSQRT_D, out_scale=1.0,
                             causal=True, round_p=False)
    o2, l2 = orc.attn_exact(q + u, k, v, causal=True)
    np.testing.assert_allclose(o1, o2, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-10)


P_SHIFT_READING = 4      # P stored as E4M3(2^4 p)
TAU_READING = 4.0        # reference max moves when a tile max exceeds it by > 4


def _e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.float8_e4m3fn).double().numpy()


@pytest.mark.parametrize("n", [16, 64, 128])
def test_single_tile_rounded_p_direct_formula(n):
    """One KV tile: P8 = E4M3(2^4 2^(t - max t)) (torch's e4m3 cast),
    O = sum P8 v / sum P8, LSE = ln2 (max t + log2 sum P8 - 4)."""
    assert orc.P_SHIFT == P_SHIFT_READING and orc.RESCALE_TAU == TAU_READING
    q, k, v = _rand_qkv(n, seed=100 + n, scale=1.3)
    o1, l1 = orc.attn_online(q, None, k, v, score_scale=LOG2E_RSQRT_D, out_scale=1.0,
                             causal=False, round_p=True)
    t = (q @ k.T) * LOG2E_RSQRT_D
    m = t.max(axis=1, keepdims=True)
    p8 = _e4m3(np.exp2(t - m) * 2.0 ** P_SHIFT_READING)
    o2 = (p8 @ v) / p8.sum(axis=1, keepdims=True)
    l2 = math.log(2) * (m[:, 0] + np.log2(p8.sum(axis=1)) - P_SHIFT_READING)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


@pytest.mark.parametrize("delta", [-3.0, 0.5, 3.9, 4.1, 7.0])
def test_two_tile_reference_max_rule(delta):
    """Two KV tiles whose maxima differ by delta (log2 units): the row's
    reference max stays at tile 0's max while delta <= 4 (P of tile 1 then
    reaches up to 2^(4+delta)), and moves to tile 1's max with the rescale
    alpha = 2^-delta once delta > 4.  Checked against a direct formula."""
    rng = np.random.default_rng(int(delta * 10) + 50)
    t0 = rng.uniform(-6, 0, 128)
    t0[5] = 0.0                                   # tile 0 max = 0
    t1 = rng.uniform(-6, 0, 128) + delta
    t1[77] = delta                                # tile 1 max = delta
    tt = np.concatenate([t0, t1])
    q = np.zeros((1, 128)); q[0, 0] = 1.0
    k = np.zeros((256, 128)); k[:, 0] = tt        # score_scale 1: t_j = k_j[0]
    v = rng.standard_normal((256, 128))
    o1, l1 = orc.attn_online(q, None, k, v, score_scale=1.0, out_scale=1.0, causal=False)
    s = 2.0 ** P_SHIFT_READING
    if delta <= TAU_READING:
        p8 = _e4m3(np.exp2(tt - 0.0) * s)
        o2 = p8 @ v / p8.sum()
        l2 = math.log(2) * (0.0 + math.log2(p8.sum()) - P_SHIFT_READING)
        if delta > 0:
            assert p8[128:].max() > s                # P above 2^s: the stale max is kept
    else:
        p0 = _e4m3(np.exp2(t0) * s)
        p1 = _e4m3(np.exp2(t1 - delta) * s)
        alpha = 2.0 ** -delta
        acc = alpha * (p0 @ v[:128]) + p1 @ v[128:]
        ell = alpha * p0.sum() + p1.sum()
        o2 = acc / ell
        l2 = math.log(2) * (delta + math.log2(ell) - P_SHIFT_READING)
    np.testing.assert_allclose(o1[0], o2, rtol=1e-12, atol=1e-13)
    assert abs(l1[0] - l2) < 1e-12


def test_shared_rounding_rows_sum_to_one():
    """The running sum adds the same rounded P codes the PV product uses, so
    V = 1 gives O = 1 exactly for every row, over many tiles and splits."""
    q, k, _ = _rand_qkv(700, seed=21, scale=2.0)
    v = np.ones((700, 128))
    for chunk in (0, 256):
        o, _ = orc.attn_online(q, None, k, v, score_scale=LOG2E_RSQRT_D, out_scale=1.0,
                               causal=True, chunk=chunk, round_p=True)
        np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-14)


def test_one_split_equals_no_split():
    q, k, v = _rand_qkv(3, nk=900, seed=31)
    a = orc.attn_online(q, None, k, v, score_scale=0.1, out_scale=1.0, causal=False,
                        kv_len=777, chunk=0)
    b = orc.attn_online(q, None, k, v, score_scale=0.1, out_scale=1.0, causal=False,
                        kv_len=777, chunk=896)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_empty_rows():
    q, k, v = _rand_qkv(2, nk=10, seed=41)
    o, l = orc.attn_online(q, None, k, v, score_scale=0.1, out_scale=1.0, causal=False,
                           kv_len=0, chunk=128)
    assert (o == 0).all() and np.isneginf(l).all()


# --------------------------------------------------------------------------
# the method end to end (oracle only)
# --------------------------------------------------------------------------

def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16).float().numpy()


def _rel_l2(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _emulate_vs_exact(Q, K, V, compensate, causal=False):
    qz = orc.quantize_q_prefill(Q, compensate)
    kz = orc.quantize_k(K)
    vz = orc.quantize_v(V)
    em = orc.prefill_emulate(qz, kz, vz, causal=causal)
    ex = orc.prefill_exact(Q, K, V, causal=causal)
    a = np.concatenate([em[h][0] for h in sorted(em)])
    b = np.concatenate([ex[h][0] for h in sorted(ex)])
    return a, b, qz


def test_zero_mean_blocks_make_compensation_vanish():
    """Rows paired (x, -x) inside every 128-row block give qbar = 0: the codes
    of Q are the same with and without the smoothing and O is identical."""
    rng = np.random.default_rng(51)
    half = _bf16(rng.standard_normal((1, 128, 1, 128)) * 1.7)
    Q = np.concatenate([half, -half], axis=1)              # [1, 256, 1, 128]
    Q = Q[:, np.r_[0:64, 128:192, 64:128, 192:256]]         # each 128-block holds x and -x
    K = _bf16(rng.standard_normal((1, 256, 1, 128)))
    V = _bf16(rng.standard_normal((1, 256, 1, 128)))
    on = orc.quantize_q_prefill(Q, True)
    off = orc.quantize_q_prefill(Q, False)
    assert (on["qbar"] == 0).all()
    assert on["s_q"] == off["s_q"]
    np.testing.assert_array_equal(on["qc"] & 0x77, off["qc"] & 0x77)   # magnitudes
    np.testing.assert_array_equal(on["qs"], off["qs"])
    assert (on["qbs"] == 0).all() and (on["qbc"] & 0x77 == 0).all()
    kz, vz = orc.quantize_k(K), orc.quantize_v(V)
    a = orc.prefill_emulate(on, kz, vz, causal=True)[(0, 0)]
    b = orc.prefill_emulate(off, kz, vz, causal=True)[(0, 0)]
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_compensation_exact_for_representable_block_means():
    """Every row of a 128-row block equal to a block mean mu_b that NVFP4
    represents exactly: with the smoothing, Q' = 0 and the rank-one term alone
    carries mu_b K^T, so O equals the unsmoothed result bit for bit, and all
    rows of a block agree.  A flipped sign, a dropped term or a wrong
    row-to-block mapping breaks the equality."""
    rng = np.random.default_rng(81)
    s = 2.0 ** -6                                         # amax = 6 * 448 * s = 42
    e4 = np.array([orc.e4m3_value(c) for c in range(0x30, 0x7F)])
    mus = []
    for b in range(3):
        codes = rng.integers(0, 16, 128)
        codes[::16] = 7 + 8 * rng.integers(0, 2, 8)       # magnitude 6 in every 16-block
        sb = rng.choice(e4, 8)
        sb[0] = 448.0
        vals = np.array([orc.e2m1_value(int(c)) for c in range(16)])[codes]
        mus.append(vals * np.repeat(sb, 16) * s)
    Q = np.repeat(np.stack(mus), 128, axis=0)[None, :, None, :].astype(np.float32)
    assert np.array_equal(_bf16(Q), Q)
    K = _bf16(rng.standard_normal((1, 384, 1, 128)))
    V = _bf16(rng.standard_normal((1, 384, 1, 128)))
    on = orc.quantize_q_prefill(Q, True)
    off = orc.quantize_q_prefill(Q, False)
    assert on["s_q"] == off["s_q"] == np.float32(s)
    np.testing.assert_array_equal(on["qbar"][0, 0], np.stack(mus).astype(np.float32))
    assert (on["qc"] & 0x77 == 0).all()                   # Q' = 0
    assert (on["qbs"][..., 1, :] == 0).all()               # mu_b exact: no residual term
    kz, vz = orc.quantize_k(K), orc.quantize_v(V)
    for causal in (False, True):
        a = orc.prefill_emulate(on, kz, vz, causal=causal)[(0, 0)]
        b = orc.prefill_emulate(off, kz, vz, causal=causal)[(0, 0)]
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])
    a = orc.prefill_emulate(on, kz, vz, causal=False)[(0, 0)][0]
    for blk in range(3):
        assert (a[blk * 128:(blk + 1) * 128] == a[blk * 128]).all()
    assert not np.array_equal(a[0], a[128])


def test_compensation_reduces_error_with_query_mean():
    """With a large per-channel offset on Q (the case the rank-one smoothing
    targets) the mean error over seeds is clearly lower with the two-term
    compensation; a dropped or sign-flipped rank-one term makes it many times
    larger instead."""
    rng = np.random.default_rng(71)
    e_on, e_off = [], []
    for _ in range(8):
        Q = _bf16(rng.standard_normal((1, 256, 1, 128)) + 6.0 * rng.standard_normal(128))
        K = _bf16(rng.standard_normal((1, 256, 1, 128)))
        V = _bf16(rng.standard_normal((1, 256, 1, 128)))
        a_on, ex, _ = _emulate_vs_exact(Q, K, V, True)
        a_off, _, _ = _emulate_vs_exact(Q, K, V, False)
        e_on.append(_rel_l2(a_on, ex))
        e_off.append(_rel_l2(a_off, ex))
    assert np.mean(e_on) < 0.8 * np.mean(e_off), (e_on, e_off)
    assert max(e_on) < 0.4


def test_decode_emulate_matches_prefill_last_row():
    """A decode query against keys [0, L) equals the prefill row L-1 of a
    causal forward with the same codes, when there is one split and no smoothing."""
    rng = np.random.default_rng(61)
    L = 384
    K = _bf16(rng.standard_normal((1, L, 1, 128)))
    V = _bf16(rng.standard_normal((1, L, 1, 128)))
    Q = _bf16(rng.standard_normal((1, L, 1, 128)))
    qz = orc.quantize_q_prefill(Q, False)
    kz, vz = orc.quantize_k(K), orc.quantize_v(V)
    pre = orc.prefill_emulate(qz, kz, vz, causal=True, rows=[L - 1])[(0, 0)]
    dq = dict(qc=qz["qc"][:, :, L - 1], qs=qz["qs"][:, :, L - 1], qbc=None, qbs=None,
              s_q=qz["s_q"])
    dec = orc.decode_emulate(dq, kz, vz, np.array([L]), chunk=0)[(0, 0)]
    np.testing.assert_array_equal(dec[0], pre[0][0])
    assert dec[1] == pre[1][0]


# --------------------------------------------------------------------------
# the score scale (t = S s_q s_k log2(e) / sqrt(d)) and the LSE it implies
# --------------------------------------------------------------------------

def _rn32(x):
    """Nearest binary32 (ties to even) of an exact rational x (fractions.Fraction),
    by integer arithmetic alone: no intermediate float rounding."""
    from fractions import Fraction
    x = Fraction(x)
    if x == 0:
        return np.float32(0.0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                       # subnormals share the smallest exponent
    scaled = a / Fraction(2) ** (e - 23)    # 24-bit significand + fraction
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    return np.float32(sign * float(Fraction(m) * Fraction(2) ** (e - 23)))


def _log2e_rsqrt_d_exact(d=128, digits=60):
    """log2(e) / sqrt(d) to `digits` decimal digits (mpmath), as a Fraction."""
    from fractions import Fraction
    import mpmath
    with mpmath.workdps(digits):
        v = 1 / (mpmath.log(2) * mpmath.sqrt(d))
        return Fraction(mpmath.nstr(v, digits, strip_zeros=False))


def test_score_scale_log2_bit_exact():
    """The factor taking accumulated code products to log2-domain logits is
    t = S * s_q * s_k * log2(e) / sqrt(d) (the explainer's attention section:
    S = Q K^T / sqrt(d), evaluated with exp2), with the fp32 roundings the
    kernels apply: c = RN32(log2(e)/sqrt(128)), then RN32(RN32(s_q s_k) c).
    The constant is derived here from 60-digit log and sqrt with exact
    rational rounding, independently of the oracle's fp64 expression."""
    from fractions import Fraction
    c = _rn32(_log2e_rsqrt_d_exact())
    assert orc.score_scale_log2(1.0, 1.0) == float(c)
    rng = np.random.default_rng(91)
    # tensor scales as the quantizers produce them (amax / 2688 for amax over a
    # wide range), plus powers of two and values whose product hits a tie
    sq = [orc.tensor_scale(a, 2688.0) for a in rng.uniform(1e-3, 3e3, 300)]
    sk = [orc.tensor_scale(a, 2688.0) for a in rng.uniform(1e-3, 3e3, 300)]
    sq += [np.float32(1.0), np.float32(2.0 ** -7), np.float32(1 + 2 ** -12)]
    sk += [np.float32(3.0), np.float32(2.0 ** 5), np.float32(1 + 2 ** -12)]
    for a, b in zip(sq, sk):
        ab = _rn32(Fraction(float(a)) * Fraction(float(b)))
        want = _rn32(Fraction(float(ab)) * Fraction(float(c)))
        assert orc.score_scale_log2(a, b) == float(want), (a, b)


def test_lse_is_natural_log_of_scaled_logits():
    """The emulated forward's LSE is ln sum_j exp(s_q s_k q_i.k_j / sqrt(d))
    over the dequantized codes (tensor scales included), and O is the softmax
    average of s_v-scaled V: checked against exact fp64 attention run on the
    scaled dequantized operands.  Unrounded P: agreement to fp32 rounding of
    the scale; rounded P (the method): within the E4M3 rounding of P."""
    rng = np.random.default_rng(93)
    n = 256
    qc = rng.integers(0, 256, (1, 1, n, 64), dtype=np.uint8)
    kc = rng.integers(0, 256, (1, 1, n, 64), dtype=np.uint8)
    qs = rng.integers(0x28, 0x40, (1, 1, n, 8), dtype=np.uint8)
    ks = rng.integers(0x28, 0x40, (1, 1, n, 8), dtype=np.uint8)
    vc = rng.integers(0, 0x7F, (1, 1, n, 128), dtype=np.uint8)
    vc[vc == 0x7F] = 0x7E
    s_q, s_k, s_v = np.float32(0.0173), np.float32(0.00911), np.float32(0.0377)
    qz = dict(qc=qc, qs=qs, qbc=None, qbs=None, s_q=s_q)
    kz = dict(kc=kc, ks=ks, s_k=s_k)
    vz = dict(vc=vc, s_v=s_v)
    q = orc.nvfp4_dequant(qc[0, 0], qs[0, 0]) * float(s_q)
    k = orc.nvfp4_dequant(kc[0, 0], ks[0, 0]) * float(s_k)
    v = orc.fp8_dequant(vc[0, 0]) * float(s_v)
    for causal in (False, True):
        o_ex, l_ex = orc.attn_exact(q, k, v, causal=causal)
        cs = orc.score_scale_log2(s_q, s_k)
        o1, l1 = orc.attn_online(orc.nvfp4_dequant(qc[0, 0], qs[0, 0]), None,
                                 orc.nvfp4_dequant(kc[0, 0], ks[0, 0]), orc.fp8_dequant(vc[0, 0]),
                                 score_scale=cs, out_scale=float(s_v), causal=causal,
                                 round_p=False)
        np.testing.assert_allclose(l1, l_ex, rtol=0, atol=1e-5 * max(1.0, np.abs(l_ex).max()))
        np.testing.assert_allclose(o1, o_ex, rtol=1e-4, atol=1e-5)
        o2, l2 = orc.prefill_emulate(qz, kz, vz, causal=causal)[(0, 0)]
        assert np.abs(l2 - l_ex).max() < math.log(1 + 2.0 ** -4)
        assert np.linalg.norm(o2 - o_ex) / np.linalg.norm(o_ex) < 0.03


# --------------------------------------------------------------------------
# decode: the rank-one block is the g query heads of one KV head
# --------------------------------------------------------------------------

def test_decode_zero_mean_groups_make_compensation_vanish():
    """Query heads of each KV head's group paired (x, -x): every group mean is
    0, so the decode codes and O are the same with and without the smoothing.
    Grouping heads by h % Hkv instead of h // g would mix x with another
    group's rows and give non-zero means."""
    rng = np.random.default_rng(95)
    B, Hkv, g, L = 2, 3, 4, 384
    x = _bf16(rng.standard_normal((B, Hkv, g // 2, 128)) * 1.3)
    q = np.concatenate([x, -x], axis=2).reshape(B, Hkv * g, 128)     # heads (x0, x1, -x0, -x1)
    K = _bf16(rng.standard_normal((B, L, Hkv, 128)))
    V = _bf16(rng.standard_normal((B, L, Hkv, 128)))
    on = orc.quantize_q_decode(q, Hkv, True, 2)
    off = orc.quantize_q_decode(q, Hkv, False)
    assert on["s_q"] == off["s_q"]
    np.testing.assert_array_equal(on["qc"] & 0x77, off["qc"] & 0x77)
    np.testing.assert_array_equal(on["qs"], off["qs"])
    assert (on["qbs"] == 0).all() and (on["qbc"] & 0x77 == 0).all()
    kz, vz = orc.quantize_k(K), orc.quantize_v(V)
    lens = np.array([L, 200])
    a = orc.decode_emulate(on, kz, vz, lens, chunk=128)
    b = orc.decode_emulate(off, kz, vz, lens, chunk=128)
    for key in a:
        np.testing.assert_array_equal(a[key][0], b[key][0])
        assert a[key][1] == b[key][1]


def test_decode_compensation_exact_for_representable_group_means():
    """All g query heads of KV head k equal to a vector mu_k that NVFP4
    represents exactly (a different mu per group): with the smoothing, q' = 0
    and the rank-one term alone carries mu_k, so decode O equals the
    unsmoothed O bit for bit.  A rank-one block other than "the g heads of KV
    head h // g" (e.g. h % Hkv) would average different mu and break it."""
    rng = np.random.default_rng(97)
    B, Hkv, g, L = 2, 2, 4, 256
    s = 2.0 ** -6
    e4 = np.array([orc.e4m3_value(c) for c in range(0x30, 0x7F)])
    vals16 = np.array([orc.e2m1_value(int(c)) for c in range(16)])
    mus = np.empty((B, Hkv, 128))
    for b in range(B):
        for hk in range(Hkv):
            codes = rng.integers(0, 16, 128)
            codes[::16] = 7 + 8 * rng.integers(0, 2, 8)
            sb = rng.choice(e4, 8)
            sb[0] = 448.0
            mus[b, hk] = vals16[codes] * np.repeat(sb, 16) * s
    q = np.repeat(mus, g, axis=1).astype(np.float32)        # head h = mu[h // g]
    assert np.array_equal(_bf16(q), q)
    K = _bf16(rng.standard_normal((B, L, Hkv, 128)))
    V = _bf16(rng.standard_normal((B, L, Hkv, 128)))
    on = orc.quantize_q_decode(q, Hkv, True, 2)
    off = orc.quantize_q_decode(q, Hkv, False)
    assert on["s_q"] == off["s_q"] == np.float32(s)
    assert (on["qc"] & 0x77 == 0).all()                     # q' = 0 in every head
    assert (on["qbs"][:, :, 1] == 0).all()                   # mu exact: no residual term
    kz, vz = orc.quantize_k(K), orc.quantize_v(V)
    lens = np.array([L, 129])
    a = orc.decode_emulate(on, kz, vz, lens, chunk=128)
    b = orc.decode_emulate(off, kz, vz, lens, chunk=128)
    for key in a:
        np.testing.assert_array_equal(a[key][0], b[key][0])
        assert a[key][1] == b[key][1]
    assert not np.array_equal(a[(0, 0)][0], a[(0, g)][0])


# --------------------------------------------------------------------------
# K-side smoothing (an addition to the pages' method, resting on the
# softmax's invariance to a per-row shift of the logits): kbar, K' and the
# LSE term
# --------------------------------------------------------------------------

def _paired_blocks(rng, B, N, H, step, lim):
    """[B, N, H, 128] values on a grid of `step` in [-lim, lim] whose every
    128-key block of every (b, h) has exactly zero channel means (rows x and
    -x inside each block)."""
    half = np.clip(np.round(rng.standard_normal((B, N // 128, 64, H, 128)) * lim / 2 / step)
                   * step, -lim, lim)
    blocks = np.concatenate([half, -half], axis=2)           # [B, nblk, 128, H, 128]
    return blocks.reshape(B, N, H, 128).astype(np.float32)


def _exact_nvfp4_rows(rng, rows, s):
    """[rows, 128] values NVFP4 represents exactly with tensor scale s (a 6 in
    every 16-element block, the first block scale 448)."""
    e4 = np.array([orc.e4m3_value(c) for c in range(0x30, 0x7F)])
    vals16 = np.array([orc.e2m1_value(int(c)) for c in range(16)])
    out = np.empty((rows, 128))
    for r in range(rows):
        codes = rng.integers(0, 16, 128)
        codes[::16] = 7 + 8 * rng.integers(0, 2, 8)
        sb = rng.choice(e4, 8)
        sb[0] = 448.0
        out[r] = vals16[codes] * np.repeat(sb, 16) * s
    return out.astype(np.float32)


def test_key_means_of_shifted_zero_mean_keys():
    """K = K0 + c with every 128-key block of K0 at exactly zero channel
    mean and c a per-(b, KV head) channel vector: kbar is c exactly, K' is
    K0, so the smoothed codes, scales and s_k equal the unsmoothed ones of
    K0.  A mean over the wrong axis, over the query heads, or a K' of
    K + kbar breaks the equalities."""
    rng = np.random.default_rng(201)
    B, N, H = 2, 384, 3
    K0 = _paired_blocks(rng, B, N, H, 0.25, 4.0)
    c = (np.round(rng.standard_normal((B, H, 128)) * 8) / 4).clip(-8, 8).astype(np.float32)
    K = (K0 + c[:, None]).astype(np.float32)
    assert np.array_equal(_bf16(K), K) and np.array_equal(K - c[:, None], K0)
    sm = orc.quantize_k(K, smooth=True)
    ref = orc.quantize_k(K0)
    np.testing.assert_array_equal(sm["kbar"], c)
    assert sm["s_k"] == ref["s_k"]
    # magnitudes: K0's -x = -0 where x = 0 codes a negative zero, K - c a positive one
    np.testing.assert_array_equal(sm["kc"] & 0x77, ref["kc"] & 0x77)
    np.testing.assert_array_equal(sm["ks"], ref["ks"])
    assert orc.quantize_k(K)["kbar"] is None


def test_key_means_are_the_mean_of_block_means():
    """Keys constant inside each 128-key block (value v_blk per channel):
    the block means are v_blk and kbar is their fp64 mean rounded to fp32,
    here exact: (1 + 2 + 3 + 6) / 4 = 3 in channel 0, and a channel-dependent
    closed form elsewhere."""
    v = np.array([1.0, 2.0, 3.0, 6.0])
    ch = np.arange(128) / 8.0 - 8.0                     # exact in bf16
    K = np.empty((1, 512, 1, 128), np.float32)
    for blk in range(4):
        K[0, blk * 128:(blk + 1) * 128, 0, :] = v[blk] * (1.0 + 0 * ch) + ch
    kb = orc.key_channel_means(K)[0, 0]
    np.testing.assert_array_equal(kb, (3.0 + ch).astype(np.float32))


def test_k_smoothing_keeps_o_and_moves_lse_by_the_dropped_logit():
    """Exactly representable Q (so the dequantized query is Q itself) against
    K = K0 + c: with K-side smoothing the emulated O is bit-identical to the
    one on K0, and the LSE differs from it by exactly what fp64 attention on
    the unquantized inputs says the shift c adds, q.c / sqrt(d) -- in
    prefill (causal and not) and in split-KV decode."""
    rng = np.random.default_rng(203)
    B, N, Hq, Hkv = 1, 256, 4, 2
    s = 2.0 ** -6
    Q = _exact_nvfp4_rows(rng, B * N * Hq, s).reshape(B, N, Hq, 128)
    K0 = _paired_blocks(rng, B, N, Hkv, 0.25, 4.0)
    c = (np.round(rng.standard_normal((B, Hkv, 128)) * 8) / 4).clip(-8, 8).astype(np.float32)
    K = (K0 + c[:, None]).astype(np.float32)
    V = _bf16(rng.standard_normal((B, N, Hkv, 128)))
    qz = orc.quantize_q_prefill(Q, False)
    assert qz["s_q"] == np.float32(s)
    np.testing.assert_array_equal(orc.query_effective(qz, 0, 1, 2), Q[0, :, 1, :])
    kz_s, kz_0, vz = orc.quantize_k(K, smooth=True), orc.quantize_k(K0), orc.quantize_v(V)
    for causal in (False, True):
        a = orc.prefill_emulate(qz, kz_s, vz, causal=causal)
        b = orc.prefill_emulate(qz, kz_0, vz, causal=causal)
        ea = orc.prefill_exact(Q, K, V, causal=causal)
        eb = orc.prefill_exact(Q, K0, V, causal=causal)
        for key in a:
            np.testing.assert_array_equal(a[key][0], b[key][0])
            np.testing.assert_allclose(ea[key][0], eb[key][0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(a[key][1] - b[key][1], ea[key][1] - eb[key][1],
                                       rtol=0, atol=1e-9)
            assert np.abs(a[key][1] - b[key][1]).max() > 0.1
    # decode: the last query row of each head against the first L keys
    q = Q[:, -1].copy()                                   # [B, Hq, 128]
    qd = orc.quantize_q_decode(q, Hkv, False)
    np.testing.assert_array_equal(orc.query_effective(qd, 0, 1, 2)[0], q[0, 1])
    lens = np.array([200])
    da = orc.decode_emulate(qd, kz_s, vz, lens, chunk=128)
    db = orc.decode_emulate(qd, kz_0, vz, lens, chunk=128)
    xa = orc.decode_exact(q, K, V, lens)
    xb = orc.decode_exact(q, K0, V, lens)
    for key in da:
        np.testing.assert_array_equal(da[key][0], db[key][0])
        assert abs((da[key][1] - db[key][1]) - (xa[key][1] - xb[key][1])) < 1e-9


def test_k_smoothing_reduces_error_on_key_offsets():
    """The tiny configuration (K channel offsets and four x20 outlier
    channels): K-side smoothing lowers the emulated output's error against
    exact fp64 attention, with and without the query-side term."""
    import mpfa_inputs as mi
    Q, K, V = mi.prefill_inputs(mi.PREFILL["tiny_n256"], "cpu", 0)
    Qn, Kn, Vn = (t.float().numpy() for t in (Q, K, V))
    ex = orc.prefill_exact(Qn, Kn, Vn, causal=False)[(0, 0)][0]
    vz = orc.quantize_v(Vn)
    for comp in (False, True):
        qz = orc.quantize_q_prefill(Qn, comp)
        e = {}
        for sm in (False, True):
            o = orc.prefill_emulate(qz, orc.quantize_k(Kn, smooth=sm), vz, causal=False)[(0, 0)][0]
            e[sm] = _rel_l2(o, ex)
        assert e[True] < 0.85 * e[False], (comp, e)


# --------------------------------------------------------------------------
# full-FP4 PV ablation (P and V^T in NVFP4)
# --------------------------------------------------------------------------

def _nvfp4_p_direct(x, s_p):
    """P in NVFP4 written out independently: per 16 values the E4M3 block
    scale (torch's cast) of fp32(max / fp32(6 s_p)), the fp32 divisor
    fp32(sb * s_p), E2M1 by the rint grid; returns the dequantized values."""
    x = np.asarray(x, np.float32)
    out = np.zeros(x.shape, np.float64)
    six_s = np.float32(np.float32(6.0) * np.float32(s_p))
    for b0 in range(0, x.shape[-1], 16):
        blk = x[..., b0:b0 + 16]
        bamax = blk.max(axis=-1, keepdims=True)
        sb = _e4m3(np.float32(bamax / six_s))
        denom = (sb.astype(np.float32) * np.float32(s_p)).astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            y = np.where(sb > 0, (blk / denom).astype(np.float32), 0.0)
        out[..., b0:b0 + 16] = _rne_grid_e2m1(y) * denom.astype(np.float64)
    return out


@pytest.mark.parametrize("n", [16, 100, 128])
def test_single_tile_fp4_p_direct_formula(n):
    """One KV tile with P in NVFP4 (round_p = 2): x = fp32(2^4 2^(t - max t)),
    P = NVFP4(x) with s_p = fp32(2^(4 + tau) / 2688) written out with torch's
    e4m3 cast and the rint E2M1 grid; O = sum P v / sum P,
    LSE = ln2 (max t + log2 sum P - 4)."""
    q, k, v = _rand_qkv(n, seed=400 + n, scale=1.3)
    o1, l1 = orc.attn_online(q, None, k, v, score_scale=LOG2E_RSQRT_D, out_scale=1.0,
                             causal=False, round_p=2)
    t = (q @ k.T) * LOG2E_RSQRT_D
    m = t.max(axis=1, keepdims=True)
    x = (np.exp2(t - m + P_SHIFT_READING)).astype(np.float32)
    pad = (-n) % 16
    xp = np.pad(x, ((0, 0), (0, pad)))
    s_p = np.float32(2.0 ** (P_SHIFT_READING + TAU_READING) / 2688.0)
    p4 = _nvfp4_p_direct(xp, s_p)[:, :n]
    o2 = (p4 @ v) / p4.sum(axis=1, keepdims=True)
    l2 = math.log(2) * (m[:, 0] + np.log2(p4.sum(axis=1)) - P_SHIFT_READING)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


def test_fp4_v_quantizer_is_nvfp4_of_v_transposed():
    """quantize_v_fp4 codes the keys of each (b, KV head, channel) row with
    the pinned NVFP4 quantizer at s_v = fp32(amax(V) / 2688)."""
    rng = np.random.default_rng(5)
    V = (rng.standard_normal((2, 256, 2, 128)) * np.exp(rng.uniform(-2, 2, (1, 256, 1, 1)))).astype(np.float32)
    vz = orc.quantize_v_fp4(V)
    assert vz["s_v"] == np.float32(np.float32(np.abs(V).max()) / np.float32(2688.0))
    for b in range(2):
        for h in range(2):
            c, sc = orc.nvfp4_quantize(np.ascontiguousarray(V[b, :, h, :].T), vz["s_v"])
            np.testing.assert_array_equal(vz["vc4"][b, h], c)
            np.testing.assert_array_equal(vz["vs4"][b, h], sc)


def test_fp4_pv_constant_v_gives_constant_o():
    """With V constant, every V^T code and block scale are equal, so the
    full-FP4 emulation's O is that one dequantized value on every row,
    causal, over several tiles: the same P codes enter l and PV."""
    B, N, Hq, Hkv = 1, 384, 2, 1
    rng = np.random.default_rng(6)
    Q = rng.standard_normal((B, N, Hq, 128)).astype(np.float32)
    K = rng.standard_normal((B, N, Hkv, 128)).astype(np.float32)
    V = np.full((B, N, Hkv, 128), 0.75, np.float32)
    qz, kz = orc.quantize_q_prefill(Q, True, 2), orc.quantize_k(K)
    vz = orc.quantize_v_fp4(V)
    val = orc.nvfp4_dequant(vz["vc4"][0, 0], vz["vs4"][0, 0]) * np.float64(vz["s_v"])
    assert np.all(val == val.flat[0])
    em = orc.prefill_emulate(qz, kz, vz, causal=True)
    for key, (o, _) in em.items():
        # exact up to the fp64 rounding of sum P v against v sum P
        np.testing.assert_allclose(o, np.full_like(o, val.flat[0]), rtol=1e-14, atol=0)


def test_fp4_pv_uniform_scores_average_v():
    """Q = 0: every visible score is 0, so every P code is the same and O is
    the plain mean of the visible rows of the dequantized V^T (closed form);
    LSE = ln(visible keys) up to the rounding of P (x = 16 maps to code 6 of
    a block scale 28)."""
    B, N, Hkv = 1, 256, 1
    rng = np.random.default_rng(7)
    Q = np.zeros((B, N, 1, 128), np.float32)
    K = rng.standard_normal((B, N, Hkv, 128)).astype(np.float32)
    V = rng.standard_normal((B, N, Hkv, 128)).astype(np.float32)
    qz, kz = orc.quantize_q_prefill(Q, False, 2), orc.quantize_k(K)
    vz = orc.quantize_v_fp4(V)
    vd = (orc.nvfp4_dequant(vz["vc4"][0, 0], vz["vs4"][0, 0]) * np.float64(vz["s_v"])).T
    (o, lse), = orc.prefill_emulate(qz, kz, vz, causal=True).values()
    want = np.cumsum(vd, axis=0) / np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, np.log(np.arange(1, N + 1)), atol=1e-6)


@pytest.mark.parametrize("delta", [2.5, 3.9, 4.5])
def test_two_tile_fp4_p_reference_max(delta):
    """Two KV tiles with P in NVFP4: while tile 1's max stays within tau of
    tile 0's, x reaches 2^(4 + delta) under the stale reference and the
    tensor scale s_p = 2^(4 + tau) / 2688 keeps the block scales unsaturated
    (a smaller s_p would clip them at 448); past tau the reference moves and
    tile 0 is rescaled by 2^-delta.  Direct formula as in the one-tile pin."""
    rng = np.random.default_rng(int(delta * 10) + 90)
    t0 = rng.uniform(-6, 0, 128)
    t0[5] = 0.0
    t1 = rng.uniform(-6, 0, 128) + delta
    t1[77] = delta
    tt = np.concatenate([t0, t1])
    q = np.zeros((1, 128)); q[0, 0] = 1.0
    k = np.zeros((256, 128)); k[:, 0] = tt
    v = rng.standard_normal((256, 128))
    o1, l1 = orc.attn_online(q, None, k, v, score_scale=1.0, out_scale=1.0, causal=False,
                             round_p=2)
    s_p = np.float32(2.0 ** (P_SHIFT_READING + TAU_READING) / 2688.0)
    sh = 2.0 ** P_SHIFT_READING
    if delta <= TAU_READING:
        p4 = _nvfp4_p_direct((np.exp2(tt) * sh).astype(np.float32)[None], s_p)[0]
        o2 = p4 @ v / p4.sum()
        l2 = math.log(2) * (math.log2(p4.sum()) - P_SHIFT_READING)
        assert p4[128:].max() > sh                 # beyond a fresh maximum's 16
    else:
        p0 = _nvfp4_p_direct((np.exp2(t0) * sh).astype(np.float32)[None], s_p)[0]
        p1 = _nvfp4_p_direct((np.exp2(t1 - delta) * sh).astype(np.float32)[None], s_p)[0]
        alpha = 2.0 ** -delta
        o2 = (alpha * (p0 @ v[:128]) + p1 @ v[128:]) / (alpha * p0.sum() + p1.sum())
        l2 = math.log(2) * (delta + math.log2(alpha * p0.sum() + p1.sum()) - P_SHIFT_READING)
    np.testing.assert_allclose(o1[0], o2, rtol=1e-12, atol=1e-13)
    assert abs(l1[0] - l2) < 1e-12
