"""Shared test helpers: run the oracle on the same seeded inputs the CUDA path
gets, and compare.  Only tests import this module."""
import numpy as np
import torch

import oracle as orc


def tiled_to_rows(tiled: np.ndarray, rows: int) -> np.ndarray:
    """Block scales in the library's 128-row tile layout -> [rows, 8]."""
    r = np.arange(rows).reshape(-1, 1)
    j = np.arange(8).reshape(1, -1)
    off = (r // 128) * 1024 + (j // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (j % 4)
    return np.asarray(tiled).reshape(-1)[off]


def np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def cosine(a, b) -> float:
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / max(np.linalg.norm(a) * np.linalg.norm(b), 1e-300))


def oracle_quantize(Q, K, V, compensate, T):
    """Oracle codes for bf16 torch tensors Q [B,N,Hq,d], K, V (any on any device)."""
    out = {}
    if Q is not None:
        out["q"] = orc.quantize_q_prefill(np_f32(Q), compensate, T)
    if K is not None:
        out["k"] = orc.quantize_k(np_f32(K))
    if V is not None:
        out["v"] = orc.quantize_v(np_f32(V))
    return out


# Full-FP4 PV: decisions that may fall either way in fp32 arithmetic
S_P = np.float32(256.0 / 2688.0)
# How far the kernel's log2 scores may sit from the oracle's fp64 ones: fp32
# accumulation of the score products in another order (relative ~1e-6 of
# scores up to ~20) plus the hardware exponential (2^-22 relative).
T_SLACK = 1e-5


def fp4p_flip_allowance(qz, kz, vz, b, h, g):
    """Single 128-key tile per row (N = 128, causal), so m is the row max and
    x = 2^(t - m + 4).  A block-scale or code decision whose x lies within
    T_SLACK (log2 units) of an E4M3 or E2M1 rounding boundary may fall either
    way in fp32 arithmetic: each such unit (a whole block if its scale moves,
    else one key) may move O by |dP (v - o)| / l and l by |sum dP|.  Returns
    the per-element sum of the O moves [rows, d] and the bound on the LSE's
    move, -ln(1 - s) with s the sum of the relative l moves [rows]."""
    q, qadd, k, _ = orc._head_operands(qz, kz, None, b, h, g)
    v = orc.nvfp4_dequant(vz["vc4"][b, h // g], vz["vs4"][b, h // g]).T * np.float64(vz["s_v"])
    return fp4p_first_tile_allowance(q + qadd, k, v, orc.score_scale_log2(qz["s_q"], kz["s_k"]),
                                     np.arange(q.shape[0]))


def fp4p_first_tile_allowance(qe, k, v, cs, rows):
    """The flip allowance of fp4p_flip_allowance for causal query rows < 128
    (rows: their indices), whose keys all lie in the first 128-key tile:
    qe the rows' effective query vectors [len(rows), d] (dequantized, rank-one
    terms added, no tensor scale), k and v the head's first 128 keys and
    values (v with its tensor scale)."""
    rows = np.asarray(rows)
    assert (rows < 128).all()
    t = qe @ k[:128].T * cs
    t = np.where(np.arange(128)[None, :] > rows[:, None], -np.inf, t)
    m = t.max(axis=1, keepdims=True)
    v = v[:128]

    def quant(tt):
        c, sc = orc.nvfp4_quantize(np.exp2(tt - m + 4).astype(np.float32), S_P)
        return orc.nvfp4_dequant(c, sc) * np.float64(S_P), sc

    P, sc = quant(t)
    l = P.sum(axis=1, keepdims=True)
    o = P @ v / l
    n = len(rows)
    allow = np.zeros_like(o)
    rel_l = np.zeros(n)
    for shift in (T_SLACK, -T_SLACK):
        Pa, sca = quant(t + shift)
        for r in range(n):
            for blk in range(8):
                sl = slice(16 * blk, 16 * blk + 16)
                if sca[r, blk] != sc[r, blk]:
                    dP = Pa[r, sl] - P[r, sl]
                    allow[r] += np.abs(dP[None, :] @ (v[sl] - o[r])).ravel() / l[r, 0]
                    rel_l[r] += abs(dP.sum()) / l[r, 0]
                else:
                    for j in np.nonzero(Pa[r, sl] != P[r, sl])[0]:
                        key = 16 * blk + j
                        dp = Pa[r, key] - P[r, key]
                        allow[r] += np.abs(dp * (v[key] - o[r])) / l[r, 0]
                        rel_l[r] += abs(dp) / l[r, 0]
    assert (rel_l < 0.5).all()
    return allow, -np.log1p(-rel_l)
