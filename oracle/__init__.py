"""CPU oracle for the MpFA QK4PV8 attention forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The product
library never imports, links or runs it, and it imports nothing from the
product package.

The arithmetic lives in ``mpfa_oracle.c`` (plain C11, fp64 where the method
leaves the precision open, fp32 exactly where the quantizer rules say fp32).
This module compiles that file with gcc on first use and composes its
functions into the method's steps, following:

* "MpFA: Hardware-Efficient Train-Free QK4V8 FlashAttention Kernels on
  Blackwell GPUs", abstract -- QK in NVFP4, P and V in FP8, rank-one smoothing
  compensation as one extra MMA, split work for decode.
* "FlashAttention压到4位" explainer, section "FP4 只有约 15 个可表示的数" --
  E2M1 codebook, NVFP4 (16-element E4M3 block scale + FP32 tensor scale).
* the same explainer, section "注意力慢在哪儿" -- tiled online softmax.

All layouts here are logical row-major (see each function); the product's
tiled scale layout is converted by the tests, not here.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mpfa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

D = 128            # head dimension the method is specified for
QBLOCK = 128       # rows per query block of the rank-one smoothing (prefill)
NVFP4_QMAX = 6.0 * 448.0
FP8_QMAX = 448.0
P_SHIFT = 4        # P is stored as E4M3(2^4 p)
RESCALE_TAU = 4.0  # the row's reference max moves only when a tile max exceeds it by > 4


def build(force: bool = False) -> str:
    """Compile ``mpfa_oracle.c`` into ``liboracle.so`` (gcc, no fast-math)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
        sig = {
            "orc_e2m1_value": (f64, [i32]),
            "orc_e4m3_value": (f64, [i32]),
            "orc_e2m1_encode": (i32, [f64]),
            "orc_e4m3_encode": (i32, [f64]),
            "orc_tensor_scale": (f32, [f32, f32]),
            "orc_nvfp4_quantize": (None, [P, i64, i64, i32, f32, P, P, i32]),
            "orc_nvfp4_dequant": (None, [P, P, i64, i32, P]),
            "orc_fp8_quantize": (None, [P, i64, f32, P]),
            "orc_fp8_dequant": (None, [P, i64, P]),
            "orc_block_means": (None, [P, i64, i32, i64, i32, P, P, i32]),
            "orc_attn_online": (None, [P, P, P, P, i64, i64, i32, f64, f64, i32, i64, i64,
                                       i32, f64, f64, P, i64, P, P, i32]),
            "orc_attn_exact": (None, [P, P, P, i64, i64, i32, f64, i32, i64, P, i64, P, P,
                                      i32]),
            "orc_e2m1_encode_array": (None, [P, i64, P]),
            "orc_e4m3_encode_array": (None, [P, i64, P]),
            "orc_bf16_round_array": (None, [P, i64, P]),
            "orc_num_threads": (i32, [i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads(requested: int = 0) -> int:
    return _L().orc_num_threads(requested)


# ----------------------------------------------------------------------------
# formats
# ----------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return _L().orc_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return _L().orc_e4m3_value(int(code))


def e2m1_encode(y) -> np.ndarray:
    y = np.ascontiguousarray(np.asarray(y, dtype=np.float64).ravel())
    out = np.empty(y.size, np.uint8)
    _L().orc_e2m1_encode_array(_p(y), y.size, _p(out))
    return out


def e4m3_encode(y) -> np.ndarray:
    y = np.ascontiguousarray(np.asarray(y, dtype=np.float64).ravel())
    out = np.empty(y.size, np.uint8)
    _L().orc_e4m3_encode_array(_p(y), y.size, _p(out))
    return out


E2M1_TABLE = None
E4M3_TABLE = None


def _tables():
    global E2M1_TABLE, E4M3_TABLE
    if E2M1_TABLE is None:
        E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], np.float64)
        E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], np.float64)
    return E2M1_TABLE, E4M3_TABLE


def bf16_round(x) -> np.ndarray:
    """uint16 bf16 bits of the nearest bf16 (ties to even) of fp64 values."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, np.uint16)
    _L().orc_bf16_round_array(_p(x), x.size, _p(out))
    return out


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# quantizers
# ----------------------------------------------------------------------------

def tensor_scale(amax: float, qmax: float) -> np.float32:
    """fp32(amax / qmax); 1 when amax == 0."""
    return np.float32(_L().orc_tensor_scale(float(np.float32(amax)), float(np.float32(qmax))))


def nvfp4_quantize(x: np.ndarray, s: float, nthreads: int = 0):
    """NVFP4 codes [rows, d/2] (low nibble = lower index) and E4M3 block
    scales [rows, d/16] of fp32 rows x [rows, d] with tensor scale s."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, d = x.shape
    codes = np.empty((rows, d // 2), np.uint8)
    scales = np.empty((rows, d // 16), np.uint8)
    _L().orc_nvfp4_quantize(_p(x), rows, d, d, float(np.float32(s)), _p(codes), _p(scales),
                            nthreads)
    return codes, scales


def nvfp4_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """code * block scale (no tensor scale), fp64 [rows, d]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, d = codes.shape[0], codes.shape[1] * 2
    out = np.empty((rows, d), np.float64)
    _L().orc_nvfp4_dequant(_p(codes), _p(scales), rows, d, _p(out))
    return out


def fp8_quantize(x: np.ndarray, s: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    _L().orc_fp8_quantize(_p(x), x.size, float(np.float32(s)), _p(out))
    return out


def fp8_dequant(codes: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, np.float64)
    _L().orc_fp8_dequant(_p(codes), codes.size, _p(out))
    return out


def block_means(x: np.ndarray, g: int, nthreads: int = 0):
    """Rank-one smoothing inputs: x [nblocks*g, d] fp32 -> (qbar [nblocks, d],
    x' = fp32(x - qbar) [nblocks*g, d])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, d = x.shape
    assert rows % g == 0
    nb = rows // g
    qbar = np.empty((nb, d), np.float32)
    xp = np.empty((rows, d), np.float32)
    _L().orc_block_means(_p(x), nb, g, d, d, _p(qbar), _p(xp), nthreads)
    return qbar, xp


def _amax(x: np.ndarray) -> np.float32:
    return np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)


# ----------------------------------------------------------------------------
# the method's quantization steps (logical layouts)
# ----------------------------------------------------------------------------

def rank_one_terms(qbar: np.ndarray, s: float, T: int, nthreads: int = 0):
    """T-term NVFP4 expansion of the block means (all terms share the tensor
    scale s): term 1 quantizes qbar; term t > 1 quantizes the fp32 residual
    r_t = fp32(r_{t-1} - fp32(fp32(code * sb) * s)) left by term t-1.
    qbar [nb, d] fp32 -> codes [nb, T, d/2], scales [nb, T, d/16]."""
    nb, d = qbar.shape
    codes = np.empty((nb, T, d // 2), np.uint8)
    scales = np.empty((nb, T, d // 16), np.uint8)
    r = np.ascontiguousarray(qbar, np.float32)
    for t in range(T):
        c, sc = nvfp4_quantize(r, s, nthreads)
        codes[:, t], scales[:, t] = c, sc
        deq = nvfp4_dequant(c, sc).astype(np.float32)           # code * sb, exact in fp32
        r = (r - (deq * np.float32(s)).astype(np.float32)).astype(np.float32)
    return codes, scales


def quantize_q_prefill(Q: np.ndarray, compensate: bool, T: int = 2, nthreads: int = 0) -> dict:
    """Quantize Q [B, N, Hq, d] (fp32 holding bf16 values).

    compensate=False: s_q = fp32(amax(Q)/2688); codes of Q.
    compensate=True:  per 128-row block of one (b, h): qbar = fp32 mean,
      Q' = fp32(Q - qbar); s_q from max(amax(Q'), amax(qbar)); codes of Q'
      and the T-term expansion of qbar (rank_one_terms) share s_q.

    Returns qc [B,Hq,N,d/2], qs [B,Hq,N,d/16], qbc [B,Hq,N/128,T,d/2] | None,
    qbs [B,Hq,N/128,T,d/16] | None, s_q (np.float32), qbar fp32 | None.
    """
    B, N, H, d = Q.shape
    qc = np.empty((B, H, N, d // 2), np.uint8)
    qs = np.empty((B, H, N, d // 16), np.uint8)
    if not compensate:
        s = tensor_scale(_amax(Q), NVFP4_QMAX)
        for b in range(B):
            for h in range(H):
                c, sc = nvfp4_quantize(np.ascontiguousarray(Q[b, :, h, :]), s, nthreads)
                qc[b, h], qs[b, h] = c, sc
        return dict(qc=qc, qs=qs, qbc=None, qbs=None, s_q=s, qbar=None)
    assert N % QBLOCK == 0
    nb = N // QBLOCK
    qbar = np.empty((B, H, nb, d), np.float32)
    amax = np.float32(0.0)
    for b in range(B):
        for h in range(H):
            mb, xp = block_means(np.ascontiguousarray(Q[b, :, h, :]), QBLOCK, nthreads)
            qbar[b, h] = mb
            amax = max(amax, _amax(xp), _amax(mb))
    s = tensor_scale(amax, NVFP4_QMAX)
    qbc = np.empty((B, H, nb, T, d // 2), np.uint8)
    qbs = np.empty((B, H, nb, T, d // 16), np.uint8)
    for b in range(B):
        for h in range(H):
            _, xp = block_means(np.ascontiguousarray(Q[b, :, h, :]), QBLOCK, nthreads)
            qc[b, h], qs[b, h] = nvfp4_quantize(xp, s, nthreads)
            qbc[b, h], qbs[b, h] = rank_one_terms(qbar[b, h], s, T, nthreads)
    return dict(qc=qc, qs=qs, qbc=qbc, qbs=qbs, s_q=s, qbar=qbar)


def key_channel_means(K: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """K-side smoothing vector (an addition to the pages' method, resting on
    the softmax's invariance to a per-row shift of the logits, the
    explainer's attention section): per (b, KV head) and channel c,
    kbar_c = fp32(fp64(sum over the 128-key blocks, in block order, of the
    block's fp32 mean) / number of blocks), each block mean being the
    correctly rounded fp32 mean of its 128 keys (the rule of the query-side
    block means).  K [B, N, Hkv, d] fp32 holding bf16 values, N a multiple
    of 128 -> kbar [B, Hkv, d] fp32."""
    B, N, H, d = K.shape
    assert N % QBLOCK == 0
    kbar = np.empty((B, H, d), np.float32)
    for b in range(B):
        for h in range(H):
            means, _ = block_means(np.ascontiguousarray(K[b, :, h, :]), QBLOCK, nthreads)
            acc = np.zeros(d, np.float64)
            for blk in range(means.shape[0]):        # sequential, in block order
                acc = acc + means[blk].astype(np.float64)
            kbar[b, h] = (acc / np.float64(means.shape[0])).astype(np.float32)
    return kbar


def quantize_k(K: np.ndarray, nthreads: int = 0, smooth: bool = False) -> dict:
    """K [B, N, Hkv, d] -> kc [B,Hkv,N,d/2], ks [B,Hkv,N,d/16], s_k.

    smooth=True (K-side smoothing): kbar = key_channel_means(K), the codes
    are those of K' = fp32(K - kbar) with s_k from amax(K'), and kbar is
    returned with them (the logits then lack q.kbar, the same for every key
    of a query row, so O is unchanged and the LSE gets it back; see
    lse_shift)."""
    B, N, H, d = K.shape
    kbar = None
    if smooth:
        kbar = key_channel_means(K, nthreads)
        K = (np.asarray(K, np.float32) - kbar[:, None, :, :]).astype(np.float32)
    s = tensor_scale(_amax(K), NVFP4_QMAX)
    kc = np.empty((B, H, N, d // 2), np.uint8)
    ks = np.empty((B, H, N, d // 16), np.uint8)
    for b in range(B):
        for h in range(H):
            kc[b, h], ks[b, h] = nvfp4_quantize(np.ascontiguousarray(K[b, :, h, :]), s, nthreads)
    return dict(kc=kc, ks=ks, s_k=s, kbar=kbar)


def quantize_v(V: np.ndarray) -> dict:
    """V [B, N, Hkv, d] -> vc [B,Hkv,N,d] (E4M3 codes), s_v = fp32(amax/448)."""
    B, N, H, d = V.shape
    s = tensor_scale(_amax(V), FP8_QMAX)
    vc = np.empty((B, H, N, d), np.uint8)
    for b in range(B):
        for h in range(H):
            vc[b, h] = fp8_quantize(np.ascontiguousarray(V[b, :, h, :]), s)
    return dict(vc=vc, s_v=s)


def quantize_v_fp4(V: np.ndarray) -> dict:
    """V [B, N, Hkv, d] fp32 for the full-FP4 PV ablation: NVFP4 of V^T along
    the keys (the reduction dimension of P V), 16-key blocks, one tensor
    scale s_v = fp32(amax(V) / 2688).  Codes [B, Hkv, d, N/2], block scales
    [B, Hkv, d, N/16] (E4M3 bytes), logical row-major."""
    B, N, H, d = V.shape
    s = tensor_scale(_amax(V), NVFP4_QMAX)
    vt = np.ascontiguousarray(np.transpose(V, (0, 2, 3, 1))).reshape(B * H * d, N)
    codes, scales = nvfp4_quantize(vt, s)
    return {"vc4": codes.reshape(B, H, d, N // 2), "vs4": scales.reshape(B, H, d, N // 16),
            "s_v": s}


def quantize_q_decode(q: np.ndarray, Hkv: int, compensate: bool, T: int = 2) -> dict:
    """Decode query q [B, Hq, d]: the rank-one block is the g = Hq/Hkv query
    heads that share one KV head.  Returns qc [B,Hq,d/2], qs [B,Hq,d/16],
    qbc [B,Hkv,T,d/2] | None, qbs [B,Hkv,T,d/16] | None, s_q."""
    B, H, d = q.shape
    g = H // Hkv
    flat = np.ascontiguousarray(q.reshape(B * H, d), dtype=np.float32)
    if not compensate:
        s = tensor_scale(_amax(flat), NVFP4_QMAX)
        c, sc = nvfp4_quantize(flat, s)
        return dict(qc=c.reshape(B, H, d // 2), qs=sc.reshape(B, H, d // 16), qbc=None,
                    qbs=None, s_q=s)
    qbar, xp = block_means(flat, g)
    s = tensor_scale(max(_amax(xp), _amax(qbar)), NVFP4_QMAX)
    c, sc = nvfp4_quantize(xp, s)
    bc, bs = rank_one_terms(qbar, s, T)
    return dict(qc=c.reshape(B, H, d // 2), qs=sc.reshape(B, H, d // 16),
                qbc=bc.reshape(B, Hkv, T, d // 2), qbs=bs.reshape(B, Hkv, T, d // 16), s_q=s)


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------

def score_scale_log2(s_q: float, s_k: float, d: int = D) -> float:
    """fp32(fp32(s_q*s_k) * fp32(log2(e)/sqrt(d))): the factor that takes the
    accumulated code products to the log2-domain logit."""
    a = np.float32(np.float32(s_q) * np.float32(s_k))
    c = np.float32(math.log2(math.e) / math.sqrt(d))
    return float(np.float32(a * c))


def attn_online(q, qadd, k, v, *, score_scale, out_scale, causal, kv_len=None, chunk=0,
                round_p=True, p_shift=P_SHIFT, tau=RESCALE_TAU, rows=None, nthreads=0):
    """Tiled online-softmax attention of one head (see orc_attn_online).
    q, qadd [nq,d] fp64 (qadd may be None), k, v [nk,d] fp64.  P is stored as
    E4M3(2^p_shift p) (round_p 1 or True), left unrounded (0 or False), or in
    NVFP4 per 16-key block (2, the full-FP4 ablation); the row's reference
    max moves only when a tile's max exceeds it by more than tau (tau = 0:
    the exact running max)."""
    q = np.ascontiguousarray(q, np.float64)
    k = np.ascontiguousarray(k, np.float64)
    v = np.ascontiguousarray(v, np.float64)
    nq, d = q.shape
    nk = k.shape[0]
    qa = None if qadd is None else np.ascontiguousarray(qadd, np.float64)
    rows = np.arange(nq, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    o = np.empty((rows.size, d), np.float64)
    lse = np.empty(rows.size, np.float64)
    _L().orc_attn_online(_p(q), None if qa is None else _p(qa), _p(k), _p(v), nq, nk, d,
                         float(score_scale), float(out_scale), int(bool(causal)),
                         nk if kv_len is None else int(kv_len), int(chunk), int(round_p),
                         float(p_shift), float(tau), _p(rows), rows.size, _p(o), _p(lse), nthreads)
    return o, lse


def attn_exact(q, k, v, *, causal, kv_len=None, rows=None, nthreads=0):
    """Exact fp64 softmax attention of one head, z = q.k / sqrt(d)."""
    q = np.ascontiguousarray(q, np.float64)
    k = np.ascontiguousarray(k, np.float64)
    v = np.ascontiguousarray(v, np.float64)
    nq, d = q.shape
    nk = k.shape[0]
    rows = np.arange(nq, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    o = np.empty((rows.size, d), np.float64)
    lse = np.empty(rows.size, np.float64)
    _L().orc_attn_exact(_p(q), _p(k), _p(v), nq, nk, d, 1.0 / math.sqrt(d), int(bool(causal)),
                        nk if kv_len is None else int(kv_len), _p(rows), rows.size, _p(o),
                        _p(lse), nthreads)
    return o, lse


def _terms_sum(codes, scales):
    """Sum over the T rank-one terms of code * block scale: codes [nb, T, d/2]
    -> fp64 [nb, d] (exact: each term is exact in fp64)."""
    nb, T = codes.shape[:2]
    tot = 0.0
    for t in range(T):
        tot = tot + nvfp4_dequant(np.ascontiguousarray(codes[:, t]),
                                  np.ascontiguousarray(scales[:, t]))
    return tot


def _head_operands(qz, kz, vz, b, h, g):
    """Dequantized operands of query head h (KV head h // g), no tensor scales."""
    hk = h // g
    q = nvfp4_dequant(qz["qc"][b, h], qz["qs"][b, h])
    qadd = None
    if qz.get("qbc") is not None:
        qb = _terms_sum(qz["qbc"][b, h], qz["qbs"][b, h])           # [nblocks, d]
        qadd = np.repeat(qb, QBLOCK, axis=0)[: q.shape[0]]
    k = nvfp4_dequant(kz["kc"][b, hk], kz["ks"][b, hk])
    v = None if vz is None else fp8_dequant(vz["vc"][b, hk])
    return q, qadd, k, v


def query_effective(qz, b, h, g):
    """The query rows the method multiplies, dequantized with the tensor
    scale: s_q * (code * block scale of Q' (or Q) + the sum of the rank-one
    terms of the row's block), fp64 [rows, d].  Prefill codes (qz from
    quantize_q_prefill, rows = N) or decode codes (quantize_q_decode,
    one row; the rank-one block is KV head h // g)."""
    qc, qs = qz["qc"][b, h], qz["qs"][b, h]
    if qc.ndim == 1:
        qc, qs = qc[None], qs[None]
    q = nvfp4_dequant(qc, qs)
    if qz.get("qbc") is not None:
        if qz["qbc"].ndim == 5:        # prefill: [B, Hq, blocks, T, d/2]
            qb = _terms_sum(qz["qbc"][b, h], qz["qbs"][b, h])
            q = q + np.repeat(qb, QBLOCK, axis=0)[: q.shape[0]]
        else:                          # decode: [B, Hkv, T, d/2]
            q = q + _terms_sum(qz["qbc"][b, h // g][None], qz["qbs"][b, h // g][None])
    return q * np.float64(qz["s_q"])


def lse_shift(qz, kz, b, h, g, d=D):
    """K-side smoothing's LSE term of query head h of batch b: the logit
    part q_eff . kbar / sqrt(d) that the smoothed keys leave out, the same
    for every key of the row (fp64 [rows]); zero without smoothing."""
    q = query_effective(qz, b, h, g)
    if kz.get("kbar") is None:
        return np.zeros(q.shape[0])
    return q @ kz["kbar"][b, h // g].astype(np.float64) / math.sqrt(d)


def prefill_emulate(qz, kz, vz, *, causal, heads=None, rows=None, nthreads=0):
    """Emulate the QK4PV8 prefill on the oracle's own codes.

    qz/kz/vz from quantize_q_prefill / quantize_k / quantize_v, or vz from
    quantize_v_fp4 for the full-FP4 PV ablation (P in NVFP4 per 16-key
    block, V^T in NVFP4 along the keys).  heads: list of (b, h) (default
    all); rows: query rows per head (default all).
    Returns {(b, h): (o fp64 [nrows, d] before the bf16 cast, lse [nrows])}."""
    B, Hq, N = qz["qc"].shape[:3]
    Hkv = kz["kc"].shape[1]
    g = Hq // Hkv
    cs = score_scale_log2(qz["s_q"], kz["s_k"])
    heads = [(b, h) for b in range(B) for h in range(Hq)] if heads is None else heads
    out = {}
    fp4 = "vc4" in vz
    for (b, h) in heads:
        if fp4:
            q, qadd, k, _ = _head_operands(qz, kz, None, b, h, g)
            v = nvfp4_dequant(vz["vc4"][b, h // g], vz["vs4"][b, h // g]).T
        else:
            q, qadd, k, v = _head_operands(qz, kz, vz, b, h, g)
        o, lse = attn_online(q, qadd, k, v, score_scale=cs, out_scale=float(vz["s_v"]),
                             causal=causal, round_p=2 if fp4 else 1, rows=rows,
                             nthreads=nthreads)
        if kz.get("kbar") is not None:
            sh = lse_shift(qz, kz, b, h, g)
            lse = lse + (sh if rows is None else sh[np.asarray(rows)])
        out[(b, h)] = (o, lse)
    return out


def prefill_exact(Q, K, V, *, causal, heads=None, rows=None, nthreads=0):
    """Exact fp64 attention on the unquantized inputs, Q [B,N,Hq,d] etc."""
    B, N, Hq, d = Q.shape
    g = Hq // K.shape[2]
    heads = [(b, h) for b in range(B) for h in range(Hq)] if heads is None else heads
    out = {}
    for (b, h) in heads:
        out[(b, h)] = attn_exact(Q[b, :, h, :], K[b, :, h // g, :], V[b, :, h // g, :],
                                 causal=causal, rows=rows, nthreads=nthreads)
    return out


def decode_emulate(qz, kz, vz, seqlens, *, chunk, heads=None, nthreads=0):
    """Emulate split-KV decode: query head h of batch b against keys
    [0, seqlens[b]) of its KV head, chunks of `chunk` keys combined by LSE.
    qz from quantize_q_decode; kz/vz: caches [B,Hkv,Lmax,...].
    Returns {(b, h): (o fp64 [d], lse)}."""
    B, Hq = qz["qc"].shape[:2]
    Hkv = kz["kc"].shape[1]
    g = Hq // Hkv
    cs = score_scale_log2(qz["s_q"], kz["s_k"])
    heads = [(b, h) for b in range(B) for h in range(Hq)] if heads is None else heads
    out = {}
    cache = {}
    for (b, h) in heads:
        hk = h // g
        if (b, hk) not in cache:
            cache.clear()
            cache[(b, hk)] = (nvfp4_dequant(kz["kc"][b, hk], kz["ks"][b, hk]),
                              fp8_dequant(vz["vc"][b, hk]))
        k, v = cache[(b, hk)]
        q = nvfp4_dequant(qz["qc"][b, h][None], qz["qs"][b, h][None])
        qadd = None
        if qz.get("qbc") is not None:
            qadd = _terms_sum(qz["qbc"][b, hk][None], qz["qbs"][b, hk][None])
        o, lse = attn_online(q, qadd, k, v, score_scale=cs, out_scale=float(vz["s_v"]),
                             causal=False, kv_len=int(seqlens[b]), chunk=chunk,
                             nthreads=nthreads)
        if kz.get("kbar") is not None:
            lse = lse + lse_shift(qz, kz, b, h, g)
        out[(b, h)] = (o[0], lse[0])
    return out


def decode_exact(q, K, V, seqlens, *, heads=None):
    """Exact fp64 decode attention: q [B,Hq,d], K/V [B,Lmax,Hkv,d]."""
    B, Hq, d = q.shape
    g = Hq // K.shape[2]
    heads = [(b, h) for b in range(B) for h in range(Hq)] if heads is None else heads
    out = {}
    for (b, h) in heads:
        o, lse = attn_exact(q[b, h][None], K[b, :, h // g, :], V[b, :, h // g, :],
                            causal=False, kv_len=int(seqlens[b]), nthreads=1)
        out[(b, h)] = (o[0], lse[0])
    return out
