"""Seeded synthetic workloads for the MpFA attention forward.

This module draws random tensors and nothing else: it holds none of the
method's arithmetic.  Both the CPU oracle (through the tests) and the CUDA
library (through the tests and ``bench.py``) take their inputs from here.

The shapes stand in for the model attention layers the MpFA abstract names
(Llama-3.1-8B: 32 query / 8 KV heads; Qwen3-14B: 40 / 8; d = 128; 16K-128K
context) and for the kernel-level shape grid of the FP4 FlashAttention-4
explainer (B1/S4096/H24, B1/S8192/H64).  No model weights or benchmark
suites are available, so activations are drawn from the stated
distributions:

* Q, K, V ~ N(0, 1) in fp32, shape [B, N, H, d] (decode: q [B, Hq, d] and a
  cache K, V [B, Lmax, Hkv, d]).
* K channel offset per (KV head, channel) ~ N(0, 2) (variance 2).
* K outlier channels: ``k_outliers`` channels per KV head, chosen by
  ``randperm``, scaled x20 (offset included).
* V outlier entries: each entry independently with probability
  ``v_outlier_p``, scaled x10.
* Optional Q channel offset per (query head, channel) ~ N(0, 2).
* Everything is cast to bf16 last.

Draw order (one ``torch.Generator`` seeded with ``seed``): Q, K, V normals;
K offset; Q offset (if any); outlier channel permutations, one per KV head;
V outlier uniforms; decode lengths (if any).  The same seed on a CPU and a
CUDA generator gives different tensors, so each caller fixes its device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    causal: bool
    k_offset: bool = True
    k_outliers: int = 0
    v_outlier_p: float = 0.0
    q_offset: bool = False
    d: int = 128

    @property
    def pairs(self) -> int:
        """(query, key) pairs the forward scores, all heads."""
        n = self.N
        per_head = n * (n + 1) // 2 if self.causal else n * n
        return self.B * self.Hq * per_head


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    Lmax: int
    len_lo: int      # lengths ~ U[len_lo, len_hi] (integers); equal -> uniform length
    len_hi: int
    k_offset: bool = True
    k_outliers: int = 1
    v_outlier_p: float = 0.001
    d: int = 128


PREFILL = {
    # Tiny non-causal forward (one head, N = 256), K offset + 4 outlier channels.
    "tiny_n256": PrefillConfig("tiny_n256", 1, 1, 1, 256, False, True, 4, 0.0),
    # Same with a per-channel Q offset, so the rank-one smoothing has a mean to remove.
    "tiny_n256_qoffset": PrefillConfig("tiny_n256_qoffset", 1, 1, 1, 256, False, True, 4, 0.0,
                                       q_offset=True),
    # Llama-3.1-8B attention shape, causal prefill at 16K.
    "llama8b_n16k_causal": PrefillConfig("llama8b_n16k_causal", 1, 32, 8, 16384, True, True, 1,
                                         0.001),
    # Qwen3-14B attention shape, causal prefill at 128K.
    "qwen14b_n128k_causal": PrefillConfig("qwen14b_n128k_causal", 1, 40, 8, 131072, True, True,
                                          1, 0.001),
    # Kernel-level non-causal grid, plain N(0,1).
    "b1_s4096_h24": PrefillConfig("b1_s4096_h24", 1, 24, 24, 4096, False, False, 0, 0.0),
    "b1_s8192_h64": PrefillConfig("b1_s8192_h64", 1, 64, 64, 8192, False, False, 0, 0.0),
}

DECODE = {
    "decode_b64_l32k": DecodeConfig("decode_b64_l32k", 64, 32, 8, 32768, 32768, 32768),
    "decode_b64_l4k_64k": DecodeConfig("decode_b64_l4k_64k", 64, 32, 8, 65536, 4096, 65536),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _outlier_channels(g, hkv, d, count, device):
    idx = []
    for _ in range(hkv):
        idx.append(torch.randperm(d, generator=g, device=device)[:count])
    return torch.stack(idx) if count > 0 else None


def _shape_k(K, g, hkv, d, cfg, device):
    """K + channel offset, then outlier channels x20 (in place on fp32 K [..., hkv, d])."""
    if cfg.k_offset:
        off = torch.randn(hkv, d, generator=g, device=device) * math.sqrt(2.0)
        K += off
    return K


def prefill_inputs(cfg: PrefillConfig, device="cpu", seed: int = 0):
    """Q [B,N,Hq,d], K, V [B,N,Hkv,d] as bf16 on `device`."""
    g = _gen(device, seed)
    B, N, d = cfg.B, cfg.N, cfg.d
    Q = torch.randn(B, N, cfg.Hq, d, generator=g, device=device)
    K = torch.randn(B, N, cfg.Hkv, d, generator=g, device=device)
    V = torch.randn(B, N, cfg.Hkv, d, generator=g, device=device)
    _shape_k(K, g, cfg.Hkv, d, cfg, device)
    if cfg.q_offset:
        Q += torch.randn(cfg.Hq, d, generator=g, device=device) * math.sqrt(2.0)
    ch = _outlier_channels(g, cfg.Hkv, d, cfg.k_outliers, device)
    if ch is not None:
        for h in range(cfg.Hkv):
            K[:, :, h, ch[h]] *= 20.0
    if cfg.v_outlier_p > 0:
        mask = torch.rand(V.shape, generator=g, device=device) < cfg.v_outlier_p
        V[mask] *= 10.0
    return Q.to(torch.bfloat16), K.to(torch.bfloat16), V.to(torch.bfloat16)


def decode_inputs(cfg: DecodeConfig, device="cpu", seed: int = 0):
    """q [B,Hq,d]; cache K, V [B,Lmax,Hkv,d] bf16; seqlens int32 [B]."""
    g = _gen(device, seed)
    B, L, d = cfg.B, cfg.Lmax, cfg.d
    q = torch.randn(B, cfg.Hq, d, generator=g, device=device)
    K = torch.randn(B, L, cfg.Hkv, d, generator=g, device=device)
    V = torch.randn(B, L, cfg.Hkv, d, generator=g, device=device)
    _shape_k(K, g, cfg.Hkv, d, cfg, device)
    ch = _outlier_channels(g, cfg.Hkv, d, cfg.k_outliers, device)
    if ch is not None:
        for h in range(cfg.Hkv):
            K[:, :, h, ch[h]] *= 20.0
    if cfg.v_outlier_p > 0:
        mask = torch.rand(V.shape, generator=g, device=device) < cfg.v_outlier_p
        V[mask] *= 10.0
    if cfg.len_lo == cfg.len_hi:
        seqlens = torch.full((B,), cfg.len_hi, dtype=torch.int32, device=device)
    else:
        seqlens = torch.randint(cfg.len_lo, cfg.len_hi + 1, (B,), generator=g, device=device,
                                dtype=torch.int32)
    return q.to(torch.bfloat16), K.to(torch.bfloat16), V.to(torch.bfloat16), seqlens


def append_inputs(B: int, n_new: int, Hkv: int, device="cpu", seed: int = 0, d: int = 128,
                  spike: float = 0.0):
    """New decode tokens to append to a cache: K, V [B, n_new, Hkv, d] bf16,
    N(0,1) draws; with spike > 0, one K channel and every 7th V element of
    the first new token of each sequence are scaled by spike (values beyond
    the cache's quantization range)."""
    g = _gen(device, seed)
    K = torch.randn(B, n_new, Hkv, d, generator=g, device=device)
    V = torch.randn(B, n_new, Hkv, d, generator=g, device=device)
    if spike > 0:
        K[:, 0, :, 3] *= spike
        V[:, 0, :, ::7] *= spike
    return K.to(torch.bfloat16), V.to(torch.bfloat16)


def custom_prefill(B, Hq, Hkv, N, causal, *, k_offset=True, k_outliers=1, v_outlier_p=0.001,
                   q_offset=False, name="custom") -> PrefillConfig:
    return PrefillConfig(name, B, Hq, Hkv, N, causal, k_offset, k_outliers, v_outlier_p,
                         q_offset)


def custom_decode(B, Hq, Hkv, Lmax, len_lo, len_hi, name="custom") -> DecodeConfig:
    return DecodeConfig(name, B, Hq, Hkv, Lmax, len_lo, len_hi)
