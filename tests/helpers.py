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
