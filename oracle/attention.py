"""Softmax attention over the dequantised cache, in float64.  Test infrastructure.

The pages describe the attention as reading the finished FP8 cache: each call
runs the new chunk's queries against all cached slots (5,788 slots of which
757 are new), 240 calls per step ([ai.info] § "La gestione della cache
spostata al momento della scrittura"; [neurocartel] § "Кэш: 240 attention
calls и работа на запись"; [wechild] ¶6).  Readings: non-causal (every query
sees every valid slot, its own chunk included), logits scaled by 1/sqrt(d),
no other mask.  The definition is written out with a library matmul:

    S = Q K^T / sqrt(d),   P = softmax_row(S),   O = P V
"""
from __future__ import annotations

import numpy as np


def attention_fp64(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """q [T][H][d], k and v [N][H][d] (any float type) -> O [T][H][d] float64."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    T, H, d = q.shape
    out = np.zeros((T, H, d), np.float64)
    if k.shape[0] == 0:
        return out
    for h in range(H):
        s = q[:, h, :] @ k[:, h, :].T / np.sqrt(d)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, h, :]
    return out


def attention_bruteforce(q, k, v):
    """Pure-Python triple loop of the same definition (tiny inputs only)."""
    import math

    T, H, d = len(q), len(q[0]), len(q[0][0])
    N = len(k)
    out = [[[0.0] * d for _ in range(H)] for _ in range(T)]
    for h in range(H):
        for i in range(T):
            logits = []
            for j in range(N):
                acc = 0.0
                for c in range(d):
                    acc += float(q[i][h][c]) * float(k[j][h][c])
                logits.append(acc / math.sqrt(d))
            m = max(logits)
            w = [math.exp(x - m) for x in logits]
            z = sum(w)
            for c in range(d):
                out[i][h][c] = sum(w[j] * float(v[j][h][c]) for j in range(N)) / z
    return out
