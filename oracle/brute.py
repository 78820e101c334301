"""Second, NumPy-only decode attention for tiny inputs (test infrastructure only).

Independent of ``pa_oracle.c``: the pool is indexed as a six-dimensional NumPy
array [num_blocks, 2, L, Hkv, B, D] (mini-infer BlockPool layout) rather than
through hand-written offsets, and the softmax is the textbook exp/sum over the
gathered scores.  Used only to cross-check the C oracle on small cases.
"""
from __future__ import annotations

import numpy as np


def decode_attention(q64: np.ndarray, pool64: np.ndarray, layer: int, block_tables,
                     context_lens, num_heads: int, scale: float) -> np.ndarray:
    nb, _, L, Hkv, B, D = pool64.shape
    g = num_heads // Hkv
    batch = len(context_lens)
    out = np.zeros((batch, num_heads, D))
    for b in range(batch):
        n = int(context_lens[b])
        if n == 0:
            continue
        blocks = [int(x) for x in block_tables[b][: -(-n // B)]]
        for h in range(num_heads):
            kvh = h // g
            K = np.concatenate([pool64[blk, 0, layer, kvh] for blk in blocks])[:n]
            V = np.concatenate([pool64[blk, 1, layer, kvh] for blk in blocks])[:n]
            s = scale * (K @ q64[b, h])
            w = np.exp(s - s.max())
            out[b, h] = (w / w.sum()) @ V
    return out
