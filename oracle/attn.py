"""CPU oracle for single-token (decode) attention over a KV cache -- TEST
INFRASTRUCTURE ONLY (same import rule as the rest of ``oracle/``: tests,
``smoke()`` and ``bench.py``'s CPU legs only; the product library never
imports it).

What it computes.  The pages ("Perplexity open-sources Lily" -- "three
workload shapes" and "Decode") describe the model's 10 full-attention layers
(grouped-query attention, 16 query heads sharing 2 KV heads), decode
attention over a KV cache that grows with the context, query heads of one KV
group sharing each KV row read ("GQA packing", +23.8 % at 32K) and a
fixed-block layout for long contexts (+40.2 % at 128K).  They print no
formula; this is scaled dot-product attention for one query token, per query
head h with KV head g = h // (Hq / Hkv):

    s_l = scale * (q_h . k_{l,g}),  p = softmax_l(s),  o_h = sum_l p_l v_{l,g}

over the L cached positions, with scale = 1 / sqrt(D) unless given.  The
oracle evaluates it in fp64 from the bf16 inputs; the GPU rounds o to bf16.

Parity status: pinned by ``tests/test_attn_oracle.py`` (equal keys give the
mean of the values, one dominant key selects its value, L = 1, invariance
under a permutation of the positions, the GQA head mapping, and agreement
with PyTorch's scaled_dot_product_attention on CPU).
"""
from __future__ import annotations

import numpy as np


def _f64(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def decode_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float | None = None) -> np.ndarray:
    """o [Hq, D] fp64 for one query token.  q [Hq, D]; k, v [L, Hkv, D]
    (bf16 bit patterns or float arrays)."""
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    Hq, D = qf.shape
    L, Hkv, _ = kf.shape
    assert Hq % Hkv == 0 and vf.shape == kf.shape and L >= 1
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.empty((Hq, D))
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = scale * (kf[:, g, :] @ qf[h])  # [L]
        p = np.exp(s - s.max())
        p /= p.sum()
        o[h] = p @ vf[:, g, :]
    return o
