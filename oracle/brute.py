"""Independent numpy statement of the MoE expert layer for tiny shapes --
TEST INFRASTRUCTURE ONLY (same import rule as the rest of ``oracle/``).

It restates the same definition as ``moe_oracle.c`` with different means, so
that a slip in either one shows up as a disagreement:
  - nibbles unpacked by shifting whole arrays, not per element;
  - bf16 rounding by integer arithmetic on the fp64 bit pattern (the C oracle
    uses frexp/floor);
  - the scatter as a stable argsort of the expert ids (the C oracle counts);
  - expert FFNs as fp64 matrix products (the C oracle loops).
Sources: "Perplexity open-sources Lily" -- "three workload shapes" (256
experts, 8 picked, one shared expert) and "Prefill" (groupwise-affine 4-bit
weights with a bf16 scale and bias per 64 weights, rebuilt to bf16; routing
histogram, scan, scatter, block map).
"""
from __future__ import annotations

import numpy as np


def bf16_value(a: np.ndarray) -> np.ndarray:
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Nearest-even bf16 of fp64 values in the normal range (or zero)."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    ok = (a == 0) | ((a >= 2.0 ** -126) & (a < 3.3e38))
    assert ok.all(), "brute-force rounding handles zero and normal values only"
    bits = v.view(np.uint64).copy()
    lsb = (bits >> np.uint64(45)) & np.uint64(1)
    bits = bits + (np.uint64(1) << np.uint64(44)) - np.uint64(1) + lsb
    bits &= ~((np.uint64(1) << np.uint64(45)) - np.uint64(1))
    f32 = bits.view(np.float64).astype(np.float32)  # exact: 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def unpack_codes(q: np.ndarray) -> np.ndarray:
    """[rows, K/8] words -> [rows, K] codes, code k at bits 4*(k%8)."""
    q = np.asarray(q, np.uint32)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    codes = (q[:, :, None] >> shifts[None, None, :]) & np.uint32(15)
    return codes.reshape(q.shape[0], -1).astype(np.float64)


def dequant(q, s, b, G: int = 64) -> np.ndarray:
    codes = unpack_codes(q)
    sc = np.repeat(bf16_value(s), G, axis=1)
    bi = np.repeat(bf16_value(b), G, axis=1)
    prod = sc * codes
    hi = prod + bi
    # the fp64 sum must be exact for this rounding to be the exact rounding
    bb = hi - prod
    lo = (prod - (hi - bb)) + (bi - bb)
    assert not np.any(lo), "inexact fp64 sum: outside the brute force's range"
    return round_bf16_bits(hi)


def select(keys: np.ndarray, k: int):
    keys = np.asarray(keys, np.float32)
    T, E = keys.shape
    nan = np.isnan(keys)
    val = np.where(nan, 0.0, keys.astype(np.float64))
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    idx = np.arange(E)
    for t in range(T):
        order = np.lexsort((idx, -val[t], nan[t]))  # last key is primary
        ids[t] = order[:k]
        l = keys[t, order[:k]].astype(np.float64)
        ex = np.exp(l - l[0])
        w[t] = ex / ex.sum()
    return ids, w


def route_maps(ids: np.ndarray, E: int):
    flat = np.asarray(ids, np.int64).ravel()
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int32)
    return counts, offsets, perm, inv


def moe_layer(x, W: dict, E: int, k: int, n_shared: int, res=None, bias=None, keys=None, G: int = 64):
    """The layer for tiny shapes.  Returns (out bf16 bits, out fp64 before
    rounding, keys, ids, w)."""
    xd = bf16_value(x)
    T, H = xd.shape
    if keys is None:
        logits = xd @ W["router"].astype(np.float64).T
        keys = logits.astype(np.float32)
        if bias is not None:
            keys = (keys + np.asarray(bias, np.float32)[None, :]).astype(np.float32)
    ids, w = select(keys, k)
    counts, offsets, perm, inv = route_maps(ids, E)

    def ffn(e, rows):
        wg = bf16_value(dequant(W["gate_q"][e], W["gate_s"][e], W["gate_b"][e], G))
        wu = bf16_value(dequant(W["up_q"][e], W["up_s"][e], W["up_b"][e], G))
        wd = bf16_value(dequant(W["down_q"][e], W["down_s"][e], W["down_b"][e], G))
        g = rows @ wg.T
        u = rows @ wu.T
        h = bf16_value(round_bf16_bits(g / (1.0 + np.exp(-g)) * u))
        return bf16_value(round_bf16_bits(h @ wd.T))

    y = np.zeros((T, k, H))
    for e in range(E):
        if counts[e] == 0:
            continue
        pairs = perm[offsets[e]:offsets[e + 1]]
        yt = ffn(e, xd[pairs // k])
        y[pairs // k, pairs % k] = yt
    acc = bf16_value(x if res is None else res).copy()
    if n_shared:
        g = 1.0  # optional shared-expert gate: sigmoid of the expert input's dot with it
        if W.get("shared_gate") is not None:
            g = (1.0 / (1.0 + np.exp(-(xd @ np.asarray(W["shared_gate"], np.float64)))))[:, None]
        acc = acc + g * ffn(E, xd)
    for j in range(k):
        acc = acc + w[:, j:j + 1] * y[:, j]
    return round_bf16_bits(acc), acc, keys, ids, w
