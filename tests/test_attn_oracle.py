"""Pins for the decode-attention oracle (CPU only): closed forms, invariances
and a library routine it must agree with."""
from __future__ import annotations

import numpy as np
import pytest

from oracle.attn import decode_attention


def _rand(seed, L, Hq=4, Hkv=2, D=16):
    r = np.random.default_rng(seed)
    return r.normal(0, 1, (Hq, D)), r.normal(0, 1, (L, Hkv, D)), r.normal(0, 1, (L, Hkv, D))


def test_equal_keys_give_the_mean_value():
    q, k, v = _rand(0, 9)
    k[:] = k[0]  # every position has the same key: uniform weights
    o = decode_attention(q, k, v)
    for h in range(4):
        np.testing.assert_allclose(o[h], v[:, h // 2].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_one_dominant_key_selects_its_value():
    q, k, v = _rand(1, 7)
    k[4] = 60.0 * q[0] / np.linalg.norm(q[0])  # score ~ 60|q| / sqrt(D): every other weight below 1e-30
    o = decode_attention(q, k, v)
    np.testing.assert_allclose(o[0], v[4, 0], rtol=1e-12, atol=1e-12)


def test_single_position_returns_its_value():
    q, k, v = _rand(2, 1)
    o = decode_attention(q, k, v)
    for h in range(4):
        np.testing.assert_allclose(o[h], v[0, h // 2], rtol=1e-14)


def test_permuting_positions_changes_nothing():
    q, k, v = _rand(3, 50)
    perm = np.random.default_rng(9).permutation(50)
    np.testing.assert_allclose(decode_attention(q, k, v), decode_attention(q, k[perm], v[perm]), rtol=1e-12,
                               atol=1e-14)


def test_query_heads_read_their_kv_head():
    # Hq = 8, Hkv = 2: heads 0-3 read KV head 0, heads 4-7 KV head 1
    q, k, v = _rand(4, 20, Hq=8, Hkv=2)
    o = decode_attention(q, k, v)
    for h in range(8):
        g = h // 4
        np.testing.assert_allclose(o[h], decode_attention(q[h:h + 1], k[:, g:g + 1], v[:, g:g + 1])[0], rtol=1e-13)


def test_agrees_with_torch_sdpa():
    torch = pytest.importorskip("torch")
    q, k, v = _rand(5, 33, Hq=16, Hkv=2, D=32)
    o = decode_attention(q, k, v, scale=0.3)
    G = 8
    qt = torch.from_numpy(q)[:, None, :]                                    # [Hq, 1, D]
    kt = torch.from_numpy(np.repeat(k.transpose(1, 0, 2), G, axis=0))       # [Hq, L, D]
    vt = torch.from_numpy(np.repeat(v.transpose(1, 0, 2), G, axis=0))
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=0.3)[:, 0, :].numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12)


def test_bf16_inputs_are_read_as_their_values():
    # q = [1, 0], keys [2, 0] and [0, 0] (0x4000 = 2), values [1, 2] and [-1, 0.5]
    q = np.array([[0x3F80, 0x0000]], np.uint16)
    k = np.array([[[0x4000, 0x0000]], [[0x0000, 0x0000]]], np.uint16)
    v = np.array([[[0x3F80, 0x4000]], [[0xBF80, 0x3F00]]], np.uint16)
    o = decode_attention(q, k, v, scale=1.0)
    w = np.exp(2.0) / (np.exp(2.0) + 1.0)
    np.testing.assert_allclose(o[0], w * np.array([1.0, 2.0]) + (1 - w) * np.array([-1.0, 0.5]), rtol=1e-14)
