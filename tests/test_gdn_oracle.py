"""Pins for the Gated DeltaNet scan oracle (CPU only).

Each test checks oracle.gdn.gdn_scan against something other than its own
loop: closed forms of special cases, the exact-retrieval property of the delta
rule with orthonormal keys, and the explicit product of the per-token
transition matrices (a different way to reach the same state).
"""
from __future__ import annotations

import numpy as np
import pytest

from oracle.gdn import gdn_scan


def _rand(seed, T, Hk, Hv, dk, dv, state=True):
    r = np.random.default_rng(seed)
    q = r.normal(0, 1 / np.sqrt(dk), (T, Hk, dk))
    k = r.normal(0, 1 / np.sqrt(dk), (T, Hk, dk))
    v = r.normal(0, 1, (T, Hv, dv))
    a = r.uniform(0.7, 1.0, (T, Hv))
    b = r.uniform(0.1, 0.9, (T, Hv))
    S0 = r.normal(0, 0.3, (Hv, dk, dv)) if state else None
    return q, k, v, a, b, S0


def test_single_step_from_empty_state():
    # S_1 = beta k v^T, so o_1 = beta (q . k) v
    q, k, v, a, b, _ = _rand(0, 1, 1, 1, 6, 5, state=False)
    o, S = gdn_scan(q, k, v, a, b)
    np.testing.assert_allclose(S[0], b[0, 0] * np.outer(k[0, 0], v[0, 0]), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(o[0, 0], b[0, 0] * (q[0, 0] @ k[0, 0]) * v[0, 0], rtol=1e-12, atol=1e-15)


def test_zero_write_strength_only_decays():
    # beta = 0: S_t = (alpha_1 ... alpha_t) S_0 and o_t = S_t^T q_t
    q, k, v, a, _, S0 = _rand(1, 7, 2, 4, 5, 3)
    o, S = gdn_scan(q, k, v, a, np.zeros_like(a), S0)
    decay = np.cumprod(a, axis=0)  # [T, Hv]
    for t in range(7):
        for h in range(4):
            want = decay[t, h] * S0[h].T @ q[t, h // 2]
            np.testing.assert_allclose(o[t, h], want, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S, decay[-1][:, None, None] * S0, rtol=1e-12)


def test_orthonormal_keys_retrieve_and_overwrite():
    # alpha = 1, beta = 1, keys e_0 .. e_{n-1}: each write stores v_i under e_i
    # exactly; a second write to e_0 replaces the first (a linear-attention
    # sum would give v + v'), and with beta = 1/2 it lands half way.
    dk, dv, n = 6, 4, 5
    r = np.random.default_rng(2)
    vals = r.normal(0, 1, (n + 1, dv))
    keys = np.zeros((n + 1, 1, dk))
    for i in range(n):
        keys[i, 0, i] = 1.0
    keys[n, 0, 0] = 1.0  # overwrite e_0
    v = vals[:, None, :]
    ones = np.ones((n + 1, 1))
    q = keys.copy()
    o, S = gdn_scan(q, keys, v, ones, ones)
    for i in range(n):
        np.testing.assert_allclose(o[i, 0], vals[i], atol=1e-14)  # reading the key just written
    np.testing.assert_allclose(S[0].T @ np.eye(dk)[0], vals[n], atol=1e-14)
    for i in range(1, n):
        np.testing.assert_allclose(S[0].T @ np.eye(dk)[i], vals[i], atol=1e-14)
    half = ones.copy()
    half[n] = 0.5
    _, S = gdn_scan(q, keys, v, ones, half)
    np.testing.assert_allclose(S[0].T @ np.eye(dk)[0], 0.5 * (vals[0] + vals[n]), atol=1e-14)


def _transition_product(q, k, v, a, b, S0, h, group):
    """S_t = A_t S_{t-1} + beta_t k_t v_t^T with A_t = alpha_t (I - beta_t k_t k_t^T),
    unrolled: S_t = (A_t ... A_1) S_0 + sum_s (A_t ... A_{s+1}) beta_s k_s v_s^T."""
    T, _, dk = k.shape
    A = [a[t, h] * (np.eye(dk) - b[t, h] * np.outer(k[t, h // group], k[t, h // group])) for t in range(T)]
    outs, states = [], []
    for t in range(T):
        P = np.eye(dk)
        for s in range(t, -1, -1):
            P = P @ A[s]
        St = P @ S0[h]
        for s in range(t + 1):
            Ps = np.eye(dk)
            for r_ in range(t, s, -1):
                Ps = Ps @ A[r_]
            St = St + Ps @ (b[s, h] * np.outer(k[s, h // group], v[s, h]))
        states.append(St)
        outs.append(St.T @ q[t, h // group])
    return np.array(outs), states[-1]


@pytest.mark.parametrize("seed", [3, 4])
def test_matches_product_of_transition_matrices(seed):
    T, Hk, Hv, dk, dv = 6, 2, 4, 5, 3
    q, k, v, a, b, S0 = _rand(seed, T, Hk, Hv, dk, dv)
    o, S = gdn_scan(q, k, v, a, b, S0)
    for h in range(Hv):
        ob, Sb = _transition_product(q, k, v, a, b, S0, h, Hv // Hk)
        np.testing.assert_allclose(o[:, h], ob, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(S[h], Sb, rtol=1e-11, atol=1e-13)


def test_value_heads_read_their_key_head():
    # Hv = 3 Hk: value head h runs the single-head scan of key head h // 3
    T, Hk, Hv, dk, dv = 5, 2, 6, 4, 3
    q, k, v, a, b, S0 = _rand(5, T, Hk, Hv, dk, dv)
    o, S = gdn_scan(q, k, v, a, b, S0)
    for h in range(Hv):
        oh, Sh = gdn_scan(q[:, h // 3:h // 3 + 1], k[:, h // 3:h // 3 + 1], v[:, h:h + 1], a[:, h:h + 1],
                          b[:, h:h + 1], S0[h:h + 1])
        np.testing.assert_allclose(o[:, h], oh[:, 0], rtol=1e-13)
        np.testing.assert_allclose(S[h], Sh[0], rtol=1e-13)


def test_prefix_of_the_scan_is_the_scan_of_the_prefix():
    q, k, v, a, b, S0 = _rand(6, 9, 1, 2, 4, 4)
    o, _ = gdn_scan(q, k, v, a, b, S0)
    o5, S5 = gdn_scan(q, k, v, a, b, S0, t_end=5)
    np.testing.assert_array_equal(o[:5], o5)
    o_rest, _ = gdn_scan(q[5:], k[5:], v[5:], a[5:], b[5:], S5)
    np.testing.assert_allclose(o[5:], o_rest, rtol=1e-13)


def test_transition_product_rejects_a_planted_mistake():
    # the same loop with the decay applied after the write instead of before
    # it disagrees with the transition-matrix product: the pin can tell
    T, dk, dv = 4, 4, 3
    q, k, v, a, b, S0 = _rand(7, T, 1, 1, dk, dv)
    S = S0[0].copy()
    wrong = []
    for t in range(T):
        u = S.T @ k[t, 0]
        S = a[t, 0] * (S + b[t, 0] * np.outer(k[t, 0], v[t, 0] - u))
        wrong.append(S.T @ q[t, 0])
    ob, _ = _transition_product(q, k, v, a, b, S0, 0, 1)
    assert not np.allclose(np.array(wrong), ob, rtol=1e-6)


def test_bf16_inputs_are_read_as_their_values():
    # bit patterns 0x3F80 = 1, 0x4000 = 2, 0xBF00 = -0.5, 0x3E80 = 0.25
    q = np.array([[[0x3F80, 0x0000]]], np.uint16)
    k = np.array([[[0x4000, 0xBF00]]], np.uint16)
    v = np.array([[[0x3E80, 0x3F80]]], np.uint16)
    o, S = gdn_scan(q, k, v, np.ones((1, 1)), np.full((1, 1), 0.5))
    # S = 0.5 * [2, -0.5]^T [0.25, 1];  o = S^T [1, 0] = 0.5 * 2 * [0.25, 1]
    np.testing.assert_array_equal(S[0], 0.5 * np.outer([2.0, -0.5], [0.25, 1.0]))
    np.testing.assert_array_equal(o[0, 0], [0.25, 1.0])
