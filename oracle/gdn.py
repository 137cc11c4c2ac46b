"""CPU oracle for the Gated DeltaNet scan -- TEST INFRASTRUCTURE ONLY (same
import rule as the rest of ``oracle/``: tests, ``smoke()`` and ``bench.py``'s
CPU legs only; the product library never imports it).

What it computes.  The pages ("Perplexity open-sources Lily", "three workload
shapes" and "Prefill") name the model's 30 Gated DeltaNet layers, call their
work a fixed-size recurrence, and credit a scan that keeps the recurrent state
in GPU registers with +5.6 % at 2K tokens; they do not print the recurrence.
This is the gated delta rule as its authors publish it (Yang, Kautz and
Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with Delta Rule", 2024),
per value head h and token t, with the state S a [dk, dv] matrix that maps
keys to values:

    S_t = alpha_t * (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
    o_t = S_t^T q_t

alpha_t in (0, 1] is the decay (the gate), beta_t in (0, 1) the write
strength.  Value head h reads query/key head h // (Hv / Hk) (the model shares
each key head between value heads).  Any normalisation or scaling of q and k
and the computation of alpha and beta from the layer's projections happen
before the scan and are not part of it.

The loop below takes the steps in that order, in fp64: decay the state, read
what it holds for k_t, write beta_t times the difference, read the output.
Inputs: bf16 q, k, v (uint16 bit patterns), fp32 alpha, beta and initial
state.  Output: o in fp64 (the GPU rounds it to bf16 once) and the final state.

Parity status: pinned by ``tests/test_gdn_oracle.py`` (single-step closed
form, beta = 0, exact retrieval and overwrite with orthonormal keys, and the
product of the per-token transition matrices).
"""
from __future__ import annotations

import numpy as np


def _bf16(a: np.ndarray) -> np.ndarray:
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gdn_scan(q: np.ndarray, k: np.ndarray, v: np.ndarray, alpha: np.ndarray, beta: np.ndarray,
             state: np.ndarray | None = None, t_end: int | None = None):
    """o [T, Hv, dv] fp64 and the final state [Hv, dk, dv] fp64 of the scan
    over tokens 0 .. t_end-1 (all by default).  q, k [T, Hk, dk] and v
    [T, Hv, dv] are bf16 bit patterns (or float arrays, taken as they are);
    alpha, beta [T, Hv]; state [Hv, dk, dv] (zeros when None)."""
    qf = _bf16(q) if np.asarray(q).dtype == np.uint16 else np.asarray(q, np.float64)
    kf = _bf16(k) if np.asarray(k).dtype == np.uint16 else np.asarray(k, np.float64)
    vf = _bf16(v) if np.asarray(v).dtype == np.uint16 else np.asarray(v, np.float64)
    T, Hk, dk = qf.shape
    Hv, dv = vf.shape[1], vf.shape[2]
    assert kf.shape == (T, Hk, dk) and vf.shape[0] == T and Hv % Hk == 0
    a = np.asarray(alpha, np.float64)
    b = np.asarray(beta, np.float64)
    S = np.zeros((Hv, dk, dv)) if state is None else np.array(state, np.float64)
    group = Hv // Hk
    head_k = np.arange(Hv) // group  # value head h reads key head h // group
    n = T if t_end is None else t_end
    o = np.zeros((n, Hv, dv))
    for t in range(n):
        kt = kf[t, head_k]  # [Hv, dk]
        qt = qf[t, head_k]
        S = a[t][:, None, None] * S                         # decay
        u = np.einsum("hij,hi->hj", S, kt)                  # what the state holds for k_t
        S = S + b[t][:, None, None] * kt[:, :, None] * (vf[t] - u)[:, None, :]  # delta write
        o[t] = np.einsum("hij,hi->hj", S, qt)               # read with q_t
    return o, S
