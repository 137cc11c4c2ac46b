"""GPU parity of the decode attention (attn_decode through the C ABI) against
the fp64 oracle on the same seeded inputs.

Tolerance, from the arithmetic: scores and sums are fp32; the softmax weights
are rounded to bf16 (2^-9 relative) before the product with V, and o is
rounded once to bf16.  So: rel-L2(o) <= 5e-3 and per element |o - ref| may
exceed half a bf16 ulp of ref by at most 2^-8 * sum_l p_l |v_l| (the weighted
mean of |v| in that dimension, from the oracle's weights) + 1e-3 * rms(ref).
"""
from __future__ import annotations

import numpy as np
import pytest

import synthetic as syn
from oracle.attn import decode_attention
from tests.tolerances import bf16_half_ulp, bf16_value

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bit_grouped_expert_gb300 as moe  # noqa: E402
from tests.gpu_util import dev, host_u16  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from bit_grouped_expert_gb300 import build
    build.build()
    syn.build()


def _run(d, L, Hq=16, Hkv=2, scale=0.0):
    ws = torch.zeros(moe.attn_decode_workspace_bytes(L, Hq, 256), dtype=torch.uint8, device="cuda:0")
    o = torch.full((Hq, 256), 0x7FC0, dtype=torch.int16, device="cuda:0")
    moe.attn_decode(dev(d["q"]), dev(d["k"]), dev(d["v"]), L, Hq, Hkv, 256, ws, o, scale=scale)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0  # the status word: no wait gave up
    return host_u16(o)


def _weighted_abs_v(d, Hq, Hkv, scale):
    """sum_l p_l |v_l| per (head, dim), with the oracle's fp64 weights."""
    q = bf16_value(d["q"]).reshape(d["q"].shape)
    k = bf16_value(d["k"]).reshape(d["k"].shape)
    v = bf16_value(d["v"]).reshape(d["v"].shape)
    out = np.empty((Hq, 256))
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = scale * (k[:, g] @ q[h])
        p = np.exp(s - s.max())
        p /= p.sum()
        out[h] = p @ np.abs(v[:, g])
    return out


def _check(o_bits, d, Hq=16, Hkv=2, scale=None, what=""):
    sc = 1.0 / 16.0 if scale is None else scale
    ref = decode_attention(d["q"], d["k"], d["v"], scale=sc)
    got = bf16_value(o_bits).reshape(ref.shape)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    allow = bf16_half_ulp(ref) + 2.0 ** -8 * _weighted_abs_v(d, Hq, Hkv, sc) + 1e-3 * rms
    worst = float((np.abs(got - ref) - allow).max())
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert worst <= 0, f"{what}: an element exceeds its allowance by {worst:.3g}"
    assert rel <= 5e-3, f"{what}: rel-L2 {rel:.3g}"


@pytest.mark.parametrize("L", [1, 7, 16, 255, 256, 257, 1000, 4099])
def test_attention_lengths(L):
    d = syn.attn_inputs(20 + L, L)
    _check(_run(d, L), d, what=f"L={L}")


@pytest.mark.parametrize("L", [32768, 131072])
def test_attention_long_contexts(L):
    d = syn.attn_inputs(3, L)
    _check(_run(d, L), d, what=f"L={L}")


def test_attention_explicit_scale_and_peaked_scores():
    # a larger scale makes the weights peaked: the running maximum must track it
    L = 3000
    d = syn.attn_inputs(5, L)
    _check(_run(d, L, scale=0.5), d, scale=0.5, what="scale 0.5")


def test_attention_more_kv_heads():
    L = 600
    d = syn.attn_inputs(6, L, Hq=32, Hkv=4)
    _check(_run(d, L, Hq=32, Hkv=4), d, Hq=32, Hkv=4, what="Hq=32 Hkv=4")


def test_attention_is_deterministic():
    L = 5000
    d = syn.attn_inputs(8, L)
    np.testing.assert_array_equal(_run(d, L), _run(d, L))
