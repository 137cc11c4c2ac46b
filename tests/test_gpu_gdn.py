"""GPU parity of the Gated DeltaNet scan (gdn_scan through the C ABI) against
the fp64 oracle on the same seeded inputs.

Tolerance, from the arithmetic: the GPU keeps the state and every sum in fp32
and rounds o once to bf16.  With |k| near 1, alpha <= 1 and beta < 1 each
token's update is a contraction, so fp32 rounding stays near 1e-6 relative
and does not grow with T.  The one bf16 rounding of o moves each element by
at most half an ulp, 2^-9 of its size, so rel-L2 from rounding alone reaches
~2e-3 on short outputs.  So: per element |o - ref| may exceed half a bf16 ulp
of ref by at most 1e-3 * rms(ref), rel-L2(o) <= 3e-3, and the final fp32
state within rel-L2 1e-5 of the oracle's.
"""
from __future__ import annotations

import numpy as np
import pytest

import synthetic as syn
from oracle.gdn import gdn_scan as oracle_scan
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


def _run(d, T, Hk, Hv, dv, state=None):
    st = dev(d["state"] if state is None else state)
    o = torch.full((T, Hv, dv), 0x7FC0, dtype=torch.int16, device="cuda:0")
    moe.gdn_scan(dev(d["q"]), dev(d["k"]), dev(d["v"]), dev(d["alpha"]), dev(d["beta"]), st, o, T, Hk, Hv, 128, dv)
    torch.cuda.synchronize()
    return host_u16(o), st.cpu().numpy()


def _check(o_bits, S, d, T, what):
    ref, S_ref = oracle_scan(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["state"])
    got = bf16_value(o_bits).reshape(ref.shape)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    beyond = np.abs(got - ref) - bf16_half_ulp(ref)
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert beyond.max() <= 1e-3 * rms, f"{what}: max beyond half-ulp {beyond.max():.3g}, rms {rms:.3g}"
    assert rel <= 3e-3, f"{what}: rel-L2 {rel:.3g}"
    srel = float(np.linalg.norm(S - S_ref) / max(np.linalg.norm(S_ref), 1e-30))
    assert srel <= 1e-5, f"{what}: state rel-L2 {srel:.3g}"


@pytest.mark.parametrize("T,Hk,Hv,dv,state_std", [(1, 1, 1, 32, 0.0), (3, 1, 2, 32, 0.1), (37, 1, 2, 64, 0.0),
                                                  (200, 2, 4, 128, 0.1), (129, 4, 4, 96, 0.05)])
def test_scan_small(T, Hk, Hv, dv, state_std):
    d = syn.gdn_inputs(10 + T, T, Hk, Hv, 128, dv, state_std=state_std)
    o, S = _run(d, T, Hk, Hv, dv)
    _check(o, S, d, T, f"T={T} Hk={Hk} Hv={Hv} dv={dv}")


def test_scan_full_size_2k():
    # one sequence of 2048 tokens, 16 key heads, 32 value heads, dk = dv = 128
    T, Hk, Hv = 2048, 16, 32
    d = syn.gdn_inputs(7, T, Hk, Hv)
    o, S = _run(d, T, Hk, Hv, 128)
    _check(o, S, d, T, "2K")


def test_scan_continues_from_its_state_bit_for_bit():
    # two calls (60 then 40 tokens) carrying the state equal one call of 100
    T, Hk, Hv, dv = 100, 2, 4, 128
    d = syn.gdn_inputs(3, T, Hk, Hv, state_std=0.1)
    o_all, S_all = _run(d, T, Hk, Hv, dv)
    first = {n: (a[:60] if n != "state" else a) for n, a in d.items()}
    o1, S1 = _run(first, 60, Hk, Hv, dv)
    second = {n: (a[60:] if n != "state" else a) for n, a in d.items()}
    o2, S2 = _run(second, 40, Hk, Hv, dv, state=S1)
    np.testing.assert_array_equal(np.concatenate([o1, o2]), o_all)
    np.testing.assert_array_equal(S2, S_all)


def test_scan_is_deterministic():
    T, Hk, Hv = 300, 4, 8
    d = syn.gdn_inputs(4, T, Hk, Hv, state_std=0.1)
    a, Sa = _run(d, T, Hk, Hv, 128)
    b, Sb = _run(d, T, Hk, Hv, 128)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(Sa, Sb)


def test_scan_zero_tokens_leaves_state():
    d = syn.gdn_inputs(5, 0, 1, 1, state_std=0.1)
    st = dev(d["state"])
    moe.gdn_scan(None, None, None, None, None, st, None, 0, 1, 1, 128, 128)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(st.cpu().numpy(), d["state"])
