"""Device-side failure reporting, made to happen from the host with no GPU
fault: a bounded wait that runs out (MOE_FLAG_TEST_WITHHOLD: the decode
kernel's CTA for expert 0 never publishes that router key and every wait is
limited to 1 ms), and the debug bounds checks (MOE_FLAG_DEBUG_CHECKS) reached
through host-made expert ids.  After each, the workspace is re-initialised and
the next call must be correct."""
from __future__ import annotations

import time

import numpy as np
import pytest

import oracle as orc
import synthetic as syn
from tests.tolerances import assert_outputs_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bit_grouped_expert_gb300 as moe  # noqa: E402
from tests.gpu_util import Layer, dev, dev_weights, host_u16  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from bit_grouped_expert_gb300 import build
    build.build()
    orc.build()
    syn.build()


@pytest.fixture(scope="module")
def real():
    W = syn.experts(0, 257, 2048, 512)
    W["router"] = syn.router(0, 256, 2048)
    return W, dev_weights(W)


def _decode_ok(L, W, Wd, seed):
    """One correct decode call on L's workspace, checked against the oracle."""
    x = syn.activations(seed, 1, 2048)
    xd = dev(x)
    out = torch.empty_like(xd)
    moe.moe_forward(L.plan, xd, None, 1, Wd, None, out, L.ws)
    torch.cuda.synchronize()
    assert L.status() == 0
    ref = orc.moe_layer(orc.Dims(), x, W, keys=L.routing(1)["keys"], intermediates=True)
    assert_outputs_close(host_u16(out), ref, "decode after a timed-out call")


def test_decode_wait_runs_out_and_the_workspace_recovers(real):
    W, Wd = real
    bad = Layer(max_tokens=1, flags=moe.MOE_FLAG_TEST_WITHHOLD)
    x = dev(syn.activations(400, 1, 2048))
    out = torch.full_like(x, 0x7FC0)
    t0 = time.perf_counter()
    moe.moe_forward(bad.plan, x, None, 1, Wd, None, out, bad.ws)
    torch.cuda.synchronize()  # the kernel returned: every CTA gave up and drained its copies
    dt = time.perf_counter() - t0
    assert bad.status() == moe.MOE_ERR_DEVICE_TIMEOUT
    assert dt < 0.5, dt  # 1 ms waits, not the default second
    assert (host_u16(out) == 0x7FC0).all()  # nothing was combined
    # a three-layer stack on the same plan stops at its first layer the same way
    r = dev(syn.activations(401, 1, 2048))
    moe.moe_decode_stack(bad.plan, r, [Wd, Wd, Wd], None, bad.ws)
    torch.cuda.synchronize()
    assert bad.status() == moe.MOE_ERR_DEVICE_TIMEOUT
    # the same workspace, re-initialised, serves a plan without the test flag
    good = Layer(max_tokens=1)
    good.ws = bad.ws
    moe.moe_workspace_init(good.plan, good.ws)
    _decode_ok(good, W, Wd, 402)
    _decode_ok(good, W, Wd, 403)


def _ids_inputs(T, E, k, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    return ids, w / w.sum(axis=1, keepdims=True)


@pytest.mark.parametrize("E,k,T", [(16, 4, 300), (40, 3, 1500)])
def test_route_from_ids_matches_the_oracle_maps(E, k, T):
    # (40, 3, 1500): 4500 pairs, three blocks of the scatter kernel
    L = Layer(H=256, E=E, k=k, I=256, max_tokens=T)
    ids, w = _ids_inputs(T, E, k, 1)
    moe.moe_route_from_ids(L.plan, dev(ids), dev(w), T, L.ws)
    torch.cuda.synchronize()
    assert L.status() == 0
    r = L.routing(T)
    np.testing.assert_array_equal(r["ids"], ids)
    np.testing.assert_array_equal(r["w"], w)
    m = orc.route_maps(ids, E, n_shared=1, BN=r["block_rows"])
    for n in ("counts", "offsets", "perm", "inv", "blockmap"):
        np.testing.assert_array_equal(r[n], m[n], err_msg=n)


def test_debug_checks_reach_the_bounds_status():
    E, k, T = 16, 4, 64
    ids, w = _ids_inputs(T, E, k, 2)
    dup = ids.copy()
    dup[5, 2] = dup[5, 0]  # token 5 names one expert twice
    oob = ids.copy()
    oob[9, 1] = E  # an id past the last expert
    dbg = Layer(H=256, E=E, k=k, I=256, max_tokens=T, flags=moe.MOE_FLAG_DEBUG_CHECKS)
    plain = Layer(H=256, E=E, k=k, I=256, max_tokens=T)
    # a repeated expert: the histogram kernel's debug check compares each id
    # with the token's earlier ones
    moe.moe_route_from_ids(dbg.plan, dev(dup), dev(w), T, dbg.ws)
    assert dbg.status() == moe.MOE_ERR_DEVICE_BOUNDS
    moe.moe_route_from_ids(plain.plan, dev(dup), dev(w), T, plain.ws)
    assert plain.status() == 0  # not looked for without the flag
    # an out-of-range id is reported with or without the flag
    for L in (dbg, plain):
        moe.moe_route_from_ids(L.plan, dev(oob), dev(w), T, L.ws)
        assert L.status() == moe.MOE_ERR_DEVICE_BOUNDS
    # valid ids after the errors: clean status, maps as the oracle's
    moe.moe_workspace_init(dbg.plan, dbg.ws)
    moe.moe_route_from_ids(dbg.plan, dev(ids), dev(w), T, dbg.ws)
    assert dbg.status() == 0
    r = dbg.routing(T)
    m = orc.route_maps(ids, E, n_shared=1, BN=r["block_rows"])
    np.testing.assert_array_equal(r["perm"], m["perm"])
