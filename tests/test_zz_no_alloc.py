"""moe_decode_static, the allocation-free single-token entry point, against
moe_forward's decode path on the same inputs.

Both run the same decode kernel on the same keys, so their outputs must agree
bit for bit; one call of each case is also checked against the CPU oracle.

Named to be collected last: the static scratch array is shared by every call
in the process, so this file also checks that it gives the same answers after
the rest of the suite has run (and when run alone, in a fresh process), and
across calls whose layer dimensions change (the array's layout changes with
them)."""
from __future__ import annotations

import numpy as np
import pytest

import bit_grouped_expert_gb300 as moe
import oracle as orc
import synthetic as syn
from tests.tolerances import assert_outputs_close


def test_rejects_layers_beyond_the_static_scratch():
    # k=16 slots of I=8192: the h vectors alone need 17 * 8192 * 2 bytes
    cfg = moe.make_config(hidden=2048, n_experts=256, top_k=16, inter=8192, n_shared=1, group_size=64)
    fake = {n: 0x30000000 + i * 0x100000 for i, n in enumerate(
        ("router", "gate_q", "up_q", "gate_s", "gate_b", "up_s", "up_b", "down_q", "down_s", "down_b"))}
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_decode_static(cfg, 0x20000000, None, fake, None, 0x40000000, stream=0)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(moe.MoeError) as ei:  # only PRENORM is a valid flag
        moe.moe_decode_static(moe.make_config(), 0x20000000, None, fake, None, 0x40000000,
                              flags=moe.MOE_FLAG_TRACE, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARGUMENT


@pytest.fixture(scope="module")
def gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from bit_grouped_expert_gb300 import build
    build.build()
    syn.build()
    orc.build()
    return torch


TINY = dict(H=256, E=16, k=4, I=256)
REAL = dict(H=2048, E=256, k=8, I=512)


def _weights(d, seed, gate=False):
    W = syn.experts(seed, d["E"] + 1, d["H"], d["I"])
    W["router"] = syn.router(seed, d["E"], d["H"])
    if gate:  # the shared expert scaled by its sigmoid gate
        W["shared_gate"] = syn.shared_gate(seed, d["H"])
    return W


def _one_call(torch, d, W, Wd, bias, seed, prenorm, status, check_oracle):
    """moe_decode_static and moe_forward's decode path on the same token:
    bitwise equal outputs, clean status; optionally against the oracle."""
    from tests.gpu_util import Layer, dev, host_u16
    cfg = moe.make_config(d["H"], d["E"], d["k"], d["I"], 1, 64)
    flags = moe.MOE_FLAG_PRENORM if prenorm else 0
    L = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=1, flags=flags)
    x = syn.activations(seed, 1, d["H"])
    res = syn.activations(seed, 1, d["H"], tensor=syn.T_RESID)
    if prenorm:  # in place over the residual stream
        r_ref, r_new = dev(res), dev(res)
        moe.moe_forward(L.plan, r_ref, None, 1, Wd, bias, r_ref, L.ws)
        moe.moe_decode_static(cfg, r_new, None, Wd, bias, r_new, status=status, flags=flags)
        want, got = r_ref, r_new
    else:
        xd, rd = dev(x), dev(res)
        want, got = torch.empty_like(xd), torch.full_like(xd, 0x7FC0)
        moe.moe_forward(L.plan, xd, rd, 1, Wd, bias, want, L.ws)
        moe.moe_decode_static(cfg, xd, rd, Wd, bias, got, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == moe.MOE_OK
    assert L.status() == 0
    np.testing.assert_array_equal(host_u16(got), host_u16(want))
    if check_oracle:
        keys = L.routing(1)["keys"]
        xin = orc.rmsnorm(res, 1e-6) if prenorm else x
        hb = None if bias is None else bias.cpu().numpy()
        ref = orc.moe_layer(orc.Dims(**d, n_shared=1), xin, W, res=res, bias=hb, keys=keys, intermediates=True)
        assert_outputs_close(host_u16(got), ref, "static decode", k=d["k"])


@pytest.mark.gpu
@pytest.mark.parametrize("prenorm,gate", [(False, False), (True, False), (True, True)])
def test_static_decode_matches_forward_on_consecutive_calls(gpu, prenorm, gate):
    torch = gpu
    from tests.gpu_util import dev, dev_weights
    W = _weights(REAL, 0, gate)
    Wd = dev_weights(W)
    bias = dev(syn.zipf_bias(0, 256))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda:0")
    for call, seed in enumerate((301, 302)):  # two calls in a row, different tokens
        _one_call(torch, REAL, W, Wd, bias, seed, prenorm, status, check_oracle=call == 0)


@pytest.mark.gpu
def test_static_decode_when_the_dimensions_change(gpu):
    # tiny, real, tiny: each change of dimensions moves the tagged words of
    # the static array to another layout, which the entry point must clear
    torch = gpu
    from tests.gpu_util import dev_weights
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda:0")
    sets = {}
    for name, d, seed in (("tiny", TINY, 5), ("real", REAL, 6)):
        W = _weights(d, seed)
        sets[name] = (d, W, dev_weights(W))
    for i, name in enumerate(("tiny", "real", "tiny", "tiny")):
        d, W, Wd = sets[name]
        _one_call(torch, d, W, Wd, None, 320 + i, prenorm=i % 2 == 1, status=status, check_oracle=i < 2)
