"""moe_decode_static, the allocation-free single-token entry point, against
moe_forward's decode path on the same inputs.

Named to be collected last: the static scratch array is shared by every call
in the process, so this file also checks that it gives the same answers after
the rest of the suite has run (and when run alone, in a fresh process)."""
from __future__ import annotations

import numpy as np
import pytest

import bit_grouped_expert_gb300 as moe
import synthetic as syn
from tests.tolerances import assert_outputs_close, bf16_value


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
    return torch


@pytest.mark.gpu
@pytest.mark.parametrize("prenorm,gate", [(False, False), (True, False), (True, True)])
def test_static_decode_matches_forward_on_consecutive_calls(gpu, prenorm, gate):
    torch = gpu
    from tests.gpu_util import Layer, dev, dev_weights, host_u16

    W = syn.experts(0, 257, 2048, 512)
    W["router"] = syn.router(0, 256, 2048)
    if gate:  # the shared expert scaled by its sigmoid gate
        W["shared_gate"] = syn.shared_gate(0, 2048)
    Wd = dev_weights(W)
    bias = dev(syn.zipf_bias(0, 256))
    cfg = moe.make_config()
    flags = moe.MOE_FLAG_PRENORM if prenorm else 0
    L = Layer(max_tokens=1, flags=flags)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda:0")
    for call, seed in enumerate((301, 302)):  # two calls in a row, different tokens
        x = syn.activations(seed, 1, 2048)
        res = syn.activations(seed, 1, 2048, tensor=syn.T_RESID)
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
        assert int(status.item()) == moe.MOE_OK, f"call {call}"
        assert L.status() == 0
        assert_outputs_close(host_u16(got), bf16_value(host_u16(want)), f"static decode call {call}")
