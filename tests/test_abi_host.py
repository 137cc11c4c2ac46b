"""Host-only checks of the C ABI: the library builds and loads, exports every
entry point the header declares, and rejects bad arguments before anything
is enqueued.  Every call here fails validation, so no kernel is launched
(safe with or without a GPU)."""
from __future__ import annotations

import ctypes
import glob
import os
import re

import pytest

import bit_grouped_expert_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bit_grouped_expert_gb300 import build
    build.build()
    return moe.lib()


def _declared():
    names = set()
    for h in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))):
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b((?:moe|gdn|attn)_[a-z_]+)\s*\(", src))
    return sorted(names)


def test_header_entry_points_exported(lib):
    names = _declared()
    assert set(names) == set(moe.EXPORTS), names
    for n in names:
        assert hasattr(lib, n), n


def test_plan_rejects_bad_dims(lib):
    good = dict(hidden=2048, n_experts=256, top_k=8, inter=512, n_shared=1, group_size=64)
    cases = [
        (dict(hidden=2000), moe.MOE_ERR_UNSUPPORTED),
        (dict(inter=500), moe.MOE_ERR_UNSUPPORTED),
        (dict(group_size=32), moe.MOE_ERR_UNSUPPORTED),
        (dict(n_experts=2048), moe.MOE_ERR_UNSUPPORTED),
        (dict(top_k=17), moe.MOE_ERR_UNSUPPORTED),
        (dict(top_k=9, n_experts=8), moe.MOE_ERR_UNSUPPORTED),
        (dict(n_shared=2), moe.MOE_ERR_UNSUPPORTED),
        (dict(top_k=0), moe.MOE_ERR_INVALID_ARGUMENT),
    ]
    for change, want in cases:
        cfg = moe.make_config(**{**good, **change})
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_plan(cfg, 256)
        assert ei.value.status == want, change
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_plan(moe.make_config(**good), 0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARGUMENT
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_plan(moe.make_config(**good), 256, flags=0x100)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARGUMENT
    h = ctypes.c_void_p()
    assert lib.moe_plan(None, 256, 0, ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARGUMENT


def test_workspace_size_covers_buffers(lib):
    plan = moe.moe_plan(moe.make_config(), 4096)
    need = moe.moe_workspace_bytes(plan)
    T, E, k, H, I = 4096, 256, 8, 2048, 512
    # keys, top-k, perm/inv, h and y, the router's bf16 split, normalised x, and
    # the x rows gathered in block-map row order for the tensor-core gate/up GEMM
    floor = (T * E * 4 + 2 * T * k * 4 + 2 * k * T * 4 + (k + 1) * T * (I + H) * 2 + 3 * E * H * 2 + T * H * 2
             + (k + 1) * T * H * 2)
    assert floor <= need <= floor * 1.01 + (1 << 20)
    assert lib.moe_workspace_bytes(None) == 0


class _FakeTensor:
    """Stands in for a device tensor: only an address and a size."""

    def __init__(self, addr, nbytes):
        self.addr, self.n = addr, nbytes

    def data_ptr(self):
        return self.addr

    def numel(self):
        return self.n

    def element_size(self):
        return 1


def test_forward_argument_errors_enqueue_nothing(lib):
    plan = moe.moe_plan(moe.make_config(), 128)
    need = moe.moe_workspace_bytes(plan)
    ws = _FakeTensor(0x10000000, need)
    x = 0x20000000
    W = {n: 0x30000000 + i * 0x100000 for i, n in enumerate(
        ("router", "gate_q", "up_q", "gate_s", "gate_b", "up_s", "up_b", "down_q", "down_s", "down_b"))}

    def status_of(**kw):
        args = dict(x=x, residual=None, T=16, weights=W, logit_bias=None, out=0x40000000, ws=ws)
        args.update(kw)
        try:
            moe.moe_forward(plan, args["x"], args["residual"], args["T"], args["weights"], args["logit_bias"],
                            args["out"], args["ws"], stream=0)
        except moe.MoeError as e:
            return e.status
        return moe.MOE_OK

    assert status_of(T=129) == moe.MOE_ERR_TOO_MANY_TOKENS
    assert status_of(T=0) == moe.MOE_ERR_INVALID_ARGUMENT
    assert status_of(ws=_FakeTensor(0x10000000, need - 1)) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert status_of(ws=_FakeTensor(0x10000008, need)) == moe.MOE_ERR_MISALIGNED
    assert status_of(x=0x20000004) == moe.MOE_ERR_MISALIGNED
    assert status_of(out=x) == moe.MOE_ERR_INVALID_ARGUMENT
    assert status_of(x=None) == moe.MOE_ERR_INVALID_ARGUMENT
    assert status_of(weights={**W, "down_q": None}) == moe.MOE_ERR_INVALID_ARGUMENT
    assert status_of(weights={**W, "up_s": W["up_s"] + 2}) == moe.MOE_ERR_MISALIGNED
    assert status_of(logit_bias=0x50000004) == moe.MOE_ERR_MISALIGNED
    assert moe.moe_last_launch_count() == 0


def test_decode_stack_argument_errors(lib):
    plan = moe.moe_plan(moe.make_config(), 1)
    need = moe.moe_workspace_bytes(plan)
    ws = _FakeTensor(0x10000000, need)
    W = {n: 0x30000000 + i * 0x100000 for i, n in enumerate(
        ("router", "gate_q", "up_q", "gate_s", "gate_b", "up_s", "up_b", "down_q", "down_s", "down_b"))}

    def status_of(r=0x20000000, Ws=(W, W), bias=None, w=ws):
        try:
            moe.moe_decode_stack(plan, r, list(Ws), bias, w, stream=0)
        except moe.MoeError as e:
            return e.status
        return moe.MOE_OK

    assert status_of(Ws=()) == moe.MOE_ERR_INVALID_ARGUMENT
    assert status_of(r=None) == moe.MOE_ERR_INVALID_ARGUMENT
    assert status_of(r=0x20000008) == moe.MOE_ERR_MISALIGNED
    assert status_of(Ws=(W, {**W, "gate_b": None})) == moe.MOE_ERR_INVALID_ARGUMENT
    assert status_of(Ws=({**W, "down_s": W["down_s"] + 4}, W)) == moe.MOE_ERR_MISALIGNED
    assert status_of(bias=[None, 0x50000004]) == moe.MOE_ERR_MISALIGNED
    assert status_of(w=_FakeTensor(0x10000000, need - 1)) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(ValueError):
        moe.moe_decode_stack(plan, 0x20000000, [W, W], [None], ws, stream=0)
    assert moe.moe_last_launch_count() == 0


def test_route_and_view_argument_errors(lib):
    plan = moe.moe_plan(moe.make_config(), 64)
    need = moe.moe_workspace_bytes(plan)
    ws = _FakeTensor(0x10000000, need)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route(plan, 0x20000000, 65, 0x30000000, None, ws, stream=0)
    assert ei.value.status == moe.MOE_ERR_TOO_MANY_TOKENS
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route(plan, None, 8, 0x30000000, None, ws, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARGUMENT
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route_from_logits(plan, 0x20000002, 8, ws, stream=0)
    assert ei.value.status == moe.MOE_ERR_MISALIGNED
    v = moe.moe_route_view(plan, 0x10000000, 64)
    assert v.keys_d >= 0x10000000 and v.y_d + 9 * 64 * 2048 * 2 <= 0x10000000 + need
    assert v.block_rows in (32, 64, 128) and v.max_tiles >= 64 * 8 // v.block_rows
    ptrs = sorted([v.keys_d, v.topk_id_d, v.topk_w_d, v.counts_d, v.offsets_d, v.perm_d, v.inv_d, v.blockmap_d,
                   v.n_tiles_d, v.h_d, v.y_d])
    assert all(p % 256 == 0 for p in ptrs) and len(set(ptrs)) == len(ptrs)
    with pytest.raises(moe.MoeError):
        moe.moe_route_view(plan, 0x10000000, 65)


def test_other_entry_point_errors(lib):
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_rmsnorm(0x1000, 4, 2047, 1e-6, 0x2000, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARGUMENT
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_rmsnorm(0x1000, 4, 2048, 1e-6, 0x1000, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARGUMENT
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_dequant(0x1000, 0x2000, 0x3000, 4, 96, 64, 0x4000, stream=0)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_dequant(0x1004, 0x2000, 0x3000, 4, 128, 64, 0x4000, stream=0)
    assert ei.value.status == moe.MOE_ERR_MISALIGNED
    assert moe.status_str(moe.MOE_ERR_NONFINITE) == "non-finite router key"


def test_gdn_scan_host_checks(lib):
    # fake, aligned device addresses: every case below is refused on the host
    q, k, v, al, be, st, o = (0x10000000 + i * 0x1000000 for i in range(7))
    ok = dict(T=64, Hk=2, Hv=4, dk=128, dv=128)

    def call(**kw):
        a = {**dict(q=q, k=k, v=v, alpha=al, beta=be, state=st, o=o), **ok, **kw}
        return lib.gdn_scan(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["state"], a["o"], a["T"], a["Hk"],
                            a["Hv"], a["dk"], a["dv"], 0)

    assert call(T=0, q=None, k=None) == moe.MOE_OK  # nothing to do, nothing enqueued
    assert call(T=-1) == moe.MOE_ERR_INVALID_ARGUMENT
    assert call(Hk=0) == moe.MOE_ERR_INVALID_ARGUMENT
    assert call(Hv=3) == moe.MOE_ERR_INVALID_ARGUMENT  # not a multiple of Hk
    assert call(dk=64) == moe.MOE_ERR_UNSUPPORTED
    assert call(dv=48) == moe.MOE_ERR_UNSUPPORTED
    assert call(beta=None) == moe.MOE_ERR_INVALID_ARGUMENT
    assert call(v=v + 8) == moe.MOE_ERR_MISALIGNED
    assert call(alpha=al + 4) == moe.MOE_ERR_MISALIGNED
    assert call(o=q + 4096) == moe.MOE_ERR_INVALID_ARGUMENT  # o overlaps q
    assert call(o=st) == moe.MOE_ERR_INVALID_ARGUMENT  # o overlaps the state


def test_attn_decode_host_checks(lib):
    import ctypes
    q, k, v, ws, o = (0x10000000 + i * 0x1000000 for i in range(5))
    need = lib.attn_decode_workspace_bytes(1000, 16, 256)
    # up to one block per 64 positions (16 here): partial outputs 16*16*256 fp32, then the max and sum rows
    assert need == 256 + 16 * 16 * 256 * 4 + 1024 + 16 * 16 * 4  # status word, then the partials
    assert lib.attn_decode_workspace_bytes(1 << 20, 16, 256) == 256 + 512 * 16 * 256 * 4 + 512 * 16 * 4 * 2
    assert lib.attn_decode_workspace_bytes(0, 16, 256) == 0
    assert lib.attn_decode_workspace_bytes(10, 16, 128) == 0

    def call(L=1000, Hq=16, Hkv=2, D=256, scale=0.0, ws_bytes=need, **kw):
        a = {**dict(q=q, k=k, v=v, ws=ws, o=o), **kw}
        return lib.attn_decode(a["q"], a["k"], a["v"], L, Hq, Hkv, D, ctypes.c_float(scale), a["ws"], ws_bytes,
                               a["o"], 0)

    assert call(L=0) == moe.MOE_ERR_INVALID_ARGUMENT
    assert call(k=None) == moe.MOE_ERR_INVALID_ARGUMENT
    assert call(scale=-1.0) == moe.MOE_ERR_INVALID_ARGUMENT
    assert call(scale=float("nan")) == moe.MOE_ERR_INVALID_ARGUMENT
    assert call(D=128) == moe.MOE_ERR_UNSUPPORTED
    assert call(Hq=8) == moe.MOE_ERR_UNSUPPORTED  # 4 query heads per KV head
    assert call(v=v + 2) == moe.MOE_ERR_MISALIGNED
    assert call(ws_bytes=need - 1) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
