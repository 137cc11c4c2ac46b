"""GPU parity for packed codes in the paired order (moe_pair_codes,
moe_weights.code_order = MOE_CODES_PAIRED).

The paired order is a permutation of the nibbles inside each packed word; the
weights it stands for are the pages' weights.  So every path is held to the
same oracle, on the pages' packing of the same seeded weights: dequantisation
bit for bit, routing bit for bit given the GPU's keys, outputs within the
layer's tolerance (tests/tolerances.py).  The CUDA-core grouped path sums the
same products in the same order for both packings, so its outputs must also
agree bit for bit; the tensor-core paths feed the products to the MMAs in a
different order within each 16-value step, so they are compared with the
oracle only."""
from __future__ import annotations

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

TINY = dict(H=256, E=16, k=4, I=256)
PATHS = {"tc": 0, "simt": moe.MOE_FLAG_SIMT_EXPERTS, "tc64": moe.MOE_FLAG_TILE_ROWS_64}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from bit_grouped_expert_gb300 import build
    build.build()
    orc.build()
    syn.build()


def _paired_host(words: np.ndarray) -> np.ndarray:
    """The paired order as the header states it: codes 2m and 2m+1 of a word
    (at bits 8m and 8m+4 of the pages' packing) move to bits 4m and 4m+16."""
    w = words.astype(np.uint64)
    out = np.zeros_like(w)
    for m in range(4):
        out |= ((w >> np.uint64(8 * m)) & np.uint64(0xF)) << np.uint64(4 * m)
        out |= ((w >> np.uint64(8 * m + 4)) & np.uint64(0xF)) << np.uint64(4 * m + 16)
    return out.astype(np.uint32)


def _paired_dev(W: dict) -> dict:
    return moe.pair_weights(dev_weights(W))


def test_pair_codes_is_the_stated_permutation():
    rng = np.random.default_rng(3)
    words = rng.integers(0, 2 ** 32, size=4096 + 12, dtype=np.uint64).astype(np.uint32)
    words[0] = 0x76543210  # every nibble distinct
    words[1] = 0xFEDCBA98
    src = dev(words)
    dst = torch.empty_like(src)
    moe.moe_pair_codes(src, dst, words.size)
    inplace = dev(words)
    moe.moe_pair_codes(inplace, inplace, words.size)
    torch.cuda.synchronize()
    want = _paired_host(words)
    assert want[0] == 0x75316420 and want[1] == 0xFDB9ECA8
    np.testing.assert_array_equal(dst.cpu().numpy().view(np.uint32), want)
    np.testing.assert_array_equal(inplace.cpu().numpy().view(np.uint32), want)
    np.testing.assert_array_equal(src.cpu().numpy().view(np.uint32), words)  # source untouched
    moe.moe_pair_codes(src, dst, 0)  # empty: nothing to do
    torch.cuda.synchronize()


def test_dequant_paired_bit_exact():
    rows, K = 64, 2048
    W = syn.experts(6, 1, K, rows)
    q, s, b = W["gate_q"][0], W["gate_s"][0].copy(), W["gate_b"][0].copy()
    # both rebuild routes and their boundary, negative and subnormal scales
    s[0, :], b[0, :] = 0x3C80, 0xBE00
    s[1, :] = 0x3CFF
    s[2, :] = 0x3D00
    s[3, :] = 0xBCFF
    s[4, :], b[4, :] = 0x0001, 0x8001
    s[5, :], b[5, :] = 0x3C00, 0x4B80
    qd = dev(q)
    moe.moe_pair_codes(qd, qd, q.size)
    wd = torch.empty((rows, K), dtype=torch.int16, device="cuda:0")
    moe.moe_dequant(qd, dev(s), dev(b), rows, K, 64, wd, code_order=moe.MOE_CODES_PAIRED)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_u16(wd), orc.dequant(q, s, b))


def _forward(L, x, Wd, res=None, bias=None):
    T = x.shape[0]
    xd = dev(x)
    out = torch.empty_like(xd)
    moe.moe_forward(L.plan, xd, None if res is None else dev(res), T, Wd, None if bias is None else dev(bias), out,
                    L.ws)
    torch.cuda.synchronize()
    return host_u16(out)


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("T", [2, 33, 300])
def test_layer_tiny_paired(path, T):
    d = TINY
    W = syn.experts(400 + T, d["E"] + 1, d["H"], d["I"])
    W["router"] = syn.router(400 + T, d["E"], d["H"])
    x = syn.activations(400 + T, T, d["H"])
    res = syn.activations(400 + T, T, d["H"], tensor=syn.T_RESID)
    bias = syn.zipf_bias(400 + T, d["E"])  # skewed: ragged and tall tiles
    flags = PATHS[path] | moe.MOE_FLAG_FORCE_GROUPED
    Lp = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=300, flags=flags)
    out = _forward(Lp, x, _paired_dev(W), res=res, bias=bias)
    keys = Lp.routing(T)["keys"]
    ref = orc.moe_layer(orc.Dims(**d, n_shared=1), x, W, res=res, keys=keys, intermediates=True)
    assert_outputs_close(out, ref, f"paired tiny T={T} {path}", k=d["k"])
    assert Lp.status() == 0
    if path == "simt":  # the same products in the same order as with the pages' packing
        L0 = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=300, flags=flags)
        np.testing.assert_array_equal(out, _forward(L0, x, dev_weights(W), res=res, bias=bias))


def test_layer_tiny_paired_no_shared_gated():
    d = TINY
    T = 65
    W = syn.experts(41, d["E"], d["H"], d["I"], centred=True)  # no shared expert
    W["router"] = syn.router(41, d["E"], d["H"])
    x = syn.activations(41, T, d["H"])
    L = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], S=0, max_tokens=T)
    out = _forward(L, x, _paired_dev(W))
    ref = orc.moe_layer(orc.Dims(**d, n_shared=0), x, W, keys=L.routing(T)["keys"], intermediates=True)
    assert_outputs_close(out, ref, "paired, no shared expert", k=d["k"], n_shared=0)
    # a shared expert with its sigmoid gate
    Wg = syn.experts(42, d["E"] + 1, d["H"], d["I"])
    Wg["router"] = syn.router(42, d["E"], d["H"])
    Wg["shared_gate"] = syn.shared_gate(42, d["H"], std=0.1)
    Lg = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=T)
    out = _forward(Lg, x, _paired_dev(Wg))
    ref = orc.moe_layer(orc.Dims(**d, n_shared=1), x, Wg, keys=Lg.routing(T)["keys"], intermediates=True)
    assert_outputs_close(out, ref, "paired, gated shared expert", k=d["k"])
    assert L.status() == 0 and Lg.status() == 0


@pytest.fixture(scope="module")
def real_paired():
    W = syn.experts(0, 257, 2048, 512)
    W["router"] = syn.router(0, 256, 2048)
    return W, _paired_dev(W)


def test_layer_t256_paired_full(real_paired):
    W, Wp = real_paired
    T = 256
    x = syn.activations(0, T, 2048)
    L = Layer(max_tokens=T)
    out = _forward(L, x, Wp)
    ref = orc.moe_layer(orc.Dims(), x, W, keys=L.routing(T)["keys"], intermediates=True)
    assert_outputs_close(out, ref, "paired T=256")
    assert L.status() == 0


@pytest.mark.parametrize("T", [2048, 4096])
def test_layer_dense_sizes_paired(real_paired, T):
    W, Wp = real_paired
    x = syn.activations(1000 + T, T, 2048)
    L = Layer(max_tokens=T)
    out = _forward(L, x, Wp)
    assert L.status() == 0
    r = L.routing(T)
    ids, _ = orc.select(r["keys"], 8)
    np.testing.assert_array_equal(r["ids"], ids)
    rows = np.random.default_rng(T + 1).choice(T, 64, replace=False)
    ref = orc.moe_layer(orc.Dims(), x[rows], W, keys=r["keys"][rows], intermediates=True)
    assert_outputs_close(out[rows], ref, f"paired T={T} (64 sampled rows)")


def test_decode_paired_t1_and_static(real_paired):
    # the decode kernel (x and h staged in natural order) and the
    # allocation-free entry point on the same paired weights
    W, Wp = real_paired
    cfg = moe.make_config()
    for seed in (0, 1):
        x = syn.activations(110 + seed, 1, 2048)
        res = syn.activations(110 + seed, 1, 2048, tensor=syn.T_RESID)
        L = Layer(max_tokens=1)
        out = _forward(L, x, Wp, res=res)
        keys = L.routing(1)["keys"]
        ref = orc.moe_layer(orc.Dims(), x, W, res=res, keys=keys, intermediates=True)
        assert_outputs_close(out, ref, f"paired decode T=1 seed {seed}")
        assert L.status() == 0
        xd, rd = dev(x), dev(res)
        got = torch.full_like(xd, 0x7FC0)
        moe.moe_decode_static(cfg, xd, rd, Wp, None, got)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host_u16(got), out)


def test_decode_stack_paired_matches_layer_by_layer():
    # three centred layers, pages' packing and paired mixed within one launch
    Ws = []
    for seed in (3, 4, 5):
        W = syn.experts(seed, 257, 2048, 512, layer=seed, centred=True)
        W["router"] = syn.router(seed, 256, 2048, layer=seed)
        Ws.append(W)
    Wds = [_paired_dev(Ws[0]), dev_weights(Ws[1]), _paired_dev(Ws[2])]
    r = syn.activations(93, 1, 2048, tensor=syn.T_RESID)
    L = Layer(max_tokens=1, flags=moe.MOE_FLAG_PRENORM)
    seq = dev(r)
    inputs = []
    for Wd in Wds:
        inputs.append(host_u16(seq))
        moe.moe_forward(L.plan, seq, None, 1, Wd, None, seq, L.ws)
    Ls = Layer(max_tokens=1)
    rs = dev(r)
    moe.moe_decode_stack(Ls.plan, rs, Wds, None, Ls.ws)
    assert moe.moe_last_launch_count() == 1
    torch.cuda.synchronize()
    assert L.status() == 0 and Ls.status() == 0
    np.testing.assert_array_equal(host_u16(rs), host_u16(seq))
    keys = Ls.routing(1)["keys"]
    ref = orc.moe_layer(orc.Dims(), orc.rmsnorm(inputs[-1], 1e-6), Ws[-1], res=inputs[-1], keys=keys,
                        intermediates=True)
    assert_outputs_close(host_u16(rs), ref, "paired stack layer 3")


def test_prefill_stack_paired_chunks_match_layer_calls_and_oracle():
    # 8192 tokens as two 4096-token chunks through 2 centred layers, paired
    T, chunk = 8192, 4096
    Ws = []
    for l in range(2):
        W = syn.experts(8, 257, 2048, 512, layer=l, centred=True)
        W["router"] = syn.router(8, 256, 2048, layer=l)
        Ws.append(W)
    Wps = [_paired_dev(W) for W in Ws]
    r0 = syn.activations(73, T, 2048, tensor=syn.T_RESID)
    L = Layer(max_tokens=chunk, flags=moe.MOE_FLAG_PRENORM)
    rd = dev(r0)
    moe.moe_prefill_stack(L.plan, rd, T, Wps, None, L.ws)
    torch.cuda.synchronize()
    assert L.status() == 0
    got = host_u16(rd)
    # the same stack as single-layer calls, tapped on sampled rows
    sample = sorted(np.random.default_rng(9).choice(T, 16, replace=False).tolist())
    Lc = Layer(max_tokens=chunk, flags=moe.MOE_FLAG_PRENORM)
    rs = dev(r0)
    for c0 in range(0, T, chunk):
        rows = [i - c0 for i in sample if c0 <= i < c0 + chunk]
        for l, Wp in enumerate(Wps):
            r_in = host_u16(rs[c0:c0 + chunk])[rows]
            moe.moe_forward(Lc.plan, rs[c0:c0 + chunk], None, chunk, Wp, None, rs[c0:c0 + chunk], Lc.ws)
            torch.cuda.synchronize()
            keys = Lc.routing(chunk)["keys"][rows]
            r_out = host_u16(rs[c0:c0 + chunk])[rows]
            ref = orc.moe_layer(orc.Dims(), orc.rmsnorm(r_in, 1e-6), Ws[l], res=r_in, keys=keys, intermediates=True)
            assert_outputs_close(r_out, ref, f"paired stack layer {l} chunk {c0 // chunk}")
    np.testing.assert_array_equal(got, host_u16(rs))
    assert Lc.status() == 0
