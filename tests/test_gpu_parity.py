"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Routing must be bit-exact given identical fp32 keys;
dequantisation bit-exact; outputs within the layer's tolerance (see
tests/tolerances.py)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as orc
import synthetic as syn
from tests.tolerances import assert_outputs_close, bf16_value, output_errors

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bit_grouped_expert_gb300 as moe  # noqa: E402
from tests.gpu_util import Layer, dev, dev_weights, host_u16  # noqa: E402

TINY = dict(H=256, E=16, k=4, I=256)  # H, I multiples of 256: both expert paths apply
PATHS = {"tc": 0, "simt": moe.MOE_FLAG_SIMT_EXPERTS}


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


def _tiny(seed, S=1, centred=False, **kw):
    d = {**TINY, **kw}
    W = syn.experts(seed, d["E"] + S, d["H"], d["I"], centred=centred)
    W["router"] = syn.router(seed, d["E"], d["H"])
    return d, W, dev_weights(W)


def _forward(L: Layer, x, Wd, res=None, bias=None, T=None):
    T = x.shape[0] if T is None else T
    xd = dev(x)
    resd = None if res is None else dev(res)
    out = torch.empty_like(xd)
    moe.moe_forward(L.plan, xd, resd, T, Wd, None if bias is None else dev(bias), out, L.ws)
    torch.cuda.synchronize()
    return host_u16(out)


def _route_ref(keys, k, E, S, BN):
    ids, w = orc.select(keys, k)
    m = orc.route_maps(ids, E, n_shared=S, BN=BN)
    return ids, w, m


def _assert_routing_equal(got, keys, k, E, S):
    ids, w, m = _route_ref(keys, k, E, S, got["block_rows"])
    np.testing.assert_array_equal(got["ids"], ids)
    np.testing.assert_allclose(got["w"], w, rtol=2e-6, atol=1e-7)
    np.testing.assert_array_equal(got["counts"], m["counts"])
    np.testing.assert_array_equal(got["offsets"], m["offsets"])
    np.testing.assert_array_equal(got["perm"], m["perm"])
    np.testing.assert_array_equal(got["inv"], m["inv"])
    assert got["n_tiles"] == m["n_tiles"]
    np.testing.assert_array_equal(got["blockmap"], m["blockmap"])
    if got["block_rows2"]:  # the down GEMM's map of taller tiles
        m2 = orc.route_maps(ids, E, n_shared=S, BN=got["block_rows2"])
        assert got["n_tiles2"] == m2["n_tiles"]
        np.testing.assert_array_equal(got["blockmap2"], m2["blockmap"])


# ---------------------------------------------------------------- dequant

def test_dequant_bit_exact():
    rows, K = 256, 2048
    W = syn.experts(5, 1, K, rows)
    q, s, b = W["gate_q"][0], W["gate_s"][0], W["gate_b"][0]
    # add the worked example and edge values: zero scale/bias, ties, tiny bias
    s = s.copy()
    b = b.copy()
    s[0, :] = 0x3C80
    b[0, :] = 0xBE00
    s[1, :] = 0
    b[1, :] = 0
    s[2, :] = 0x3F81
    b[2, :] = 0
    b[3, :] = 0x0001  # subnormal bias
    # both rebuild routes and their boundary: scales below 2^-5 take the
    # masked-code route, 2^-5 and above the 0x4300 | q route
    s[4, :] = 0x3CFF   # largest scale of the masked-code route
    s[5, :] = 0x3D00   # 2^-5: the other route
    s[6, :] = 0xBCFF   # negative scale
    s[7, :] = 0x0001   # subnormal scale
    b[7, :] = 0x8001
    s[8, :] = 0x3A80
    b[8, :] = 0xBC40   # bias cancelling s*q for some codes
    s[9, :] = 0x3C00
    b[9, :] = 0x4B80   # bias far above s*q
    wd = torch.empty((rows, K), dtype=torch.int16, device="cuda:0")
    moe.moe_dequant(dev(q), dev(s), dev(b), rows, K, 64, wd)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_u16(wd), orc.dequant(q, s, b))


# ---------------------------------------------------------------- routing

@pytest.mark.parametrize("T", [16, 256, 300, 2048])
def test_router_keys_within_fp32_bound(real, T):
    # T >= 32 runs the tensor-core router (3 x bf16 split), T = 16 the CUDA-core one
    W, Wd = real
    x = syn.activations(T, T, 2048)
    bias = syn.zipf_bias(T, 256)
    L = Layer(max_tokens=T)
    moe.moe_route(L.plan, dev(x), T, Wd["router"], dev(bias), L.ws)
    torch.cuda.synchronize()
    got = L.routing(T)["keys"].astype(np.float64)
    ref = orc.logits(x, W["router"], bias).astype(np.float64)
    mag = np.abs(bf16_value(x)) @ np.abs(W["router"].astype(np.float64)).T + np.abs(bias)[None, :]
    bound = 2048 * 2.0 ** -24 * mag + np.abs(ref) * 2.0 ** -23
    assert (np.abs(got - ref) <= bound).all()


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("T,zipf", [(256, False), (512, True), (77, False)])
def test_routing_bit_exact_given_keys(real, path, T, zipf):
    W, Wd = real
    x = syn.activations(T, T, 2048)
    bias = syn.zipf_bias(T, 256) if zipf else None
    L = Layer(max_tokens=T, flags=PATHS[path])
    moe.moe_route(L.plan, dev(x), T, Wd["router"], None if bias is None else dev(bias), L.ws)
    torch.cuda.synchronize()
    got = L.routing(T)
    _assert_routing_equal(got, got["keys"], 8, 256, 1)
    assert L.status() == 0


@pytest.mark.parametrize("path", sorted(PATHS))
def test_routing_edge_cases_from_keys(path):
    E, k = 16, 4
    L = Layer(H=256, E=E, k=k, I=256, max_tokens=520, flags=PATHS[path])
    v = L.view(1)
    BN = max(v.block_rows, v.block_rows2)  # groups of BN-1, BN, BN+1 rows in the taller tiles
    rng = np.random.default_rng(3)
    T = 2 * BN + 5
    keys = rng.normal(size=(T, E)).astype(np.float32)
    # about BN-1, BN, BN+1 rows on experts 1, 2, 3 (rows 5-7 below add a few);
    # expert 15 is never picked
    keys[:, 0] = -100
    keys[:, 15] = -100
    keys[: BN - 1, 1] = 50
    keys[:BN, 2] = 49
    keys[: BN + 1, 3] = 48
    keys[5, :] = 0.0          # all-equal row -> experts 0..3
    keys[6, 4:8] = 7.0        # ties -> lower index first
    keys[7, 9] = -0.0
    keys[7, 10] = 0.0
    kd = dev(keys)
    moe.moe_route_from_logits(L.plan, kd, T, L.ws)
    torch.cuda.synchronize()
    got = L.routing(T)
    np.testing.assert_array_equal(got["keys"], keys)
    _assert_routing_equal(got, keys, k, E, 1)
    assert list(got["ids"][5]) == [0, 1, 2, 3] and np.all(got["w"][5] == 0.25)
    assert L.status() == 0


@pytest.mark.parametrize("E,k,T", [(40, 3, 1500), (1024, 16, 300), (256, 8, 4096)])
def test_routing_spans_scatter_chunks(E, k, T):
    # the scatter kernel takes 2048 (token, slot) pairs a block: several
    # blocks here, tokens whose pairs straddle two blocks (k = 3), the most
    # experts a plan takes (E = 1024), and three hot experts whose pairs run
    # through every block
    L = Layer(H=256, E=E, k=k, I=256, max_tokens=T)
    rng = np.random.default_rng(E + k)
    keys = rng.normal(size=(T, E)).astype(np.float32)
    keys[:, :3] += 2.0
    moe.moe_route_from_logits(L.plan, dev(keys), T, L.ws)
    torch.cuda.synchronize()
    got = L.routing(T)
    assert T * k > 2 * 2048
    _assert_routing_equal(got, keys, k, E, 1)
    assert L.status() == 0


@pytest.mark.parametrize("T", [16, 300, 4096])
def test_routing_resets_between_calls(real, T):
    # a second call on the same workspace routes only its own tokens: the
    # histograms start from zero each call (cleared by a memset below 32
    # tokens, by the tensor-core router itself above), so the counts, the
    # offsets and the maps match the oracle for the second input alone
    W, Wd = real
    L = Layer(max_tokens=T)
    for seed in (21, 22):
        x = syn.activations(seed, T, 2048)
        moe.moe_route(L.plan, dev(x), T, Wd["router"], None, L.ws)
        torch.cuda.synchronize()
    got = L.routing(T)
    _assert_routing_equal(got, got["keys"], 8, 256, 1)
    assert int(got["counts"].sum()) == 8 * T
    assert L.status() == 0


def test_routing_is_deterministic(real):
    W, Wd = real
    T = 512
    x = syn.activations(9, T, 2048)
    L = Layer(max_tokens=T)
    outs = []
    for _ in range(2):
        moe.moe_route(L.plan, dev(x), T, Wd["router"], None, L.ws)
        torch.cuda.synchronize()
        r = L.routing(T)
        outs.append(np.concatenate([r["perm"], r["inv"], r["ids"].ravel(), r["w"].view(np.int32).ravel()]))
    np.testing.assert_array_equal(outs[0], outs[1])


# ---------------------------------------------------------------- layer, tiny dims

def test_default_plan_uses_tensor_core_path():
    # the second map's tile height follows the down GEMM's mode for T tokens:
    # taller tiles from k T / E >= 96, short tiles below 12
    L = Layer(max_tokens=4096)
    assert (L.view(4096).block_rows, L.view(4096).block_rows2) == (128, 192)
    assert L.view(8).block_rows2 == 64
    v = Layer(max_tokens=8, flags=moe.MOE_FLAG_TILE_ROWS_64).view(1)
    assert (v.block_rows, v.block_rows2) == (64, 64)
    v = Layer(max_tokens=8, flags=moe.MOE_FLAG_SIMT_EXPERTS).view(1)
    assert (v.block_rows, v.block_rows2) == (32, 0)


@pytest.mark.parametrize("T", [1, 5, 64, 129, 300])
def test_tc_tile_rows_64_tiny(T):
    d, W, Wd = _tiny(40 + T)
    x = syn.activations(40 + T, T, d["H"])
    bias = syn.zipf_bias(40 + T, d["E"])
    L = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=300,
              flags=moe.MOE_FLAG_TILE_ROWS_64 | moe.MOE_FLAG_FORCE_GROUPED)
    out = _forward(L, x, Wd, bias=bias)
    ref = orc.moe_layer(orc.Dims(**d, n_shared=1), x, W, bias=bias, keys=L.routing(T)["keys"], intermediates=True)
    assert_outputs_close(out, ref, f"tc64 T={T}", k=d["k"])
    assert L.status() == 0

@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("T", [2, 3, 7, 33, 100, 300])
def test_layer_tiny_dims(path, T):
    d, W, Wd = _tiny(T)
    x = syn.activations(T, T, d["H"])
    res = syn.activations(T, T, d["H"], tensor=syn.T_RESID)
    bias = syn.zipf_bias(T, d["E"])
    L = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=300, flags=PATHS[path])
    out = _forward(L, x, Wd, res=res, bias=bias)
    r = L.routing(T)
    keys = r["keys"]
    ref = orc.moe_layer(orc.Dims(**d, n_shared=1), x, W, res=res, keys=keys, intermediates=True)
    assert_outputs_close(out, ref, f"tiny T={T} {path}", k=d["k"])
    assert L.status() == 0


@pytest.mark.parametrize("T", [40, 300, 700])
def test_layer_tiny_dims_both_down_modes(T):
    # k T / E < 12 (T = 40): the down GEMM takes two output tiles per item,
    # two items in flight, over the second map cut into 64-row tiles (as do
    # the tiny-dims tests below T = 48 and the real-dims T = 256 tests, whose
    # shared expert spans four such tiles); k T / E < 96 (T = 300):
    # two output tiles per item over the 128-row map; T = 700: one output
    # tile per item over the 192-row map, where the skew puts more than 128
    # rows in a tile
    d, W, Wd = _tiny(500 + T)
    x = syn.activations(500 + T, T, d["H"])
    bias = syn.zipf_bias(500 + T, d["E"])
    L = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=T)
    out = _forward(L, x, Wd, bias=bias)
    r = L.routing(T)
    if T == 700:
        assert d["k"] * T >= 96 * d["E"] and (r["blockmap2"][:, 2] > 128).any()
    elif T == 300:
        assert d["k"] * T < 96 * d["E"] and (r["blockmap"][:, 2] > 64).any()
    else:
        assert d["k"] * T < 12 * d["E"] and r["block_rows2"] == 64 and (r["blockmap2"][:, 2] <= 64).all()
    ref = orc.moe_layer(orc.Dims(**d, n_shared=1), x, W, bias=bias, keys=r["keys"], intermediates=True)
    assert_outputs_close(out, ref, f"tiny T={T} down modes", k=d["k"])
    assert L.status() == 0


@pytest.mark.parametrize("path", sorted(PATHS))
def test_layer_tiny_no_shared_centred(path):
    T = 65
    d, W, Wd = _tiny(11, S=0, centred=True)
    x = syn.activations(11, T, d["H"])
    L = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], S=0, max_tokens=T, flags=PATHS[path])
    out = _forward(L, x, Wd)
    ref = orc.moe_layer(orc.Dims(**d, n_shared=0), x, W, keys=L.routing(T)["keys"], intermediates=True)
    assert_outputs_close(out, ref, k=d["k"], n_shared=0)


# ---------------------------------------------------------------- shared-expert sigmoid gate

def _gated(W, seed, H, std=0.1):
    """W with a shared-expert gate vector, and the same weights without one."""
    Wg = dict(W)
    Wg["shared_gate"] = syn.shared_gate(seed, H, std=std)
    return Wg


def _gate_matters(out, d, x, W, keys, res=None):
    # the ungated layer is not within tolerance of the result: the test above
    # would catch a path that ignores the gate
    ref0 = orc.moe_layer(orc.Dims(**d, n_shared=1) if d else orc.Dims(), x, W, res=res, keys=keys)
    assert not output_errors(out, ref0["out_exact"])["ok"]


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("T", [1, 7, 300])
def test_layer_tiny_shared_gate(path, T):
    d, W, _ = _tiny(40 + T)
    Wg = _gated(W, 40 + T, d["H"])
    x = syn.activations(40 + T, T, d["H"])
    res = syn.activations(40 + T, T, d["H"], tensor=syn.T_RESID)
    L = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=300, flags=PATHS[path])
    out = _forward(L, x, dev_weights(Wg), res=res)
    keys = L.routing(T)["keys"]
    ref = orc.moe_layer(orc.Dims(**d, n_shared=1), x, Wg, res=res, keys=keys, intermediates=True)
    assert_outputs_close(out, ref, f"gated tiny T={T} {path}", k=d["k"])
    _gate_matters(out, d, x, W, keys, res=res)
    assert L.status() == 0


@pytest.mark.parametrize("T", [1, 256])
def test_layer_real_dims_shared_gate(real, T):
    # T=1: the decode kernel (gate row on the router CTAs); T=256: the grouped
    # path's combine kernel
    W, Wd = real
    Wg = _gated(W, 7, 2048, std=0.02)
    Wgd = dict(Wd)
    Wgd["shared_gate"] = dev(Wg["shared_gate"])
    x = syn.activations(60 + T, T, 2048)
    res = syn.activations(60 + T, T, 2048, tensor=syn.T_RESID)
    L = Layer(max_tokens=T)
    out = _forward(L, x, Wgd, res=res)
    keys = L.routing(T)["keys"]
    ref = orc.moe_layer(orc.Dims(), x, Wg, res=res, keys=keys, intermediates=True)
    assert_outputs_close(out, ref, f"gated T={T}")
    _gate_matters(out, None, x, W, keys, res=res)
    assert L.status() == 0


# ---------------------------------------------------------------- layer, real dims

@pytest.mark.parametrize("path", sorted(PATHS))
def test_layer_t256_full(real, path):
    W, Wd = real
    T = 256
    x = syn.activations(0, T, 2048)
    L = Layer(max_tokens=T, flags=PATHS[path])
    out = _forward(L, x, Wd)
    ref = orc.moe_layer(orc.Dims(), x, W, keys=L.routing(T)["keys"], intermediates=True)
    assert_outputs_close(out, ref, f"T=256 {path}")
    assert L.status() == 0


def test_layer_t256_centred_full():
    W = syn.experts(1, 257, 2048, 512, centred=True)
    W["router"] = syn.router(1, 256, 2048)
    Wd = dev_weights(W)
    T = 256
    x = syn.activations(1, T, 2048)
    L = Layer(max_tokens=T)
    out = _forward(L, x, Wd)
    ref = orc.moe_layer(orc.Dims(), x, W, keys=L.routing(T)["keys"], intermediates=True)
    assert_outputs_close(out, ref, "T=256 centred")


def test_layer_t512_zipf_sampled(real):
    W, Wd = real
    T = 512
    x = syn.activations(2, T, 2048)
    bias = syn.zipf_bias(2, 256)
    L = Layer(max_tokens=T)
    out = _forward(L, x, Wd, bias=bias)
    r = L.routing(T)
    assert (r["counts"] == 0).sum() > 50  # skewed: many experts get no token
    rows = np.random.default_rng(0).choice(T, 40, replace=False)
    ref = orc.moe_layer(orc.Dims(), x[rows], W, keys=r["keys"][rows], intermediates=True)
    assert_outputs_close(out[rows], ref, "T=512 zipf sample")


@pytest.mark.parametrize("T", [512, 4096])
def test_layer_all_tokens_to_eight_experts(real, T):
    # the degenerate routing: a bias that puts experts 0..7 first for every
    # token, so eight experts take all T rows each (several full tiles, over
    # the down GEMM's taller tiles at T = 4096) and the other 248 none
    W, Wd = real
    x = syn.activations(5, T, 2048)
    bias = np.zeros(256, np.float32)
    bias[:8] = 50.0
    L = Layer(max_tokens=T)
    out = _forward(L, x, Wd, bias=bias)
    r = L.routing(T)
    np.testing.assert_array_equal(r["counts"][:8], np.full(8, T))
    assert int(r["counts"][8:].sum()) == 0
    _assert_routing_equal(r, r["keys"], 8, 256, 1)
    rows = np.random.default_rng(1).choice(T, 40, replace=False)
    ref = orc.moe_layer(orc.Dims(), x[rows], W, keys=r["keys"][rows], intermediates=True)
    assert_outputs_close(out[rows], ref, f"T={T}, every token to experts 0..7")
    assert L.status() == 0


# ---------------------------------------------------------------- decode path

def test_decode_t1_matches_oracle_and_grouped(real):
    W, Wd = real
    for seed in (0, 1, 2):
        x = syn.activations(100 + seed, 1, 2048)
        res = syn.activations(100 + seed, 1, 2048, tensor=syn.T_RESID)
        Ld = Layer(max_tokens=1)
        out_d = _forward(Ld, x, Wd, res=res)
        keys = Ld.routing(1)["keys"]
        ref = orc.moe_layer(orc.Dims(), x, W, res=res, keys=keys, intermediates=True)
        assert_outputs_close(out_d, ref, "decode T=1")
        ids, w = orc.select(keys, 8)
        np.testing.assert_array_equal(Ld.routing(1)["ids"], ids)
        Lg = Layer(max_tokens=1, flags=moe.MOE_FLAG_FORCE_GROUPED)
        out_g = _forward(Lg, x, Wd, res=res)
        assert_outputs_close(out_g, ref, "grouped T=1")
        assert Ld.status() == 0 and Lg.status() == 0


def test_decode_tiny_dims_in_place_residual():
    d, W, Wd = _tiny(21)
    x = syn.activations(21, 1, d["H"])
    res = syn.activations(21, 1, d["H"], tensor=syn.T_RESID)
    L = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=4)
    xd, rd = dev(x), dev(res)
    moe.moe_forward(L.plan, xd, rd, 1, Wd, None, rd, L.ws)  # out aliases residual
    torch.cuda.synchronize()
    ref = orc.moe_layer(orc.Dims(**d, n_shared=1), x, W, res=res, keys=L.routing(1)["keys"], intermediates=True)
    assert_outputs_close(host_u16(rd), ref, k=d["k"])


@pytest.mark.parametrize("T", [1, 37])
def test_prenorm_in_place_matches_oracle(T):
    # pre-norm block: out = r + MoE(RMSNorm(r)), written over r
    d, W, Wd = _tiny(60 + T)
    r = syn.activations(60 + T, T, d["H"], tensor=syn.T_RESID)
    L = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=64, flags=moe.MOE_FLAG_PRENORM)
    rd = dev(r)
    moe.moe_forward(L.plan, rd, None, T, Wd, None, rd, L.ws)
    torch.cuda.synchronize()
    x = orc.rmsnorm(r, 1e-6)
    ref = orc.moe_layer(orc.Dims(**d, n_shared=1), x, W, res=r, keys=L.routing(T)["keys"], intermediates=True)
    assert_outputs_close(host_u16(rd), ref, f"prenorm T={T}", k=d["k"])
    assert L.status() == 0


def test_decode_real_dims_prenorm_and_deterministic(real):
    W, Wd = real
    r = syn.activations(77, 1, 2048, tensor=syn.T_RESID)
    L = Layer(max_tokens=1, flags=moe.MOE_FLAG_PRENORM)
    outs = []
    for _ in range(3):
        rd = dev(r)
        moe.moe_forward(L.plan, rd, None, 1, Wd, None, rd, L.ws)
        torch.cuda.synchronize()
        outs.append(host_u16(rd))
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])
    ref = orc.moe_layer(orc.Dims(), orc.rmsnorm(r, 1e-6), W, res=r, keys=L.routing(1)["keys"], intermediates=True)
    assert_outputs_close(outs[0], ref, "decode prenorm")
    assert L.status() == 0


@pytest.mark.parametrize("E,k", [(512, 8), (40, 16)])
def test_decode_expert_counts(E, k):
    # E > 256: the CTA-wide selection; E=40, k=16: half of the warp's lanes
    # hold two keys and the k-th lane maximum sits among them
    d, W, Wd = _tiny(30 + E, E=E, k=k)
    x = syn.activations(30 + E, 1, d["H"])
    res = syn.activations(30 + E, 1, d["H"], tensor=syn.T_RESID)
    L = Layer(H=d["H"], E=E, k=k, I=d["I"], max_tokens=1)
    out = _forward(L, x, Wd, res=res)
    r = L.routing(1)
    ids, w = orc.select(r["keys"], k)
    np.testing.assert_array_equal(r["ids"], ids)
    np.testing.assert_allclose(r["w"], w, rtol=2e-6, atol=1e-7)
    ref = orc.moe_layer(orc.Dims(**d, n_shared=1), x, W, res=res, keys=r["keys"], intermediates=True)
    assert_outputs_close(out, ref, f"decode E={E} k={k}", k=k)
    assert L.status() == 0


def test_decode_tied_keys_take_the_lower_expert(real):
    # router rows repeated in pairs: every key ties with its neighbour's
    W, _ = real
    W2 = dict(W)
    W2["router"] = np.repeat(W["router"][::2], 2, axis=0)
    Wd = dev_weights(W2)
    x = syn.activations(123, 1, 2048)
    L = Layer(max_tokens=1)
    out = _forward(L, x, Wd)
    r = L.routing(1)
    assert np.all(r["keys"][0, ::2] == r["keys"][0, 1::2])
    ids, w = orc.select(r["keys"], 8)
    np.testing.assert_array_equal(r["ids"], ids)
    assert set(ids[0, 0::2] % 2) == {0} and set(ids[0, 1::2] % 2) == {1}  # pairs, lower index first
    ref = orc.moe_layer(orc.Dims(), x, W2, keys=r["keys"], intermediates=True)
    assert_outputs_close(out, ref, "decode tied keys")


def _stack_vs_layers(d, Ws, biases, r):
    """moe_decode_stack over the layers against one PRENORM moe_forward per
    layer; returns (stack result, per-layer inputs of the sequential run, the
    plan used by the stack)."""
    L = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=1, flags=moe.MOE_FLAG_PRENORM)
    Wds = [dev_weights(W) for W in Ws]
    bds = [None if b is None else dev(b) for b in biases]
    seq = dev(r)
    inputs = []
    for Wd, b in zip(Wds, bds):
        inputs.append(host_u16(seq))
        moe.moe_forward(L.plan, seq, None, 1, Wd, b, seq, L.ws)
    torch.cuda.synchronize()
    Ls = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=1)
    rs = dev(r)
    moe.moe_decode_stack(Ls.plan, rs, Wds, bds if any(b is not None for b in biases) else None, Ls.ws)
    launches = moe.moe_last_launch_count()
    torch.cuda.synchronize()
    assert L.status() == 0 and Ls.status() == 0
    np.testing.assert_array_equal(host_u16(rs), host_u16(seq))
    return host_u16(rs), inputs, Ls, launches


def _centred_layers(seeds):
    # centred weights: with the literal generator's mean weight a stack's
    # residual stream runs away after its first layer (or the later layers'
    # gates saturate and add exactly nothing), which a stack test would not see
    Ws = []
    for seed in seeds:
        W = syn.experts(seed, 257, 2048, 512, layer=seed, centred=True)
        W["router"] = syn.router(seed, 256, 2048, layer=seed)
        Ws.append(W)
    return Ws


def test_decode_stack_real_dims_matches_layer_by_layer():
    # three distinct layers at the model's dims: one launch, bit-identical to
    # three single-layer calls; the last layer also against the oracle
    Ws = _centred_layers((0, 1, 2))
    biases = [None, syn.zipf_bias(5, 256), None]
    r = syn.activations(88, 1, 2048, tensor=syn.T_RESID)
    out, inputs, Ls, launches = _stack_vs_layers(dict(H=2048, E=256, k=8, I=512), Ws, biases, r)
    assert launches == 1
    r_last = inputs[-1]
    keys = Ls.routing(1)["keys"]
    ref = orc.moe_layer(orc.Dims(), orc.rmsnorm(r_last, 1e-6), Ws[-1], res=r_last, keys=keys, intermediates=True)
    assert_outputs_close(out, ref, "stack layer 3")


def test_decode_stack_tiny_dims_spans_launches():
    # nine layers at tiny dims: more layers than one launch carries
    Ws, biases = [], []
    for l in range(9):
        d, W, _ = _tiny(200 + l)
        Ws.append(W)
        biases.append(syn.zipf_bias(200 + l, d["E"]) if l % 3 == 1 else None)
    r = syn.activations(90, 1, d["H"], tensor=syn.T_RESID)
    out, inputs, Ls, launches = _stack_vs_layers(d, Ws, biases, r)
    assert launches == 2
    keys = Ls.routing(1)["keys"]
    ref = orc.moe_layer(orc.Dims(**d, n_shared=1), orc.rmsnorm(inputs[-1], 1e-6), Ws[-1], res=inputs[-1],
                        keys=keys, intermediates=True)
    assert_outputs_close(out, ref, "stack layer 9", k=d["k"])


def test_decode_stack_mixed_shared_gates():
    # eight tiny layers, a gate vector on every other one: the gate row's
    # copy size and tagged word change from layer to layer within a launch
    Ws = []
    for l in range(8):
        d, W, _ = _tiny(300 + l)
        Ws.append(_gated(W, 300 + l, d["H"]) if l % 2 == 0 else W)
    r = syn.activations(92, 1, d["H"], tensor=syn.T_RESID)
    out, inputs, Ls, launches = _stack_vs_layers(d, Ws, [None] * 8, r)
    assert launches == 2
    keys = Ls.routing(1)["keys"]
    ref = orc.moe_layer(orc.Dims(**d, n_shared=1), orc.rmsnorm(inputs[-1], 1e-6), Ws[-1], res=inputs[-1],
                        keys=keys, intermediates=True)
    assert_outputs_close(out, ref, "gated stack layer 8", k=d["k"])


def test_decode_stack_repeated_tokens_seven_layers():
    # one full launch (7 layers) per token, several tokens in a row on one
    # workspace: the tagged exchange must hand every launch its own values
    Wds = [dev_weights(W) for W in _centred_layers(range(7))]
    L = Layer(max_tokens=1, flags=moe.MOE_FLAG_PRENORM)
    Ls = Layer(max_tokens=1)
    for t in range(6):
        r = syn.activations(500 + t, 1, 2048, tensor=syn.T_RESID)
        seq, rs = dev(r), dev(r)
        for Wd in Wds:
            moe.moe_forward(L.plan, seq, None, 1, Wd, None, seq, L.ws)
        moe.moe_decode_stack(Ls.plan, rs, Wds, None, Ls.ws)
        torch.cuda.synchronize()
        assert L.status() == 0 and Ls.status() == 0, f"token {t}"
        np.testing.assert_array_equal(host_u16(rs), host_u16(seq), err_msg=f"token {t}")


def test_decode_stack_single_layer(real):
    W, _ = real
    r = syn.activations(91, 1, 2048, tensor=syn.T_RESID)
    _, _, _, launches = _stack_vs_layers(dict(H=2048, E=256, k=8, I=512), [W], [None], r)
    assert launches == 1


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("T", [1, 40])
def test_zero_expert_weights_return_residual(T):
    d, W, _ = _tiny(3)
    for n in ("gate_s", "gate_b", "up_s", "up_b", "down_s", "down_b"):
        W[n][:] = 0
    Wd = dev_weights(W)
    x = syn.activations(4, T, d["H"])
    res = syn.activations(4, T, d["H"], tensor=syn.T_RESID)
    for flags in PATHS.values():
        L = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=64, flags=flags)
        np.testing.assert_array_equal(_forward(L, x, Wd, res=res), res)


def test_nonfinite_router_key_sets_status():
    d, W, Wd = _tiny(5)
    x = syn.activations(5, 9, d["H"])
    x[4, 17] = 0x7FC0  # NaN
    for T, xs in ((9, x), (1, x[4:5])):
        L = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=16)
        _forward(L, xs, Wd)
        assert L.status() == moe.MOE_ERR_NONFINITE
        assert L.status() == 0  # reset by the previous read


def test_max_tokens_and_ragged_tail():
    d, W, Wd = _tiny(6)
    T = 257
    x = syn.activations(6, T, d["H"])
    L = Layer(H=d["H"], E=d["E"], k=d["k"], I=d["I"], max_tokens=T)
    out = _forward(L, x, Wd)
    ref = orc.moe_layer(orc.Dims(**d, n_shared=1), x, W, keys=L.routing(T)["keys"], intermediates=True)
    assert_outputs_close(out, ref, k=d["k"])
    with pytest.raises(moe.MoeError) as ei:
        _forward(L, syn.activations(6, T + 1, d["H"]), Wd)
    assert ei.value.status == moe.MOE_ERR_TOO_MANY_TOKENS


def test_layer_output_deterministic(real):
    W, Wd = real
    x = syn.activations(8, 300, 2048)
    L = Layer(max_tokens=300)
    a = _forward(L, x, Wd)
    b = _forward(L, x, Wd)
    np.testing.assert_array_equal(a, b)


def test_rmsnorm_matches_oracle():
    r = syn.activations(12, 33, 2048)
    xd = torch.empty((33, 2048), dtype=torch.int16, device="cuda:0")
    moe.moe_rmsnorm(dev(r), 33, 2048, 1e-6, xd)
    torch.cuda.synchronize()
    got = bf16_value(host_u16(xd))
    want = bf16_value(orc.rmsnorm(r, 1e-6))
    # fp32 vs fp64 norm: at most one bf16 step apart
    assert (np.abs(got - want) <= np.abs(want) * 2.0 ** -7 + 1e-30).all()
    assert (got == want).mean() > 0.99


def test_forward_captures_into_cuda_graph(real):
    W, Wd = real
    for T in (1, 64):
        x = syn.activations(13, T, 2048)
        L = Layer(max_tokens=64)
        eager = _forward(L, x, Wd)
        xd = dev(x)
        out = torch.empty_like(xd)
        cw = moe.make_weights(Wd)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                moe.moe_forward(L.plan, xd, None, T, cw, None, out, L.ws, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host_u16(out), eager)
