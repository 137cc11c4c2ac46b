"""Pins for the CPU oracle: each check ties it to something other than itself
(the pages' printed figures, hand-derived worked examples, closed forms,
invariants, an independent numpy brute force and library routines)."""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as orc
import synthetic as syn
from oracle import brute
from tests.tolerances import assert_outputs_close, bf16_value

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits_of(v: float) -> int:
    return int(np.float32(v).view(np.uint32)) >> 16


def _exact_rne_bf16(x: Fraction) -> int:
    """Independent exact nearest-even rounding of a rational to bf16 bits."""
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    a = -x if x < 0 else x
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    quantum = Fraction(2) ** (e - 7)
    m = a / quantum
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign | _bf16_bits_of(float(fl * quantum))


def _pack_codes(codes: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, np.uint32).reshape(codes.shape[0], -1, 8)
    words = np.zeros(codes.shape[:2], np.uint32)
    for i in range(8):
        words |= codes[:, :, i] << np.uint32(4 * i)
    return words


# --------------------------------------------------------------- pages' figures

def _pages_figures():
    vals = {}
    with open(os.path.join(GOLDEN, "pages_figures.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, value = line.split()[:2]
            vals[name] = float(value)
    return vals


def test_format_bytes_match_pages_ratio():
    fig = _pages_figures()
    H, I, G = 2048, 512, int(fig["group_size"])
    weights = 3 * H * I
    bits_per_weight = fig["code_bits"] + 2 * fig["affine_param_bits"] / G  # 4.5
    assert bits_per_weight == 4.5
    assert orc.expert_bytes(H, I, G) == 1_769_472 == weights * bits_per_weight / 8
    # ~70 GB bf16 -> 19.4 GB: 35e9 params at 2 bytes is 70 GB, at 4.5 bits 19.7 GB
    params = fig["total_params_b"] * 1e9
    assert abs(params * 2 / 1e9 - fig["bf16_checkpoint_gb"]) < 1e-9
    assert abs(params * bits_per_weight / 8 / 1e9 - fig["packed_checkpoint_gb"]) / fig["packed_checkpoint_gb"] < 0.02
    # the MoE weights of 40 layers stay inside the model's size
    moe_params = (fig["routed_experts"] + fig["shared_experts"]) * weights * (fig["attention_layers"] + fig["deltanet_layers"])
    assert moe_params < params
    active = (fig["experts_per_token"] + fig["shared_experts"]) * weights * 40
    assert active < fig["active_params_b"] * 1e9


# --------------------------------------------------------------- dequantisation

def _golden_dequant_rows():
    rows = []
    with open(os.path.join(GOLDEN, "dequant_worked_example.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                s, b, q, w = line.split()
                rows.append((int(s, 16), int(b, 16), int(q), int(w, 16)))
    return rows


def test_dequant_worked_examples():
    rows = _golden_dequant_rows()
    assert len(rows) >= 16
    for s, b, q, want in rows:
        codes = np.full((1, 64), q, np.uint32)
        w = orc.dequant(_pack_codes(codes), np.array([[s]], np.uint16), np.array([[b]], np.uint16))
        assert (w == want).all(), (hex(s), hex(b), q, hex(int(w[0, 0])), hex(want))


def test_packing_pattern_low_nibble_first():
    words = np.array([[0x76543210, 0xFEDCBA98] * 4], np.uint32)  # one row, 64 columns
    one, zero = np.array([[0x3F80]], np.uint16), np.array([[0]], np.uint16)
    w = orc.dequant(words, one, zero)
    assert list(bf16_value(w[0, :16])) == list(range(16))
    np.testing.assert_array_equal(w, brute.dequant(words, one, zero))


def test_dequant_groups_index_along_k():
    # two rows, 128 columns: each (row, group) has its own scale and bias
    codes = np.tile(np.arange(16, dtype=np.uint32), (2, 8))
    s = np.array([[_bf16_bits_of(1.0), _bf16_bits_of(2.0)], [_bf16_bits_of(4.0), _bf16_bits_of(0.5)]], np.uint16)
    b = np.array([[_bf16_bits_of(0.0), _bf16_bits_of(-1.0)], [_bf16_bits_of(3.0), _bf16_bits_of(0.25)]], np.uint16)
    w = bf16_value(orc.dequant(_pack_codes(codes), s, b))
    q = codes.astype(np.float64)
    want = np.empty_like(q)
    want[0, :64], want[0, 64:] = q[0, :64] * 1.0, q[0, 64:] * 2.0 - 1.0
    want[1, :64], want[1, 64:] = q[1, :64] * 4.0 + 3.0, q[1, 64:] * 0.5 + 0.25
    np.testing.assert_array_equal(w, want)


def test_dequant_sweep_exact_rounding():
    rng = np.random.default_rng(7)
    n = 3000
    s = rng.uniform(0.005, 0.02, n)
    b = rng.normal(0, 0.01, n)
    # force exponent gaps well beyond fp64's 53 bits and exact ties
    b[:200] = rng.normal(0, 1e-20, 200)
    b[200:260] = 0.0
    s_bits = np.array([_bf16_bits_of(v) for v in s], np.uint16)
    b_bits = np.array([_bf16_bits_of(v) for v in b], np.uint16)
    q = rng.integers(0, 16, n)
    codes = np.zeros((n, 64), np.uint32)
    codes[:, 0] = q
    w = orc.dequant(_pack_codes(codes), s_bits[:, None], b_bits[:, None])[:, 0]
    for i in range(n):
        sv = Fraction(float(bf16_value(s_bits[i])))
        bv = Fraction(float(bf16_value(b_bits[i])))
        assert int(w[i]) == _exact_rne_bf16(sv * int(q[i]) + bv), i


def test_round_bf16_ties_and_sticky_low_part():
    one_plus_half = 1.0 + 2.0 ** -8  # midpoint of 1.0 and 1 + 2^-7
    assert orc.round_bf16(one_plus_half) == 0x3F80
    assert orc.round_bf16(one_plus_half, 1e-30) == 0x3F81
    assert orc.round_bf16(one_plus_half, -1e-30) == 0x3F80
    assert orc.round_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert orc.round_bf16(-one_plus_half, -1e-30) == 0xBF81
    assert orc.round_bf16(0.0) == 0 and orc.round_bf16(-0.0) == 0x8000
    assert orc.round_bf16(1e39) == 0x7F80
    assert orc.round_bf16(2.0 ** -133) == 0x0001  # smallest subnormal


# --------------------------------------------------------------- routing

def test_router_logits_match_library_dot():
    x = syn.activations(3, 17, 256)
    Wr = syn.router(3, 16, 256)
    bias = syn.zipf_bias(3, 16)
    keys = orc.logits(x, Wr, bias)
    ref = bf16_value(x) @ Wr.astype(np.float64).T
    want = (ref.astype(np.float32) + bias[None, :]).astype(np.float32)
    # fp64 sums in a different order may round to the neighbouring fp32
    np.testing.assert_allclose(keys, want, rtol=0, atol=np.abs(want).max() * 2 ** -22)
    assert (keys == want).mean() > 0.99


def test_select_all_equal_and_descending():
    k = 8
    ids, w = orc.select(np.zeros((3, 256), np.float32), k)
    assert (ids == np.arange(8)).all() and (w == 0.125).all()
    ids, _ = orc.select(-np.arange(256, dtype=np.float32)[None, :], k)
    assert list(ids[0]) == list(range(8))
    ids, _ = orc.select(np.arange(256, dtype=np.float32)[None, :], k)
    assert list(ids[0]) == list(range(255, 247, -1))


def test_select_ties_signed_zero_and_nan():
    keys = np.full((1, 16), -5.0, np.float32)
    keys[0, [3, 9]] = 2.0          # tie -> lower index first
    keys[0, 5] = -0.0
    keys[0, 1] = 0.0               # -0 == +0 -> index order 1, 5
    keys[0, 0] = np.nan            # NaN ranks below every number
    ids, w = orc.select(keys, 5)
    assert list(ids[0]) == [3, 9, 1, 5, 2]
    l = np.array([2.0, 2.0, 0.0, 0.0, -5.0])
    np.testing.assert_allclose(w[0], np.exp(l - 2) / np.exp(l - 2).sum(), rtol=1e-15)
    ids, _ = orc.select(np.full((1, 4), np.nan, np.float32), 2)
    assert list(ids[0]) == [0, 1]


def test_select_matches_brute_on_heavy_ties():
    rng = np.random.default_rng(11)
    keys = rng.integers(-3, 3, size=(200, 64)).astype(np.float32)
    keys[rng.random(keys.shape) < 0.02] = np.nan
    ids, w = orc.select(keys, 8)
    bids, bw = brute.select(keys, 8)
    np.testing.assert_array_equal(ids, bids)
    np.testing.assert_allclose(w, bw, rtol=1e-14)


def test_softmax_weights_equal_renormalised_full_softmax():
    keys = syn.router(5, 40, 256)  # any fp32 numbers
    ids, w = orc.select(keys, 8)
    full = np.exp(keys.astype(np.float64) - keys.max(axis=1, keepdims=True))
    full /= full.sum(axis=1, keepdims=True)
    pick = np.take_along_axis(full, ids, axis=1)
    np.testing.assert_allclose(w, pick / pick.sum(axis=1, keepdims=True), rtol=1e-12)
    assert np.abs(w.sum(axis=1) - 1).max() <= 8 * 2.0 ** -52
    assert (np.diff(w, axis=1) <= 0).all()  # slot order = descending weight


@pytest.mark.parametrize("T,E,k,BN", [(1, 256, 8, 128), (300, 16, 4, 7), (97, 256, 8, 32), (0, 8, 2, 4)])
def test_route_maps_invariants(T, E, k, BN):
    rng = np.random.default_rng(T + E)
    ids = np.array([rng.choice(E, k, replace=False) for _ in range(T)], np.int32).reshape(T, k)
    m = orc.route_maps(ids, E, n_shared=1, BN=BN)
    c, off, perm, inv = m["counts"], m["offsets"], m["perm"], m["inv"]
    P = T * k
    assert c.sum() == P and off[0] == 0 and off[E] == P and (np.diff(off) == c).all()
    assert sorted(perm.tolist()) == list(range(P))
    assert (inv[perm] == np.arange(P)).all() and (perm[inv] == np.arange(P)).all()
    flat = ids.ravel()
    for e in range(E):
        seg = perm[off[e]:off[e + 1]]
        assert (flat[seg] == e).all()
        assert (np.diff(seg) > 0).all()  # stable: ascending token order
    bc, boff, bperm, binv = brute.route_maps(ids, E)
    np.testing.assert_array_equal(c, bc)
    np.testing.assert_array_equal(off, boff)
    np.testing.assert_array_equal(perm, bperm)
    np.testing.assert_array_equal(inv, binv)
    bm = m["blockmap"]
    want_tiles = sum(-(-int(ce) // BN) for ce in c) + -(-T // BN)
    assert m["n_tiles"] == want_tiles == len(bm)
    routed = bm[bm[:, 0] < E]
    assert routed[:, 2].sum() == P and (bm[:, 2] <= BN).all() and (bm[:, 2] >= 1).all()
    shared = bm[bm[:, 0] == E]
    assert shared[:, 2].sum() == T and (shared[:, 1] >= P).all()
    # rows covered exactly once
    cover = np.zeros(P + T, np.int32)
    for e, r0, n, _ in bm:
        cover[r0:r0 + n] += 1
        if e < E:
            assert off[e] <= r0 and r0 + n <= off[e + 1]
    assert (cover == 1).all()


# --------------------------------------------------------------- whole layer

TINY = dict(H=256, E=16, k=4, I=128)


def _tiny_weights(seed, n_shared=1, centred=False, **dims):
    d = {**TINY, **dims}
    W = syn.experts(seed, d["E"] + n_shared, d["H"], d["I"], centred=centred)
    W["router"] = syn.router(seed, d["E"], d["H"])
    return orc.Dims(n_shared=n_shared, **d), W


@pytest.mark.parametrize("T", [1, 2, 3, 7, 33, 300])
@pytest.mark.parametrize("n_shared,centred,with_bias", [(1, False, False), (0, True, True), (1, True, False)])
def test_layer_matches_brute_force(T, n_shared, centred, with_bias):
    d, W = _tiny_weights(T, n_shared, centred)
    x = syn.activations(T, T, d.H)
    res = syn.activations(T, T, d.H, tensor=syn.T_RESID)
    bias = syn.zipf_bias(T, d.E) if with_bias else None
    r = orc.moe_layer(d, x, W, res=res, bias=bias, intermediates=True)
    bo, bx, keys, ids, w = brute.moe_layer(x, W, d.E, d.k, n_shared, res=res, bias=bias, keys=r["keys"])
    np.testing.assert_array_equal(ids, r["ids"])
    np.testing.assert_allclose(w, r["w"], rtol=1e-13)
    np.testing.assert_allclose(bx, r["out_exact"], rtol=0, atol=1e-10 * max(1.0, np.abs(bx).max()))
    assert (bo != r["out"]).mean() < 1e-3
    # and the oracle's own keys agree with a library dot product
    lib = (bf16_value(x) @ W["router"].astype(np.float64).T).astype(np.float32)
    if bias is not None:
        lib = (lib + bias[None, :]).astype(np.float32)
    np.testing.assert_allclose(r["keys"], lib, rtol=0, atol=np.abs(lib).max() * 2 ** -22)


@pytest.mark.parametrize("T", [1, 7, 33])
def test_layer_shared_gate_matches_brute_force(T):
    """The optional shared-expert gate, sigmoid(x . gate) on the shared
    expert's output, against the numpy statement (separate residual: the gate
    reads the expert input x, not the residual)."""
    d, W = _tiny_weights(50 + T)
    W["shared_gate"] = syn.shared_gate(50 + T, d.H)
    x = syn.activations(50 + T, T, d.H)
    res = syn.activations(50 + T, T, d.H, tensor=syn.T_RESID)
    r = orc.moe_layer(d, x, W, res=res, intermediates=True)
    bo, bx, keys, ids, w = brute.moe_layer(x, W, d.E, d.k, 1, res=res, keys=r["keys"])
    np.testing.assert_array_equal(ids, r["ids"])
    np.testing.assert_allclose(bx, r["out_exact"], rtol=0, atol=1e-10 * max(1.0, np.abs(bx).max()))


def test_layer_zero_shared_gate_halves_the_shared_expert():
    """gate = 0 gives sigmoid(0) = 1/2: the output moves by exactly half the
    shared expert's (bf16) output against the ungated layer."""
    d, W = _tiny_weights(61)
    x = syn.activations(61, 20, d.H)
    plain = orc.moe_layer(d, x, W, intermediates=True)
    W["shared_gate"] = np.zeros(d.H, np.float32)
    gated = orc.moe_layer(d, x, W, intermediates=True)
    y_sh = bf16_value(plain["y"][d.k * 20:])
    np.testing.assert_array_equal(plain["y"], gated["y"])
    np.testing.assert_allclose(gated["out_exact"], plain["out_exact"] - 0.5 * y_sh, rtol=0,
                               atol=1e-12 * np.abs(plain["out_exact"]).max())


def test_layer_zero_expert_weights_return_residual():
    d, W = _tiny_weights(1)
    for n in ("gate_s", "gate_b", "up_s", "up_b", "down_s", "down_b"):
        W[n][:] = 0
    x = syn.activations(2, 40, d.H)
    res = syn.activations(2, 40, d.H, tensor=syn.T_RESID)
    r = orc.moe_layer(d, x, W, res=res)
    np.testing.assert_array_equal(r["out"], res)


def test_layer_silu_of_zero_is_zero():
    d, W = _tiny_weights(2)
    W["gate_s"][:] = 0
    W["gate_b"][:] = 0  # g == 0 for every row -> h = silu(0) * u = 0
    x = syn.activations(3, 9, d.H)
    r = orc.moe_layer(d, x, W, intermediates=True)
    assert (r["h"] & 0x7FFF == 0).all()
    np.testing.assert_array_equal(r["out"], x)


def test_layer_constant_weights_closed_form():
    d, W = _tiny_weights(4)
    c = 2.0 ** -7
    for n in ("gate", "up", "down"):
        W[n + "_s"][:] = 0
        W[n + "_b"][:] = _bf16_bits_of(c)
    x = syn.activations(5, 12, d.H)
    r = orc.moe_layer(d, x, W)
    xs = bf16_value(x)
    for t in range(x.shape[0]):
        g = c * math.fsum(xs[t])  # g == u for every row of every expert
        h = float(bf16_value(np.array([orc.round_bf16(g / (1 + math.exp(-g)) * g)]))[0])
        y = float(bf16_value(np.array([orc.round_bf16(c * d.I * h)]))[0])
        # every expert gives the same y; the k weights sum to one; shared adds 1
        want = xs[t] + y + y
        np.testing.assert_allclose(r["out_exact"][t], want, rtol=1e-12, atol=1e-12)


def _dense_reference(x, W, e, res_add):
    """Library check: dequantise (brute force) and run the SwiGLU MLP with torch."""
    import torch
    xs = torch.tensor(bf16_value(x), dtype=torch.float64)
    wg = torch.tensor(bf16_value(brute.dequant(W["gate_q"][e], W["gate_s"][e], W["gate_b"][e])))
    wu = torch.tensor(bf16_value(brute.dequant(W["up_q"][e], W["up_s"][e], W["up_b"][e])))
    wd = torch.tensor(bf16_value(brute.dequant(W["down_q"][e], W["down_s"][e], W["down_b"][e])))
    h = torch.nn.functional.silu(xs @ wg.T) * (xs @ wu.T)
    h = torch.tensor(bf16_value(brute.round_bf16_bits(h.numpy())))
    y = torch.tensor(bf16_value(brute.round_bf16_bits((h @ wd.T).numpy())))
    return y.numpy()


def test_layer_single_expert_is_dense_swiglu_mlp():
    d, W = _tiny_weights(6, n_shared=0, E=1, k=1)
    x = syn.activations(6, 21, d.H)
    r = orc.moe_layer(d, x, W)
    want = bf16_value(x) + _dense_reference(x, W, 0, None)
    np.testing.assert_allclose(r["out_exact"], want, rtol=1e-12, atol=1e-9)


def test_layer_top_k_equals_E_is_full_softmax_mixture():
    d, W = _tiny_weights(8, n_shared=1, E=4, k=4, centred=True)
    x = syn.activations(8, 10, d.H)
    r = orc.moe_layer(d, x, W)
    keys = orc.logits(x, W["router"])
    p = np.exp(keys.astype(np.float64) - keys.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    want = bf16_value(x) + _dense_reference(x, W, 4, None)
    for e in range(4):
        want = want + p[:, e:e + 1] * _dense_reference(x, W, e, None)
    np.testing.assert_allclose(r["out_exact"], want, rtol=1e-10, atol=1e-9 * np.abs(want).max())


def test_layer_real_dims_brute_force_tokens():
    # real dims, a few tokens: oracle vs the numpy brute force at full size
    d = orc.Dims()
    W = syn.experts(0, 257, 2048, 512)
    W["router"] = syn.router(0, 256, 2048)
    x = syn.activations(0, 3, 2048)
    r = orc.moe_layer(d, x, W, intermediates=True)
    bo, bx, keys, ids, w = brute.moe_layer(x, W, 256, 8, 1, keys=r["keys"])
    np.testing.assert_array_equal(ids, r["ids"])
    np.testing.assert_allclose(bx, r["out_exact"], rtol=1e-12, atol=1e-9)
    assert_outputs_close(r["out"], bx)


def test_rmsnorm_closed_form_and_library():
    r = np.full((2, 256), _bf16_bits_of(3.0), np.uint16)
    x = orc.rmsnorm(r, 0.0)
    assert (x == _bf16_bits_of(1.0)).all()
    r = syn.activations(9, 20, 2048)
    x = bf16_value(orc.rmsnorm(r, 1e-6))
    rv = bf16_value(r)
    want = rv / np.sqrt((rv ** 2).mean(axis=1, keepdims=True) + 1e-6)
    np.testing.assert_array_equal(x, bf16_value(brute.round_bf16_bits(want)))
