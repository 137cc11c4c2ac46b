"""The output tolerance accepts the oracle's own bf16 rounding and one-ulp
flips of the bf16 expert outputs, and rejects plausible mistakes planted in
the oracle's result (a dropped term, a wrong row, a perturbed element)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as orc
import synthetic as syn
from tests.tolerances import bf16_half_ulp, bf16_value, intermediate_allowance, output_errors


@pytest.fixture(scope="module")
def layer():
    d = orc.Dims(H=256, E=16, k=4, I=128, n_shared=1)
    W = syn.experts(31, 17, 256, 128, centred=True)
    W["router"] = syn.router(31, 16, 256)
    x = syn.activations(31, 64, 256)
    ref = orc.moe_layer(d, x, W, intermediates=True)
    return d, W, x, ref


def _recombine(ref, k, T, y, w=None, drop_shared=False):
    """fp64 combine of bf16 rows y (block-map row order) -> bf16 bits."""
    from oracle import brute
    ids = ref["ids"]
    w = ref["w"] if w is None else w
    perm = np.argsort(ids.ravel(), kind="stable")
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    yv = bf16_value(y)
    acc = bf16_value(ref["x"]).copy()
    if not drop_shared:
        acc += yv[k * T:k * T + T]
    for j in range(k):
        acc += w[:, j:j + 1] * yv[inv[np.arange(T) * k + j]]
    return brute.round_bf16_bits(acc)


def test_oracle_rounded_output_passes(layer):
    d, W, x, ref = layer
    r = output_errors(ref["out"], ref["out_exact"], intermediate_allowance(ref, d.k, 1))
    assert r["ok"] and r["max_beyond_half_ulp"] <= 0


def test_one_ulp_flips_of_y_pass(layer):
    d, W, x, ref = layer
    T = x.shape[0]
    rng = np.random.default_rng(0)
    y = ref["y"].copy()
    flip = rng.random(y.shape) < 0.01
    y[flip] = y[flip] + np.where(rng.random(flip.sum()) < 0.5, 1, -1).astype(np.uint16)  # +-1 ulp
    out = _recombine({**ref, "x": x}, d.k, T, y)
    assert output_errors(out, ref["out_exact"], intermediate_allowance(ref, d.k, 1))["ok"]


def test_planted_mistakes_fail(layer):
    d, W, x, ref = layer
    T, k = x.shape[0], d.k
    allow = intermediate_allowance(ref, k, 1)
    base = {**ref, "x": x}
    # dropped shared-expert term
    out = _recombine(base, k, T, ref["y"], drop_shared=True)
    assert not output_errors(out, ref["out_exact"], allow)["ok"]
    # one token reads a wrong expert row
    y = ref["y"].copy()
    y[[0, 1]] = y[[1, 0]]
    out = _recombine(base, k, T, y)
    assert not output_errors(out, ref["out_exact"], allow)["ok"]
    # slot weights swapped for one token
    w = ref["w"].copy()
    w[3, [0, k - 1]] = w[3, [k - 1, 0]]
    out = _recombine(base, k, T, ref["y"], w=w)
    assert not output_errors(out, ref["out_exact"], allow)["ok"]
    # one element off by 5% of rms
    out = ref["out"].copy()
    rms = np.sqrt(np.mean(ref["out_exact"] ** 2))
    v = bf16_value(out[7:8, 11:12]) + 0.05 * rms + bf16_half_ulp(bf16_value(out[7:8, 11:12]))
    from oracle import brute
    out[7, 11] = brute.round_bf16_bits(v)[0, 0]
    assert not output_errors(out, ref["out_exact"], allow)["ok"]
