"""Pins of the FP8 cache oracle (oracle.fp8) against what the E4M3
definition and the mathematics fix, none of which retypes the oracle:

* hand-derived code/value pairs of the E4M3 layout (tests/golden/e4m3_examples.json);
* every finite code decodes and encodes back to itself;
* encoding equals the exhaustive nearest finite code (ties to even);
* encoding equals torch's float8_e4m3fn cast (a library routine) in range;
* bf16 rounding equals torch's bfloat16 cast;
* the row quantiser: a hand example, rows that are exactly representable
  come back exactly, the largest element takes the largest code, every
  value lies within half a code step, power-of-two scaling commutes, zero
  rows, and the decode over dequantised rows nears the exact decode.

``test_planted_*`` plant slips in the oracle and check that a pin fails.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import fp8
from oracle import mla as omla
from synth.workloads import Dims

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_examples.json")
FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def check_golden():
    g = _golden()
    for code, value in g["decode"]:
        assert fp8.e4m3_decode(np.array([code]))[0] == value, (code, value)
    for value, code in g["encode"]:
        assert fp8.e4m3_encode(np.array([value]))[0] == code, (value, code)


def check_roundtrip():
    v = fp8.e4m3_decode(FINITE)
    assert np.array_equal(fp8.e4m3_encode(v), FINITE)


def check_nearest(n=4000, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=n) * np.exp2(rng.uniform(-11, 9, size=n))
    x = np.concatenate([x, fp8.e4m3_decode(FINITE[:-1]) / 2 + fp8.e4m3_decode(FINITE[1:]) / 2])
    vals = fp8.e4m3_decode(FINITE)
    got = fp8.e4m3_encode(x)
    for xi, ci in zip(x, got):
        t = min(max(xi, -448.0), 448.0)
        d = np.abs(vals - t)
        best = FINITE[d == d.min()]
        if len(best) > 1:   # a tie: the even mantissa (the two differ in the last bit)
            best = best[(best & 1) == 0]
            if len(best) > 1:   # +0 and -0
                best = best[np.signbit(fp8.e4m3_decode(best)) == np.signbit(t)]
        assert ci == best[0], (xi, ci, best)


def check_row_quantiser():
    # hand example (d_c = 4, d_R = 2): amax 1, s = fp32(1/448), x = 448 c
    rows = np.array([[1.0, -0.5, 0.25, 0.0, 2.0, -1.0]])
    q = fp8.quantize_rows(rows, 4)
    assert q["codes"].tolist() == [[0x7E, 0xF6, 0x6E, 0x00]]
    assert q["scale"][0] == np.float32(1.0) / np.float32(448.0)
    assert q["kr"].tolist() == [[896.0, -448.0]]
    # exactly representable rows come back exactly: codes with 448 present,
    # scale 2^-4 (then 448/amax = 16 exactly)
    rng = np.random.default_rng(3)
    codes = rng.choice(FINITE, size=(16, 32))
    codes[:, 0] = 0x7E
    c = fp8.e4m3_decode(codes) * 2.0 ** -4
    kr = fp8.bf16_round(rng.normal(size=(16, 8)).astype(np.float32)).astype(np.float64)
    q = fp8.quantize_rows(np.concatenate([c, kr], axis=1), 32)
    got = fp8.e4m3_decode(q["codes"])
    assert np.array_equal(got, fp8.e4m3_decode(codes))   # -0 and +0 may swap codes
    assert np.all(q["scale"] == np.float32(2.0 ** -4))
    assert np.array_equal(q["deq"], np.concatenate([c, kr], axis=1))
    # random rows: the largest element takes +-448; every value within half a
    # code step of the (bf16) input; never a NaN code
    rows = rng.normal(size=(64, 40)) * np.exp2(rng.uniform(-8, 8, size=(64, 1)))
    q = fp8.quantize_rows(rows, 32)
    cb = fp8.bf16_round(rows[:, :32].astype(np.float32)).astype(np.float64)
    amax_at = np.argmax(np.abs(cb), axis=1)
    assert np.all(np.abs(fp8.e4m3_decode(q["codes"][np.arange(64), amax_at])) == 448.0)
    assert not np.any((q["codes"] & 0x7F) == 0x7F)
    x = cb / q["scale"][:, None].astype(np.float64)
    step = np.where(np.abs(x) < 2.0 ** -6, 2.0 ** -9,
                    np.exp2(np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -6)))) / 8.0)
    err = np.abs(q["deq"][:, :32] - cb) / q["scale"][:, None]
    assert np.all(err <= 0.5 * step * (1 + 1e-5) + 1e-6 * np.abs(x))
    # power-of-two scaling of a row commutes with quantisation
    q2 = fp8.quantize_rows(rows * 2.0 ** 5, 32)
    assert np.array_equal(q2["codes"], q["codes"])
    assert np.array_equal(q2["scale"], q["scale"] * np.float32(32.0))
    # an all-zero latent: scale 1, codes 0, k^R stored as is
    z = fp8.quantize_rows(np.array([[0.0] * 4 + [0.5, -3.0]]), 4)
    assert z["scale"][0] == 1.0 and not z["codes"].any() and z["kr"].tolist() == [[0.5, -3.0]]


def test_golden():
    check_golden()


def test_roundtrip_every_finite_code():
    check_roundtrip()


def test_encode_is_nearest_with_ties_to_even():
    check_nearest()


def test_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    x = (rng.normal(size=100000) * np.exp2(rng.uniform(-12, 8, size=100000)))
    x = np.clip(x, -448, 448).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x.astype(np.float64)), ref)


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(2)
    x = (rng.normal(size=100000) * np.exp2(rng.uniform(-30, 30, size=100000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(fp8.bf16_round(x), ref)


def test_row_quantiser():
    check_row_quantiser()


def test_fp8_decode_nears_the_exact_decode():
    """The decode over dequantised rows departs from the exact decode by the
    quantisation alone: within a few per cent of u on random rows, and not
    at all when the rows are exactly representable."""
    d = Dims(d_model=32, n_heads=4, d_nope=8, d_v=8, d_latent=16, d_rope=4, page_size=4)
    rng = np.random.default_rng(5)
    w = {"w_uk": rng.normal(size=(32, 16)) / 4, "w_uv": rng.normal(size=(32, 16)) / 4,
         "w_o": rng.normal(size=(32, 32)) / 6}
    rows = rng.normal(size=(40, 20))
    q = rng.normal(size=(2, 4, 12))
    exact = omla.decode_explicit(d, rows, q, w, 2)["u"]
    quant = omla.decode_explicit(d, fp8.quantize_rows(rows, 16)["deq"], q, w, 2)["u"]
    s = omla.error_stats(quant, exact)
    assert 1e-4 < s["mean_rel"] < 0.06, s


# ---------------------------------------------------------------------------
# planted mistakes: each must be caught by one of the pins above
# ---------------------------------------------------------------------------
def _fails(check):
    with pytest.raises(AssertionError):
        check()


def test_pins_pass_unplanted():
    check_golden()
    check_roundtrip()
    check_nearest(500)
    check_row_quantiser()


def test_planted_exponent_bias(monkeypatch):
    orig = fp8.e4m3_decode
    monkeypatch.setattr(fp8, "e4m3_decode", lambda c: orig(c) / 2.0)
    _fails(check_golden)


def test_planted_flushed_subnormals(monkeypatch):
    orig = fp8.e4m3_encode
    monkeypatch.setattr(fp8, "e4m3_encode",
                        lambda x: np.where(np.abs(np.asarray(x)) < 2.0 ** -6, 0, orig(x)).astype(np.uint8))
    _fails(check_golden)


def test_planted_round_half_up(monkeypatch):
    orig = fp8.e4m3_encode

    def bad(x):
        x = np.asarray(x, dtype=np.float64)
        c = orig(x)
        v = fp8.e4m3_decode(c)
        up = orig(x * (1 + 2.0 ** -12))   # nudged past a tie
        return np.where(np.abs(x) == np.abs(v), c, up).astype(np.uint8)
    monkeypatch.setattr(fp8, "e4m3_encode", bad)
    _fails(lambda: check_nearest(500))


def test_planted_no_saturation(monkeypatch):
    orig = fp8.e4m3_encode
    monkeypatch.setattr(fp8, "e4m3_encode",
                        lambda x: np.where(np.abs(np.asarray(x)) > 448, 0x7F, orig(x)).astype(np.uint8))
    _fails(check_golden)


def test_planted_scale_from_256(monkeypatch):
    orig = fp8.quantize_rows

    def bad(rows, d_latent):
        q = orig(rows, d_latent)
        q["scale"] = q["scale"] * np.float32(448.0 / 256.0)
        q["deq"][:, :d_latent] *= 448.0 / 256.0
        return q
    monkeypatch.setattr(fp8, "quantize_rows", bad)
    _fails(check_row_quantiser)


def test_planted_rope_key_not_divided(monkeypatch):
    orig = fp8.quantize_rows

    def bad(rows, d_latent):
        q = orig(rows, d_latent)
        q["kr"] = fp8.bf16_round(np.asarray(rows[:, d_latent:], dtype=np.float32))
        return q
    monkeypatch.setattr(fp8, "quantize_rows", bad)
    _fails(check_row_quantiser)
