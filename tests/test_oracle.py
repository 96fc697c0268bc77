"""Pins of the fp64 oracle against things other than itself (CPU only).

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong scale) fails at least one
of them; ``test_planted_*`` plant such slips in the oracle and check that
the pins catch them.
"""
import dataclasses
import json
import math
import os

import numpy as np
import pytest

from oracle import brute, mla
from synth.workloads import TINY, V2, Dims

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _rand_case(dims, S, T, seed):
    rng = np.random.default_rng(seed)
    d = dims
    w = {
        "w_dkv": rng.standard_normal((d.d_latent, d.d_model)) / math.sqrt(d.d_model),
        "w_kr": rng.standard_normal((d.d_rope, d.d_model)) / math.sqrt(d.d_model),
        "w_uk": rng.standard_normal((d.n_heads * d.d_nope, d.d_latent)) / math.sqrt(d.d_latent),
        "w_uv": rng.standard_normal((d.n_heads * d.d_v, d.d_latent)) / math.sqrt(d.d_latent),
        "w_o": rng.standard_normal((d.d_model, d.n_heads * d.d_v)) / math.sqrt(d.n_heads * d.d_v),
    }
    h = rng.standard_normal((S, d.d_model))
    q = rng.standard_normal((T, d.n_heads, d.d_nope + d.d_rope))
    return w, h, q


def _rows(dims, w, h):
    return mla.latent_rows(h, w["w_dkv"], w["w_kr"], np.arange(h.shape[0]), dims.rope_base)


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


SMALL_SHAPES = [
    Dims(d_model=6, n_heads=1, d_nope=3, d_v=2, d_latent=4, d_rope=2, page_size=4),
    Dims(d_model=8, n_heads=2, d_nope=4, d_v=3, d_latent=5, d_rope=4, page_size=4),
    TINY,
]


# --------------------------------------------------------------------------
# closed forms printed on the pages
# --------------------------------------------------------------------------
def test_cache_size_closed_forms():
    g = _load("cache_sizes.json")
    assert mla.mha_cache_elems(128, 128) == g["mha_elems_per_token_layer"]
    assert mla.mla_cache_elems(512, 64) == g["mla_elems_per_token_layer"]
    assert mla.mla_cache_elems(512, 64, layers=60) == g["mla_elems_60_layers"]
    assert mla.mha_cache_elems(128, 128, layers=60) == g["mha_elems_60_layers"]
    assert mla.gqa_equivalent_groups(512, 64, 128) == g["gqa_equivalent_groups"]
    ratio = mla.mla_cache_elems(512, 64) / mla.mha_cache_elems(128, 128)
    assert ratio == g["mla_over_mha"]
    assert mla.mla_cache_elems(512, 64) * 2 == g["bf16_row_bytes"]
    assert V2.row_width == 576
    # the quoted 93.3% is vs DeepSeek 67B and does not follow from these widths
    assert abs((1 - ratio) - g["quoted_reduction_vs_67B_context_only"]) > 0.04


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------
def test_rope_golden_pairs():
    for case in _load("rope_pairs.json")["cases"]:
        got = mla.rope(np.array(case["x"]), case["pos"], case["base"])
        np.testing.assert_allclose(got, case["expect"], rtol=0, atol=1e-15)


def test_rope_invariants():
    rng = np.random.default_rng(3)
    x, y = rng.standard_normal(64), rng.standard_normal(64)
    np.testing.assert_array_equal(mla.rope(x, 0), x)
    for pos in (1, 7, 131071):
        assert abs(np.linalg.norm(mla.rope(x, pos)) - np.linalg.norm(x)) < 1e-12
    # <R_m x, R_n y> depends on m - n only
    a = mla.rope(x, 5) @ mla.rope(y, 3)
    b = mla.rope(x, 9) @ mla.rope(y, 7)
    assert abs(a - b) < 1e-12
    # vectorised positions equal scalar calls
    X = rng.standard_normal((4, 8))
    P = np.array([0, 3, 10, 99])
    np.testing.assert_allclose(mla.rope(X, P), np.stack([mla.rope(X[i], P[i]) for i in range(4)]),
                               rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# paged addressing
# --------------------------------------------------------------------------
def test_slot_of_hand_example_and_bijection():
    assert mla.slot_of(np.array([[5, 2]]), 0, 6, 4) == 10
    assert mla.slot_of(np.array([[5, 2]]), 0, 3, 4) == 23
    rng = np.random.default_rng(0)
    P, lens = 8, [13, 1, 24, 8]
    pages = [(L + P - 1) // P for L in lens]
    perm = rng.permutation(sum(pages))
    bt = np.full((len(lens), max(pages)), -1)
    k = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[k:k + n]
        k += n
    slots = [mla.slot_of(bt, b, p, P) for b, L in enumerate(lens) for p in range(L)]
    assert len(set(slots)) == sum(lens)
    assert min(slots) >= 0 and max(slots) < sum(pages) * P
    for b, L in enumerate(lens):
        for p in range(L):
            assert mla.slot_of(bt, b, p, P) // P == bt[b, p // P]


# --------------------------------------------------------------------------
# worked examples (hand-derived exact answers)
# --------------------------------------------------------------------------
WORKED_DIMS = Dims(d_model=3, n_heads=1, d_nope=1, d_v=1, d_latent=1, d_rope=2, page_size=4)


def _worked(case, decode_fn):
    w = {k: np.array(case[k], dtype=np.float64) for k in ("w_dkv", "w_kr", "w_uk", "w_uv", "w_o")}
    h = np.array(case["h"])
    rows = _rows(WORKED_DIMS, w, h)
    q = np.array(case["q"]).reshape(1, 1, 3)
    return decode_fn(WORKED_DIMS, rows, q, w, 1)["u"][0]


@pytest.mark.parametrize("form", ["explicit", "absorbed"])
def test_worked_examples(form):
    fn = mla.decode_explicit if form == "explicit" else mla.decode_absorbed
    for case in _load("worked_examples.json")["cases"]:
        np.testing.assert_allclose(_worked(case, fn), case["expect_u"], rtol=0, atol=1e-14,
                                   err_msg=case["name"])


def test_worked_examples_brute():
    for case in _load("worked_examples.json")["cases"]:
        w = {k: case[k] for k in ("w_dkv", "w_kr", "w_uk", "w_uv", "w_o")}
        u = brute.decode(WORKED_DIMS, case["h"], [[case["q"][0]]], w, 1)[0]
        np.testing.assert_allclose(u, case["expect_u"], rtol=0, atol=1e-14, err_msg=case["name"])


# --------------------------------------------------------------------------
# brute force vs vectorised explicit; absorbed vs explicit
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dims", SMALL_SHAPES)
@pytest.mark.parametrize("S,T", [(1, 1), (5, 1), (5, 2), (64, 1)])
def test_brute_force_agrees(dims, S, T):
    if dims is TINY and S != 64 and T == 1:
        pytest.skip("tiny widths run at S=64 and the T=2 case only")
    w, h, q = _rand_case(dims, S, T, seed=S * 10 + T)
    ref = mla.decode_explicit(dims, _rows(dims, w, h), q, w, T)["u"]
    bw = {k: v.tolist() for k, v in w.items()}
    got = np.array(brute.decode(dims, h.tolist(), q.tolist(), bw, T))
    assert _rel(got, ref) < 1e-12


@pytest.mark.parametrize("dims", SMALL_SHAPES + [
    dataclasses.replace(V2, d_model=256, n_heads=4)])
@pytest.mark.parametrize("S,T", [(1, 1), (70, 1), (70, 2)])
def test_absorbed_equals_explicit(dims, S, T):
    w, h, q = _rand_case(dims, S, T, seed=S + T)
    rows = _rows(dims, w, h)
    e = mla.decode_explicit(dims, rows, q, w, T)
    a = mla.decode_absorbed(dims, rows, q, w, T)
    assert _rel(a["u"], e["u"]) < 1e-12
    assert _rel(a["o"], e["o"]) < 1e-12
    # latent output and value recovery: o_i = W^UV_i o_lat_i
    w_uv = w["w_uv"].reshape(dims.n_heads, dims.d_v, dims.d_latent)
    assert _rel(np.einsum("hvc,thc->thv", w_uv, a["o_lat"]), e["o"]) < 1e-12


# --------------------------------------------------------------------------
# softmax and masking invariants, special cases
# --------------------------------------------------------------------------
def test_softmax_rows_and_causal_mask():
    dims = TINY
    w, h, q = _rand_case(dims, 40, 2, seed=1)
    rows = _rows(dims, w, h)
    a = mla.decode_explicit(dims, rows, q, w, 2, return_attn=True)["attn"]
    assert (a >= 0).all()
    np.testing.assert_allclose(a.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert (a[0, :, 39] == 0).all()          # token at 38 does not see 39
    assert (a[1, :, 39] > 0).all()
    for t in range(2):
        for hd in range(dims.n_heads):
            np.testing.assert_allclose(
                mla.attention_weights_absorbed(dims, rows, q, w, 2, t, hd),
                a[t, hd, :38 + t + 1], rtol=0, atol=1e-12)


def test_single_slot_ignores_query():
    dims = TINY
    w, h, q = _rand_case(dims, 1, 1, seed=2)
    rows = _rows(dims, w, h)
    u1 = mla.decode_explicit(dims, rows, q, w, 1)["u"]
    u2 = mla.decode_explicit(dims, rows, 3.0 * q + 1.0, w, 1)["u"]
    c0 = rows[0, :dims.d_latent]
    expect = w["w_o"] @ (w["w_uv"] @ c0)      # a = [1]: o_i = W^UV_i c_0
    assert _rel(u1[0], expect) < 1e-12 and _rel(u2[0], expect) < 1e-12


def test_equal_rows_give_single_slot_answer():
    dims = TINY
    w, h, q = _rand_case(dims, 1, 1, seed=4)
    rows = np.repeat(_rows(dims, w, h), 17, axis=0)
    u = mla.decode_absorbed(dims, rows, q, w, 1)["u"]
    expect = w["w_o"] @ (w["w_uv"] @ rows[0, :dims.d_latent])
    assert _rel(u[0], expect) < 1e-12


def test_zero_query_and_rope_key_is_uniform():
    dims = TINY
    w, h, q = _rand_case(dims, 33, 1, seed=5)
    w["w_kr"] = np.zeros_like(w["w_kr"])
    q = np.zeros_like(q)
    rows = _rows(dims, w, h)
    o = mla.decode_explicit(dims, rows, q, w, 1)["o"][0]
    c_mean = rows[:, :dims.d_latent].mean(axis=0)
    expect = (w["w_uv"] @ c_mean).reshape(dims.n_heads, dims.d_v)
    assert _rel(o, expect) < 1e-12


def test_two_tokens_equal_two_single_decodes():
    dims = TINY
    w, h, q = _rand_case(dims, 30, 2, seed=6)
    rows = _rows(dims, w, h)
    both = mla.decode_explicit(dims, rows, q, w, 2)["u"]
    first = mla.decode_explicit(dims, rows[:29], q[:1], w, 1)["u"]
    second = mla.decode_explicit(dims, rows, q[1:], w, 1)["u"]
    assert _rel(both[0], first[0]) < 1e-13 and _rel(both[1], second[0]) < 1e-13


@pytest.mark.parametrize("T", [5, 40])
def test_chunk_of_tokens_equals_successive_single_decodes(T):
    """A chunk of T new tokens (prefill) is T single-token decodes, token t
    seeing the cache up to itself: the causal mask inside the chunk."""
    dims = SMALL_SHAPES[1]
    S = 70
    w, h, q = _rand_case(dims, S, T, seed=7 + T)
    rows = _rows(dims, w, h)
    chunk = mla.decode_explicit(dims, rows, q, w, T)["u"]
    for t in range(T):
        one = mla.decode_explicit(dims, rows[:S - T + t + 1], q[t:t + 1], w, 1)["u"][0]
        assert _rel(chunk[t], one) < 1e-12
    brute_u = brute.decode(dims, h.tolist(), q.tolist(), {k: v.tolist() for k, v in w.items()}, T)
    assert _rel(chunk, np.array(brute_u)) < 1e-12


def test_rope_key_is_shared_and_in_row():
    """k^R occupies columns d_c.. of the row, is the same for every head and
    carries the position (caching only c^KV would lose it)."""
    dims = TINY
    w, h, _ = _rand_case(dims, 3, 1, seed=7)
    rows = _rows(dims, w, h)
    np.testing.assert_allclose(rows[:, :dims.d_latent], h @ w["w_dkv"].T, rtol=0, atol=1e-13)
    raw = h @ w["w_kr"].T
    for p in range(3):
        np.testing.assert_allclose(rows[p, dims.d_latent:], mla.rope(raw[p], p), rtol=0, atol=1e-13)
    moved = mla.latent_rows(h, w["w_dkv"], w["w_kr"], np.arange(3) + 5)
    assert np.abs(moved[:, dims.d_latent:] - rows[:, dims.d_latent:]).max() > 1e-3


def test_error_stats():
    s = mla.error_stats(np.array([1.0, -2.0, 2.5]), np.array([1.0, -2.0, 3.0]))
    assert s["max_rel"] == pytest.approx(0.5 / 3.0) and s["mean_rel"] == pytest.approx(0.5 / 6.0)


# --------------------------------------------------------------------------
# planted mistakes: each must be caught by one of the pins above
# --------------------------------------------------------------------------
def _pins_pass():
    try:
        test_rope_golden_pairs()
        for form in ("explicit", "absorbed"):
            test_worked_examples(form)
        test_brute_force_agrees(SMALL_SHAPES[1], 5, 2)
        test_absorbed_equals_explicit(SMALL_SHAPES[1], 70, 2)
        test_softmax_rows_and_causal_mask()
    except AssertionError:
        return False
    return True


def test_planted_rope_sign(monkeypatch):
    orig = mla.rope
    monkeypatch.setattr(mla, "rope", lambda x, pos, base=10000.0: orig(x, -np.asarray(pos), base))
    assert not _pins_pass()


def test_planted_rope_frequency(monkeypatch):
    orig = mla.rope
    monkeypatch.setattr(mla, "rope", lambda x, pos, base=10000.0: orig(x, pos, base * 2))
    assert not _pins_pass()


def test_planted_scale(monkeypatch):
    monkeypatch.setattr(Dims, "softmax_scale", property(lambda s: 1.0 / math.sqrt(s.d_nope)))
    assert not _pins_pass()


def test_planted_head_slicing(monkeypatch):
    orig = mla.decode_explicit

    def bad(dims, rows, q, w, T, return_attn=False):
        w2 = dict(w)
        H, dn = dims.n_heads, dims.d_nope
        w2["w_uk"] = np.asarray(w["w_uk"]).reshape(dn, H, -1).transpose(1, 0, 2).reshape(H * dn, -1)
        return orig(dims, rows, q, w2, T, return_attn)
    monkeypatch.setattr(mla, "decode_explicit", bad)
    assert not _pins_pass()


def test_planted_dropped_rope_key(monkeypatch):
    orig = mla.latent_rows

    def bad(h, w_dkv, w_kr, positions, base=10000.0):
        r = orig(h, w_dkv, w_kr, positions, base)
        r[:, np.asarray(w_dkv).shape[0]:] = 0.0
        return r
    monkeypatch.setattr(mla, "latent_rows", bad)
    assert not _pins_pass()


def test_planted_unmasked_future(monkeypatch):
    orig = mla.decode_explicit

    def bad(dims, rows, q, w, T, return_attn=False):
        # every query sees every row (drops the causal mask between new tokens)
        out = {"u": [], "o": []}
        for t in range(T):
            r = orig(dims, rows, q[t:t + 1], w, 1, return_attn)
            out["u"].append(r["u"][0])
            out["o"].append(r["o"][0])
        res = {k: np.stack(v) for k, v in out.items()}
        if return_attn:
            res["attn"] = np.stack([orig(dims, rows, q[t:t + 1], w, 1, True)["attn"][0]
                                    for t in range(T)])
        return res
    monkeypatch.setattr(mla, "decode_explicit", bad)
    assert not _pins_pass()


# --------------------------------------------------------------------------
# query path: c^Q = W^DQ h, q^C = W^UQ c^Q, q^R = W^QR h
# --------------------------------------------------------------------------
QW = ("w_dkv", "w_kr", "w_uk", "w_uv", "w_o", "w_dq", "w_uq", "w_qr")


def _qdims(case):
    return dataclasses.replace(WORKED_DIMS, n_heads=case["n_heads"])


def _query_worked(case, decode_fn):
    dims = _qdims(case)
    w = {k: np.array(case[k], dtype=np.float64) for k in QW}
    h = np.array(case["h"])
    rows = _rows(dims, w, h)
    q = mla.query_from_hidden(dims, h[-1:], w["w_dq"], w["w_uq"], w["w_qr"])
    return q, decode_fn(dims, rows, q, w, 1)["u"][0]


@pytest.mark.parametrize("form", ["explicit", "absorbed"])
def test_query_path_worked_examples(form):
    fn = mla.decode_explicit if form == "explicit" else mla.decode_absorbed
    for case in _load("query_path_examples.json")["cases"]:
        q, u = _query_worked(case, fn)
        np.testing.assert_allclose(q, case["expect_q"], rtol=0, atol=1e-14, err_msg=case["name"])
        np.testing.assert_allclose(u, case["expect_u"], rtol=0, atol=1e-14, err_msg=case["name"])


def test_query_path_worked_examples_brute():
    for case in _load("query_path_examples.json")["cases"]:
        dims = _qdims(case)
        w = {k: case[k] for k in QW}
        q = brute.query(dims, case["h"][-1], w)
        np.testing.assert_allclose(q, case["expect_q"][0], rtol=0, atol=1e-14, err_msg=case["name"])
        u = brute.decode(dims, case["h"], [q], w, 1)[0]
        np.testing.assert_allclose(u, case["expect_u"], rtol=0, atol=1e-14, err_msg=case["name"])


@pytest.mark.parametrize("dims", SMALL_SHAPES)
@pytest.mark.parametrize("d_cq", [3, 7])
def test_query_path_brute_force_agrees(dims, d_cq):
    rng = np.random.default_rng(d_cq)
    d = dims
    w = {"w_dq": rng.standard_normal((d_cq, d.d_model)),
         "w_uq": rng.standard_normal((d.n_heads * d.d_nope, d_cq)),
         "w_qr": rng.standard_normal((d.n_heads * d.d_rope, d.d_model))}
    h = rng.standard_normal((3, d.d_model))
    q = mla.query_from_hidden(d, h, w["w_dq"], w["w_uq"], w["w_qr"])
    ref = [brute.query(d, list(r), {k: v.tolist() for k, v in w.items()}) for r in h]
    assert _rel(q, np.array(ref)) < 1e-12


def _query_pins_pass():
    try:
        test_query_path_worked_examples("explicit")
        test_query_path_brute_force_agrees(SMALL_SHAPES[1], 3)
    except AssertionError:
        return False
    return True


def test_query_pins_pass_unplanted():
    assert _query_pins_pass()


def test_planted_query_rope_from_latent(monkeypatch):
    """q^R taken from c^Q instead of h (a plausible misreading)."""
    def bad(dims, h, w_dq, w_uq, w_qr):
        H, dn, dr = dims.n_heads, dims.d_nope, dims.d_rope
        c_q = np.asarray(h) @ np.asarray(w_dq).T
        q_c = (c_q @ np.asarray(w_uq).T).reshape(-1, H, dn)
        w_qr = np.asarray(w_qr)
        if w_qr.shape[1] != c_q.shape[1]:
            return np.full(q_c.shape[:2] + (dn + dr,), np.nan)
        q_r = (c_q @ w_qr.T).reshape(-1, H, dr)
        return np.concatenate([q_c, q_r], axis=2)
    monkeypatch.setattr(mla, "query_from_hidden", bad)
    assert not _query_pins_pass()


def test_planted_query_head_order(monkeypatch):
    """W^QR rows taken head-interleaved instead of head-major."""
    orig = mla.query_from_hidden

    def bad(dims, h, w_dq, w_uq, w_qr):
        H, dr = dims.n_heads, dims.d_rope
        w2 = np.asarray(w_qr).reshape(dr, H, -1).transpose(1, 0, 2).reshape(H * dr, -1)
        return orig(dims, h, w_dq, w_uq, w2)
    monkeypatch.setattr(mla, "query_from_hidden", bad)
    assert not _query_pins_pass()


def test_planted_query_dropped_up_projection(monkeypatch):
    """q^C = c^Q (W^UQ dropped) where the widths allow it."""
    def bad(dims, h, w_dq, w_uq, w_qr):
        H, dn, dr = dims.n_heads, dims.d_nope, dims.d_rope
        c_q = np.asarray(h) @ np.asarray(w_dq).T
        q_c = np.resize(c_q, (c_q.shape[0], H * dn)).reshape(-1, H, dn)
        q_r = (np.asarray(h) @ np.asarray(w_qr).T).reshape(-1, H, dr)
        return np.concatenate([q_c, q_r], axis=2)
    monkeypatch.setattr(mla, "query_from_hidden", bad)
    assert not _query_pins_pass()


def test_planted_query_swapped_parts(monkeypatch):
    """[q^R ; q^C] instead of [q^C ; q^R] per head."""
    orig = mla.query_from_hidden

    def bad(dims, h, w_dq, w_uq, w_qr):
        q = orig(dims, h, w_dq, w_uq, w_qr)
        return np.concatenate([q[..., dims.d_nope:], q[..., :dims.d_nope]], axis=2)[..., :q.shape[2]]
    monkeypatch.setattr(mla, "query_from_hidden", bad)
    assert not _query_pins_pass()


# --------------------------------------------------------------------------
# multi-layer step: h_{j+1} = h_j + u_j, each layer with its own cache
# --------------------------------------------------------------------------
def _stack_case():
    case = _load("layer_stack_examples.json")["cases"][0]
    layers = []
    for L in case["layers"]:
        w = {k: np.array(L[k], dtype=np.float64) for k in QW}
        rows = _rows(WORKED_DIMS, w, np.array(L["prefix_h"]))
        layers.append({"w": w, "prefix_rows": rows})
    return case, layers


@pytest.mark.parametrize("form", ["explicit", "absorbed"])
def test_layer_stack_worked_example(form):
    case, layers = _stack_case()
    r = mla.decode_layers(WORKED_DIMS, layers, np.array(case["h_new"]), 1, form=form)
    np.testing.assert_allclose(r["u"], case["expect_u"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(r["h"], case["expect_h"], rtol=0, atol=1e-14)


def test_layer_stack_worked_example_brute():
    case = _load("layer_stack_examples.json")["cases"][0]
    layers = [{"w": {k: L[k] for k in QW}, "prefix_h": L["prefix_h"]} for L in case["layers"]]
    h = brute.decode_layers(WORKED_DIMS, layers, case["h_new"], 1)
    np.testing.assert_allclose(h, case["expect_h"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("T", [1, 2])
def test_layer_stack_brute_force_agrees(T):
    d = dataclasses.replace(SMALL_SHAPES[1], d_cq=3)
    rng = np.random.default_rng(11 + T)
    layers, blayers = [], []
    for _ in range(3):
        w = {"w_dkv": rng.standard_normal((d.d_latent, d.d_model)),
             "w_kr": rng.standard_normal((d.d_rope, d.d_model)),
             "w_uk": rng.standard_normal((d.n_heads * d.d_nope, d.d_latent)),
             "w_uv": rng.standard_normal((d.n_heads * d.d_v, d.d_latent)),
             "w_o": rng.standard_normal((d.d_model, d.n_heads * d.d_v)) * 0.3,
             "w_dq": rng.standard_normal((3, d.d_model)),
             "w_uq": rng.standard_normal((d.n_heads * d.d_nope, 3)),
             "w_qr": rng.standard_normal((d.n_heads * d.d_rope, d.d_model))}
        ph = rng.standard_normal((4, d.d_model))
        layers.append({"w": w, "prefix_rows": _rows(d, w, ph)})
        blayers.append({"w": {k: v.tolist() for k, v in w.items()}, "prefix_h": ph.tolist()})
    h0 = rng.standard_normal((T, d.d_model))
    r = mla.decode_layers(d, layers, h0, T)
    hb = brute.decode_layers(d, blayers, h0.tolist(), T)
    assert _rel(r["h"], np.array(hb)) < 1e-12


def _stack_pins_pass():
    try:
        test_layer_stack_worked_example("explicit")
        test_layer_stack_brute_force_agrees(2)
    except AssertionError:
        return False
    return True


def test_planted_stack_without_residual(monkeypatch):
    orig = mla.decode_layers

    def bad(dims, layers, h_new, T, base=None, form="explicit"):
        h = np.asarray(h_new, dtype=np.float64)
        us = []
        for layer in layers:
            r = orig(dims, [layer], h, T, base, form)
            us.append(r["u"][0])
            h = r["u"][0]          # the residual dropped
        return {"h": h, "u": np.stack(us)}
    monkeypatch.setattr(mla, "decode_layers", bad)
    assert not _stack_pins_pass()


def test_planted_stack_same_input_every_layer(monkeypatch):
    orig = mla.decode_layers

    def bad(dims, layers, h_new, T, base=None, form="explicit"):
        h0 = np.asarray(h_new, dtype=np.float64)
        h, us = h0, []
        for layer in layers:
            r = orig(dims, [layer], h0, T, base, form)   # every layer reads h_0
            us.append(r["u"][0])
            h = h + r["u"][0]
        return {"h": h, "u": np.stack(us)}
    monkeypatch.setattr(mla, "decode_layers", bad)
    assert not _stack_pins_pass()
